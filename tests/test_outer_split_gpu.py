"""Outer split (qStartIdx / kvStartIdx): per-sequence global starts of the
query and key/value chunks shift the window onto global positions.  The CUDA
path is compared with the oracle given the same starts, and a sequence cut
into query chunks must reproduce the whole-sequence result."""

import numpy as np
import pytest
import torch

from varlen_flashattention_backward_gb300 import binding as fa
from varlen_flashattention_backward_gb300 import build as fb
from varlen_flashattention_backward_gb300 import workloads as wl

from _helpers import TOL, assert_close, f64, gpu_forward_backward, oracle_full, rel_err

pytestmark = pytest.mark.gpu
BIG = wl.UNBOUNDED
DEV = torch.device("cuda:0")
IMPLS = {"simt": fa.FA_BWD_SIMT, "tcgen05": fa.FA_BWD_TCGEN05}

CASES = {
    # second query chunk of a causal sequence against its whole key range, and
    # a key chunk that starts inside the sequence
    "causal_chunks": (wl.Workload(60, "bf16", [100, 140], 2, 128, BIG, 0, seed=21,
                                  lens_kv=[260, 140]), [160, 0], [0, 30]),
    "band_gqa_dropout": (wl.Workload(61, "bf16", [130, 70], 4, 128, 50, 10, keep_prob=0.85,
                                     seed=22, n_heads_kv=2, lens_kv=[90, 200]), [40, 7], [0, 100]),
    "fp32_band": (wl.Workload(62, "fp32", [65, 30], 2, 64, 20, 3, seed=23), [5, 1000], [0, 990]),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    fb.build()
    fa.lib()
    torch.cuda.set_device(DEV)


@pytest.mark.parametrize("impl", ["simt", "tcgen05"])
@pytest.mark.parametrize("name", list(CASES))
def test_starts_against_oracle(name, impl):
    w, qs, ks = CASES[name]
    if impl == "tcgen05" and (w.dtype == "fp32" or w.head_dim not in (64, 128)):
        pytest.skip("tcgen05 kernel not built for this case")
    tensors = wl.make_tensors(w)
    mask_np = wl.make_keep_mask(w)
    mask = None if mask_np is None else torch.from_numpy(mask_np).to(DEV)
    out = gpu_forward_backward(w, tensors, DEV, IMPLS[impl], mask, q_start=qs, kv_start=ks)
    ref = oracle_full(w, tensors, mask_np, q_start=qs, kv_start=ks)
    assert_close(out, ref, TOL[w.dtype])


def test_query_chunks_reproduce_the_whole_sequence():
    """A causal 2048-token sequence cut into three query chunks: each chunk's
    backward (with its global start) gives the whole run's dQ rows, and the
    chunks' dK, dV add up to the whole run's (a context-parallel caller)."""
    L, cuts = 2048, [0, 700, 1536, 2048]
    w = wl.Workload(63, "bf16", [L], 4, 128, BIG, 0, seed=24)
    q, k, v, dy = (t.to(DEV) for t in wl.make_tensors(w))
    y, m, l = fa.fwd(q, k, v, [L], [L], w.scale, BIG, 0)
    dq, dk, dv = fa.bwd(q, k, v, dy, y, m, l, [L], [L], w.scale, BIG, 0)
    dk_sum = torch.zeros(dk.shape, dtype=torch.float32, device=DEV)
    dv_sum = torch.zeros_like(dk_sum)
    for a, b in zip(cuts[:-1], cuts[1:]):
        yc, mc, lc = fa.fwd(q[a:b], k, v, [b - a], [L], w.scale, BIG, 0, q_start=[a],
                            kv_start=[0])
        dqc, dkc, dvc = fa.bwd(q[a:b], k, v, dy[a:b], yc, mc, lc, [b - a], [L], w.scale, BIG, 0,
                               q_start=[a], kv_start=[0])
        torch.cuda.synchronize()
        assert rel_err(f64(yc), f64(y[a:b])) <= 1e-2
        assert rel_err(f64(dqc), f64(dq[a:b])) <= 1e-2
        dk_sum += dkc.float()
        dv_sum += dvc.float()
    assert rel_err(f64(dk_sum), f64(dk)) <= 1e-2
    assert rel_err(f64(dv_sum), f64(dv)) <= 1e-2


MODE_CASES = {
    # Lq < Lk, Lq > Lk and a zero-length sequence, for both lower-triangular modes
    "mode2": (wl.Workload(64, "bf16", [100, 260, 0, 37], 2, 128, 3, 5, seed=25,
                          lens_kv=[230, 140, 9, 37]), 2),
    "mode3": (wl.Workload(65, "bf16", [100, 260, 0, 37], 2, 128, 3, 5, seed=26,
                          lens_kv=[230, 140, 9, 37]), 3),
    "mode3_gqa_dropout": (wl.Workload(66, "bf16", [150, 64], 4, 128, 0, 0, keep_prob=0.8,
                                      seed=27, n_heads_kv=2, lens_kv=[300, 40]), 3),
    "mode4_fp32": (wl.Workload(67, "fp32", [70, 33], 2, 64, 9, 2, seed=28,
                               lens_kv=[50, 90]), 4),
}


@pytest.mark.parametrize("impl", ["simt", "tcgen05"])
@pytest.mark.parametrize("name", list(MODE_CASES))
def test_sparse_modes_against_oracle(name, impl):
    w, mode = MODE_CASES[name]
    if impl == "tcgen05" and (w.dtype == "fp32" or w.head_dim not in (64, 128)):
        pytest.skip("tcgen05 kernel not built for this case")
    tensors = wl.make_tensors(w)
    mask_np = wl.make_keep_mask(w)
    mask = None if mask_np is None else torch.from_numpy(mask_np).to(DEV)
    q, k, v, dy = (t.to(DEV) for t in tensors)
    y, m, l = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens,
                     w.keep_prob, mask, sparse_mode=mode)
    dq, dk, dv = fa.bwd(q, k, v, dy, y, m, l, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                        w.next_tokens, w.keep_prob, mask, impl=IMPLS[impl], sparse_mode=mode)
    torch.cuda.synchronize()
    qn, kn, vn, dyn = (f64(t) for t in tensors)
    import oracle
    ry, rm, rl = oracle.varlen_forward(qn, kn, vn, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                                       w.next_tokens, mask_np, w.keep_prob, sparse_mode=mode)
    rdq, rdk, rdv = oracle.varlen_backward(qn, kn, vn, dyn, ry, rm, rl, w.lens, w.lens_kv,
                                           w.scale, w.pre_tokens, w.next_tokens, mask_np,
                                           w.keep_prob, sparse_mode=mode)
    assert_close(dict(y=y, dq=dq, dk=dk, dv=dv), dict(y=ry, dq=rdq, dk=rdk, dv=rdv),
                 TOL[w.dtype])


def _random_mask(w, seed, density, pitch16=False):
    """Seeded uint8 mask, a few rows / columns wider than the longest
    sequence; with pitch16 its row pitch is a multiple of 16 bytes (the
    tensor-core kernel then loads its tiles by TMA)."""
    g = np.random.default_rng(seed)
    rows, cols = max(w.lens) + 3, max(w.lens_kv) + 5
    if pitch16:
        cols = (cols + 15) // 16 * 16
    elif cols % 16 == 0:
        cols += 1
    return (g.random((rows, cols)) < density).astype(np.uint8)


MASK_CASES = {
    "mode1_ragged": (wl.Workload(68, "bf16", [100, 260, 0, 37], 2, 128, 0, 0, seed=29,
                                 lens_kv=[230, 140, 9, 37]), 1, 0.3),
    "mode0_band_and_mask_gqa": (wl.Workload(69, "bf16", [200, 90], 4, 128, 60, 10, seed=30,
                                            n_heads_kv=2), 0, 0.2),
    "mode1_dropout": (wl.Workload(70, "bf16", [150, 64], 2, 128, 0, 0, keep_prob=0.85, seed=31),
                      1, 0.5),
    "mode1_fp32": (wl.Workload(71, "fp32", [70, 33], 2, 64, 0, 0, seed=32, lens_kv=[50, 90]),
                   1, 0.3),
    "mode1_d64": (wl.Workload(72, "bf16", [140, 70], 2, 64, 0, 0, seed=33, lens_kv=[90, 200]),
                  1, 0.3),
}


@pytest.mark.parametrize("pitch16", [False, True])
@pytest.mark.parametrize("impl", ["simt", "tcgen05"])
@pytest.mark.parametrize("name", list(MASK_CASES))
def test_atten_mask_against_oracle(name, impl, pitch16):
    w, mode, density = MASK_CASES[name]
    if impl == "tcgen05" and (w.dtype == "fp32" or w.head_dim not in (64, 128)):
        pytest.skip("tcgen05 kernel not built for this case")
    am_np = _random_mask(w, w.seed, density, pitch16)
    am = torch.from_numpy(am_np).to(DEV)
    tensors = wl.make_tensors(w)
    mask_np = wl.make_keep_mask(w)
    mask = None if mask_np is None else torch.from_numpy(mask_np).to(DEV)
    q, k, v, dy = (t.to(DEV) for t in tensors)
    y, m, l = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens,
                     w.keep_prob, mask, sparse_mode=mode, atten_mask=am)
    dq, dk, dv = fa.bwd(q, k, v, dy, y, m, l, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                        w.next_tokens, w.keep_prob, mask, impl=IMPLS[impl], sparse_mode=mode,
                        atten_mask=am)
    torch.cuda.synchronize()
    import oracle
    qn, kn, vn, dyn = (f64(t) for t in tensors)
    ry, rm, rl = oracle.varlen_forward(qn, kn, vn, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                                       w.next_tokens, mask_np, w.keep_prob, sparse_mode=mode,
                                       atten_mask=am_np)
    rdq, rdk, rdv = oracle.varlen_backward(qn, kn, vn, dyn, ry, rm, rl, w.lens, w.lens_kv,
                                           w.scale, w.pre_tokens, w.next_tokens, mask_np,
                                           w.keep_prob, sparse_mode=mode, atten_mask=am_np)
    assert_close(dict(y=y, dq=dq, dk=dk, dv=dv), dict(y=ry, dq=rdq, dk=rdk, dv=rdv),
                 TOL[w.dtype])
