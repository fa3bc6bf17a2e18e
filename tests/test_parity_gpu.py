"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.  Bar: max|err| <= 1e-4 * max|ref| per output tensor
for fp32 and <= 2e-2 * max|ref| for 16-bit types.

Small problems are compared element by element over the whole batch; the
full-size workloads 3-5 are run in the launch configuration bench.py times
(default kernel choice) and compared element by element on whole sampled
(sequence, head) units, with sum invariants checked over every unit."""

import math

import numpy as np
import pytest
import torch

import oracle
from varlen_flashattention_backward_gb300 import binding as fa
from varlen_flashattention_backward_gb300 import build as fb
from varlen_flashattention_backward_gb300 import workloads as wl

from _helpers import (TOL, assert_close, device_mask, f64, gpu_forward_backward, oracle_full,
                      rel_err, unit_check)

pytestmark = pytest.mark.gpu
BIG = wl.UNBOUNDED
DEV = torch.device("cuda:0")

IMPLS = {"simt": fa.FA_BWD_SIMT, "tcgen05": fa.FA_BWD_TCGEN05}


@pytest.fixture(scope="module", autouse=True)
def built():
    fb.build()
    fa.lib()
    torch.cuda.set_device(DEV)


def _impl_or_skip(name, w):
    impl = IMPLS[name]
    try:
        fa.bwd_workspace_size(w.lens, w.lens_kv, w.n_heads, w.n_heads_kv, w.head_dim,
                              w.torch_dtype, w.keep_prob, w.pre_tokens, w.next_tokens, impl)
    except fa.FaError as e:
        if e.status == fa.FA_ERR_UNSUPPORTED and name == "tcgen05":
            pytest.skip("tcgen05 kernel not built for this case")
        raise
    return impl


SMALL = {
    "w1_fp32": wl.workload(1),
    "w2_causal": wl.workload(2),
    "ragged_causal": wl.Workload(10, "bf16", [1, 0, 37, 65, 127, 129, 200], 2, 128, BIG, 0,
                                 seed=3),
    "gqa_band_dropout": wl.Workload(11, "bf16", [300, 0, 150], 4, 128, 100, 20, keep_prob=0.8,
                                    seed=4, n_heads_kv=2),
    "d64_nomask": wl.Workload(12, "bf16", [130, 70], 2, 64, BIG, BIG, seed=5),
    "d32_band": wl.Workload(16, "bf16", [90, 0, 141], 2, 32, 25, 7, seed=9),
    "d64_causal_ragged_fp16": wl.Workload(20, "fp16", [1, 0, 37, 65, 127, 129, 300], 2, 64,
                                          BIG, 0, seed=13),
    "d64_gqa_band_dropout": wl.Workload(21, "bf16", [300, 0, 150], 4, 64, 100, 20,
                                        keep_prob=0.8, seed=14, n_heads_kv=2),
    "d64_w7": wl.workload(7),
    "d64_odd_kv_heads": wl.Workload(22, "bf16", [129, 0, 64, 250], 3, 64, BIG, 0, seed=15),
    "d64_gqa_odd_kv_heads": wl.Workload(23, "bf16", [200, 77], 6, 64, 50, 5, seed=16,
                                        n_heads_kv=3),
    "d96_causal_gqa_fp16": wl.Workload(17, "fp16", [77, 130], 4, 96, BIG, 0, seed=10,
                                       n_heads_kv=2),
    "d192_dropout": wl.Workload(18, "bf16", [66, 129], 2, 192, BIG, BIG, keep_prob=0.85,
                                seed=11),
    "d96_fp32": wl.Workload(19, "fp32", [40, 71], 2, 96, 30, 30, seed=12),
    "fp16_causal": wl.Workload(13, "fp16", [100, 33], 2, 128, BIG, 0, seed=6),
    "lq_ne_lk": wl.Workload(14, "bf16", [50, 90], 2, 128, 30, 10, seed=7, lens_kv=[120, 40]),
    "fp32_dropout_band": wl.Workload(15, "fp32", [70, 45], 2, 128, 20, 3, keep_prob=0.7, seed=8),
    # Key lengths that are multiples of 128: the tensor-core kernel copies
    # the keep bits of each stage into shared memory (ragged query lengths,
    # an empty sequence, grouped heads, Lq != Lk).
    "dropout_rows16_gqa": wl.Workload(24, "bf16", [256, 0, 384, 128], 4, 128, 100, 20,
                                      keep_prob=0.8, seed=17, n_heads_kv=2),
    "dropout_rows16_lq_ne_lk": wl.Workload(25, "bf16", [200, 50, 131], 2, 128, BIG, 40,
                                           keep_prob=0.9, seed=18, lens_kv=[256, 128, 384]),
    "d64_dropout_rows16": wl.Workload(26, "bf16", [256, 77, 128], 3, 64, 90, 0, keep_prob=0.85,
                                      seed=19, lens_kv=[256, 128, 128]),
    # No key reaches query rows 0-129 (nextTokens = -130): query tiles 0 and
    # 1 have no key tile at all, so their dQ rows come only from the
    # accumulator rows the preprocess zeroes.
    "unvisited_query_tiles": wl.Workload(27, "bf16", [300, 200], 2, 128, BIG, -130, seed=20),
}


@pytest.mark.parametrize("impl", ["simt", "tcgen05"])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_end_to_end(name, impl):
    """GPU forward -> GPU backward, against oracle forward -> oracle backward."""
    w = SMALL[name]
    impl_id = _impl_or_skip(impl, w)
    tensors = wl.make_tensors(w)
    mask_np = wl.make_keep_mask(w)
    mask = None if mask_np is None else torch.from_numpy(mask_np).to(DEV)
    out = gpu_forward_backward(w, tensors, DEV, impl_id, mask)
    ref = oracle_full(w, tensors, mask_np)
    assert_close(out, ref, TOL[w.dtype])
    gm, gl = f64(out["smax"]), f64(out["ssum"])
    assert np.all(gm == gm[..., :1]) and np.all(gl == gl[..., :1])     # 8 equal lanes
    np.testing.assert_allclose(gl[..., 0], ref["ssum"][..., 0], rtol=1e-4, atol=0)
    ok = np.isfinite(ref["smax"][..., 0])
    np.testing.assert_allclose(gm[..., 0][ok], ref["smax"][..., 0][ok], rtol=1e-4, atol=1e-5)


@pytest.mark.parametrize("impl", ["simt", "tcgen05"])
@pytest.mark.parametrize("name", ["w2_causal", "gqa_band_dropout", "fp32_dropout_band"])
def test_small_backward_only(name, impl):
    """The backward alone, fed the oracle's Y and statistics (rounded to the
    storage types), against the oracle backward on the same rounded inputs."""
    w = SMALL[name]
    impl_id = _impl_or_skip(impl, w)
    tensors = wl.make_tensors(w)
    mask_np = wl.make_keep_mask(w)
    ref = oracle_full(w, tensors, mask_np)
    y_st = torch.from_numpy(ref["y"]).to(w.torch_dtype)
    m32 = torch.from_numpy(ref["smax"]).float()
    l32 = torch.from_numpy(ref["ssum"]).float()
    q, k, v, dy = (f64(t) for t in tensors)
    rdq, rdk, rdv = oracle.varlen_backward(q, k, v, dy, f64(y_st), f64(m32), f64(l32), w.lens,
                                           w.lens_kv, w.scale, w.pre_tokens, w.next_tokens,
                                           mask_np, w.keep_prob)
    qd, kd, vd, dyd = (t.to(DEV) for t in tensors)
    mask = None if mask_np is None else torch.from_numpy(mask_np).to(DEV)
    dq, dk, dv = fa.bwd(qd, kd, vd, dyd, y_st.to(DEV), m32.to(DEV), l32.to(DEV), w.lens,
                        w.lens_kv, w.scale, w.pre_tokens, w.next_tokens, w.keep_prob, mask,
                        impl=impl_id)
    torch.cuda.synchronize()
    for nm, got, r in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
        assert rel_err(f64(got), r) <= TOL[w.dtype], nm


def test_page_call_example():
    """The FAG-V2 page's call example: all-ones fp32 {256,1,128}, statistics
    3.0, scale 0.088388.  dS is exactly 0, so dQ = dK = 0 exactly and every
    dV element is 256 * exp(0.088388 * 128 - 3) / 3."""
    import json, os  # noqa: E401
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_example.json")))
    t, n, d = g["shape"]
    ones = torch.ones(t, n, d, dtype=torch.float32, device=DEV)
    stats = torch.full((t, n, 8), g["stat_value"], dtype=torch.float32, device=DEV)
    dq, dk, dv = fa.bwd(ones, ones, ones, ones, ones, stats, stats, g["lens"], g["lens"],
                        g["scale"], g["pre_tokens"], g["next_tokens"])
    torch.cuda.synchronize()
    assert float(dq.abs().max()) == 0.0 and float(dk.abs().max()) == 0.0
    assert rel_err(f64(dv), np.full((t, n, d), g["dv_value"])) <= 1e-4


@pytest.mark.parametrize("impl", ["simt", "tcgen05"])
def test_guard_regions_and_full_overwrite(impl):
    """Outputs sit inside NaN-filled buffers: every output element must be
    written (no NaN left) and no guard element touched."""
    w = SMALL["ragged_causal"]
    impl_id = _impl_or_skip(impl, w)
    q, k, v, dy = (t.to(DEV) for t in wl.make_tensors(w))
    y, smax, ssum = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens)
    G = 4096
    outs = []
    for like in (q, k, v):
        buf = torch.full((like.numel() + 2 * G,), float("nan"), dtype=like.dtype, device=DEV)
        outs.append((buf, buf[G:G + like.numel()].view(like.shape)))
    fa.bwd(q, k, v, dy, y, smax, ssum, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens,
           dq=outs[0][1], dk=outs[1][1], dv=outs[2][1], impl=impl_id)
    torch.cuda.synchronize()
    for buf, view in outs:
        assert not torch.isnan(view).any()
        assert torch.isnan(buf[:G]).all() and torch.isnan(buf[-G:]).all()


def test_empty_queries_give_zero_key_gradients():
    w = wl.Workload(16, "bf16", [0, 0], 2, 128, BIG, 0, lens_kv=[40, 9])
    q = torch.empty(0, 2, 128, dtype=torch.bfloat16, device=DEV)
    k = torch.randn(49, 2, 128, device=DEV).bfloat16()
    v = torch.randn(49, 2, 128, device=DEV).bfloat16()
    st = torch.empty(0, 2, 8, device=DEV)
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    fa.bwd(q, k, v, q, q, st, st, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens,
           dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert float(dk.abs().max()) == 0.0 and float(dv.abs().max()) == 0.0


# Rows whose window holds a single key: the softmax gives P = 1 there (Z /
# keep_prob under dropout) and Y = P V_j, so dP = dY V_j^T and D = dY Y^T
# agree and dS = P (dP Z / keep_prob - D) vanishes; dQ and dK are zero in
# exact arithmetic and dV is the only nonzero gradient.  An error relative
# to an all-zero reference means nothing, so dQ and dK are held to the
# tolerance times the size of the terms that cancel.  The first case came
# from a seeded random search: an outer split leaves one row with one key.
SINGLE_KEY = {
    "fp16_d32_gqa_dropout_split": (
        wl.Workload(60, "fp16", [22], 4, 32, 86, 0, keep_prob=0.85, seed=526, mask_seed=24301,
                    n_heads_kv=2), [86], [107]),
    "bf16_d128_diagonal": (wl.Workload(61, "bf16", [200, 77], 2, 128, 0, 0, seed=61), None, None),
    "bf16_d64_diagonal_dropout": (
        wl.Workload(62, "bf16", [130, 64], 4, 64, 0, 0, keep_prob=0.8, seed=62, n_heads_kv=2),
        None, None),
}


@pytest.mark.parametrize("impl", ["simt", "tcgen05"])
@pytest.mark.parametrize("name", list(SINGLE_KEY))
def test_single_key_rows(name, impl):
    w, qs, ks = SINGLE_KEY[name]
    impl_id = _impl_or_skip(impl, w)
    tensors = wl.make_tensors(w)
    mask = device_mask(w, DEV)
    out = gpu_forward_backward(w, tensors, DEV, impl_id, mask, q_start=qs, kv_start=ks)
    mask_np = None if mask is None else mask.cpu().numpy()
    ref = oracle_full(w, tensors, mask_np, q_start=qs, kv_start=ks)
    assert_close(out, ref, TOL[w.dtype], keys=("y", "dv"))
    # |dS| terms: |dP| Z / keep_prob <= |dY| |V| / keep_prob, and |D| <= |dY| |Y|
    # with |Y| <= max |V_j| / keep_prob; one key per row.
    q, k, v, dy = (f64(t) for t in tensors)
    norm = lambda x: float(np.sqrt((x * x).sum(-1)).max())
    ds_terms = 2.0 * norm(dy) * norm(v) / w.keep_prob
    bound = {"dq": w.scale * ds_terms * float(np.abs(k).max()),
             "dk": w.scale * ds_terms * float(np.abs(q).max())}
    for key in ("dq", "dk"):
        assert float(np.abs(ref[key]).max()) <= 1e-9 * bound[key], key   # the premise
        err = float(np.abs(f64(out[key]) - ref[key]).max())
        assert err <= TOL[w.dtype] * bound[key], (key, err, bound[key])


def test_keep_mask_generator_matches_cpu_twin():
    w = wl.workload(5)
    mask = fa.gen_keep_mask(w.mask_bits, w.mask_seed, w.keep_prob, device=DEV)
    torch.cuda.synchronize()
    nbytes = (w.mask_bits + 7) // 8
    assert mask.numel() == nbytes
    rng = np.random.default_rng(1)
    for start in [0, nbytes - 4096] + list(rng.integers(0, nbytes - 4096, 6)):
        start = int(start)
        cpu = wl.keep_mask_bytes(w.mask_seed, w.keep_prob, w.mask_bits, start, 4096)
        assert np.array_equal(mask[start:start + 4096].cpu().numpy(), cpu)
    # odd sizes: tail bits beyond nbits are zero
    m = fa.gen_keep_mask(1001, 99, 0.5, device=DEV)
    torch.cuda.synchronize()
    assert np.array_equal(m.cpu().numpy(), wl.keep_mask_bytes(99, 0.5, 1001))


def _full_size_run(cid):
    w = wl.workload(cid)
    tensors = wl.make_tensors(w)
    mask = device_mask(w, DEV)
    out = gpu_forward_backward(w, tensors, DEV, fa.FA_BWD_AUTO, mask)
    return w, tensors, out


def _invariants(w, tensors, out):
    """Identities of the exact backward, checked on every (sequence, kv head)
    unit of a full-size run, each against the size of its own terms (bound
    tol * sum of |terms|, tol the parity tolerance):
    - sum_j dK_j = 0 for every column d (each dS row sums to 0);
    - sum dQ o Q over the unit's query heads = sum dK o K (both equal
      sum_ij dS_ij S_ij);
    - sum dV o V = sum dY o Y over the unit's query heads (Y = P V).
    A unit with a wrong or missing key tile, or with dQ rows of another
    unit, breaks at least one of them; nothing may be non-finite."""
    for name in ("dq", "dk", "dv", "y"):
        assert torch.isfinite(out[name]).all(), name
    tol = TOL[w.dtype]
    cq, ck = oracle.cu_seqlens(w.lens), oracle.cu_seqlens(w.lens_kv)
    group = w.n_heads // w.n_heads_kv
    dev = out["dk"].device
    q, k, v, dy = (t.to(dev) for t in tensors)
    for b in range(len(w.lens)):
        qs, ks = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
        if cq[b + 1] == cq[b] or ck[b + 1] == ck[b]:
            continue
        for h in range(w.n_heads_kv):
            hs = slice(h * group, (h + 1) * group)
            dk = out["dk"][ks, h].double()
            kk = k[ks, h].double()
            s = dk.sum(dim=0).abs()
            a = dk.abs().sum(dim=0)
            assert bool((s <= tol * a + 1e-30).all()), (b, h, float(s.max()), float(a.max()))
            qq = q[qs, hs].double()
            dq = out["dq"][qs, hs].double()
            lhs, rhs = (dq * qq).sum(), (dk * kk).sum()
            bound = tol * ((dq * qq).abs().sum() + (dk * kk).abs().sum())
            assert abs(float(lhs - rhs)) <= float(bound), (b, h, float(lhs), float(rhs))
            dv, vv = out["dv"][ks, h].double(), v[ks, h].double()
            yy, dyy = out["y"][qs, hs].double(), dy[qs, hs].double()
            lhs, rhs = (dv * vv).sum(), (dyy * yy).sum()
            bound = tol * ((dv * vv).abs().sum() + (dyy * yy).abs().sum())
            assert abs(float(lhs - rhs)) <= float(bound), (b, h, float(lhs), float(rhs))


@pytest.mark.parametrize("cid,units", [
    (3, "longest2+shortest2"),
    (4, [(0, 0), (0, 7), (1, 0), (1, 7)]),
    (5, [(0, 0), (0, 15), (3, 0), (3, 15)]),
])
def test_full_size_sampled_units(cid, units):
    w, tensors, out = _full_size_run(cid)
    _invariants(w, tensors, out)
    if units == "longest2+shortest2":
        lo, hi = int(np.argmin(w.lens)), int(np.argmax(w.lens))
        units = [(hi, 0), (hi, w.n_heads - 1), (lo, 5), (lo, w.n_heads - 1)]
    for b, n in units:
        errs = unit_check(w, tensors, out, b, n)
        tol = TOL[w.dtype]
        assert errs["lse"] <= 1e-3, (b, n, errs)
        for k in ("y", "dq", "dk", "dv"):
            assert errs[k] <= tol, (b, n, errs)


def test_repeat_calls_agree():
    """dQ is summed with atomics (non-deterministic order): two calls agree to
    a few fp32 ulps of the accumulator, dK/dV bit for bit."""
    w = SMALL["w2_causal"]
    q, k, v, dy = (t.to(DEV) for t in wl.make_tensors(w))
    y, m, l = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens)
    a = fa.bwd(q, k, v, dy, y, m, l, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens)
    b = fa.bwd(q, k, v, dy, y, m, l, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert rel_err(f64(a[0]), f64(b[0])) <= 1e-2
