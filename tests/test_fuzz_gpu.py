"""Seeded random problems through both backward kernels against the fp64
oracle: element types, head dims 64 and 128, grouped heads, ragged and
empty sequences, Lq != Lk, windows of every sparse mode, explicit masks,
dropout, outer-split starts and the deterministic mode, in combination.
Each case draws its own configuration from its seed, so a failure names a
reproducible case."""

import numpy as np
import pytest
import torch

import oracle
from varlen_flashattention_backward_gb300 import binding as fa
from varlen_flashattention_backward_gb300 import build as fb
from varlen_flashattention_backward_gb300 import workloads as wl

from _helpers import TOL, assert_close, f64

pytestmark = pytest.mark.gpu
BIG = wl.UNBOUNDED
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    fb.build()
    fa.lib()
    torch.cuda.set_device(DEV)


def _case(seed, dims=(64, 128), dtypes=("bf16", "fp16")):
    g = np.random.default_rng(1000 + seed)
    b = int(g.integers(1, 5))
    lens = [int(x) for x in g.integers(0, 300, b)]
    lens[int(g.integers(0, b))] = int(g.integers(1, 300))     # never all empty
    lens_kv = lens if g.random() < 0.5 else [int(x) for x in g.integers(1, 300, b)]
    n_kv = int(g.choice([1, 2, 3]))
    n = n_kv * int(g.choice([1, 2]))
    d = int(g.choice(list(dims)))
    dtype = str(g.choice(list(dtypes)))
    mode = int(g.choice([0, 0, 1, 2, 3, 4]))
    pre = int(g.choice([BIG, int(g.integers(0, 200))]))
    nxt = int(g.choice([BIG, 0, int(g.integers(0, 50))]))
    keep = float(g.choice([1.0, 1.0, 0.85]))
    starts = g.random() < 0.3
    qs = [int(x) for x in g.integers(0, 200, b)] if starts else None
    ks = [int(x) for x in g.integers(0, 200, b)] if starts else None
    am = None
    if mode == 1 or (mode in (0, 4) and g.random() < 0.3):
        am = (g.random((max(lens) + 2, max(lens_kv) + 3)) < 0.3).astype(np.uint8)
    det = bool(g.random() < 0.3)
    w = wl.Workload(200 + seed, dtype, lens, n, d, pre, nxt, keep_prob=keep, seed=300 + seed,
                    n_heads_kv=n_kv, lens_kv=lens_kv)
    return w, mode, am, qs, ks, det


def _run_case(w, mode, am_np, qs, ks, det, impl):
    tensors = wl.make_tensors(w)
    mask_np = wl.make_keep_mask(w)
    mask = None if mask_np is None else torch.from_numpy(mask_np).to(DEV)
    am = None if am_np is None else torch.from_numpy(am_np).to(DEV)
    q, k, v, dy = (t.to(DEV) for t in tensors)
    y, m, l = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens,
                     w.keep_prob, mask, q_start=qs, kv_start=ks, sparse_mode=mode, atten_mask=am)
    ws = torch.empty(fa.bwd_workspace_size(w.lens, w.lens_kv, w.n_heads, w.n_heads_kv,
                                           w.head_dim, q.dtype, w.keep_prob, w.pre_tokens,
                                           w.next_tokens, impl, mode, am),
                     dtype=torch.uint8, device=DEV)
    dq, dk, dv = fa.bwd(q, k, v, dy, y, m, l, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                        w.next_tokens, w.keep_prob, mask, workspace=ws, impl=impl,
                        deterministic=det, q_start=qs, kv_start=ks, sparse_mode=mode,
                        atten_mask=am)
    torch.cuda.synchronize()
    assert fa.read_error(ws) == 0
    qn, kn, vn, dyn = (f64(t) for t in tensors)
    ry, rm, rl = oracle.varlen_forward(qn, kn, vn, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                                       w.next_tokens, mask_np, w.keep_prob, q_start=qs,
                                       kv_start=ks, sparse_mode=mode, atten_mask=am_np)
    rdq, rdk, rdv = oracle.varlen_backward(qn, kn, vn, dyn, ry, rm, rl, w.lens, w.lens_kv,
                                           w.scale, w.pre_tokens, w.next_tokens, mask_np,
                                           w.keep_prob, q_start=qs, kv_start=ks,
                                           sparse_mode=mode, atten_mask=am_np)
    assert_close(dict(y=y, dq=dq, dk=dk, dv=dv), dict(y=ry, dq=rdq, dk=rdk, dv=rdv),
                 TOL[w.dtype])


@pytest.mark.parametrize("seed", range(24))
def test_random_problem_tcgen05(seed):
    _run_case(*_case(seed), fa.FA_BWD_TCGEN05)


@pytest.mark.parametrize("seed", range(12))
def test_random_problem_cuda_cores(seed):
    """The CUDA-core kernel: every element type and every head dim it has."""
    _run_case(*_case(100 + seed, dims=(32, 64, 96, 128, 192), dtypes=("fp32", "bf16", "fp16")),
              fa.FA_BWD_SIMT)
