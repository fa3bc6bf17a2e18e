"""Failure detection without a GPU fault: a kernel's bounded wait on a
barrier that nothing completes must give up, record a timeout code that the
host reads as FA_ERR_TIMEOUT, and leave the context usable."""

import time

import pytest
import torch

from varlen_flashattention_backward_gb300 import binding as fa
from varlen_flashattention_backward_gb300 import build as fb
from varlen_flashattention_backward_gb300 import workloads as wl

from _helpers import TOL, f64, oracle_full, rel_err

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    fb.build()
    fa.lib()
    torch.cuda.set_device(DEV)


@pytest.mark.gpu
def test_expired_wait_reports_timeout_and_context_survives():
    ws = torch.full((256,), 0xFF, dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    fa.selftest_wait_timeout(ws, 20_000_000)          # 20 ms
    code = fa.read_error(ws)                          # synchronises
    elapsed = time.perf_counter() - t0
    assert code == 0x100 + 7
    assert elapsed >= 0.015
    st = fa.lib().fa_varlen_read_error(fa._ptr(ws), ws.numel(), fa._stream(None),
                                       fa.ctypes.byref(fa.ctypes.c_int32()))
    assert st == fa.FA_ERR_TIMEOUT
    # the context is still usable: a normal backward gives correct results
    w = wl.Workload(30, "bf16", [150, 77], 2, 128, wl.UNBOUNDED, 0, seed=9)
    t = wl.make_tensors(w)
    q, k, v, dy = (x.to(DEV) for x in t)
    y, m, l = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens)
    out = fa.bwd(q, k, v, dy, y, m, l, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens)
    torch.cuda.synchronize()
    ref = oracle_full(w, t)
    for name, g in zip(("dq", "dk", "dv"), out):
        assert rel_err(f64(g), ref[name]) <= TOL["bf16"], name
