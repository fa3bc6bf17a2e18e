"""The no-allocation backward, fa_varlen_bwd_static_scratch.

Code running inside a custom allocator or a memory-pool callback, or under a
runtime that owns all device memory, cannot always call cudaMalloc for a
workspace.  fa_varlen_bwd_static_scratch serves such callers from a 64 MiB
device array that the library reserves when it is loaded.  These tests call
it through the C ABI and check that:
- it gives the same dQ, dK, dV as fa_varlen_bwd, within the bf16 parity
  tolerance, on two calls in a row (the array keeps the previous call's
  contents, so the second call checks that nothing stale leaks through);
- it refuses a problem whose scratch would not fit.

The file name makes pytest collect it last, and it needs nothing from the
other test files, so it passes both alone in a fresh process and after the
rest of the suite."""

import pytest
import torch

from varlen_flashattention_backward_gb300 import binding as fa
from varlen_flashattention_backward_gb300 import build as fb
from varlen_flashattention_backward_gb300 import workloads as wl

from _helpers import TOL, f64, rel_err

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    fb.build()
    fa.lib()
    torch.cuda.set_device(DEV)


def test_static_scratch_matches_workspace_entry_point_twice():
    # The benchmark workload: bf16, lengths [512, 1024, 2048, 512], N = 16,
    # D = 128, causal.  Its scratch (about 34 MB) fits in the 64 MiB array.
    w = wl.workload(2)
    q, k, v, dy = (t.to(DEV) for t in wl.make_tensors(w))
    y, smax, ssum = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens)
    ref = fa.bwd(q, k, v, dy, y, smax, ssum, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                 w.next_tokens)
    torch.cuda.synchronize()
    outs = [(torch.full_like(q, float("nan")), torch.full_like(k, float("nan")),
             torch.full_like(v, float("nan"))) for _ in range(2)]
    before = torch.cuda.memory_allocated(DEV)
    for dq, dk, dv in outs:
        fa.bwd_static_scratch(q, k, v, dy, y, smax, ssum, w.lens, w.lens_kv, w.scale,
                              w.pre_tokens, w.next_tokens, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated(DEV) == before
    for call, got in enumerate(outs):
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert not torch.isnan(g).any(), (call, name)
            assert rel_err(f64(g), f64(r)) <= TOL[w.dtype], (call, name)


def test_static_scratch_rejects_problems_that_do_not_fit():
    # Workload 4 (2 x 32768 tokens, N = 8, D = 128) needs a 268 MB fp32 dQ
    # accumulator alone: refused before any launch.
    w = wl.workload(4)
    assert fa.bwd_workspace_size(w.lens, w.lens_kv, w.n_heads, w.n_heads_kv, w.head_dim,
                                 torch.bfloat16) > (64 << 20)
    t = torch.empty(8, dtype=torch.bfloat16, device=DEV)
    st = torch.empty(8, dtype=torch.float32, device=DEV)
    shp_q = (w.total_q, w.n_heads, w.head_dim)
    fake_q = t.as_strided(shp_q, (0, 0, 0))
    with pytest.raises(fa.FaError) as e:
        fa.bwd_static_scratch(fake_q, fake_q, fake_q, fake_q, fake_q, st, st, w.lens, w.lens_kv,
                              w.scale, w.pre_tokens, w.next_tokens, dq=fake_q, dk=fake_q,
                              dv=fake_q)
    assert e.value.status == fa.FA_ERR_WORKSPACE
