"""The no-allocation backward, fa_varlen_bwd_static_scratch.

Code running inside a custom allocator or a memory-pool callback, or under a
runtime that owns all device memory, cannot always call cudaMalloc for a
workspace.  fa_varlen_bwd_static_scratch serves such callers from a 64 MiB
device array that the library's module holds in each CUDA context.  These
tests call it through the C ABI and check that:
- it gives the same dQ, dK, dV as fa_varlen_bwd, within the parity
  tolerance of the element type, on two calls in a row (the array keeps the
  previous call's contents, so the second call checks that nothing stale
  leaks through), on the tensor-core kernel (head dim 128, and head dim 64
  with two kv heads per work item) and on the CUDA-core kernel (fp32);
- the device's free memory, as the driver reports it, does not move across
  those calls (torch's allocator statistics would miss a cudaMalloc);
- its error word reads back as 0 through
  fa_varlen_bwd_static_scratch_read_error;
- in a second CUDA context on the same device (made through the driver
  API, as some runtimes do) it finds that context's own copy of the array;
- it refuses a problem whose scratch would not fit.

The file name makes pytest collect it last, and it needs nothing from the
other test files, so it passes both alone in a fresh process and after the
rest of the suite."""

import os
import subprocess
import sys

import pytest
import torch

from varlen_flashattention_backward_gb300 import binding as fa
from varlen_flashattention_backward_gb300 import build as fb
from varlen_flashattention_backward_gb300 import workloads as wl

from _helpers import TOL, f64, rel_err

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    fb.build()
    fa.lib()
    torch.cuda.set_device(DEV)


def _static(q, k, v, dy, y, smax, ssum, w, outs):
    fa.bwd_static_scratch(q, k, v, dy, y, smax, ssum, w.lens, w.lens_kv, w.scale,
                          w.pre_tokens, w.next_tokens, dq=outs[0], dk=outs[1], dv=outs[2])


# 2: bf16, lengths [512, 1024, 2048, 512], N = 16, D = 128, causal (about
#    34 MB of scratch), tensor-core kernel;
# 7: the same lengths with N = 32, D = 64 (two kv heads per work item);
# 1: fp32, lengths [37, 64], N = 2, D = 64, no mask: CUDA-core kernel.
@pytest.mark.parametrize("cid", [2, 7, 1])
def test_static_scratch_matches_workspace_entry_point_twice(cid):
    w = wl.workload(cid)
    q, k, v, dy = (t.to(DEV) for t in wl.make_tensors(w))
    y, smax, ssum = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens)
    ref = fa.bwd(q, k, v, dy, y, smax, ssum, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                 w.next_tokens)
    outs = [(torch.full_like(q, float("nan")), torch.full_like(k, float("nan")),
             torch.full_like(v, float("nan"))) for _ in range(3)]
    # One warm call first: the first use of a kernel in a context loads it.
    _static(q, k, v, dy, y, smax, ssum, w, outs[2])
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info(DEV)
    torch_before = torch.cuda.memory_allocated(DEV)
    for o in outs[:2]:
        _static(q, k, v, dy, y, smax, ssum, w, o)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info(DEV)
    assert free_after == free_before
    assert torch.cuda.memory_allocated(DEV) == torch_before
    assert fa.static_scratch_read_error() == 0
    for call, got in enumerate(outs[:2]):
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


# Runs in a fresh process: the primary context (through torch), then a
# second context made with the driver API, then the primary one again.
_SECOND_CONTEXT = r"""
import ctypes, sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
sys.path.insert(0, ROOT + "/tests")
from varlen_flashattention_backward_gb300 import binding as fa
from varlen_flashattention_backward_gb300 import build as fb
from varlen_flashattention_backward_gb300 import workloads as wl
from _helpers import TOL, rel_err

fb.build()
lib = fa.lib()
dev = torch.device("cuda:0")
torch.cuda.set_device(dev)
w = wl.workload(2)
q, k, v, dy = (t.to(dev) for t in wl.make_tensors(w))
y, smax, ssum = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens)
ref = [t.double().cpu().numpy() for t in
       fa.bwd(q, k, v, dy, y, smax, ssum, w.lens, w.lens_kv, w.scale, w.pre_tokens,
              w.next_tokens)]

def check(outs, where):
    for name, g, r in zip(("dq", "dk", "dv"), outs, ref):
        assert not np.isnan(g).any(), (where, name)
        e = rel_err(g, r)
        assert e <= TOL["bf16"], (where, name, e)

def primary(where):
    o = fa.bwd_static_scratch(q, k, v, dy, y, smax, ssum, w.lens, w.lens_kv, w.scale,
                              w.pre_tokens, w.next_tokens)
    torch.cuda.synchronize()
    check([t.double().cpu().numpy() for t in o], where)

primary("primary context, first call")
torch.cuda.synchronize()

ins = [t.contiguous().cpu() for t in (q, k, v, dy, y, smax, ssum)]
host = [t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy() for t in ins]
cu = ctypes.CDLL("libcuda.so.1")
def ok(r, what):
    assert r == 0, (what, r)
ok(cu.cuInit(0), "cuInit")
cdev = ctypes.c_int(0)
ok(cu.cuDeviceGet(ctypes.byref(cdev), 0), "cuDeviceGet")
ctx = ctypes.c_void_p()
if hasattr(cu, "cuCtxCreate_v2"):
    ok(cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, cdev), "cuCtxCreate_v2")
else:
    ok(cu.cuCtxCreate_v4(ctypes.byref(ctx), None, 0, cdev), "cuCtxCreate_v4")
bufs = []
def alloc(nbytes):
    p = ctypes.c_uint64(0)
    ok(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc")
    bufs.append(p)
    return p.value
d_in = []
for h in host:
    p = alloc(h.nbytes)
    ok(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(p), h.ctypes.data_as(ctypes.c_void_p),
                          ctypes.c_size_t(h.nbytes)), "cuMemcpyHtoD")
    d_in.append(p)
d_out = [alloc(host[i].nbytes) for i in (0, 1, 2)]
lq, b, _ = fa._lens(w.lens)
lk, _, _ = fa._lens(w.lens_kv)
vp = ctypes.c_void_p
for call in range(2):
    st = lib.fa_varlen_bwd_static_scratch(
        vp(d_in[0]), vp(d_in[1]), vp(d_in[2]), vp(d_in[3]), None, 0, vp(d_in[5]),
        vp(d_in[6]), vp(d_in[4]), lq, lk, b, sum(w.lens), sum(w.lens_kv), w.n_heads, w.n_heads_kv,
        w.head_dim, 2, b"TND", float(w.scale), 1.0, int(w.pre_tokens), int(w.next_tokens), 0,
        vp(d_out[0]), vp(d_out[1]), vp(d_out[2]), None)
    assert st == 0, ("second context", fa.status_string(st))
    ok(cu.cuCtxSynchronize(), "cuCtxSynchronize")
    code = ctypes.c_int32(-1)
    assert lib.fa_varlen_bwd_static_scratch_read_error(None, ctypes.byref(code)) == 0
    assert code.value == 0
    outs = []
    for i, p in enumerate(d_out):
        h = np.empty_like(host[i])
        ok(cu.cuMemcpyDtoH_v2(h.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(p),
                              ctypes.c_size_t(h.nbytes)), "cuMemcpyDtoH")
        outs.append(torch.from_numpy(h).view(torch.bfloat16).double().numpy())
    check(outs, "second context, call %d" % call)
for p in bufs:
    ok(cu.cuMemFree_v2(p), "cuMemFree")
ok(cu.cuCtxDestroy_v2(ctx), "cuCtxDestroy")
primary("primary context, after the second context")
print("second context ok")
"""


def test_static_scratch_in_a_second_context():
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + _SECOND_CONTEXT],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "second context ok" in r.stdout, r.stdout + r.stderr
