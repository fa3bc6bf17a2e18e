"""The largest problems the page's constraint section allows, on the GPU
against the fp64 oracle.

- T = 2^20 query and key rows (the bound T <= 1M), as 256 sequences of
  4096, with N = 8 and D = 128: every bf16 tensor is 2 GiB and the fp32 dQ
  accumulator 4 GiB, so byte offsets pass 2^31.  Whole (sequence, head)
  units at both ends and in the middle are compared element by element, and
  every sequence's dK rows must sum to zero.
- 2048 sequences (the bound on the number of sequences) of ragged lengths,
  zeros included, compared over the whole batch.
- N = 256 query heads (the bound on N), with one, 16 and 256 key/value
  heads, compared over the whole batch."""

import numpy as np
import pytest
import torch

from varlen_flashattention_backward_gb300 import binding as fa
from varlen_flashattention_backward_gb300 import build as fb
from varlen_flashattention_backward_gb300 import workloads as wl

from _helpers import TOL, assert_close, gpu_forward_backward, oracle_full, unit_check

pytestmark = pytest.mark.gpu
BIG = wl.UNBOUNDED
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    fb.build()
    fa.lib()
    torch.cuda.set_device(DEV)


def test_max_tokens_with_offsets_past_2_31_bytes():
    w = wl.Workload(60, "bf16", [4096] * 256, 8, 128, BIG, 0, seed=61)
    assert w.total_q == 1 << 20
    tensors = wl.make_tensors_on_device(w, DEV)
    out = gpu_forward_backward(w, tensors, DEV)
    for name in ("y", "dq", "dk", "dv"):
        assert torch.isfinite(out[name]).all(), name
    seg = out["dk"].view(256, 4096, 8, 128).double()
    s = seg.sum(dim=1).abs().amax(dim=(1, 2))
    a = seg.abs().sum(dim=1).amax(dim=(1, 2))
    assert bool((s <= 2e-2 * a).all())
    del seg
    for b, n in [(0, 0), (128, 3), (255, 7)]:
        errs = unit_check(w, tensors, out, b, n)
        assert errs["lse"] <= 1e-3, (b, n, errs)
        for k in ("y", "dq", "dk", "dv"):
            assert errs[k] <= TOL[w.dtype], (b, n, errs)


def test_max_sequence_count():
    rng = np.random.default_rng(62)
    lens = [int(x) for x in rng.integers(0, 97, 2048)]
    lens[0], lens[-1] = 0, 96
    w = wl.Workload(61, "bf16", lens, 2, 128, BIG, 0, seed=63)
    tensors = wl.make_tensors(w)
    out = gpu_forward_backward(w, tensors, DEV)
    assert_close(out, oracle_full(w, tensors), TOL[w.dtype])


@pytest.mark.parametrize("n_kv", [1, 16, 256])
@pytest.mark.parametrize("impl", ["simt", "tcgen05"])
def test_max_heads(n_kv, impl):
    w = wl.Workload(62, "bf16", [100, 37], 256, 128, 40, 5, seed=64 + n_kv, n_heads_kv=n_kv)
    tensors = wl.make_tensors(w)
    code = fa.FA_BWD_SIMT if impl == "simt" else fa.FA_BWD_TCGEN05
    out = gpu_forward_backward(w, tensors, DEV, code)
    assert_close(out, oracle_full(w, tensors), TOL[w.dtype])
