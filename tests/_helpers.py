"""Shared pieces of the GPU parity tests: run the CUDA path through the
binding, run the fp64 oracle on the same seeded inputs, compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from varlen_flashattention_backward_gb300 import binding as fa
from varlen_flashattention_backward_gb300 import workloads as wl

# max|err| <= TOL * max|ref| per output tensor
TOL = {"fp32": 1e-4, "bf16": 2e-2, "fp16": 2e-2}


def f64(t) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def rel_err(got, ref) -> float:
    ref = np.asarray(ref)
    den = np.abs(ref).max() if ref.size else 0.0
    if den == 0.0:
        return float(np.abs(np.asarray(got)).max()) if np.asarray(got).size else 0.0
    return float(np.abs(np.asarray(got) - ref).max() / den)


def device_mask(w: wl.Workload, dev):
    """Keep mask on the device.  Small masks are drawn on the CPU and copied;
    large ones come from the library's SplitMix64 twin."""
    if w.keep_prob >= 1.0:
        return None
    if w.mask_bits <= (1 << 27):
        return torch.from_numpy(wl.make_keep_mask(w)).to(dev)
    return fa.gen_keep_mask(w.mask_bits, w.mask_seed, w.keep_prob, device=dev)


def nan_workspace(w: wl.Workload, dev, impl=fa.FA_BWD_AUTO):
    """A backward workspace whose every byte is 0xFF (every fp32 word a NaN),
    so that any scratch the backward reads before writing poisons its
    outputs."""
    nbytes = fa.bwd_workspace_size(w.lens, w.lens_kv, w.n_heads, w.n_heads_kv, w.head_dim,
                                   w.torch_dtype, w.keep_prob, w.pre_tokens, w.next_tokens,
                                   impl)
    return torch.full((nbytes,), 255, dtype=torch.uint8, device=dev)


def gpu_forward_backward(w: wl.Workload, tensors, dev, impl=fa.FA_BWD_AUTO, mask=None,
                         q_start=None, kv_start=None):
    q, k, v, dy = (t.to(dev) for t in tensors)
    y, smax, ssum = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens,
                           w.keep_prob, mask, q_start=q_start, kv_start=kv_start)
    dq, dk, dv = fa.bwd(q, k, v, dy, y, smax, ssum, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                        w.next_tokens, w.keep_prob, mask, impl=impl, q_start=q_start,
                        kv_start=kv_start, workspace=nan_workspace(w, dev, impl))
    torch.cuda.synchronize()
    return dict(y=y, smax=smax, ssum=ssum, dq=dq, dk=dk, dv=dv)


def cpu_keep_rows(w: wl.Workload, b: int, n: int):
    """Oracle-side keep bits of unit (b, n), drawn from the CPU generator."""
    if w.keep_prob >= 1.0:
        return None, None
    off = int(oracle.mask_bit_offsets(w.lens, w.lens_kv, w.n_heads)[b])
    lq, lk = w.lens[b], w.lens_kv[b]
    base = off + n * lq * lk

    def rows(r):
        r = np.asarray(r, dtype=np.int64)[:, None]
        return wl.keep_bits(w.mask_seed, w.keep_prob,
                            base + r * lk + np.arange(lk)[None, :]).astype(np.float64)

    def cols(c):
        c = np.asarray(c, dtype=np.int64)[None, :]
        return wl.keep_bits(w.mask_seed, w.keep_prob,
                            base + np.arange(lq)[:, None] * lk + c).astype(np.float64)

    return rows, cols


def oracle_full(w: wl.Workload, tensors, mask_np=None, q_start=None, kv_start=None):
    """Oracle forward + backward over the whole packed batch."""
    q, k, v, dy = (f64(t) for t in tensors)
    y, m, l = oracle.varlen_forward(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                                    w.next_tokens, mask_np, w.keep_prob, q_start=q_start,
                                    kv_start=kv_start)
    dq, dk, dv = oracle.varlen_backward(q, k, v, dy, y, m, l, w.lens, w.lens_kv, w.scale,
                                        w.pre_tokens, w.next_tokens, mask_np, w.keep_prob,
                                        q_start=q_start, kv_start=kv_start)
    return dict(y=y, smax=m, ssum=l, dq=dq, dk=dk, dv=dv)


def assert_close(got: dict, ref: dict, tol: float, keys=("y", "dq", "dk", "dv")):
    errs = {k: rel_err(f64(got[k]), ref[k]) for k in keys}
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, f"rel errors {errs} exceed {tol}"
    return errs


def unit_check(w: wl.Workload, tensors, out: dict, b: int, n: int):
    """Oracle forward + backward of one whole (sequence, head) unit of a
    full-size run, compared element by element with the GPU outputs of that
    unit (max|ref| taken over the unit).  The inputs may live on the host or
    the device; only the unit's slices are copied.  Returns the relative
    errors."""
    cq, ck = oracle.cu_seqlens(w.lens), oracle.cu_seqlens(w.lens_kv)
    group = w.n_heads // w.n_heads_kv
    q, k, v, dy = tensors
    qs = f64(q[cq[b]:cq[b + 1], n])
    ks = f64(k[ck[b]:ck[b + 1], n // group])
    vs = f64(v[ck[b]:ck[b + 1], n // group])
    dys = f64(dy[cq[b]:cq[b + 1], n])
    keep_rows, _ = cpu_keep_rows(w, b, n)
    y, m, l = oracle.unit_forward(qs, ks, vs, w.scale, w.pre_tokens, w.next_tokens,
                                  keep_rows, w.keep_prob)
    dq, dk, dv = oracle.unit_backward(qs, ks, vs, dys, y, m, l, w.scale, w.pre_tokens,
                                      w.next_tokens, keep_rows, w.keep_prob)
    g = lambda name, sl, h: f64(out[name][sl, h])  # noqa: E731
    qsl, ksl = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
    errs = {"y": rel_err(g("y", qsl, n), y), "dq": rel_err(g("dq", qsl, n), dq)}
    # dK/dV of a shared key/value head sum over its query heads; compare only
    # when the group has one head.
    if group == 1:
        errs["dk"] = rel_err(g("dk", ksl, n), dk)
        errs["dv"] = rel_err(g("dv", ksl, n), dv)
    gm = f64(out["smax"][qsl, n, 0])
    gl = f64(out["ssum"][qsl, n, 0])
    ok = l > 0
    errs["lse"] = float(np.abs((gm + np.log(gl))[ok] - (m + np.log(l))[ok]).max())
    return errs
