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


def gpu_forward_backward(w: wl.Workload, tensors, dev, impl=fa.FA_BWD_AUTO, mask=None):
    q, k, v, dy = (t.to(dev) for t in tensors)
    y, smax, ssum = fa.fwd(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens, w.next_tokens,
                           w.keep_prob, mask)
    dq, dk, dv = fa.bwd(q, k, v, dy, y, smax, ssum, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                        w.next_tokens, w.keep_prob, mask, impl=impl)
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


def oracle_full(w: wl.Workload, tensors, mask_np=None):
    """Oracle forward + backward over the whole packed batch."""
    q, k, v, dy = (f64(t) for t in tensors)
    y, m, l = oracle.varlen_forward(q, k, v, w.lens, w.lens_kv, w.scale, w.pre_tokens,
                                    w.next_tokens, mask_np, w.keep_prob)
    dq, dk, dv = oracle.varlen_backward(q, k, v, dy, y, m, l, w.lens, w.lens_kv, w.scale,
                                        w.pre_tokens, w.next_tokens, mask_np, w.keep_prob)
    return dict(y=y, smax=m, ssum=l, dq=dq, dk=dk, dv=dv)


def assert_close(got: dict, ref: dict, tol: float, keys=("y", "dq", "dk", "dv")):
    errs = {k: rel_err(f64(got[k]), ref[k]) for k in keys}
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, f"rel errors {errs} exceed {tol}"
    return errs


def sampled_unit_check(w: wl.Workload, tensors, out: dict, b: int, n: int, n_rows=48,
                       n_cols=48, seed=0):
    """Oracle on one (sequence, head) unit: the whole forward, dQ at sampled
    query rows and dK/dV at sampled key rows.  Returns the relative errors."""
    rng = np.random.default_rng(seed + 97 * b + n)
    cq, ck = oracle.cu_seqlens(w.lens), oracle.cu_seqlens(w.lens_kv)
    lq, lk = w.lens[b], w.lens_kv[b]
    group = w.n_heads // w.n_heads_kv
    q, k, v, dy = tensors
    qs = q[cq[b]:cq[b + 1], n].double().numpy()
    ks = k[ck[b]:ck[b + 1], n // group].double().numpy()
    vs = v[ck[b]:ck[b + 1], n // group].double().numpy()
    dys = dy[cq[b]:cq[b + 1], n].double().numpy()
    keep_rows, keep_cols = cpu_keep_rows(w, b, n)
    y, m, l = oracle.unit_forward(qs, ks, vs, w.scale, w.pre_tokens, w.next_tokens,
                                  keep_rows, w.keep_prob)
    edge = [0, 1, 63, 64, 127, 128, lq - 1]
    rows = np.unique(np.concatenate([[r for r in edge if 0 <= r < lq],
                                     rng.integers(0, lq, n_rows)]))
    edge = [0, 1, 127, 128, lk - 1]
    cols = np.unique(np.concatenate([[c for c in edge if 0 <= c < lk],
                                     rng.integers(0, lk, n_cols)]))
    dq = oracle.unit_backward_rows(rows, qs, ks, vs, dys, y, m, l, w.scale, w.pre_tokens,
                                   w.next_tokens, keep_rows, w.keep_prob)
    dk, dv = oracle.unit_backward_cols(cols, qs, ks, vs, dys, y, m, l, w.scale, w.pre_tokens,
                                       w.next_tokens, keep_cols, w.keep_prob)
    g = lambda name, sl, h: f64(out[name][sl, h])  # noqa: E731
    gy = g("y", slice(cq[b], cq[b + 1]), n)
    gdq = g("dq", slice(cq[b], cq[b + 1]), n)[rows]
    # dK/dV of a shared key/value head sum over its query heads; compare only
    # when the group has one head.
    errs = {"y": rel_err(gy, y), "dq": rel_err(gdq, dq)}
    if group == 1:
        errs["dk"] = rel_err(g("dk", slice(ck[b], ck[b + 1]), n)[cols], dk)
        errs["dv"] = rel_err(g("dv", slice(ck[b], ck[b + 1]), n)[cols], dv)
    gm = f64(out["smax"][cq[b]:cq[b + 1], n, 0])
    gl = f64(out["ssum"][cq[b]:cq[b + 1], n, 0])
    errs["lse"] = float(np.abs((gm + np.log(gl)) - (m + np.log(l))).max())
    return errs
