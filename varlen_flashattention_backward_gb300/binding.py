"""Thin ctypes binding over libfavarlen.so (argument marshalling only).

Every function here forwards to the C entry point of the same name in
``include/fa_varlen.h``; all arithmetic runs in the library's CUDA kernels.
torch provides device memory and the current stream.  If the library has
not been built, the first call raises: there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

FA_OK, FA_ERR_NULLPTR, FA_ERR_INVALID, FA_ERR_UNSUPPORTED = 0, 1, 2, 3
FA_ERR_WORKSPACE, FA_ERR_CUDA, FA_ERR_TIMEOUT = 4, 5, 6
FA_BWD_AUTO, FA_BWD_SIMT, FA_BWD_TCGEN05 = 0, 1, 2

_DTYPE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

_LIB = None

_i64, _f64, _sz, _vp = ctypes.c_int64, ctypes.c_double, ctypes.c_size_t, ctypes.c_void_p
_i32, _cp = ctypes.c_int32, ctypes.c_char_p
_pi64 = ctypes.POINTER(ctypes.c_int64)
_psz = ctypes.POINTER(ctypes.c_size_t)


class BwdOptions(ctypes.Structure):
    _fields_ = [("impl", ctypes.c_int32), ("deterministic", ctypes.c_int32),
                ("wait_timeout_ns", ctypes.c_int64), ("events", ctypes.POINTER(ctypes.c_void_p)),
                ("q_start_idx", ctypes.POINTER(ctypes.c_int64)),
                ("kv_start_idx", ctypes.POINTER(ctypes.c_int64)),
                ("atten_mask", ctypes.c_void_p), ("atten_mask_rows", ctypes.c_int64),
                ("atten_mask_cols", ctypes.c_int64)]


class FwdOptions(ctypes.Structure):
    _fields_ = [("q_start_idx", ctypes.POINTER(ctypes.c_int64)),
                ("kv_start_idx", ctypes.POINTER(ctypes.c_int64)),
                ("atten_mask", ctypes.c_void_p), ("atten_mask_rows", ctypes.c_int64),
                ("atten_mask_cols", ctypes.c_int64)]


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


_SCALARS = [_pi64, _pi64, _i64, _i64, _i64, _i64, _i64, _i64, _i32, _cp]

_SIGS = {
    "fa_varlen_version": ([], _i32),
    "fa_status_string": ([_i32], _cp),
    "fa_varlen_fwd_workspace_size": (_SCALARS + [_f64, _i64, _i64, _i64, _psz], _i32),
    "fa_varlen_bwd_workspace_size": (_SCALARS + [_f64, _i64, _i64, _i64, _psz], _i32),
    "fa_varlen_bwd_workspace_size_ex": (
        _SCALARS + [_f64, _i64, _i64, _i64, ctypes.POINTER(BwdOptions), _psz], _i32),
    "fa_varlen_fwd": ([_vp, _vp, _vp, _vp, _i64] + _SCALARS[:8] + [_i32, _cp, _f64, _f64, _i64,
                      _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "fa_varlen_fwd_ex": ([_vp, _vp, _vp, _vp, _i64] + _SCALARS[:8] + [_i32, _cp, _f64, _f64,
                         _i64, _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp,
                         ctypes.POINTER(FwdOptions)], _i32),
    "fa_varlen_bwd": ([_vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp] + _SCALARS[:8] +
                      [_i32, _cp, _f64, _f64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp],
                      _i32),
    "fa_varlen_bwd_ex": ([_vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp] + _SCALARS[:8] +
                         [_i32, _cp, _f64, _f64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp,
                          ctypes.POINTER(BwdOptions)], _i32),
    "fa_varlen_read_error": ([_vp, _sz, _vp, ctypes.POINTER(ctypes.c_int32)], _i32),
    "fa_gen_keep_mask": ([_vp, _i64, ctypes.c_uint64, _f64, _vp], _i32),
    "fa_varlen_bwd_static_scratch": ([_vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp] +
                                     _SCALARS[:8] + [_i32, _cp, _f64, _f64, _i64, _i64, _i64,
                                                     _vp, _vp, _vp, _vp], _i32),
    "fa_varlen_bwd_static_scratch_read_error": ([_vp, ctypes.POINTER(ctypes.c_int32)], _i32),
    "fa_varlen_selftest_wait_timeout": ([_vp, _sz, _i64, _vp], _i32),
    "fa_varlen_bwd_schedule": ([_pi64, _pi64, _i64, _i64, _i64, _i64, _i32,
                                ctypes.POINTER(ctypes.c_int32), _i64, _pi64], _i32),
    "fa_varlen_bwd_schedule_ex": ([_pi64, _pi64, _i64, _i64, _i64, _i64, _i32, _i64, _i64, _i32,
                                   _i64, _i64, _i32, ctypes.POINTER(ctypes.c_int32), _i64, _pi64],
                                  _i32),
}

EXPORTS = tuple(_SIGS)


def library_path() -> str:
    return _build.library_path()


def lib():
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libfavarlen.so is not built ({path}); run "
                               "varlen_flashattention_backward_gb300.build.build() first")
        handle = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = handle
    return _LIB


def status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def version() -> int:
    return int(lib().fa_varlen_version())


def _check(status: int, where: str):
    if status != FA_OK:
        raise FaError(status, where)


def _lens(lens):
    lens = [int(x) for x in lens]
    return (ctypes.c_int64 * max(1, len(lens)))(*lens), len(lens), sum(lens)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _starts(starts):
    """Host int64 array of per-sequence chunk starts, or None."""
    if starts is None:
        return None
    vals = [int(x) for x in starts]
    return (ctypes.c_int64 * max(1, len(vals)))(*vals)


def _mask_fields(atten_mask):
    """(pointer, rows, cols) of a 2-D uint8 device mask, or (None, 0, 0)."""
    if atten_mask is None:
        return None, 0, 0
    rows, cols = atten_mask.shape
    return ctypes.c_void_p(atten_mask.data_ptr()), int(rows), int(cols)


def _opts(impl=FA_BWD_AUTO, wait_timeout_ns=0, events=None, deterministic=False,
          q_start=None, kv_start=None, atten_mask=None):
    ev = None
    if events is not None:
        arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
        ev = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
        ev._keep = arr
    qs, ks = _starts(q_start), _starts(kv_start)
    am, am_rows, am_cols = _mask_fields(atten_mask)
    opt = BwdOptions(int(impl), int(bool(deterministic)), int(wait_timeout_ns), ev,
                     ctypes.cast(qs, ctypes.POINTER(ctypes.c_int64)) if qs is not None else None,
                     ctypes.cast(ks, ctypes.POINTER(ctypes.c_int64)) if ks is not None else None,
                     am, am_rows, am_cols)
    opt._keep = (qs, ks)
    return opt


def fwd_workspace_size(lens_q, lens_kv, n, n_kv, d, dtype, keep_prob=1.0,
                       pre_tokens=2 ** 31 - 1, next_tokens=2 ** 31 - 1, sparse_mode=0) -> int:
    lq, b, tq = _lens(lens_q)
    lk, _, tk = _lens(lens_kv)
    out = ctypes.c_size_t(0)
    _check(lib().fa_varlen_fwd_workspace_size(lq, lk, b, tq, tk, n, n_kv, d, _DTYPE[dtype], b"TND",
                                              keep_prob, pre_tokens, next_tokens,
                                              int(sparse_mode), ctypes.byref(out)),
           "fa_varlen_fwd_workspace_size")
    return out.value


def bwd_workspace_size(lens_q, lens_kv, n, n_kv, d, dtype, keep_prob=1.0,
                       pre_tokens=2 ** 31 - 1, next_tokens=2 ** 31 - 1,
                       impl=FA_BWD_AUTO, sparse_mode=0, atten_mask=None) -> int:
    lq, b, tq = _lens(lens_q)
    lk, _, tk = _lens(lens_kv)
    out = ctypes.c_size_t(0)
    opt = _opts(impl, atten_mask=atten_mask)
    _check(lib().fa_varlen_bwd_workspace_size_ex(lq, lk, b, tq, tk, n, n_kv, d, _DTYPE[dtype],
                                                 b"TND", keep_prob, pre_tokens, next_tokens,
                                                 int(sparse_mode), ctypes.byref(opt),
                                                 ctypes.byref(out)),
           "fa_varlen_bwd_workspace_size_ex")
    return out.value


def fwd(q, k, v, lens_q, lens_kv, scale, pre_tokens, next_tokens, keep_prob=1.0,
        drop_mask=None, y=None, softmax_max=None, softmax_sum=None, workspace=None,
        stream=None, q_start=None, kv_start=None, sparse_mode=0, atten_mask=None):
    """Y and the [T, N, 8] statistics (fa_varlen_fwd_ex).  ``q_start`` /
    ``kv_start``: per-sequence global chunk starts (outer split), or None.
    ``sparse_mode``: 0 or 4 (preTokens / nextTokens band), 1 (``atten_mask``
    alone), 2 (lower triangle from the top-left corner), 3 (lower triangle
    from the bottom-right).  ``atten_mask``: 2-D uint8 device tensor, 1 =
    excluded, at each sequence's chunk-local (i, j); read in modes 0, 1, 4."""
    tq, n, d = q.shape
    n_kv = k.shape[1]
    lq, b, _ = _lens(lens_q)
    lk, _, _ = _lens(lens_kv)
    dev = q.device
    if y is None:
        y = torch.empty_like(q)
    if softmax_max is None:
        softmax_max = torch.empty(tq, n, 8, dtype=torch.float32, device=dev)
    if softmax_sum is None:
        softmax_sum = torch.empty(tq, n, 8, dtype=torch.float32, device=dev)
    if workspace is None:
        ws = fwd_workspace_size(lens_q, lens_kv, n, n_kv, d, q.dtype, keep_prob, pre_tokens,
                                next_tokens, sparse_mode)
        workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
    mask_bytes = 0 if drop_mask is None else drop_mask.numel()
    qs, ks = _starts(q_start), _starts(kv_start)
    am, am_rows, am_cols = _mask_fields(atten_mask)
    opt = FwdOptions(ctypes.cast(qs, ctypes.POINTER(ctypes.c_int64)) if qs is not None else None,
                     ctypes.cast(ks, ctypes.POINTER(ctypes.c_int64)) if ks is not None else None,
                     am, am_rows, am_cols)
    _check(lib().fa_varlen_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(drop_mask), mask_bytes, lq, lk,
                                  b, tq, k.shape[0], n, n_kv, d, _DTYPE[q.dtype], b"TND",
                                  float(scale), float(keep_prob), int(pre_tokens),
                                  int(next_tokens), int(sparse_mode), _ptr(y), _ptr(softmax_max),
                                  _ptr(softmax_sum), _ptr(workspace), workspace.numel(),
                                  _stream(stream), ctypes.byref(opt)), "fa_varlen_fwd_ex")
    return y, softmax_max, softmax_sum


def bwd(q, k, v, dy, y, softmax_max, softmax_sum, lens_q, lens_kv, scale, pre_tokens,
        next_tokens, keep_prob=1.0, drop_mask=None, dq=None, dk=None, dv=None,
        workspace=None, stream=None, impl=FA_BWD_AUTO, wait_timeout_ns=0, events=None,
        deterministic=False, q_start=None, kv_start=None, sparse_mode=0, atten_mask=None):
    """dQ, dK, dV (fa_varlen_bwd_ex).  ``events``: four torch.cuda.Event
    (already recorded once, so that they exist) recorded around the kernels.
    ``deterministic``: add the dQ partials in a fixed order (bitwise
    reproducible dQ).  ``q_start`` / ``kv_start`` / ``sparse_mode``: as in
    ``fwd`` (give the forward the same values)."""
    tq, n, d = q.shape
    n_kv = k.shape[1]
    lq, b, _ = _lens(lens_q)
    lk, _, _ = _lens(lens_kv)
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    if workspace is None:
        ws = bwd_workspace_size(lens_q, lens_kv, n, n_kv, d, q.dtype, keep_prob, pre_tokens,
                                next_tokens, impl, sparse_mode, atten_mask)
        workspace = torch.empty(ws, dtype=torch.uint8, device=q.device)
    mask_bytes = 0 if drop_mask is None else drop_mask.numel()
    opt = _opts(impl, wait_timeout_ns, events, deterministic, q_start, kv_start, atten_mask)
    _check(lib().fa_varlen_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(drop_mask),
                                  mask_bytes, _ptr(softmax_max), _ptr(softmax_sum), _ptr(y), lq,
                                  lk, b, tq, k.shape[0], n, n_kv, d, _DTYPE[q.dtype], b"TND",
                                  float(scale), float(keep_prob), int(pre_tokens),
                                  int(next_tokens), int(sparse_mode), _ptr(dq), _ptr(dk),
                                  _ptr(dv),
                                  _ptr(workspace), workspace.numel(), _stream(stream),
                                  ctypes.byref(opt)), "fa_varlen_bwd_ex")
    return dq, dk, dv


def bwd_static_scratch(q, k, v, dy, y, softmax_max, softmax_sum, lens_q, lens_kv, scale,
                       pre_tokens, next_tokens, keep_prob=1.0, drop_mask=None, dq=None, dk=None,
                       dv=None, stream=None):
    """dQ, dK, dV through fa_varlen_bwd_static_scratch: no workspace is
    allocated; the library's 64 MiB device array serves as scratch."""
    tq, n, d = q.shape
    n_kv = k.shape[1]
    lq, b, _ = _lens(lens_q)
    lk, _, _ = _lens(lens_kv)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    mask_bytes = 0 if drop_mask is None else drop_mask.numel()
    _check(lib().fa_varlen_bwd_static_scratch(
        _ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(drop_mask), mask_bytes, _ptr(softmax_max),
        _ptr(softmax_sum), _ptr(y), lq, lk, b, tq, k.shape[0], n, n_kv, d, _DTYPE[q.dtype],
        b"TND", float(scale), float(keep_prob), int(pre_tokens), int(next_tokens), 0, _ptr(dq),
        _ptr(dk), _ptr(dv), _stream(stream)), "fa_varlen_bwd_static_scratch")
    return dq, dk, dv


def static_scratch_read_error(stream=None) -> int:
    """Raw error word of the last fa_varlen_bwd_static_scratch call in the
    current context (fa_varlen_bwd_static_scratch_read_error; synchronises
    `stream`)."""
    code = ctypes.c_int32(0)
    st = lib().fa_varlen_bwd_static_scratch_read_error(_stream(stream), ctypes.byref(code))
    if st not in (FA_OK, FA_ERR_TIMEOUT):
        _check(st, "fa_varlen_bwd_static_scratch_read_error")
    return int(code.value)


def selftest_wait_timeout(workspace, wait_timeout_ns, stream=None):
    """fa_varlen_selftest_wait_timeout: a kernel whose bounded wait on a
    barrier nothing completes must expire and record a timeout code."""
    _check(lib().fa_varlen_selftest_wait_timeout(_ptr(workspace), workspace.numel(),
                                                 int(wait_timeout_ns), _stream(stream)),
           "fa_varlen_selftest_wait_timeout")


def read_error(workspace, stream=None) -> int:
    """Raw error word of the last call on `workspace` (synchronises)."""
    code = ctypes.c_int32(0)
    st = lib().fa_varlen_read_error(_ptr(workspace), workspace.numel(), _stream(stream),
                                    ctypes.byref(code))
    if st not in (FA_OK, FA_ERR_TIMEOUT):
        _check(st, "fa_varlen_read_error")
    return int(code.value)


def bwd_schedule(lens_q, lens_kv, n_kv, pre_tokens, next_tokens, kv_tile):
    """The backward work list as a list of (seq, kv_head, kv_tile, q_lo, q_count)."""
    lq, b, _ = _lens(lens_q)
    lk, _, _ = _lens(lens_kv)
    n = ctypes.c_int64(0)
    _check(lib().fa_varlen_bwd_schedule(lq, lk, b, n_kv, pre_tokens, next_tokens, kv_tile, None,
                                        0, ctypes.byref(n)), "fa_varlen_bwd_schedule")
    buf = (ctypes.c_int32 * max(4, 4 * n.value))()
    _check(lib().fa_varlen_bwd_schedule(lq, lk, b, n_kv, pre_tokens, next_tokens, kv_tile, buf,
                                        n.value, ctypes.byref(n)), "fa_varlen_bwd_schedule")
    out = []
    for i in range(n.value):
        s, h, t, r = buf[4 * i:4 * i + 4]
        out.append((s, h, t, r & 0xFFFF, (r >> 16) & 0xFFFF))
    return out


def bwd_schedule_ex(lens_q, lens_kv, n, n_kv, d, dtype, pre_tokens, next_tokens, kv_tile,
                    l2_bytes=0, tail_items=0, head_pairs=False):
    """fa_varlen_bwd_schedule_ex: the work list in launch order, as a list of
    (seq, first kv head, kv heads, kv_tile, q_lo, q_count)."""
    lq, b, _ = _lens(lens_q)
    lk, _, _ = _lens(lens_kv)
    cnt = ctypes.c_int64(0)
    args = (lq, lk, b, n, n_kv, d, _DTYPE[dtype], pre_tokens, next_tokens, kv_tile,
            int(l2_bytes), int(tail_items), int(bool(head_pairs)))
    _check(lib().fa_varlen_bwd_schedule_ex(*args, None, 0, ctypes.byref(cnt)),
           "fa_varlen_bwd_schedule_ex")
    buf = (ctypes.c_int32 * max(4, 4 * cnt.value))()
    _check(lib().fa_varlen_bwd_schedule_ex(*args, buf, cnt.value, ctypes.byref(cnt)),
           "fa_varlen_bwd_schedule_ex")
    out = []
    for i in range(cnt.value):
        s_, h, t, r = buf[4 * i:4 * i + 4]
        out.append((s_, h & 0xFFFF, 1 + (h >> 16), t, r & 0xFFFF, (r >> 16) & 0xFFFF))
    return out


def gen_keep_mask(nbits: int, seed: int, keep_prob: float, device="cuda", out=None,
                  stream=None):
    """SplitMix64 keep mask of `nbits` bits on the device (fa_gen_keep_mask)."""
    nbytes = (int(nbits) + 7) // 8
    if out is None:
        out = torch.empty(max(1, nbytes), dtype=torch.uint8, device=device)
    _check(lib().fa_gen_keep_mask(_ptr(out), int(nbits), int(seed) & (2 ** 64 - 1),
                                  float(keep_prob), _stream(stream)), "fa_gen_keep_mask")
    return out
