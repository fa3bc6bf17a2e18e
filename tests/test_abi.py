"""CPU tests of the C ABI: the library loads and exports what include/*.h
declares, the argument checks return the documented status codes without
touching a GPU, and the host tile scheduler covers exactly the allowed
(query, key) pairs."""

import ctypes
import glob
import os
import re

import numpy as np
import pytest
import torch

from varlen_flashattention_backward_gb300 import binding as fa
from varlen_flashattention_backward_gb300 import build as fb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BIG = 2 ** 31 - 1


@pytest.fixture(scope="module", autouse=True)
def built():
    fb.build()
    fa.lib()


def header_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b([a-z_][a-z0-9_]*)\s*\(", text):
            if m.group(1).startswith("fa_"):
                names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol():
    declared = header_functions()
    assert {"fa_varlen_bwd", "fa_varlen_fwd", "fa_varlen_bwd_workspace_size",
            "fa_status_string"} <= declared
    handle = ctypes.CDLL(fb.library_path())
    for name in sorted(declared):
        assert hasattr(handle, name), name
    # the binding wraps every declared entry point under the same name
    assert declared == set(fa.EXPORTS)


def test_status_strings_and_version():
    for s in range(7):
        assert fa.status_string(s).startswith("FA_")
    assert fa.version() >= 100


def _ws(lens_q=(37, 64), lens_kv=None, n=2, nkv=2, d=64, dt=torch.float32, keep=1.0,
        pre=BIG, nxt=BIG, layout=b"TND", sparse=0, batch=None, tq=None, tk=None):
    lens_kv = lens_q if lens_kv is None else lens_kv
    lq = (ctypes.c_int64 * len(lens_q))(*lens_q)
    lk = (ctypes.c_int64 * len(lens_kv))(*lens_kv)
    out = ctypes.c_size_t(0)
    b = len(lens_q) if batch is None else batch
    tq = sum(lens_q) if tq is None else tq
    tk = sum(lens_kv) if tk is None else tk
    return fa.lib().fa_varlen_bwd_workspace_size(lq, lk, b, tq, tk, n, nkv, d, fa._DTYPE[dt],
                                                 layout, keep, pre, nxt, sparse,
                                                 ctypes.byref(out)), out.value


def test_workspace_size_checks():
    st, size = _ws()
    assert st == fa.FA_OK and size > 0
    assert _ws(layout=b"BSND")[0] == fa.FA_ERR_INVALID
    assert _ws(n=0)[0] == fa.FA_ERR_INVALID
    assert _ws(n=257, nkv=1)[0] == fa.FA_ERR_INVALID
    assert _ws(n=4, nkv=3)[0] == fa.FA_ERR_INVALID
    assert _ws(d=0)[0] == fa.FA_ERR_INVALID
    assert _ws(d=769)[0] == fa.FA_ERR_INVALID
    assert _ws(keep=0.0)[0] == fa.FA_ERR_INVALID
    assert _ws(keep=1.5)[0] == fa.FA_ERR_INVALID
    assert _ws(batch=0)[0] == fa.FA_ERR_INVALID
    assert _ws(lens_q=tuple([1] * 2049))[0] == fa.FA_ERR_INVALID
    assert _ws(lens_q=(5, -1))[0] == fa.FA_ERR_INVALID
    assert _ws(tq=100)[0] == fa.FA_ERR_INVALID
    assert _ws(lens_q=(1 << 20, 1))[0] == fa.FA_ERR_INVALID
    for d in (16, 80, 256, 768):
        assert _ws(d=d)[0] == fa.FA_ERR_UNSUPPORTED
    for d in (32, 64, 96, 128, 192):
        assert _ws(d=d)[0] == fa.FA_OK
    assert _ws(sparse=1)[0] == fa.FA_OK
    for mode in (6, 7, 8):
        assert _ws(sparse=mode)[0] == fa.FA_ERR_UNSUPPORTED
    for mode in (-1, 5, 9):
        assert _ws(sparse=mode)[0] == fa.FA_ERR_INVALID
    for mode in (0, 2, 3, 4):
        assert _ws(sparse=mode)[0] == fa.FA_OK
    assert _ws(lens_q=(0, 5, 0))[0] == fa.FA_OK


def test_nullptr_checks():
    lq = (ctypes.c_int64 * 1)(8)
    out = ctypes.c_size_t(0)
    L = fa.lib()
    assert L.fa_varlen_bwd_workspace_size(None, lq, 1, 8, 8, 1, 1, 64, 0, b"TND", 1.0, BIG, BIG, 0,
                                          ctypes.byref(out)) == fa.FA_ERR_NULLPTR
    assert L.fa_varlen_bwd_workspace_size(lq, lq, 1, 8, 8, 1, 1, 64, 0, None, 1.0, BIG, BIG, 0,
                                          ctypes.byref(out)) == fa.FA_ERR_NULLPTR
    assert L.fa_varlen_bwd_workspace_size(lq, lq, 1, 8, 8, 1, 1, 64, 0, b"TND", 1.0, BIG, BIG, 0,
                                          None) == fa.FA_ERR_NULLPTR


def _bwd_call(**over):
    """fa_varlen_bwd with fake (never dereferenced) device pointers; every case
    below fails a host check before any CUDA call."""
    fake = ctypes.c_void_p(0x1000)
    args = dict(q=fake, k=fake, v=fake, dy=fake, mask=None, mask_bytes=0, smax=fake, ssum=fake,
                y=fake, lens=(8,), n=1, nkv=1, d=64, dt=2, layout=b"TND", scale=0.125, keep=1.0,
                pre=BIG, nxt=BIG, sparse=0, dq=fake, dk=fake, dv=fake, ws=fake, ws_bytes=0)
    args.update(over)
    lens = (ctypes.c_int64 * len(args["lens"]))(*args["lens"])
    t = sum(args["lens"])
    return fa.lib().fa_varlen_bwd(args["q"], args["k"], args["v"], args["dy"], args["mask"],
                                  args["mask_bytes"], args["smax"], args["ssum"], args["y"], lens,
                                  lens, len(args["lens"]), t, t, args["n"], args["nkv"], args["d"],
                                  args["dt"], args["layout"], args["scale"], args["keep"],
                                  args["pre"], args["nxt"], args["sparse"], args["dq"], args["dk"],
                                  args["dv"], args["ws"], args["ws_bytes"], None)


def test_bwd_argument_checks_before_any_launch():
    for name in ("q", "k", "v", "dy", "smax", "ssum", "y", "dq", "dk", "dv"):
        assert _bwd_call(**{name: None}) == fa.FA_ERR_NULLPTR, name
    assert _bwd_call(keep=0.5) == fa.FA_ERR_NULLPTR            # dropout needs a mask
    assert _bwd_call(keep=0.5, mask=ctypes.c_void_p(0x1000), mask_bytes=7) == fa.FA_ERR_INVALID
    assert _bwd_call(layout=b"BNSD") == fa.FA_ERR_INVALID
    assert _bwd_call(dt=7) == fa.FA_ERR_INVALID
    assert _bwd_call(scale=float("nan")) == fa.FA_ERR_INVALID
    assert _bwd_call(n=3, nkv=2) == fa.FA_ERR_INVALID
    assert _bwd_call(d=80) == fa.FA_ERR_UNSUPPORTED
    assert _bwd_call(sparse=6) == fa.FA_ERR_UNSUPPORTED
    assert _bwd_call(sparse=1) == fa.FA_ERR_NULLPTR           # mode 1 reads the attention mask
    assert _bwd_call(sparse=5) == fa.FA_ERR_INVALID
    assert _bwd_call(ws_bytes=16) == fa.FA_ERR_WORKSPACE
    assert _bwd_call(ws=None, ws_bytes=1 << 20) == fa.FA_ERR_NULLPTR
    assert _bwd_call(lens=(0,)) == fa.FA_OK                    # empty input: nothing to do


def test_gen_mask_and_read_error_checks():
    L = fa.lib()
    assert L.fa_gen_keep_mask(None, 8, 1, 0.9, None) == fa.FA_ERR_NULLPTR
    assert L.fa_gen_keep_mask(ctypes.c_void_p(0x1000), -1, 1, 0.9, None) == fa.FA_ERR_INVALID
    assert L.fa_gen_keep_mask(ctypes.c_void_p(0x1000), 8, 1, 0.0, None) == fa.FA_ERR_INVALID
    assert L.fa_gen_keep_mask(ctypes.c_void_p(0x1000), 0, 1, 0.9, None) == fa.FA_OK
    code = ctypes.c_int32(0)
    assert L.fa_varlen_read_error(None, 256, None, ctypes.byref(code)) == fa.FA_ERR_NULLPTR


# ---------------------------------------------------------------------------
# scheduler
# ---------------------------------------------------------------------------

def _allowed_pairs(lq, lk, pre, nxt):
    i = np.arange(lq)[:, None]
    j = np.arange(lk)[None, :]
    return (j >= i - pre) & (j <= i + nxt)


SCHED_CASES = [
    ([512, 1024, 2048, 512], 1, BIG, 0),
    ([37, 64, 0, 1, 129], 2, BIG, BIG),
    ([300, 200], 1, 70, 0),
    ([250], 1, 5, 40),
    ([0, 0, 7], 3, BIG, 0),
]


@pytest.mark.parametrize("kv_tile", [64, 128])
@pytest.mark.parametrize("case", SCHED_CASES)
def test_schedule_covers_exactly_the_allowed_pairs(case, kv_tile):
    lens, nkv, pre, nxt = case
    items = fa.bwd_schedule(lens, lens, nkv, pre, nxt, kv_tile)
    n_tiles = sum((L + kv_tile - 1) // kv_tile for L in lens) * nkv
    assert len(items) == n_tiles
    # the items of one (sequence, head) unit are contiguous and longest first;
    # units are ordered by their longest item, longest first
    units = []
    for b, h, t, lo, cnt in items:
        if not units or units[-1][0] != (b, h):
            units.append(((b, h), []))
        units[-1][1].append(cnt)
    assert len({u for u, _ in units}) == len(units)
    for _, counts in units:
        assert counts == sorted(counts, reverse=True)
    heads = [counts[0] for _, counts in units]
    assert heads == sorted(heads, reverse=True)
    seen = set()
    for b, h, t, lo, cnt in items:
        assert (b, h, t) not in seen
        seen.add((b, h, t))
        L = lens[b]
        allowed = _allowed_pairs(L, L, pre, nxt)
        k0, k1 = t * kv_tile, min(L, (t + 1) * kv_tile)
        cols = allowed[:, k0:k1]
        rows_needed = np.nonzero(cols.any(axis=1))[0]
        covered = np.zeros(L, bool)
        covered[lo * 64:(lo + cnt) * 64] = True
        # every query with an allowed key in this tile is visited ...
        assert covered[rows_needed].all()
        # ... and no visited query tile is entirely masked for this key tile
        for qt in range(lo, lo + cnt):
            assert cols[qt * 64:(qt + 1) * 64].any(), (b, t, qt)


def test_selftest_argument_checks():
    L = fa.lib()
    fake = ctypes.c_void_p(0x1000)
    assert L.fa_varlen_selftest_wait_timeout(None, 256, 10**6, None) == fa.FA_ERR_NULLPTR
    assert L.fa_varlen_selftest_wait_timeout(fake, 64, 10**6, None) == fa.FA_ERR_WORKSPACE
    assert L.fa_varlen_selftest_wait_timeout(fake, 256, 10, None) == fa.FA_ERR_INVALID
    assert L.fa_varlen_selftest_wait_timeout(fake, 256, 10**11, None) == fa.FA_ERR_INVALID


@pytest.mark.parametrize("kv_tile", [64, 128])
@pytest.mark.parametrize("case", SCHED_CASES + [([50, 300], 2, 30, 10), ([700, 1], 1, 0, 0)])
def test_key_tiles_of_a_query_tile_are_contiguous(case, kv_tile):
    """The deterministic mode adds the dQ partials of a query tile in key-tile
    order, ranked from the first key tile that visits it; that needs the key
    tiles visiting any one query tile to form a contiguous range."""
    lens, nkv, pre, nxt = case
    items = fa.bwd_schedule(lens, lens, nkv, pre, nxt, kv_tile)
    cover = {}
    for b, h, t, lo, cnt in items:
        if h != 0:
            continue
        for qt in range(lo, lo + cnt):
            cover.setdefault((b, qt), []).append(t)
    for key, tiles in cover.items():
        tiles.sort()
        assert tiles == list(range(tiles[0], tiles[-1] + 1)), (key, tiles)


def test_deterministic_option_accepted():
    lq = (ctypes.c_int64 * 2)(37, 64)
    out = ctypes.c_size_t(0)
    opt = fa.BwdOptions(fa.FA_BWD_AUTO, 1, 0, None)
    assert fa.lib().fa_varlen_bwd_workspace_size_ex(lq, lq, 2, 101, 101, 2, 2, 64,
                                                    fa._DTYPE[torch.float32], b"TND", 1.0, BIG,
                                                    BIG, 0, ctypes.byref(opt),
                                                    ctypes.byref(out)) == fa.FA_OK
    assert out.value > 0


def test_negative_chunk_start_is_invalid():
    lq = (ctypes.c_int64 * 1)(8)
    out = ctypes.c_size_t(0)
    neg = (ctypes.c_int64 * 1)(-1)
    opt = fa.BwdOptions(fa.FA_BWD_AUTO, 0, 0, None,
                        ctypes.cast(neg, ctypes.POINTER(ctypes.c_int64)), None)
    assert fa.lib().fa_varlen_bwd_workspace_size_ex(lq, lq, 1, 8, 8, 1, 1, 64,
                                                    fa._DTYPE[torch.float32], b"TND", 1.0, BIG,
                                                    BIG, 0, ctypes.byref(opt),
                                                    ctypes.byref(out)) == fa.FA_ERR_INVALID
    fake = ctypes.c_void_p(0x1000)
    fo = fa.FwdOptions(ctypes.cast(neg, ctypes.POINTER(ctypes.c_int64)), None)
    st = fa.lib().fa_varlen_fwd_ex(fake, fake, fake, None, 0, lq, lq, 1, 8, 8, 1, 1, 64,
                                   fa._DTYPE[torch.float32], b"TND", 0.125, 1.0, BIG, BIG, 0,
                                   fake, fake, fake, fake, 1 << 20, None, ctypes.byref(fo))
    assert st == fa.FA_ERR_INVALID


# ---------------------------------------------------------------------------
# launch-order rules of the scheduler (fa_varlen_bwd_schedule_ex)
# ---------------------------------------------------------------------------

ORDER_CASES = [
    ([512, 1024, 2048, 512], 16, 16, 128, BIG, 0),
    ([37, 64, 0, 1, 129, 700], 4, 2, 128, 100, 20),
    ([300, 200, 1000], 6, 3, 64, BIG, 0),
]


def _item_key(it):
    s_, h, nh, t, lo, cnt = it
    return (s_, h, nh, t, lo, cnt)


def _length(it):
    return it[5] * it[2]


@pytest.mark.parametrize("case", ORDER_CASES)
def test_whole_list_longest_first_when_it_fits_in_l2(case):
    lens, n, nkv, d, pre, nxt = case
    unit = fa.bwd_schedule_ex(lens, lens, n, nkv, d, torch.bfloat16, pre, nxt, 128)
    fit = fa.bwd_schedule_ex(lens, lens, n, nkv, d, torch.bfloat16, pre, nxt, 128,
                             l2_bytes=1 << 40)
    small = fa.bwd_schedule_ex(lens, lens, n, nkv, d, torch.bfloat16, pre, nxt, 128,
                               l2_bytes=1 << 10)
    assert sorted(map(_item_key, fit)) == sorted(map(_item_key, unit))
    lengths = [_length(it) for it in fit]
    assert lengths == sorted(lengths, reverse=True)
    # stable: equal lengths keep their unit order
    pos = {_item_key(it): i for i, it in enumerate(unit)}
    for a, b in zip(fit, fit[1:]):
        if _length(a) == _length(b):
            assert pos[_item_key(a)] < pos[_item_key(b)]
    # a working set larger than L2 keeps unit order
    assert small == unit


@pytest.mark.parametrize("tail", [1, 5, 40, 10**6])
def test_tail_of_the_unit_order_is_sorted(tail):
    lens, n, nkv, d, pre, nxt = ORDER_CASES[1]
    unit = fa.bwd_schedule_ex(lens, lens, n, nkv, d, torch.bfloat16, pre, nxt, 128)
    got = fa.bwd_schedule_ex(lens, lens, n, nkv, d, torch.bfloat16, pre, nxt, 128,
                             tail_items=tail)
    k = len(unit) if tail >= len(unit) else tail
    if tail >= len(unit):
        assert got == unit     # no tail sort when the tail would be the whole list
        return
    assert got[:-k] == unit[:-k]
    assert sorted(map(_item_key, got[-k:])) == sorted(map(_item_key, unit[-k:]))
    lengths = [_length(it) for it in got[-k:]]
    assert lengths == sorted(lengths, reverse=True)


@pytest.mark.parametrize("nkv", [1, 2, 3, 8])
def test_head_pairs_cover_every_kv_head_once(nkv):
    lens = [300, 0, 129, 64]
    single = fa.bwd_schedule_ex(lens, lens, 2 * nkv, nkv, 64, torch.bfloat16, BIG, 0, 128)
    pairs = fa.bwd_schedule_ex(lens, lens, 2 * nkv, nkv, 64, torch.bfloat16, BIG, 0, 128,
                               head_pairs=True)
    assert len(pairs) == sum((L + 127) // 128 for L in lens) * ((nkv + 1) // 2)
    covered = []
    for s_, h, nh, t, lo, cnt in pairs:
        assert h % 2 == 0 and nh == min(2, nkv - h)
        for hh in range(h, h + nh):
            covered.append((s_, hh, t, lo, cnt))
    assert sorted(covered) == sorted((s_, h, t, lo, cnt) for s_, h, nh, t, lo, cnt in single)


def test_schedule_ex_argument_checks():
    L = fa.lib()
    lq = (ctypes.c_int64 * 2)(37, 64)
    n = ctypes.c_int64(0)
    ok = (lq, lq, 2, 4, 2, 128, 2, BIG, BIG, 128, 0, 0, 0, None, 0, ctypes.byref(n))
    assert L.fa_varlen_bwd_schedule_ex(*ok) == fa.FA_OK
    for i, v in ((3, 3), (5, 1000), (6, 7), (10, -1), (11, -1), (9, 32)):
        bad = list(ok)
        bad[i] = v
        assert L.fa_varlen_bwd_schedule_ex(*bad) == fa.FA_ERR_INVALID, (i, v)
