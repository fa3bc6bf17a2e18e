"""Pins for the fp64 oracle against things other than itself.

Each test fixes the oracle to mathematics or to the FAG-V2 page (the web page
"CANN/ops-transformer FlashAttention梯度V2" documenting
aclnnFlashAttentionUnpaddingScoreGradV2): hand-enumerated fixtures, central
finite differences, closed forms, invariants, torch fp64 autograd of the
explicit forward graph, and the page's own call example.  Chosen so that a
dropped term, a wrong sign or index, or a transposed operand anywhere in the
oracle fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from varlen_flashattention_backward_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
BIG = 65536


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_problem(rng, lens_q, lens_kv, n, nkv, d, dv=None):
    dv = dv or d
    tq, tk = sum(lens_q), sum(lens_kv)
    q = rng.standard_normal((tq, n, d))
    k = rng.standard_normal((tk, nkv, d))
    v = rng.standard_normal((tk, nkv, dv))
    dy = rng.standard_normal((tq, n, dv))
    return q, k, v, dy


def _mask_for(rng, lens_q, lens_kv, n, p_keep=0.7):
    nbits = sum(n * a * b for a, b in zip(lens_q, lens_kv))
    bits = (rng.random(nbits) < p_keep).astype(np.uint8)
    bits = np.concatenate([bits, np.zeros((-nbits) % 8, np.uint8)])
    return np.packbits(bits.reshape(-1, 8), axis=1, bitorder="little").reshape(-1)


# ---------------------------------------------------------------------------
# hand fixtures: window, mask bits, offsets, statistics
# ---------------------------------------------------------------------------

def test_window_fixture():
    for c in _load("window_cases.json")["cases"]:
        got = oracle.window_allowed(c["lq"], c["lk"], c["pre"], c["next"])
        assert got.astype(int).tolist() == c["allowed"], c


def test_mask_bits_fixture():
    g = _load("mask_bits.json")
    for c in g["cases"]:
        got = oracle.keep_bits_unit(np.array(c["bytes"], np.uint8), c["bit_offset"],
                                    c["lq"], c["lk"])
        assert got.astype(int).tolist() == c["keep"], c
    o = g["offsets"]
    assert oracle.mask_bit_offsets(o["lens_q"], o["lens_kv"], o["n_heads"]).tolist() == o["expected"]


def test_stats_closed_form():
    # q = [1], k = [[0], [1]], scale 1: S = [0, 1], max = 1, sum = 1 + e^-1.
    q = np.array([[[1.0]]]); k = np.array([[[0.0]], [[1.0]]]); v = np.array([[[2.0]], [[5.0]]])
    y, m, l = oracle.varlen_forward(q, k, v, [1], [2], 1.0, BIG, BIG)
    assert m[0, 0, 0] == 1.0 and np.all(m[0, 0] == 1.0)
    assert l[0, 0, 0] == pytest.approx(1.0 + math.exp(-1.0), rel=1e-15)
    p = np.array([math.exp(-1.0), 1.0]) / (1.0 + math.exp(-1.0))
    assert y[0, 0, 0] == pytest.approx(2.0 * p[0] + 5.0 * p[1], rel=1e-15)
    # causal: the only allowed key of query 0 is key 0.
    y, m, l = oracle.varlen_forward(q, k, v, [1], [2], 1.0, BIG, 0)
    assert (m[0, 0, 0], l[0, 0, 0], y[0, 0, 0]) == (0.0, 1.0, 2.0)


def test_empty_row_stats_and_grads():
    rng = np.random.default_rng(3)
    q, k, v, dy = _rand_problem(rng, [3], [3], 1, 1, 2)
    # pre=1, next=-1: row 0 has no allowed key.
    y, m, l = oracle.varlen_forward(q, k, v, [3], [3], 0.5, 1, -1)
    assert m[0, 0, 0] == -np.inf and l[0, 0, 0] == 0.0 and np.all(y[0] == 0.0)
    dq, dk, dv = oracle.varlen_backward(q, k, v, dy, y, m, l, [3], [3], 0.5, 1, -1)
    assert np.all(dq[0] == 0.0)
    # key 2 is allowed for no query -> zero gradients.
    assert np.all(dk[2] == 0.0) and np.all(dv[2] == 0.0)


# ---------------------------------------------------------------------------
# finite differences of L = sum(Y * dY)
# ---------------------------------------------------------------------------

def _loss(q, k, v, dy, lens_q, lens_kv, scale, pre, nxt, mask, kp):
    y, _, _ = oracle.varlen_forward(q, k, v, lens_q, lens_kv, scale, pre, nxt, mask, kp)
    return float((y * dy).sum())


FD_CASES = [
    # lens_q, lens_kv, n, nkv, d, pre, next, dropout
    ([3, 5], [3, 5], 2, 2, 4, BIG, BIG, False),
    ([3, 5], [3, 5], 2, 2, 4, BIG, 0, False),
    ([4, 2], [4, 2], 2, 1, 3, 1, 0, False),
    ([3, 4], [3, 4], 1, 1, 4, BIG, 0, True),
    ([2, 5], [4, 3], 2, 2, 2, 2, 1, True),
    ([3], [3], 1, 1, 2, 1, -1, False),
]


@pytest.mark.parametrize("case", FD_CASES)
def test_finite_differences(case):
    lens_q, lens_kv, n, nkv, d, pre, nxt, drop = case
    rng = np.random.default_rng(11)
    q, k, v, dy = _rand_problem(rng, lens_q, lens_kv, n, nkv, d)
    scale = 0.7
    mask = _mask_for(rng, lens_q, lens_kv, n) if drop else None
    kp = 0.8 if drop else 1.0
    y, m, l = oracle.varlen_forward(q, k, v, lens_q, lens_kv, scale, pre, nxt, mask, kp)
    dq, dk, dv = oracle.varlen_backward(q, k, v, dy, y, m, l, lens_q, lens_kv, scale,
                                        pre, nxt, mask, kp)
    h = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, dy, lens_q, lens_kv, scale, pre, nxt, mask, kp)
            x[idx] = old - h
            lm = _loss(q, k, v, dy, lens_q, lens_kv, scale, pre, nxt, mask, kp)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - g).max() / max(1e-12, np.abs(num).max())
        assert err <= 1e-6, (name, err)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("drop", [False, True])
def test_ds_rows_sum_to_zero(drop):
    rng = np.random.default_rng(5)
    lq = lk = 37
    q, k, v, dy = (rng.standard_normal((lq, 8)) for _ in range(4))
    kb = None
    kp = 1.0
    if drop:
        z = (rng.random((lq, lk)) < 0.6).astype(np.float64)
        kb = lambda rows: z[rows]  # noqa: E731
        kp = 0.6
    y, m, l = oracle.unit_forward(q, k, v, 0.3, 9, 0, kb, kp)
    dq, dk, dv, ds = oracle.unit_backward(q, k, v, dy, y, m, l, 0.3, 9, 0, kb, kp,
                                          return_ds=True)
    assert np.abs(ds.sum(axis=1)).max() <= 1e-12 * np.abs(ds).max() * lk
    # sum_j dK_j = scale * sum_i (sum_j dS_ij) Q_i = 0
    assert np.abs(dk.sum(axis=0)).max() <= 1e-12 * np.abs(dk).max() * lk
    if not drop:
        # every row has an allowed key and P rows sum to 1: sum_j dV_j = sum_i dY_i
        np.testing.assert_allclose(dv.sum(axis=0), dy.sum(axis=0), rtol=1e-12, atol=1e-12)


def test_packed_equals_each_alone():
    rng = np.random.default_rng(8)
    lens = [5, 1, 0, 7]
    q, k, v, dy = _rand_problem(rng, lens, lens, 2, 2, 3)
    mask = _mask_for(rng, lens, lens, 2)
    args = (0.5, 3, 1, mask, 0.75)
    y, m, l = oracle.varlen_forward(q, k, v, lens, lens, *args)
    dq, dk, dv = oracle.varlen_backward(q, k, v, dy, y, m, l, lens, lens, *args)
    cu = oracle.cu_seqlens(lens)
    offs = oracle.mask_bit_offsets(lens, lens, 2)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        s = slice(cu[b], cu[b + 1])
        # the sequence alone: its mask bits start at bit 0
        nb = 2 * L * L
        bits = oracle.keep_bits_unit(mask, int(offs[b]), 1, nb).reshape(-1).astype(np.uint8)
        bits = np.concatenate([bits, np.zeros((-nb) % 8, np.uint8)])
        sub = np.packbits(bits.reshape(-1, 8), axis=1, bitorder="little").reshape(-1)
        a = (0.5, 3, 1, sub, 0.75)
        y1, m1, l1 = oracle.varlen_forward(q[s], k[s], v[s], [L], [L], *a)
        dq1, dk1, dv1 = oracle.varlen_backward(q[s], k[s], v[s], dy[s], y1, m1, l1,
                                               [L], [L], *a)
        for got, ref in ((y[s], y1), (m[s], m1), (l[s], l1), (dq[s], dq1),
                         (dk[s], dk1), (dv[s], dv1)):
            assert np.array_equal(got, ref)


def test_length_one_causal():
    rng = np.random.default_rng(2)
    q, k, v, dy = _rand_problem(rng, [1], [1], 2, 2, 4)
    y, m, l = oracle.varlen_forward(q, k, v, [1], [1], 0.5, BIG, 0)
    assert np.array_equal(y, v)
    assert np.all(l == 1.0)
    dq, dk, dv = oracle.varlen_backward(q, k, v, dy, y, m, l, [1], [1], 0.5, BIG, 0)
    assert np.array_equal(dv, dy)
    # dS = P (dP - D) with dP = dY.V and D = dY.Y, Y = V: zero up to fp64 round-off
    assert np.abs(dq).max() <= 1e-14 and np.abs(dk).max() <= 1e-14


def test_uniform_attention_closed_form():
    rng = np.random.default_rng(4)
    L, d, scale = 9, 5, 0.4
    q = np.zeros((L, d)); k = rng.standard_normal((L, d))
    v = rng.standard_normal((L, d)); dy = rng.standard_normal((L, d))
    y, m, l = oracle.unit_forward(q, k, v, scale, BIG, BIG)
    np.testing.assert_allclose(y, np.tile(v.mean(axis=0), (L, 1)), rtol=1e-13, atol=1e-14)
    dq, dk, dv = oracle.unit_backward(q, k, v, dy, y, m, l, scale, BIG, BIG)
    np.testing.assert_allclose(dv, np.tile(dy.mean(axis=0), (L, 1)), rtol=1e-13, atol=1e-14)
    assert np.all(dk == 0.0)
    vbar = v.mean(axis=0)
    ref = (scale / L) * ((dy @ (v - vbar).T) @ k)
    np.testing.assert_allclose(dq, ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# library routine: torch fp64 autograd of the explicit forward graph
# ---------------------------------------------------------------------------

def _torch_graph(q, k, v, dy, lens_q, lens_kv, scale, pre, nxt, mask, kp):
    tq = [torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v)]
    qt, kt, vt = tq
    n, nkv = q.shape[1], k.shape[1]
    group = n // nkv
    cq, ck = oracle.cu_seqlens(lens_q), oracle.cu_seqlens(lens_kv)
    offs = oracle.mask_bit_offsets(lens_q, lens_kv, n)
    ys = torch.zeros(q.shape[0], n, v.shape[2], dtype=torch.float64)
    lse = torch.zeros(q.shape[0], n, dtype=torch.float64)
    outs = []
    for b in range(len(lens_q)):
        lq, lk = lens_q[b], lens_kv[b]
        for h in range(n):
            qs = qt[cq[b]:cq[b + 1], h]
            ks = kt[ck[b]:ck[b + 1], h // group]
            vs = vt[ck[b]:ck[b + 1], h // group]
            i = torch.arange(lq)[:, None]
            j = torch.arange(lk)[None, :]
            allowed = (j >= i - pre) & (j <= i + nxt)
            s = (scale * qs @ ks.T).masked_fill(~allowed, float("-inf"))
            p = torch.softmax(s, dim=-1)
            if mask is not None and kp < 1.0:
                idx = int(offs[b]) + h * lq * lk + i * lk + j
                bits = torch.tensor(mask.astype(np.int64))[idx // 8] >> (idx % 8) & 1
                p = p * bits.to(torch.float64) / kp
            outs.append(((cq[b], cq[b + 1], h), p @ vs, torch.logsumexp(s, dim=-1)))
    loss = 0
    for (a, b_, h), y, lz in outs:
        ys[a:b_, h] = y.detach()
        lse[a:b_, h] = lz.detach()
        loss = loss + (y * torch.tensor(dy[a:b_, h])).sum()
    loss.backward()
    return ys.numpy(), lse.numpy(), [t.grad.numpy() for t in tq]


@pytest.mark.parametrize("case", [
    # lens_q, lens_kv, n, nkv, d, pre, next, dropout
    ([37, 64], [37, 64], 2, 2, 64, BIG, BIG, False),            # workload 1's shape
    ([33, 70, 5], [33, 70, 5], 4, 2, 16, BIG, 0, False),         # causal, GQA
    ([40, 17], [40, 17], 2, 2, 8, 6, 0, True),                   # band + dropout
    ([21], [30], 1, 1, 8, 4, 3, False),                          # Lq != Lk, two-sided band
])
def test_against_torch_autograd(case):
    lens_q, lens_kv, n, nkv, d, pre, nxt, drop = case
    rng = np.random.default_rng(21)
    q, k, v, dy = _rand_problem(rng, lens_q, lens_kv, n, nkv, d)
    mask = _mask_for(rng, lens_q, lens_kv, n, 0.9) if drop else None
    kp = 0.9 if drop else 1.0
    scale = 1 / math.sqrt(d)
    y, m, l = oracle.varlen_forward(q, k, v, lens_q, lens_kv, scale, pre, nxt, mask, kp)
    dq, dk, dv = oracle.varlen_backward(q, k, v, dy, y, m, l, lens_q, lens_kv, scale,
                                        pre, nxt, mask, kp)
    ty, tlse, (tdq, tdk, tdv) = _torch_graph(q, k, v, dy, lens_q, lens_kv, scale, pre,
                                             nxt, mask, kp)
    np.testing.assert_allclose(y, ty, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(m[..., 0] + np.log(l[..., 0]), tlse, rtol=1e-12, atol=1e-12)
    for a, b in ((dq, tdq), (dk, tdk), (dv, tdv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------------------
# the page's call example
# ---------------------------------------------------------------------------

def test_page_call_example():
    g = _load("page_example.json")
    t, n, d = g["shape"]
    ones = np.ones((t, n, d))
    stats = np.full((t, n, 8), g["stat_value"])
    dq, dk, dv = oracle.varlen_backward(ones, ones, ones, ones, ones, stats, stats,
                                        g["lens"], g["lens"], g["scale"],
                                        g["pre_tokens"], g["next_tokens"])
    # closed form: dS = 0, every P_ij = exp(scale*d - 3)/3, dV = T * P_ij
    closed = t * math.exp(g["scale"] * d - g["stat_value"]) / g["stat_value"]
    assert np.abs(dq).max() == g["dq_max_abs"] == 0.0
    assert np.abs(dk).max() == g["dk_max_abs"] == 0.0
    assert g["dv_value"] == pytest.approx(closed, rel=1e-13)
    np.testing.assert_allclose(dv, g["dv_value"], rtol=1e-13)


# ---------------------------------------------------------------------------
# the sampled variants agree with the whole-unit backward
# ---------------------------------------------------------------------------

def test_rows_and_cols_match_full_unit():
    rng = np.random.default_rng(9)
    lq, lk, d = 50, 61, 8
    q, dy = rng.standard_normal((lq, d)), rng.standard_normal((lq, d))
    k, v = rng.standard_normal((lk, d)), rng.standard_normal((lk, d))
    z = (rng.random((lq, lk)) < 0.8).astype(np.float64)
    kr = lambda rows: z[np.asarray(rows)]  # noqa: E731
    kc = lambda cols: z[:, np.asarray(cols)]  # noqa: E731
    y, m, l = oracle.unit_forward(q, k, v, 0.35, 20, 3, kr, 0.8, block=16)
    dq, dk, dv = oracle.unit_backward(q, k, v, dy, y, m, l, 0.35, 20, 3, kr, 0.8, block=7)
    rows = [0, 13, 49]
    cols = [0, 31, 60]
    np.testing.assert_allclose(
        oracle.unit_backward_rows(rows, q, k, v, dy, y, m, l, 0.35, 20, 3, kr, 0.8),
        dq[rows], rtol=1e-12, atol=1e-13)
    gk, gv = oracle.unit_backward_cols(cols, q, k, v, dy, y, m, l, 0.35, 20, 3, kc, 0.8)
    np.testing.assert_allclose(gk, dk[cols], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(gv, dv[cols], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# the input generator
# ---------------------------------------------------------------------------

def test_splitmix64_published_vector():
    # SplitMix64 seeded with 1234567: the first three outputs of the
    # published test vector.
    got = [int(x) for x in wl.splitmix64(1234567, np.arange(3))]
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423]


def test_keep_mask_packing_and_rate():
    nbits = 1000003
    b = wl.keep_mask_bytes(7, 0.9, nbits, chunk=4096)
    bits = np.unpackbits(b, bitorder="little")[:nbits]
    assert np.array_equal(bits, wl.keep_bits(7, 0.9, np.arange(nbits)))
    assert abs(bits.mean() - 0.9) < 3e-3
    part = wl.keep_mask_bytes(7, 0.9, nbits, byte_start=1234, byte_count=77)
    assert np.array_equal(part, b[1234:1234 + 77])


def test_workload_shapes():
    w3 = wl.workload(3)
    assert len(w3.lens) == 16 and all(128 <= x <= 4096 for x in w3.lens)
    assert wl.workload(2).total_q == 4096
    assert wl.workload(4).total_q == 65536 and wl.workload(5).total_q == 65536
    assert wl.workload(5).mask_bits == 4 * 16 * 16384 * 16384
    q, k, v, dy = wl.make_tensors(wl.workload(1))
    assert q.shape == (101, 2, 64) and q.dtype == torch.float32


# ---------------------------------------------------------------------------
# outer split (qStartIdx / kvStartIdx)
# ---------------------------------------------------------------------------

def test_window_split_fixture():
    for c in _load("window_split_cases.json")["cases"]:
        got = oracle.window_allowed(c["lq"], c["lk"], c["pre"], c["next"],
                                    q_start=c["q_start"], kv_start=c["kv_start"])
        assert got.astype(int).tolist() == c["allowed"], c


@pytest.mark.parametrize("pre,nxt", [(2 ** 31 - 1, 0), (20, 5)])
def test_query_chunks_reproduce_the_whole_sequence(pre, nxt):
    """Cutting one sequence's queries into chunks, each run against the whole
    key/value sequence with its global start, reproduces the rows of the
    whole run (forward and dQ), and the chunks' dK, dV add up to the whole
    run's: the context-parallel use the outer-split parameters exist for."""
    rng = np.random.default_rng(11)
    L, n, d, cut = 70, 2, 8, 33
    q, k, v, dy = (rng.standard_normal((L, n, d)) for _ in range(4))
    sc = 0.3
    y, m, l = oracle.varlen_forward(q, k, v, [L], [L], sc, pre, nxt)
    dq, dk, dv = oracle.varlen_backward(q, k, v, dy, y, m, l, [L], [L], sc, pre, nxt)
    dk_sum, dv_sum = np.zeros_like(dk), np.zeros_like(dv)
    for a, b in ((0, cut), (cut, L)):
        yc, mc, lc = oracle.varlen_forward(q[a:b], k, v, [b - a], [L], sc, pre, nxt,
                                           q_start=[a], kv_start=[0])
        np.testing.assert_allclose(yc, y[a:b], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(np.isinf(mc), np.isinf(m[a:b]))
        np.testing.assert_allclose(lc, l[a:b], rtol=1e-12, atol=0)
        dqc, dkc, dvc = oracle.varlen_backward(q[a:b], k, v, dy[a:b], yc, mc, lc, [b - a], [L],
                                               sc, pre, nxt, q_start=[a], kv_start=[0])
        np.testing.assert_allclose(dqc, dq[a:b], rtol=0, atol=1e-12)
        dk_sum += dkc
        dv_sum += dvc
    np.testing.assert_allclose(dk_sum, dk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv_sum, dv, rtol=0, atol=1e-12)


def test_key_chunks_reproduce_the_whole_sequence():
    """With the whole run's statistics, backward over key/value chunks (each
    with its global start) gives the whole run's dK, dV rows, and the
    chunks' dQ add up to the whole run's dQ."""
    rng = np.random.default_rng(12)
    L, n, d, cut = 64, 2, 8, 29
    q, k, v, dy = (rng.standard_normal((L, n, d)) for _ in range(4))
    sc, pre, nxt = 0.25, 2 ** 31 - 1, 0
    y, m, l = oracle.varlen_forward(q, k, v, [L], [L], sc, pre, nxt)
    dq, dk, dv = oracle.varlen_backward(q, k, v, dy, y, m, l, [L], [L], sc, pre, nxt)
    dq_sum = np.zeros_like(dq)
    for a, b in ((0, cut), (cut, L)):
        dqc, dkc, dvc = oracle.varlen_backward(q, k[a:b], v[a:b], dy, y, m, l, [L], [b - a],
                                               sc, pre, nxt, q_start=[0], kv_start=[a])
        np.testing.assert_allclose(dkc, dk[a:b], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dvc, dv[a:b], rtol=0, atol=1e-12)
        dq_sum += dqc
    np.testing.assert_allclose(dq_sum, dq, rtol=0, atol=1e-12)


def test_equal_starts_change_nothing():
    """Only the difference of the two starts matters: shifting both by the
    same amount leaves every output unchanged."""
    rng = np.random.default_rng(13)
    lens = [23, 17]
    T = sum(lens)
    q, k, v, dy = (rng.standard_normal((T, 2, 8)) for _ in range(4))
    base = oracle.varlen_forward(q, k, v, lens, lens, 0.3, 5, 2)
    moved = oracle.varlen_forward(q, k, v, lens, lens, 0.3, 5, 2, q_start=[100, 7],
                                  kv_start=[100, 7])
    for a, b in zip(base, moved):
        np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------
# sparseMode readings
# ---------------------------------------------------------------------------

def test_sparse_mode_fixture():
    for c in _load("sparse_mode_cases.json")["cases"]:
        pre_b, next_b = oracle.mode_window(c["mode"], c["pre"], c["next"], c["lq"], c["lk"])
        got = oracle.window_allowed(c["lq"], c["lk"], pre_b, next_b)
        assert got.astype(int).tolist() == c["allowed"], c


def test_lower_triangular_modes_agree_on_square_sequences():
    """For Lq = Lk the two lower-triangular modes and the causal window of
    mode 0 are one mask, so every output agrees."""
    rng = np.random.default_rng(14)
    lens = [19, 33]
    T = sum(lens)
    q, k, v, dy = (rng.standard_normal((T, 2, 8)) for _ in range(4))
    ref = oracle.varlen_forward(q, k, v, lens, lens, 0.3, 2 ** 31 - 1, 0)
    gref = oracle.varlen_backward(q, k, v, dy, *ref, lens, lens, 0.3, 2 ** 31 - 1, 0)
    for mode in (2, 3):
        got = oracle.varlen_forward(q, k, v, lens, lens, 0.3, 5, 7, sparse_mode=mode)
        for a, b in zip(got, ref):
            np.testing.assert_array_equal(a, b)
        g = oracle.varlen_backward(q, k, v, dy, *got, lens, lens, 0.3, 5, 7, sparse_mode=mode)
        for a, b in zip(g, gref):
            np.testing.assert_array_equal(a, b)


def test_bottom_right_mode_is_the_top_left_mode_of_the_last_rows():
    """Mode 3 on (Lq, Lk) with Lq <= Lk aligns the triangle at the last key:
    it equals the top-left triangle of queries that start at global position
    Lk - Lq, i.e. mode 2 with the outer-split start Lk - Lq."""
    rng = np.random.default_rng(15)
    lq, lk = 21, 50
    q, dy = (rng.standard_normal((lq, 2, 8)) for _ in range(2))
    k, v = (rng.standard_normal((lk, 2, 8)) for _ in range(2))
    a = oracle.varlen_forward(q, k, v, [lq], [lk], 0.3, 0, 0, sparse_mode=3)
    b = oracle.varlen_forward(q, k, v, [lq], [lk], 0.3, 0, 0, sparse_mode=2,
                              q_start=[lk - lq], kv_start=[0])
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


# ---------------------------------------------------------------------------
# explicit attention mask
# ---------------------------------------------------------------------------

def test_atten_mask_fixture_through_uniform_attention():
    """With Q = 0 every allowed key gets the same weight, and with one-hot
    value rows Y_i is 1/|allowed_i| on the allowed keys and 0 elsewhere (0
    for a row with no allowed key): the forward's output spells out the
    allowed set, which must match the hand-enumerated matrix."""
    g = _load("atten_mask_cases.json")
    mask = np.array(g["mask"], np.uint8)
    for c in g["cases"]:
        lq, lk = c["lq"], c["lk"]
        q = np.zeros((lq, 1, 8))
        k = np.random.default_rng(1).standard_normal((lk, 1, 8))
        v = np.zeros((lk, 1, 8))
        v[np.arange(lk), 0, np.arange(lk)] = 1.0
        y, m, l = oracle.varlen_forward(q, k, v, [lq], [lk], 0.5, c["pre"], c["next"],
                                        sparse_mode=c["mode"], atten_mask=mask)
        allowed = np.array(c["allowed"], float)
        cnt = allowed.sum(axis=1, keepdims=True)
        want = np.divide(allowed, cnt, out=np.zeros_like(allowed), where=cnt > 0)
        np.testing.assert_allclose(y[:, 0, :lk], want, rtol=0, atol=1e-15)
        assert np.all(np.isinf(m[cnt[:, 0] == 0]))


def test_causal_mask_tensor_equals_the_causal_mode():
    """Mode 1 with the lower-triangular mask tensor (masked iff j > i) is the
    top-left causal mode 2; mode 0 with an all-zero mask is mode 0 alone."""
    rng = np.random.default_rng(16)
    lens = [23, 40]
    T = sum(lens)
    q, k, v, dy = (rng.standard_normal((T, 2, 8)) for _ in range(4))
    tri = (np.arange(48)[None, :] > np.arange(48)[:, None]).astype(np.uint8)
    a = oracle.varlen_forward(q, k, v, lens, lens, 0.3, 0, 0, sparse_mode=1, atten_mask=tri)
    b = oracle.varlen_forward(q, k, v, lens, lens, 0.3, 0, 0, sparse_mode=2)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    ga = oracle.varlen_backward(q, k, v, dy, *a, lens, lens, 0.3, 0, 0, sparse_mode=1,
                                atten_mask=tri)
    gb = oracle.varlen_backward(q, k, v, dy, *b, lens, lens, 0.3, 0, 0, sparse_mode=2)
    for x, y in zip(ga, gb):
        np.testing.assert_array_equal(x, y)
    zero = np.zeros((48, 48), np.uint8)
    c = oracle.varlen_forward(q, k, v, lens, lens, 0.3, 6, 3, atten_mask=zero)
    d = oracle.varlen_forward(q, k, v, lens, lens, 0.3, 6, 3)
    for x, y in zip(c, d):
        np.testing.assert_array_equal(x, y)


def test_atten_mask_gradients_by_finite_differences():
    """dQ, dK, dV under a random mask (mode 1) against central differences
    of L = sum(Y * dY)."""
    rng = np.random.default_rng(17)
    lq, lk, d = 5, 6, 3
    q, dy = rng.standard_normal((lq, 1, d)), rng.standard_normal((lq, 1, d))
    k, v = rng.standard_normal((lk, 1, d)), rng.standard_normal((lk, 1, d))
    mask = (rng.random((lq, lk)) < 0.35).astype(np.uint8)
    sc = 0.7

    def loss(qq, kk, vv):
        y, _, _ = oracle.varlen_forward(qq, kk, vv, [lq], [lk], sc, 0, 0, sparse_mode=1,
                                        atten_mask=mask)
        return float((y * dy).sum())

    y, m, l = oracle.varlen_forward(q, k, v, [lq], [lk], sc, 0, 0, sparse_mode=1,
                                    atten_mask=mask)
    g = oracle.varlen_backward(q, k, v, dy, y, m, l, [lq], [lk], sc, 0, 0, sparse_mode=1,
                               atten_mask=mask)
    h = 1e-6
    for which, x in enumerate((q, k, v)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            num[idx] = (up - loss(*args)) / (2 * h)
        np.testing.assert_allclose(g[which], num, rtol=1e-6, atol=1e-8)
