"""Plain fp64 CPU restatement of FAG-V2's attention forward and backward.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Shares no code with
the CUDA library.

The FAG-V2 page, section "功能说明 / 计算公式" (function description /
formulas), defines, per sequence and head:

    S  = Mask(Q K^T / sqrt(d) + pse, atten_mask)
    P  = Dropout(Softmax(S), keep_prob)
    Y  = P V
    dV = P^T dY
    dQ = (dS K) / sqrt(d)
    dK = (dS^T Q) / sqrt(d)

This module writes those formulas out in numpy float64, one (sequence, head)
unit at a time, in blocks of query rows only so that a long sequence's S is
never held whole (every block computes exactly the rows the formula asks
for; there is no reordering of the arithmetic inside a row).

Readings taken where the page is silent or ambiguous:

* scale.  The parameter table's scaleValue replaces 1/sqrt(d) in all three
  places it appears.
* Mask.  Only the sliding window of the parameter table's preTokens /
  nextTokens rows is modelled (sparseMode 0, no pse, no atten_mask tensor):
  key j is allowed for query i iff ``i - preTokens <= j <= i + nextTokens``,
  both bounds inclusive, indices 0-based inside each sequence.  Causal is
  ``nextTokens = 0`` with ``preTokens >= Lq``.
* Softmax statistics.  softmaxMax is the row maximum of the scaled, masked
  logits S; softmaxSum is sum_j exp(S_ij - max_i) with the natural
  exponential.  The constraint section fixes their TND layout as [T, N, 8];
  all 8 lanes hold the same value.  A row with no allowed key has max = -inf,
  sum = 0 and a zero P row.
* The backward takes the statistics as inputs, as the operator does:
  P_ij = exp(S_ij - max_i) / sum_i.
* Dropout is inverted dropout: Pd = P * Z / keep_prob with Z the keep bit
  (1 = keep).  keep_prob = 1 ignores the mask.  The dropMask parameter is a
  1-D UINT8 tensor; the bit layout read here packs one bit per
  (b, n, i, j) at index ``O_b + (n * Lq_b + i) * Lk_b + j`` with
  ``O_b = N * sum_{b' < b} Lq_b' * Lk_b'`` (the per-segment [N, Sq_i, Skv_i]
  flattening the constraint section gives for TND pse), least significant
  bit first within a byte (the bit-per-boolean convention of the sibling
  operator aclnnFusedLinearCrossEntropyLossGrad's targetMask).
* dS is the gradient of the loss with respect to S:
  ``dS = P * (dP * Z / keep_prob - D)`` with ``dP = dY V^T`` and
  ``D_i = sum_d dY_id * Y_id`` (Y = the attentionIn input).
* Grouped heads (the constraint section allows Nq/Nkv integer): query head
  n reads key/value head ``n // (Nq / Nkv)``.
* sparseMode (parameter table: 0..8, 5 unsupported; constraint section:
  modes 1, 2 and 3 ignore preTokens / nextTokens, modes 0 and 4 need the
  attention mask to agree with the preTokens / nextTokens window, and modes
  0, 2 and 3 are the lower-triangular mask cases).  The per-mode doc is not
  on the page.  Readings: modes 0 and 4 are the preTokens / nextTokens
  window; mode 2 is the lower-triangular mask aligned at the top-left corner
  (j <= i); mode 3 is the lower-triangular mask aligned at the bottom-right
  corner (j <= i + Lk - Lq).  Other modes are not modelled.
* attenMaskOptional (parameter table: 1 = the position does not take part,
  0 = it does; shapes [B,N,Sq,Skv] ... [Sq,Skv]).  Reading: one [Sq, Skv]
  matrix shared by every sequence and head, indexed by the chunk-local
  (i, j) of each sequence; sparseMode 1 applies it alone (no window), modes
  0 and 4 apply it together with the preTokens / nextTokens window (the
  constraint section asks the two to agree), modes 2 and 3 do not read it.
* Outer split (the parameter table's qStartIdxOptional / kvStartIdxOptional:
  the global start index of this chunk's query / key-value sequence).  The
  window is evaluated on global positions: key j of the chunk is allowed
  for query i iff ``(qs + i) - preTokens <= ks + j <= (qs + i) + nextTokens``
  with qs, ks the chunk's starts (one pair per sequence, 0 when absent).
  The keep-mask bits stay indexed by the chunk-local (i, j).
"""

from __future__ import annotations

import numpy as np

ROW_BLOCK = 512


# ---------------------------------------------------------------------------
# index helpers
# ---------------------------------------------------------------------------

def cu_seqlens(lens) -> np.ndarray:
    """Start offset of each sequence in the packed T axis (TND layout: the
    constraint section packs every batch's tokens tightly along T)."""
    lens = np.asarray(lens, dtype=np.int64)
    out = np.zeros(len(lens) + 1, dtype=np.int64)
    out[1:] = np.cumsum(lens)
    return out


def mask_bit_offsets(lens_q, lens_kv, n_heads: int) -> np.ndarray:
    """First dropout-mask bit of each sequence, O_b = N * sum_{b'<b} Lq*Lk
    (reading of the parameter table's 1-D UINT8 dropMaskOptional)."""
    lq = np.asarray(lens_q, dtype=np.int64)
    lk = np.asarray(lens_kv, dtype=np.int64)
    per = n_heads * lq * lk
    out = np.zeros(len(lq), dtype=np.int64)
    out[1:] = np.cumsum(per)[:-1]
    return out


UNBOUNDED = 2 ** 31 - 1


def mode_window(sparse_mode: int, pre_tokens: int, next_tokens: int, lq: int, lk: int):
    """(pre, next) window of one sequence under the sparseMode readings of
    the module docstring."""
    if sparse_mode in (0, 4):
        return pre_tokens, next_tokens
    if sparse_mode == 1:
        return UNBOUNDED, UNBOUNDED
    if sparse_mode == 2:
        return UNBOUNDED, 0
    if sparse_mode == 3:
        return UNBOUNDED, lk - lq
    raise ValueError(f"sparse mode {sparse_mode} is not modelled")


def window_allowed(lq: int, lk: int, pre_tokens: int, next_tokens: int,
                   rows=None, q_start: int = 0, kv_start: int = 0) -> np.ndarray:
    """Allowed (i, j) pairs of one sequence for the preTokens/nextTokens
    sliding window of the parameter table, on global positions
    ``gi = q_start + i``, ``gj = kv_start + j``: ``gi - pre <= gj <= gi + next``."""
    i = (np.arange(lq, dtype=np.int64) if rows is None
         else np.asarray(rows, dtype=np.int64))[:, None] + int(q_start)
    j = np.arange(lk, dtype=np.int64)[None, :] + int(kv_start)
    return (j >= i - pre_tokens) & (j <= i + next_tokens)


def keep_bits_unit(mask_u8: np.ndarray, bit_offset: int, lq: int, lk: int,
                   rows=None, cols=None) -> np.ndarray:
    """Keep bits Z[i, j] (0.0 or 1.0) of one (sequence, head) unit whose bits
    start at ``bit_offset``: bit ``bit_offset + i * lk + j``, LSB first."""
    i = (np.arange(lq, dtype=np.int64) if rows is None
         else np.asarray(rows, dtype=np.int64))[:, None]
    j = (np.arange(lk, dtype=np.int64) if cols is None
         else np.asarray(cols, dtype=np.int64))[None, :]
    idx = np.int64(bit_offset) + i * np.int64(lk) + j
    byte = np.asarray(mask_u8, dtype=np.uint8)[idx >> 3]
    return ((byte >> (idx & 7).astype(np.uint8)) & 1).astype(np.float64)


# ---------------------------------------------------------------------------
# one (sequence, head) unit
# ---------------------------------------------------------------------------

def unit_logits(q_rows: np.ndarray, k: np.ndarray, scale: float,
                allowed_rows: np.ndarray) -> np.ndarray:
    """S = Mask(scale * Q K^T): masked entries are -inf (formula for S)."""
    s = scale * (q_rows @ k.T)
    return np.where(allowed_rows, s, -np.inf)


def _softmax_stats(s: np.ndarray):
    """Row max and row sum of exp(S - max); empty rows give (-inf, 0)."""
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 for masked entries
    l = e.sum(axis=1)
    m = np.where(empty, -np.inf, m)
    l = np.where(empty, 0.0, l)
    return m, l


def _probs(s: np.ndarray, m: np.ndarray, l: np.ndarray) -> np.ndarray:
    """P_ij = exp(S_ij - max_i) / sum_i from given statistics; rows whose
    sum is 0 (no allowed key) and masked entries give 0."""
    ok = (l > 0) & np.isfinite(m)
    m_safe = np.where(ok, m, 0.0)
    l_safe = np.where(ok, l, 1.0)
    p = np.exp(s - m_safe[:, None]) / l_safe[:, None]
    return np.where(ok[:, None], p, 0.0)


def _zscale(keep_rows, r0, r1, lk, keep_prob):
    """Z / keep_prob for rows [r0, r1); all ones when dropout is off."""
    if keep_rows is None or keep_prob >= 1.0:
        return np.ones((r1 - r0, lk))
    return keep_rows(np.arange(r0, r1)) / keep_prob


def unit_forward(q, k, v, scale, pre_tokens, next_tokens, keep_rows=None,
                 keep_prob=1.0, block=ROW_BLOCK, q_start=0, kv_start=0, masked=None):
    """Y = Dropout(Softmax(S), keep_prob) V for one unit, plus the softmax
    statistics (max, sum) the forward hands to the backward.

    ``keep_rows(rows) -> [len(rows), Lk]`` returns keep bits, or None."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    lq, lk = q.shape[0], k.shape[0]
    y = np.zeros((lq, v.shape[1]))
    m = np.full(lq, -np.inf)
    l = np.zeros(lq)
    for r0 in range(0, lq, block):
        r1 = min(lq, r0 + block)
        allowed = window_allowed(lq, lk, pre_tokens, next_tokens, np.arange(r0, r1),
                                 q_start, kv_start)
        if masked is not None:
            allowed &= ~masked[r0:r1]
        s = unit_logits(q[r0:r1], k, scale, allowed)
        mb, lb = _softmax_stats(s)
        p = _probs(s, mb, lb)
        pd = p * _zscale(keep_rows, r0, r1, lk, keep_prob)
        y[r0:r1] = pd @ v
        m[r0:r1] = mb
        l[r0:r1] = lb
    return y, m, l


def unit_backward(q, k, v, dy, y, m, l, scale, pre_tokens, next_tokens,
                  keep_rows=None, keep_prob=1.0, block=ROW_BLOCK,
                  return_ds=False, q_start=0, kv_start=0, masked=None):
    """dQ, dK, dV of one unit from the backward formulas, using the given
    forward output ``y`` (attentionIn) and statistics ``m``/``l``.

    dV = Pd^T dY;  dP = dY V^T;  D = rowsum(dY * Y);
    dS = P * (dP * Z / keep_prob - D);  dQ = scale dS K;  dK = scale dS^T Q.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); dy = np.asarray(dy, np.float64)
    y = np.asarray(y, np.float64)
    m = np.asarray(m, np.float64); l = np.asarray(l, np.float64)
    lq, lk = q.shape[0], k.shape[0]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros((lk, v.shape[1]))
    ds_all = np.zeros((lq, lk)) if return_ds else None
    dsum = (dy * y).sum(axis=1)
    for r0 in range(0, lq, block):
        r1 = min(lq, r0 + block)
        allowed = window_allowed(lq, lk, pre_tokens, next_tokens, np.arange(r0, r1),
                                 q_start, kv_start)
        if masked is not None:
            allowed &= ~masked[r0:r1]
        s = unit_logits(q[r0:r1], k, scale, allowed)
        p = _probs(s, m[r0:r1], l[r0:r1])
        z = _zscale(keep_rows, r0, r1, lk, keep_prob)
        dv += (p * z).T @ dy[r0:r1]
        dp = dy[r0:r1] @ v.T
        ds = p * (dp * z - dsum[r0:r1, None])
        dq[r0:r1] = scale * (ds @ k)
        dk += scale * (ds.T @ q[r0:r1])
        if return_ds:
            ds_all[r0:r1] = ds
    if return_ds:
        return dq, dk, dv, ds_all
    return dq, dk, dv


def unit_backward_rows(rows, q, k, v, dy, y, m, l, scale, pre_tokens,
                       next_tokens, keep_rows=None, keep_prob=1.0, q_start=0, kv_start=0,
                       masked=None):
    """dQ at the given query rows only (each row of dS needs only its own
    row of S, dP and D)."""
    rows = np.asarray(rows, dtype=np.int64)
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); dy = np.asarray(dy, np.float64)
    y = np.asarray(y, np.float64)
    lq, lk = q.shape[0], k.shape[0]
    allowed = window_allowed(lq, lk, pre_tokens, next_tokens, rows, q_start, kv_start)
    if masked is not None:
        allowed &= ~masked[rows]
    s = unit_logits(q[rows], k, scale, allowed)
    p = _probs(s, np.asarray(m, np.float64)[rows], np.asarray(l, np.float64)[rows])
    if keep_rows is None or keep_prob >= 1.0:
        z = np.ones_like(p)
    else:
        z = keep_rows(rows) / keep_prob
    dp = dy[rows] @ v.T
    dsum = (dy[rows] * y[rows]).sum(axis=1)
    ds = p * (dp * z - dsum[:, None])
    return scale * (ds @ k)


def unit_backward_cols(cols, q, k, v, dy, y, m, l, scale, pre_tokens,
                       next_tokens, keep_cols=None, keep_prob=1.0, q_start=0, kv_start=0,
                       masked=None):
    """dK and dV at the given key rows only (column j of P and dS runs over
    every query row i, so the full statistics m, l and D are used).

    ``keep_cols(cols) -> [Lq, len(cols)]`` returns keep bits, or None."""
    cols = np.asarray(cols, dtype=np.int64)
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); dy = np.asarray(dy, np.float64)
    y = np.asarray(y, np.float64)
    m = np.asarray(m, np.float64); l = np.asarray(l, np.float64)
    lq, lk = q.shape[0], k.shape[0]
    i = np.arange(lq, dtype=np.int64)[:, None] + int(q_start)
    j = cols[None, :] + int(kv_start)
    allowed = (j >= i - pre_tokens) & (j <= i + next_tokens)
    if masked is not None:
        allowed &= ~masked[:, cols]
    s = np.where(allowed, scale * (q @ k[cols].T), -np.inf)
    p = _probs(s, m, l)
    if keep_cols is None or keep_prob >= 1.0:
        z = np.ones_like(p)
    else:
        z = keep_cols(cols) / keep_prob
    dp = dy @ v[cols].T
    dsum = (dy * y).sum(axis=1)
    ds = p * (dp * z - dsum[:, None])
    dk = scale * (ds.T @ q)
    dv = (p * z).T @ dy
    return dk, dv


# ---------------------------------------------------------------------------
# packed varlen (TND) wrappers
# ---------------------------------------------------------------------------

def _keep_fns(mask_u8, bit_off, lq, lk):
    if mask_u8 is None:
        return None, None
    rows_fn = lambda rows: keep_bits_unit(mask_u8, bit_off, lq, lk, rows=rows)  # noqa: E731
    cols_fn = lambda cols: keep_bits_unit(mask_u8, bit_off, lq, lk, cols=cols)  # noqa: E731
    return rows_fn, cols_fn


def _unit_mask(atten_mask, sparse_mode, lq, lk):
    """The attention mask's [lq, lk] corner as booleans (True = masked out),
    or None where the mode does not read it."""
    if atten_mask is None or sparse_mode not in (0, 1, 4):
        return None
    return np.asarray(atten_mask)[:lq, :lk] != 0


def _starts(starts, batch):
    return [0] * batch if starts is None else [int(x) for x in starts]


def varlen_forward(q, k, v, lens_q, lens_kv, scale, pre_tokens, next_tokens,
                   mask_u8=None, keep_prob=1.0, q_start=None, kv_start=None, sparse_mode=0,
                   atten_mask=None):
    """Forward over a packed batch: q [Tq, N, D], k/v [Tk, Nkv, D*].
    ``q_start`` / ``kv_start``: per-sequence global start indices of the
    chunks (outer split), or None for zeros.
    Returns y [Tq, N, Dv], softmax_max [Tq, N, 8], softmax_sum [Tq, N, 8]."""
    qs0, ks0 = _starts(q_start, len(lens_q)), _starts(kv_start, len(lens_q))
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n_heads, n_kv = q.shape[1], k.shape[1]
    group = n_heads // n_kv
    cq, ck = cu_seqlens(lens_q), cu_seqlens(lens_kv)
    offs = mask_bit_offsets(lens_q, lens_kv, n_heads)
    y = np.zeros((q.shape[0], n_heads, v.shape[2]))
    smax = np.full((q.shape[0], n_heads, 8), -np.inf)
    ssum = np.zeros((q.shape[0], n_heads, 8))
    for b in range(len(lens_q)):
        lq, lk = int(lens_q[b]), int(lens_kv[b])
        if lq == 0:
            continue
        for n in range(n_heads):
            kv = n // group
            rows_fn, _ = _keep_fns(mask_u8, int(offs[b]) + n * lq * lk, lq, lk)
            pre_b, next_b = mode_window(sparse_mode, pre_tokens, next_tokens, lq, lk)
            yb, mb, lb = unit_forward(q[cq[b]:cq[b + 1], n], k[ck[b]:ck[b + 1], kv],
                                      v[ck[b]:ck[b + 1], kv], scale, pre_b, next_b,
                                      rows_fn, keep_prob, q_start=qs0[b], kv_start=ks0[b],
                                      masked=_unit_mask(atten_mask, sparse_mode, lq, lk))
            y[cq[b]:cq[b + 1], n] = yb
            smax[cq[b]:cq[b + 1], n, :] = mb[:, None]
            ssum[cq[b]:cq[b + 1], n, :] = lb[:, None]
    return y, smax, ssum


def varlen_backward(q, k, v, dy, y, softmax_max, softmax_sum, lens_q, lens_kv,
                    scale, pre_tokens, next_tokens, mask_u8=None, keep_prob=1.0,
                    q_start=None, kv_start=None, sparse_mode=0, atten_mask=None):
    """Backward over a packed batch; reads lane 0 of the [T, N, 8] statistics.
    Returns dq [Tq, N, D], dk [Tk, Nkv, D], dv [Tk, Nkv, Dv] (grouped query
    heads add into their shared key/value head)."""
    qs0, ks0 = _starts(q_start, len(lens_q)), _starts(kv_start, len(lens_q))
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); dy = np.asarray(dy, np.float64)
    y = np.asarray(y, np.float64)
    smax = np.asarray(softmax_max, np.float64)
    ssum = np.asarray(softmax_sum, np.float64)
    n_heads, n_kv = q.shape[1], k.shape[1]
    group = n_heads // n_kv
    cq, ck = cu_seqlens(lens_q), cu_seqlens(lens_kv)
    offs = mask_bit_offsets(lens_q, lens_kv, n_heads)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(len(lens_q)):
        lq, lk = int(lens_q[b]), int(lens_kv[b])
        if lq == 0 or lk == 0:
            continue
        qs, ks = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
        for n in range(n_heads):
            kv = n // group
            rows_fn, _ = _keep_fns(mask_u8, int(offs[b]) + n * lq * lk, lq, lk)
            pre_b, next_b = mode_window(sparse_mode, pre_tokens, next_tokens, lq, lk)
            dqb, dkb, dvb = unit_backward(q[qs, n], k[ks, kv], v[ks, kv], dy[qs, n],
                                          y[qs, n], smax[qs, n, 0], ssum[qs, n, 0],
                                          scale, pre_b, next_b, rows_fn,
                                          keep_prob, q_start=qs0[b], kv_start=ks0[b],
                                          masked=_unit_mask(atten_mask, sparse_mode, lq, lk))
            dq[qs, n] = dqb
            dk[ks, kv] += dkb
            dv[ks, kv] += dvb
    return dq, dk, dv
