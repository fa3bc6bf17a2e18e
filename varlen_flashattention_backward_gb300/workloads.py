"""Seeded synthetic workloads for the varlen attention backward.

This module only draws inputs: shapes, sequence lengths, N(0, 1) tensors
and dropout keep bits.  It holds none of the attention arithmetic, so both
the fp64 oracle (through the tests) and the CUDA library can be fed from it.

The five workloads are the ones the library is measured and checked on:

1. fp32, lengths [37, 64] (T = 101), N = 2, D = 64, no mask.
2. bf16, lengths [512, 1024, 2048, 512] (T = 4096), N = 16, D = 128, causal.
3. bf16, 16 lengths uniform in [128, 4096] drawn from the seed, N = 32,
   D = 128, causal, dY ~ 0.1 * N(0, 1).
4. bf16, 2 x 32768 (T = 65536), N = 8, D = 128, causal.
5. bf16, 4 x 16384 (T = 65536), N = 16, D = 128, sliding window
   preTokens = 4096 / nextTokens = 0, dropout keep_prob = 0.9.

Workload 6 is the profiling case: bf16, 8 x 2048 (T = 16384), N = 16,
D = 128, causal.  Its inputs (335 MB) exceed L2 while one backward launch
stays well under a millisecond.  Workloads 15 and 16 are workload 5 cut to
2 x 8192 tokens (the same window and heads), with and without dropout: the
dropout path's profiling pair (0.5 GB of inputs and keep bits).

Every workload uses scale = 1/sqrt(D).  Q, K, V and dY are drawn in fp32
from one ``torch.Generator`` seeded with ``seed`` (order: lengths when they
are random, then Q, K, V, dY) and rounded to the storage dtype.

Dropout keep bits come from SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014; finaliser constants
of the published reference implementation): bit g of the mask is
``splitmix64(seed, g) < floor(keep_prob * 2**64)``, where
``splitmix64(seed, g)`` is the generator's output number g + 1 after seeding
its state with ``seed``.  Bits are packed least significant bit first.  The
CUDA library carries a twin of this generator (``fa_gen_keep_mask``) so that
multi-gigabyte masks can be produced on the device; the tests compare the
two bit for bit.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

UNBOUNDED = 2 ** 31 - 1          # preTokens / nextTokens value meaning "no bound"

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)


@dataclass
class Workload:
    cid: int
    dtype: str                    # "fp32" | "bf16" | "fp16"
    lens: list
    n_heads: int
    head_dim: int
    pre_tokens: int
    next_tokens: int
    keep_prob: float = 1.0
    dy_std: float = 1.0
    seed: int = 0
    mask_seed: int = 0x5EED
    n_heads_kv: int = 0           # 0 -> same as n_heads
    lens_kv: list = field(default=None)
    sparse_mode: int = 0
    q_start: list = field(default=None)    # outer split: per-sequence chunk starts
    kv_start: list = field(default=None)
    mask_density: float = 0.0     # > 0: an explicit attention mask, this share excluded

    def __post_init__(self):
        if not self.n_heads_kv:
            self.n_heads_kv = self.n_heads
        if self.lens_kv is None:
            self.lens_kv = list(self.lens)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def total_q(self) -> int:
        return int(sum(self.lens))

    @property
    def total_kv(self) -> int:
        return int(sum(self.lens_kv))

    @property
    def mask_bits(self) -> int:
        return int(sum(self.n_heads * a * b for a, b in zip(self.lens, self.lens_kv)))

    @property
    def torch_dtype(self):
        return {"fp32": torch.float32, "bf16": torch.bfloat16,
                "fp16": torch.float16}[self.dtype]

    def describe(self) -> str:
        mask = ("causal" if self.next_tokens == 0 and self.pre_tokens >= max(self.lens_kv, default=0)
                else "none" if self.pre_tokens >= max(self.lens_kv, default=0)
                and self.next_tokens >= max(self.lens_kv, default=0)
                else f"band pre={self.pre_tokens} next={self.next_tokens}")
        s = (f"{self.dtype} TND lens={_short(self.lens)} T={self.total_q} "
             f"N={self.n_heads} D={self.head_dim} mask={mask}")
        if self.keep_prob < 1.0:
            s += f" dropout keep_prob={self.keep_prob}"
        if self.lens_kv != self.lens:
            s += f" lens_kv={_short(self.lens_kv)}"
        if self.n_heads_kv != self.n_heads:
            s += f" Nkv={self.n_heads_kv}"
        if self.sparse_mode:
            s += f" sparse_mode={self.sparse_mode}"
        if self.q_start is not None:
            s += f" q_start={_short(self.q_start)} kv_start={_short(self.kv_start)}"
        if self.mask_density > 0:
            s += f" atten_mask density={self.mask_density}"
        return s


def _short(lens):
    if len(lens) <= 6:
        return "[" + ",".join(str(x) for x in lens) + "]"
    return f"[{len(lens)} seqs {min(lens)}..{max(lens)}]"


def config3_lengths(seed: int = 0) -> list:
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(128, 4097, (16,), generator=g)]


def workload(cid: int, seed: int = 0) -> Workload:
    """The five reference workloads (see the module docstring)."""
    if cid == 1:
        return Workload(1, "fp32", [37, 64], 2, 64, UNBOUNDED, UNBOUNDED, seed=seed)
    if cid == 2:
        return Workload(2, "bf16", [512, 1024, 2048, 512], 16, 128, UNBOUNDED, 0, seed=seed)
    if cid == 3:
        return Workload(3, "bf16", config3_lengths(seed), 32, 128, UNBOUNDED, 0,
                        dy_std=0.1, seed=seed)
    if cid == 4:
        return Workload(4, "bf16", [32768, 32768], 8, 128, UNBOUNDED, 0, seed=seed)
    if cid == 5:
        return Workload(5, "bf16", [16384] * 4, 16, 128, 4096, 0, keep_prob=0.9, seed=seed)
    if cid == 6:
        return Workload(6, "bf16", [2048] * 8, 16, 128, UNBOUNDED, 0, seed=seed)
    if cid == 7:
        # head dim 64: the bench mix with twice the heads (the same bytes)
        return Workload(7, "bf16", [512, 1024, 2048, 512], 32, 64, UNBOUNDED, 0, seed=seed)
    bench_lens = [512, 1024, 2048, 512]
    if cid == 8:
        # grouped-query heads: 32 query heads on 8 key/value heads
        return Workload(8, "bf16", bench_lens, 32, 128, UNBOUNDED, 0, seed=seed, n_heads_kv=8)
    if cid == 9:
        return Workload(9, "fp16", bench_lens, 16, 128, UNBOUNDED, 0, seed=seed)
    if cid == 10:
        # outer split: the second half of four causal 2048-token sequences
        return Workload(10, "bf16", [1024] * 4, 16, 128, UNBOUNDED, 0, seed=seed,
                        lens_kv=[2048] * 4, q_start=[1024] * 4, kv_start=[0] * 4)
    if cid == 11:
        # bottom-right causal (sparseMode 3): queries are the last part of the keys
        return Workload(11, "bf16", [256, 512, 1024, 256], 16, 128, UNBOUNDED, 0, seed=seed,
                        lens_kv=[1024, 2048, 4096, 1024], sparse_mode=3)
    if cid == 12:
        # an explicit mask (sparseMode 1), 30% of the pairs excluded
        return Workload(12, "bf16", bench_lens, 16, 128, UNBOUNDED, UNBOUNDED, seed=seed,
                        sparse_mode=1, mask_density=0.3)
    if cid == 13:
        # head dim 96 (zero-padded to 128 on the tensor cores)
        return Workload(13, "bf16", bench_lens, 16, 96, UNBOUNDED, 0, seed=seed)
    if cid == 14:
        # head dim 32 (zero-padded to 64 on the tensor cores)
        return Workload(14, "bf16", bench_lens, 32, 32, UNBOUNDED, 0, seed=seed)
    if cid in (15, 16):
        # workload 5 cut to two sequences of 8192 tokens, with (15) and
        # without (16) dropout
        return Workload(cid, "bf16", [8192] * 2, 16, 128, 4096, 0,
                        keep_prob=0.9 if cid == 15 else 1.0, seed=seed)
    raise ValueError(f"unknown workload {cid}")


def make_tensors(w: Workload):
    """Q, K, V, dY as CPU torch tensors in the workload's dtype, TND layout."""
    g = torch.Generator().manual_seed(w.seed)
    if w.cid == 3:
        torch.randint(128, 4097, (16,), generator=g)   # the lengths' draw comes first
    shp_q = (w.total_q, w.n_heads, w.head_dim)
    shp_k = (w.total_kv, w.n_heads_kv, w.head_dim)
    q = torch.randn(shp_q, generator=g, dtype=torch.float32)
    k = torch.randn(shp_k, generator=g, dtype=torch.float32)
    v = torch.randn(shp_k, generator=g, dtype=torch.float32)
    dy = torch.randn(shp_q, generator=g, dtype=torch.float32) * w.dy_std
    dt = w.torch_dtype
    return q.to(dt), k.to(dt), v.to(dt), dy.to(dt)


def make_atten_mask(w: Workload):
    """The workload's explicit attention mask (uint8, 1 = excluded), drawn
    from its seed, or None."""
    if w.mask_density <= 0:
        return None
    g = np.random.default_rng(w.seed + 77)
    rows, cols = max(w.lens), max(w.lens_kv)
    return (g.random((rows, cols)) < w.mask_density).astype(np.uint8)


def make_tensors_on_device(w: Workload, device):
    """Q, K, V, dY drawn on ``device`` by torch's seeded generator there.

    For inputs of billions of values, where drawing them on the host would
    take minutes; the values differ from ``make_tensors`` but are fixed by
    the seed.  Callers hand slices of them to the oracle."""
    g = torch.Generator(device=device).manual_seed(w.seed)
    shp_q = (w.total_q, w.n_heads, w.head_dim)
    shp_k = (w.total_kv, w.n_heads_kv, w.head_dim)
    dt = w.torch_dtype
    out = []
    for shp, std in ((shp_q, 1.0), (shp_k, 1.0), (shp_k, 1.0), (shp_q, w.dy_std)):
        t = torch.randn(shp, generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            t.mul_(std)
        out.append(t.to(dt))
        del t
    return tuple(out)


# ---------------------------------------------------------------------------
# SplitMix64 dropout keep bits (CPU side of the generator pair)
# ---------------------------------------------------------------------------

def splitmix64(seed: int, index) -> np.ndarray:
    """Output number ``index + 1`` of SplitMix64 seeded with ``seed``."""
    idx = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & (2 ** 64 - 1)) + (idx + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
        z = z ^ (z >> np.uint64(31))
    return z


def keep_threshold(keep_prob: float) -> int:
    """floor(keep_prob * 2**64); 2**64 means keep everything."""
    if keep_prob >= 1.0:
        return 2 ** 64
    return int(math.floor(keep_prob * 2.0 ** 64))


def keep_bits(seed: int, keep_prob: float, index) -> np.ndarray:
    """Keep bit (0/1, uint8) at each global bit index."""
    thr = keep_threshold(keep_prob)
    idx = np.asarray(index, dtype=np.int64)
    if thr >= 2 ** 64:
        return np.ones(idx.shape, dtype=np.uint8)
    return (splitmix64(seed, idx.astype(np.uint64)) < np.uint64(thr)).astype(np.uint8)


def keep_mask_bytes(seed: int, keep_prob: float, nbits: int, byte_start: int = 0,
                    byte_count: int | None = None, chunk: int = 1 << 22) -> np.ndarray:
    """Packed mask bytes [byte_start, byte_start + byte_count) of an
    ``nbits``-bit mask (bits past ``nbits`` in the last byte are 0)."""
    total = (nbits + 7) // 8
    if byte_count is None:
        byte_count = total - byte_start
    out = np.zeros(byte_count, dtype=np.uint8)
    weights = (1 << np.arange(8, dtype=np.uint16)).astype(np.uint16)
    for c0 in range(0, byte_count, chunk):
        c1 = min(byte_count, c0 + chunk)
        bits = (np.arange((byte_start + c0) * 8, (byte_start + c1) * 8, dtype=np.int64))
        kb = keep_bits(seed, keep_prob, bits)
        kb[bits >= nbits] = 0
        out[c0:c1] = (kb.reshape(-1, 8).astype(np.uint16) * weights).sum(axis=1).astype(np.uint8)
    return out


def make_keep_mask(w: Workload) -> np.ndarray | None:
    """The whole packed mask on the CPU (only sensible for small workloads)."""
    if w.keep_prob >= 1.0:
        return None
    return keep_mask_bytes(w.mask_seed, w.keep_prob, w.mask_bits)
