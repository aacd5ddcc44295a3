"""Seeded synthetic inputs for paged MLA decode.

This module only draws random numbers and lays them out: it holds none of the
decode arithmetic.  Both the CUDA path's tests/bench and the fp64 oracle take
their inputs from here, as plain numpy arrays of the exact bits the GPU gets:

  q_bits       uint16 [B, Sq, H, 576]          bf16 bit patterns, ~N(0, 1)
  cache        uint16 [P, page_size, 576]      bf16 bits, ~N(0, 1)      (bf16 cache)
               uint8  [P, page_size, 576]      e4m3 codes of N(0,1)/s  (fp8 cache)
  kv_scale     float  s = amax / 448 for fp8, 1.0 for bf16
  block_table  int32  [B, max_blocks]          a seeded random permutation of pages
  seq_lens     int32  [B]

Random numbers come from numpy's counter-based Philox generator, one stream
per (seed, tag, chunk), so large tensors are drawn in chunks and redrawn
identically.  The workload shapes follow the sweeps on the pages: the nh128
batch x context grid of the HK MLA decode table, the fp8 long-context gather
shapes at page_size 64, the MTP head/token pairs, and a ragged batch.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

D_QK = 576
D_V = 512
KV_BF16 = 0
KV_FP8_E4M3 = 1
E4M3_MAX = 448.0
DEFAULT_SCALE = 1.0 / math.sqrt(192.0)

_CHUNK = 1 << 22  # elements per random chunk


def _rng(seed: int, tag: int, chunk: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[seed & 0xFFFFFFFFFFFFFFFF,
                                                     (tag << 32) | chunk]))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Saturating float32 -> fp8 E4M3FN codes (nearest-even, via torch's cast)."""
    import torch
    t = torch.from_numpy(np.clip(np.ascontiguousarray(x, np.float32), -E4M3_MAX, E4M3_MAX))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _normal_f32(seed: int, tag: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float32)
    for c, lo in enumerate(range(0, n, _CHUNK)):
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = _rng(seed, tag, c).standard_normal(hi - lo, dtype=np.float32)
    return out


@dataclass
class Problem:
    """One decode call's inputs, as the exact bits both sides consume."""
    q_bits: np.ndarray
    cache: np.ndarray
    kv_dtype: int
    kv_scale: float
    page_size: int
    block_table: np.ndarray
    seq_lens: np.ndarray
    softmax_scale: float
    causal: bool
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.q_bits.shape[0])

    @property
    def sq(self) -> int:
        return int(self.q_bits.shape[1])

    @property
    def heads(self) -> int:
        return int(self.q_bits.shape[2])

    @property
    def num_pages(self) -> int:
        return int(self.cache.shape[0])


def make_block_table(seed: int, seq_lens, page_size: int, extra_pages: int = 0,
                     poison: bool = False):
    """Give every sequence ceil(ctx/ps) pages drawn from one shuffled pool.

    Returns (block_table [B, max_blocks] int32, num_pages).  Entries past a
    sequence's last page are -1 when ``poison`` (they must never be read),
    else 0.
    """
    seq_lens = np.asarray(seq_lens, np.int64)
    nblk = (seq_lens + page_size - 1) // page_size
    total = int(nblk.sum()) + int(extra_pages)
    total = max(total, 1)
    perm = _rng(seed, 7).permutation(total).astype(np.int32)
    width = max(1, int(nblk.max()) if len(nblk) else 1)
    bt = np.full((len(seq_lens), width), -1 if poison else 0, np.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[off:off + n]
        off += int(n)
    return bt, total


def make_problem(batch: int, sq: int, heads: int, seq_lens, page_size: int,
                 kv_dtype: int = KV_BF16, causal: bool = False, seed: int = 0,
                 softmax_scale: float = DEFAULT_SCALE, outlier_frac: float = 0.0,
                 outlier_mult: float = 8.0, poison: bool = False, extra_pages: int = 0,
                 name: str = "") -> Problem:
    """Draw q ~ N(0,1) and a paged latent cache ~ N(0,1) (bf16 or fp8)."""
    seq_lens = np.asarray(seq_lens, np.int32).reshape(batch)
    bt, num_pages = make_block_table(seed, seq_lens, page_size, extra_pages, poison)
    q = _normal_f32(seed, 1, batch * sq * heads * D_QK)
    q_bits = f32_to_bf16_bits(q).reshape(batch, sq, heads, D_QK)
    n_rows = num_pages * page_size
    x = _normal_f32(seed, 2, n_rows * D_QK).reshape(n_rows, D_QK)
    if outlier_frac > 0:
        k = max(1, int(round(outlier_frac * n_rows)))
        idx = _rng(seed, 3).choice(n_rows, size=k, replace=False)
        x[idx] *= np.float32(outlier_mult)
    if kv_dtype == KV_BF16:
        cache = f32_to_bf16_bits(x).reshape(num_pages, page_size, D_QK)
        kv_scale = 1.0
    else:
        amax = float(np.abs(x).max())
        kv_scale = float(np.float32(amax / E4M3_MAX))
        cache = np.empty(n_rows * D_QK, np.uint8)
        flat = x.reshape(-1)
        inv = np.float32(1.0) / np.float32(kv_scale)
        for lo in range(0, flat.size, _CHUNK):
            cache[lo:lo + _CHUNK] = f32_to_e4m3(flat[lo:lo + _CHUNK] * inv)
        cache = cache.reshape(num_pages, page_size, D_QK)
    del x
    if poison:
        # Slots past each sequence's last key in its last page hold NaN: a
        # correct kernel never reads them.
        nan = np.uint16(0x7FC0) if kv_dtype == KV_BF16 else np.uint8(0x7F)
        for b in range(batch):
            ctx = int(seq_lens[b])
            if ctx % page_size:
                cache[bt[b, ctx // page_size], ctx % page_size:, :] = nan
        used = np.zeros(num_pages, bool)
        for b in range(batch):
            n = (int(seq_lens[b]) + page_size - 1) // page_size
            used[bt[b, :n]] = True
        cache[~used] = nan
    return Problem(q_bits=q_bits, cache=cache, kv_dtype=kv_dtype, kv_scale=kv_scale,
                   page_size=page_size, block_table=bt, seq_lens=seq_lens,
                   softmax_scale=float(softmax_scale), causal=bool(causal), name=name)


def ragged_lens(batch: int, lo: int = 21, hi: int = 131072, seed: int = 0) -> np.ndarray:
    """Context lengths drawn log-uniform in [lo, hi] (floor of exp(U[ln lo, ln hi]))."""
    u = _rng(seed, 11).random(batch)
    v = np.floor(np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))).astype(np.int64)
    return np.clip(v, lo, hi).astype(np.int32)


# Named workloads (the shapes of the pages' sweeps).
DENSE_BATCHES = (1, 3, 5, 16, 32, 64, 128, 256)
DENSE_CTXS = (21, 64, 256, 512, 1200, 3200, 5200, 8192, 23333)
FP8_LONG_CTXS = (4096, 32000, 65536, 109440)
MTP_SHAPES = ((64, 2), (32, 4), (16, 8), (16, 4))
MTP_PAGE_SIZES = (1, 16, 64)


def tiny(seed: int = 0, **kw) -> Problem:
    """B1 Sq1 H16 ctx64 page_size 1 bf16, no mask."""
    return make_problem(1, 1, 16, [64], 1, KV_BF16, False, seed, name="tiny_b1_h16_ctx64", **kw)


def dense(batch: int, ctx: int, seed: int = 0, **kw) -> Problem:
    """H128 Sq1 page_size 1 bf16, uniform context."""
    return make_problem(batch, 1, 128, [ctx] * batch, 1, KV_BF16, False, seed,
                        name=f"dense_h128_b{batch}_ctx{ctx}_ps1_bf16", **kw)


def fp8_long(ctx: int, batch: int = 8, seed: int = 0, **kw) -> Problem:
    """H16 Sq1 page_size 64 fp8-e4m3 cache with a per-tensor scale."""
    return make_problem(batch, 1, 16, [ctx] * batch, 64, KV_FP8_E4M3, False, seed,
                        name=f"fp8_h16_b{batch}_ctx{ctx}_ps64", **kw)


def mtp(heads: int, sq: int, page_size: int, batch: int = 32, ctx: int = 8192,
        seed: int = 0, **kw) -> Problem:
    """Causal MTP decode, bf16, 1% of cache rows scaled x8."""
    return make_problem(batch, sq, heads, [ctx] * batch, page_size, KV_BF16, True, seed,
                        outlier_frac=0.01, name=f"mtp_h{heads}_sq{sq}_b{batch}_ctx{ctx}_ps{page_size}",
                        **kw)


def ragged(kv_dtype: int = KV_BF16, batch: int = 64, seed: int = 0, **kw) -> Problem:
    """B64 H128 Sq1 page_size 16, log-uniform contexts in [21, 131072]."""
    lens = ragged_lens(batch, seed=seed)
    tag = "bf16" if kv_dtype == KV_BF16 else "fp8"
    return make_problem(batch, 1, 128, lens, 16, kv_dtype, False, seed,
                        name=f"ragged_h128_b{batch}_ps16_{tag}", **kw)
