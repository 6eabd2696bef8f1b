"""Seeded synthetic inputs for GQA decode and for the K/V mean-pool conversion.

This module is the only code that both the CUDA path's tests/bench and the CPU
oracle use.  It holds none of the method's arithmetic: it draws random numbers,
rounds them to bf16 storage, and lays them out.  Everything downstream (the
oracle in ``oracle/`` and the CUDA library) receives the same bytes.

Workload shapes follow the pages' model settings:
  * T5-XXL with 64 heads and the G sweep of the group-count figure
    ("Grouped-query attention (GQA)" concept page, "Choosing the group count G",
    fig. 6);
  * Mistral 7B with 32 query heads and 8 K/V heads (same page, "Decoder-only
    models with GQA", arxiv:2310.06825 tab. 1);
  * a Llama-3-70B-shaped batch (64 query heads, 8 K/V heads; the explainer
    "Grouped-query attention" (whatisai.fyi), "Where it's used").
Head dims, batch sizes and cache lengths are the workload definitions of this
library's benchmark; the pages give no such numbers.  No dataset or checkpoint
is involved: every value is drawn i.i.d. N(0, 1) from a fixed seed.

Recipe (also stated in the design notes):
  * seeds: ``SeedSequence(20230522 + config_id, spawn_key=(variant,)).spawn(5)``
    gives the streams for q, k, v, seq_lens and the outlier mask (PCG64);
  * values: ``standard_normal`` in float32, then rounded to bf16
    (round-to-nearest-even);
  * seq_lens: ``integers(lo, hi + 1)`` per sequence (inclusive), or fixed;
  * outliers (Llama shape): a Bernoulli(0.01) mask per (b, t) position; keys of
    every K/V head at that position are multiplied by 4 in float32 before the
    bf16 rounding (exact: a power-of-two scale);
  * cache positions t >= seq_lens[b] hold bf16 NaN when ``poison_tail`` is set
    (tests), zeros otherwise (bench).  They are never part of the result.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

BF16_QNAN = np.uint16(0x7FC0)

SEED_BASE = 20230522


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    """One GQA decode workload: B sequences, H query heads, G K/V heads."""

    name: str
    config_id: int
    B: int
    H: int
    G: int
    d: int
    Lmax: int
    seq_lo: int = 0
    seq_hi: int = 0
    fixed_seq: Optional[tuple] = None
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    variant: int = 0

    @property
    def n(self) -> int:
        """Query heads per group, H/G."""
        return self.H // self.G

    @property
    def scale(self) -> np.float32:
        """The score scale 1/sqrt(d) as the fp32 value both sides receive."""
        return np.float32(1.0 / math.sqrt(self.d))

    def with_G(self, G: int) -> "DecodeConfig":
        return dataclasses.replace(self, G=G, variant=G, name=f"{self.name}_G{G}")

    def with_(self, **kw) -> "DecodeConfig":
        return dataclasses.replace(self, **kw)


# The five workloads.  The sweep entry is expanded with .with_G(G).
TINY = DecodeConfig("tiny", 0, B=1, H=8, G=2, d=64, Lmax=128, seq_lo=128, seq_hi=128)
MISTRAL_7B = DecodeConfig("mistral7b", 1, B=16, H=32, G=8, d=128, Lmax=4096,
                          seq_lo=1024, seq_hi=4096)
T5XXL_SWEEP = DecodeConfig("t5xxl_sweep", 2, B=32, H=64, G=8, d=64, Lmax=2048,
                           seq_lo=2048, seq_hi=2048)
T5XXL_SWEEP_GS = (1, 2, 4, 8, 16, 32, 64)
LLAMA3_70B = DecodeConfig("llama3_70b", 3, B=64, H=64, G=8, d=128, Lmax=8192,
                          seq_lo=2048, seq_hi=8192, outlier_frac=0.01, outlier_scale=4.0)
LONG_RAGGED = DecodeConfig("long_ragged", 4, B=4, H=32, G=8, d=128, Lmax=131072,
                           fixed_seq=(131072, 65536, 8192, 1024))

CONFIGS = {c.name: c for c in (TINY, MISTRAL_7B, T5XXL_SWEEP, LLAMA3_70B, LONG_RAGGED)}

# Mean-pool conversion workload: a random fp32 K (or V) projection stored
# head-major [H, h, d_model] = [8, 64, 512], pooled to [G=2, 64, 512].
MEANPOOL_TINY = dict(H=8, G=2, h=64, d_model=512, config_id=0)
# Checkpoint-sized conversion: one K (or V) projection of T5-XXL, 64 heads of
# 64 over a 4096-wide model (64 MiB fp32), pooled to G groups (G = 8 in the
# GQA paper's main setting).
MEANPOOL_T5XXL = dict(H=64, G=8, h=64, d_model=4096, config_id=2)
# A whole checkpoint in one call: every K and V projection of a T5-XXL-shaped
# encoder-decoder (24 encoder layers with self-attention, 24 decoder layers with
# self- and cross-attention: 72 attention blocks x {K, V} = 144 projections of
# [64, 64, 4096]), as [outer = 144, H, h * d_model] fp32, 9.66 GB, pooled to G = 8.
MEANPOOL_T5XXL_CHECKPOINT = dict(H=64, G=8, h=64, d_model=4096, config_id=3, outer=144)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (storage conversion)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _streams(cfg: DecodeConfig):
    ss = np.random.SeedSequence(SEED_BASE + cfg.config_id, spawn_key=(cfg.variant,))
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(5)]


def draw_seq_lens(cfg: DecodeConfig) -> np.ndarray:
    """Per-sequence valid cache lengths, int32 [B]."""
    _, _, _, rs, _ = _streams(cfg)
    if cfg.fixed_seq is not None:
        s = np.asarray(cfg.fixed_seq, dtype=np.int64)
        assert s.shape == (cfg.B,)
    else:
        s = rs.integers(cfg.seq_lo, cfg.seq_hi + 1, size=cfg.B)
    return s.astype(np.int32)


@dataclasses.dataclass
class DecodeInputs:
    cfg: DecodeConfig
    q: np.ndarray          # uint16 bf16 bits [B, H, d]
    k: np.ndarray          # uint16 bf16 bits [B, G, Lmax, d]
    v: np.ndarray          # uint16 bf16 bits [B, G, Lmax, d]
    seq_lens: np.ndarray   # int32 [B]
    scale: np.float32

    @property
    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one decode step reads: sum_b seq_b * G * d * 2 B * 2."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.cfg.G * self.cfg.d * 2 * 2


def make_decode_inputs(cfg: DecodeConfig, poison_tail: bool = True,
                       seq_lens: Optional[Sequence[int]] = None) -> DecodeInputs:
    """Draw q, k, v and seq_lens for ``cfg``.

    Only the valid region t < seq_lens[b] is drawn, batch by batch, so the large
    caches cost time proportional to their valid bytes.  ``seq_lens`` overrides
    the drawn lengths (edge-case tests); it must lie in [0, Lmax].
    """
    qs, ks, vs, _, ms = _streams(cfg)
    B, H, G, d, L = cfg.B, cfg.H, cfg.G, cfg.d, cfg.Lmax
    if seq_lens is None:
        sl = draw_seq_lens(cfg)
    else:
        sl = np.asarray(seq_lens, dtype=np.int32)
        assert sl.shape == (B,) and sl.min(initial=0) >= 0 and sl.max(initial=0) <= L
    q = f32_to_bf16_bits(qs.standard_normal((B, H, d), dtype=np.float32))
    fill = BF16_QNAN if poison_tail else np.uint16(0)
    k = np.full((B, G, L, d), fill, dtype=np.uint16)
    v = np.full((B, G, L, d), fill, dtype=np.uint16)
    for b in range(B):
        t = int(sl[b])
        if t == 0:
            continue
        kb = ks.standard_normal((G, t, d), dtype=np.float32)
        if cfg.outlier_frac > 0.0:
            mask = ms.random(t) < cfg.outlier_frac
            kb[:, mask, :] *= np.float32(cfg.outlier_scale)
        k[b, :, :t, :] = f32_to_bf16_bits(kb)
        del kb
        v[b, :, :t, :] = f32_to_bf16_bits(vs.standard_normal((G, t, d), dtype=np.float32))
    return DecodeInputs(cfg, q, k, v, sl, cfg.scale)


def make_meanpool_input(H: int, G: int, h: int, d_model: int, config_id: int = 0,
                        outer: int = 1) -> np.ndarray:
    """A random fp32 projection, [outer, H, h * d_model] viewed as head-major.

    With outer == 1 this is the [H, h, d_model] head-major tensor of the tiny
    workload.  Values are N(0, 1) float32 (no bf16 rounding: the conversion runs
    in fp32).
    """
    ss = np.random.SeedSequence(SEED_BASE + config_id, spawn_key=(1000 + H * 131 + G,))
    rng = np.random.Generator(np.random.PCG64(ss))
    w = rng.standard_normal((outer, H, h * d_model), dtype=np.float32)
    return w if outer > 1 else w.reshape(H, h, d_model)


def make_paged_layout(inp: DecodeInputs, page_size: int, seed: int = 0, spare_pages: int = 0,
                      shuffle: bool = True):
    """The contiguous caches of ``inp`` laid out as a page pool, pages in random pool order.

    Returns (k_pages, v_pages, block_table): pools [num_pages, G, page_size, d]
    (uint16 bf16 bits) and the int32 table [B, ceil(Lmax / page_size)]: position
    t of sequence b is row t % page_size of page block_table[b, t // page_size].
    With ``shuffle=False`` the pages follow one another in sequence order.
    Each sequence gets the pages its length needs; entries past them are -1 and
    the ``spare_pages`` unused pages, like the rows past a length, hold bf16 NaN.
    This only moves data: it is an input layout, not part of the method.
    """
    cfg = inp.cfg
    B, G, L, d = inp.k.shape
    max_pages = -(-L // page_size)
    need = [-(-int(t) // page_size) for t in inp.seq_lens]
    num_pages = sum(need) + spare_pages
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(SEED_BASE + cfg.config_id,
                                                                      spawn_key=(2000 + page_size, seed))))
    order = rng.permutation(num_pages) if shuffle else np.arange(num_pages)
    kp = np.full((num_pages, G, page_size, d), BF16_QNAN, dtype=np.uint16)
    vp = np.full((num_pages, G, page_size, d), BF16_QNAN, dtype=np.uint16)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    nxt = 0
    for b in range(B):
        for p in range(need[b]):
            page = int(order[nxt])
            nxt += 1
            table[b, p] = page
            lo, hi = p * page_size, min((p + 1) * page_size, L)
            kp[page, :, :hi - lo] = inp.k[b, :, lo:hi]
            vp[page, :, :hi - lo] = inp.v[b, :, lo:hi]
    return kp, vp, table


def make_new_rows(cfg: DecodeConfig, seed: int = 0):
    """The new token's K and V rows [B, G, d] for a fused append (N(0,1) -> bf16)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(SEED_BASE + cfg.config_id,
                                                                      spawn_key=(3000, seed))))
    k = f32_to_bf16_bits(rng.standard_normal((cfg.B, cfg.G, cfg.d), dtype=np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((cfg.B, cfg.G, cfg.d), dtype=np.float32))
    return k, v
