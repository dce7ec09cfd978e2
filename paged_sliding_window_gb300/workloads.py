"""Seeded synthetic workloads for paged sliding-window attention.

This module only draws inputs: sequence lengths, block tables, query and
key/value rows, and the initial contents of the page pools. It holds none of
the attention arithmetic and no slot mapping; the CUDA library and the CPU
oracle both consume what it returns, each through its own cache-write and
attention code.

Input recipe (shared by the tests and the benchmark):

* Every random draw comes from numpy's PCG64, seeded per workload. Bulk
  normal draws are split into fixed chunks, each with a child stream of the
  workload's ``SeedSequence``; the values are the same for any thread count.
* Values are float32 N(0, 1). When the workload says "RMS-normalised", each
  head vector is divided by ``sqrt(mean(x^2) + 1e-6)`` (unit weight). Values
  are then rounded to bf16 with round-to-nearest-even and carried as uint16
  bit patterns.
* Lengths: "uniform in [a, b]" is integer-inclusive; "log-uniform" is
  ``floor(exp(U(ln a, ln b)))``; "lognormal, median m" is
  ``floor(exp(N(ln m, sigma)))`` clipped to ``[1, cap]``; "past up to X" is
  integer-uniform in ``[0, X]``.
* Block tables: each sequence owns ``ceil(total_len / 16)`` pages. Physical
  block ids are a seed-permuted list of the pool's ids dealt out in sequence
  order; unused table entries hold -1.
* Pools start filled with a NaN canary in every slot. Each side then writes
  the retained history (``hist_*``) into its own pools with its own cache
  write, so nothing about the page layout is computed here. A sliding layer
  retains only the positions its first query of the step can still see
  (``W - 1`` tokens before it); every other slot keeps the canary, so a read
  outside the visible range shows up as NaN.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16
# bf16 quiet NaN with a payload: never produced by rounding finite values.
CANARY_BF16 = np.uint16(0x7FD1)
_CHUNK = 1 << 22  # elements per child stream in bulk normal draws


@dataclass(frozen=True)
class Layer:
    """Per-layer attention parameters (mirrors psw_layer_t)."""
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    window: int = 0          # 0 = full attention
    softcap: float = 0.0     # 0 = off
    scale: float = 1.0
    k_eq_v: bool = False     # V aliases the K pages
    block_size: int = BLOCK_SIZE

    def as_dict(self) -> dict:
        return dict(n_q_heads=self.n_q_heads, n_kv_heads=self.n_kv_heads,
                    head_dim=self.head_dim, window=self.window, softcap=self.softcap,
                    scale=self.scale, k_eq_v=int(self.k_eq_v), block_size=self.block_size)


# --------------------------------------------------------------------------- #
# value generation
# --------------------------------------------------------------------------- #
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = ((u + rounding) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_f32(seedseq: np.random.SeedSequence, n: int, threads: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    n_chunks = max(1, math.ceil(n / _CHUNK))
    children = seedseq.spawn(n_chunks)

    def fill(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(children[i]))
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    if n_chunks == 1 or threads <= 1:
        for i in range(n_chunks):
            fill(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out


def normal_bf16(seedseq: np.random.SeedSequence, shape, rms_norm: bool,
                threads: int = 8) -> np.ndarray:
    """N(0,1) float32 of ``shape``, optionally RMS-normalised over the last axis,
    rounded to bf16 bits."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    x = _normal_f32(seedseq, n, threads).reshape(shape)
    if rms_norm and n > 0:
        ms = np.mean(np.square(x, dtype=np.float32), axis=-1, keepdims=True, dtype=np.float32)
        x = x / np.sqrt(ms + np.float32(1e-6), dtype=np.float32)
    return f32_to_bf16_bits(x)


# --------------------------------------------------------------------------- #
# lengths and block tables
# --------------------------------------------------------------------------- #
def uniform_int(rng, lo, hi, n):
    return rng.integers(lo, hi + 1, size=n).astype(np.int64)


def log_uniform_int(rng, lo, hi, n):
    return np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))).astype(np.int64)


def lognormal_int(rng, median, sigma, cap, n):
    v = np.floor(np.exp(rng.normal(math.log(median), sigma, size=n))).astype(np.int64)
    return np.clip(v, 1, cap)


def pages_for(total_len) -> np.ndarray:
    return (np.asarray(total_len, dtype=np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE


def deal_block_table(rng, pages_per_seq, num_blocks: int | None = None,
                     slack: float = 1.25):
    """Seed-permuted pool ids dealt out in sequence order. Returns
    (block_table int32 [n_seqs, max_pages] with -1 padding, num_blocks)."""
    pages_per_seq = np.asarray(pages_per_seq, dtype=np.int64)
    need = int(pages_per_seq.sum())
    if num_blocks is None:
        num_blocks = max(1, math.ceil(slack * need))
    if need > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need} pages")
    perm = rng.permutation(num_blocks).astype(np.int32)
    width = max(1, int(pages_per_seq.max()) if len(pages_per_seq) else 1)
    table = np.full((len(pages_per_seq), width), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages_per_seq):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, int(num_blocks)


def cu_from_lens(lens) -> np.ndarray:
    lens = np.asarray(lens, dtype=np.int64)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    return cu


# --------------------------------------------------------------------------- #
# workloads
# --------------------------------------------------------------------------- #
@dataclass
class Cache:
    """One layer's pools plus the history to write into them before the step."""
    layer: Layer
    num_blocks: int
    hist_k: np.ndarray          # [n_hist_total, n_kv, hd] bf16 bits
    hist_v: np.ndarray | None   # None when V aliases K
    hist_cu: np.ndarray         # int32 [n_seqs + 1]
    hist_past: np.ndarray       # int32 [n_seqs]: first history position per seq

    def empty_pools(self):
        """Canary-filled host pools [num_blocks, 16, n_kv, hd] (K, V or None)."""
        shape = (self.num_blocks, self.layer.block_size, self.layer.n_kv_heads,
                 self.layer.head_dim)
        k = np.full(shape, CANARY_BF16, dtype=np.uint16)
        v = None if self.layer.k_eq_v else np.full(shape, CANARY_BF16, dtype=np.uint16)
        return k, v

    @property
    def pool_shape(self):
        return (self.num_blocks, self.layer.block_size, self.layer.n_kv_heads,
                self.layer.head_dim)


@dataclass
class Step:
    """New tokens of one step for one layer: cache write, then attention.

    Decode sequences have ``new_lens == 1`` and query ``q`` at seq_len - 1;
    prefill sequences carry a chunk of ``new_lens[b]`` rows."""
    layer: Layer
    block_table: np.ndarray     # int32 [n_seqs, max_pages]
    past_lens: np.ndarray       # int32 [n_seqs]: tokens already cached
    new_lens: np.ndarray        # int32 [n_seqs]
    cu_new: np.ndarray          # int32 [n_seqs + 1]
    q: np.ndarray               # [n_new_total, n_q, hd] bf16 bits
    new_k: np.ndarray           # [n_new_total, n_kv, hd]
    new_v: np.ndarray | None
    cache: Cache

    @property
    def n_seqs(self) -> int:
        return int(self.past_lens.shape[0])

    @property
    def seq_lens(self) -> np.ndarray:
        return (self.past_lens.astype(np.int64) + self.new_lens).astype(np.int32)


@dataclass
class Workload:
    name: str
    seed: int
    kind: str                    # "decode", "prefill" or "mixed"
    steps: list = field(default_factory=list)       # per layer
    decode_seqs: int = 0         # mixed: first decode_seqs rows are decode
    notes: str = ""


def _retained_start(layer: Layer, first_query_pos: np.ndarray) -> np.ndarray:
    """First history position a sliding layer keeps (full layers keep all)."""
    if layer.window == 0:
        return np.zeros_like(first_query_pos)
    return np.maximum(0, first_query_pos - layer.window + 1)


def make_step(layer: Layer, seedseq: np.random.SeedSequence, block_table, num_blocks,
              past_lens, new_lens, q_rms: bool, kv_rms: bool, threads: int = 8) -> Step:
    past_lens = np.asarray(past_lens, dtype=np.int64)
    new_lens = np.asarray(new_lens, dtype=np.int64)
    s_q, s_hk, s_hv, s_nk, s_nv = seedseq.spawn(5)
    hist_lo = _retained_start(layer, past_lens)
    hist_lens = past_lens - hist_lo
    n_hist = int(hist_lens.sum())
    n_new = int(new_lens.sum())
    kv_shape = (layer.n_kv_heads, layer.head_dim)
    hist_k = normal_bf16(s_hk, (n_hist,) + kv_shape, kv_rms, threads)
    hist_v = None if layer.k_eq_v else normal_bf16(s_hv, (n_hist,) + kv_shape, kv_rms, threads)
    cache = Cache(layer=layer, num_blocks=int(num_blocks), hist_k=hist_k, hist_v=hist_v,
                  hist_cu=cu_from_lens(hist_lens), hist_past=hist_lo.astype(np.int32))
    q = normal_bf16(s_q, (n_new, layer.n_q_heads, layer.head_dim), q_rms, threads)
    new_k = normal_bf16(s_nk, (n_new,) + kv_shape, kv_rms, threads)
    new_v = None if layer.k_eq_v else normal_bf16(s_nv, (n_new,) + kv_shape, kv_rms, threads)
    return Step(layer=layer, block_table=np.ascontiguousarray(block_table, dtype=np.int32),
                past_lens=past_lens.astype(np.int32), new_lens=new_lens.astype(np.int32),
                cu_new=cu_from_lens(new_lens), q=q, new_k=new_k, new_v=new_v, cache=cache)


# Layers of the synthetic workloads ---------------------------------------- #
SLIDING_256 = Layer(n_q_heads=16, n_kv_heads=8, head_dim=256, window=1024)
FULL_512_KEQV = Layer(n_q_heads=32, n_kv_heads=4, head_dim=512, window=0, k_eq_v=True)


def tiny_decode(seed: int = 1, threads: int = 8) -> Workload:
    """1 sequence of 64 tokens, sliding hd256 4q/2kv W=32, 8 shuffled physical
    blocks, RMS-normalised bf16 inputs, scale 1.0, no softcap."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    layer = Layer(n_q_heads=4, n_kv_heads=2, head_dim=256, window=32)
    seq_lens = np.array([64])
    table, nb = deal_block_table(rng, pages_for(seq_lens), num_blocks=8)
    step = make_step(layer, ss.spawn(1)[0], table, nb, seq_lens - 1, np.ones(1, np.int64),
                     True, True, threads)
    return Workload("tiny paged decode", seed, "decode", [step])


def sliding_decode(seed: int = 2, threads: int = 8, n_seqs: int = 64) -> Workload:
    """64 sequences, lengths uniform in [512, 4096], hd256 16q/8kv W=1024,
    pool of 32768 blocks, RMS-normalised bf16 K/V and q, scale 1.0."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    seq_lens = uniform_int(rng, 512, 4096, n_seqs)
    table, nb = deal_block_table(rng, pages_for(seq_lens), num_blocks=32768)
    step = make_step(SLIDING_256, ss.spawn(1)[0], table, nb, seq_lens - 1,
                     np.ones(n_seqs, np.int64), True, True, threads)
    return Workload("sliding-layer decode batch", seed, "decode", [step])


def full_keqv_decode(seed: int = 3, threads: int = 8, n_seqs: int = 32) -> Workload:
    """32 sequences, lengths log-uniform in [1024, 32768], hd512 32q/4kv, V
    aliases the K pages, full causal attention, RMS-normalised bf16."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    seq_lens = log_uniform_int(rng, 1024, 32768, n_seqs)
    table, nb = deal_block_table(rng, pages_for(seq_lens))
    step = make_step(FULL_512_KEQV, ss.spawn(1)[0], table, nb, seq_lens - 1,
                     np.ones(n_seqs, np.int64), True, True, threads)
    return Workload("full-layer k_eq_v decode", seed, "decode", [step])


def chunked_prefill(seed: int = 4, threads: int = 8, n_seqs: int = 8,
                    chunk: int = 512) -> Workload:
    """8 sequences, past uniform in [0, 8192], chunk 512; sliding W=1024 hd256
    8q/4kv, softcap 50, scale 1/sqrt(256); plain N(0,1) bf16."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    past = uniform_int(rng, 0, 8192, n_seqs)
    new = np.full(n_seqs, chunk, dtype=np.int64)
    table, nb = deal_block_table(rng, pages_for(past + new))
    layer = Layer(n_q_heads=8, n_kv_heads=4, head_dim=256, window=1024, softcap=50.0,
                  scale=1.0 / 16.0)
    step = make_step(layer, ss.spawn(1)[0], table, nb, past, new, False, False, threads)
    return Workload("chunked prefill with softcap", seed, "prefill", [step])


def _mixed_lengths(rng, n_decode, n_prefill, sigma):
    dec_lens = lognormal_int(rng, 2048, sigma, 65536, n_decode)
    pre_past = uniform_int(rng, 0, 16384, n_prefill)
    return dec_lens, pre_past


def mixed_hybrid_lengths(seed: int = 5, n_decode: int = 256, n_prefill: int = 4,
                         sigma: float = 1.0):
    """(decode sequence lengths, prefill past lengths) of mixed_hybrid, without
    drawing any values."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    return _mixed_lengths(rng, n_decode, n_prefill, sigma)


def mixed_hybrid(seed: int = 5, threads: int = 8, n_decode: int = 256, n_prefill: int = 4,
                 chunk: int = 2048, sigma: float = 1.0) -> Workload:
    """6-layer hybrid stack in the 5:1 pattern (5 sliding hd256 W=1024 16q/8kv,
    then 1 full hd512 32q/4kv k_eq_v); 256 decode sequences with lognormal
    lengths (median 2048, sigma 1.0, cap 65536) plus 4 prefill chunks of 2048
    tokens with past uniform in [0, 16384]; scale 1.0, no softcap. All layers
    share one block table; each layer has its own pools and values."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    dec_lens, pre_past = _mixed_lengths(rng, n_decode, n_prefill, sigma)
    past = np.concatenate([dec_lens - 1, pre_past])
    new = np.concatenate([np.ones(n_decode, np.int64), np.full(n_prefill, chunk, np.int64)])
    table, nb = deal_block_table(rng, pages_for(past + new))
    layers = [SLIDING_256] * 5 + [FULL_512_KEQV]
    layer_seeds = ss.spawn(1)[0].spawn(len(layers))
    steps = [make_step(layer, layer_seeds[i], table, nb, past, new, True, True, threads)
             for i, layer in enumerate(layers)]
    return Workload("mixed hybrid step", seed, "mixed", steps, decode_seqs=n_decode)


def custom_step(layer: Layer, seed: int, past_lens, new_lens, num_blocks=None,
                q_rms: bool = True, kv_rms: bool = True, threads: int = 1) -> Step:
    """Small ad-hoc steps for tests (edge cases: ragged, empty, page boundaries)."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    past_lens = np.asarray(past_lens, dtype=np.int64)
    new_lens = np.asarray(new_lens, dtype=np.int64)
    table, nb = deal_block_table(rng, pages_for(past_lens + new_lens), num_blocks)
    return make_step(layer, ss.spawn(1)[0], table, nb, past_lens, new_lens, q_rms, kv_rms,
                     threads)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "sliding_decode": sliding_decode,
    "full_keqv_decode": full_keqv_decode,
    "chunked_prefill": chunked_prefill,
    "mixed_hybrid": mixed_hybrid,
}
