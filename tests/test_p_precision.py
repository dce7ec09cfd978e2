"""Why P enters PV as a bf16 high part plus a bf16 remainder (both GPU
kernels): with the scale 1.0 that follows QK-norm (P3 Gemma-3 item 1) the
softmax of head-normalised vectors is peaked, a few keys carry P close to 1,
and P rounded once to bf16 (relative error up to 2^-9) times |V| of a few
units breaks the absolute part of the bar, 2e-3. The same rows with the
high part and remainder, as the kernels form them (each part truncated to
bf16), stay far inside it. Plain numpy over the oracle's pools: fp64 scores,
the two ways of carrying P into PV, l from the unrounded P."""
import numpy as np

from paged_sliding_window_gb300 import workloads as wl
from paged_sliding_window_gb300.workloads import Layer

ATOL, RTOL = 2e-3, 1e-2


def bf16_rne(x):
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return (((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(np.float32)


def bf16_trunc(x):
    return (np.asarray(x, np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)


def worst_ratio(step, kp, vp, carry):
    L = step.layer
    G = L.n_q_heads // L.n_kv_heads
    q = wl.bf16_bits_to_f32(step.q).astype(np.float64)
    K = wl.bf16_bits_to_f32(kp).astype(np.float64).reshape(-1, L.n_kv_heads, L.head_dim)
    V = wl.bf16_bits_to_f32(vp).astype(np.float64).reshape(-1, L.n_kv_heads, L.head_dim)
    worst = 0.0
    for b in range(step.n_seqs):
        p = int(step.seq_lens[b]) - 1
        pos = np.arange(max(0, p - L.window + 1) if L.window else 0, p + 1)
        slot = step.block_table[b][pos // 16] * 16 + pos % 16
        for h in range(L.n_q_heads):
            g = h // G
            s = L.scale * (K[slot, g] @ q[b, h])
            e = np.exp(s - s.max())
            ref = e @ V[slot, g] / e.sum()
            e32 = e.astype(np.float32)
            got = carry(e32) @ V[slot, g] / e32.astype(np.float64).sum()
            worst = max(worst, float((np.abs(got - ref) / (ATOL + RTOL * np.abs(ref))).max()))
    return worst


def test_p_needs_its_remainder_at_scale_one():
    import oracle
    orc = oracle.default()
    # the sliding layer of the decode batch (W = 1024, scale 1.0), 16 sequences
    layer = Layer(16, 8, 256, window=1024, scale=1.0)
    lens = [1072, 809, 935, 1245, 1023, 633, 971, 917, 329, 271, 992, 665, 917, 587, 470, 380]
    step = wl.custom_step(layer, 102, lens, [1] * len(lens))
    c = step.cache
    k0, v0 = c.empty_pools()
    k1, v1, _ = orc.kv_cache_write(c.hist_k, c.hist_v, c.hist_cu, c.hist_past, step.block_table,
                                   k0, v0)
    kp, vp, _ = orc.kv_cache_write(step.new_k, step.new_v, step.cu_new, step.past_lens,
                                   step.block_table, k1, v1)

    def single(e32):
        return bf16_rne(e32).astype(np.float64)

    def hi_lo(e32):
        hi = bf16_trunc(e32)
        return hi.astype(np.float64) + bf16_trunc(e32 - hi)

    assert worst_ratio(step, kp, vp, single) > 1.0     # one bf16 rounding breaks the bar
    assert worst_ratio(step, kp, vp, hi_lo) < 0.05     # high part + remainder: far inside
