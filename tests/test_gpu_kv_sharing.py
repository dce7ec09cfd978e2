"""KV sharing across layers on the GPU, over the 35-layer topology printed for
Gemma 4 E2B ("MNN supports the full Gemma4 family", KV-sharing section):
layers 0-14 own their caches, each of layers 15-34 reads the cache of layer
13 (sliding) or 14 (full), as psw_kv_share_map gives it.

A cache-owning layer runs the fused pre-attention step (norm, RoPE, cache
write) and then decode and chunked prefill on its own pools; a sharing layer
runs the fused step on q alone ("Gemma 4 model architecture analysis",
section 4.3: RoPE on q only, no cache write) and attends over its target's
pools. Every layer's outputs are compared with the oracle running the same
topology on its own pools, and the target pools must come out of the sharing
layers bit for bit unchanged. Scale 1/16 keeps the softmax away from near
ties, where a one-unit bf16 difference in the fused step's outputs could
move an attention output by more than the bar; the topology, not the
rounding, is what this test is about."""
import numpy as np
import pytest
import torch

from gpu_harness import assert_close, host_bits
from paged_sliding_window_gb300 import binding
from paged_sliding_window_gb300 import workloads as wl
from paged_sliding_window_gb300.staging import GpuStep, dev_bf16
from paged_sliding_window_gb300.workloads import Layer

pytestmark = pytest.mark.gpu

N_LAYERS, PATTERN, N_SHARED = 35, 5, 20
SLIDING = Layer(8, 1, 256, window=512, scale=1.0 / 16)
FULL = Layer(8, 1, 512, window=0, scale=1.0 / 16)
ROPE = {False: (1e4, 1.0), True: (1e6, 0.25)}  # (theta, rotated fraction) per layer type
EPS = 1e-6


def test_e2b_kv_sharing_topology():
    import oracle
    orc = oracle.default()
    is_full, target = binding.kv_share_map(N_LAYERS, PATTERN, N_SHARED)
    rng = np.random.default_rng(9)
    dec_lens = rng.integers(200, 3000, size=6)
    past = np.concatenate([dec_lens - 1, [100, 700]])
    new = np.concatenate([np.ones(6, np.int64), [64, 100]])
    nd = 6
    table, nb = wl.deal_block_table(rng, wl.pages_for(past + new))
    seeds = np.random.SeedSequence(77).spawn(N_LAYERS)
    steps = [wl.make_step(FULL if is_full[i] else SLIDING, seeds[i], table, nb, past, new,
                          False, False, threads=4) for i in range(N_LAYERS)]

    gpu_state, orc_pools, owner_bits = {}, {}, {}
    for i in range(N_LAYERS):
        st, layer = steps[i], steps[i].layer
        theta, factor = ROPE[is_full[i]]
        ra = int(factor * layer.head_dim / 2)
        owner = target[i] == i
        # ---- GPU
        if owner:
            g = GpuStep(st)  # this layer's pools, history written
            gpu_state[i] = g
        g_t = gpu_state[target[i]]
        rn = binding.make_norm_rope(theta, factor, EPS)
        q = dev_bf16(st.q)
        q_rot = torch.empty_like(q)
        if owner:
            binding.qkv_norm_rope_cache_write(layer, rn, q, dev_bf16(st.new_k),
                                              dev_bf16(st.new_v), g_t.cu_new, g_t.past,
                                              g_t.pages, q_rot, g_t.k_pool, g_t.v_pool)
        else:
            binding.qkv_norm_rope_cache_write(layer, rn, q, None, None, g_t.cu_new, g_t.past,
                                              None, q_rot, None, None)
        out = torch.full((q.shape[0], layer.n_q_heads, layer.head_dim), float("nan"),
                         device="cuda")
        lse = torch.full((q.shape[0], layer.n_q_heads), float("nan"), device="cuda")
        pages_dec = binding.make_pages(g_t.table[:nd].contiguous(), st.cache.num_blocks)
        binding.attn_decode_paged(layer, q_rot[:nd], g_t.k_pool, g_t.v_pool, pages_dec,
                                  g_t.seq_lens[:nd].contiguous(), out[:nd], lse[:nd], g_t.ws)
        row0 = int(st.cu_new[nd])
        pre_table = g_t.table[nd:].contiguous()
        binding.attn_prefill_chunked(layer, q_rot[row0:], (g_t.cu_new[nd:] - row0).contiguous(),
                                     g_t.past[nd:].contiguous(), int(new[nd:].max()),
                                     g_t.k_pool, g_t.v_pool,
                                     binding.make_pages(pre_table, st.cache.num_blocks),
                                     out[row0:], lse[row0:], g_t.ws)
        torch.cuda.synchronize()
        assert binding.get_error() == 0, f"layer {i}"
        if owner:
            owner_bits[i] = (host_bits(g_t.k_pool), host_bits(g_t.v_pool))
        # ---- oracle, same topology
        rq, rk, rv = orc.qkv_norm_rope(st.q, st.new_k if owner else None,
                                       st.new_v if owner else None, st.cu_new, st.past_lens,
                                       EPS, theta, ra)
        rq = orc.to_bf16(rq)
        if owner:
            c = st.cache
            kp, vp = c.empty_pools()
            orc.kv_cache_write(c.hist_k, c.hist_v, c.hist_cu, c.hist_past, table, kp, vp,
                               in_place=True)
            orc.kv_cache_write(orc.to_bf16(rk), orc.to_bf16(rv), st.cu_new, st.past_lens,
                               table, kp, vp, in_place=True)
            orc_pools[i] = (kp, vp)
        kp, vp = orc_pools[target[i]]
        L = layer.as_dict()
        ref_o, ref_l, _ = orc.decode(L, rq[:nd], kp, vp, table[:nd], st.seq_lens[:nd])
        assert_close(out[:nd].cpu().numpy(), ref_o, f"layer {i} decode out")
        assert_close(lse[:nd].cpu().numpy(), ref_l, f"layer {i} decode lse")
        rows = np.arange(row0, int(st.cu_new[-1]))
        ref_o, ref_l, _ = orc.prefill(L, rq, st.cu_new, st.past_lens, kp, vp, table, rows=rows)
        assert_close(out[row0:].cpu().numpy(), ref_o, f"layer {i} prefill out")
        assert_close(lse[row0:].cpu().numpy(), ref_l, f"layer {i} prefill lse")

    # the sharing layers wrote nothing into their targets' pools
    for src, (kb, vb) in owner_bits.items():
        g = gpu_state[src]
        assert np.array_equal(host_bits(g.k_pool), kb), f"layer {src} K pool changed"
        assert np.array_equal(host_bits(g.v_pool), vb), f"layer {src} V pool changed"
    # 15 layers own caches, 20 read layer 13 or 14
    assert sorted(gpu_state) == list(range(15))
    assert [target[i] for i in range(15, 35)] == [14 if is_full[i] else 13 for i in range(15, 35)]
