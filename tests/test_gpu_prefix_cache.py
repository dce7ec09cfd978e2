"""Prefix caching end to end: block-table rows come from the host page
allocator (psw_block_pool_admit / commit), a second request whose prompt
shares 48 tokens with the first gets the first request's three full pages
in its row and writes only its own tokens, and its chunked prefill over the
shared pages matches the oracle computing the same request alone on private
pages ("Gemma 4 model architecture analysis", section 6.6: a shared system
prompt's KV is computed once)."""
import numpy as np
import pytest
import torch

from gpu_harness import assert_close, host_bits
from paged_sliding_window_gb300 import binding
from paged_sliding_window_gb300 import workloads as wl
from paged_sliding_window_gb300.staging import dev_bf16, dev_i32
from paged_sliding_window_gb300.workloads import Layer

pytestmark = pytest.mark.gpu

LAYER = Layer(8, 4, 256, window=0)
MAX_BLOCKS = 8


def kv_rows(tokens, start):
    """K and V rows of tokens at positions start.. (a function of the token
    and its position only, so equal prefixes have equal rows)."""
    ks, vs = [], []
    for i, t in enumerate(tokens):
        ss = np.random.SeedSequence([int(t), start + i])
        ks.append(wl.normal_bf16(ss.spawn(1)[0], (LAYER.n_kv_heads, LAYER.head_dim), True, 1))
        vs.append(wl.normal_bf16(ss.spawn(2)[1], (LAYER.n_kv_heads, LAYER.head_dim), True, 1))
    return np.stack(ks), np.stack(vs)


def test_prefix_shared_pages_feed_the_prefill():
    import oracle
    orc = oracle.default()
    a = list(range(1000, 1078))
    b = a[:48] + list(range(5000, 5020))
    num_blocks = 32
    pool = binding.BlockPool(num_blocks)
    canary = int(wl.CANARY_BF16)
    shape = (num_blocks, 16, LAYER.n_kv_heads, LAYER.head_dim)
    k_pool = torch.full(shape, canary, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    v_pool = torch.full(shape, canary, dtype=torch.int16, device="cuda").view(torch.bfloat16)

    def write(tokens, row, past):
        k, v = kv_rows(tokens[past:], past)
        table = dev_i32(np.array([row], np.int32))
        binding.kv_cache_write(LAYER, dev_bf16(k), dev_bf16(v), dev_i32([0, len(tokens) - past]),
                               dev_i32([past]), binding.make_pages(table, num_blocks), k_pool,
                               v_pool)
        return table

    rc, row_a, cached_a = pool.admit(a, MAX_BLOCKS)
    assert rc == 0 and cached_a == 0
    write(a, row_a, 0)
    assert pool.commit(a, row_a) == 0
    before = host_bits(k_pool)
    rc, row_b, cached_b = pool.admit(b, MAX_BLOCKS)
    assert rc == 0 and cached_b == 48 and row_b[:3] == row_a[:3]
    assert all(pool.ref_count(x) == 2 for x in row_b[:3])
    table_b = write(b, row_b, cached_b)
    after = host_bits(k_pool)
    assert np.array_equal(after[row_a[:3]], before[row_a[:3]]), "a shared page was rewritten"

    n_new = len(b) - cached_b
    rng = np.random.default_rng(3)
    q = wl.f32_to_bf16_bits(rng.standard_normal((n_new, LAYER.n_q_heads, LAYER.head_dim))
                            .astype(np.float32))
    out = torch.empty((n_new, LAYER.n_q_heads, LAYER.head_dim), device="cuda")
    lse = torch.empty((n_new, LAYER.n_q_heads), device="cuda")
    ws = binding.alloc_workspace(LAYER, 1, len(b))
    binding.attn_prefill_chunked(LAYER, dev_bf16(q), dev_i32([0, n_new]), dev_i32([cached_b]),
                                 n_new, k_pool, v_pool, binding.make_pages(table_b, num_blocks),
                                 out, lse, ws)
    torch.cuda.synchronize()
    assert binding.get_error() == 0

    # oracle: request b alone, every row of its prompt on private pages
    k, v = kv_rows(b, 0)
    pages = (len(b) + 15) // 16
    table = np.arange(pages, dtype=np.int32)[None, :]
    kp = np.full((pages, 16, LAYER.n_kv_heads, LAYER.head_dim), wl.CANARY_BF16, np.uint16)
    vp = kp.copy()
    orc.kv_cache_write(k, v, [0, len(b)], [0], table, kp, vp, in_place=True)
    ref_o, ref_l, _ = orc.prefill(LAYER.as_dict(), q, [0, n_new], [cached_b], kp, vp, table)
    assert_close(out.cpu().numpy(), ref_o, "prefill over shared pages")
    assert_close(lse.cpu().numpy(), ref_l, "prefill lse over shared pages")
    # both requests done: every page back in the free queue
    assert pool.release([x for x in row_b if x >= 0][::-1]) == 0
    assert pool.release([x for x in row_a if x >= 0][::-1]) == 0
    assert pool.num_free() == num_blocks
