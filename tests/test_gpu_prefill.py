"""Chunked-prefill parity on the GPU: kv_cache_write of the chunk then
attn_prefill_chunked through the C ABI, against the fp64 oracle. Pools are
compared bit for bit; outputs within 2e-3 + 1e-2 |ref|."""
import numpy as np
import pytest
import torch

from gpu_harness import GpuStep, OracleStep, assert_close, host_bits
from paged_sliding_window_gb300 import binding
from paged_sliding_window_gb300 import workloads as wl
from paged_sliding_window_gb300.workloads import Layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.default()


def sample_rows(step, every=7, edge=64):
    """First and last `edge` rows of each chunk, every `every`-th row, and the
    rows around the window boundary of each chunk."""
    rows = set()
    W = step.layer.window
    for b in range(step.n_seqs):
        lo, hi = int(step.cu_new[b]), int(step.cu_new[b + 1])
        n = hi - lo
        rows.update(range(lo, min(hi, lo + edge)))
        rows.update(range(max(lo, hi - edge), hi))
        rows.update(range(lo, hi, every))
        if W > 0:
            past = int(step.past_lens[b])
            for i in (W - past - 2, W - past - 1, W - past, W - past + 1):
                if 0 <= i < n:
                    rows.add(lo + i)
    return np.array(sorted(rows), dtype=np.int64)


def run_prefill(orc, step, rows=None, check_pools=True):
    g = GpuStep(step)
    g.write_new()
    g.prefill()
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    o = OracleStep(orc, step)
    if check_pools:
        assert np.array_equal(host_bits(g.k_pool), o.k_pool), "K pool differs from the oracle"
        if g.v_pool is not None:
            assert np.array_equal(host_bits(g.v_pool), o.v_pool), "V pool differs from the oracle"
    ref_out, ref_lse = o.prefill(rows)
    got_out = g.out.cpu().numpy()
    got_lse = g.lse.cpu().numpy()
    if rows is not None:
        got_out, got_lse = got_out[rows], got_lse[rows]
    assert_close(got_out, ref_out, "prefill out")
    assert_close(got_lse, ref_lse, "prefill lse")
    return g


def test_chunked_prefill_softcap_full_size(orc):
    """Every row of the chunked-prefill workload (8 chunks of 512 tokens after
    0-8192 cached ones, window 1024, softcap 50) against the oracle."""
    step = wl.chunked_prefill().steps[0]
    g = run_prefill(orc, step)
    assert torch.isfinite(g.out).all() and torch.isfinite(g.lse).all()
    assert not g.ws[:binding.WORKSPACE_COUNTER_BYTES].any(), "counter block written"


PREFILL_CASES = [
    # layer, past lens, chunk lens
    pytest.param(Layer(8, 4, 256, window=64, softcap=50.0, scale=0.0625),
                 [0, 10, 63, 64, 65, 200, 1000], [1, 70, 64, 63, 129, 5, 300], id="hd256-g2-w64-cap"),
    pytest.param(Layer(16, 8, 256, window=1024), [0, 3000, 1020, 17], [700, 65, 9, 1024],
                 id="hd256-g2-w1024"),
    pytest.param(Layer(8, 8, 256, window=0), [0, 5, 130], [130, 33, 64], id="hd256-g1-full"),
    pytest.param(Layer(16, 2, 256, window=40, softcap=20.0), [0, 77, 500], [50, 33, 17],
                 id="hd256-g8-w40-cap"),
    pytest.param(Layer(32, 2, 256, window=0, scale=0.3), [0, 12], [40, 9], id="hd256-g16-full"),
    pytest.param(Layer(32, 4, 512, window=0, k_eq_v=True), [0, 100, 1500], [48, 17, 200],
                 id="hd512-g8-keqv"),
    pytest.param(Layer(8, 2, 512, window=48), [0, 30, 400], [100, 3, 60], id="hd512-g4-w48"),
    pytest.param(Layer(16, 2, 512, window=100, k_eq_v=True, softcap=30.0), [0, 300, 1000],
                 [130, 64, 70], id="hd512-g8-w100-keqv-cap"),
    pytest.param(Layer(4, 4, 256, window=0, k_eq_v=True), [0, 31], [31, 66], id="hd256-g1-keqv"),
    pytest.param(Layer(12, 4, 256, window=33), [0, 50], [45, 20], id="hd256-g3-w33"),
    # empty chunks between (and after) non-empty ones: cu_q[b + 1] == cu_q[b]
    pytest.param(Layer(8, 4, 256, window=64, softcap=50.0, scale=0.0625),
                 [100, 40, 0, 300, 7], [70, 0, 65, 0, 0], id="hd256-g2-empty-chunks"),
    pytest.param(Layer(32, 4, 512, window=0, k_eq_v=True), [0, 500, 33], [0, 40, 129],
                 id="hd512-g8-keqv-empty-first"),
]


@pytest.mark.parametrize("layer,past,chunks", PREFILL_CASES)
def test_prefill_edge_cases(orc, layer, past, chunks):
    step = wl.custom_step(layer, 31, past, chunks)
    run_prefill(orc, step)


def test_prefill_last_row_matches_decode():
    """Row i of a chunk and a decode at seq_len = past + i + 1 see the same keys
    (the decode tail rule equals the band rule); the two kernels agree."""
    layer = Layer(16, 8, 256, window=256, softcap=30.0)
    past, chunk = np.array([700, 40, 300]), np.array([64, 100, 1])
    step = wl.custom_step(layer, 41, past, chunk)
    g = GpuStep(step)
    g.write_new()
    g.prefill()
    last = step.cu_new[1:] - 1
    q_last = g.q[torch.from_numpy(last.astype(np.int64)).cuda()].contiguous()
    out = torch.empty((3, 16, 256), dtype=torch.float32, device="cuda")
    lse = torch.empty((3, 16), dtype=torch.float32, device="cuda")
    seq_lens = torch.from_numpy((past + chunk).astype(np.int32)).cuda()
    binding.attn_decode_paged(layer, q_last, g.k_pool, g.v_pool, g.pages, seq_lens, out, lse,
                              g.ws)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    assert_close(out.cpu().numpy(), g.out[torch.from_numpy(last.astype(np.int64)).cuda()].cpu().numpy(),
                 "decode vs prefill last row")


def test_prefill_invalid_block_is_flagged():
    layer = Layer(8, 4, 256, window=64)
    step = wl.custom_step(layer, 51, [100, 20], [40, 40])
    g = GpuStep(step)
    g.write_new()
    assert binding.get_error() == 0
    bad = g.table.clone()
    bad[0, 7] = step.cache.num_blocks + 1
    g.pages = binding.make_pages(bad, step.cache.num_blocks)
    g.prefill()
    assert binding.get_error() & binding.DEVERR_BLOCK_ID


def _crafted_scores(step, row, key_pos_to_dim0):
    """Query `row`, head 0 = 16 e_0 (RMS 1) and keys of KV head 0 = c e_0, so
    that the scale-1 score of key j is 16 c_j exactly (all values bf16)."""
    q = np.zeros(step.layer.head_dim, np.float32)
    q[0] = 16.0
    step.q[row, 0] = wl.f32_to_bf16_bits(q)
    past = int(step.past_lens[0])
    c = step.cache
    for j, cj in key_pos_to_dim0.items():
        k = np.zeros(step.layer.head_dim, np.float32)
        k[0] = cj
        bits = wl.f32_to_bf16_bits(k)
        if j >= past:
            step.new_k[int(step.cu_new[0]) + j - past, 0] = bits
        else:
            step.cache.hist_k[int(c.hist_cu[0]) + j - int(c.hist_past[0]), 0] = bits


def _low_first_then_growth():
    """Keys 0-63 score -100, keys 64-127 score -12, key 128 scores -10 and keys
    129-130 score -100 for the query at position 130: the row's maximum grows
    by about 130 (log2 units) in two steps, and the second step's tile carries
    90 % of the weight."""
    keys = {j: -6.25 for j in range(64)}
    keys.update({j: -0.75 for j in range(64, 128)})
    keys.update({128: -0.625, 129: -6.25, 130: -6.25})
    return keys


def test_prefill_rescale_after_low_first_maximum(orc):
    """A row whose first key tile holds only very low scores, then a tile far
    above them, then a slightly higher key: the running maximum is raised
    twice and the earlier tiles must keep their weight through the rescale."""
    layer = Layer(4, 4, 256, window=0, scale=1.0)
    step = wl.custom_step(layer, 61, [0], [192])
    _crafted_scores(step, 130, _low_first_then_growth())
    run_prefill(orc, step)


def test_decode_rescale_after_low_first_maximum(orc):
    """The same scores seen by a decode query at position 130."""
    layer = Layer(4, 4, 256, window=0, scale=1.0)
    step = wl.custom_step(layer, 62, [130], [1])
    _crafted_scores(step, 0, _low_first_then_growth())
    g = GpuStep(step)
    g.write_new()
    g.decode()
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    ref_out, ref_lse = OracleStep(orc, step).decode()
    assert_close(g.out.cpu().numpy(), ref_out, "decode out")
    assert_close(g.lse.cpu().numpy(), ref_lse, "decode lse")


def test_prefill_without_lse(orc):
    """lse = NULL: the output alone is written, identical to a call with lse."""
    layer = Layer(16, 2, 512, window=100, k_eq_v=True, softcap=30.0)
    step = wl.custom_step(layer, 71, [0, 300, 1000], [130, 64, 70])
    g = GpuStep(step)
    g.write_new()
    g.prefill()
    with_lse = g.out.clone()
    out = torch.full_like(g.out, float("nan"))
    max_q = int(step.new_lens.max())
    binding.attn_prefill_chunked(layer, g.q, g.cu_new, g.past, max_q, g.k_pool, g.v_pool,
                                 g.pages, out, None, g.ws)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    assert torch.equal(out, with_lse)
    ref_out, _ = OracleStep(orc, step).prefill()
    assert_close(out.cpu().numpy(), ref_out, "prefill out (lse NULL)")
