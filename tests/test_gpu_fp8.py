"""FP8 KV pages on the GPU (kv_cache_write_fp8, attn_decode_paged_fp8)
against the fp64 oracle of the same format: the cache write's codes and
scales bit for bit (both sides take each rounding decision in fp32, the
conversion to E4M3 rounding to nearest even), and decode over the
dequantised pages within 2e-3 + 1e-2 |ref| of the oracle's attention over the
same dequantised values."""
import numpy as np
import pytest
import torch

from gpu_harness import assert_close
from paged_sliding_window_gb300 import binding
from paged_sliding_window_gb300 import workloads as wl
from paged_sliding_window_gb300.staging import FP8_CANARY, GpuStepFP8
from paged_sliding_window_gb300.workloads import Layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.default()


def oracle_pools_fp8(orc, step):
    c = step.cache
    shape = c.pool_shape
    k8 = np.full(shape, FP8_CANARY, np.uint8)
    ks = np.full(shape[:3], np.nan, np.float32)
    v8 = None if step.layer.k_eq_v else np.full(shape, FP8_CANARY, np.uint8)
    vs = None if step.layer.k_eq_v else np.full(shape[:3], np.nan, np.float32)
    assert orc.kv_cache_write_fp8(c.hist_k, c.hist_v, c.hist_cu, c.hist_past, step.block_table,
                                  k8, v8, ks, vs) == 0
    assert orc.kv_cache_write_fp8(step.new_k, step.new_v, step.cu_new, step.past_lens,
                                  step.block_table, k8, v8, ks, vs) == 0
    return k8, v8, ks, vs


def _bits(t):
    return t.cpu().numpy().view(np.uint32) if t.dtype == torch.float32 else t.cpu().numpy()


def run_fp8(orc, step, check_pools=True, seqs=None):
    g = GpuStepFP8(step)
    g.write_new()
    g.decode()
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    k8, v8, ks, vs = oracle_pools_fp8(orc, step)
    if check_pools:
        assert np.array_equal(g.k_pool8.cpu().numpy(), k8), "K codes differ from the oracle"
        assert np.array_equal(_bits(g.k_scale), ks.view(np.uint32)), "K scales differ"
        if v8 is not None:
            assert np.array_equal(g.v_pool8.cpu().numpy(), v8), "V codes differ from the oracle"
            assert np.array_equal(_bits(g.v_scale), vs.view(np.uint32)), "V scales differ"
    ref_o, ref_l, _ = orc.decode_fp8(step.layer.as_dict(), step.q, k8, v8, ks, vs,
                                     step.block_table, step.seq_lens, seqs=seqs)
    got_o, got_l = g.out.cpu().numpy(), g.lse.cpu().numpy()
    if seqs is not None:
        got_o, got_l = got_o[seqs], got_l[seqs]
    assert_close(got_o, ref_o, "fp8 decode out")
    assert_close(got_l, ref_l, "fp8 decode lse")
    return g


def test_fp8_sliding_decode_batch_full_size(orc):
    """The sliding-layer decode batch on FP8 pages, every output."""
    run_fp8(orc, wl.sliding_decode().steps[0], check_pools=True)


def test_fp8_full_keqv_decode_full_size(orc):
    run_fp8(orc, wl.full_keqv_decode().steps[0], check_pools=False)


EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 200, 1000]


@pytest.mark.parametrize("layer", [
    pytest.param(Layer(16, 8, 256, window=64), id="hd256-g2-w64"),
    pytest.param(Layer(8, 8, 256, window=0, softcap=30.0, scale=0.0625), id="hd256-g1-cap"),
    pytest.param(Layer(32, 4, 512, window=0, k_eq_v=True), id="hd512-g8-keqv"),
    pytest.param(Layer(8, 2, 512, window=48), id="hd512-g4-w48"),
    pytest.param(Layer(4, 4, 256, window=0, k_eq_v=True, scale=0.5), id="hd256-g1-keqv"),
    pytest.param(Layer(16, 2, 512, window=200, softcap=20.0), id="hd512-g8-w200-cap"),
    pytest.param(Layer(32, 2, 256, window=0), id="hd256-g16-two-query-chunks"),
])
def test_fp8_decode_edge_lengths(orc, layer):
    lens = np.array(EDGE_LENS)
    run_fp8(orc, wl.custom_step(layer, 91, lens - 1, np.ones_like(lens)))


def test_fp8_cache_write_zero_rows_and_wide_range(orc):
    """All-zero rows (scale 0) and rows spanning many binades, through the
    cache write and the decode that reads them."""
    layer = Layer(8, 4, 256, window=0)
    step = wl.custom_step(layer, 92, [40, 7], [1, 1], kv_rms=False)
    rng = np.random.default_rng(3)

    def spread(rows):
        s = np.exp2(rng.uniform(-30, 30, rows.shape[:2] + (1,))).astype(np.float32)
        return wl.f32_to_bf16_bits(wl.bf16_bits_to_f32(rows) * s)

    c = step.cache
    c.hist_k, c.hist_v = spread(c.hist_k), spread(c.hist_v)
    step.new_k, step.new_v = spread(step.new_k), spread(step.new_v)
    step.new_v[1] = 0
    step.new_k[0, 1] = 0
    c.hist_k[5, 2] = 0
    run_fp8(orc, step)
