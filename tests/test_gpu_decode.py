"""Decode parity on the GPU: kv_cache_write + attn_decode_paged through the C
ABI against the fp64 oracle, at the workloads' full sizes and on edge cases.
Pools are compared bit for bit, outputs within 2e-3 + 1e-2 |ref|."""
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


def run_decode(orc, step, seqs=None, check_pools=True, zero_lens=()):
    g = GpuStep(step)
    g.write_new()
    o = OracleStep(orc, step)
    seq_lens = step.seq_lens.copy()
    for i in zero_lens:
        seq_lens[i] = 0
    if zero_lens:
        g.seq_lens.copy_(torch.from_numpy(seq_lens).cuda())
    g.decode()
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    if check_pools:
        assert np.array_equal(host_bits(g.k_pool), o.k_pool), "K pool differs from the oracle"
        if g.v_pool is not None:
            assert np.array_equal(host_bits(g.v_pool), o.v_pool), "V pool differs from the oracle"
    ref_out, ref_lse, _ = orc.decode(step.layer.as_dict(), step.q, o.k_pool, o.v_pool,
                                     step.block_table, seq_lens, seqs=seqs)
    got_out = g.out.cpu().numpy()
    got_lse = g.lse.cpu().numpy()
    if seqs is not None:
        got_out, got_lse = got_out[seqs], got_lse[seqs]
    assert_close(got_out, ref_out, "decode out")
    assert_close(got_lse, ref_lse, "decode lse")
    return g


def test_tiny_paged_decode(orc):
    run_decode(orc, wl.tiny_decode().steps[0])


def test_sliding_decode_batch_full_size(orc):
    run_decode(orc, wl.sliding_decode().steps[0], check_pools=False)


def test_full_keqv_decode_full_size(orc):
    """Every sequence of the full-layer k_eq_v batch (32 sequences up to 32768
    keys, head_dim 512, V read from the K pages)."""
    g = run_decode(orc, wl.full_keqv_decode().steps[0], check_pools=False)
    assert torch.isfinite(g.out).all() and torch.isfinite(g.lse).all()
    assert not g.ws[:binding.WORKSPACE_COUNTER_BYTES].any(), "merge tickets left non-zero"


EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 47, 48, 49, 63, 64, 65, 79, 80, 81, 127, 128, 129,
             200, 1000]

EDGE_LAYERS = [
    pytest.param(Layer(16, 8, 256, window=64), id="hd256-g2-w64"),
    pytest.param(Layer(8, 8, 256, window=0, softcap=30.0, scale=0.0625), id="hd256-g1-full-cap"),
    pytest.param(Layer(32, 4, 512, window=0, k_eq_v=True), id="hd512-g8-keqv"),
    pytest.param(Layer(32, 2, 256, window=100, softcap=5.0), id="hd256-g16-w100-cap"),
    pytest.param(Layer(8, 2, 512, window=48), id="hd512-g4-w48"),
    pytest.param(Layer(4, 4, 256, window=0, k_eq_v=True, scale=0.5), id="hd256-g1-keqv"),
    pytest.param(Layer(12, 4, 256, window=33), id="hd256-g3-w33"),
    pytest.param(Layer(32, 4, 512, window=0, k_eq_v=True, softcap=30.0, scale=0.0625),
                 id="hd512-g8-keqv-cap"),
    pytest.param(Layer(16, 2, 512, window=200, softcap=20.0), id="hd512-g8-w200-cap"),
]


@pytest.mark.parametrize("layer", EDGE_LAYERS)
def test_decode_edge_lengths(orc, layer):
    lens = np.array(EDGE_LENS)
    step = wl.custom_step(layer, 7, lens - 1, np.ones_like(lens))
    run_decode(orc, step)


def test_decode_many_sequences_split_units(orc):
    """More tiles than CTAs: units are cut across CTAs and merged; the merge
    tickets are back at zero afterwards."""
    rng = np.random.default_rng(3)
    lens = rng.integers(1, 3000, size=300)
    step = wl.custom_step(Layer(16, 8, 256, window=1024), 11, lens - 1, np.ones_like(lens),
                          threads=8)
    g = run_decode(orc, step, check_pools=False)
    assert not g.ws[:binding.WORKSPACE_COUNTER_BYTES].any(), "merge tickets left non-zero"


def test_decode_workspace_reused_by_smaller_then_larger_batches(orc):
    """One zero-filled workspace serves calls of different batch sizes in a
    row (tickets left at zero by each call)."""
    layer = Layer(16, 8, 256, window=512, softcap=40.0)
    rng = np.random.default_rng(17)
    big = rng.integers(1, 2500, size=200)
    small = rng.integers(1, 6000, size=7)
    steps = [wl.custom_step(layer, 18 + i, lens - 1, np.ones_like(lens), threads=8)
             for i, lens in enumerate((big, small, big))]
    ws = binding.alloc_workspace(layer, 200, 6000)
    for step in steps:
        g = GpuStep(step)
        g.ws = ws
        g.write_new()
        g.decode()
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        o = OracleStep(orc, step)
        ref_out, ref_lse = o.decode()
        assert_close(g.out.cpu().numpy(), ref_out, "decode out")
        assert_close(g.lse.cpu().numpy(), ref_lse, "decode lse")
        assert not ws[:binding.WORKSPACE_COUNTER_BYTES].any(), "merge tickets left non-zero"


def test_decode_without_lse(orc):
    """lse = NULL: the output alone is written, identical to a call with lse."""
    step = wl.custom_step(Layer(32, 4, 512, window=0, k_eq_v=True), 19,
                          np.array([20000, 5, 700]), np.ones(3, np.int64), threads=8)
    g = GpuStep(step)
    g.write_new()
    g.decode()
    with_lse = g.out.clone()
    out = torch.full_like(g.out, float("nan"))
    binding.attn_decode_paged(step.layer, g.q, g.k_pool, g.v_pool, g.pages, g.seq_lens, out,
                              None, g.ws)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    assert torch.equal(out, with_lse)
    ref_out, _ = OracleStep(orc, step).decode()
    assert_close(out.cpu().numpy(), ref_out, "decode out (lse NULL)")


def test_decode_single_long_sequence(orc):
    """One unit spread over every CTA of the grid."""
    step = wl.custom_step(Layer(32, 4, 512, window=0, k_eq_v=True), 12, [40000], [1], threads=8)
    run_decode(orc, step, check_pools=False)


def test_decode_empty_sequence(orc):
    lens = np.array([5, 40, 17, 3])
    step = wl.custom_step(Layer(16, 8, 256, window=32), 13, lens - 1, np.ones_like(lens))
    g = run_decode(orc, step, zero_lens=(1,))
    assert torch.all(g.out[1] == 0) and torch.all(torch.isneginf(g.lse[1]))


def test_decode_deterministic_and_workspace_reuse(orc):
    step = wl.custom_step(Layer(16, 8, 256, window=1024), 14, [3000, 20, 700], [1, 1, 1])
    g = GpuStep(step)
    g.write_new()
    g.decode()
    first = g.out.clone()
    g.out.fill_(float("nan"))
    g.decode()
    torch.cuda.synchronize()
    assert torch.equal(first, g.out)


def test_device_error_block_id_is_flagged_not_fatal():
    layer = Layer(16, 8, 256, window=64)
    step = wl.custom_step(layer, 15, [100, 50], [1, 1])
    g = GpuStep(step)
    assert binding.get_error() == 0
    bad = g.table.clone()
    bad[0, 3] = step.cache.num_blocks + 5
    g.pages = binding.make_pages(bad, step.cache.num_blocks)
    g.decode()
    assert binding.get_error() & binding.DEVERR_BLOCK_ID
    g.write_new()  # seq 0 writes page 6 (valid), seq 1 page 3 (valid)
    assert binding.get_error() == 0
    bad[1, 3] = -7
    g.write_new()
    assert binding.get_error() & binding.DEVERR_BLOCK_ID
    torch.cuda.synchronize()


def test_device_error_capacity_is_flagged():
    layer = Layer(16, 8, 256, window=64)
    step = wl.custom_step(layer, 16, [100, 50], [1, 1])
    g = GpuStep(step)
    g.seq_lens[1] = 10_000  # longer than the table row
    g.decode()
    assert binding.get_error() & binding.DEVERR_CAPACITY
    g.seq_lens[1] = -3
    g.decode()
    assert binding.get_error() & binding.DEVERR_LENGTH
