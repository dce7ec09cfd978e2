"""attn_decode_paged_append: the decode step fused into one launch (each
sequence's new K/V row written at position seq_len - 1 and attended to in
the same pass). Pools must equal the oracle's cache write bit for bit and
the outputs the oracle's decode over those pools, within 2e-3 + 1e-2 |ref|;
the fused call must also give the same outputs, bit for bit, as
kv_cache_write followed by attn_decode_paged."""
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


def run_append(orc, step, seqs=None):
    g = GpuStep(step)
    g.decode_append()
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    o = OracleStep(orc, step)
    assert np.array_equal(host_bits(g.k_pool), o.k_pool), "K pool differs from the oracle"
    if g.v_pool is not None:
        assert np.array_equal(host_bits(g.v_pool), o.v_pool), "V pool differs from the oracle"
    ref_o, ref_l = o.decode(seqs)
    got_o, got_l = g.out.cpu().numpy(), g.lse.cpu().numpy()
    if seqs is not None:
        got_o, got_l = got_o[seqs], got_l[seqs]
    assert_close(got_o, ref_o, "append decode out")
    assert_close(got_l, ref_l, "append decode lse")
    # the two-call step on fresh pools gives the same bits
    g2 = GpuStep(step)
    g2.write_new()
    g2.decode()
    torch.cuda.synchronize()
    assert torch.equal(g2.out, g.out) and torch.equal(g2.lse, g.lse)
    return g


def test_append_sliding_decode_batch_full_size(orc):
    run_append(orc, wl.sliding_decode().steps[0])


def test_append_full_keqv_decode_full_size(orc):
    run_append(orc, wl.full_keqv_decode().steps[0])


EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 1000]


@pytest.mark.parametrize("layer", [
    pytest.param(Layer(16, 8, 256, window=64), id="hd256-g2-w64"),
    pytest.param(Layer(8, 8, 256, window=0, softcap=30.0, scale=0.0625), id="hd256-g1-cap"),
    pytest.param(Layer(32, 4, 512, window=0, k_eq_v=True), id="hd512-g8-keqv"),
    pytest.param(Layer(32, 2, 256, window=0), id="hd256-g16-two-query-chunks"),
    pytest.param(Layer(16, 2, 512, window=48), id="hd512-g8-w48"),
    pytest.param(Layer(4, 4, 256, window=0, k_eq_v=True), id="hd256-g1-keqv"),
])
def test_append_edge_lengths(orc, layer):
    lens = np.array(EDGE_LENS)
    run_append(orc, wl.custom_step(layer, 93, lens - 1, np.ones_like(lens)))


def test_append_with_empty_sequences(orc):
    """Sequences of length 0 between others: no write, a zero row."""
    layer = Layer(16, 8, 256, window=1024)
    step = wl.custom_step(layer, 94, [40, 0, 300], [1, 1, 1])
    g = GpuStep(step)
    lens = step.seq_lens.copy()
    lens[1] = 0
    g.seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    before = host_bits(g.k_pool)
    g.decode_append()
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    after = host_bits(g.k_pool)
    # only the two non-empty sequences' new slots changed
    changed = np.argwhere(np.any(before != after, axis=-1))
    assert len(np.unique(changed[:, :2], axis=0)) == 2
    assert not g.out[1].any() and torch.isinf(g.lse[1]).all()
