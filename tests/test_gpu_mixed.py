"""The mixed serving step over the 6-layer hybrid stack (5 sliding hd256
layers, then 1 full hd512 k_eq_v layer; 256 decode sequences plus 4 prefill
chunks of 2048 tokens): every layer runs kv_cache_write, attn_decode_paged and
attn_prefill_chunked through the C ABI. Outputs are compared with the oracle on
every decode row of every layer and on sampled prefill rows (all prefill rows
are about 4 TFLOP of fp64 work, too much for a CPU pass); every output is
checked finite."""
import numpy as np
import pytest
import torch

from gpu_harness import assert_close
from paged_sliding_window_gb300 import binding
from paged_sliding_window_gb300 import workloads as wl
from paged_sliding_window_gb300.staging import MixedLayerStep

pytestmark = pytest.mark.gpu


def prefill_sample(step, n_decode, every=97, edge=16):
    rows = set()
    W = step.layer.window
    for b in range(n_decode, step.n_seqs):
        lo, hi = int(step.cu_new[b]), int(step.cu_new[b + 1])
        rows.update(range(lo, lo + edge))
        rows.update(range(hi - edge, hi))
        rows.update(range(lo, hi, every))
        if W > 0:
            past = int(step.past_lens[b])
            for i in (W - past - 1, W - past):
                if 0 <= i < hi - lo:
                    rows.add(lo + i)
    return np.array(sorted(rows), dtype=np.int64)


def test_mixed_hybrid_step_all_layers():
    import oracle
    orc = oracle.default()
    work = wl.mixed_hybrid(threads=16)
    nd = work.decode_seqs
    for li, step in enumerate(work.steps):
        m = MixedLayerStep(step, nd)
        m.run()
        torch.cuda.synchronize()
        assert binding.get_error() == 0, f"layer {li}: device error"
        g = m.g
        assert torch.isfinite(g.out).all() and torch.isfinite(g.lse).all(), f"layer {li}"
        assert not g.ws[:binding.WORKSPACE_COUNTER_BYTES].any(), f"layer {li}: tickets"
        got_out = g.out.cpu().numpy()
        got_lse = g.lse.cpu().numpy()
        # oracle pools for this layer, written in place
        c = step.cache
        kp, vp = c.empty_pools()
        orc.kv_cache_write(c.hist_k, c.hist_v, c.hist_cu, c.hist_past, step.block_table, kp, vp,
                           in_place=True)
        orc.kv_cache_write(step.new_k, step.new_v, step.cu_new, step.past_lens,
                           step.block_table, kp, vp, in_place=True)
        L = step.layer.as_dict()
        lens = step.seq_lens[:nd]
        # every decode row of every layer (the full layer's rows reach 65536
        # keys: about 25 G multiply-adds of fp64 oracle work)
        seqs = list(range(nd))
        ref_o, ref_l, _ = orc.decode(L, step.q[:nd], kp, vp, step.block_table[:nd], lens,
                                     seqs=seqs)
        # decode rows are the first nd rows of q/out (one new token each)
        assert_close(got_out[seqs], ref_o, f"layer {li} decode out")
        assert_close(got_lse[seqs], ref_l, f"layer {li} decode lse")
        rows = prefill_sample(step, nd)
        ref_o, ref_l, _ = orc.prefill(L, step.q, step.cu_new, step.past_lens, kp, vp,
                                      step.block_table, rows=rows)
        assert_close(got_out[rows], ref_o, f"layer {li} prefill out")
        assert_close(got_lse[rows], ref_l, f"layer {li} prefill lse")
        del m, g, kp, vp
        torch.cuda.empty_cache()
