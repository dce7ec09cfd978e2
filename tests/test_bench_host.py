"""Host-side checks of the benchmark's end-to-end packing (no GPU needed):
every input of a decode step lands bit for bit in its piece of the packed
buffer, every piece starts 256 bytes into alignment, and the output pieces
cover out and lse."""
import types

import numpy as np
import torch

import bench
from paged_sliding_window_gb300 import binding
from paged_sliding_window_gb300 import workloads as wl


def test_packed_step_io_layout(monkeypatch):
    # pinned memory and the ABI's page descriptor need a GPU; their stand-ins
    # keep the tensors and record what would be passed
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)
    monkeypatch.setattr(binding, "make_pages", lambda t, nb: (t.data_ptr(), t.shape[1], nb))
    step = wl.custom_step(wl.Layer(16, 8, 256, window=1024), 7, [100, 3000, 17], [1, 1, 1])
    g = types.SimpleNamespace(out=torch.empty((3, 16, 256)), lse=torch.empty((3, 16)))
    h_in, d_in, h_out, d_out = bench.packed_step_io(step, g, device="cpu")
    d_in.copy_(h_in)

    def bits(t):
        return t.view(torch.int16).numpy().view(np.uint16)

    assert np.array_equal(bits(g.q), step.q)
    assert np.array_equal(bits(g.new_k), step.new_k)
    assert np.array_equal(bits(g.new_v), step.new_v)
    assert np.array_equal(g.cu_new.numpy(), step.cu_new)
    assert np.array_equal(g.past.numpy(), step.past_lens)
    assert np.array_equal(g.seq_lens.numpy(), step.seq_lens)
    assert np.array_equal(g.table.numpy(), step.block_table)
    assert g.pages[1:] == (step.block_table.shape[1], step.cache.num_blocks)
    for t in (g.q, g.new_k, g.new_v, g.cu_new, g.past, g.seq_lens, g.table):
        assert (t.data_ptr() - d_in.data_ptr()) % 256 == 0 and t.is_contiguous()
    expect_in = sum((a.nbytes + 255) // 256 * 256 for a in (
        step.q, step.new_k, step.new_v, step.cu_new.astype(np.int32),
        step.past_lens.astype(np.int32), step.seq_lens.astype(np.int32),
        step.block_table.astype(np.int32)))
    assert h_in.numel() == expect_in
    assert g.out.shape == (3, 16, 256) and g.lse.shape == (3, 16)
    g.out.fill_(1.5)
    g.lse.fill_(-2.0)
    h_out.copy_(d_out)
    raw = h_out.numpy()
    n_out = g.out.numel() * 4
    assert np.all(raw[:n_out].view(np.float32) == 1.5)
    lse_off = (g.lse.data_ptr() - d_out.data_ptr())
    assert np.all(raw[lse_off:lse_off + g.lse.numel() * 4].view(np.float32) == -2.0)
