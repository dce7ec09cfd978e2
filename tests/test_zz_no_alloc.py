"""attn_decode_paged_noalloc: decode for callers that cannot allocate device
memory (their memory belongs to another allocator with a fixed budget, or
they must not call cudaMalloc once serving has started). The entry point
takes its scratch from a static buffer inside the library instead of a
caller workspace.

Checked through the C ABI against attn_decode_paged on the same inputs, within
the tolerance of the other parity tests, on two calls in a row with different
batches (the second call must not be affected by what the first left in the
shared buffer). Runs last so a failure here never hides another test's
result, and works alone in a fresh process too."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_harness import ATOL, RTOL, GpuStep
from paged_sliding_window_gb300 import binding
from paged_sliding_window_gb300 import workloads as wl
from paged_sliding_window_gb300.workloads import Layer


def _within(got: torch.Tensor, ref: torch.Tensor) -> bool:
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    both_inf = np.isneginf(g) & np.isneginf(r)
    return bool(np.all((np.abs(g - r) <= ATOL + RTOL * np.abs(r)) | both_inf))


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_twice():
    steps = [
        wl.custom_step(Layer(16, 8, 256, window=1024), 21, [3000, 17, 900, 64, 1500],
                       [1, 1, 1, 1, 1]),
        wl.custom_step(Layer(32, 4, 512, window=0, k_eq_v=True), 22, [5000, 40, 2047],
                       [1, 1, 1]),
    ]
    for step in steps:
        g = GpuStep(step)
        g.write_new()
        g.decode()
        ref_out, ref_lse = g.out.clone(), g.lse.clone()
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        binding.attn_decode_paged_noalloc(step.layer, g.q, g.k_pool, g.v_pool, g.pages,
                                          g.seq_lens, out, lse)
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        assert _within(out, ref_out), "no-alloc decode output differs from attn_decode_paged"
        assert _within(lse, ref_lse), "no-alloc decode lse differs from attn_decode_paged"


@pytest.mark.gpu
def test_noalloc_rejects_batches_beyond_the_static_buffer():
    layer = binding.make_layer(Layer(16, 8, 256, window=1024))
    too_many = 4096  # 4096 * 8 units need far more than the static buffer holds
    assert binding.workspace_bytes(Layer(16, 8, 256, window=1024), too_many, 1) > \
        16 * 1024 * 1024
    pages = binding.PswPages(0x10000, 4, 1024)
    rc = binding.load().attn_decode_paged_noalloc(
        ctypes.byref(layer), 0x10000, 0x10000, 0x10000, ctypes.byref(pages), 0x10000, too_many,
        0x10000, None, None)
    assert rc == -16  # PSW_ESCRATCH, returned before anything runs
