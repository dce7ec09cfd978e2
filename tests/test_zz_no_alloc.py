"""attn_decode_paged_noalloc: decode for callers that cannot allocate device
memory (their memory belongs to another allocator with a fixed budget, or
they must not call cudaMalloc once serving has started). The entry point
takes its scratch from a static buffer inside the library instead of a
caller workspace.

Checked through the C ABI on several calls in a row, each against
attn_decode_paged on the same inputs (bit for bit: both run the same kernels
in the same order, so any leftover in the shared buffer would show) and
against the fp64 oracle (the stated tolerance): a sliding-layer batch, a
full-layer k_eq_v batch, and the sliding batch again with fewer sequences
after the larger one. A child process checks the one-time set-up under both
CUDA module-loading modes. Runs last, so a failure here never hides another
test's result, and works alone in a fresh process too."""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

from gpu_harness import GpuStep, OracleStep, assert_close
from paged_sliding_window_gb300 import binding
from paged_sliding_window_gb300 import workloads as wl
from paged_sliding_window_gb300.workloads import Layer

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _steps():
    sliding = Layer(16, 8, 256, window=1024)
    return [
        wl.custom_step(sliding, 21, [3000, 17, 900, 64, 1500, 5000, 2047, 1],
                       [1] * 8, threads=8),
        wl.custom_step(Layer(32, 4, 512, window=0, k_eq_v=True), 22, [5000, 40, 2047],
                       [1, 1, 1], threads=8),
        wl.custom_step(sliding, 23, [700, 2], [1, 1], threads=8),
    ]


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_and_oracle():
    import oracle
    orc = oracle.default()
    for step in _steps():
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
        assert torch.equal(out, ref_out), "no-alloc output differs from attn_decode_paged"
        assert torch.equal(lse, ref_lse), "no-alloc lse differs from attn_decode_paged"
        o_out, o_lse = OracleStep(orc, step).decode()
        assert_close(out.cpu().numpy(), o_out, "no-alloc decode out")
        assert_close(lse.cpu().numpy(), o_lse, "no-alloc decode lse")


@pytest.mark.gpu
def test_noalloc_rejects_batches_beyond_the_static_buffer():
    layer = binding.make_layer(Layer(16, 8, 256, window=1024))
    too_many = 4096  # 4096 * 8 units need far more than the static buffer holds
    assert binding.workspace_bytes(Layer(16, 8, 256, window=1024), too_many, 1) > \
        16 * 1024 * 1024
    fake = 0x10000  # aligned, non-null: only the size check can fail
    pages = binding.PswPages(fake, 4, 1024)
    rc = binding.load().attn_decode_paged_noalloc(
        ctypes.byref(layer), fake, fake, fake, ctypes.byref(pages), fake, too_many, fake, None,
        None)
    assert rc == -16  # PSW_ESCRATCH, returned before anything runs


_CHILD = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    import numpy as np, torch
    from paged_sliding_window_gb300 import binding
    from paged_sliding_window_gb300 import workloads as wl
    from paged_sliding_window_gb300.staging import GpuStep
    torch.cuda.set_device(0)
    step = wl.custom_step(wl.Layer(16, 8, 256, window=1024), 24, [4000, 33, 1200], [1, 1, 1],
                          threads=8)
    g = GpuStep(step)
    g.write_new()
    # set-up call at start-up: no sequences, valid pointers, nothing launched
    import ctypes
    rc = binding.load().attn_decode_paged_noalloc(
        ctypes.byref(binding.make_layer(step.layer)), g.q.data_ptr(), g.k_pool.data_ptr(),
        g.v_pool.data_ptr(), ctypes.byref(g.pages), g.seq_lens.data_ptr(), 0,
        g.out.data_ptr(), g.lse.data_ptr(), None)
    assert rc == 0, rc
    g.decode()
    out = torch.full_like(g.out, float("nan"))
    lse = torch.full_like(g.lse, float("nan"))
    for _ in range(2):
        binding.attn_decode_paged_noalloc(step.layer, g.q, g.k_pool, g.v_pool, g.pages,
                                          g.seq_lens, out, lse)
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        assert torch.equal(out, g.out) and torch.equal(lse, g.lse)
    print("child ok")
""")


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["LAZY", "EAGER"])
def test_noalloc_setup_call_in_a_fresh_process(mode):
    """A fresh process under either module-loading mode: the set-up call
    (n_seqs = 0) finds the buffer, later calls match attn_decode_paged."""
    env = dict(os.environ, CUDA_MODULE_LOADING=mode)
    res = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT)], env=env,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0 and "child ok" in res.stdout, res.stdout + res.stderr
