"""The bounded pipeline waits, made to run out on purpose in the allowed way:
through the library's testing hook, the TMA producer of one CTA leaves one
tile copy unissued, so the consumer's wait for it has nothing that will ever
complete it. The wait must give up after its bound (about a second), the call
must come back with PSW_DEVERR_PIPELINE in the device error word, and the
context must stay usable: the next call on the same buffers, with the hook
off, matches the oracle. For the prefill kernel this also shows that the
CTA freed its tensor memory (the next launch allocates it again) and drained
its copies before exiting."""
import time

import numpy as np
import pytest
import torch

from gpu_harness import GpuStep, OracleStep, assert_close
from paged_sliding_window_gb300 import binding
from paged_sliding_window_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.default()


@pytest.fixture(autouse=True)
def hook_off():
    binding.testing_stall(binding.STALL_OFF)
    yield
    binding.testing_stall(binding.STALL_OFF)


def test_decode_wait_runs_out_and_the_next_call_is_exact(orc):
    step = wl.sliding_decode().steps[0]  # 27 tiles per CTA: CTA 0 reaches copy 2
    g = GpuStep(step)
    g.write_new()
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    binding.testing_stall(binding.STALL_DECODE, 0, 2)
    t0 = time.time()
    g.decode()
    err = binding.get_error()
    elapsed = time.time() - t0
    binding.testing_stall(binding.STALL_OFF)
    assert err & binding.DEVERR_PIPELINE, err
    assert 0.3 < elapsed < 30, elapsed  # the wait's bound, not a hang nor an instant return
    # same buffers, hook off: the counter block is zeroed as documented
    g.ws[:binding.WORKSPACE_COUNTER_BYTES].zero_()
    g.out.fill_(float("nan"))
    g.lse.fill_(float("nan"))
    g.decode()
    assert binding.get_error() == 0
    seqs = np.arange(0, step.n_seqs, 3)
    ref_o, ref_l = OracleStep(orc, step).decode(seqs)
    assert_close(g.out.cpu().numpy()[seqs], ref_o, "decode after a stalled call")
    assert_close(g.lse.cpu().numpy()[seqs], ref_l, "decode lse after a stalled call")


def test_prefill_wait_runs_out_and_the_next_call_is_exact(orc):
    step = wl.chunked_prefill().steps[0]
    g = GpuStep(step)
    g.write_new()
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    binding.testing_stall(binding.STALL_PREFILL, 0, 1)
    t0 = time.time()
    g.prefill()
    err = binding.get_error()
    elapsed = time.time() - t0
    binding.testing_stall(binding.STALL_OFF)
    assert err & binding.DEVERR_PIPELINE, err
    assert 0.3 < elapsed < 30, elapsed
    g.out.fill_(float("nan"))
    g.lse.fill_(float("nan"))
    g.prefill()  # allocates tensor memory on every SM again
    assert binding.get_error() == 0
    rows = np.arange(0, int(step.cu_new[-1]), 37)
    ref_o, ref_l = OracleStep(orc, step).prefill(rows)
    assert_close(g.out.cpu().numpy()[rows], ref_o, "prefill after a stalled call")
    assert_close(g.lse.cpu().numpy()[rows], ref_l, "prefill lse after a stalled call")
