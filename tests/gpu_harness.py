"""Runs a workloads.Step through the C ABI on the GPU and through the CPU
oracle, so the parity tests can compare the two. Both sides start from the
same seeded inputs and each writes the history into its own canary-filled
pools with its own cache write."""
from __future__ import annotations

import os

import numpy as np
import torch  # noqa: F401

from paged_sliding_window_gb300 import workloads as wl

# bar of the benchmark spec: |err| <= 2e-3 + 1e-2 |ref| elementwise
ATOL, RTOL = 2e-3, 1e-2


from paged_sliding_window_gb300.staging import GpuStep, dev_bf16, dev_i32, host_bits  # noqa: F401


class OracleStep:
    """Host pools with history and new rows written by the oracle."""

    def __init__(self, orc, step: wl.Step):
        self.orc, self.step = orc, step
        layer, c = step.layer, step.cache
        k0, v0 = c.empty_pools()
        k1, v1, st = orc.kv_cache_write(c.hist_k, c.hist_v, c.hist_cu, c.hist_past,
                                        step.block_table, k0, v0)
        assert st == 0
        self.k_pool, self.v_pool, st = orc.kv_cache_write(step.new_k, step.new_v, step.cu_new,
                                                          step.past_lens, step.block_table, k1, v1)
        assert st == 0

    def decode(self, seqs=None):
        out, lse, _ = self.orc.decode(self.step.layer.as_dict(), self.step.q, self.k_pool,
                                      self.v_pool, self.step.block_table, self.step.seq_lens,
                                      seqs=seqs)
        return out, lse

    def prefill(self, rows=None):
        out, lse, _ = self.orc.prefill(self.step.layer.as_dict(), self.step.q, self.step.cu_new,
                                       self.step.past_lens, self.k_pool, self.v_pool,
                                       self.step.block_table, rows=rows)
        return out, lse


# (test, what, elements, max |err|, max |err| / (atol + rtol |ref|)) of every
# comparison in this session; conftest prints them at the end of the run
PARITY_LOG: list = []


def assert_close(got: np.ndarray, ref: np.ndarray, what: str, atol=ATOL, rtol=RTOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    both_neg_inf = np.isneginf(got) & np.isneginf(ref)
    err = np.abs(got - ref)
    bad = ~((err <= atol + rtol * np.abs(ref)) | both_neg_inf)
    finite = ~both_neg_inf
    with np.errstate(invalid="ignore"):
        e = np.where(finite, err, 0.0)
        ratio = np.where(finite, err / (atol + rtol * np.abs(np.where(finite, ref, 0.0))), 0.0)
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    PARITY_LOG.append((test, what, int(got.size), float(np.nanmax(e)) if e.size else 0.0,
                       float(np.nanmax(ratio)) if ratio.size else 0.0))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside "
            f"{atol} + {rtol}|ref|; max err {np.nanmax(np.where(both_neg_inf, 0, err)):.3e}; "
            f"first {idx.tolist()} got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")
