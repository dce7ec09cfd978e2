"""Runs a workloads.Step through the C ABI on the GPU and through the CPU
oracle, so the parity tests can compare the two. Both sides start from the
same seeded inputs and each writes the history into its own canary-filled
pools with its own cache write."""
from __future__ import annotations

import os

import numpy as np
import torch

from paged_sliding_window_gb300 import binding

from paged_sliding_window_gb300 import workloads as wl

# the parity bar for bf16 inputs with fp32 accumulation: |err| <= 2e-3 + 1e-2 |ref|,
# elementwise
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


# --------------------------------------------------------------- pre-attention step
def _ordered(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def bf16_values(bits) -> np.ndarray:
    return wl.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


def assert_norm_rope_close(got_bits, exact, pre, rotated: bool, what: str):
    """Bar of the fused pre-attention step, from its arithmetic: the kernel
    forms each result in fp32, y = x / rms * w to about 2^-21 relative (its
    reciprocal square root is good to about 2^-22) and
    out = y_d cos - y_partner sin from cos and sin good to 2^-22, so before its
    single rounding to bf16 it is within 2^-20 (|y_d| + |y_partner|) of the
    exact value; the rounding adds at most half a bf16 unit of the result.
    `exact` is the oracle's fp64 result, `pre` its normalised values before
    the rotation (partner = the other dim of the rotation pair). A
    cancelling rotation can leave a result far smaller than its terms, so a
    bar of whole bf16 units of the result would be wrong there."""
    got = bf16_values(got_bits)
    exact = np.asarray(exact, dtype=np.float64)
    pre = np.asarray(pre, dtype=np.float64)
    hd = exact.shape[-1]
    partner = np.roll(pre, hd // 2, axis=-1) if rotated else np.zeros_like(pre)
    mag = np.abs(exact)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    half_unit = np.where(mag > 0, np.exp2(np.maximum(e, -126.0) - 8.0), 2.0 ** -134)
    bound = half_unit + 2.0 ** -20 * (np.abs(pre) + np.abs(partner))
    err = np.abs(got - exact)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} beyond the bar; "
                           f"worst err/bar {float(np.max(err / bound)):.3f}")


def _weights(rng, hd, spread):
    return None if spread is None else (1.0 + spread * rng.standard_normal(hd)).astype(np.float32)


class NormRopeCase:
    """Raw (un-normalised) projections of one step plus history, run on the
    GPU through the fused step and on the CPU through the oracle."""

    def __init__(self, orc, layer, past, new, seed, theta, factor, eps=1e-6, w_spread=0.1,
                 v_weight=False, v_from_k=False, scale_raw=3.0):
        self.layer, self.theta, self.factor, self.eps = layer, theta, factor, eps
        self.step = wl.custom_step(layer, seed, past, new, q_rms=False, kv_rms=False, threads=8)
        st = self.step
        hd = layer.head_dim
        rng = np.random.default_rng(seed)
        # raw projections: plain N(0, 1) scaled, so the norm has work to do
        self.q_raw = wl.f32_to_bf16_bits(wl.bf16_bits_to_f32(st.q) * scale_raw)
        self.k_raw = wl.f32_to_bf16_bits(wl.bf16_bits_to_f32(st.new_k) * scale_raw)
        self.v_raw = None
        if not layer.k_eq_v:
            self.v_raw = self.k_raw if v_from_k else wl.f32_to_bf16_bits(
                wl.bf16_bits_to_f32(st.new_v) * scale_raw)
        self.qw, self.kw = _weights(rng, hd, w_spread), _weights(rng, hd, w_spread)
        self.vw = _weights(rng, hd, w_spread) if v_weight else None
        self.rope_angles = int(factor * hd / 2)
        self.orc = orc

    def oracle_exact(self, with_kv=True, rotate=True):
        """fp64 (q, k, v) rows; rotate=False gives the normalised rows before
        the rotation (all frequencies zero)."""
        return self.orc.qkv_norm_rope(
            self.q_raw, self.k_raw if with_kv else None, self.v_raw if with_kv else None,
            self.step.cu_new, self.step.past_lens, self.eps, self.theta,
            self.rope_angles if rotate else 0, q_w=self.qw, k_w=self.kw, v_w=self.vw)

    def oracle(self, with_kv=True):
        """The oracle's rows rounded to bf16 (what its cache write stores)."""
        to = self.orc.to_bf16
        qo, ko, vo = self.oracle_exact(with_kv)
        return to(qo), (None if ko is None else to(ko)), (None if vo is None else to(vo))

    def gpu(self, g, with_kv=True, q_out=None):
        dev = lambda w: None if w is None else torch.from_numpy(w).cuda()
        self._w = [dev(self.qw), dev(self.kw), dev(self.vw)]
        rn = binding.make_norm_rope(self.theta, self.factor, self.eps, *self._w)
        q = dev_bf16(self.q_raw)
        out = torch.empty_like(q) if q_out is None else q_out
        k = dev_bf16(self.k_raw) if with_kv else None
        v = dev_bf16(self.v_raw) if (with_kv and self.v_raw is not None) else None
        binding.qkv_norm_rope_cache_write(
            self.layer, rn, q, k, v, g.cu_new, g.past, g.pages if with_kv else None, out,
            g.k_pool if with_kv else None, g.v_pool if with_kv else None)
        return out


