"""Pins of the oracle's pre-attention step (per-head RMS-norm of q, k and v,
then the proportional rotary embedding of q and k) and of its bf16 rounding,
against facts fixed outside the oracle:

* closed forms of RMS-norm: mean square of the output, scale invariance,
  the weight multiplying each dim;
* the defining property of a rotary embedding: the dot product of a rotated
  query and key depends only on their position difference, and each rotated
  pair keeps its length;
* position 0 is the identity; V is never rotated;
* the frequency rule printed in "Gemma 4 model architecture analysis",
  challenge 5: pair i turns by pos * theta^(-2i / head_size) for i below the
  rotated count and not at all beyond it (head size, not the rotated size, in
  the exponent's denominator), the pair being dims i and i + head_size / 2;
* bf16 rounding: exact values stay, ties go to even, everything else agrees
  with torch's float32 -> bfloat16 conversion on values that are exact in
  float32.
"""
from __future__ import annotations

import math

import numpy as np

from paged_sliding_window_gb300 import workloads as wl


def _bits(x):
    return wl.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _vec(seed, hd, scale=1.0):
    rng = np.random.default_rng(seed)
    return _bits(rng.standard_normal(hd).astype(np.float32) * scale)


def _f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def check_rms_norm_closed_form(orc):
    """Without rotation or weight, mean(y^2) = ms / (ms + eps) exactly."""
    for hd, eps in ((256, 1e-6), (512, 0.5)):
        x = _vec(11 + hd, hd, 3.0)
        y = orc.norm_rope_row(x, eps, rotate=False)
        ms = float(np.mean(_f64(x) ** 2))
        assert abs(float(np.mean(y * y)) - ms / (ms + eps)) < 1e-12
        # direction kept: y is a positive multiple of x
        r = y / _f64(x)
        assert np.all(np.abs(r - r[0]) < 1e-12) and r[0] > 0


def check_rms_norm_scale_invariant_and_weight(orc):
    x = _vec(21, 256)
    y1 = orc.norm_rope_row(x, 0.0, rotate=False)
    y2 = orc.norm_rope_row(_bits(_f64(x) * 8.0), 0.0, rotate=False)  # exact power of two
    assert np.max(np.abs(y1 - y2)) < 1e-12
    w = (np.arange(256) % 7 + 0.5).astype(np.float32)
    yw = orc.norm_rope_row(x, 0.0, weight=w, rotate=False)
    assert np.max(np.abs(yw - y1 * w.astype(np.float64))) < 1e-12


def check_rope_position_zero_is_identity(orc):
    x = _vec(31, 512)
    a = orc.norm_rope_row(x, 1e-6, rotate=True, theta=1e6, pos=0)
    b = orc.norm_rope_row(x, 1e-6, rotate=False)
    assert np.array_equal(a, b)


def check_rope_relative_position(orc):
    """<R_m q, R_n k> depends on m - n only (the rotary embedding's defining
    property), for full and partial rotation."""
    for hd, theta, ra in ((256, 1e4, 128), (512, 1e6, 64)):
        q, k = _vec(41, hd), _vec(42, hd)
        base = None
        for shift in (0, 7, 1000, 40000):
            qm = orc.norm_rope_row(q, 1e-6, theta=theta, rope_angles=ra, pos=90 + shift)
            kn = orc.norm_rope_row(k, 1e-6, theta=theta, rope_angles=ra, pos=17 + shift)
            d = float(np.dot(qm, kn))
            if base is None:
                base = d
            assert abs(d - base) < 1e-9 * max(1.0, abs(base)), (hd, shift, d, base)
        # and it does change with the difference itself
        q2 = orc.norm_rope_row(q, 1e-6, theta=theta, rope_angles=ra, pos=91)
        k2 = orc.norm_rope_row(k, 1e-6, theta=theta, rope_angles=ra, pos=17)
        assert abs(float(np.dot(q2, k2)) - base) > 1e-6


def check_rope_pairs_keep_length(orc):
    x = _vec(51, 512)
    y = orc.norm_rope_row(x, 1e-6, rotate=False)
    z = orc.norm_rope_row(x, 1e-6, theta=1e6, rope_angles=200, pos=12345)
    h = 256
    assert np.max(np.abs((z[:h] ** 2 + z[h:] ** 2) - (y[:h] ** 2 + y[h:] ** 2))) < 1e-12


def check_rope_frequency_rule(orc):
    """A vector whose only non-zero dims are i and i + hd/2 turns by
    pos * theta^(-2i/hd) when i < rope_angles and stays put otherwise."""
    for hd, theta, ra, pos in ((256, 1e4, 128, 33), (512, 1e6, 64, 5000), (512, 1e6, 64, 7)):
        h = hd // 2
        for i in (0, 1, 5, ra - 1, ra, h - 1):
            if i >= h:
                continue
            x = np.zeros(hd, np.float32)
            x[i], x[i + h] = 0.75, -1.25
            xb = _bits(x)
            z = orc.norm_rope_row(xb, 0.0, theta=theta, rope_angles=ra, pos=pos)
            y = orc.norm_rope_row(xb, 0.0, rotate=False)
            others = np.delete(np.arange(hd), [i, i + h])
            assert np.all(z[others] == 0.0)
            freq = theta ** (-2.0 * i / hd) if i < ra else 0.0
            want = (math.atan2(y[i + h], y[i]) + pos * freq) % (2 * math.pi)
            got = math.atan2(z[i + h], z[i]) % (2 * math.pi)
            diff = abs(got - want)
            diff = min(diff, 2 * math.pi - diff)
            assert diff < 1e-9, (hd, i, pos, got, want)


def check_v_not_rotated_and_layer_step(orc):
    """The layer step: q and k rotated at each token's position, v only
    normalised; positions come from past_lens and cu_new."""
    n_q, n_kv, hd = 4, 2, 256
    rng = np.random.default_rng(61)
    cu = np.array([0, 3, 3, 5], np.int32)  # the middle sequence has no new token
    past = np.array([10, 0, 2000], np.int32)
    n = int(cu[-1])
    q = _bits(rng.standard_normal((n, n_q, hd)).astype(np.float32))
    k = _bits(rng.standard_normal((n, n_kv, hd)).astype(np.float32))
    v = _bits(rng.standard_normal((n, n_kv, hd)).astype(np.float32))
    qw = (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32)
    qo, ko, vo = orc.qkv_norm_rope(q, k, v, cu, past, 1e-6, 1e4, 128, q_w=qw)
    pos = [10, 11, 12, 2000, 2001]
    for t in range(n):
        for hq in range(n_q):
            want = orc.norm_rope_row(q[t, hq], 1e-6, weight=qw, theta=1e4, pos=pos[t])
            assert np.array_equal(qo[t, hq], want)
        for g in range(n_kv):
            assert np.array_equal(ko[t, g], orc.norm_rope_row(k[t, g], 1e-6, theta=1e4,
                                                              pos=pos[t]))
            assert np.array_equal(vo[t, g], orc.norm_rope_row(v[t, g], 1e-6, rotate=False))
    # a shared-cache layer: q only
    qo2, ko2, vo2 = orc.qkv_norm_rope(q, None, None, cu, past, 1e-6, 1e4, 128, q_w=qw)
    assert ko2 is None and vo2 is None and np.array_equal(qo2, qo)


def check_bf16_rounding(orc):
    import torch
    exact = np.array([1.0, -2.5, 0.0078125, 2.0 ** -130], np.float64)  # bf16 values
    assert np.array_equal(orc.to_bf16(exact), _bits(exact.astype(np.float32)))
    # ties to even: 1 + 2^-8 -> 1, 1 + 3 * 2^-8 -> 1 + 2^-6
    assert orc.to_bf16([1.0 + 2 ** -8])[0] == 0x3F80
    assert orc.to_bf16([1.0 + 3 * 2 ** -8])[0] == 0x3F82
    rng = np.random.default_rng(71)
    vals = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                           [1e-40, -5e-39, 3.3e38, -3.4e38]]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.to_bf16(vals.astype(np.float64)), ref)


ROPE_CHECKS = [
    check_rms_norm_closed_form, check_rms_norm_scale_invariant_and_weight,
    check_rope_position_zero_is_identity, check_rope_relative_position,
    check_rope_pairs_keep_length, check_rope_frequency_rule,
    check_v_not_rotated_and_layer_step, check_bf16_rounding,
]
