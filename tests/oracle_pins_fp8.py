"""Pins of the oracle's FP8 pages (E4M3 codes with one fp32 scale per slot
and KV head) against facts fixed outside the oracle:

* the E4M3 format itself, through torch's float8_e4m3fn: the value of every
  one of the 256 codes, and round-to-nearest-even of float32 values inside
  the finite range;
* closed forms of the per-row quantisation: the row's largest magnitude maps
  to code +-448 exactly, every value is recovered to within half a code step
  (2^-4 relative for normal codes, 2^-10 of the scale for subnormal ones),
  an all-zero row gets scale 0;
* the FP8 attention path reduces to the (separately pinned) bf16 path when
  every scale is 1, since E4M3 values are exact in bf16; and a scale enters
  linearly: doubling every K scale is doubling the score scale, doubling
  every V scale doubles the output.
"""
from __future__ import annotations

import numpy as np

from paged_sliding_window_gb300 import workloads as wl


def _decode_torch(codes):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def check_e4m3_code_values(orc):
    codes = np.arange(256, dtype=np.uint8)
    got, ref = orc.e4m3_decode(codes), _decode_torch(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # S.1111.111
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def check_e4m3_rounding(orc):
    import torch
    rng = np.random.default_rng(81)
    mags = np.exp2(rng.uniform(-14, np.log2(440.0), 20000))
    x = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    # exact ties between neighbouring codes, in every binade
    ties = []
    vals = np.unique(np.abs(orc.e4m3_decode(np.arange(0x7F, dtype=np.uint8))))
    vals = vals[np.isfinite(vals)]
    ties = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, ties, -ties])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(x), ref)
    # saturation at the largest finite value
    assert list(orc.e4m3_encode(np.array([448.0, 470.0, 1e30, -1e30], np.float32))) == \
        [0x7E, 0x7E, 0x7E, 0xFE]


def _quantise(orc, rows):
    """Rows through the oracle's FP8 cache write (one token per row, one
    sequence, identity block table): (codes, scales)."""
    n, hd = rows.shape
    k8 = np.zeros(((n + 15) // 16, 16, 1, hd), np.uint8)
    ks = np.zeros(((n + 15) // 16, 16, 1), np.float32)
    table = np.arange(k8.shape[0], dtype=np.int32)[None, :]
    st = orc.kv_cache_write_fp8(rows[:, None, :], None, [0, n], [0], table, k8, None, ks, None)
    assert st == 0
    return k8.reshape(-1, hd)[:n], ks.reshape(-1)[:n]


def check_fp8_row_quantisation(orc):
    rng = np.random.default_rng(82)
    rows = wl.f32_to_bf16_bits((rng.standard_normal((40, 256)) *
                                np.exp2(rng.uniform(-20, 20, (40, 1)))).astype(np.float32))
    rows[3] = 0  # an all-zero row
    codes, scales = _quantise(orc, rows)
    x = wl.bf16_bits_to_f32(rows).astype(np.float64)
    amax = np.abs(x).max(axis=1)
    assert scales[3] == 0.0 and not codes[3].any()
    nz = amax > 0
    # the largest magnitude of each row is code +-448
    for r in np.nonzero(nz)[0]:
        j = int(np.argmax(np.abs(x[r])))
        assert codes[r, j] & 0x7F == 0x7E, r
        assert abs(float(scales[r]) - amax[r] / 448.0) <= 2.0 ** -23 * amax[r] / 448.0
    xhat = orc.e4m3_decode(codes) * scales[:, None].astype(np.float64)
    err = np.abs(xhat - x)
    bound = 2.0 ** -4 * np.abs(xhat) + 2.0 ** -10 * scales[:, None] + 2.0 ** -20 * np.abs(x)
    assert np.all(err[nz] <= bound[nz])


def _fp8_case(orc, seed, hd=64, n_q=4, n_kv=2, lens=(37, 70, 5), k_eq_v=False):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens)
    pages = (lens + 15) // 16
    table = np.full((len(lens), int(pages.max())), -1, np.int32)
    perm = rng.permutation(int(pages.sum()) + 3).astype(np.int32)
    off = 0
    for b, p in enumerate(pages):
        table[b, :p] = perm[off:off + p]
        off += p
    nb = int(pages.sum()) + 3
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    k8 = rng.choice(finite, (nb, 16, n_kv, hd)).astype(np.uint8)
    v8 = None if k_eq_v else rng.choice(finite, (nb, 16, n_kv, hd)).astype(np.uint8)
    q = wl.f32_to_bf16_bits(rng.standard_normal((len(lens), n_q, hd)).astype(np.float32) * 0.05)
    layer = dict(n_q_heads=n_q, n_kv_heads=n_kv, head_dim=hd, window=32, softcap=0.0,
                 scale=0.02, k_eq_v=int(k_eq_v), block_size=16)
    return layer, q, k8, v8, table, lens


def check_fp8_attention_unit_scales_is_bf16_attention(orc):
    for k_eq_v in (False, True):
        layer, q, k8, v8, table, lens = _fp8_case(orc, 83, k_eq_v=k_eq_v)
        ones = np.ones(k8.shape[:3], np.float32)
        o8, l8, _ = orc.decode_fp8(layer, q, k8, v8, ones, None if k_eq_v else ones, table,
                                   lens, threads=1)
        to_bf16 = lambda c: wl.f32_to_bf16_bits(orc.e4m3_decode(c).astype(np.float32))
        kb = to_bf16(k8)
        vb = None if k_eq_v else to_bf16(v8)
        ob, lb, _ = orc.decode(layer, q, kb, vb, table, lens, threads=1)
        assert np.array_equal(o8, ob) and np.array_equal(l8, lb), k_eq_v


def check_fp8_scales_enter_linearly(orc):
    layer, q, k8, v8, table, lens = _fp8_case(orc, 84)
    rng = np.random.default_rng(85)
    ks = rng.uniform(0.5, 2.0, k8.shape[:3]).astype(np.float32)
    vs = rng.uniform(0.5, 2.0, k8.shape[:3]).astype(np.float32)
    o, l, _ = orc.decode_fp8(layer, q, k8, v8, ks, vs, table, lens, threads=1)
    o2, l2, _ = orc.decode_fp8(dict(layer, scale=layer["scale"] * 2), q, k8, v8, ks, vs, table,
                               lens, threads=1)
    o3, l3, _ = orc.decode_fp8(layer, q, k8, v8, ks * 2, vs, table, lens, threads=1)
    assert np.array_equal(o2, o3) and np.array_equal(l2, l3)
    o4, l4, _ = orc.decode_fp8(layer, q, k8, v8, ks, vs * 2, table, lens, threads=1)
    assert np.array_equal(o4, 2 * o) and np.array_equal(l4, l)


FP8_CHECKS = [
    check_e4m3_code_values, check_e4m3_rounding, check_fp8_row_quantisation,
    check_fp8_attention_unit_scales_is_bf16_attention, check_fp8_scales_enter_linearly,
]
