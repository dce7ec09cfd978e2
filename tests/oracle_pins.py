"""Checks that pin the CPU oracle to facts fixed outside the oracle itself.

Each ``check_*`` takes an oracle instance (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with:

* the worked examples printed on the pages (``tests/golden/``),
* closed forms of softmax attention (one visible key, uniform scores,
  identical keys, the window's key count read off ``lse``),
* an independent dense brute force over contiguous per-sequence K/V arrays,
  and torch's ``scaled_dot_product_attention`` in float64 with an explicit
  boolean mask,
* structural identities: paged == contiguous layout, decode == last chunk row,
  chunked prefill == sequential decodes, k_eq_v == explicit V copy,
  softcap -> identity as cap -> infinity.

The same checks run against deliberately broken copies of the oracle in
``test_oracle_mutants.py`` to show that each planted mistake is caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from oracle_pins_fp8 import FP8_CHECKS
from oracle_pins_rope import ROPE_CHECKS
from paged_sliding_window_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f64(bits) -> np.ndarray:
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def layer_dict(n_q, n_kv, hd, window=0, softcap=0.0, scale=1.0, k_eq_v=False, bs=16):
    return dict(n_q_heads=n_q, n_kv_heads=n_kv, head_dim=hd, window=window,
                softcap=softcap, scale=scale, k_eq_v=int(k_eq_v), block_size=bs)


class Case:
    """Logical per-sequence K/V (contiguous) written into canary-filled paged
    pools through the oracle's own cache write."""

    def __init__(self, orc, layer, seq_lens, seed, num_blocks=None, identity=False,
                 kv=None, q=None, new_per_seq=1):
        self.layer = layer
        self.seq_lens = np.asarray(seq_lens, dtype=np.int64)
        n_kv, hd, bs = layer["n_kv_heads"], layer["head_dim"], layer["block_size"]
        ss = np.random.SeedSequence(seed)
        rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
        pages = (self.seq_lens + bs - 1) // bs
        if identity:
            nb = int(pages.sum()) if num_blocks is None else num_blocks
            table = np.full((len(pages), max(1, int(pages.max()))), -1, dtype=np.int32)
            off = 0
            for b, n in enumerate(pages):
                table[b, :n] = np.arange(off, off + n)
                off += n
        else:
            table, nb = wl.deal_block_table(rng, pages, num_blocks)
        self.table, self.num_blocks = table, nb
        total = int(self.seq_lens.sum())
        s_k, s_v, s_q = ss.spawn(3)
        if kv is None:
            k_all = wl.normal_bf16(s_k, (total, n_kv, hd), True, 1)
            v_all = wl.normal_bf16(s_v, (total, n_kv, hd), True, 1)
        else:
            k_all, v_all = kv
        if layer["k_eq_v"]:
            v_all = k_all
        self.k_all, self.v_all = k_all, v_all
        self.cu = wl.cu_from_lens(self.seq_lens)
        shape = (nb, bs, n_kv, hd)
        k_pool = np.full(shape, wl.CANARY_BF16, dtype=np.uint16)
        v_pool = None if layer["k_eq_v"] else np.full(shape, wl.CANARY_BF16, dtype=np.uint16)
        self.k_pool, self.v_pool, st = orc.kv_cache_write(
            k_all, None if layer["k_eq_v"] else v_all, self.cu,
            np.zeros(len(self.seq_lens), np.int32), table, k_pool, v_pool, bs)
        assert st == 0
        n_q = layer["n_q_heads"]
        # queries: one per sequence (decode) or per row (prefill), drawn on demand
        self.q_all = (wl.normal_bf16(s_q, (total, n_q, hd), True, 1) if q is None else q)

    def logical(self, b):
        lo, hi = int(self.cu[b]), int(self.cu[b + 1])
        return f64(self.k_all[lo:hi]), f64(self.v_all[lo:hi])

    def q_at(self, b, p):
        """Query bits for sequence b at position p (taken from the q table)."""
        return self.q_all[int(self.cu[b]) + p]

    def decode(self, orc):
        q = np.stack([self.q_at(b, int(L) - 1) for b, L in enumerate(self.seq_lens)])
        out, lse, _ = orc.decode(self.layer, q, self.k_pool, self.v_pool, self.table,
                                 self.seq_lens, threads=2)
        return q, out, lse

    def prefill(self, orc, chunk_lens):
        """Prefill the last chunk_lens[b] positions of each sequence."""
        chunk_lens = np.asarray(chunk_lens, dtype=np.int64)
        past = self.seq_lens - chunk_lens
        rows = []
        for b in range(len(self.seq_lens)):
            for i in range(int(chunk_lens[b])):
                rows.append(self.q_at(b, int(past[b]) + i))
        q = np.stack(rows) if rows else np.zeros((0, self.layer["n_q_heads"],
                                                   self.layer["head_dim"]), np.uint16)
        out, lse, _ = orc.prefill(self.layer, q, wl.cu_from_lens(chunk_lens), past,
                                  self.k_pool, self.v_pool, self.table, threads=2)
        return q, out, lse, past


def brute(layer, q_bits, K, V, p):
    """Dense brute force for one query at absolute position p over contiguous
    logical K/V [L, n_kv, hd] (float64)."""
    n_q, n_kv = layer["n_q_heads"], layer["n_kv_heads"]
    group = n_q // n_kv
    q = f64(q_bits)
    out = np.zeros((n_q, layer["head_dim"]))
    lse = np.full(n_q, -np.inf)
    if p < 0:
        return out, lse
    keys = np.arange(p + 1)
    if layer["window"] > 0:
        keys = keys[p - keys < layer["window"]]
    for h in range(n_q):
        kv = h // group
        s = layer["scale"] * (K[keys, kv, :] @ q[h])
        if layer["softcap"] > 0:
            s = layer["softcap"] * np.tanh(s / layer["softcap"])
        mx = s.max()
        w = np.exp(s - mx)
        out[h] = (w[:, None] * V[keys, kv, :]).sum(0) / w.sum()
        lse[h] = mx + math.log(w.sum())
    return out, lse


def _close(a, b, tol=1e-12, what=""):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    ok = np.isclose(a, b, rtol=tol, atol=tol) | (np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b)))
    assert ok.all(), f"{what}: max diff {np.nanmax(np.abs(a - b))}"


# --------------------------------------------------------------------------- #
# golden examples printed on the pages
# --------------------------------------------------------------------------- #
def check_slot_golden(orc):
    g = json.load(open(os.path.join(GOLDEN, "slot_mapping_example.json")))
    bs, pos = g["block_size"], g["token_position"]
    row = np.array([40, 17, 93, 5], dtype=np.int32)  # arbitrary physical ids
    got = orc.slot(row, pos, bs)
    assert got == row[g["logical_block"]] * bs + g["offset"], got
    # every position of the first four pages maps into the right block/offset
    for p in range(4 * bs):
        s = orc.slot(row, p, bs)
        assert s // bs == row[p // bs] and s % bs == p % bs


def check_kv_size_golden(orc):
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_size_example.json")))
    hd = g["d_model"] // g["n_heads"]
    mha = orc.kv_cache_bytes(1, g["seq_len"], 1, g["n_heads"], hd, g["dtype_bytes"], True)
    gqa = orc.kv_cache_bytes(1, g["seq_len"], 1, g["n_kv_heads_gqa"], hd, g["dtype_bytes"], True)
    assert f"{mha / 1024**3:.2f}" == f"{g['mha_gib_printed']:.2f}", mha
    assert f"{gqa / 1024**3:.2f}" == f"{g['gqa_gib_printed']:.2f}", gqa
    assert abs((1 - gqa / mha) * 100 - g["saving_percent_printed"]) < 1e-9
    # K only is half
    k_only = orc.kv_cache_bytes(1, g["seq_len"], 1, g["n_kv_heads_gqa"], hd, g["dtype_bytes"], False)
    assert k_only * 2 == gqa


# --------------------------------------------------------------------------- #
# cache write
# --------------------------------------------------------------------------- #
def check_cache_write(orc):
    n_kv, hd, bs = 2, 16, 16
    ss = np.random.SeedSequence(11)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    past = np.array([0, 5, 16, 31])
    new = np.array([3, 11, 16, 2])
    table, nb = wl.deal_block_table(rng, wl.pages_for(past + new), num_blocks=20)
    total = int(new.sum())
    k_new = wl.normal_bf16(ss.spawn(1)[0], (total, n_kv, hd), False, 1)
    v_new = wl.normal_bf16(ss.spawn(1)[0], (total, n_kv, hd), False, 1)
    shape = (nb, bs, n_kv, hd)
    k0 = np.full(shape, wl.CANARY_BF16, np.uint16)
    v0 = np.full(shape, wl.CANARY_BF16, np.uint16)
    cu = wl.cu_from_lens(new)
    k1, v1, st = orc.kv_cache_write(k_new, v_new, cu, past, table, k0, v0, bs)
    assert st == 0
    # restated loop: for each token, block = table[b][pos // bs], offset = pos % bs
    ek, ev = k0.copy(), v0.copy()
    t = 0
    for b in range(len(past)):
        for i in range(int(new[b])):
            pos = int(past[b]) + i
            blk, off = table[b][pos // bs], pos % bs
            ek[blk, off] = k_new[t]
            ev[blk, off] = v_new[t]
            t += 1
    assert np.array_equal(k1, ek) and np.array_equal(v1, ev)
    # k_eq_v: only K written
    k2, v2, st = orc.kv_cache_write(k_new, None, cu, past, table, k0, None, bs)
    assert st == 0 and v2 is None and np.array_equal(k2, ek)
    # a block id outside the pool is reported and nothing is written for it
    bad = table.copy()
    bad[0, 0] = nb + 3
    k3, _, st = orc.kv_cache_write(k_new, v_new, cu, past, bad, k0, v0, bs)
    assert st != 0
    assert np.array_equal(k3[table[1:][table[1:] >= 0]], ek[table[1:][table[1:] >= 0]])


# --------------------------------------------------------------------------- #
# brute force and library cross-checks
# --------------------------------------------------------------------------- #
BRUTE_LAYERS = [
    layer_dict(4, 2, 16, window=8),
    layer_dict(4, 4, 32, window=0),
    layer_dict(8, 2, 16, window=5, softcap=3.0, scale=0.7),
    layer_dict(6, 2, 32, window=17, softcap=0.5, scale=2.0),
    layer_dict(4, 1, 16, window=0, k_eq_v=True),
    layer_dict(8, 4, 256, window=32),
]


def check_brute_decode(orc):
    for li, layer in enumerate(BRUTE_LAYERS):
        lens = [1, 7, 16, 17, 33, 40][: 6 if layer["head_dim"] < 256 else 3]
        case = Case(orc, layer, lens, seed=100 + li)
        q, out, lse = case.decode(orc)
        for b, L in enumerate(case.seq_lens):
            K, V = case.logical(b)
            eo, el = brute(layer, q[b], K, V, int(L) - 1)
            _close(out[b], eo, 1e-11, f"decode out layer {li} seq {b}")
            _close(lse[b], el, 1e-11, f"decode lse layer {li} seq {b}")


def check_brute_prefill(orc):
    for li, layer in enumerate(BRUTE_LAYERS[:5]):
        lens = np.array([9, 20, 40, 5])
        chunks = np.array([4, 20, 13, 1])
        case = Case(orc, layer, lens, seed=200 + li)
        q, out, lse, past = case.prefill(orc, chunks)
        r = 0
        for b in range(len(lens)):
            K, V = case.logical(b)
            for i in range(int(chunks[b])):
                eo, el = brute(layer, q[r], K, V, int(past[b]) + i)
                _close(out[r], eo, 1e-11, f"prefill out layer {li} row {r}")
                _close(lse[r], el, 1e-11, f"prefill lse layer {li} row {r}")
                r += 1


def check_sdpa(orc):
    import torch
    import torch.nn.functional as F
    for li, layer in enumerate([BRUTE_LAYERS[0], BRUTE_LAYERS[1], layer_dict(4, 2, 16, 6, scale=0.3)]):
        lens = np.array([30, 12])
        chunks = np.array([10, 12])
        case = Case(orc, layer, lens, seed=300 + li)
        q, out, lse, past = case.prefill(orc, chunks)
        G = layer["n_q_heads"] // layer["n_kv_heads"]
        r = 0
        for b in range(len(lens)):
            K, V = case.logical(b)
            L, n = int(lens[b]), int(chunks[b])
            qb = torch.from_numpy(f64(q[r:r + n])).permute(1, 0, 2)          # [n_q, n, hd]
            kb = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)  # [n_q, L, hd]
            vb = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)
            pos = torch.arange(n)[:, None] + int(past[b])
            j = torch.arange(L)[None, :]
            mask = j <= pos
            if layer["window"] > 0:
                mask &= (pos - j) < layer["window"]
            ref = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=layer["scale"])
            _close(out[r:r + n], ref.permute(1, 0, 2).numpy(), 1e-10, f"sdpa layer {li} seq {b}")
            r += n


# --------------------------------------------------------------------------- #
# closed forms
# --------------------------------------------------------------------------- #
def check_window_one_is_self(orc):
    layer = layer_dict(4, 2, 32, window=1, softcap=2.0, scale=1.3)
    case = Case(orc, layer, [1, 9, 16, 17, 50], seed=400)
    q, out, lse = case.decode(orc)
    for b, L in enumerate(case.seq_lens):
        K, V = case.logical(b)
        for h in range(4):
            g = h // 2
            assert np.array_equal(out[b, h], V[L - 1, g]), (b, h)
            s = 1.3 * float(K[L - 1, g] @ f64(q[b, h]))
            _close(lse[b, h], 2.0 * math.tanh(s / 2.0), 1e-12, "lse of a single key")


def check_zero_query_counts_window(orc):
    """q = 0 makes every score 0: out is the mean of the visible V rows and
    lse = log(number of visible keys) = log(min(p + 1, W))."""
    W = 16
    layer = layer_dict(2, 1, 16, window=W)
    lens = [1, 15, 16, 17, 31, 32, 33, 64]
    total = sum(lens)
    qz = np.zeros((total, 2, 16), np.uint16)  # +0.0 in bf16
    case = Case(orc, layer, lens, seed=410, q=qz)
    q, out, lse = case.decode(orc)
    for b, L in enumerate(lens):
        K, V = case.logical(b)
        n_vis = min(L, W)
        _close(lse[b], [math.log(n_vis)] * 2, 1e-12, f"lse count L={L}")
        _close(out[b, 0], V[L - n_vis:L, 0].mean(0), 1e-12, f"mean L={L}")
    # prefill rows see the band: row at p sees min(p + 1, W) keys
    q2, out2, lse2, past = case.prefill(orc, [1, 5, 16, 17, 31, 32, 33, 64])
    r = 0
    for b, L in enumerate(lens):
        for i in range([1, 5, 16, 17, 31, 32, 33, 64][b]):
            p = int(past[b]) + i
            _close(lse2[r], [math.log(min(p + 1, W))] * 2, 1e-12, f"band count p={p}")
            r += 1


def check_identical_keys_uniform(orc):
    layer = layer_dict(4, 2, 16, window=0, softcap=1.5, scale=3.0)
    lens = [5, 23]
    total = sum(lens)
    ss = np.random.SeedSequence(420)
    k_row = wl.normal_bf16(ss.spawn(1)[0], (1, 2, 16), True, 1)
    k_all = np.repeat(k_row, total, axis=0)
    v_all = wl.normal_bf16(ss.spawn(1)[0], (total, 2, 16), True, 1)
    case = Case(orc, layer, lens, seed=421, kv=(k_all, v_all))
    q, out, lse = case.decode(orc)
    for b, L in enumerate(lens):
        K, V = case.logical(b)
        for h in range(4):
            _close(out[b, h], V[:, h // 2].mean(0), 1e-12, "identical keys -> mean")


def check_softcap_closed_form(orc):
    """Two visible keys with known dot products: the cap sits on the scaled
    score and before the softmax."""
    hd = 16
    layer = layer_dict(1, 1, hd, window=0, softcap=2.0, scale=3.0)
    k_rows = np.zeros((2, 1, hd), np.float32)
    k_rows[0, 0, 0], k_rows[1, 0, 0] = 1.5, -0.5
    v_rows = np.zeros((2, 1, hd), np.float32)
    v_rows[0, 0, :] = 1.0
    v_rows[1, 0, :] = -2.0
    q_rows = np.zeros((2, 1, hd), np.float32)
    q_rows[:, 0, 0] = 2.0
    kv = (wl.f32_to_bf16_bits(k_rows), wl.f32_to_bf16_bits(v_rows))
    case = Case(orc, layer, [2], seed=430, kv=kv, q=wl.f32_to_bf16_bits(q_rows))
    _, out, lse = case.decode(orc)
    s0 = 2.0 * math.tanh(3.0 * 3.0 / 2.0)   # q.k0 = 3
    s1 = 2.0 * math.tanh(3.0 * -1.0 / 2.0)  # q.k1 = -1
    w0, w1 = math.exp(s0), math.exp(s1)
    _close(out[0, 0], [(w0 * 1.0 + w1 * -2.0) / (w0 + w1)] * hd, 1e-13, "softcap closed form")
    _close(lse[0, 0], math.log(w0 + w1), 1e-13, "softcap lse")


def check_gqa_grouping(orc):
    """q heads h use kv head h // (n_q / n_kv): make kv head 1's V constant."""
    layer = layer_dict(4, 2, 16, window=0)
    lens = [12]
    ss = np.random.SeedSequence(440)
    k_all = wl.normal_bf16(ss.spawn(1)[0], (12, 2, 16), True, 1)
    v_f = wl.bf16_bits_to_f32(wl.normal_bf16(ss.spawn(1)[0], (12, 2, 16), True, 1)).copy()
    v_f[:, 1, :] = 0.75
    case = Case(orc, layer, lens, seed=441, kv=(k_all, wl.f32_to_bf16_bits(v_f)))
    _, out, _ = case.decode(orc)
    _close(out[0, 2], np.full(16, 0.75), 1e-14, "head 2 uses kv head 1")
    _close(out[0, 3], np.full(16, 0.75), 1e-14, "head 3 uses kv head 1")
    assert not np.allclose(out[0, 1], 0.75) and not np.allclose(out[0, 0], 0.75)


def check_empty_sequence(orc):
    layer = layer_dict(4, 2, 16, window=8)
    case = Case(orc, layer, [5], seed=450)
    q = np.zeros((1, 4, 16), np.uint16)
    out, lse, _ = orc.decode(layer, q, case.k_pool, case.v_pool, case.table, [0], threads=1)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))


# --------------------------------------------------------------------------- #
# structural identities
# --------------------------------------------------------------------------- #
def check_paged_equals_contiguous(orc):
    layer = layer_dict(4, 2, 32, window=20, softcap=4.0)
    lens = [3, 16, 47, 64]
    a = Case(orc, layer, lens, seed=500, identity=True)
    b = Case(orc, layer, lens, seed=500, num_blocks=37)
    assert not np.array_equal(a.table, b.table)
    _, oa, la = a.decode(orc)
    _, ob, lb = b.decode(orc)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def check_decode_equals_last_prefill_row(orc):
    layer = layer_dict(4, 2, 32, window=12, softcap=1.0, scale=0.5)
    lens = np.array([5, 12, 13, 40])
    case = Case(orc, layer, lens, seed=510)
    qd, od, ld = case.decode(orc)
    chunks = np.array([5, 3, 13, 7])
    qp, op, lp, past = case.prefill(orc, chunks)
    last = np.cumsum(chunks) - 1
    assert np.array_equal(op[last], od) and np.array_equal(lp[last], ld)


def check_prefill_equals_sequential_decodes(orc):
    layer = layer_dict(4, 2, 32, window=9, softcap=2.0)
    lens = np.array([30, 11])
    chunks = np.array([14, 11])
    case = Case(orc, layer, lens, seed=520)
    qp, op, lp, past = case.prefill(orc, chunks)
    r = 0
    for b in range(2):
        for i in range(int(chunks[b])):
            p = int(past[b]) + i
            seq_lens = np.zeros(2, np.int64)
            seq_lens[b] = p + 1
            qd = np.stack([qp[r]] * 2)
            od, ld, _ = orc.decode(layer, qd, case.k_pool, case.v_pool, case.table, seq_lens,
                                   seqs=[b], threads=1)
            assert np.array_equal(od[0], op[r]) and np.array_equal(ld[0], lp[r])
            r += 1
    # a chunk split in two gives the same rows
    q1, o1, l1, _ = case.prefill(orc, [6, 4])
    qa, oa, la, _ = case.prefill(orc, [14, 11])
    a_rows = list(range(14 - 6, 14)) + list(range(14 + 11 - 4, 25))
    assert np.array_equal(o1, oa[a_rows])


def check_softcap_to_identity(orc):
    base = layer_dict(4, 2, 32, window=0)
    capped = dict(base, softcap=1e7)
    case = Case(orc, base, [20, 33], seed=530)
    _, o0, l0 = case.decode(orc)
    q = np.stack([case.q_at(b, int(L) - 1) for b, L in enumerate(case.seq_lens)])
    o1, l1, _ = orc.decode(capped, q, case.k_pool, case.v_pool, case.table, case.seq_lens,
                           threads=1)
    _close(o1, o0, 1e-9, "softcap to identity")
    _close(l1, l0, 1e-9, "softcap to identity lse")


def check_k_eq_v_equals_copy(orc):
    keqv = layer_dict(4, 1, 32, window=0, k_eq_v=True)
    case = Case(orc, keqv, [9, 40], seed=540)
    q = np.stack([case.q_at(b, int(L) - 1) for b, L in enumerate(case.seq_lens)])
    o1, l1, _ = orc.decode(keqv, q, case.k_pool, None, case.table, case.seq_lens, threads=1)
    plain = dict(keqv, k_eq_v=0)
    o2, l2, _ = orc.decode(plain, q, case.k_pool, case.k_pool.copy(), case.table,
                           case.seq_lens, threads=1)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


ALL_CHECKS = [
    check_slot_golden, check_kv_size_golden, check_cache_write, check_brute_decode,
    check_brute_prefill, check_sdpa, check_window_one_is_self,
    check_zero_query_counts_window, check_identical_keys_uniform, check_softcap_closed_form,
    check_gqa_grouping, check_empty_sequence, check_paged_equals_contiguous,
    check_decode_equals_last_prefill_row, check_prefill_equals_sequential_decodes,
    check_softcap_to_identity, check_k_eq_v_equals_copy,
] + ROPE_CHECKS + FP8_CHECKS
