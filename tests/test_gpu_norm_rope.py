"""The fused pre-attention step on the GPU (qkv_norm_rope_cache_write: per-head
RMS-norm, proportional RoPE of q and k, cache write of k and v) against the
fp64 oracle.

Bar (derived in gpu_harness.assert_norm_rope_close): each bf16 result within
half a bf16 unit of the oracle's exact fp64 value plus the kernel's fp32
error, 2^-20 (|y_d| + |y_partner|) in the normalised values of its rotation
pair. In practice nearly every result is the oracle's own rounding; the
share that is not is also bounded (below 1e-3). Every pool slot that is not
written must keep its bits."""
import numpy as np
import pytest
import torch

from gpu_harness import GpuStep, NormRopeCase, assert_close, assert_norm_rope_close, host_bits
from paged_sliding_window_gb300 import binding
from paged_sliding_window_gb300 import workloads as wl
from paged_sliding_window_gb300.staging import dev_bf16
from paged_sliding_window_gb300.workloads import Layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.default()


def _written_slots(step):
    """Pool rows (block, offset) of the step's new tokens."""
    rows = []
    for b in range(step.n_seqs):
        for i in range(int(step.new_lens[b])):
            pos = int(step.past_lens[b]) + i
            rows.append((int(step.block_table[b, pos // 16]), pos % 16))
    return rows


def _check_pools(g_pool, before, exact, pre, rotated, step, what):
    """New rows within the bar of the oracle's exact rows, every other slot
    unchanged."""
    got = host_bits(g_pool)
    slots = _written_slots(step)
    idx = tuple(np.array(slots).T)
    assert_norm_rope_close(got[idx], exact, pre, rotated, f"{what} new rows")
    mask = np.ones(got.shape[:2], bool)
    mask[idx] = False
    assert np.array_equal(got[mask], before[mask]), f"{what}: a slot outside the step changed"


def _check_q(case, got_bits, with_kv=True):
    exact_q = case.oracle_exact(with_kv)[0]
    pre_q = case.oracle_exact(with_kv, rotate=False)[0]
    assert_norm_rope_close(got_bits, exact_q, pre_q, True, "q_out")
    ref_q = case.oracle(with_kv)[0]
    assert float((got_bits != ref_q).mean()) < 1e-3, "q_out: too many results off the oracle's rounding"


def run_case(orc, case, check_v=True):
    g = GpuStep(case.step)
    k_before = host_bits(g.k_pool)
    v_before = None if g.v_pool is None else host_bits(g.v_pool)
    out = case.gpu(g)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    _check_q(case, host_bits(out))
    _, ek, ev = case.oracle_exact()
    _, pk, pv = case.oracle_exact(rotate=False)
    _check_pools(g.k_pool, k_before, ek, pk, True, case.step, "K")
    if check_v and g.v_pool is not None:
        _check_pools(g.v_pool, v_before, ev, pv, False, case.step, "V")
    return g, out


def test_norm_rope_sliding_layer(orc):
    """Sliding layer (head_dim 256, theta 1e4, every dim rotated, weighted q/k
    norms, weightless v norm): decode tokens and prefill chunks, ragged."""
    layer = Layer(16, 8, 256, window=1024)
    past = [0, 1, 15, 16, 1000, 4095, 3000, 0, 777]
    new = [1, 1, 1, 1, 1, 1, 200, 130, 64]
    run_case(orc, NormRopeCase(orc, layer, past, new, 101, 1e4, 1.0))


def test_norm_rope_many_heads(orc):
    """48 query and 16 KV heads (80 head vectors per token, more than one
    warp's share in the earlier layout): units of four head vectors, twelve
    of q and four each of k and v per token."""
    layer = Layer(48, 16, 256, window=1024)
    run_case(orc, NormRopeCase(orc, layer, [5, 100, 0], [3, 17, 1], 112, 1e4, 1.0))


def test_norm_rope_full_layer_partial_k_eq_v(orc):
    """Full layer (head_dim 512, theta 1e6, a quarter of the dims rotated), V
    aliasing the K pages: only K is written."""
    layer = Layer(32, 4, 512, window=0, k_eq_v=True)
    run_case(orc, NormRopeCase(orc, layer, [0, 20000, 5, 2047], [3, 1, 100, 17], 102, 1e6, 0.25,
                               eps=1e-5))


def test_norm_rope_v_from_the_k_projection(orc):
    """A layer without its own V projection that keeps a V cache: V is the
    same raw rows as K, only normalised (with a v weight), K normalised and
    rotated."""
    layer = Layer(16, 2, 512, window=0)
    run_case(orc, NormRopeCase(orc, layer, [10, 300], [40, 1], 103, 1e6, 0.5, v_from_k=True,
                               v_weight=True))


def test_norm_rope_large_positions(orc):
    """Positions up to about 70000, where a float angle would be off by far
    more than a bf16 unit."""
    layer = Layer(4, 2, 512, window=0)
    run_case(orc, NormRopeCase(orc, layer, [65530, 69000, 40000], [8, 1, 3], 104, 1e6, 1.0))


@pytest.mark.parametrize("n_q,n_kv", [(4, 2), (3, 1)])
def test_norm_rope_many_sequences_with_empty_chunks(orc, n_q, n_kv):
    """1100 sequences (the warp's sequence search takes three rounds past 961)
    with new lengths 0, 1, 2 or 5 and pasts across page boundaries: every
    token lands in its own sequence's slot, empty sequences write nothing.
    Few KV heads keep the pools small; the head counts give units of two
    head vectors and of one."""
    layer = Layer(n_q, n_kv, 256, window=1024)
    rng = np.random.default_rng(109)
    n = 1100
    new = rng.choice([0, 0, 1, 2, 5], size=n)
    past = rng.integers(0, 40, size=n)
    run_case(orc, NormRopeCase(orc, layer, past, new, 110, 1e4, 1.0))


@pytest.mark.parametrize("hd,theta,factor", [(256, 1e4, 1.0), (512, 1e6, 0.25)])
def test_norm_rope_positions_past_2_22(orc, hd, theta, factor):
    """q-only calls (no cache write, so no pages) at positions where the
    float angle reduction takes its second step (2^22 to 2^24), across the
    switch to double at 2^24, and on to 2^26 (where the oracle's own fp64
    product is still good to about 1.5e-8 rad)."""
    layer = Layer(8, 4, hd, window=0)
    rng = np.random.default_rng(108)
    past = np.array([2**22 - 5, 2**23 + 11, 2**24 - 4, 2**24 + 1, 2**25 + 3, 2**26 - 9],
                    np.int32)
    new = np.array([9, 3, 8, 2, 4, 7], np.int32)
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    n = int(cu[-1])
    q_raw = wl.f32_to_bf16_bits((3.0 * rng.standard_normal((n, 8, hd))).astype(np.float32))
    qw = (1.0 + 0.1 * rng.standard_normal(hd)).astype(np.float32)
    angles = int(factor * hd / 2)
    exact = orc.qkv_norm_rope(q_raw, None, None, cu, past, 1e-6, theta, angles, q_w=qw)[0]
    pre = orc.qkv_norm_rope(q_raw, None, None, cu, past, 1e-6, theta, 0, q_w=qw)[0]
    w_dev = torch.from_numpy(qw).cuda()
    rn = binding.make_norm_rope(theta, factor, 1e-6, w_dev, None, None)
    q = dev_bf16(q_raw)
    out = torch.empty_like(q)
    binding.qkv_norm_rope_cache_write(layer, rn, q, None, None, torch.from_numpy(cu).cuda(),
                                      torch.from_numpy(past).cuda(), None, out, None, None)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    assert_norm_rope_close(host_bits(out), exact, pre, True, f"q_out hd {hd}")


def test_norm_rope_q_only_leaves_pools(orc):
    """A layer reading another layer's cache: only q is processed, in place,
    and no pool changes."""
    layer = Layer(16, 8, 256, window=1024)
    case = NormRopeCase(orc, layer, [100, 3000], [1, 33], 105, 1e4, 1.0)
    g = GpuStep(case.step)
    k_before, v_before = host_bits(g.k_pool), host_bits(g.v_pool)
    q = dev_bf16(case.q_raw)
    case.gpu(g, with_kv=False, q_out=q)  # in place
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    _check_q(case, host_bits(q), with_kv=False)
    assert np.array_equal(host_bits(g.k_pool), k_before)
    assert np.array_equal(host_bits(g.v_pool), v_before)


def test_norm_rope_bad_block_is_flagged_q_still_written(orc):
    layer = Layer(16, 8, 256, window=64)
    case = NormRopeCase(orc, layer, [100, 20], [1, 1], 106, 1e4, 1.0)
    g = GpuStep(case.step)
    bad = g.table.clone()
    bad[0, 100 // 16] = case.step.cache.num_blocks + 3
    g.pages = binding.make_pages(bad, case.step.cache.num_blocks)
    out = case.gpu(g)
    assert binding.get_error() & binding.DEVERR_BLOCK_ID
    _check_q(case, host_bits(out))


def test_norm_rope_bad_lengths_are_flagged(orc):
    """A sequence with a negative past length is skipped whole (flagged as a
    length error: no q_out row, no cache write); a sequence past the end of
    its block-table row still gets its q_out rows at their positions, only
    its K/V rows are dropped (a capacity error). The third sequence is
    processed as usual, and no other pool slot changes."""
    layer = Layer(8, 4, 256, window=1024)
    case = NormRopeCase(orc, layer, [10, 20, 30], [2, 3, 2], 111, 1e4, 1.0)
    st = case.step
    g = GpuStep(st)
    k_before, v_before = host_bits(g.k_pool), host_bits(g.v_pool)
    max_blocks = int(g.table.shape[1])
    past = st.past_lens.astype(np.int32).copy()
    past[1] = -7                   # every token of sequence 1 at a negative position
    past[2] = max_blocks * 16      # sequence 2 beyond its block-table row
    g.past = torch.from_numpy(past).cuda()
    nan_bits = 0x7FC0
    out = torch.from_numpy(np.full(case.q_raw.shape, nan_bits, np.uint16).view(np.int16)).cuda()
    out = out.view(torch.bfloat16)
    case.gpu(g, q_out=out)
    torch.cuda.synchronize()
    err = binding.get_error()
    assert err & binding.DEVERR_LENGTH and err & binding.DEVERR_CAPACITY, err
    got = host_bits(out)
    cu = st.cu_new.astype(np.int32)
    past_ok = past.copy()
    past_ok[1] = 0  # the oracle needs some position; those rows are not compared
    exact = orc.qkv_norm_rope(case.q_raw, None, None, cu, past_ok, case.eps, case.theta,
                              case.rope_angles, q_w=case.qw)[0]
    pre = orc.qkv_norm_rope(case.q_raw, None, None, cu, past_ok, case.eps, case.theta, 0,
                            q_w=case.qw)[0]
    for b in (0, 2):
        rows = slice(int(cu[b]), int(cu[b + 1]))
        assert_norm_rope_close(got[rows], exact[rows], pre[rows], True, f"q_out of sequence {b}")
    assert np.all(got[int(cu[1]):int(cu[2])] == nan_bits), "a skipped token's q_out row was written"
    # pools: only sequence 0's slots change
    _, ek, ev = case.oracle_exact()
    _, pk, pv = case.oracle_exact(rotate=False)
    n0 = int(cu[1])
    slots = [(int(st.block_table[0, (int(st.past_lens[0]) + i) // 16]), (int(st.past_lens[0]) + i) % 16)
             for i in range(n0)]
    idx = tuple(np.array(slots).T)
    for pool, before, ex, pr, rot, what in ((g.k_pool, k_before, ek, pk, True, "K"),
                                           (g.v_pool, v_before, ev, pv, False, "V")):
        bits = host_bits(pool)
        assert_norm_rope_close(bits[idx], ex[:n0], pr[:n0], rot, f"{what} rows of sequence 0")
        mask = np.ones(bits.shape[:2], bool)
        mask[idx] = False
        assert np.array_equal(bits[mask], before[mask]), f"{what}: a slot outside sequence 0 changed"


@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_fused_step_then_attention_matches_oracle_pipeline(orc, mode):
    """The layer path from raw projections: fused step, then decode or chunked
    prefill, against the oracle doing the same (its own rounding, its own
    cache write, its own attention). Scale 1/16 keeps the softmax away from
    near ties, where a one-unit bf16 difference in an input could move the
    output by more than the attention bar."""
    layer = Layer(8, 4, 256, window=256, softcap=50.0, scale=1.0 / 16)
    if mode == "decode":
        past, new = [300, 17, 1000, 2], [1, 1, 1, 1]
    else:
        past, new = [0, 200, 900], [100, 64, 300]
    case = NormRopeCase(orc, layer, past, new, 107, 1e4, 1.0)
    g = GpuStep(case.step)
    q = case.gpu(g)
    g.q = q
    if mode == "decode":
        g.decode()
    else:
        g.prefill()
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    # oracle pipeline: history, then the step's own rounded rows, then attention
    ref_q, ref_k, ref_v = case.oracle()
    st = case.step
    c = st.cache
    kp, vp = c.empty_pools()
    orc.kv_cache_write(c.hist_k, c.hist_v, c.hist_cu, c.hist_past, st.block_table, kp, vp,
                       in_place=True)
    orc.kv_cache_write(ref_k, ref_v, st.cu_new, st.past_lens, st.block_table, kp, vp,
                       in_place=True)
    L = layer.as_dict()
    if mode == "decode":
        ref_o, ref_l, _ = orc.decode(L, ref_q, kp, vp, st.block_table, st.seq_lens)
    else:
        ref_o, ref_l, _ = orc.prefill(L, ref_q, st.cu_new, st.past_lens, kp, vp, st.block_table)
    assert_close(g.out.cpu().numpy(), ref_o, f"{mode} out after the fused step")
    assert_close(g.lse.cpu().numpy(), ref_l, f"{mode} lse after the fused step")
