"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point declared in include/psw.h, sizes its
workspace by pure arithmetic, and rejects every invalid argument with its
documented code before touching a device."""
import ctypes
import os
import re

import pytest

from paged_sliding_window_gb300 import binding, build
from paged_sliding_window_gb300.workloads import Layer

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "psw.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^PSW_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)


def header_codes():
    text = open(HEADER).read()
    return {name: int(val) for name, val in re.findall(r"#define\s+(PSW_E\w+|PSW_OK)\s+(-?\d+)", text)}


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(binding.EXPORTED)
    for name in names:
        assert hasattr(lib, name), name


def test_error_codes_match_header():
    codes = header_codes()
    for code, name in binding.ERRORS.items():
        assert codes[name] == code
    assert codes["PSW_OK"] == 0


def test_strerror_covers_every_code(lib):
    for code in list(binding.ERRORS) + [0]:
        msg = lib.psw_strerror(code).decode()
        assert msg and msg != "unknown error", code
    assert lib.psw_strerror(12345).decode() == "unknown error"


SLIDING = Layer(n_q_heads=16, n_kv_heads=8, head_dim=256, window=1024)
FULL = Layer(n_q_heads=32, n_kv_heads=4, head_dim=512, window=0, k_eq_v=True)


def test_workspace_bytes_arithmetic(lib):
    # a 2048-byte counter block (one merge ticket per decode CTA), then for
    # decode (max CTAs + units) slots of 8 query heads x (head_dim floats +
    # (m, l)), and for prefill a 64-byte header plus one 8-byte entry per
    # block of 128 / G chunk tokens of every sequence; the larger of the two
    def expect(layer, n_seqs, max_len):
        G = layer.n_q_heads // layer.n_kv_heads
        units = n_seqs * layer.n_kv_heads * ((G + 7) // 8)
        slots = 512 + units
        align = lambda x: (x + 255) // 256 * 256
        decode = 2048 + align(slots * 8 * layer.head_dim * 4) + align(slots * 8 * 8)
        T = 128 // G
        prefill = align(2048 + 64 + n_seqs * ((max_len + T - 1) // T) * 8)
        return max(decode, prefill)
    for layer, n, max_len in ((SLIDING, 64, 4096), (FULL, 32, 4096), (SLIDING, 0, 4096),
                              (FULL, 1000, 4096), (FULL, 4, 1 << 24), (SLIDING, 2, 0)):
        assert binding.workspace_bytes(layer, n, max_len) == expect(layer, n, max_len)
    # the prefill term dominates for few, very long sequences
    assert expect(FULL, 4, 1 << 24) > expect(FULL, 4, 4096)


def test_counter_block_size_matches_header():
    text = open(HEADER).read()
    m = re.search(r"#define\s+PSW_WORKSPACE_COUNTER_BYTES\s+(\d+)", text)
    assert m and int(m.group(1)) == binding.WORKSPACE_COUNTER_BYTES


FAKE = 0x10000  # aligned fake device address; validation never dereferences


def _layer(**kw):
    base = dict(n_q_heads=16, n_kv_heads=8, head_dim=256, window=1024, softcap=0.0,
                scale=1.0, k_eq_v=0, block_size=16)
    base.update(kw)
    return binding.PswLayer(**base)


def _pages(table=FAKE, mbps=64, nb=1024):
    return binding.PswPages(table, mbps, nb)


def _decode(lib, layer, q=FAKE, k=FAKE, v=FAKE, pages=None, seq=FAKE, n=4, out=FAKE, ws=FAKE,
            ws_bytes=1 << 30):
    pages = pages or _pages()
    return lib.attn_decode_paged(ctypes.byref(layer), q, k, v, ctypes.byref(pages), seq, n, out,
                                 None, ws, ws_bytes, None)


def _write(lib, layer, k=FAKE, v=FAKE, cu=FAKE, past=FAKE, n=4, pages=None, kp=FAKE, vp=FAKE):
    pages = pages or _pages()
    return lib.kv_cache_write(ctypes.byref(layer), k, v, cu, past, n, ctypes.byref(pages), kp, vp,
                              None)


def _prefill(lib, layer, q=FAKE, cu=FAKE, past=FAKE, n=4, maxq=512, k=FAKE, v=FAKE, pages=None,
             out=FAKE):
    pages = pages or _pages()
    return lib.attn_prefill_chunked(ctypes.byref(layer), q, cu, past, n, 4 * 512, maxq, k, v,
                                    ctypes.byref(pages), out, None, FAKE, 1 << 30, None)


@pytest.mark.parametrize("kw,code", [
    (dict(n_q_heads=12, n_kv_heads=8), -2),
    (dict(n_q_heads=0), -2),
    (dict(n_kv_heads=0), -2),
    (dict(head_dim=128), -3),
    (dict(head_dim=384), -3),
    (dict(softcap=-1.0), -4),
    (dict(softcap=float("inf")), -4),
    (dict(softcap=float("nan")), -4),
    (dict(window=-1), -5),
    (dict(block_size=32), -6),
    (dict(scale=0.0), -8),
    (dict(scale=-1.0), -8),
    (dict(scale=float("nan")), -8),
    (dict(k_eq_v=2), -7),
])
def test_layer_validation_all_entry_points(lib, kw, code):
    layer = _layer(**kw)
    assert _decode(lib, layer) == code
    assert _write(lib, layer) == code
    assert _prefill(lib, layer) == code
    size = ctypes.c_size_t(0)
    assert lib.psw_workspace_bytes(ctypes.byref(layer), 4, 100, ctypes.byref(size)) == code


def test_k_eq_v_pointer_rules(lib):
    keqv = _layer(k_eq_v=1, n_q_heads=32, n_kv_heads=4, head_dim=512, window=0)
    assert _decode(lib, keqv, v=FAKE) == -7          # V pool given with k_eq_v
    assert _write(lib, keqv, v=FAKE, vp=None) == -7  # V rows given with k_eq_v
    assert _write(lib, keqv, v=None, vp=FAKE) == -7  # V pool given with k_eq_v
    assert _prefill(lib, keqv, v=FAKE) == -7
    plain = _layer()
    assert _decode(lib, plain, v=None) == -7         # V pool missing
    assert _write(lib, plain, v=None) == -7
    assert _prefill(lib, plain, v=None) == -7


def test_null_pointers(lib):
    layer = _layer()
    assert lib.attn_decode_paged(None, FAKE, FAKE, FAKE, ctypes.byref(_pages()), FAKE, 1, FAKE,
                                 None, FAKE, 1 << 30, None) == -1
    assert _decode(lib, layer, q=None) == -1
    assert _decode(lib, layer, k=None) == -1
    assert _decode(lib, layer, seq=None) == -1
    assert _decode(lib, layer, out=None) == -1
    assert _decode(lib, layer, pages=_pages(table=None)) == -1
    assert _write(lib, layer, k=None) == -1
    assert _write(lib, layer, cu=None) == -1
    assert _prefill(lib, layer, cu=None) == -1
    assert lib.psw_get_error(None, None) == -1


def test_capacity_alignment_nseqs(lib):
    layer = _layer()
    assert _decode(lib, layer, pages=_pages(mbps=0)) == -11
    assert _decode(lib, layer, pages=_pages(nb=0)) == -11
    assert _decode(lib, layer, pages=_pages(nb=(1 << 27) + 1)) == -11
    assert _decode(lib, layer, n=-1) == -9
    assert _write(lib, layer, n=-1) == -9
    assert _prefill(lib, layer, maxq=-1) == -11
    assert _decode(lib, layer, q=FAKE + 8) == -12
    assert _decode(lib, layer, k=FAKE + 2) == -12
    assert _write(lib, layer, kp=FAKE + 4) == -12
    assert _decode(lib, layer, ws=None) == -10
    assert _decode(lib, layer, ws_bytes=16) == -10


def test_empty_batch_is_a_no_op(lib):
    layer = _layer()
    assert _decode(lib, layer, n=0, ws=None, ws_bytes=0) == 0
    assert _write(lib, layer, n=0) == 0
    assert _prefill(lib, layer, n=0) == 0


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="host without a GPU only")
def test_valid_call_without_gpu_fails_loudly(lib):
    """No silent CPU path: a valid call on a host without a GPU is refused."""
    assert _decode(lib, _layer()) == -13
    assert _write(lib, _layer()) == -13


def _noalloc(lib, layer, q=FAKE, k=FAKE, v=FAKE, pages=None, seq=FAKE, n=4, out=FAKE):
    pages = pages or _pages()
    return lib.attn_decode_paged_noalloc(ctypes.byref(layer), q, k, v, ctypes.byref(pages), seq,
                                         n, out, None, None)


def test_noalloc_reports_argument_errors_before_the_scratch_limit(lib):
    """The no-allocation decode checks pointers and alignment like
    attn_decode_paged before it compares the batch with its static buffer."""
    layer = _layer()
    too_many = 4096  # far beyond the static buffer at head_dim 256
    assert binding.workspace_bytes(SLIDING, too_many, 1) > 16 * 1024 * 1024
    assert _noalloc(lib, layer, q=None, n=too_many) == -1
    assert _noalloc(lib, layer, out=None, n=too_many) == -1
    assert _noalloc(lib, layer, q=FAKE + 8, n=too_many) == -12
    assert _noalloc(lib, layer, v=None, n=too_many) == -7
    assert _noalloc(lib, layer, n=-1) == -9
    assert _noalloc(lib, _layer(head_dim=128), n=too_many) == -3
    assert _noalloc(lib, layer, n=too_many) == -16


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="host without a GPU only")
def test_noalloc_without_gpu_fails_loudly(lib):
    """Valid arguments on a host without a GPU: the one-time address lookup
    cannot run, and nothing falls back to the CPU."""
    assert _noalloc(lib, _layer(), n=0) == -13
    assert _noalloc(lib, _layer(), n=4) == -13


def _norm_rope(lib, layer, rn=None, q=FAKE, k=FAKE, v=FAKE, cu=FAKE, past=FAKE, n=4,
               pages=None, q_out=FAKE, kp=FAKE, vp=FAKE, use_pages=True):
    rn = rn or binding.PswNormRope(10000.0, 1.0, 1e-6, None, None, None)
    pages = pages or _pages()
    return lib.qkv_norm_rope_cache_write(ctypes.byref(layer), ctypes.byref(rn), q, k, v, cu,
                                         past, n, ctypes.byref(pages) if use_pages else None,
                                         q_out, kp, vp, None)


def test_norm_rope_argument_checks(lib):
    layer = _layer()
    for bad in (binding.PswNormRope(0.0, 1.0, 1e-6, None, None, None),
                binding.PswNormRope(float("inf"), 1.0, 1e-6, None, None, None),
                binding.PswNormRope(1e4, 0.0, 1e-6, None, None, None),
                binding.PswNormRope(1e4, 1.5, 1e-6, None, None, None),
                binding.PswNormRope(1e4, 1.0, -1.0, None, None, None),
                binding.PswNormRope(1e4, 1.0, float("nan"), None, None, None)):
        assert _norm_rope(lib, layer, rn=bad) == -17
    assert _norm_rope(lib, _layer(head_dim=128)) == -3
    assert _norm_rope(lib, layer, q=None) == -1
    assert _norm_rope(lib, layer, q_out=None) == -1
    assert _norm_rope(lib, layer, kp=None) == -1
    assert _norm_rope(lib, layer, v=None) == -7          # V rows missing on a k_eq_v = 0 layer
    keqv = _layer(k_eq_v=1, n_q_heads=32, n_kv_heads=4, head_dim=512, window=0)
    assert _norm_rope(lib, keqv) == -7                   # V rows given on a k_eq_v layer
    assert _norm_rope(lib, layer, k=None) == -1          # q only, but V rows named
    assert _norm_rope(lib, layer, q=FAKE + 8) == -12
    assert _norm_rope(lib, layer, n=-1) == -9
    assert _norm_rope(lib, layer, pages=_pages(mbps=0)) == -11
    w = binding.PswNormRope(1e4, 1.0, 1e-6, FAKE + 4, None, None)
    assert _norm_rope(lib, layer, rn=w) == -12
    assert _norm_rope(lib, layer, n=0) == 0
    # q only (a layer reading another layer's cache): no pages needed
    assert _norm_rope(lib, layer, k=None, v=None, kp=None, vp=None, n=0, use_pages=False) == 0


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="host without a GPU only")
def test_norm_rope_without_gpu_fails_loudly(lib):
    assert _norm_rope(lib, _layer()) == -13
    # any number of heads per token passes the argument checks (the kernel
    # takes a token's head vectors a few at a time): it reaches the device
    # step, which has no GPU here
    assert _norm_rope(lib, _layer(n_q_heads=128, n_kv_heads=16)) == -13
    assert _norm_rope(lib, _layer(n_q_heads=96, n_kv_heads=8, head_dim=512, window=0)) == -13


def _decode8(lib, layer, q=FAKE, k=FAKE, v=FAKE, ks=FAKE, vs=FAKE, pages=None, seq=FAKE, n=4,
             out=FAKE, ws=FAKE, ws_bytes=1 << 30):
    pages = pages or _pages()
    return lib.attn_decode_paged_fp8(ctypes.byref(layer), q, k, v, ks, vs, ctypes.byref(pages),
                                     seq, n, out, None, ws, ws_bytes, None)


def _write8(lib, layer, k=FAKE, v=FAKE, cu=FAKE, past=FAKE, n=4, pages=None, kp=FAKE, vp=FAKE,
            ks=FAKE, vs=FAKE):
    pages = pages or _pages()
    return lib.kv_cache_write_fp8(ctypes.byref(layer), k, v, cu, past, n, ctypes.byref(pages),
                                  kp, vp, ks, vs, None)


def test_fp8_argument_checks(lib):
    layer = _layer()
    assert _decode8(lib, _layer(head_dim=128)) == -3
    assert _write8(lib, _layer(head_dim=128)) == -3
    assert _decode8(lib, layer, ks=None) == -1
    assert _write8(lib, layer, ks=None) == -1
    assert _decode8(lib, layer, vs=None) == -7           # V scales missing on a k_eq_v = 0 layer
    assert _write8(lib, layer, vs=None) == -7
    keqv = _layer(k_eq_v=1, n_q_heads=32, n_kv_heads=4, head_dim=512, window=0)
    assert _decode8(lib, keqv, v=None) == -7             # V scales given on a k_eq_v layer
    assert _decode8(lib, keqv, v=None, vs=None, n=0) == 0
    assert _write8(lib, keqv, v=None, vp=None) == -7
    assert _write8(lib, keqv, v=None, vp=None, vs=None, n=0) == 0
    assert _decode8(lib, layer, ks=FAKE + 2) == -12      # scales: 4-byte aligned
    assert _write8(lib, layer, vs=FAKE + 1) == -12
    assert _write8(lib, layer, kp=FAKE + 8) == -12       # code pools: 16-byte aligned
    assert _decode8(lib, layer, ws=None) == -10
    assert _decode8(lib, layer, n=-1) == -9
    assert _write8(lib, layer, n=-1) == -9
    assert _decode8(lib, layer, n=0, ws=None, ws_bytes=0) == 0
    assert _write8(lib, layer, n=0) == 0


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="host without a GPU only")
def test_fp8_without_gpu_fails_loudly(lib):
    assert _decode8(lib, _layer()) == -13
    assert _write8(lib, _layer()) == -13


def test_testing_stall_argument_checks(lib):
    assert lib.psw_testing_stall(3, 0, 0) == -9
    assert lib.psw_testing_stall(-1, 0, 0) == -9
    assert lib.psw_testing_stall(1, -1, 0) == -9
    assert lib.psw_testing_stall(2, 0, -1) == -9
    assert lib.psw_testing_stall(1, 0, 2) == 0
    assert lib.psw_testing_stall(0, -1, -1) == 0


def _append(lib, layer, q=FAKE, kn=FAKE, vn=FAKE, k=FAKE, v=FAKE, pages=None, seq=FAKE, n=4,
            out=FAKE, ws=FAKE, ws_bytes=1 << 30):
    pages = pages or _pages()
    return lib.attn_decode_paged_append(ctypes.byref(layer), q, kn, vn, k, v,
                                        ctypes.byref(pages), seq, n, out, None, ws, ws_bytes, None)


def test_append_argument_checks(lib):
    layer = _layer()
    assert _append(lib, _layer(head_dim=128)) == -3
    assert _append(lib, layer, kn=None) == -1
    assert _append(lib, layer, q=None) == -1
    assert _append(lib, layer, vn=None) == -7          # new V rows missing on a k_eq_v = 0 layer
    keqv = _layer(k_eq_v=1, n_q_heads=32, n_kv_heads=4, head_dim=512, window=0)
    assert _append(lib, keqv, v=None) == -7            # new V rows given on a k_eq_v layer
    assert _append(lib, keqv, v=None, vn=None, n=0) == 0
    assert _append(lib, layer, kn=FAKE + 8) == -12
    assert _append(lib, layer, vn=FAKE + 2) == -12
    assert _append(lib, layer, ws=None) == -10
    assert _append(lib, layer, n=-1) == -9
    assert _append(lib, layer, n=0, ws=None, ws_bytes=0) == 0


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="host without a GPU only")
def test_append_without_gpu_fails_loudly(lib):
    assert _append(lib, _layer()) == -13
