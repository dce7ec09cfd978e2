"""Thin ctypes binding of libpsw.so (the C ABI declared in include/psw.h).

Argument marshalling only: every function takes torch tensors that already
live on the GPU, checks dtypes and shapes, and passes raw pointers, sizes and
the current CUDA stream to the C entry point of the same name. All arithmetic
runs in the CUDA kernels of the library; there is no fallback. If the
library cannot be loaded, every call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

PSW_OK = 0
ERRORS = {
    -1: "PSW_ENULL", -2: "PSW_EINVAL_HEADS", -3: "PSW_EINVAL_HDIM", -4: "PSW_EINVAL_SOFTCAP",
    -5: "PSW_EINVAL_WINDOW", -6: "PSW_EINVAL_BLOCKSIZE", -7: "PSW_EINVAL_KEQV",
    -8: "PSW_EINVAL_SCALE", -9: "PSW_EINVAL_NSEQS", -10: "PSW_EWORKSPACE",
    -11: "PSW_ECAPACITY", -12: "PSW_EALIGN", -13: "PSW_EDEVICE", -14: "PSW_ELAUNCH",
    -15: "PSW_ETENSORMAP", -16: "PSW_ESCRATCH", -17: "PSW_EINVAL_ROPE",
    -18: "PSW_EINVAL_LAYERS", -19: "PSW_ENOBLOCKS", -20: "PSW_EBLOCK",
}
DEVERR_BLOCK_ID, DEVERR_CAPACITY, DEVERR_LENGTH, DEVERR_PIPELINE = 1, 2, 4, 8
EXPORTED = ("psw_workspace_bytes", "kv_cache_write", "attn_decode_paged",
            "attn_prefill_chunked", "psw_get_error", "psw_strerror",
            "attn_decode_paged_noalloc", "qkv_norm_rope_cache_write", "psw_kv_share_map",
            "psw_block_pool_create", "psw_block_pool_destroy", "psw_block_pool_num_free",
            "psw_block_pool_allocate", "psw_block_pool_free", "psw_block_pool_get_cached",
            "psw_block_pool_cache", "psw_block_pool_ref_count", "psw_block_hash",
            "psw_block_pool_admit", "psw_block_pool_commit", "kv_cache_write_fp8",
            "attn_decode_paged_fp8", "psw_testing_stall", "attn_decode_paged_append")


class PswLayer(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("window", ctypes.c_int32),
                ("softcap", ctypes.c_float), ("scale", ctypes.c_float),
                ("k_eq_v", ctypes.c_int32), ("block_size", ctypes.c_int32)]


class PswPages(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64)]


class PswNormRope(ctypes.Structure):
    _fields_ = [("theta", ctypes.c_float), ("partial_rotary_factor", ctypes.c_float),
                ("eps", ctypes.c_float), ("q_weight", ctypes.c_void_p),
                ("k_weight", ctypes.c_void_p), ("v_weight", ctypes.c_void_p)]


class PswError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({strerror(code)})")
        self.code = code


_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads libpsw.so (building it first if asked and missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"libpsw.so not built ({path})")
            path = _build.build()
        lib = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        lp = ctypes.POINTER(PswLayer)
        pp = ctypes.POINTER(PswPages)
        lib.psw_workspace_bytes.argtypes = [lp, i32, i32, ctypes.POINTER(sz)]
        lib.kv_cache_write.argtypes = [lp, vp, vp, vp, vp, i32, pp, vp, vp, vp]
        lib.attn_decode_paged.argtypes = [lp, vp, vp, vp, pp, vp, i32, vp, vp, vp, sz, vp]
        lib.attn_prefill_chunked.argtypes = [lp, vp, vp, vp, i32, i32, i32, vp, vp, pp, vp, vp,
                                             vp, sz, vp]
        lib.attn_decode_paged_noalloc.argtypes = [lp, vp, vp, vp, pp, vp, i32, vp, vp, vp]
        lib.attn_decode_paged_noalloc.restype = ctypes.c_int
        lib.qkv_norm_rope_cache_write.argtypes = [lp, ctypes.POINTER(PswNormRope), vp, vp, vp,
                                                  vp, vp, i32, pp, vp, vp, vp, vp]
        lib.qkv_norm_rope_cache_write.restype = ctypes.c_int
        lib.psw_kv_share_map.argtypes = [i32, i32, i32, ctypes.POINTER(i32),
                                         ctypes.POINTER(i32)]
        lib.psw_kv_share_map.restype = ctypes.c_int
        i32p, u64 = ctypes.POINTER(i32), ctypes.c_uint64
        lib.psw_block_pool_create.argtypes = [i64, i32, ctypes.POINTER(vp)]
        lib.psw_block_pool_destroy.argtypes = [vp]
        lib.psw_block_pool_destroy.restype = None
        lib.psw_block_pool_num_free.argtypes = [vp]
        lib.psw_block_pool_num_free.restype = i64
        lib.psw_block_pool_allocate.argtypes = [vp, i32, i32p]
        lib.psw_block_pool_free.argtypes = [vp, i32p, i32]
        lib.psw_block_pool_get_cached.argtypes = [vp, u64, i32p]
        lib.psw_block_pool_cache.argtypes = [vp, i32, u64]
        lib.psw_block_pool_ref_count.argtypes = [vp, i32, i32p]
        lib.psw_block_hash.argtypes = [u64, i32p, i32]
        lib.psw_block_hash.restype = u64
        lib.psw_block_pool_admit.argtypes = [vp, i32p, i32, i32p, i32, i32p]
        lib.psw_block_pool_commit.argtypes = [vp, i32p, i32, i32p]
        for name in ("psw_block_pool_create", "psw_block_pool_allocate", "psw_block_pool_free",
                     "psw_block_pool_get_cached", "psw_block_pool_cache",
                     "psw_block_pool_ref_count", "psw_block_pool_admit",
                     "psw_block_pool_commit"):
            getattr(lib, name).restype = ctypes.c_int
        lib.kv_cache_write_fp8.argtypes = [lp, vp, vp, vp, vp, i32, pp, vp, vp, vp, vp, vp]
        lib.kv_cache_write_fp8.restype = ctypes.c_int
        lib.attn_decode_paged_fp8.argtypes = [lp, vp, vp, vp, vp, vp, pp, vp, i32, vp, vp, vp, sz,
                                              vp]
        lib.attn_decode_paged_fp8.restype = ctypes.c_int
        lib.attn_decode_paged_append.argtypes = [lp, vp, vp, vp, vp, vp, pp, vp, i32, vp, vp, vp,
                                                 sz, vp]
        lib.attn_decode_paged_append.restype = ctypes.c_int
        lib.psw_testing_stall.argtypes = [i32, i32, i32]
        lib.psw_testing_stall.restype = ctypes.c_int
        lib.psw_get_error.argtypes = [vp, ctypes.POINTER(i32)]
        lib.psw_strerror.argtypes = [ctypes.c_int]
        lib.psw_strerror.restype = ctypes.c_char_p
        for name in ("psw_workspace_bytes", "kv_cache_write", "attn_decode_paged",
                     "attn_prefill_chunked", "psw_get_error"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def strerror(code: int) -> str:
    try:
        return load(build_if_missing=False).psw_strerror(int(code)).decode()
    except Exception:
        return ERRORS.get(code, str(code))


def make_layer(layer) -> PswLayer:
    """From any object with the psw_layer_t fields (e.g. workloads.Layer)."""
    return PswLayer(int(layer.n_q_heads), int(layer.n_kv_heads), int(layer.head_dim),
                    int(layer.window), float(layer.softcap), float(layer.scale),
                    int(bool(layer.k_eq_v)), int(getattr(layer, "block_size", 16)))


def make_pages(block_table: torch.Tensor, num_blocks: int) -> PswPages:
    _check(block_table, torch.int32, "block_table")
    return PswPages(block_table.data_ptr(), int(block_table.shape[1]), int(num_blocks))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _raise(rc, what):
    if rc != PSW_OK:
        raise PswError(rc, what)


def workspace_bytes(layer, n_seqs: int, max_seq_len: int) -> int:
    out = ctypes.c_size_t(0)
    _raise(load().psw_workspace_bytes(ctypes.byref(make_layer(layer)), int(n_seqs),
                                      int(max_seq_len), ctypes.byref(out)), "psw_workspace_bytes")
    return int(out.value)


WORKSPACE_COUNTER_BYTES = 2048  # PSW_WORKSPACE_COUNTER_BYTES


def alloc_workspace(layer, n_seqs: int, max_seq_len: int, device="cuda") -> torch.Tensor:
    """A caller-owned workspace of the size the library asks for, zero-filled
    once (its counter block must start at zero; calls keep it zero)."""
    return torch.zeros(max(workspace_bytes(layer, n_seqs, max_seq_len), 256), dtype=torch.uint8,
                       device=device)


def kv_cache_write(layer, k, v, cu_new, past_lens, pages: PswPages, k_pool, v_pool,
                   stream=None) -> None:
    for t, n in ((k, "k"), (v, "v"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        _check(t, torch.bfloat16, n)
    _check(cu_new, torch.int32, "cu_new")
    _check(past_lens, torch.int32, "past_lens")
    rc = load().kv_cache_write(ctypes.byref(make_layer(layer)), _ptr(k), _ptr(v), _ptr(cu_new),
                               _ptr(past_lens), int(past_lens.shape[0]), ctypes.byref(pages),
                               _ptr(k_pool), _ptr(v_pool), _stream(stream))
    _raise(rc, "kv_cache_write")


def attn_decode_paged(layer, q, k_pool, v_pool, pages: PswPages, seq_lens, out, lse=None,
                      ws=None, stream=None) -> None:
    _check(q, torch.bfloat16, "q")
    _check(k_pool, torch.bfloat16, "k_pool")
    _check(v_pool, torch.bfloat16, "v_pool")
    _check(seq_lens, torch.int32, "seq_lens")
    _check(out, torch.float32, "out")
    _check(lse, torch.float32, "lse")
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = load().attn_decode_paged(ctypes.byref(make_layer(layer)), _ptr(q), _ptr(k_pool),
                                  _ptr(v_pool), ctypes.byref(pages), _ptr(seq_lens),
                                  int(seq_lens.shape[0]), _ptr(out), _ptr(lse), _ptr(ws),
                                  ws_bytes, _stream(stream))
    _raise(rc, "attn_decode_paged")


def attn_prefill_chunked(layer, q, cu_q, past_lens, max_q_len: int, k_pool, v_pool,
                         pages: PswPages, out, lse=None, ws=None, stream=None) -> None:
    _check(q, torch.bfloat16, "q")
    _check(cu_q, torch.int32, "cu_q")
    _check(past_lens, torch.int32, "past_lens")
    _check(k_pool, torch.bfloat16, "k_pool")
    _check(v_pool, torch.bfloat16, "v_pool")
    _check(out, torch.float32, "out")
    _check(lse, torch.float32, "lse")
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = load().attn_prefill_chunked(ctypes.byref(make_layer(layer)), _ptr(q), _ptr(cu_q),
                                     _ptr(past_lens), int(past_lens.shape[0]), int(q.shape[0]),
                                     int(max_q_len),
                                     _ptr(k_pool), _ptr(v_pool), ctypes.byref(pages), _ptr(out),
                                     _ptr(lse), _ptr(ws), ws_bytes, _stream(stream))
    _raise(rc, "attn_prefill_chunked")


def attn_decode_paged_noalloc(layer, q, k_pool, v_pool, pages: PswPages, seq_lens, out,
                              lse=None, stream=None) -> None:
    """attn_decode_paged without a workspace, for callers that cannot allocate
    device memory: the library uses its own static device buffer (see
    include/psw.h for the size limit and the rule that overlapping calls race)."""
    _check(q, torch.bfloat16, "q")
    _check(k_pool, torch.bfloat16, "k_pool")
    _check(v_pool, torch.bfloat16, "v_pool")
    _check(seq_lens, torch.int32, "seq_lens")
    _check(out, torch.float32, "out")
    _check(lse, torch.float32, "lse")
    rc = load().attn_decode_paged_noalloc(ctypes.byref(make_layer(layer)), _ptr(q),
                                          _ptr(k_pool), _ptr(v_pool), ctypes.byref(pages),
                                          _ptr(seq_lens), int(seq_lens.shape[0]), _ptr(out),
                                          _ptr(lse), _stream(stream))
    _raise(rc, "attn_decode_paged_noalloc")


def attn_decode_paged_append(layer, q, k_new, v_new, k_pool, v_pool, pages: PswPages, seq_lens,
                             out, lse=None, ws=None, stream=None) -> None:
    """One decode step in one launch: each sequence's new K/V row written at
    position seq_len - 1 and attended to (kv_cache_write + attn_decode_paged)."""
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_pool, "k_pool"),
                 (v_pool, "v_pool")):
        _check(t, torch.bfloat16, n)
    _check(seq_lens, torch.int32, "seq_lens")
    _check(out, torch.float32, "out")
    _check(lse, torch.float32, "lse")
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = load().attn_decode_paged_append(ctypes.byref(make_layer(layer)), _ptr(q), _ptr(k_new),
                                         _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                         ctypes.byref(pages), _ptr(seq_lens),
                                         int(seq_lens.shape[0]), _ptr(out), _ptr(lse), _ptr(ws),
                                         ws_bytes, _stream(stream))
    _raise(rc, "attn_decode_paged_append")


def kv_cache_write_fp8(layer, k, v, cu_new, past_lens, pages: PswPages, k_pool8, v_pool8,
                       k_scale, v_scale, stream=None) -> None:
    """kv_cache_write into FP8 pools (uint8 codes, fp32 per-row scales)."""
    _check(k, torch.bfloat16, "k")
    _check(v, torch.bfloat16, "v")
    _check(k_pool8, torch.uint8, "k_pool8")
    _check(v_pool8, torch.uint8, "v_pool8")
    _check(k_scale, torch.float32, "k_scale")
    _check(v_scale, torch.float32, "v_scale")
    _check(cu_new, torch.int32, "cu_new")
    _check(past_lens, torch.int32, "past_lens")
    rc = load().kv_cache_write_fp8(ctypes.byref(make_layer(layer)), _ptr(k), _ptr(v),
                                   _ptr(cu_new), _ptr(past_lens), int(past_lens.shape[0]),
                                   ctypes.byref(pages), _ptr(k_pool8), _ptr(v_pool8),
                                   _ptr(k_scale), _ptr(v_scale), _stream(stream))
    _raise(rc, "kv_cache_write_fp8")


def attn_decode_paged_fp8(layer, q, k_pool8, v_pool8, k_scale, v_scale, pages: PswPages,
                          seq_lens, out, lse=None, ws=None, stream=None) -> None:
    """attn_decode_paged over FP8 pools."""
    _check(q, torch.bfloat16, "q")
    _check(k_pool8, torch.uint8, "k_pool8")
    _check(v_pool8, torch.uint8, "v_pool8")
    _check(k_scale, torch.float32, "k_scale")
    _check(v_scale, torch.float32, "v_scale")
    _check(seq_lens, torch.int32, "seq_lens")
    _check(out, torch.float32, "out")
    _check(lse, torch.float32, "lse")
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = load().attn_decode_paged_fp8(ctypes.byref(make_layer(layer)), _ptr(q), _ptr(k_pool8),
                                      _ptr(v_pool8), _ptr(k_scale), _ptr(v_scale),
                                      ctypes.byref(pages), _ptr(seq_lens),
                                      int(seq_lens.shape[0]), _ptr(out), _ptr(lse), _ptr(ws),
                                      ws_bytes, _stream(stream))
    _raise(rc, "attn_decode_paged_fp8")


STALL_OFF, STALL_DECODE, STALL_PREFILL = 0, 1, 2


def testing_stall(kernel: int, cta: int = -1, tile: int = -1) -> None:
    """Testing hook: CTA `cta` of the next launches of `kernel` leaves its
    tile copy `tile` unissued, so a bounded wait runs out (STALL_OFF: off)."""
    _raise(load().psw_testing_stall(kernel, cta, tile), "psw_testing_stall")


def make_norm_rope(theta: float, partial_rotary_factor: float = 1.0, eps: float = 1e-6,
                   q_weight=None, k_weight=None, v_weight=None) -> PswNormRope:
    """psw_norm_rope_t from device fp32 weight tensors (or None)."""
    for t, n in ((q_weight, "q_weight"), (k_weight, "k_weight"), (v_weight, "v_weight")):
        _check(t, torch.float32, n)
    return PswNormRope(float(theta), float(partial_rotary_factor), float(eps),
                       None if q_weight is None else q_weight.data_ptr(),
                       None if k_weight is None else k_weight.data_ptr(),
                       None if v_weight is None else v_weight.data_ptr())


def qkv_norm_rope_cache_write(layer, rn: PswNormRope, q, k, v, cu_new, past_lens,
                              pages: PswPages | None, q_out, k_pool, v_pool,
                              stream=None) -> None:
    """The fused pre-attention step (per-head RMS-norm, proportional RoPE of q
    and k, cache write of k and v). k = v = pools = None processes q only."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (q_out, "q_out"), (k_pool, "k_pool"),
                 (v_pool, "v_pool")):
        _check(t, torch.bfloat16, n)
    _check(cu_new, torch.int32, "cu_new")
    _check(past_lens, torch.int32, "past_lens")
    rc = load().qkv_norm_rope_cache_write(
        ctypes.byref(make_layer(layer)), ctypes.byref(rn), _ptr(q), _ptr(k), _ptr(v),
        _ptr(cu_new), _ptr(past_lens), int(past_lens.shape[0]),
        None if pages is None else ctypes.byref(pages), _ptr(q_out), _ptr(k_pool), _ptr(v_pool),
        _stream(stream))
    _raise(rc, "qkv_norm_rope_cache_write")


def kv_share_map(n_layers: int, pattern: int, n_shared: int = 0):
    """(is_full, target) lists of a hybrid stack (psw_kv_share_map): layer i is
    full when (i + 1) % pattern == 0; the last n_shared layers read the cache of
    the last cache-owning layer of their type."""
    full = (ctypes.c_int32 * n_layers)()
    tgt = (ctypes.c_int32 * n_layers)()
    _raise(load().psw_kv_share_map(int(n_layers), int(pattern), int(n_shared), full, tgt),
           "psw_kv_share_map")
    return [bool(x) for x in full], [int(x) for x in tgt]


def _i32_array(values):
    arr = (ctypes.c_int32 * max(1, len(values)))(*[int(v) for v in values])
    return arr


def block_hash(parent: int, tokens) -> int:
    """psw_block_hash: chained FNV-1a hash of one page's tokens."""
    return int(load().psw_block_hash(int(parent), _i32_array(tokens), len(tokens)))


class BlockPool:
    """Host page allocator with prefix caching (psw_block_pool_*): ctypes
    marshalling only; the pool lives in libpsw."""

    def __init__(self, num_blocks: int, prefix_cache: bool = True):
        self._lib = load()
        h = ctypes.c_void_p()
        _raise(self._lib.psw_block_pool_create(int(num_blocks), int(bool(prefix_cache)),
                                               ctypes.byref(h)), "psw_block_pool_create")
        self._h = h

    def close(self):
        if self._h:
            self._lib.psw_block_pool_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return int(self._lib.psw_block_pool_num_free(self._h))

    def allocate(self, n: int):
        """(status, ids)."""
        out = (ctypes.c_int32 * max(1, n))()
        rc = self._lib.psw_block_pool_allocate(self._h, int(n), out)
        return rc, (list(out[:n]) if rc == PSW_OK else [])

    def release(self, ids) -> int:
        return self._lib.psw_block_pool_free(self._h, _i32_array(ids), len(ids))

    def get_cached(self, h: int) -> int:
        out = ctypes.c_int32(-1)
        _raise(self._lib.psw_block_pool_get_cached(self._h, int(h), ctypes.byref(out)),
               "psw_block_pool_get_cached")
        return int(out.value)

    def cache(self, block: int, h: int) -> int:
        return self._lib.psw_block_pool_cache(self._h, int(block), int(h))

    def ref_count(self, block: int) -> int:
        out = ctypes.c_int32(0)
        _raise(self._lib.psw_block_pool_ref_count(self._h, int(block), ctypes.byref(out)),
               "psw_block_pool_ref_count")
        return int(out.value)

    def admit(self, tokens, max_blocks: int):
        """(status, block-table row, tokens whose KV is already cached)."""
        row = (ctypes.c_int32 * max(1, max_blocks))()
        cached = ctypes.c_int32(0)
        rc = self._lib.psw_block_pool_admit(self._h, _i32_array(tokens), len(tokens), row,
                                            int(max_blocks), ctypes.byref(cached))
        return rc, (list(row[:max_blocks]) if rc == PSW_OK else None), int(cached.value)

    def commit(self, tokens, row) -> int:
        return self._lib.psw_block_pool_commit(self._h, _i32_array(tokens), len(tokens),
                                               _i32_array(row))


def get_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error word."""
    val = ctypes.c_int32(0)
    _raise(load().psw_get_error(_stream(stream), ctypes.byref(val)), "psw_get_error")
    return int(val.value)
