"""Plain fp64 CPU oracle for paged sliding-window attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code
with the CUDA library (``paged_sliding_window_gb300``) and never imports it;
the library never imports this package.

The arithmetic lives in ``psw_oracle.c`` (plain C, double precision, one
pthread per core). This module only compiles it with gcc, marshals numpy
arrays and maps the two operations onto query rows:

* decode: the query of sequence ``b`` sits at absolute position
  ``seq_len[b] - 1`` (the sliding-window decode tail of InfiniLM PR 581,
  Gemma-3 item 3: only the last ``min(total, W)`` keys are read);
* chunked prefill: chunk row ``i`` of sequence ``b`` sits at
  ``past_len[b] + i`` (same passage: the band rule composed with the aligned
  causal rule).

bf16 tensors are passed as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "psw_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpsw_oracle.so")

_lock = threading.Lock()
_default = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)


def compile_source(src_path: str, lib_path: str) -> str:
    """gcc -O2 a C source of the oracle into a shared library."""
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-o", tmp, src_path, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib_path)
    return lib_path


def build(force: bool = False) -> str:
    """Compile psw_oracle.c into a shared library with gcc; returns its path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _ptr(a, ctype):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctype))
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_slot.restype = ctypes.c_int64
        lib.oracle_slot.argtypes = [_i32p, ctypes.c_int64, ctypes.c_int32]
        lib.oracle_kv_cache_bytes.restype = ctypes.c_double
        lib.oracle_kv_cache_bytes.argtypes = [ctypes.c_int64] * 6 + [ctypes.c_int32]
        lib.oracle_kv_cache_write.restype = ctypes.c_int32
        lib.oracle_kv_cache_write.argtypes = [
            _u16p, _u16p, _i32p, _i32p, ctypes.c_int32, _i32p, ctypes.c_int32,
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            _u16p, _u16p]
        lib.oracle_num_cores.restype = ctypes.c_int32
        lib.oracle_num_cores.argtypes = []
        lib.oracle_norm_rope_row.restype = None
        lib.oracle_norm_rope_row.argtypes = [
            _u16p, ctypes.c_int32, ctypes.c_double, _f32p, ctypes.c_int32, ctypes.c_double,
            ctypes.c_int32, ctypes.c_int64, _f64p]
        lib.oracle_to_bf16.restype = ctypes.c_uint16
        lib.oracle_to_bf16.argtypes = [ctypes.c_double]
        _u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_e4m3_encode_array.argtypes = [_f32p, _u8p, ctypes.c_int64]
        lib.oracle_e4m3_decode_array.restype = None
        lib.oracle_e4m3_decode_array.argtypes = [_u8p, _f64p, ctypes.c_int64]
        lib.oracle_kv_cache_write_fp8.restype = ctypes.c_int32
        lib.oracle_kv_cache_write_fp8.argtypes = [
            _u16p, _u16p, _i32p, _i32p, ctypes.c_int32, _i32p, ctypes.c_int32,
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            _u8p, _u8p, _f32p, _f32p]
        lib.oracle_attention_rows_fp8.restype = ctypes.c_int32
        lib.oracle_attention_rows_fp8.argtypes = [
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_double, ctypes.c_double, ctypes.c_int32, ctypes.c_int32,
            _u16p, _i32p, _i64p, ctypes.c_int64, _u8p, _u8p, _f32p, _f32p, _i32p,
            ctypes.c_int32, _f64p, _f64p, ctypes.c_int32]
        lib.oracle_to_bf16_array.restype = None
        lib.oracle_to_bf16_array.argtypes = [_f64p, _u16p, ctypes.c_int64]
        lib.oracle_qkv_norm_rope.restype = None
        lib.oracle_qkv_norm_rope.argtypes = [
            _u16p, _u16p, _u16p, _i32p, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_double, _f32p, _f32p, _f32p, ctypes.c_double,
            ctypes.c_int32, _f64p, _f64p, _f64p]
        lib.oracle_attention_rows.restype = ctypes.c_int32
        lib.oracle_attention_rows.argtypes = [
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_double, ctypes.c_double, ctypes.c_int32, ctypes.c_int32,
            _u16p, _i32p, _i64p, ctypes.c_int64, _u16p, _u16p, _i32p,
            ctypes.c_int32, _f64p, _f64p, ctypes.c_int32]
        self.lib = lib
        self.path = lib_path

    def num_cores(self) -> int:
        return int(self.lib.oracle_num_cores())

    def slot(self, block_table_row, pos: int, block_size: int) -> int:
        """Physical slot of logical position ``pos`` (vLLM compute_slot_mapping)."""
        row = np.ascontiguousarray(block_table_row, dtype=np.int32)
        return int(self.lib.oracle_slot(_ptr(row, ctypes.c_int32), int(pos), int(block_size)))

    def kv_cache_bytes(self, batch, seq_len, n_layers, n_kv_heads, head_dim, dtype_bytes,
                       with_v: bool = True) -> float:
        return float(self.lib.oracle_kv_cache_bytes(batch, seq_len, n_layers, n_kv_heads,
                                                    head_dim, dtype_bytes, int(with_v)))

    def kv_cache_write(self, k_new, v_new, cu_new, past_lens, block_table, k_pool, v_pool,
                       block_size: int = 16, in_place: bool = False):
        """Returns (k_pool', v_pool', status): the pools with the new rows
        written (copies, or the given arrays themselves when ``in_place``).
        ``v_pool`` None means V aliases the K pages."""
        k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
        cu_new = np.ascontiguousarray(cu_new, dtype=np.int32)
        past_lens = np.ascontiguousarray(past_lens, dtype=np.int32)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        if in_place:
            assert k_pool.dtype == np.uint16 and k_pool.flags["C_CONTIGUOUS"]
            k_out, v_out = k_pool, v_pool
        else:
            k_out = np.array(k_pool, dtype=np.uint16, copy=True, order="C")
            v_out = None if v_pool is None else np.array(v_pool, dtype=np.uint16, copy=True,
                                                         order="C")
        v_new_c = None if v_pool is None else np.ascontiguousarray(v_new, dtype=np.uint16)
        n_seqs = past_lens.shape[0]
        num_blocks, bs, n_kv, hd = k_out.shape
        assert bs == block_size
        status = self.lib.oracle_kv_cache_write(
            _ptr(k_new, ctypes.c_uint16), _ptr(v_new_c, ctypes.c_uint16),
            _ptr(cu_new, ctypes.c_int32), _ptr(past_lens, ctypes.c_int32), n_seqs,
            _ptr(block_table, ctypes.c_int32), block_table.shape[1], num_blocks,
            n_kv, hd, block_size, _ptr(k_out, ctypes.c_uint16), _ptr(v_out, ctypes.c_uint16))
        return k_out, v_out, int(status)

    def attention_rows(self, layer: dict, q_rows, row_seq, row_pos, k_pool, v_pool,
                       block_table, threads: int = 0):
        """Attention for explicit query rows. Returns (out fp64 [n_rows, n_q, hd],
        lse fp64 [n_rows, n_q], threads_used)."""
        q_rows = np.ascontiguousarray(q_rows, dtype=np.uint16)
        row_seq = np.ascontiguousarray(row_seq, dtype=np.int32)
        row_pos = np.ascontiguousarray(row_pos, dtype=np.int64)
        k_pool = np.ascontiguousarray(k_pool, dtype=np.uint16)
        v_pool = None if v_pool is None else np.ascontiguousarray(v_pool, dtype=np.uint16)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        n_rows = row_pos.shape[0]
        n_q, hd = int(layer["n_q_heads"]), int(layer["head_dim"])
        out = np.zeros((n_rows, n_q, hd), dtype=np.float64)
        lse = np.zeros((n_rows, n_q), dtype=np.float64)
        if n_rows == 0:
            return out, lse, 0
        used = self.lib.oracle_attention_rows(
            n_q, int(layer["n_kv_heads"]), hd, int(layer["window"]),
            float(layer["softcap"]), float(layer["scale"]), int(layer["k_eq_v"]),
            int(layer.get("block_size", 16)),
            _ptr(q_rows, ctypes.c_uint16), _ptr(row_seq, ctypes.c_int32),
            _ptr(row_pos, ctypes.c_int64), n_rows, _ptr(k_pool, ctypes.c_uint16),
            _ptr(v_pool, ctypes.c_uint16), _ptr(block_table, ctypes.c_int32),
            block_table.shape[1], _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
            int(threads))
        if used < 0:
            raise ValueError(f"oracle_attention_rows failed ({used})")
        return out, lse, int(used)

    def decode(self, layer: dict, q, k_pool, v_pool, block_table, seq_lens, seqs=None,
               threads: int = 0):
        """Decode attention: one query per sequence at position seq_len - 1.

        q: [n_seqs, n_q, hd] bf16 bits. ``seqs`` optionally restricts the rows
        to a subset of sequences (outputs follow that order)."""
        seq_lens = np.asarray(seq_lens, dtype=np.int64)
        idx = np.arange(seq_lens.shape[0]) if seqs is None else np.asarray(seqs, dtype=np.int64)
        row_pos = seq_lens[idx] - 1
        return self.attention_rows(layer, np.asarray(q)[idx], idx.astype(np.int32), row_pos,
                                   k_pool, v_pool, block_table, threads)

    def prefill(self, layer: dict, q, cu_q, past_lens, k_pool, v_pool, block_table,
                rows=None, threads: int = 0):
        """Chunked-prefill attention: chunk row i of sequence b sits at past_b + i.

        q: [n_q_total, n_q, hd] bf16 bits; cu_q: [n_seqs + 1] offsets. ``rows``
        optionally restricts the computation to a subset of flat row indices."""
        cu_q = np.asarray(cu_q, dtype=np.int64)
        past_lens = np.asarray(past_lens, dtype=np.int64)
        n_total = int(cu_q[-1])
        seq_of_row = np.searchsorted(cu_q, np.arange(n_total), side="right") - 1
        idx = np.arange(n_total) if rows is None else np.asarray(rows, dtype=np.int64)
        seq = seq_of_row[idx]
        row_pos = past_lens[seq] + (idx - cu_q[seq])
        return self.attention_rows(layer, np.asarray(q)[idx], seq.astype(np.int32), row_pos,
                                   k_pool, v_pool, block_table, threads)


    # ---------------------------------------------------------- pre-attention step
    def norm_rope_row(self, x, eps: float, weight=None, rotate: bool = True,
                      theta: float = 10000.0, rope_angles: int | None = None, pos: int = 0):
        """One head vector (bf16 bits): RMS-norm (optional weight), then the
        proportional rotary embedding at ``pos`` when ``rotate``. fp64 out."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        hd = x.shape[-1]
        ra = hd // 2 if rope_angles is None else int(rope_angles)
        w = None if weight is None else np.ascontiguousarray(weight, dtype=np.float32)
        out = np.zeros(hd, dtype=np.float64)
        self.lib.oracle_norm_rope_row(_ptr(x, ctypes.c_uint16), hd, float(eps),
                                      _ptr(w, ctypes.c_float), int(bool(rotate)), float(theta),
                                      ra, int(pos), _ptr(out, ctypes.c_double))
        return out

    def qkv_norm_rope(self, q, k, v, cu_new, past_lens, eps: float, theta: float,
                      rope_angles: int, q_w=None, k_w=None, v_w=None):
        """The pre-attention step of one layer: returns (q_out, k_rows, v_rows)
        in fp64 (k_rows / v_rows None when k / v is None)."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        n_tok, n_q, hd = q.shape
        cu_new = np.ascontiguousarray(cu_new, dtype=np.int32)
        past_lens = np.ascontiguousarray(past_lens, dtype=np.int32)
        k = None if k is None else np.ascontiguousarray(k, dtype=np.uint16)
        v = None if v is None else np.ascontiguousarray(v, dtype=np.uint16)
        n_kv = k.shape[1] if k is not None else (v.shape[1] if v is not None else 1)
        ws = [None if w is None else np.ascontiguousarray(w, dtype=np.float32)
              for w in (q_w, k_w, v_w)]
        q_out = np.zeros((n_tok, n_q, hd), dtype=np.float64)
        k_rows = None if k is None else np.zeros((n_tok, n_kv, hd), dtype=np.float64)
        v_rows = None if v is None else np.zeros((n_tok, n_kv, hd), dtype=np.float64)
        self.lib.oracle_qkv_norm_rope(
            _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
            _ptr(cu_new, ctypes.c_int32), _ptr(past_lens, ctypes.c_int32),
            past_lens.shape[0], n_q, n_kv, hd, float(eps),
            _ptr(ws[0], ctypes.c_float), _ptr(ws[1], ctypes.c_float),
            _ptr(ws[2], ctypes.c_float), float(theta), int(rope_angles),
            _ptr(q_out, ctypes.c_double), _ptr(k_rows, ctypes.c_double),
            _ptr(v_rows, ctypes.c_double))
        return q_out, k_rows, v_rows

    def to_bf16(self, values) -> np.ndarray:
        """Round fp64 values to bf16 bits (nearest, ties to even)."""
        a = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.oracle_to_bf16_array(_ptr(a, ctypes.c_double), _ptr(out, ctypes.c_uint16),
                                      a.size)
        return out


    # ---------------------------------------------------------- FP8 pages
    def e4m3_encode(self, x) -> np.ndarray:
        """OCP E4M3 codes of float32 values (nearest even, saturating at 448)."""
        a = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(a.shape, dtype=np.uint8)
        self.lib.oracle_e4m3_encode_array(_ptr(a, ctypes.c_float), _ptr(out, ctypes.c_uint8),
                                          a.size)
        return out

    def e4m3_decode(self, codes) -> np.ndarray:
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(c.shape, dtype=np.float64)
        self.lib.oracle_e4m3_decode_array(_ptr(c, ctypes.c_uint8), _ptr(out, ctypes.c_double),
                                          c.size)
        return out

    def kv_cache_write_fp8(self, k_new, v_new, cu_new, past_lens, block_table, k8, v8,
                           k_scale, v_scale, block_size: int = 16) -> int:
        """Quantised cache write into FP8 pools (uint8 [nb, bs, n_kv, hd]) and
        scale pools (fp32 [nb, bs, n_kv]), in place. v8 None: K only."""
        k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
        v_new = None if v8 is None else np.ascontiguousarray(v_new, dtype=np.uint16)
        cu_new = np.ascontiguousarray(cu_new, dtype=np.int32)
        past_lens = np.ascontiguousarray(past_lens, dtype=np.int32)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        for a in (k8, v8, k_scale, v_scale):
            assert a is None or a.flags["C_CONTIGUOUS"]
        num_blocks, bs, n_kv, hd = k8.shape
        return int(self.lib.oracle_kv_cache_write_fp8(
            _ptr(k_new, ctypes.c_uint16), _ptr(v_new, ctypes.c_uint16),
            _ptr(cu_new, ctypes.c_int32), _ptr(past_lens, ctypes.c_int32), past_lens.shape[0],
            _ptr(block_table, ctypes.c_int32), block_table.shape[1], num_blocks, n_kv, hd,
            block_size, _ptr(k8, ctypes.c_uint8), _ptr(v8, ctypes.c_uint8),
            _ptr(k_scale, ctypes.c_float), _ptr(v_scale, ctypes.c_float)))

    def decode_fp8(self, layer: dict, q, k8, v8, k_scale, v_scale, block_table, seq_lens,
                   seqs=None, threads: int = 0):
        """Decode attention over FP8 pages (values code * scale)."""
        seq_lens = np.asarray(seq_lens, dtype=np.int64)
        idx = np.arange(seq_lens.shape[0]) if seqs is None else np.asarray(seqs, dtype=np.int64)
        q_rows = np.ascontiguousarray(np.asarray(q)[idx], dtype=np.uint16)
        row_seq = np.ascontiguousarray(idx.astype(np.int32))
        row_pos = np.ascontiguousarray(seq_lens[idx] - 1, dtype=np.int64)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        n_rows = row_pos.shape[0]
        n_q, hd = int(layer["n_q_heads"]), int(layer["head_dim"])
        out = np.zeros((n_rows, n_q, hd), dtype=np.float64)
        lse = np.zeros((n_rows, n_q), dtype=np.float64)
        if n_rows == 0:
            return out, lse, 0
        used = self.lib.oracle_attention_rows_fp8(
            n_q, int(layer["n_kv_heads"]), hd, int(layer["window"]), float(layer["softcap"]),
            float(layer["scale"]), int(layer["k_eq_v"]), int(layer.get("block_size", 16)),
            _ptr(q_rows, ctypes.c_uint16), _ptr(row_seq, ctypes.c_int32),
            _ptr(row_pos, ctypes.c_int64), n_rows, _ptr(k8, ctypes.c_uint8),
            _ptr(v8, ctypes.c_uint8), _ptr(k_scale, ctypes.c_float),
            _ptr(v_scale, ctypes.c_float), _ptr(block_table, ctypes.c_int32),
            block_table.shape[1], _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
            int(threads))
        if used < 0:
            raise ValueError(f"oracle_attention_rows_fp8 failed ({used})")
        return out, lse, int(used)


def default() -> Oracle:
    """The oracle built from psw_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def num_cores() -> int:
    return default().num_cores()


def slot(block_table_row, pos, block_size):
    return default().slot(block_table_row, pos, block_size)


def kv_cache_bytes(*args, **kw):
    return default().kv_cache_bytes(*args, **kw)


def kv_cache_write(*args, **kw):
    return default().kv_cache_write(*args, **kw)


def attention_rows(*args, **kw):
    return default().attention_rows(*args, **kw)


def decode(*args, **kw):
    return default().decode(*args, **kw)


def prefill(*args, **kw):
    return default().prefill(*args, **kw)


def norm_rope_row(*args, **kw):
    return default().norm_rope_row(*args, **kw)


def qkv_norm_rope(*args, **kw):
    return default().qkv_norm_rope(*args, **kw)


def to_bf16(values):
    return default().to_bf16(values)


def kv_cache_write_fp8(*args, **kw):
    return default().kv_cache_write_fp8(*args, **kw)


def decode_fp8(*args, **kw):
    return default().decode_fp8(*args, **kw)
