"""Stages a seeded workload step on the GPU for the C ABI: device copies of
the step's inputs, canary-filled pools with the retained history written by
the library's own kv_cache_write, output buffers and the workspace. Used by
the benchmark and the GPU tests; all compute goes through ``binding``."""
from __future__ import annotations

import numpy as np
import torch

from . import binding
from . import workloads as wl


def dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def dev_i32(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


class GpuStep:
    """Device copies of one step's inputs plus pools with the history written."""

    def __init__(self, step: wl.Step, device="cuda"):
        self.step = step
        layer = step.layer
        c = step.cache
        shape = c.pool_shape
        canary = int(wl.CANARY_BF16)  # < 0x8000, so the same bits as int16
        self.k_pool = torch.full(shape, canary, dtype=torch.int16, device=device).view(torch.bfloat16)
        self.v_pool = None if layer.k_eq_v else torch.full(
            shape, canary, dtype=torch.int16, device=device).view(torch.bfloat16)
        self.table = dev_i32(step.block_table, device)
        self.pages = binding.make_pages(self.table, c.num_blocks)
        if c.hist_k.shape[0] > 0:
            binding.kv_cache_write(layer, dev_bf16(c.hist_k, device),
                                   None if layer.k_eq_v else dev_bf16(c.hist_v, device),
                                   dev_i32(c.hist_cu, device), dev_i32(c.hist_past, device),
                                   self.pages, self.k_pool, self.v_pool)
        self.q = dev_bf16(step.q, device)
        self.new_k = dev_bf16(step.new_k, device)
        self.new_v = None if layer.k_eq_v else dev_bf16(step.new_v, device)
        self.cu_new = dev_i32(step.cu_new, device)
        self.past = dev_i32(step.past_lens, device)
        self.seq_lens = dev_i32(step.seq_lens, device)
        n_rows = step.q.shape[0]
        self.out = torch.full((n_rows, layer.n_q_heads, layer.head_dim), float("nan"),
                              dtype=torch.float32, device=device)
        self.lse = torch.full((n_rows, layer.n_q_heads), float("nan"), dtype=torch.float32,
                              device=device)
        max_len = int(step.seq_lens.max()) if step.n_seqs else 0
        self.ws = binding.alloc_workspace(layer, step.n_seqs, max_len, device)

    def write_new(self):
        binding.kv_cache_write(self.step.layer, self.new_k, self.new_v, self.cu_new, self.past,
                               self.pages, self.k_pool, self.v_pool)

    def decode(self):
        binding.attn_decode_paged(self.step.layer, self.q, self.k_pool, self.v_pool, self.pages,
                                  self.seq_lens, self.out, self.lse, self.ws)

    def decode_append(self):
        """The fused step: writes the new rows and decodes (one new token per
        sequence, as in a decode step)."""
        binding.attn_decode_paged_append(self.step.layer, self.q, self.new_k, self.new_v,
                                         self.k_pool, self.v_pool, self.pages, self.seq_lens,
                                         self.out, self.lse, self.ws)

    def prefill(self):
        max_q = int(self.step.new_lens.max()) if self.step.n_seqs else 0
        binding.attn_prefill_chunked(self.step.layer, self.q, self.cu_new, self.past, max_q,
                                     self.k_pool, self.v_pool, self.pages, self.out, self.lse,
                                     self.ws)


class MixedLayerStep:
    """One layer of a mixed serving step on the GPU: the first ``n_decode``
    sequences decode one token each, the rest prefill a chunk. One cache write
    covers every new token; decode and prefill then run on their own rows of
    the shared block table."""

    def __init__(self, step: wl.Step, n_decode: int, device="cuda"):
        self.g = GpuStep(step, device)
        self.step, self.n_decode = step, n_decode
        g = self.g
        nd = n_decode
        self.dec_q = g.q[:nd]
        self.dec_lens = g.seq_lens[:nd]
        self.dec_out = g.out[:nd]
        self.dec_lse = g.lse[:nd]
        self.dec_table = g.table[:nd]
        self.dec_pages = binding.make_pages(self.dec_table, step.cache.num_blocks)
        row0 = int(step.cu_new[nd])
        self.pre_q = g.q[row0:]
        self.pre_cu = (g.cu_new[nd:] - row0).contiguous()
        self.pre_past = g.past[nd:].contiguous()
        self.pre_out = g.out[row0:]
        self.pre_lse = g.lse[row0:]
        self.pre_table = g.table[nd:].contiguous()
        self.pre_pages = binding.make_pages(self.pre_table, step.cache.num_blocks)
        self.max_chunk = int(step.new_lens[nd:].max()) if step.n_seqs > nd else 0

    def run(self):
        g, L = self.g, self.step.layer
        g.write_new()
        binding.attn_decode_paged(L, self.dec_q, g.k_pool, g.v_pool, self.dec_pages,
                                  self.dec_lens, self.dec_out, self.dec_lse, g.ws)
        binding.attn_prefill_chunked(L, self.pre_q, self.pre_cu, self.pre_past, self.max_chunk,
                                     g.k_pool, g.v_pool, self.pre_pages, self.pre_out,
                                     self.pre_lse, g.ws)


FP8_CANARY = 0x7F  # an E4M3 NaN code: a read of a never-written slot shows


class GpuStepFP8:
    """A step on FP8 pages: e4m3 code pools (canary-filled), fp32 scale pools
    (NaN-filled), the history written by the library's FP8 cache write."""

    def __init__(self, step: wl.Step, device="cuda"):
        self.step = step
        layer = step.layer
        c = step.cache
        shape = c.pool_shape
        self.k_pool8 = torch.full(shape, FP8_CANARY, dtype=torch.uint8, device=device)
        self.k_scale = torch.full(shape[:3], float("nan"), dtype=torch.float32, device=device)
        self.v_pool8 = None if layer.k_eq_v else torch.full(shape, FP8_CANARY, dtype=torch.uint8,
                                                            device=device)
        self.v_scale = None if layer.k_eq_v else torch.full(shape[:3], float("nan"),
                                                            dtype=torch.float32, device=device)
        self.table = dev_i32(step.block_table, device)
        self.pages = binding.make_pages(self.table, c.num_blocks)
        if c.hist_k.shape[0] > 0:
            binding.kv_cache_write_fp8(layer, dev_bf16(c.hist_k, device),
                                       None if layer.k_eq_v else dev_bf16(c.hist_v, device),
                                       dev_i32(c.hist_cu, device), dev_i32(c.hist_past, device),
                                       self.pages, self.k_pool8, self.v_pool8, self.k_scale,
                                       self.v_scale)
        self.q = dev_bf16(step.q, device)
        self.new_k = dev_bf16(step.new_k, device)
        self.new_v = None if layer.k_eq_v else dev_bf16(step.new_v, device)
        self.cu_new = dev_i32(step.cu_new, device)
        self.past = dev_i32(step.past_lens, device)
        self.seq_lens = dev_i32(step.seq_lens, device)
        n_rows = step.q.shape[0]
        self.out = torch.full((n_rows, layer.n_q_heads, layer.head_dim), float("nan"),
                              dtype=torch.float32, device=device)
        self.lse = torch.full((n_rows, layer.n_q_heads), float("nan"), dtype=torch.float32,
                              device=device)
        max_len = int(step.seq_lens.max()) if step.n_seqs else 0
        self.ws = binding.alloc_workspace(layer, step.n_seqs, max_len, device)

    def write_new(self):
        binding.kv_cache_write_fp8(self.step.layer, self.new_k, self.new_v, self.cu_new,
                                   self.past, self.pages, self.k_pool8, self.v_pool8,
                                   self.k_scale, self.v_scale)

    def decode(self):
        binding.attn_decode_paged_fp8(self.step.layer, self.q, self.k_pool8, self.v_pool8,
                                      self.k_scale, self.v_scale, self.pages, self.seq_lens,
                                      self.out, self.lse, self.ws)
