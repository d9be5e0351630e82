"""Helpers for the GPU parity tests: move generator output to the device, run the library
through its binding, and compare with the oracle under the stated tolerance."""
from __future__ import annotations

import os

import numpy as np

import workloads as W

# Tolerance for bf16 I/O with fp32 accumulation, against the fp32 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3

# Host threads for the oracle on full-size batches (each thread runs the single-threaded C oracle
# on its own rows; the arithmetic per row is unchanged).
ORACLE_THREADS = os.cpu_count() or 8


def torch_mod():
    import torch
    return torch


def dev_bf16(a: np.ndarray):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def dev_i32(a: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host_bits(t) -> np.ndarray:
    torch = torch_mod()
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f32(t) -> np.ndarray:
    return W.bf16_bits_to_f32(host_bits(t))


def compare(got: np.ndarray, want: np.ndarray, what: str = ""):
    """Assert max-abs <= 2e-2 and mean-abs <= 2e-3; return the stats (relative L2 too)."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - want)
    stats = {
        "max_abs": float(err.max()) if err.size else 0.0,
        "mean_abs": float(err.mean()) if err.size else 0.0,
        "rel_l2": float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)),
    }
    assert stats["max_abs"] <= MAX_ABS and stats["mean_abs"] <= MEAN_ABS, f"{what}: {stats}"
    return stats


class DeviceBatch:
    """A ``workloads.PagedBatch`` resident on the GPU (pool built from the block seeds)."""

    def __init__(self, batch: W.PagedBatch, kc: np.ndarray | None = None, vc: np.ndarray | None = None):
        torch = torch_mod()
        self.b = batch
        if kc is None:
            kc, vc = batch.cache()
        self.kc_host0, self.vc_host0 = kc, vc
        self.k_cache = dev_bf16(kc)
        self.v_cache = dev_bf16(vc)
        self.q = dev_bf16(batch.q)
        self.k_new = dev_bf16(batch.k_new)
        self.v_new = dev_bf16(batch.v_new)
        self.slot_mapping = dev_i32(batch.slot_mapping)
        self.block_tables = dev_i32(batch.block_tables)
        self.seq_lens = dev_i32(batch.seq_lens)
        self.cu_q = dev_i32(batch.cu_seqlens_q)
        self.cu_k = dev_i32(batch.cu_seqlens_k)
        self.d_err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def store(self):
        import paged_kv_attention_store_gb300 as nv
        nv.nv_store_kvcache(self.k_new, self.v_new, self.slot_mapping, self.k_cache, self.v_cache, d_err=self.d_err)

    def decode(self, max_context_len=None, q=None):
        import paged_kv_attention_store_gb300 as nv
        if max_context_len is None:
            max_context_len = int(self.b.seq_lens.max()) if self.b.num_seqs else 1
        return nv.nv_paged_decode_attn(self.q if q is None else q, self.k_cache, self.v_cache, self.block_tables,
                                       self.seq_lens, self.b.scale, max_context_len=max_context_len,
                                       d_err=self.d_err)

    def prefill(self, max_seqlen_q=None, q=None):
        import paged_kv_attention_store_gb300 as nv
        if max_seqlen_q is None:
            max_seqlen_q = int(self.b.q_lens.max())
        return nv.nv_paged_prefill_attn(self.q if q is None else q, self.k_cache, self.v_cache, self.cu_q, self.cu_k,
                                        self.block_tables, self.b.scale, max_seqlen_q=max_seqlen_q, d_err=self.d_err)

    def err(self) -> int:
        torch = torch_mod()
        torch.cuda.synchronize()
        return int(self.d_err.item())


def oracle_store_in_place(orc, batch, kc, vc):
    """The oracle's store applied to host caches in place (for multi-GB pools not needed afterwards)."""
    orc.store_kvcache(batch.k_new, batch.v_new, batch.slot_mapping, kc, vc)
    return kc, vc


def oracle_cache_after_store(orc, batch, kc, vc):
    kc, vc = kc.copy(), vc.copy()
    orc.store_kvcache(batch.k_new, batch.v_new, batch.slot_mapping, kc, vc)
    return kc, vc


def oracle_decode(orc, batch, kc, vc, threads=8):
    return orc.decode_attn(batch.q, kc, vc, batch.block_tables, batch.context_lens, batch.num_kv_heads,
                           batch.block_size, batch.scale, threads=threads)


def oracle_prefill(orc, batch, kc, vc, rows=None, threads=8):
    return orc.prefill_attn(batch.q, kc, vc, batch.cu_seqlens_q, batch.cu_seqlens_k, batch.block_tables,
                            batch.num_kv_heads, batch.block_size, batch.scale, rows=rows, threads=threads)
