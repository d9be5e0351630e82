#!/usr/bin/env python3
"""Benchmark of the paged KV attention store on GB300.

One JSON line on rank 0.  Two phases run in one invocation and together cover every step
of the hot path (slot scatter, paged decode attention, varlen prefill attention):

* decode phase (the headline line): K engine decode steps on the Qwen3-8B-shaped batch
  (512 sequences, context lengths U[1024, 4096], 32 q / 8 kv heads, head_dim 128, block
  size 256): store the 512 new K/V rows, then decode.  ``value`` is the KV bytes the
  decode attention must read per step (4096 B per attended position: K and V of 8 heads
  x 128 dims in bf16) times K, over the device time of the K steps: paged-decode KV GB/s.
* prefill phase (the ``prefill`` object): K engine prefill steps on the chunked-prefill
  workload (16 sequences, 16384 new tokens, cached prefixes 256*U{0..8}, 16 q / 8 kv
  heads): store the 16384 new rows, then causal prefill.  TFLOP/s counts the causally
  visible (query, key) pairs only: 4 * D * Hq per pair.

``--impl reference`` times the CPU oracle (the only reference implementation this project
has) on bounded samples of the same workloads.  Multi-GPU runs (torchrun) give every rank
its own batch (weak scaling; the path needs no collective): barrier + synchronize around
the timed region, max time over ranks, whole-job throughput on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "paged-decode KV GB/s (% of HBM peak); prefill attn TFLOP/s; attended tok/s"
KV_BYTES_PER_TOKEN_PER_KVHEAD = 128 * 2 * 2          # K and V rows of one kv head, bf16
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------------------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def decode_algorithmic_bytes(b: W.PagedBatch) -> int:
    """KV rows read + q read + out written + block-table entries and lengths read."""
    kv = int(b.seq_lens.astype(np.int64).sum()) * b.num_kv_heads * KV_BYTES_PER_TOKEN_PER_KVHEAD
    qo = 2 * b.num_seqs * b.num_q_heads * 128 * 2
    meta = sum(W.blocks_needed(int(L), b.block_size) for L in b.seq_lens) * 4 + b.num_seqs * 4
    return kv + qo + meta


def decode_kv_bytes(b: W.PagedBatch) -> int:
    return int(b.seq_lens.astype(np.int64).sum()) * b.num_kv_heads * KV_BYTES_PER_TOKEN_PER_KVHEAD


def prefill_pairs(b: W.PagedBatch) -> int:
    P = b.meta["prefix_lens"].astype(np.int64)
    Lq = b.q_lens.astype(np.int64)
    return int((Lq * P + Lq * (Lq + 1) // 2).sum())


def prefill_flops(b: W.PagedBatch) -> int:
    return 4 * 128 * b.num_q_heads * prefill_pairs(b)


def source_hash(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_attention_store_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key: str, sources) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_sha") != source_hash(*sources):
        return None
    return float(e["dram_bytes_per_launch"])


def reduce_over_ranks(x: float, op: str, world: int, device="cpu") -> float:
    """Max or sum of a host scalar over the ranks of the default process group (identity at 1 rank)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def measure_decode_config(batch: W.PagedBatch, steps: int, warmup: int, dev) -> dict:
    """Store + decode on another decode configuration; CUDA events around the decode call only."""
    import torch

    import paged_kv_attention_store_gb300 as nv

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    kc, vc = batch.cache()
    k_cache, v_cache = to_dev(kc), to_dev(vc)
    del kc, vc
    q, k_new, v_new, slots = to_dev(batch.q), to_dev(batch.k_new), to_dev(batch.v_new), to_dev(batch.slot_mapping)
    bt, lens = to_dev(batch.block_tables), to_dev(batch.seq_lens)
    out = torch.empty_like(q)
    maxc = int(batch.seq_lens.max())
    ws = torch.zeros(max(nv.nv_paged_decode_workspace_size(batch.num_seqs, batch.num_q_heads, 128, maxc), 16),
                     dtype=torch.uint8, device=dev)
    d_err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(warmup + steps):
        nv.nv_store_kvcache(k_new, v_new, slots, k_cache, v_cache, d_err=d_err)
        if i >= warmup:
            evs[i - warmup][0].record(stream)
        nv.nv_paged_decode_attn(q, k_cache, v_cache, bt, lens, batch.scale, out=out, max_context_len=maxc,
                                workspace=ws, d_err=d_err)
        if i >= warmup:
            evs[i - warmup][1].record(stream)
    torch.cuda.synchronize()
    assert int(d_err.item()) == 0, f"device error flags {int(d_err.item())}"
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    logical = decode_kv_bytes(batch)
    used = batch.used_blocks([i for i in range(batch.num_seqs) if batch.seq_lens[i] > 0])
    unique = len(used) * batch.block_size * batch.num_kv_heads * KV_BYTES_PER_TOKEN_PER_KVHEAD
    del k_cache, v_cache
    torch.cuda.empty_cache()
    return {"ms_per_decode": round(ms, 4),
            "attended_tok_s": round(float(batch.seq_lens.astype(np.int64).sum()) / (ms * 1e-3), 1),
            "logical_kv_gbs": round(logical / (ms * 1e-3) / 1e9, 1),
            "unique_kv_gbs": round(unique / (ms * 1e-3) / 1e9, 1),
            "logical_kv_bytes": logical, "unique_kv_bytes": unique}


def rank_decode_batch(rank: int, num_seqs: int = 512) -> W.PagedBatch:
    """Each rank's own Qwen3-8B-shaped decode batch (weak scaling: same shape, different seed)."""
    return W.qwen8_decode(seed=rank, num_seqs=num_seqs)


def rank_prefill_batch(rank: int) -> W.PagedBatch:
    return W.prefill_chunk(seed=rank)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import paged_kv_attention_store_gb300 as nv
    from paged_kv_attention_store_gb300 import build as lib_build

    lib_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    red_dev = dev if (world > 1 and dist.get_backend() == "nccl") else "cpu"

    def max_over_ranks(x: float) -> float:
        return reduce_over_ranks(x, "max", world, red_dev)

    def sum_over_ranks(x: float) -> float:
        return reduce_over_ranks(x, "sum", world, red_dev)

    pk, pk_kind = peaks()

    # ---------------- decode phase: store + decode on the Qwen3-8B batch ----------------
    db = rank_decode_batch(rank)
    kc, vc = db.cache()
    k_cache, v_cache = to_dev(kc), to_dev(vc)
    del kc, vc
    q, k_new, v_new = to_dev(db.q), to_dev(db.k_new), to_dev(db.v_new)
    slots, bt, ctx = to_dev(db.slot_mapping), to_dev(db.block_tables), to_dev(db.seq_lens)
    out = torch.empty_like(q)
    maxc = int(db.seq_lens.max())
    ws_bytes = nv.nv_paged_decode_workspace_size(db.num_seqs, db.num_q_heads, 128, maxc)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)      # split counters start at zero
    d_err = torch.zeros(1, dtype=torch.int32, device=dev)

    def decode_step(ev=None):
        nv.nv_store_kvcache(k_new, v_new, slots, k_cache, v_cache, d_err=d_err)
        if ev is not None:
            ev[0].record(stream)
        nv.nv_paged_decode_attn(q, k_cache, v_cache, bt, ctx, db.scale, out=out, max_context_len=maxc, workspace=ws,
                                d_err=d_err)
        if ev is not None:
            ev[1].record(stream)

    launches_per_decode_step = 2        # store, then decode (split merge inside the decode kernel)

    sampler = ClockSampler(local_rank)
    sampler.__enter__()
    try:
        for _ in range(args.warmup):
            decode_step()
        barrier()
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            decode_step(kev[i])
        t_end.record(stream)
        barrier()
        dec_ms = t_start.elapsed_time(t_end)
        dec_kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
        assert int(d_err.item()) == 0, f"device error flags {int(d_err.item())}"
        dec_out_bits = host_bits(out)             # checked against the oracle's sample below

        # e2e: the same step through the public API from pinned HOST memory: the step's inputs (q, the new
        # K/V rows, slots, block tables, lengths) packed back to back in one staging buffer and copied in
        # with one transfer, and the output read back, every step
        host_parts = [db.q.view(np.uint8).ravel(), db.k_new.view(np.uint8).ravel(), db.v_new.view(np.uint8).ravel(),
                      db.slot_mapping.view(np.uint8).ravel(), db.block_tables.view(np.uint8).ravel(),
                      db.seq_lens.view(np.uint8).ravel()]
        offs, total = [], 0
        for a in host_parts:
            offs.append(total)
            total += (a.size + 255) // 256 * 256
        h_stage = torch.zeros(total, dtype=torch.uint8).pin_memory()
        hs = h_stage.numpy()
        for o, a in zip(offs, host_parts):
            hs[o:o + a.size] = a
        d_stage = torch.empty(total, dtype=torch.uint8, device=dev)

        def staged(k, like):
            return d_stage[offs[k]:offs[k] + like.numel() * like.element_size()].view(like.dtype).view(like.shape)

        q_e, k_e, v_e = staged(0, q), staged(1, k_new), staged(2, v_new)
        s_e, bt_e, ctx_e = staged(3, slots), staged(4, bt), staged(5, ctx)
        h_out = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
        h2d = total
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step():
            d_stage.copy_(h_stage, non_blocking=True)
            nv.nv_store_kvcache(k_e, v_e, s_e, k_cache, v_cache, d_err=d_err)
            nv.nv_paged_decode_attn(q_e, k_cache, v_cache, bt_e, ctx_e, db.scale, out=out, max_context_len=maxc,
                                    workspace=ws, d_err=d_err)
            h_out.copy_(out, non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        barrier()
        e2e_ms = e0.elapsed_time(e1)
        torch.cuda.synchronize()
        assert np.array_equal(h_out.view(torch.int16).numpy().view(np.uint16), dec_out_bits), \
            "the staged end-to-end step must reproduce the device-resident step's output"

        # fused store + decode (one pass, nv_store_decode_attn) on the same batch
        def fused_step():
            nv.nv_store_decode_attn(q, k_new, v_new, slots, k_cache, v_cache, bt, ctx, db.scale, out=out,
                                    max_context_len=maxc, workspace=ws, d_err=d_err)

        for _ in range(args.warmup):
            fused_step()
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps):
            fused_step()
        f1.record(stream)
        barrier()
        fused_ms = f0.elapsed_time(f1)
        assert int(d_err.item()) == 0, f"device error flags {int(d_err.item())}"

        # device-side attention metadata for the same decode batch (NEXT-3) against the pages' host path
        pd_out = tuple(torch.empty(db.num_seqs, dtype=torch.int32, device=dev) for _ in range(3))
        for _ in range(args.warmup):
            nv.nv_prepare_decode(ctx, bt, db.block_size, db.num_blocks, out=pd_out, d_err=d_err)
        # captured in a CUDA graph so the number is device time, not the binding's launch rate
        g_meta = torch.cuda.CUDAGraph()
        cap_stream = torch.cuda.Stream()
        cap_stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(g_meta, stream=cap_stream):
                for _ in range(20):
                    nv.nv_prepare_decode(ctx, bt, db.block_size, db.num_blocks, out=pd_out, d_err=d_err)
        torch.cuda.current_stream().wait_stream(cap_stream)
        g_meta.replay()
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(1, args.steps // 20)
        m0.record(stream)
        for _ in range(reps):
            g_meta.replay()
        m1.record(stream)
        torch.cuda.synchronize()
        meta_dev_us = m0.elapsed_time(m1) * 1e3 / (reps * 20)
        assert torch.equal(pd_out[2].cpu(), torch.from_numpy(db.slot_mapping)), "device slots differ"
        from paged_kv_attention_store_gb300 import metadata as host_meta
        seqs_host = [(db.block_tables[i][db.block_tables[i] >= 0].tolist(), int(db.seq_lens[i]))
                     for i in range(db.num_seqs)]
        host_steps = max(5, min(args.steps, 50))
        torch.cuda.synchronize()
        t_h = time.perf_counter()
        for _ in range(host_steps):
            hm = host_meta.prepare_decode(seqs_host, db.block_size, width=db.block_tables.shape[1])
            for arr in (hm.positions, hm.slot_mapping, hm.context_lens, hm.block_tables):
                torch.from_numpy(arr).pin_memory().to(dev, non_blocking=True)
        torch.cuda.synchronize()
        meta_host_us = (time.perf_counter() - t_h) * 1e6 / host_steps

        # sampler (exponential race) over the decode batch's rows and the Qwen3 vocabulary
        V_SAMPLE = 151936
        srng = np.random.default_rng([rank, 17])
        s_logits = to_dev(W.f32_to_bf16_bits((srng.standard_normal((db.num_seqs, V_SAMPLE)) * 3.0)
                                             .astype(np.float32)))
        s_temps = torch.from_numpy(srng.uniform(0.5, 1.5, db.num_seqs).astype(np.float32)).to(dev)
        s_draws = torch.from_numpy(srng.exponential(1.0, (db.num_seqs, V_SAMPLE)).astype(np.float32)).to(dev)
        s_tok = torch.empty(db.num_seqs, dtype=torch.int64, device=dev)
        s_ws = torch.zeros(max(nv.load_library().nv_sample_workspace_size(db.num_seqs, V_SAMPLE), 16),
                           dtype=torch.uint8, device=dev)     # zero-filled once: per-row counters
        for _ in range(args.warmup):
            nv.nv_sample_exponential_race(s_logits, s_temps, s_draws, tokens=s_tok, workspace=s_ws, d_err=d_err)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(args.steps):
            nv.nv_sample_exponential_race(s_logits, s_temps, s_draws, tokens=s_tok, workspace=s_ws, d_err=d_err)
        s1.record(stream)
        torch.cuda.synchronize()
        sample_ms = s0.elapsed_time(s1) / args.steps
        sample_bytes = db.num_seqs * V_SAMPLE * (2 + 4) + db.num_seqs * (4 + 8)
        del s_logits, s_draws
        assert int(d_err.item()) == 0, f"device error flags {int(d_err.item())}"

        # ---------------- prefill phase: store + prefill on the chunked-prefill batch ----------------
        del k_cache, v_cache, ws
        torch.cuda.empty_cache()
        pb = rank_prefill_batch(rank)
        pkc, pvc = pb.cache()
        pk_cache, pv_cache = to_dev(pkc), to_dev(pvc)
        del pkc, pvc
        pq, pk_new, pv_new = to_dev(pb.q), to_dev(pb.k_new), to_dev(pb.v_new)
        pslots, pbt = to_dev(pb.slot_mapping), to_dev(pb.block_tables)
        pcu_q, pcu_k = to_dev(pb.cu_seqlens_q), to_dev(pb.cu_seqlens_k)
        pout = torch.empty_like(pq)
        mq = int(pb.q_lens.max())
        pws = torch.empty(nv.nv_paged_prefill_workspace_size(pb.num_seqs, int(pb.q_lens.sum()), mq, pb.num_q_heads,
                                                             pb.num_kv_heads), dtype=torch.uint8, device=dev)
        # L2 flush between timed calls: a 256 MB write (more than the 129 MB L2) evicts every input and
        # the previous call's outputs; a 256 MB read of a second buffer then evicts the write's own dirty
        # lines, so their write-back to HBM happens here and not inside the next timed call.
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        flush_rd = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)

        def flush_l2(i):
            flush.fill_(i & 0xFF)
            flush_rd.sum()

        def prefill_step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            nv.nv_store_kvcache(pk_new, pv_new, pslots, pk_cache, pv_cache, d_err=d_err)
            if ev is not None:
                ev[1].record(stream)
            nv.nv_paged_prefill_attn(pq, pk_cache, pv_cache, pcu_q, pcu_k, pbt, pb.scale, max_seqlen_q=mq, out=pout,
                                     workspace=pws, d_err=d_err)
            if ev is not None:
                ev[2].record(stream)

        # the warm-up runs the flush too: the first call of its kernels (lazily loaded by the runtime)
        # stalled the host for ~60 us inside the first timed step, which then measured 84 us
        for i in range(args.warmup):
            flush_l2(i)
            prefill_step()
        barrier()
        pev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2(i)                    # L2 flush between steps, outside the step's events
            prefill_step(pev[i])
        barrier()
        pf_out_bits = host_bits(pout)
        store_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in pev)
        pf_ms = statistics.mean(b.elapsed_time(c) for _, b, c in pev)
        pf_step_ms = statistics.mean(a.elapsed_time(c) for a, _, c in pev)

        # attention prologue (QK-norm + RoPE + K/V store) on the same batch's 16384 new tokens
        pi = W.prologue_inputs(pb, rank)
        pqkv, ppos = to_dev(pi.qkv), to_dev(pi.positions)
        pqw, pkw = to_dev(pi.q_weight), to_dev(pi.k_weight)
        pq_out = torch.empty_like(pq)

        def prologue_step():
            nv.nv_qk_norm_rope_store(pqkv, ppos, pqw, pkw, pslots, pk_cache, pv_cache, pb.num_q_heads,
                                     rms_eps=pi.eps, rope_theta=pi.theta, q_out=pq_out, d_err=d_err)

        for i in range(args.warmup):
            flush_l2(i)
            prologue_step()
        barrier()
        rev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2(i)
            rev[i][0].record(stream)
            prologue_step()
            rev[i][1].record(stream)
        barrier()
        pro_ms = statistics.mean(a.elapsed_time(b) for a, b in rev)
        assert int(d_err.item()) == 0, f"device error flags {int(d_err.item())}"

        # the other decode configurations: Qwen3-0.6B decode with graph padding, long shared prefix
        del flush, flush_rd
        torch.cuda.empty_cache()
        extra_steps = max(5, min(args.steps, 50))
        cfg_q06 = measure_decode_config(W.qwen06_decode(seed=rank), extra_steps, args.warmup, dev)
        cfg_64 = measure_decode_config(W.qwen8_decode(seed=rank, num_seqs=64), extra_steps, args.warmup, dev)
        cfg_sp = {bs: measure_decode_config(W.shared_prefix(seed=rank, block_size=bs), extra_steps, args.warmup, dev)
                  for bs in (256, 16)}
    finally:
        sampler.__exit__(None, None, None)

    # the prefill under sustained load: back-to-back calls for about a second, after the timed phases and
    # with a clock sampler of its own (a GPU at its power cap shows sw_power_cap there, not in the headline's
    # clock record); no L2 flush between the calls
    sus_calls = max(50, int(args.sustained_seconds / max(pf_ms * 1e-3, 1e-5)))
    barrier()
    sus_sampler = ClockSampler(local_rank)
    sus_sampler.__enter__()
    try:
        time.sleep(0.3)                        # a few clock samples from before the load starts
        s0e, s1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0e.record(stream)
        for _ in range(sus_calls):
            nv.nv_paged_prefill_attn(pq, pk_cache, pv_cache, pcu_q, pcu_k, pbt, pb.scale, max_seqlen_q=mq, out=pout,
                                     workspace=pws, d_err=d_err)
        s1e.record(stream)
        torch.cuda.synchronize()
    finally:
        sus_sampler.__exit__(None, None, None)
    assert int(d_err.item()) == 0, f"device error flags {int(d_err.item())}"
    sus_ms_max = max_over_ranks(s0e.elapsed_time(s1e) / sus_calls)
    del pk_cache, pv_cache

    dec_ms_max = max_over_ranks(dec_ms)
    e2e_ms_max = max_over_ranks(e2e_ms)
    dec_kernel_ms_max = max_over_ranks(dec_kernel_ms)
    fused_ms_max = max_over_ranks(fused_ms)
    pf_ms_max = max_over_ranks(pf_ms)
    pf_step_ms_max = max_over_ranks(pf_step_ms)
    store_ms_max = max_over_ranks(store_ms)
    pro_ms_max = max_over_ranks(pro_ms)

    kv_total = sum_over_ranks(float(decode_kv_bytes(db))) * args.steps
    tok_total = sum_over_ranks(float(db.seq_lens.astype(np.int64).sum())) * args.steps
    value = kv_total / (dec_ms_max * 1e-3) / 1e9
    e2e_value = kv_total / (e2e_ms_max * 1e-3) / 1e9
    alg_bytes = decode_algorithmic_bytes(db)
    achieved = alg_bytes / (dec_kernel_ms_max * 1e-3) / 1e9
    pf_flops_rank = prefill_flops(pb)
    pf_flops = sum_over_ranks(float(pf_flops_rank))
    pf_tflops = pf_flops / (pf_ms_max * 1e-3) / 1e12
    pf_tflops_rank = pf_flops_rank / (pf_ms_max * 1e-3) / 1e12
    pf_tok = sum_over_ranks(float(prefill_pairs(pb)))
    store_bytes = 2 * 2 * int(pb.q_lens.sum()) * pb.num_kv_heads * 128 * 2     # read + write, K and V
    n_pf = int(pb.q_lens.sum())
    # prologue: read q|k|v rows, write roped q and the stored k and v, plus positions and slots
    pro_bytes = n_pf * (pb.num_q_heads + 2 * pb.num_kv_heads) * 128 * 2 * 2 + n_pf * 8

    if rank != 0:
        return None
    dec_want, pf_want = {}, {}
    cpu = None if args.no_cpu_baseline else cpu_baseline_decode(db, args.cpu_seconds, collect=dec_want)
    cpu_pf = None if args.no_cpu_baseline else cpu_baseline_prefill(pb, args.cpu_seconds, collect=pf_want)
    parity = None
    if dec_want and pf_want:
        ds = sorted(dec_want)
        pr = np.array(sorted(pf_want), np.int64)
        parity = {
            "decode": dict(output_error(dec_out_bits[ds], np.stack([dec_want[i] for i in ds])),
                           sample=f"{len(ds)} sequences x {db.num_q_heads} heads of the timed batch"),
            "prefill": dict(output_error(pf_out_bits[pr], np.stack([pf_want[int(i)] for i in pr])),
                            sample=f"{pr.size} query rows x {pb.num_q_heads} heads of the timed batch"),
            "bar": {"max_abs": 2e-2, "mean_abs": 2e-3},
            "note": "GPU outputs of the timed runs against the fp32 oracle's outputs for the rows its baseline "
                    "leg computed",
        }
    clocks = sampler.summary()
    hbm_peak = float(pk["hbm_gbs"])
    tc_peak = float(pk["bf16_tflops"])
    tc_peak_sus = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dec_ms_max / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) values rounded to bf16, block tables dealt from a shuffled pool",
        "config": {
            "workload": "qwen3-8b-shaped decode step (store 512 new K/V rows + paged decode): 512 seqs, "
                        "ctx U[1024,4096], 32 q / 8 kv heads, head_dim 128, block_size 256, 1 layer",
            "num_seqs": db.num_seqs, "sum_context": int(db.seq_lens.sum()), "max_context": maxc,
            "kv_bytes_per_step": decode_kv_bytes(db),
            "l2": "inputs larger than L2 (decode KV 5.4 GB per step); L2 flushed between prefill and prologue steps (256 MB write, then a 256 MB read of another buffer so the flush leaves no dirty lines)",
            "parallelism": f"replicas x{world} (each rank its own batch; no collective on the path)",
        },
        "hbm_frac_of_peak": round(value / hbm_peak, 4),
        "attended_tok_s": round(tok_total / (dec_ms_max * 1e-3), 1),
        "roofline": {
            "kernel": "paged_decode_kernel, split merge fused in (nv_paged_decode_attn)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4),
            "peak_source": f"{pk_kind} hbm_gbs",
            "algorithmic_bytes_per_launch": alg_bytes,
            "traffic": profiled_traffic("decode_qwen8", ["paged_decode.cu", "nv_common.cuh"]),
        },
        "cpu_baseline": cpu,
        "parity": parity,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms_max / args.steps, 4)},
        "fused_store_decode": {
            "kernel": "paged_decode_kernel<4, 8, fused> (nv_store_decode_attn)",
            "value": round(kv_total / (fused_ms_max * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(fused_ms_max / args.steps, 4),
            "separate_ms_per_step": round(dec_ms_max / args.steps, 4),
            "note": "same step as the headline (store 512 rows + decode) in one pass: the new rows are read once "
                    "from the inputs and written to the pool by the decode kernel",
        },
        "prepare_decode": {
            "kernel": "prepare_decode_kernel (nv_prepare_decode)", "rows": db.num_seqs,
            "device_us_per_call": round(meta_dev_us, 2),
            "device_timing": "20 calls captured in a CUDA graph, replayed; CUDA events around the replays",
            "host_path_us_per_step": round(meta_host_us, 1),
            "note": "the pages build positions / slot_mapping / context_lens / block tables in Python each decode step "
                    "and copy them from pinned memory; the device call derives the first three from lengths and "
                    "tables already on the GPU (slots checked equal to the host-built ones)",
        },
        "sampler": {
            "kernel": "sample_partial_kernel, row merge fused in (nv_sample_exponential_race)",
            "workload": f"{db.num_seqs} rows x 151936-entry vocabulary: bf16 logits N(0, 9), T ~ U[0.5, 1.5], "
                        "float32 Exp(1) draws; inputs (467 MB) larger than L2",
            "ms": round(sample_ms, 4),
            "roofline": {"bound": "hbm", "achieved": round(sample_bytes / (sample_ms * 1e-3) / 1e9, 1),
                         "peak": float(pk["hbm_gbs"]), "unit": "GB/s",
                         "frac": round(sample_bytes / (sample_ms * 1e-3) / 1e9 / float(pk["hbm_gbs"]), 4),
                         "algorithmic_bytes_per_launch": sample_bytes},
        },
        "gpu_launches": launches_per_decode_step * args.steps,
        "gpu_launches_note": "kernels of this library launched in the headline timed region (store + split-KV decode "
                             "per step); all timed phases together: see gpu_launches_all_phases",
        # per step: headline and e2e (store + decode each), fused (1), prepare_decode (1), sampler (1), prefill
        # (store + pre-pass + attention), prologue (1); then the decode call of the three extra configs
        # (the extra configs: qwen06 one split-KV launch; the 64-sequence and shared-prefix batches a
        # pre-pass and the tile kernel each)
        "gpu_launches_all_phases": (launches_per_decode_step * 2 + 1 + 1 + 1 + 3 + 1) * args.steps
                                   + (1 + 2 + 2 + 2) * max(5, min(args.steps, 50)) + 2 * sus_calls,
        "clocks": clocks,
        "prefill": {
            "workload": "chunked prefill with prefix cache (store 16384 new rows + causal varlen prefill): 16 seqs, "
                        "prefixes 256*U{0..8}, chunks a uniform composition of 16384, 16 q / 8 kv heads, bs 256",
            "value": round(pf_tflops, 1), "unit": "TFLOP/s",
            "flops_per_step": pf_flops_rank, "causal_pairs_per_step": prefill_pairs(pb),
            "ms_prefill_kernel": round(pf_ms_max, 4), "ms_per_step": round(pf_step_ms_max, 4),
            "attended_pairs_s": round(pf_tok / (pf_ms_max * 1e-3), 1),
            "roofline": {
                "kernel": "paged_prefill_kernel (nv_paged_prefill_attn)",
                "bound": "tensor", "achieved": round(pf_tflops_rank, 1), "peak": tc_peak, "unit": "TFLOP/s",
                "frac": round(pf_tflops_rank / tc_peak, 4), "peak_source": f"{pk_kind} bf16_tflops (burst)",
                "traffic": profiled_traffic("prefill_chunk", ["paged_prefill.cu", "nv_common.cuh"]),
            },
            "store": {"ms": round(store_ms_max, 4), "gbs": round(store_bytes / (store_ms_max * 1e-3) / 1e9, 1),
                      "bytes_per_step": store_bytes},
            "sustained": {
                "calls": sus_calls, "ms_per_call": round(sus_ms_max, 4),
                "value": round(pf_flops / (sus_ms_max * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                "frac_of_sustained_peak": round(pf_flops_rank / (sus_ms_max * 1e-3) / 1e12 / tc_peak_sus, 4),
                "peak": tc_peak_sus, "peak_source": f"{pk_kind} bf16_tflops_sustained",
                "clocks": sus_sampler.summary(),
                "note": "back-to-back calls for about a second after the timed phases, no L2 flush between them; "
                        "its own clock record",
            },
            "cpu_baseline": cpu_pf,
        },
        "qwen06_decode": {
            "workload": "Qwen3-0.6B decode step: 256 seqs, ctx U[100, 2048], 16 q / 8 kv heads, bs 256, plus 32 "
                        "graph-padding rows (slot -1, context 0); store 288 rows + decode",
            **cfg_q06, "hbm_frac_of_peak": round(cfg_q06["logical_kv_gbs"] / hbm_peak, 4),
        },
        "qwen8_decode_64seq": {
            "workload": "the Qwen3-8B decode shape with 64 sequences (ctx U[1024, 4096], 32 q / 8 kv heads, bs 256); "
                        "store 64 rows + decode, which runs on the tcgen05 tile kernel (a split-KV grid this short "
                        "ends in a partly filled wave)",
            **cfg_64, "hbm_frac_of_peak": round(cfg_64["logical_kv_gbs"] / hbm_peak, 4),
        },
        "shared_prefix": {
            "workload": "64 seqs at context 4096, 32 q / 8 kv heads, the first 3072 tokens in the same physical "
                        "blocks; logical KV 1.07 GB, unique 281 MB; decode on the tcgen05 tile kernel",
            "bs256": cfg_sp[256], "bs16": cfg_sp[16],
            "bs16_slowdown": round(cfg_sp[16]["ms_per_decode"] / cfg_sp[256]["ms_per_decode"], 3),
        },
        "prologue": {
            "kernel": "qk_norm_rope_store_kernel (nv_qk_norm_rope_store)",
            "workload": "QK-norm + RoPE (theta 1e6) + K/V store for the chunked-prefill batch's 16384 new tokens, "
                        "16 q / 8 kv heads; L2 flushed before each call",
            "ms": round(pro_ms_max, 4),
            "roofline": {"bound": "hbm", "achieved": round(pro_bytes / (pro_ms_max * 1e-3) / 1e9, 1),
                         "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(pro_bytes / (pro_ms_max * 1e-3) / 1e9 / hbm_peak, 4),
                         "algorithmic_bytes_per_launch": pro_bytes},
        },
    }
    return line


# ----------------------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ----------------------------------------------------------------------------------------

def host_bits(t) -> np.ndarray:
    """bf16 tensor -> host uint16 bit patterns (a synchronous copy)."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def output_error(got_bits: np.ndarray, want: np.ndarray) -> dict:
    """max-abs, mean-abs and relative L2 error of bf16 outputs against fp32 oracle outputs."""
    got = W.bf16_bits_to_f32(got_bits).astype(np.float64)
    want = np.asarray(want, np.float64)
    err = np.abs(got - want)
    return {"max_abs": float(err.max()), "mean_abs": float(err.mean()),
            "rel_l2": float(np.linalg.norm(got - want) / max(float(np.linalg.norm(want)), 1e-30))}


def host_cpu() -> dict:
    """The host the CPU legs run on: its core count and CPU model (``lscpu``'s model name where
    /proc/cpuinfo has none, as on Arm hosts)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.strip().lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return {"host_cores": os.cpu_count(), "cpu_model": model or platform.machine()}


def cpu_baseline_decode(b: W.PagedBatch, seconds: float, max_seqs: int | None = None, collect: dict | None = None):
    """Oracle decode, single thread, sequence by sequence until ~`seconds` of CPU work (outputs into
    `collect`, by sequence, when given)."""
    import oracle
    orc = oracle.default()
    done, tokens, spent = 0, 0, 0.0
    order = np.random.default_rng(7).permutation(b.num_seqs)
    for s in order:
        sub, ids = b.subset([int(s)])
        kc, vc = sub.cache(ids, threads=1)
        orc.store_kvcache(sub.k_new, sub.v_new, sub.slot_mapping, kc, vc)
        t0 = time.perf_counter()
        o = orc.decode_attn(sub.q, kc, vc, sub.block_tables, sub.context_lens, sub.num_kv_heads, sub.block_size,
                            sub.scale, threads=1)
        spent += time.perf_counter() - t0
        if collect is not None:
            collect[int(s)] = o[0]
        done += 1
        tokens += int(sub.seq_lens.sum())
        if spent >= seconds or (max_seqs and done >= max_seqs):
            break
    kv = tokens * b.num_kv_heads * KV_BYTES_PER_TOKEN_PER_KVHEAD
    return {"value": round(kv / spent / 1e9, 4), "unit": "GB/s", "cores": 1, **host_cpu(), "kind": "oracle",
            "sample": f"{done} of {b.num_seqs} sequences ({tokens} attended positions x {b.num_q_heads} heads) "
                      f"of the same decode batch, one thread, {spent:.1f} s",
            "seconds": round(spent, 2), "attended_tok_s": round(tokens / spent, 1)}


def cpu_baseline_prefill(b: W.PagedBatch, seconds: float, collect: dict | None = None):
    """Oracle prefill, single thread, on a random sample of query rows until ~`seconds` (outputs into
    `collect`, by row, when given)."""
    import oracle
    orc = oracle.default()
    kc, vc = b.cache(threads=1)
    orc.store_kvcache(b.k_new, b.v_new, b.slot_mapping, kc, vc)
    rows_all = np.random.default_rng(8).permutation(int(b.q_lens.sum()))
    cu = b.cu_seqlens_q
    P = b.meta["prefix_lens"]
    spent, done, pairs, i = 0.0, 0, 0, 0
    while spent < seconds and i < rows_all.size:
        chunk = rows_all[i:i + 16]
        i += 16
        t0 = time.perf_counter()
        o = orc.prefill_attn(b.q, kc, vc, b.cu_seqlens_q, b.cu_seqlens_k, b.block_tables, b.num_kv_heads,
                             b.block_size, b.scale, rows=chunk, threads=1)
        spent += time.perf_counter() - t0
        if collect is not None:
            for j, r in enumerate(chunk):
                collect[int(r)] = o[j]
        for r in chunk:
            s = int(np.searchsorted(cu, r, side="right") - 1)
            pairs += int(P[s]) + int(r - cu[s]) + 1
        done += chunk.size
    flops = 4 * 128 * b.num_q_heads * pairs
    return {"value": round(flops / spent / 1e12, 6), "unit": "TFLOP/s", "cores": 1, **host_cpu(), "kind": "oracle",
            "sample": f"{done} of {int(b.q_lens.sum())} query rows ({pairs} causal pairs x {b.num_q_heads} heads) "
                      f"of the same prefill batch, one thread, {spent:.1f} s",
            "seconds": round(spent, 2)}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on rank 0 only; other ranks exit without work."""
    if rank != 0:
        return None
    db = W.qwen8_decode(seed=0)
    per_step = max(1, int(args.ref_seqs_per_step))
    # warm-up steps (untimed), then K timed steps, each a bounded sample of the batch
    for _ in range(min(args.warmup, 1)):
        cpu_baseline_decode(db, 0.0, max_seqs=1)
    t0 = time.perf_counter()
    kv = 0.0
    spent = 0.0
    toks = 0
    for k in range(args.steps):
        r = cpu_baseline_decode(db, 1e9, max_seqs=per_step)
        spent += r["seconds"]
        toks += int(r["attended_tok_s"] * r["seconds"])
        kv += r["value"] * 1e9 * r["seconds"]
    wall = time.perf_counter() - t0
    value = kv / spent / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(spent / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded N(0,1) values rounded to bf16, block tables dealt from a shuffled pool",
        "config": {"workload": "qwen3-8b-shaped decode step (store + paged decode), "
                               f"{per_step} sampled sequence(s) per step", "num_seqs": db.num_seqs},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, **host_cpu(), "kind": "oracle",
                         "sample": f"{per_step} sequence(s) of the 512-sequence batch per step, one thread"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 2),
    }


def run_profile_case(case: str):
    """Run one small case three times (store + attention) for an ncu capture, then exit.

    decode-16seq: the first 16 sequences' shapes of the Qwen3-8B decode batch (about 170 MB of KV,
    above the 129 MB L2), which decode on the same split-KV kernel as the full 512-sequence batch;
    decode-64seq: the first 64 sequences (about 0.7 GB of KV), which decode on the tile kernel;
    decode-g8-64seq: the same lengths with 64 query heads over the 8 kv heads (Qwen3-32B's attention
    shape, group 8); prefill-chunk: the full chunked-prefill workload (about 0.3 GB).  Each holds
    a few GB on the device at most."""
    import torch

    import paged_kv_attention_store_gb300 as nv
    from paged_kv_attention_store_gb300 import build as lib_build
    lib_build.build()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    if case == "sampler-256rows":
        # 256 rows x the 151936-entry vocabulary: 233 MB of logits + draws, above the L2
        rng = np.random.default_rng([0, 17])
        lg = to_dev(W.f32_to_bf16_bits((rng.standard_normal((256, 151936)) * 3.0).astype(np.float32)))
        tm = torch.from_numpy(rng.uniform(0.5, 1.5, 256).astype(np.float32)).cuda()
        dr = torch.from_numpy(rng.exponential(1.0, (256, 151936)).astype(np.float32)).cuda()
        d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(3):
            nv.nv_sample_exponential_race(lg, tm, dr, d_err=d_err)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": case, "d_err": int(d_err.item()),
                          "algorithmic_bytes": 256 * 151936 * 6 + 256 * 12}))
        return
    if case in ("decode-16seq", "decode-64seq"):
        n = 16 if case == "decode-16seq" else 64
        ctx = np.random.default_rng([0, 200]).integers(1024, 4097, size=512)[:n]
        b = W.make_decode(f"qwen3-8b-decode-{n}", 0, ctx, 32, 8, 128, 256)
    elif case == "decode-g8-64seq":
        ctx = np.random.default_rng([0, 200]).integers(1024, 4097, size=512)[:64]
        b = W.make_decode("group8-decode-64", 0, ctx, 64, 8, 128, 256)
    elif case.startswith("shared-prefix-bs"):
        b = W.shared_prefix(block_size=int(case[len("shared-prefix-bs"):]))
    else:
        b = W.prefill_chunk()
    kc, vc = b.cache()
    k_cache, v_cache = to_dev(kc), to_dev(vc)
    q, k_new, v_new, slots = to_dev(b.q), to_dev(b.k_new), to_dev(b.v_new), to_dev(b.slot_mapping)
    bt, lens = to_dev(b.block_tables), to_dev(b.seq_lens)
    cu_q, cu_k = to_dev(b.cu_seqlens_q), to_dev(b.cu_seqlens_k)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if case == "prologue-chunk":
        pi = W.prologue_inputs(b, 0)
        qkv, pos = to_dev(pi.qkv), to_dev(pi.positions)
        qw, kw = to_dev(pi.q_weight), to_dev(pi.k_weight)
        for _ in range(3):
            nv.nv_qk_norm_rope_store(qkv, pos, qw, kw, slots, k_cache, v_cache, b.num_q_heads, rms_eps=pi.eps,
                                     rope_theta=pi.theta, d_err=d_err)
        torch.cuda.synchronize()
        n = int(b.q_lens.sum())
        print(json.dumps({"profile_case": case, "d_err": int(d_err.item()),
                          "algorithmic_bytes": n * (b.num_q_heads + 2 * b.num_kv_heads) * 128 * 4 + n * 8}))
        return
    for _ in range(3):
        nv.nv_store_kvcache(k_new, v_new, slots, k_cache, v_cache, d_err=d_err)
        if b.kind == "decode":
            nv.nv_paged_decode_attn(q, k_cache, v_cache, bt, lens, b.scale, max_context_len=int(b.seq_lens.max()),
                                    d_err=d_err)
        else:
            nv.nv_paged_prefill_attn(q, k_cache, v_cache, cu_q, cu_k, bt, b.scale, max_seqlen_q=int(b.q_lens.max()),
                                     d_err=d_err)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": case, "d_err": int(d_err.item()),
                      "algorithmic_bytes": decode_algorithmic_bytes(b) if b.kind == "decode" else None,
                      "flops": prefill_flops(b) if b.kind == "prefill" else None}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU work per oracle baseline leg")
    ap.add_argument("--sustained-seconds", type=float, default=1.0,
                    help="back-to-back prefill calls after the timed phases (the prefill under sustained load)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seqs-per-step", type=int, default=1)
    ap.add_argument("--profile-case", choices=["decode-16seq", "decode-64seq", "decode-g8-64seq", "prefill-chunk", "prologue-chunk",
                                               "sampler-256rows",
                                               "shared-prefix-bs256", "shared-prefix-bs16"],
                    help="run one small case three times for an ncu capture and exit")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)
    try:
        line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world,
                                                                                         local_rank)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
