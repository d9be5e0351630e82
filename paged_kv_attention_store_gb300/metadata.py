"""Host-side attention metadata: what a caller builds before the three library calls.

These are the caller's side of the boundary, restated from the nano-vLLM field guide
(Step 07.5 "prepare_prefill", Step 07.6 "prepare_decode", Step 07.7
"prepare_block_tables", Step 07.8 graph-replay padding).  They run on the host on
plain Python ints and return NumPy arrays ready to copy to the device; the kernels
never depend on them.

A block table lists a sequence's physical block ids in logical order.  Position
``pos`` lives in block ``table[pos // block_size]`` at row ``pos % block_size``, so its
slot (row index into the flattened ``[num_blocks * block_size, Hkv * D]`` pool) is
``table[pos // block_size] * block_size + pos % block_size``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def slot_for(block_table, pos: int, block_size: int) -> int:
    """Slot of logical position ``pos`` of a sequence with ``block_table``."""
    return int(block_table[pos // block_size]) * block_size + pos % block_size


def slots_for_range(block_table, start: int, end: int, block_size: int) -> list[int]:
    """Slots of positions ``start .. end-1``, walked block by block as ``prepare_prefill`` does:
    the first block starts at ``start % block_size``, the last stops at ``end``, and the blocks
    in between contribute all of their rows."""
    out: list[int] = []
    if end <= start:
        return out
    first = start // block_size
    last = (end + block_size - 1) // block_size
    for i in range(first, last):
        base = int(block_table[i]) * block_size
        lo = start % block_size if i == first else 0
        hi = end - i * block_size if i == last - 1 else block_size
        out.extend(range(base + lo, base + hi))
    return out


def pad_block_tables(tables, width: int | None = None) -> np.ndarray:
    """int32 ``[B, W]``: each table padded with -1 to the longest (or to ``width``)."""
    w = max((len(t) for t in tables), default=0) if width is None else int(width)
    out = np.full((len(tables), max(w, 1)), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        if len(t) > w:
            raise ValueError(f"block table {i} has {len(t)} entries, wider than {w}")
        out[i, :len(t)] = t
    return out


@dataclass
class PrefillMeta:
    positions: np.ndarray       # [total_q] int64
    slot_mapping: np.ndarray    # [total_q] int32
    cu_seqlens_q: np.ndarray    # [B+1] int32
    cu_seqlens_k: np.ndarray    # [B+1] int32
    max_seqlen_q: int
    max_seqlen_k: int
    block_tables: np.ndarray    # [B, W] int32 (always built; the pages pass it only with a cached prefix)
    has_prefix: bool            # cu_seqlens_k[-1] > cu_seqlens_q[-1]


def prepare_prefill(seqs, block_size: int) -> PrefillMeta:
    """``seqs``: iterable of ``(block_table, num_cached_tokens, num_scheduled_tokens)``.

    Sequence b contributes queries for positions ``[cached, cached + scheduled)`` and
    attends to ``seqlen_k = cached + scheduled`` keys (its cached prefix plus the chunk)."""
    positions, slots, tables = [], [], []
    cu_q, cu_k = [0], [0]
    max_q = max_k = 0
    for table, cached, scheduled in seqs:
        start, end = int(cached), int(cached) + int(scheduled)
        positions.extend(range(start, end))
        cu_q.append(cu_q[-1] + (end - start))
        cu_k.append(cu_k[-1] + end)
        max_q = max(max_q, end - start)
        max_k = max(max_k, end)
        slots.extend(slots_for_range(table, start, end, block_size))
        tables.append(list(table))
    return PrefillMeta(
        positions=np.asarray(positions, dtype=np.int64),
        slot_mapping=np.asarray(slots, dtype=np.int32),
        cu_seqlens_q=np.asarray(cu_q, dtype=np.int32),
        cu_seqlens_k=np.asarray(cu_k, dtype=np.int32),
        max_seqlen_q=max_q, max_seqlen_k=max_k,
        block_tables=pad_block_tables(tables),
        has_prefix=cu_k[-1] > cu_q[-1])


@dataclass
class DecodeMeta:
    positions: np.ndarray       # [B] int64: len(seq) - 1
    context_lens: np.ndarray    # [B] int32: len(seq), including the token stored this step
    slot_mapping: np.ndarray    # [B] int32: slot of the newest token
    block_tables: np.ndarray    # [B, W] int32, -1 padded


def prepare_decode(seqs, block_size: int, width: int | None = None) -> DecodeMeta:
    """``seqs``: iterable of ``(block_table, num_tokens)``; one new token per sequence.

    The newest token sits at position ``num_tokens - 1``; its slot is the last block's base
    plus the number of tokens in that block minus one."""
    positions, ctx, slots, tables = [], [], [], []
    for table, n in seqs:
        n = int(n)
        nblocks = (n + block_size - 1) // block_size
        last_block_tokens = n - (nblocks - 1) * block_size
        positions.append(n - 1)
        ctx.append(n)
        slots.append(int(table[nblocks - 1]) * block_size + last_block_tokens - 1)
        tables.append(list(table))
    return DecodeMeta(positions=np.asarray(positions, dtype=np.int64),
                      context_lens=np.asarray(ctx, dtype=np.int32),
                      slot_mapping=np.asarray(slots, dtype=np.int32),
                      block_tables=pad_block_tables(tables, width))


def pad_decode_to_bucket(meta: DecodeMeta, bucket: int) -> DecodeMeta:
    """Pad a decode batch to a CUDA-graph bucket: extra rows store nothing (slot -1) and attend
    to nothing (context length 0); their block-table rows are -1."""
    B = meta.context_lens.shape[0]
    if bucket < B:
        raise ValueError(f"bucket {bucket} smaller than batch {B}")
    pad = bucket - B
    W = meta.block_tables.shape[1]
    return DecodeMeta(
        positions=np.concatenate([meta.positions, np.zeros(pad, np.int64)]),
        context_lens=np.concatenate([meta.context_lens, np.zeros(pad, np.int32)]),
        slot_mapping=np.concatenate([meta.slot_mapping, np.full(pad, -1, np.int32)]),
        block_tables=np.concatenate([meta.block_tables, np.full((pad, W), -1, np.int32)]))


GRAPH_BUCKETS = [1, 2, 4, 8] + list(range(16, 513, 16))


def graph_bucket(batch: int, max_bs: int = 512) -> int:
    """Smallest captured decode batch size that holds ``batch`` rows (1, 2, 4, 8, then multiples of 16)."""
    for b in GRAPH_BUCKETS:
        if b > max_bs:
            break
        if b >= batch:
            return b
    raise ValueError(f"no graph bucket holds {batch} rows (max {max_bs})")
