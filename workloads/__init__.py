"""Seeded synthetic inputs for the paged KV attention store.

This module is shared by the tests and the bench and feeds both the CUDA path and
the CPU oracle.  It holds no attention arithmetic: only random draws, exact
rounding of those draws to bf16, and the bookkeeping a block allocator does
(dealing physical block ids out of a shuffled pool and recording which physical
slot holds which logical position of a sequence, as the nano-vLLM field guide's
"Blocks, block tables and slots" section describes).

All values are bf16 bit patterns held in ``np.uint16`` arrays.  Cache contents
are drawn block by block from their own counter-keyed streams
(``default_rng([seed, tag, block_id])``), so a subset of blocks can be rebuilt
without materialising a multi-GB pool on the host.

Workload shapes follow the Qwen3 models the pages serve (16 q / 8 kv heads for
Qwen3-0.6B, 32 q / 8 kv for Qwen3-8B, head_dim 128); the per-config recipes are
the functions ``tiny``, ``qwen06_decode``, ``qwen8_decode``, ``prefill_chunk``
and ``shared_prefix`` at the bottom.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field

import numpy as np

BF16_NAN_SENTINEL = np.uint16(0x7FC1)   # quiet-NaN pattern used to poison slots nobody may read

# Stream tags: distinct random streams for the distinct kinds of draw.
_TAG_CACHE_K = 1
_TAG_CACHE_V = 2
_TAG_QKV = 3
_TAG_PROLOGUE = 4


# ----------------------------------------------------------------------------
# bf16 helpers (exact bit manipulation; no rounding beyond the one RNE step)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return bit patterns."""
    x = np.asarray(x, dtype=np.float32)
    u = np.ascontiguousarray(x).view(np.uint32).reshape(x.shape)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) float32 draws rounded to bf16 bit patterns."""
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


# ----------------------------------------------------------------------------
# Block dealing and cache contents
# ----------------------------------------------------------------------------

def blocks_needed(length: int, block_size: int) -> int:
    return (int(length) + block_size - 1) // block_size


def deal_block_tables(rng, lengths, block_size, width=None, shared_prefix_blocks=0):
    """Deal physical block ids to sequences out of a shuffled pool sized to the need.

    Returns ``(block_tables [B, W] int32 padded with -1, num_blocks)``.  With
    ``shared_prefix_blocks = s`` the first ``s`` logical blocks of every sequence
    map to the same ``s`` physical blocks (prefix-cache hits); the rest are distinct.
    """
    lengths = [int(x) for x in lengths]
    need = [blocks_needed(n, block_size) for n in lengths]
    s = int(shared_prefix_blocks)
    if s:
        assert all(n > s for n in need), "every sequence must extend past the shared prefix"
    total = s + sum(n - s for n in need)
    perm = rng.permutation(total).astype(np.int32)
    W = max(need) if width is None else int(width)
    assert W >= max(need)
    bt = np.full((len(lengths), W), -1, dtype=np.int32)
    shared = perm[:s]
    cur = s
    for b, n in enumerate(need):
        bt[b, :s] = shared
        bt[b, s:n] = perm[cur:cur + n - s]
        cur += n - s
    return bt, total


def physical_slots(block_table_row: np.ndarray, block_size: int, length: int) -> np.ndarray:
    """Physical slot of every logical position ``0..length-1`` of one sequence.

    This is the allocator's own record of where it put each position: block
    ``block_table_row[i]`` holds positions ``i*bs .. i*bs+bs-1`` in its rows
    ``0..bs-1``.  Built by expanding the table, not by a per-position formula.
    """
    n = blocks_needed(length, block_size)
    rows = np.arange(block_size, dtype=np.int64)
    slots = (block_table_row[:n].astype(np.int64)[:, None] * block_size + rows[None, :]).reshape(-1)
    return slots[:length]


def cache_block(seed: int, block_id: int, block_size: int, num_kv_heads: int, head_dim: int):
    """K and V contents of one physical block: ``([bs, Hkv, D], [bs, Hkv, D])`` bf16 bits."""
    shape = (block_size, num_kv_heads, head_dim)
    k = normal_bf16(np.random.default_rng([seed, _TAG_CACHE_K, int(block_id)]), shape)
    v = normal_bf16(np.random.default_rng([seed, _TAG_CACHE_V, int(block_id)]), shape)
    return k, v


def fill_cache(seed, block_ids, block_size, num_kv_heads, head_dim, k_out, v_out, threads=None):
    """Fill ``k_out[i], v_out[i]`` (shape ``[n, bs, Hkv, D]``) with the contents of ``block_ids[i]``."""
    block_ids = list(int(b) for b in block_ids)

    def work(i):
        k, v = cache_block(seed, block_ids[i], block_size, num_kv_heads, head_dim)
        k_out[i] = k
        v_out[i] = v

    threads = threads or min(16, os.cpu_count() or 1)
    if len(block_ids) < 8 or threads <= 1:
        for i in range(len(block_ids)):
            work(i)
    else:
        with _cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(len(block_ids))))


# ----------------------------------------------------------------------------
# Batches
# ----------------------------------------------------------------------------

@dataclass
class PagedBatch:
    """One attention call's worth of inputs over a paged pool.

    ``kind`` is ``"decode"`` (one new token per sequence, at position L-1) or
    ``"prefill"`` (a chunk of ``Lq`` new tokens after ``P`` cached ones).
    ``q``/``k_new``/``v_new`` are packed over new tokens; ``slot_mapping`` has one
    entry per new-token row (``-1`` for padding rows).  The pool itself is not
    stored here; ``cache(...)`` builds it (or a subset) from the block seeds.
    """
    name: str
    kind: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    block_tables: np.ndarray          # [B, W] int32
    seq_lens: np.ndarray              # [B] int32: keys visible to the last query (L or Lk)
    q_lens: np.ndarray                # [B] int32: new tokens per sequence (1 in decode, 0 for padding)
    q: np.ndarray                     # [Nq, Hq, D] uint16
    k_new: np.ndarray                 # [Nq, Hkv, D] uint16
    v_new: np.ndarray                 # [Nq, Hkv, D] uint16
    slot_mapping: np.ndarray          # [Nq] int32
    scale: float
    poison_tail: bool = False         # positions >= L inside each last block hold NaN patterns
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self):
        return int(self.block_tables.shape[0])

    @property
    def context_lens(self):
        """Decode: ``[B]`` int32 keys per sequence (0 for padding rows)."""
        return self.seq_lens.astype(np.int32)

    @property
    def cu_seqlens_q(self):
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def cu_seqlens_k(self):
        return np.concatenate([[0], np.cumsum(self.seq_lens)]).astype(np.int32)

    @property
    def kv_row_elems(self):
        return self.num_kv_heads * self.head_dim

    def used_blocks(self, seqs=None):
        seqs = range(self.num_seqs) if seqs is None else seqs
        out = []
        for b in seqs:
            n = blocks_needed(int(self.seq_lens[b]), self.block_size)
            out.extend(int(x) for x in self.block_tables[b, :n])
        return sorted(set(out))

    def cache(self, block_ids=None, threads=None):
        """Initial pool ``(k_cache, v_cache)`` as ``[n, bs, Hkv, D]`` uint16.

        With ``block_ids=None`` the whole pool (``num_blocks`` blocks, in id order);
        otherwise only the listed blocks, in the listed order.
        """
        ids = list(range(self.num_blocks)) if block_ids is None else list(block_ids)
        shape = (len(ids), self.block_size, self.num_kv_heads, self.head_dim)
        kc = np.empty(shape, dtype=np.uint16)
        vc = np.empty(shape, dtype=np.uint16)
        fill_cache(self.seed, ids, self.block_size, self.num_kv_heads, self.head_dim, kc, vc, threads)
        if self.poison_tail:
            pos_of = {bid: i for i, bid in enumerate(ids)}
            for b in range(self.num_seqs):
                L = int(self.seq_lens[b])
                if L <= 0:
                    continue
                nb = blocks_needed(L, self.block_size)
                last = int(self.block_tables[b, nb - 1])
                off = L - (nb - 1) * self.block_size
                if last in pos_of:
                    kc[pos_of[last], off:] = BF16_NAN_SENTINEL
                    vc[pos_of[last], off:] = BF16_NAN_SENTINEL
        return kc, vc

    def subset(self, seqs):
        """The same work restricted to ``seqs``, over a compact pool relabelled 0..n-1.

        Relabelling physical blocks leaves attention unchanged (a pinned oracle
        property), so the oracle can check sampled sequences of a multi-GB batch.
        Returns ``(sub_batch, block_ids)`` where ``block_ids[i]`` is the original id
        of compact block ``i`` (pass it to ``cache``).
        """
        seqs = [int(s) for s in seqs]
        ids = self.used_blocks(seqs)
        relabel = {bid: i for i, bid in enumerate(ids)}
        nb = [blocks_needed(int(self.seq_lens[b]), self.block_size) for b in seqs]
        W = max(max(nb), 1)
        bt = np.full((len(seqs), W), -1, dtype=np.int32)
        for r, b in enumerate(seqs):
            bt[r, :nb[r]] = [relabel[int(x)] for x in self.block_tables[b, :nb[r]]]
        cu = self.cu_seqlens_q
        rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in seqs]).astype(np.int64) \
            if seqs else np.zeros(0, np.int64)
        sub_slots = []
        for r, b in enumerate(seqs):
            L = int(self.seq_lens[b])
            nq = int(self.q_lens[b])
            if nq == 0:
                continue
            sl = physical_slots(bt[r], self.block_size, L)
            sub_slots.extend(sl[L - nq:L].tolist())
        sub = PagedBatch(
            name=f"{self.name}[subset]", kind=self.kind, seed=self.seed,
            num_q_heads=self.num_q_heads, num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
            block_size=self.block_size, num_blocks=len(ids), block_tables=bt,
            seq_lens=self.seq_lens[seqs].copy(), q_lens=self.q_lens[seqs].copy(),
            q=self.q[rows].copy(), k_new=self.k_new[rows].copy(), v_new=self.v_new[rows].copy(),
            slot_mapping=np.asarray(sub_slots, dtype=np.int32).reshape(-1), scale=self.scale,
            poison_tail=self.poison_tail, meta=dict(self.meta, parent_rows=rows, parent_seqs=seqs))
        return sub, ids


def _new_rows(seed, n, hq, hkv, d):
    rng = np.random.default_rng([seed, _TAG_QKV])
    q = normal_bf16(rng, (n, hq, d))
    k = normal_bf16(rng, (n, hkv, d))
    v = normal_bf16(rng, (n, hkv, d))
    return q, k, v


@dataclass
class PrologueInputs:
    """Inputs of the attention prologue (QK-norm + RoPE + store) for the new rows of a batch."""
    qkv: np.ndarray          # uint16 [N, (Hq + 2 Hkv) * D]: q | k | v of each new token
    positions: np.ndarray    # int32 [N]
    q_weight: np.ndarray     # uint16 [D]
    k_weight: np.ndarray     # uint16 [D]
    eps: float
    theta: float


def prologue_inputs(batch: "PagedBatch", seed: int = 0, eps: float = 1e-6, theta: float = 1e6) -> PrologueInputs:
    """Projection rows N(0,1) (bf16) for every new token of ``batch`` (one per slot_mapping entry),
    the tokens' positions (prefix + index for prefill, L-1 for decode, 0 for padding rows), and
    random-init norm weights N(1, 0.1^2) (bf16) -- Qwen3's layer shapes with synthetic values."""
    rng = np.random.default_rng([seed, _TAG_PROLOGUE])
    n = int(batch.slot_mapping.shape[0])
    width = (batch.num_q_heads + 2 * batch.num_kv_heads) * batch.head_dim
    qkv = normal_bf16(rng, (n, width))
    w = f32_to_bf16_bits(1.0 + 0.1 * rng.standard_normal((2, batch.head_dim)).astype(np.float32))
    if batch.kind == "decode":
        pos = np.maximum(batch.seq_lens.astype(np.int64) - 1, 0)
    else:
        pos = np.concatenate([np.arange(int(p), int(p) + int(lq)) for p, lq in
                              zip(batch.meta["prefix_lens"], batch.q_lens)]) if n else np.zeros(0, np.int64)
    return PrologueInputs(qkv=qkv, positions=pos.astype(np.int32), q_weight=w[0].copy(), k_weight=w[1].copy(),
                          eps=float(eps), theta=float(theta))


def make_decode(name, seed, ctx_lens, hq, hkv, d, block_size, n_pad=0, width=None,
                shared_prefix_blocks=0, poison_tail=False, scale=None):
    """A decode step: sequence b has ``ctx_lens[b]`` keys, the last of which is its new token.

    ``n_pad`` extra rows mimic CUDA-graph bucket padding: context length 0 and slot -1.
    """
    rng = np.random.default_rng([seed, 0])
    ctx = np.asarray(ctx_lens, dtype=np.int64)
    bt, num_blocks = deal_block_tables(rng, ctx, block_size, width, shared_prefix_blocks)
    B = len(ctx)
    if n_pad:
        bt = np.concatenate([bt, np.full((n_pad, bt.shape[1]), -1, np.int32)])
    n = B + n_pad
    q, k, v = _new_rows(seed, n, hq, hkv, d)
    slots = np.full(n, -1, dtype=np.int32)
    for b in range(B):
        slots[b] = physical_slots(bt[b], block_size, int(ctx[b]))[-1]
    seq_lens = np.concatenate([ctx, np.zeros(n_pad, np.int64)]).astype(np.int32)
    q_lens = np.concatenate([np.ones(B, np.int64), np.zeros(n_pad, np.int64)]).astype(np.int32)
    return PagedBatch(name=name, kind="decode", seed=seed, num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=d, block_size=block_size, num_blocks=num_blocks, block_tables=bt,
                      seq_lens=seq_lens, q_lens=q_lens, q=q, k_new=k, v_new=v, slot_mapping=slots,
                      scale=float(d ** -0.5 if scale is None else scale), poison_tail=poison_tail,
                      meta={"n_pad": n_pad})


def make_prefill(name, seed, prefix_lens, chunk_lens, hq, hkv, d, block_size, width=None,
                 poison_tail=False, scale=None):
    """A prefill step: sequence b has ``prefix_lens[b]`` cached tokens and ``chunk_lens[b]`` new ones."""
    rng = np.random.default_rng([seed, 0])
    P = np.asarray(prefix_lens, dtype=np.int64)
    Lq = np.asarray(chunk_lens, dtype=np.int64)
    Lk = P + Lq
    bt, num_blocks = deal_block_tables(rng, Lk, block_size, width)
    total_q = int(Lq.sum())
    q, k, v = _new_rows(seed, total_q, hq, hkv, d)
    slots = []
    for b in range(len(Lk)):
        sl = physical_slots(bt[b], block_size, int(Lk[b]))
        slots.extend(sl[int(P[b]):int(Lk[b])].tolist())
    return PagedBatch(name=name, kind="prefill", seed=seed, num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=d, block_size=block_size, num_blocks=num_blocks, block_tables=bt,
                      seq_lens=Lk.astype(np.int32), q_lens=Lq.astype(np.int32), q=q, k_new=k, v_new=v,
                      slot_mapping=np.asarray(slots, dtype=np.int32), scale=float(d ** -0.5 if scale is None else scale),
                      poison_tail=poison_tail, meta={"prefix_lens": P.astype(np.int32)})


# ----------------------------------------------------------------------------
# The five workload recipes
# ----------------------------------------------------------------------------

def tiny(seed=0):
    """1 layer, 16 q / 8 kv heads, D 128, bs 256, pool of 8 blocks, contexts [1, 17, 256, 300]."""
    rng = np.random.default_rng([seed, 0])
    ctx = [1, 17, 256, 300]
    # A random permutation of the 8-block pool, dealt in order (5 blocks are used).
    perm = rng.permutation(8).astype(np.int32)
    bt = np.full((4, 2), -1, np.int32)
    cur = 0
    for b, L in enumerate(ctx):
        n = blocks_needed(L, 256)
        bt[b, :n] = perm[cur:cur + n]
        cur += n
    q, k, v = _new_rows(seed, 4, 16, 8, 128)
    slots = np.array([physical_slots(bt[b], 256, ctx[b])[-1] for b in range(4)], np.int32)
    return PagedBatch(name="tiny", kind="decode", seed=seed, num_q_heads=16, num_kv_heads=8,
                      head_dim=128, block_size=256, num_blocks=8, block_tables=bt,
                      seq_lens=np.asarray(ctx, np.int32), q_lens=np.ones(4, np.int32), q=q, k_new=k,
                      v_new=v, slot_mapping=slots, scale=1.0 / np.sqrt(128.0), poison_tail=True,
                      meta={"n_pad": 0})


def qwen06_decode(seed=0, block_size=256):
    """Qwen3-0.6B heads, 256 sequences with L ~ U[100, 2048] plus 32 graph-padding rows."""
    rng = np.random.default_rng([seed, 100])
    ctx = rng.integers(100, 2049, size=256)
    return make_decode("qwen3-0.6b-decode", seed, ctx, 16, 8, 128, block_size, n_pad=32)


def qwen8_decode(seed=0, block_size=256, num_seqs=512):
    """Qwen3-8B heads (32 q / 8 kv), 512 sequences with L ~ U[1024, 4096]: the HBM headline."""
    rng = np.random.default_rng([seed, 200])
    ctx = rng.integers(1024, 4097, size=num_seqs)
    return make_decode("qwen3-8b-decode", seed, ctx, 32, 8, 128, block_size)


def prefill_chunk(seed=0, block_size=256, total_new=16384, num_seqs=16):
    """Qwen3-0.6B heads, 16 sequences, prefixes 256*U{0..8}, chunk lengths a uniform composition of 16384."""
    rng = np.random.default_rng([seed, 300])
    cuts = np.sort(rng.choice(np.arange(1, total_new), size=num_seqs - 1, replace=False))
    chunks = np.diff(np.concatenate([[0], cuts, [total_new]]))
    prefix = 256 * rng.integers(0, 9, size=num_seqs)
    return make_prefill("qwen3-0.6b-chunked-prefill", seed, prefix, chunks, 16, 8, 128, block_size)


def shared_prefix(seed=0, block_size=256):
    """Qwen3-8B heads, 64 sequences at context 4096 whose first 3072 tokens share physical blocks."""
    shared = 3072 // block_size
    return make_decode(f"shared-prefix-bs{block_size}", seed, [4096] * 64, 32, 8, 128, block_size,
                       shared_prefix_blocks=shared)


CONFIGS = {
    "tiny": tiny,
    "qwen06_decode": qwen06_decode,
    "qwen8_decode": qwen8_decode,
    "prefill_chunk": prefill_chunk,
    "shared_prefix": shared_prefix,
}
