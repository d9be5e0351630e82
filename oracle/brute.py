"""Float64 NumPy brute force for tiny inputs -- TEST INFRASTRUCTURE ONLY (pins the C oracle).

It reaches the same quantities by a different route from ``oracle.c``:

* un-paging goes through the 4-D pool view ``[num_blocks, bs, Hkv, D]``: the blocks a
  sequence owns are gathered in table order and concatenated (no slot arithmetic);
* attention is one dense float64 matrix product per sequence with an explicit
  bottom-right causal mask (nano-vLLM field guide, Step 10.3: with fewer queries than
  keys the mask is aligned to the bottom-right corner), then a max-subtracted softmax;
* GQA repeats each kv head over its group of ``Hq / Hkv`` query heads.
"""
from __future__ import annotations

import numpy as np


def widen(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def unpage(cache4: np.ndarray, table_row, length: int) -> np.ndarray:
    """Contiguous ``[length, Hkv, D]`` history of one sequence from a ``[nb, bs, Hkv, D]`` pool."""
    bs = cache4.shape[1]
    n = (length + bs - 1) // bs
    ids = [int(x) for x in table_row[:n]]
    if n == 0:
        return cache4[:0].reshape(0, *cache4.shape[2:])
    return np.concatenate([cache4[i] for i in ids], axis=0)[:length]


def attention(q_rows, k_seq, v_seq, scale, num_queries_total_keys_offset):
    """Dense causal attention in float64.

    ``q_rows``: ``[Lq, Hq, D]`` (float64), ``k_seq``/``v_seq``: ``[Lk, Hkv, D]`` (float64).
    Query i may see keys ``0 .. offset + i`` where ``offset = Lk - Lq``.
    Returns ``[Lq, Hq, D]`` float64.
    """
    Lq, hq, d = q_rows.shape
    Lk, hkv, _ = k_seq.shape
    g = hq // hkv
    K = np.repeat(k_seq, g, axis=1)          # [Lk, Hq, D]
    V = np.repeat(v_seq, g, axis=1)
    S = np.einsum("ihd,jhd->hij", q_rows, K) * scale     # [Hq, Lq, Lk]
    off = num_queries_total_keys_offset
    allowed = np.arange(Lk)[None, :] <= (off + np.arange(Lq))[:, None]
    S = np.where(allowed[None], S, -np.inf)
    S = S - S.max(axis=-1, keepdims=True)
    Pm = np.exp(S)
    Pm /= Pm.sum(axis=-1, keepdims=True)
    return np.einsum("hij,jhd->ihd", Pm, V)


def decode(q, k_cache4, v_cache4, block_tables, context_lens, scale):
    """``[B, Hq, D]`` float64: each sequence's one query over its ``context_lens[b]`` keys."""
    q = widen(q)
    B, hq, d = q.shape
    out = np.zeros((B, hq, d))
    for b in range(B):
        L = int(context_lens[b])
        if L <= 0:
            continue
        K = widen(unpage(k_cache4, block_tables[b], L))
        V = widen(unpage(v_cache4, block_tables[b], L))
        out[b] = attention(q[b:b + 1], K, V, scale, L - 1)[0]
    return out


def prefill(q, k_cache4, v_cache4, cu_q, cu_k, block_tables, scale):
    """``[total_q, Hq, D]`` float64 causal prefill over cached prefix + chunk."""
    q = widen(q)
    out = np.zeros(q.shape)
    for b in range(len(cu_q) - 1):
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        Lk = int(cu_k[b + 1] - cu_k[b])
        if q1 == q0:
            continue
        K = widen(unpage(k_cache4, block_tables[b], Lk))
        V = widen(unpage(v_cache4, block_tables[b], Lk))
        out[q0:q1] = attention(q[q0:q1], K, V, scale, Lk - (q1 - q0))
    return out


def round_bf16(x) -> np.ndarray:
    """Round to bf16 (nearest even) and widen back to float64; via float32, then the bit trick."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def rms_norm(x_bits, w_bits, eps):
    """Qwen3's per-head RMSNorm in float64: x / sqrt(mean(x^2) + eps) rounded to bf16, then the
    bf16 product with the weight (rounded to bf16)."""
    x = widen(x_bits)
    r = 1.0 / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    return round_bf16(round_bf16(x * r) * widen(w_bits))


def norm_rope(x_bits, w_bits, eps, theta, positions):
    """Float64 restatement of Qwen3's QK-norm + RoPE for head vectors ``x_bits`` ``[N, H, D]``
    (bf16 bits) at ``positions`` ``[N]``: RMSNorm over D (cast to bf16, then the bf16 product with
    the weight), then the rotate-half rotation by position * theta^(-2j/D).  Returns float64
    values already rounded to bf16 (the pages' output dtype)."""
    n = rms_norm(x_bits, w_bits, eps)
    d = n.shape[-1]
    j = np.arange(d // 2, dtype=np.float64)
    ang = np.asarray(positions, np.float64)[:, None, None] * theta ** (-2.0 * j / d)
    x1, x2 = n[..., : d // 2], n[..., d // 2:]
    return np.concatenate([round_bf16(x1 * np.cos(ang) - x2 * np.sin(ang)),
                           round_bf16(x2 * np.cos(ang) + x1 * np.sin(ang))], axis=-1)
