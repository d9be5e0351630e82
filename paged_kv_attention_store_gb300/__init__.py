"""Paged KV attention store for NVIDIA GB300 (sm_103a): Python binding of the C ABI.

The three calls of the hot path, same names as the C entry points declared in
``include/nv_paged_kv.h``:

* ``nv_store_kvcache``      -- scatter new K/V rows into their cache slots;
* ``nv_paged_decode_attn``  -- split-KV decode attention over block tables (GQA);
* ``nv_paged_prefill_attn`` -- varlen causal prefill over a cached prefix (tcgen05).

This module only marshals arguments: it reads shapes, strides and raw device pointers
from torch tensors and the current CUDA stream, and calls the shared library through
ctypes.  Every step of the computation runs in the library's kernels; there is no other
implementation to fall back to, and importing fails loudly if the library is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import metadata  # noqa: F401  (host-side slot / cu_seqlens builders)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libnv_paged_kv.so")

NV_OK = 0
NV_DERR_SLOT_RANGE = 0x1
NV_DERR_BLOCK_RANGE = 0x2
NV_DERR_LENGTH = 0x4
NV_DERR_TIMEOUT = 0x8
NV_DERR_SLOT_MISMATCH = 0x10
NV_DERR_VALUE = 0x20

EXPORTED = ("nv_status_string", "nv_store_kvcache", "nv_paged_decode_workspace_size", "nv_paged_decode_attn",
            "nv_store_decode_attn", "nv_paged_decode_attn_noalloc", "nv_paged_prefill_workspace_size",
            "nv_paged_prefill_attn", "nv_qk_norm_rope_store", "nv_prepare_decode", "nv_prepare_prefill",
            "nv_sample_workspace_size", "nv_sample_exponential_race")


class NvError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} returned {status}: {text}")
        self.status = status


_lib = None


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle of the CUDA library.

    Raises ``RuntimeError`` if it has not been built -- run
    ``python -m paged_kv_attention_store_gb300.build`` (or ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing "
                           "(run `python -m paged_kv_attention_store_gb300.build`)")
    L = ctypes.CDLL(p)
    V, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    L.nv_status_string.argtypes = [ctypes.c_int]
    L.nv_status_string.restype = ctypes.c_char_p
    L.nv_store_kvcache.argtypes = [V, i64, V, i64, V, i32, V, V, i64, i32, i32, V, V]
    L.nv_store_kvcache.restype = ctypes.c_int
    L.nv_paged_decode_workspace_size.argtypes = [i32, i32, i32, i32]
    L.nv_paged_decode_workspace_size.restype = sz
    L.nv_paged_decode_attn.argtypes = [V, V, V, V, i32, V, i32, i32, i32, i32, i32, i32, i32, f32, V, V, sz, V, V]
    L.nv_paged_decode_attn.restype = ctypes.c_int
    L.nv_sample_workspace_size.argtypes = [i32, i32]
    L.nv_sample_workspace_size.restype = sz
    L.nv_sample_exponential_race.argtypes = [V, i64, V, V, i64, i32, i32, V, V, sz, V, V]
    L.nv_sample_exponential_race.restype = ctypes.c_int
    L.nv_prepare_decode.argtypes = [V, V, i32, i32, i32, i32, i32, V, V, V, V, V]
    L.nv_prepare_decode.restype = ctypes.c_int
    L.nv_prepare_prefill.argtypes = [V, V, V, i32, i32, i32, i32, i32, V, V, V, V, V, V, V]
    L.nv_prepare_prefill.restype = ctypes.c_int
    L.nv_qk_norm_rope_store.argtypes = [V, i64, V, V, V, f32, f32, V, i32, i32, i32, i32, V, V, V, i64, V, V]
    L.nv_qk_norm_rope_store.restype = ctypes.c_int
    L.nv_store_decode_attn.argtypes = [V, V, i64, V, i64, V, V, V, V, i32, V, i32, i32, i32, i32, i32, i32, i32, f32,
                                       V, V, sz, V, V]
    L.nv_store_decode_attn.restype = ctypes.c_int
    L.nv_paged_decode_attn_noalloc.argtypes = [V, V, V, V, i32, V, i32, i32, i32, i32, i32, i32, i32, f32, V, V, V]
    L.nv_paged_decode_attn_noalloc.restype = ctypes.c_int
    L.nv_paged_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.nv_paged_prefill_workspace_size.restype = sz
    L.nv_paged_prefill_attn.argtypes = [V, V, V, V, V, V, i32, i32, i32, i32, i32, i32, i32, i32, i32, f32, V, V, sz,
                                        V, V]
    L.nv_paged_prefill_attn.restype = ctypes.c_int
    if path is None:
        _lib = L
    return L


def _check(fn, rc):
    if rc != NV_OK:
        raise NvError(fn, rc, load_library().nv_status_string(rc).decode())


def _ptr(t):
    return None if t is None else t.data_ptr()      # ctypes passes an int as the c_void_p argument


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream                            # an int, passed as the c_void_p argument


def _need(cond, msg):
    """Raise ValueError(msg) unless ``cond``; ``msg`` may be a callable, formatted only on failure."""
    if not cond:
        raise ValueError(msg() if callable(msg) else msg)


def _dtypes(bf16=(), i32=(), f32=()):
    """Each (name, tensor) pair has the element type the C entry point reads (None = absent)."""
    import torch
    for want, group in ((torch.bfloat16, bf16), (torch.int32, i32), (torch.float32, f32)):
        for name, t in group:
            if t is not None and t.dtype != want:
                raise ValueError(f"{name} must be {str(want).replace('torch.', '')}, not {t.dtype}")


def _on_one_gpu(*named):
    """Every tensor given (None = absent) lives on the same CUDA device; returns that device."""
    first = None
    for name, t in named:
        if t is None:
            continue
        _need(t.is_cuda, lambda: f"{name} must be a CUDA tensor (it is on {t.device})")
        if first is None:
            first, idx = t, t.get_device()
        elif t.get_device() != idx:
            raise ValueError(f"{name} is on {t.device}, the other tensors on {first.device}")
    return None if first is None else first.device


# Default workspaces: one per (device, stream, kind), grown when a call needs more and kept, so a
# call that passes none allocates only the first time (or when a batch outgrows it) instead of
# every step.  Keyed by stream because calls on one stream never overlap; zero-filled when made
# (the decode and sampler workspaces keep their counters zero between calls).  Not used under
# CUDA-graph capture, where the caller must pass a workspace the graph can own.
_ws_lock = threading.Lock()
_ws_cache: dict = {}


def _default_workspace(kind: str, nbytes: int, device, stream):
    import torch
    _need(not torch.cuda.is_current_stream_capturing(),
          "pass a workspace when capturing a CUDA graph (the default one is not allocated during capture)")
    s = torch.cuda.current_stream(device) if stream is None else stream
    key = (device.index, s.cuda_stream, kind)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            size = 1 << max(12, (int(nbytes) - 1).bit_length())      # a power of two: few regrowths
            with torch.cuda.stream(s):      # allocated on the stream that uses it
                ws = torch.zeros(size, dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
        return ws


def _pool_shape(k_cache, v_cache):
    _need(k_cache.dim() == 4 and k_cache.shape == v_cache.shape,
          "caches must be [num_blocks, block_size, num_kv_heads, head_dim]")
    _need(k_cache.is_contiguous() and v_cache.is_contiguous(), "caches must be contiguous")
    return tuple(int(x) for x in k_cache.shape)


def nv_store_kvcache(k, v, slot_mapping, k_cache, v_cache, d_err=None, stream=None):
    """Scatter ``k``/``v`` rows ``[N, Hkv, D]`` into ``k_cache``/``v_cache`` at ``slot_mapping`` (-1 = skip).

    ``k`` and ``v`` need contiguous heads and may have any row stride (e.g. ``v`` a view
    into a fused QKV output).  Caches are ``[num_blocks, block_size, Hkv, D]`` contiguous."""
    nb, bs, hkv, d = _pool_shape(k_cache, v_cache)
    _need(slot_mapping.dim() == 1 and slot_mapping.is_contiguous(), "slot_mapping must be a contiguous [N]")
    n = int(slot_mapping.shape[0])
    for name, t in (("k", k), ("v", v)):
        _need(t.dim() == 3 and tuple(t.shape) == (n, hkv, d), lambda: f"{name} must be [N, Hkv, D] = {(n, hkv, d)}")
        _need(t.stride(2) == 1 and t.stride(1) == d, lambda: f"{name} heads must be contiguous")
    _dtypes(bf16=(("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache)),
            i32=(("slot_mapping", slot_mapping), ("d_err", d_err)))
    _on_one_gpu(("k", k), ("v", v), ("slot_mapping", slot_mapping), ("k_cache", k_cache), ("v_cache", v_cache),
                ("d_err", d_err))
    rc = load_library().nv_store_kvcache(_ptr(k), k.stride(0), _ptr(v), v.stride(0), _ptr(slot_mapping), n,
                                         _ptr(k_cache), _ptr(v_cache), nb * bs, hkv, d, _ptr(d_err), _stream(stream))
    _check("nv_store_kvcache", rc)


def release_default_workspaces():
    """Drop the workspaces the calls below allocate when none is passed (the next call makes fresh,
    zero-filled ones).  Call it after a decode or sampler call flagged NV_DERR_VALUE, whose counters
    are then no longer known to be zero, or to give the memory back."""
    with _ws_lock:
        _ws_cache.clear()


def _ws_arg(workspace, name):
    """(pointer, bytes) of a caller-supplied uint8 workspace on the call's device."""
    import torch
    if workspace is None:
        return None, 0
    _need(workspace.dtype == torch.uint8 and workspace.is_contiguous(), lambda: f"{name} must be a contiguous uint8 tensor")
    return _ptr(workspace), workspace.numel()


def _check_out(out, shape, name="out"):
    """A caller's output tensor (None = allocate one) has the shape, bf16 type and layout written."""
    import torch
    if out is None:
        return
    _need(tuple(out.shape) == tuple(shape), lambda: f"{name} must be {tuple(shape)}, not {tuple(out.shape)}")
    _need(out.dtype == torch.bfloat16, lambda: f"{name} must be bfloat16, not {out.dtype}")
    _need(out.is_contiguous(), lambda: f"{name} must be contiguous")


def _out_like(out, ref, shape):
    import torch
    return torch.empty(shape, dtype=torch.bfloat16, device=ref.device) if out is None else out


def _vec(t, name, n=None):
    _need(t.dim() == 1 and t.is_contiguous(), lambda: f"{name} must be a contiguous 1-D tensor")
    _need(n is None or int(t.shape[0]) == n, lambda: f"{name} must have {n} entries, not {int(t.shape[0])}")


def _table(bt, rows):
    _need(bt.dim() == 2 and int(bt.shape[0]) == rows and bt.stride(1) == 1,
          "block_tables must be [B, W] with unit column stride")


def nv_sample_exponential_race(logits, temperatures, draws, tokens=None, workspace=None, d_err=None, stream=None):
    """Token per row: argmax_i softmax(logits / T)_i / max(E_i, 1e-10) with ``draws`` E (int64 ``[B]``).

    ``workspace`` (uint8, ``nv_sample_workspace_size`` bytes, zero-filled once) defaults to one kept
    per device and stream."""
    import torch
    _need(logits.dim() == 2 and logits.stride(1) == 1 and draws.dim() == 2 and draws.stride(1) == 1,
          "logits and draws must be [B, V] with unit column stride")
    B, V = (int(x) for x in logits.shape)
    _need(tuple(draws.shape) == (B, V) and int(temperatures.shape[0]) == B, "one temperature and V draws per row")
    _vec(temperatures, "temperatures", B)
    _dtypes(bf16=(("logits", logits),), f32=(("temperatures", temperatures), ("draws", draws)),
            i32=(("d_err", d_err),))
    if tokens is not None:
        _need(tuple(tokens.shape) == (B,) and tokens.dtype == torch.int64 and tokens.is_contiguous(),
              "tokens must be a contiguous int64 [B]")
    dev = _on_one_gpu(("logits", logits), ("temperatures", temperatures), ("draws", draws), ("tokens", tokens),
                      ("workspace", workspace), ("d_err", d_err))
    if tokens is None:
        tokens = torch.empty(B, dtype=torch.int64, device=dev)
    if workspace is None:
        workspace = _default_workspace("sampler", max(int(load_library().nv_sample_workspace_size(B, V)), 16), dev,
                                       stream)
    ws_p, ws_n = _ws_arg(workspace, "workspace")
    rc = load_library().nv_sample_exponential_race(_ptr(logits), logits.stride(0), _ptr(temperatures), _ptr(draws),
                                                   draws.stride(0), B, V, _ptr(tokens), ws_p, ws_n, _ptr(d_err),
                                                   _stream(stream))
    _check("nv_sample_exponential_race", rc)
    return tokens


def nv_prepare_decode(seq_lens, block_tables, block_size, num_blocks, padded_seqs=None, out=None, d_err=None,
                      stream=None):
    """Device-side decode metadata: returns ``(context_lens, positions, slot_mapping)`` int32 ``[padded]``
    for sequences of ``seq_lens`` tokens (new token included) over ``block_tables``."""
    import torch
    _vec(seq_lens, "seq_lens")
    B = int(seq_lens.shape[0])
    pad = B if padded_seqs is None else int(padded_seqs)
    _need(pad >= B, "padded_seqs must be >= the number of sequences")
    _need(block_tables.dim() == 2 and block_tables.shape[0] >= B and block_tables.stride(1) == 1,
          "block_tables must be [B, W] with unit column stride")
    if out is not None:
        _need(len(out) == 3, "out must be (context_lens, positions, slot_mapping)")
        for name, t in zip(("context_lens", "positions", "slot_mapping"), out):
            _vec(t, name, pad)
    named = [("seq_lens", seq_lens), ("block_tables", block_tables), ("d_err", d_err)]
    if out is not None:
        named += list(zip(("context_lens", "positions", "slot_mapping"), out))
    _dtypes(i32=named)
    dev = _on_one_gpu(*named)
    if out is None:
        out = tuple(torch.empty(pad, dtype=torch.int32, device=dev) for _ in range(3))
    cl, pos, sm = out
    rc = load_library().nv_prepare_decode(_ptr(seq_lens), _ptr(block_tables), block_tables.stride(0), B, pad,
                                          int(block_size), int(num_blocks), _ptr(cl), _ptr(pos), _ptr(sm), _ptr(d_err),
                                          _stream(stream))
    _check("nv_prepare_decode", rc)
    return cl, pos, sm


def nv_prepare_prefill(num_cached, num_scheduled, block_tables, block_size, num_blocks, total_q, d_err=None,
                       stream=None):
    """Device-side prefill metadata: returns ``(cu_seqlens_q, cu_seqlens_k, positions, slot_mapping, max_seqlens)``."""
    import torch
    _vec(num_cached, "num_cached")
    B = int(num_cached.shape[0])
    _vec(num_scheduled, "num_scheduled", B)
    _need(block_tables.dim() == 2 and block_tables.shape[0] >= B and block_tables.stride(1) == 1,
          "block_tables must be [B, W] with unit column stride")
    named = (("num_cached", num_cached), ("num_scheduled", num_scheduled), ("block_tables", block_tables),
             ("d_err", d_err))
    _dtypes(i32=named)
    dev = _on_one_gpu(*named)
    cq = torch.empty(B + 1, dtype=torch.int32, device=dev)
    ck = torch.empty(B + 1, dtype=torch.int32, device=dev)
    pos = torch.empty(max(int(total_q), 1), dtype=torch.int32, device=dev)
    sm = torch.empty(max(int(total_q), 1), dtype=torch.int32, device=dev)
    mx = torch.empty(2, dtype=torch.int32, device=dev)
    rc = load_library().nv_prepare_prefill(_ptr(num_cached), _ptr(num_scheduled), _ptr(block_tables),
                                           block_tables.stride(0), B, int(total_q), int(block_size), int(num_blocks),
                                           _ptr(cq), _ptr(ck), _ptr(pos), _ptr(sm), _ptr(mx), _ptr(d_err),
                                           _stream(stream))
    _check("nv_prepare_prefill", rc)
    return cq, ck, pos[:int(total_q)], sm[:int(total_q)], mx


def nv_qk_norm_rope_store(qkv, positions, q_norm_weight, k_norm_weight, slot_mapping, k_cache, v_cache,
                          num_q_heads, rms_eps=1e-6, rope_theta=1e6, q_out=None, d_err=None, stream=None):
    """QK-norm + RoPE on the q and k heads of ``qkv`` ``[N, (Hq + 2 Hkv) * D]`` (rows may be strided),
    roped q returned (``[N, Hq, D]``), roped k and v stored at ``slot_mapping`` (-1 = skip)."""
    nb, bs, hkv, d = _pool_shape(k_cache, v_cache)
    _need(qkv.dim() == 2 and qkv.stride(1) == 1, "qkv must be [N, row] with unit column stride")
    n = int(qkv.shape[0])
    _need(int(qkv.shape[1]) >= (num_q_heads + 2 * hkv) * d, "qkv rows are too short for q | k | v")
    _need(int(positions.shape[0]) == n and int(slot_mapping.shape[0]) == n, "one position and slot per token")
    _need(q_norm_weight.numel() == d and k_norm_weight.numel() == d, "norm weights must have head_dim values")
    _vec(positions, "positions", n)
    _vec(slot_mapping, "slot_mapping", n)
    _need(q_norm_weight.is_contiguous() and k_norm_weight.is_contiguous(), "norm weights must be contiguous")
    _dtypes(bf16=(("qkv", qkv), ("q_norm_weight", q_norm_weight), ("k_norm_weight", k_norm_weight),
                  ("k_cache", k_cache), ("v_cache", v_cache)),
            i32=(("positions", positions), ("slot_mapping", slot_mapping), ("d_err", d_err)))
    _check_out(q_out, (n, int(num_q_heads), d), "q_out")
    _on_one_gpu(("qkv", qkv), ("positions", positions), ("q_norm_weight", q_norm_weight),
                ("k_norm_weight", k_norm_weight), ("slot_mapping", slot_mapping), ("k_cache", k_cache),
                ("v_cache", v_cache), ("q_out", q_out), ("d_err", d_err))
    q_out = _out_like(q_out, qkv, (n, int(num_q_heads), d))
    rc = load_library().nv_qk_norm_rope_store(
        _ptr(qkv), qkv.stride(0), _ptr(positions), _ptr(q_norm_weight), _ptr(k_norm_weight), float(rms_eps),
        float(rope_theta), _ptr(slot_mapping), n, int(num_q_heads), hkv, d, _ptr(q_out), _ptr(k_cache),
        _ptr(v_cache), nb * bs, _ptr(d_err), _stream(stream))
    _check("nv_qk_norm_rope_store", rc)
    return q_out


def nv_paged_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len) -> int:
    return int(load_library().nv_paged_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len))


def _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, d_err, workspace=None, new_rows=()):
    """Shared checks of the decode entry points (``new_rows``: the fused store's bf16 ``k``, ``v``
    and int32 ``slot_mapping``, as (name, tensor) pairs); returns (pool shape, B, Hq, out)."""
    nb, bs, hkv, d = _pool_shape(k_cache, v_cache)
    _need(q.dim() == 3, "q must be contiguous [B, Hq, D]")
    B, hq, dq = (int(x) for x in q.shape)
    _need(dq == d and q.is_contiguous(), "q must be contiguous [B, Hq, D]")
    _table(block_tables, B)
    _vec(context_lens, "context_lens", B)
    _dtypes(bf16=(("q", q), ("k_cache", k_cache), ("v_cache", v_cache)) + tuple(new_rows[:2]),
            i32=(("block_tables", block_tables), ("context_lens", context_lens), ("d_err", d_err))
            + tuple(new_rows[2:]))
    _check_out(out, (B, hq, d))
    _on_one_gpu(("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("block_tables", block_tables),
                ("context_lens", context_lens), ("out", out), ("d_err", d_err), ("workspace", workspace), *new_rows)
    return (nb, bs, hkv, d), B, hq, _out_like(out, q, (B, hq, d))


def nv_paged_decode_attn(q, k_cache, v_cache, block_tables, context_lens, scale, out=None, max_context_len=None,
                         workspace=None, d_err=None, stream=None):
    """Decode attention: ``q`` ``[B, Hq, D]`` over each sequence's ``context_lens[b]`` keys.

    ``max_context_len`` (a host int bounding every context length) sizes the split-KV grid;
    by default it is the block table's capacity ``W * block_size``, which needs no device
    read.  ``workspace`` (uint8): when not given, one kept per device and stream is used (made
    zero-filled, grown when a batch needs more); a workspace passed in must have been zero-filled
    when it was allocated (its split counters are zero between calls), and may then be reused
    for any batch."""
    (nb, bs, hkv, d), B, hq, out = _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, d_err,
                                                 workspace)
    if max_context_len is None:
        max_context_len = int(block_tables.shape[1]) * bs
    ws_need = nv_paged_decode_workspace_size(B, hq, d, int(max_context_len))
    if workspace is None and ws_need:
        workspace = _default_workspace("decode", ws_need, q.device, stream)
    ws_p, ws_n = _ws_arg(workspace, "workspace")
    rc = load_library().nv_paged_decode_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.stride(0), _ptr(context_lens), B, hq,
        hkv, d, bs, nb, int(max_context_len), float(scale), _ptr(out), ws_p, ws_n, _ptr(d_err), _stream(stream))
    _check("nv_paged_decode_attn", rc)
    return out


def nv_store_decode_attn(q, k, v, slot_mapping, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                         max_context_len=None, workspace=None, d_err=None, stream=None):
    """Store each sequence's new K/V row (``k``/``v`` ``[B, Hkv, D]`` at ``slot_mapping``) and run decode
    attention over the history that ends with it, in one pass (same result as ``nv_store_kvcache``
    then ``nv_paged_decode_attn``).  ``workspace`` as for ``nv_paged_decode_attn``."""
    nb, bs, hkv, d = _pool_shape(k_cache, v_cache)
    _need(q.dim() == 3, "q must be contiguous [B, Hq, D]")
    B = int(q.shape[0])
    _need(slot_mapping.dim() == 1 and int(slot_mapping.shape[0]) == B,
          "slot_mapping must have one entry per sequence")
    _vec(slot_mapping, "slot_mapping", B)
    for name, t in (("k", k), ("v", v)):
        _need(t.dim() == 3 and tuple(t.shape) == (B, hkv, d), lambda: f"{name} must be [B, Hkv, D] = {(B, hkv, d)}")
        _need(t.stride(2) == 1 and t.stride(1) == d, lambda: f"{name} heads must be contiguous")
    (nb, bs, hkv, d), B, hq, out = _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, d_err,
                                                 workspace, (("k", k), ("v", v), ("slot_mapping", slot_mapping)))
    if max_context_len is None:
        max_context_len = int(block_tables.shape[1]) * bs
    ws_need = nv_paged_decode_workspace_size(B, hq, d, int(max_context_len))
    if workspace is None and ws_need:
        workspace = _default_workspace("decode", ws_need, q.device, stream)
    ws_p, ws_n = _ws_arg(workspace, "workspace")
    rc = load_library().nv_store_decode_attn(
        _ptr(q), _ptr(k), k.stride(0), _ptr(v), v.stride(0), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), block_tables.stride(0), _ptr(context_lens), B, hq, hkv, d, bs, nb, int(max_context_len),
        float(scale), _ptr(out), ws_p, ws_n, _ptr(d_err), _stream(stream))
    _check("nv_store_decode_attn", rc)
    return out


def nv_paged_decode_attn_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                                 max_context_len=None, d_err=None, stream=None):
    """``nv_paged_decode_attn`` for callers that cannot allocate device memory: no workspace, the
    split-KV partials live in a fixed array inside the library (see the C header for the limit).
    Calls sharing that array must not overlap on the GPU.  ``out`` must be given to allocate nothing."""
    (nb, bs, hkv, d), B, hq, out = _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, d_err)
    if max_context_len is None:
        max_context_len = int(block_tables.shape[1]) * bs
    rc = load_library().nv_paged_decode_attn_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.stride(0), _ptr(context_lens), B, hq,
        hkv, d, bs, nb, int(max_context_len), float(scale), _ptr(out), _ptr(d_err), _stream(stream))
    _check("nv_paged_decode_attn_noalloc", rc)
    return out


def nv_paged_prefill_workspace_size(num_seqs, total_q, max_seqlen_q, num_q_heads, num_kv_heads) -> int:
    return int(load_library().nv_paged_prefill_workspace_size(num_seqs, total_q, max_seqlen_q, num_q_heads,
                                                              num_kv_heads))


def nv_paged_prefill_attn(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, scale, max_seqlen_q=None,
                          out=None, workspace=None, d_err=None, stream=None):
    """Causal varlen prefill: packed ``q`` ``[total_q, Hq, D]`` over cached prefix + chunk.

    ``max_seqlen_q`` (host int) bounds every chunk's length; by default ``total_q``, an upper
    bound that needs no device read.  ``workspace`` (uint8, ``nv_paged_prefill_workspace_size``
    bytes): when not given, one kept per device and stream is used (grown when a batch needs more)."""
    nb, bs, hkv, d = _pool_shape(k_cache, v_cache)
    _need(q.dim() == 3, "q must be contiguous [total_q, Hq, D]")
    total_q, hq, dq = (int(x) for x in q.shape)
    _need(dq == d and q.is_contiguous(), "q must be contiguous [total_q, Hq, D]")
    B = int(cu_seqlens_q.shape[0]) - 1
    _need(int(cu_seqlens_k.shape[0]) == B + 1, "cu_seqlens_q and cu_seqlens_k must both have B+1 entries")
    _table(block_tables, B)
    _vec(cu_seqlens_q, "cu_seqlens_q")
    _vec(cu_seqlens_k, "cu_seqlens_k")
    _dtypes(bf16=(("q", q), ("k_cache", k_cache), ("v_cache", v_cache)),
            i32=(("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k), ("block_tables", block_tables),
                 ("d_err", d_err)))
    _check_out(out, (total_q, hq, d))
    _on_one_gpu(("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("cu_seqlens_q", cu_seqlens_q),
                ("cu_seqlens_k", cu_seqlens_k), ("block_tables", block_tables), ("out", out), ("d_err", d_err),
                ("workspace", workspace))
    out = _out_like(out, q, (total_q, hq, d))
    mq = int(total_q if max_seqlen_q is None else max_seqlen_q)
    if workspace is None and B > 0 and total_q > 0 and mq > 0:
        workspace = _default_workspace("prefill", nv_paged_prefill_workspace_size(B, total_q, mq, hq, hkv), q.device,
                                       stream)
    ws_p, ws_n = _ws_arg(workspace, "workspace")
    rc = load_library().nv_paged_prefill_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(block_tables),
        block_tables.stride(0), B, total_q, mq, hq, hkv, d, bs, nb, float(scale), _ptr(out), ws_p, ws_n,
        _ptr(d_err), _stream(stream))
    _check("nv_paged_prefill_attn", rc)
    return out
