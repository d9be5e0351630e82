"""CPU oracle for the paged KV attention store -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The product library never does, and this
package imports nothing from it.

Two independent statements of what the hot path computes:

* ``oracle.c`` (loaded through ctypes): plain single-threaded C that follows the
  nano-vLLM field guide's definitions, query by query, key by key, in float.
* ``brute``: a NumPy float64 brute force on tiny inputs that un-pages the pool into
  contiguous per-sequence K/V through the 4-D ``[blocks, bs, Hkv, D]`` view and
  applies a dense masked softmax.  It exists to pin the C oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_default = None

_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]


def compile_c(src_path: str, out_path: str) -> str:
    """Compile one oracle C source into a shared library (gcc, no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", *_CFLAGS, src_path, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` if it is missing or stale."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_c(_SRC, _LIB_PATH)
    return _LIB_PATH


def _load(path: str):
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    L.oracle_slot_of.argtypes = [P, i32, i32]
    L.oracle_slot_of.restype = i32
    L.oracle_store_kvcache.argtypes = [P, i64, P, i64, P, i64, P, P, i64, i32]
    L.oracle_store_kvcache.restype = i64
    L.oracle_decode_attn.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, f32, P]
    L.oracle_decode_attn.restype = i32
    L.oracle_prefill_attn.argtypes = [P, P, P, P, P, P, i32, i32, P, i64, i32, i32, i32, i32, f32, P]
    L.oracle_prefill_attn.restype = i32
    L.oracle_qk_norm_rope_store.argtypes = [P, i64, P, P, P, f32, f32, P, i64, i32, i32, i32, P, P, P, i64]
    L.oracle_qk_norm_rope_store.restype = i64
    L.oracle_prepare_decode.argtypes = [P, P, i32, i32, i32, i32, P, P, P]
    L.oracle_prepare_decode.restype = i64
    L.oracle_prepare_prefill.argtypes = [P, P, P, i32, i32, i32, P, P, P, P, P]
    L.oracle_prepare_prefill.restype = i64
    L.oracle_sample_exponential_race.argtypes = [P, i64, P, P, i64, i32, i32, P]
    L.oracle_sample_exponential_race.restype = None
    return L


def lib():
    """The ctypes handle of the default oracle library (built on first use)."""
    return default().lib


def default() -> "Oracle":
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """Thin ctypes wrapper around one compiled copy of ``oracle.c``."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        self.lib = _load(lib_path)

    def slot_of(self, table, pos: int, block_size: int) -> int:
        t = _c(table, np.int32)
        return int(self.lib.oracle_slot_of(_ptr(t), int(pos), int(block_size)))

    def store_kvcache(self, k, v, slot_mapping, k_cache, v_cache) -> int:
        """Scatter new K/V rows into ``k_cache``/``v_cache`` in place; return the number of rejected slots.

        ``k``/``v``: uint16 ``[N, Hkv, D]`` or 2-D ``[N, stride]`` views whose first ``Hkv*D``
        columns are the row (row stride taken from the array).  Caches: uint16, any shape whose
        trailing dims flatten to ``[num_slots, Hkv*D]``, C-contiguous (modified in place).
        """
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
        sm = _c(slot_mapping, np.int32)
        n = sm.shape[0]
        row_elems = int(np.prod(k_cache.shape[2:])) if k_cache.ndim == 4 else int(k_cache.shape[-1])
        num_slots = k_cache.size // row_elems

        def rowview(x):
            x = np.asarray(x)
            assert x.dtype == np.uint16
            if x.ndim == 3:
                assert x.strides[2] == 2 and x.strides[1] == x.shape[2] * 2
            base = x.reshape(n, -1) if x.flags.c_contiguous else x
            stride = base.strides[0] // 2 if n > 0 else row_elems
            return base, stride

        kb, ks = rowview(k)
        vb, vs = rowview(v)
        return int(self.lib.oracle_store_kvcache(_ptr(kb), ks, _ptr(vb), vs, _ptr(sm), n, _ptr(k_cache),
                                              _ptr(v_cache), num_slots, row_elems))

    def decode_attn(self, q, k_cache, v_cache, block_tables, context_lens, num_kv_heads, block_size, scale,
                    threads: int = 1):
        """float32 ``[B, Hq, D]`` attention of each sequence's single query over its L keys.

        ``threads > 1`` splits sequences across Python threads (each runs the single-threaded
        C routine on its own range; ctypes releases the GIL)."""
        q = _c(q, np.uint16)
        B, hq, d = q.shape
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        kc = _c(k_cache, np.uint16)
        vc = _c(v_cache, np.uint16)
        out = np.zeros((B, hq, d), np.float32)
        L = self.lib

        def run(lo, hi):
            rc = L.oracle_decode_attn(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl), lo, hi,
                                      hq, int(num_kv_heads), d, int(block_size), float(scale), _ptr(out))
            assert rc == 0, rc

        _parallel(run, B, threads)
        return out

    def prefill_attn(self, q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, num_kv_heads, block_size,
                     scale, rows=None, threads: int = 1):
        """float32 ``[len(rows), Hq, D]`` causal attention of packed query rows over prefix + chunk."""
        q = _c(q, np.uint16)
        total_q, hq, d = q.shape
        cq = _c(cu_seqlens_q, np.int32)
        ck = _c(cu_seqlens_k, np.int32)
        bt = _c(block_tables, np.int32)
        kc = _c(k_cache, np.uint16)
        vc = _c(v_cache, np.uint16)
        rows = np.arange(total_q, dtype=np.int64) if rows is None else _c(rows, np.int64)
        out = np.zeros((rows.shape[0], hq, d), np.float32)
        L = self.lib

        def run(lo, hi):
            sub_rows = rows[lo:hi]
            sub_out = np.zeros((hi - lo, hq, d), np.float32)
            rc = L.oracle_prefill_attn(_ptr(q), _ptr(kc), _ptr(vc), _ptr(cq), _ptr(ck), _ptr(bt), bt.shape[1],
                                       cq.shape[0] - 1, _ptr(sub_rows), hi - lo, hq, int(num_kv_heads), d,
                                       int(block_size), float(scale), _ptr(sub_out))
            assert rc == 0, rc
            out[lo:hi] = sub_out

        _parallel(run, rows.shape[0], threads)
        return out

    def qk_norm_rope_store(self, qkv, positions, q_weight, k_weight, eps, theta, slot_mapping, num_q_heads,
                           num_kv_heads, k_cache, v_cache):
        """QK-norm + RoPE + store: returns ``(q_out [N, Hq, D] uint16, rejected)``; stores into the caches.

        ``qkv``: uint16 ``[N, row_stride]`` (q | k | v per row); caches as for ``store_kvcache``."""
        qkv = np.asarray(qkv)
        assert qkv.dtype == np.uint16 and qkv.ndim == 2 and qkv.strides[1] == 2
        n = qkv.shape[0]
        d = int(np.asarray(q_weight).shape[0])
        pos = _c(positions, np.int32)
        sm = _c(slot_mapping, np.int32)
        qw, kw = _c(q_weight, np.uint16), _c(k_weight, np.uint16)
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        num_slots = k_cache.size // (num_kv_heads * d)
        q_out = np.zeros((n, num_q_heads, d), np.uint16)
        stride = qkv.strides[0] // 2 if n else qkv.shape[1]
        rej = self.lib.oracle_qk_norm_rope_store(_ptr(qkv), stride, _ptr(pos), _ptr(qw), _ptr(kw), float(eps),
                                                 float(theta), _ptr(sm), n, int(num_q_heads), int(num_kv_heads), d,
                                                 _ptr(q_out), _ptr(k_cache), _ptr(v_cache), num_slots)
        return q_out, int(rej)

    def prepare_decode(self, seq_lens, block_tables, block_size, padded_seqs=None):
        """``(context_lens, positions, slot_mapping, bad_rows)`` for a decode step (int32 arrays)."""
        sl = _c(seq_lens, np.int32)
        bt = _c(block_tables, np.int32)
        b = sl.shape[0]
        pad = b if padded_seqs is None else int(padded_seqs)
        cl, pos, sm = (np.zeros(pad, np.int32) for _ in range(3))
        bad = self.lib.oracle_prepare_decode(_ptr(sl), _ptr(bt), bt.shape[1], b, pad, int(block_size), _ptr(cl),
                                             _ptr(pos), _ptr(sm))
        return cl, pos, sm, int(bad)

    def prepare_prefill(self, num_cached, num_scheduled, block_tables, block_size):
        """``(cu_seqlens_q, cu_seqlens_k, positions, slot_mapping, (max_seqlen_q, max_seqlen_k))``."""
        nc, ns = _c(num_cached, np.int32), _c(num_scheduled, np.int32)
        bt = _c(block_tables, np.int32)
        b = nc.shape[0]
        total = int(ns.sum())
        cq, ck = np.zeros(b + 1, np.int32), np.zeros(b + 1, np.int32)
        pos, sm = np.zeros(max(total, 1), np.int32), np.zeros(max(total, 1), np.int32)
        mx = np.zeros(2, np.int32)
        n = self.lib.oracle_prepare_prefill(_ptr(nc), _ptr(ns), _ptr(bt), bt.shape[1], b, int(block_size), _ptr(cq),
                                            _ptr(ck), _ptr(pos), _ptr(sm), _ptr(mx))
        assert n == total, n
        return cq, ck, pos[:total], sm[:total], (int(mx[0]), int(mx[1]))

    def sample(self, logits, temperatures, draws, threads: int = 1):
        """int64 ``[B]``: argmax_i softmax(logits/T)_i / max(E_i, 1e-10) per row (first index on ties)."""
        lg = _c(logits, np.uint16)
        ex = _c(draws, np.float32)
        tm = _c(temperatures, np.float32)
        B, V = lg.shape
        out = np.zeros(B, np.int64)

        def run(lo, hi):
            sub = np.zeros(hi - lo, np.int64)
            self.lib.oracle_sample_exponential_race(_ptr(lg[lo:hi]), V, _ptr(tm[lo:hi]), _ptr(ex[lo:hi]), V, hi - lo,
                                                    V, _ptr(sub))
            out[lo:hi] = sub

        _parallel(run, B, threads)
        return out


def slot_of(table, pos, block_size):
    return default().slot_of(table, pos, block_size)


def store_kvcache(k, v, slot_mapping, k_cache, v_cache):
    return default().store_kvcache(k, v, slot_mapping, k_cache, v_cache)


def decode_attn(*args, **kw):
    return default().decode_attn(*args, **kw)


def prefill_attn(*args, **kw):
    return default().prefill_attn(*args, **kw)


def qk_norm_rope_store(*args, **kw):
    return default().qk_norm_rope_store(*args, **kw)


def _parallel(run, n, threads):
    """Run ``run(lo, hi)`` over [0, n) on ``threads`` Python threads (the C routines release the GIL).

    The range is cut into about eight pieces per thread, handed out in order as threads come free,
    so a few expensive rows (long contexts) do not leave the other threads idle."""
    threads = max(1, min(int(threads), n))
    if threads == 1:
        if n:
            run(0, n)
        return
    pieces = min(n, threads * 8)
    bounds = np.linspace(0, n, pieces + 1).astype(int)
    nxt = [0]
    lock = threading.Lock()
    errors = []

    def worker():
        while True:
            with lock:
                i = nxt[0]
                nxt[0] += 1
            if i >= pieces or errors:
                return
            try:
                run(int(bounds[i]), int(bounds[i + 1]))
            except BaseException as e:  # re-raised on the calling thread below
                errors.append(e)
                return

    ts = [threading.Thread(target=worker) for _ in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errors:
        raise errors[0]
