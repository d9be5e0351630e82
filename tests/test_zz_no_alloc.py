"""The allocation-free decode entry point, called through the C ABI, against the allocating one.

Some callers cannot allocate device memory when they run decode: an engine whose KV pool already
took all the memory its allocator may hand out, a host application that lends the library only
its tensors, or C code with no CUDA allocator at hand.  nv_paged_decode_attn_noalloc serves them:
its split-KV partials live in a fixed device array inside the library.  Two calls in a row must
each match nv_paged_decode_attn (the array keeps the previous call's contents, and nothing may
depend on them).  This file is collected last, so a run that stops at the first failure has run
every other test before it."""
import ctypes

import numpy as np
import pytest

import workloads as W
from tests.gpu_util import DeviceBatch, compare, host_f32

pytestmark = pytest.mark.gpu

V, I32, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
NV_ERR_WORKSPACE = -5


def _c_entry():
    import paged_kv_attention_store_gb300 as nv
    f = nv.load_library().nv_paged_decode_attn_noalloc
    f.argtypes = [V, V, V, V, I32, V, I32, I32, I32, I32, I32, I32, I32, F32, V, V, V]
    f.restype = ctypes.c_int
    return f


def _call(f, db, out, max_ctx):
    import torch
    b = db.b
    nb, bs, hkv, d = (int(x) for x in db.k_cache.shape)
    return f(db.q.data_ptr(), db.k_cache.data_ptr(), db.v_cache.data_ptr(), db.block_tables.data_ptr(),
             db.block_tables.stride(0), db.seq_lens.data_ptr(), b.num_seqs, b.num_q_heads, hkv, d, bs, nb,
             max_ctx, b.scale, out.data_ptr(), db.d_err.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _group8():
    ctx = np.random.default_rng([0, 200]).integers(1024, 4097, size=96)
    return W.make_decode("group8", 3, ctx, 64, 8, 128, 256, n_pad=5)


def _group16():
    return W.make_decode("group16", 4, [1, 300, 2048, 700], 128, 8, 128, 16, n_pad=2)


def _group4_mid():
    return W.qwen8_decode(num_seqs=64)


def _group2_few_long():
    return W.make_decode("group2-few-long", 8, [40000, 300], 16, 8, 128, 256, n_pad=1)


def _group4_one_long():
    return W.make_decode("group4-one-long", 9, [70000], 32, 8, 128, 256)


@pytest.mark.parametrize("make", [W.qwen06_decode, W.qwen8_decode, _group8, _group16, _group4_mid, _group2_few_long,
                                  _group4_one_long],
                         ids=["qwen3-0.6b", "qwen3-8b", "group8-tiles", "group16-tiles", "group4-64seq-tiles",
                              "group2-few-long-tiles", "group4-one-long-tiles"])
def test_noalloc_matches_allocating_entry_point_twice(make):
    import torch
    b = make()
    db = DeviceBatch(b)
    db.store()
    max_ctx = int(b.seq_lens.max())
    want = host_f32(db.decode(max_context_len=max_ctx))           # the allocating entry point
    assert db.err() == 0
    f = _c_entry()
    for call in range(2):
        out = torch.full_like(db.q, float("nan"))
        assert _call(f, db, out, max_ctx) == 0
        got = host_f32(out)
        assert db.err() == 0
        rows = b.seq_lens > 0
        compare(got[rows], want[rows], f"noalloc call {call}")
        assert not got[~rows].any()


def test_noalloc_headline_batch_coarsened_split_against_oracle():
    """The 512-sequence headline batch: its usual split (512 positions, 8 per sequence) needs more
    partials than the static array holds, so the entry point doubles the split until they fit.  Every
    sequence of that coarsened-split result is compared with the oracle itself."""
    import torch
    import oracle
    from tests.gpu_util import ORACLE_THREADS, oracle_decode, oracle_store_in_place
    b = W.qwen8_decode()
    db = DeviceBatch(b)
    db.store()
    max_ctx = int(b.seq_lens.max())
    out = torch.full_like(db.q, float("nan"))
    assert _call(_c_entry(), db, out, max_ctx) == 0
    got = host_f32(out)
    assert db.err() == 0
    kc, vc = oracle_store_in_place(oracle.default(), b, db.kc_host0, db.vc_host0)
    compare(got, oracle_decode(oracle.default(), b, kc, vc, threads=ORACLE_THREADS), "noalloc qwen8 vs oracle")


def test_noalloc_many_splits_use_the_merge_launch():
    """Three long contexts in a tiny batch are cut into 64-position splits (up to 128 per sequence),
    more than the decode kernel merges itself, so the partials in the static array are combined by
    the separate merge launch.  Two calls in a row against the allocating entry point and the oracle."""
    import torch
    import oracle
    from tests.gpu_util import oracle_cache_after_store, oracle_decode
    b = W.make_decode("long3", 5, [8192, 7999, 5000], 32, 8, 128, 256)
    db = DeviceBatch(b)
    db.store()
    max_ctx = int(b.seq_lens.max())
    want = host_f32(db.decode(max_context_len=max_ctx))
    assert db.err() == 0
    kc, vc = oracle_cache_after_store(oracle.default(), b, db.kc_host0, db.vc_host0)
    ref = oracle_decode(oracle.default(), b, kc, vc)
    f = _c_entry()
    for call in range(2):
        out = torch.full_like(db.q, float("nan"))
        assert _call(f, db, out, max_ctx) == 0
        got = host_f32(out)
        assert db.err() == 0
        compare(got, want, f"noalloc many splits, call {call}")
        compare(got, ref, f"noalloc many splits vs oracle, call {call}")


def test_noalloc_rejects_a_batch_beyond_the_static_array():
    """1024 sequences x 64 q heads (16 kv heads: group 4, the split-KV kernel) x 8192 positions need
    more partials than the array holds even at the longest split: rejected on the host, nothing
    enqueued (the pointers are never touched)."""
    f = _c_entry()
    fake = 0x10000
    rc = f(fake, fake, fake, fake, 32, fake, 1024, 64, 16, 128, 256, 64, 8192, 0.088, fake, None, None)
    assert rc == NV_ERR_WORKSPACE
