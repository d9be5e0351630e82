"""nv_paged_prefill_attn on the GPU against the oracle (store the chunk first, then prefill)."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gpu_util import (ORACLE_THREADS, DeviceBatch, compare, host_bits, host_f32, oracle_cache_after_store,
                            oracle_prefill, oracle_store_in_place)

pytestmark = pytest.mark.gpu


def _run(batch, max_seqlen_q=None):
    db = DeviceBatch(batch)
    db.store()
    out = db.prefill(max_seqlen_q)
    assert db.err() == 0
    kc1, vc1 = oracle_cache_after_store(oracle.default(), batch, db.kc_host0, db.vc_host0)
    return db, host_f32(out), kc1, vc1


CASES = [
    # name, prefix lens, chunk lens, Hq, Hkv, block_size
    ("g2-bs256-fresh", [0, 0], [1, 300], 16, 8, 256),
    ("g2-bs256-prefix", [256, 512, 0, 1024], [64, 65, 128, 200], 16, 8, 256),
    ("g2-bs16-ragged", [0, 48, 16, 160], [63, 1, 129, 77], 16, 8, 16),
    ("g1-bs64", [64, 0, 320], [130, 5, 300], 8, 8, 64),
    ("g4-bs128", [128, 0, 256], [33, 97, 250], 32, 8, 128),
    ("g8-bs32", [32, 0], [40, 17], 16, 2, 32),
    ("g16-bs256", [256], [20], 16, 1, 256),
    ("unaligned-prefix", [100, 37, 255], [60, 200, 3], 16, 8, 16),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_shapes(case):
    name, P, Lq, hq, hkv, bs = case
    b = W.make_prefill(name, 31, P, Lq, hq, hkv, 128, bs, poison_tail=True)
    db, got, kc, vc = _run(b)
    want = oracle_prefill(oracle.default(), b, kc, vc)
    compare(got, want, name)


def test_prefill_single_key_is_exact():
    b = W.make_prefill("one", 32, [0], [1], 16, 8, 128, 256, poison_tail=True)
    db = DeviceBatch(b)
    db.store()
    bits = host_bits(db.prefill())
    g = 2
    for h in range(16):
        assert np.array_equal(bits[0, h], b.v_new[0, h // g])


def test_prefill_chunked_equals_full():
    """One sequence prefilled whole, and as a cached prefix + chunk over the same pool."""
    import torch
    import paged_kv_attention_store_gb300 as nv
    from tests.gpu_util import dev_i32
    full = W.make_prefill("full", 33, [0], [700], 16, 8, 128, 64)
    db = DeviceBatch(full)
    db.store()
    out_full = host_f32(db.prefill())
    P = 384
    out_chunk = nv.nv_paged_prefill_attn(db.q[P:].contiguous(), db.k_cache, db.v_cache, dev_i32(np.array([0, 700 - P])),
                                         dev_i32(np.array([0, 700])), db.block_tables, full.scale)
    compare(host_f32(out_chunk), out_full[P:], "chunk vs full")


def test_prefill_last_row_equals_decode():
    b = W.make_prefill("lastrow", 34, [128, 0], [77, 200], 16, 8, 128, 64)
    db = DeviceBatch(b)
    db.store()
    out = host_f32(db.prefill())
    import paged_kv_attention_store_gb300 as nv
    from tests.gpu_util import dev_i32
    last = b.cu_seqlens_q[1:] - 1
    q_last = db.q[last.tolist()].contiguous()
    dec = nv.nv_paged_decode_attn(q_last, db.k_cache, db.v_cache, db.block_tables, db.seq_lens, b.scale)
    compare(host_f32(dec), out[last], "decode vs last prefill row")


def test_prefill_chunk_budget_full_size():
    """The chunked-prefill workload at full size (16 sequences, 16384 new tokens, prefixes up to
    2048): every query row and head compared element by element with the oracle."""
    b = W.prefill_chunk()
    db = DeviceBatch(b)
    db.store()
    got = host_f32(db.prefill())
    assert db.err() == 0
    kc, vc = oracle_store_in_place(oracle.default(), b, db.kc_host0, db.vc_host0)
    want = oracle_prefill(oracle.default(), b, kc, vc, threads=ORACLE_THREADS)
    compare(got, want, "prefill chunk budget")


def test_prefill_grid_hint_smaller_than_chunk_is_flagged():
    import paged_kv_attention_store_gb300 as nv
    b = W.make_prefill("hint", 35, [0], [300], 16, 8, 128, 256)
    db = DeviceBatch(b)
    db.store()
    db.prefill(max_seqlen_q=100)
    assert db.err() & nv.NV_DERR_LENGTH


def test_prefill_many_sequences_and_long_chunk_sampled():
    """1200 sequences (more than the pre-pass has threads, and many sharing one sort bucket) with
    short chunks over assorted prefixes, plus one 2500-token chunk (more query tiles than a warp
    has lanes): every listed tile must be computed once, whatever its place in the work list."""
    rng = np.random.default_rng(7)
    n = 1200
    prefix = (rng.integers(0, 9, n) * 64).tolist() + [300]
    chunk = rng.integers(1, 40, n).tolist() + [2500]
    b = W.make_prefill("many", 41, prefix, chunk, 16, 8, 128, 64)
    db, got, kc, vc = _run(b)
    cu = b.cu_seqlens_q
    rows = set(rng.choice(int(cu[-1]) - 2500, 160, replace=False).tolist())
    lo = int(cu[-2])
    rows |= {lo, lo + 63, lo + 64, lo + 2047, lo + 2048, lo + 2111, lo + 2112, lo + 2499}
    rows |= set((lo + rng.choice(2500, 40, replace=False)).tolist())
    rows = np.array(sorted(rows), np.int64)
    want = oracle_prefill(oracle.default(), b, kc, vc, rows=rows, threads=ORACLE_THREADS)
    compare(got[rows], want, "prefill many sequences")


def test_prefill_at_the_sequence_limit():
    """65535 sequences (the most the work list addresses; one more is refused on the host), chunks of
    1-3 tokens over prefixes of 0-32, group 8 (8 q / 1 kv head), block size 16: every row against the
    oracle."""
    rng = np.random.default_rng(43)
    n = 65535
    b = W.make_prefill("max-seqs", 43, (rng.integers(0, 3, n) * 16).tolist(), rng.integers(1, 4, n).tolist(),
                       8, 1, 128, 16)
    shape = (b.num_blocks, b.block_size, b.num_kv_heads, b.head_dim)
    kc0, vc0 = W.normal_bf16(rng, shape), W.normal_bf16(rng, shape)   # one draw each: quick to build
    db = DeviceBatch(b, kc0, vc0)
    db.store()
    got = host_f32(db.prefill())
    assert db.err() == 0
    kc, vc = oracle_cache_after_store(oracle.default(), b, kc0, vc0)
    compare(got, oracle_prefill(oracle.default(), b, kc, vc, threads=ORACLE_THREADS), "65535 sequences")

