"""nv_store_decode_attn (store + decode in one pass) on the GPU.

The fused call must leave the same pool and produce the same output as ``nv_store_kvcache``
followed by ``nv_paged_decode_attn`` (bit for bit: the new rows are the same bf16 values, read
from the inputs instead of the pool), and therefore match the oracle's store-then-decode within
the attention tolerance."""
import numpy as np
import pytest

import oracle
import paged_kv_attention_store_gb300 as nv
import workloads as W
from tests.gpu_util import (ORACLE_THREADS, DeviceBatch, compare, host_bits, host_f32, oracle_cache_after_store,
                            oracle_decode, oracle_store_in_place)

pytestmark = pytest.mark.gpu


def _fused(db, slot_mapping=None, max_context_len=None):
    b = db.b
    if max_context_len is None:
        max_context_len = int(b.seq_lens.max()) if b.num_seqs else 1
    return nv.nv_store_decode_attn(db.q, db.k_new, db.v_new, db.slot_mapping if slot_mapping is None else slot_mapping,
                                   db.k_cache, db.v_cache, db.block_tables, db.seq_lens, b.scale,
                                   max_context_len=max_context_len, d_err=db.d_err)


def _fused_vs_separate(batch):
    kc, vc = batch.cache()
    sep = DeviceBatch(batch, kc, vc)
    sep.store()
    out_sep = sep.decode()
    assert sep.err() == 0
    fus = DeviceBatch(batch, kc, vc)
    out_fus = _fused(fus)
    assert fus.err() == 0
    # identical pools (every byte) and identical outputs
    assert np.array_equal(host_bits(fus.k_cache), host_bits(sep.k_cache))
    assert np.array_equal(host_bits(fus.v_cache), host_bits(sep.v_cache))
    assert np.array_equal(host_bits(out_fus), host_bits(out_sep))
    return fus, host_f32(out_fus), kc, vc


CASES = [
    # name, ctx lens, Hq, Hkv, block_size, n_pad
    ("g2-bs256", [1, 7, 255, 256, 257, 600, 1500], 16, 8, 256, 3),
    ("g4-bs64", [3, 64, 65, 700, 2049, 4100], 32, 8, 64, 0),
    ("g1-bs16", [1, 8, 9, 16, 17, 333], 8, 8, 16, 2),
    ("g8-bs32", [10, 32, 33, 900], 16, 2, 32, 1),
    ("g2-hkv16", [2, 40, 513], 32, 16, 16, 0),
    ("g8-hkv8", [1, 257, 1100, 3000], 64, 8, 256, 1),   # store pass + tile kernel, keys split
    ("g8-long", [5, 9000], 64, 8, 64, 0),
    ("g4-hkv12", [4, 129, 700], 48, 12, 32, 0),
    # group 4 with 17-40 sequences decodes on the tile kernel: store pass + tile decode
    ("g4-tiles-24", list(np.random.default_rng(5).integers(1, 3000, 24)), 32, 8, 128, 2),
    ("g4-tiles-40-bs16", list(np.random.default_rng(6).integers(1, 2000, 40)), 32, 8, 16, 0),
    # group 4, a few long contexts (>= 32768 keys in all): also the tile kernel, keys split
    ("g4-few-long", [40000, 7, 1300], 32, 8, 256, 1),
    ("g2-few-long", [35000, 3], 16, 8, 256, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_equals_store_then_decode(case):
    name, ctx, hq, hkv, bs, pad = case
    b = W.make_decode(name, 23, ctx, hq, hkv, 128, bs, n_pad=pad, poison_tail=True)
    fus, got, kc, vc = _fused_vs_separate(b)
    orc = oracle.default()
    kc1, vc1 = oracle_cache_after_store(orc, b, kc, vc)
    assert np.array_equal(host_bits(fus.k_cache), kc1)
    assert np.array_equal(host_bits(fus.v_cache), vc1)
    compare(got, oracle_decode(orc, b, kc1, vc1), name)
    assert not got[b.seq_lens == 0].any()


def test_fused_qwen06_with_padding_rows():
    """256 sequences plus 32 graph-padding rows (slot -1, context 0): every real row checked."""
    b = W.qwen06_decode()
    fus, got, kc, vc = _fused_vs_separate(b)
    orc = oracle.default()
    kc1, vc1 = oracle_cache_after_store(orc, b, kc, vc)
    compare(got[:256], oracle_decode(orc, b, kc1, vc1, threads=ORACLE_THREADS)[:256], "qwen06")
    assert not got[256:].any()


def test_fused_qwen8_full_size():
    """The headline decode batch at full size through the fused store + decode: the pool equals the
    oracle's store bit for bit, and every sequence's output matches the oracle."""
    b = W.qwen8_decode()
    fus = DeviceBatch(b)
    got = host_f32(_fused(fus))
    assert fus.err() == 0
    orc = oracle.default()
    kc, vc = oracle_store_in_place(orc, b, fus.kc_host0, fus.vc_host0)
    assert np.array_equal(host_bits(fus.k_cache), kc)
    assert np.array_equal(host_bits(fus.v_cache), vc)
    compare(got, oracle_decode(orc, b, kc, vc, threads=ORACLE_THREADS), "qwen8 fused")


def test_fused_single_key_is_the_new_v_row():
    b = W.tiny()
    fus = DeviceBatch(b)
    out = host_bits(_fused(fus))
    assert fus.err() == 0
    g = b.num_q_heads // b.num_kv_heads
    for h in range(b.num_q_heads):            # sequence 0 has L = 1: its only key is the new row
        assert np.array_equal(out[0, h], b.v_new[0, h // g])


def test_fused_rejects_a_foreign_slot():
    """A slot that is not position L-1's is not written; position L-1 is read from the pool."""
    b = W.make_decode("mismatch", 29, [300, 40, 5], 16, 8, 128, 16)
    kc, vc = b.cache()
    fus = DeviceBatch(b, kc, vc)
    bad = b.slot_mapping.copy()
    victim = int(W.physical_slots(b.block_tables[1], b.block_size, 40)[3])   # a slot of another history
    bad[0] = victim
    from tests.gpu_util import dev_i32
    out = _fused(fus, slot_mapping=dev_i32(bad))
    assert fus.err() & nv.NV_DERR_SLOT_MISMATCH
    k_after = host_bits(fus.k_cache).reshape(-1, b.num_kv_heads, 128)
    assert np.array_equal(k_after[victim], kc.reshape(-1, b.num_kv_heads, 128)[victim])
    # rows 1 and 2 were stored and attended normally; row 0 attended over the pool as it was
    orc = oracle.default()
    good = b.slot_mapping.copy()
    good[0] = -1
    kc1, vc1 = kc.copy(), vc.copy()
    orc.store_kvcache(b.k_new, b.v_new, good, kc1, vc1)
    compare(host_f32(out), oracle_decode(orc, b, kc1, vc1), "mismatch")


def test_fused_padding_row_with_a_slot_is_flagged():
    b = W.make_decode("padslot", 31, [20, 9], 16, 8, 128, 16, n_pad=1)
    fus = DeviceBatch(b)
    bad = b.slot_mapping.copy()
    bad[2] = 0                                 # padding row (L = 0) given a slot
    from tests.gpu_util import dev_i32
    out = host_f32(_fused(fus, slot_mapping=dev_i32(bad)))
    assert fus.err() & nv.NV_DERR_SLOT_MISMATCH
    assert not out[2].any()
