"""nv_paged_decode_attn on the GPU against the oracle (store first, then decode)."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gpu_util import (ORACLE_THREADS, DeviceBatch, compare, dev_i32, host_bits, host_f32,
                            oracle_cache_after_store, oracle_decode, oracle_store_in_place)

pytestmark = pytest.mark.gpu


def _run(batch, max_context_len=None, kc=None, vc=None):
    db = DeviceBatch(batch, kc, vc)
    db.store()
    out = db.decode(max_context_len)
    assert db.err() == 0
    kc1, vc1 = oracle_cache_after_store(oracle.default(), batch, db.kc_host0, db.vc_host0)
    return db, host_f32(out), kc1, vc1


def test_decode_tiny_parity_and_pins():
    b = W.tiny()
    db, got, kc, vc = _run(b)
    want = oracle_decode(oracle.default(), b, kc, vc)
    compare(got, want, "tiny")
    # single key (L = 1): the output is that V row, bit for bit after bf16 rounding
    g = b.num_q_heads // b.num_kv_heads
    out_bits = host_bits(db.decode())
    for h in range(b.num_q_heads):
        assert np.array_equal(out_bits[0, h], b.v_new[0, h // g])
    # equal scores: q = 0 -> mean of V rows
    import torch
    zero_q = torch.zeros_like(db.q)
    got0 = host_f32(db.decode(q=zero_q))
    want0 = oracle.decode_attn(np.zeros_like(b.q), kc, vc, b.block_tables, b.context_lens, b.num_kv_heads,
                               b.block_size, b.scale)
    compare(got0, want0, "tiny q=0")


CASES = [
    # name, ctx lens, Hq, Hkv, block_size, n_pad
    ("g1-bs16", [1, 7, 8, 9, 15, 16, 17, 100, 333], 8, 8, 16, 2),
    ("g2-bs256", [1, 255, 256, 257, 511, 600, 1500], 16, 8, 256, 3),
    ("g4-bs64", [3, 64, 65, 700, 2049, 4100], 32, 8, 64, 0),
    ("g8-bs32", [10, 31, 32, 33, 900], 16, 2, 32, 1),
    ("g4-hkv1", [5, 130, 1025], 4, 1, 128, 0),
    ("g2-hkv16", [2, 40, 513], 32, 16, 16, 0),
    ("g8-hkv8", [1, 9, 255, 256, 1100, 3000], 64, 8, 256, 1),   # two consumer warps per kv head
    ("g8-hkv16", [3, 500, 1300], 128, 16, 16, 0),
    ("g4-hkv12", [5, 300, 2100], 48, 12, 128, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_decode_shapes(case):
    name, ctx, hq, hkv, bs, pad = case
    b = W.make_decode(name, 21, ctx, hq, hkv, 128, bs, n_pad=pad, poison_tail=True)
    db, got, kc, vc = _run(b)
    want = oracle_decode(oracle.default(), b, kc, vc)
    compare(got, want, name)
    assert not got[b.seq_lens == 0].any()


def test_decode_max_context_hint_larger_than_needed():
    b = W.make_decode("hint", 22, [20, 300, 64], 16, 8, 128, 16)
    _, got, kc, vc = _run(b, max_context_len=b.block_tables.shape[1] * 16)
    compare(got, oracle_decode(oracle.default(), b, kc, vc), "hint")


def test_decode_qwen06_full():
    """256 sequences (L ~ U[100, 2048]) plus 32 graph-padding rows: every real row checked."""
    b = W.qwen06_decode()
    _, got, kc, vc = _run(b)
    want = oracle_decode(oracle.default(), b, kc, vc, threads=ORACLE_THREADS)
    compare(got[:256], want[:256], "qwen06")
    assert not got[256:].any()


def _full(batch, label):
    """Store + decode on the GPU, then every real row against the oracle (host threads over rows)."""
    db = DeviceBatch(batch)
    db.store()
    got = host_f32(db.decode())
    assert db.err() == 0
    kc, vc = oracle_store_in_place(oracle.default(), batch, db.kc_host0, db.vc_host0)
    want = oracle_decode(oracle.default(), batch, kc, vc, threads=ORACLE_THREADS)
    real = batch.seq_lens > 0
    assert not got[~real].any()
    return compare(got[real], want[real], label)


def test_decode_qwen8_full_size():
    """The headline batch (512 sequences, L ~ U[1024, 4096], 32/8 heads) at full size: every
    sequence and head compared element by element with the oracle."""
    _full(W.qwen8_decode(), "qwen8")


@pytest.mark.parametrize("bs", [256, 16])
def test_decode_shared_prefix_full(bs):
    """64 sequences at context 4096 sharing their first 3072 tokens' blocks: every sequence checked."""
    _full(W.shared_prefix(block_size=bs), f"shared-prefix-bs{bs}")


@pytest.mark.parametrize("num_seqs", [17, 64, 200])
def test_decode_group4_mid_batches_on_tiles(num_seqs):
    """Group 4 batches of 17 to a few hundred sequences decode on the tcgen05 tile kernel (their
    split-KV grid would end in a partly filled wave): every sequence against the oracle."""
    _full(W.qwen8_decode(num_seqs=num_seqs), f"group4 {num_seqs} seqs")


@pytest.mark.parametrize("lens,bs,pad", [([40000], 256, 0), ([20000, 13000, 7], 256, 0), ([33000, 2], 16, 1)],
                         ids=["one-40k", "three-mixed", "bs16-with-padding-row"])
def test_decode_group4_few_long_contexts_on_tiles(lens, bs, pad):
    """Group 4 with a few long contexts (num_seqs x max_context_len >= 32768 keys) decodes on the tile
    kernel with its keys split into ranges: every sequence against the oracle (a padding row gets zeros)."""
    _full(W.make_decode("g4-few-long", 31, lens, 32, 8, 128, bs, n_pad=pad), f"group4 few long {lens}")


@pytest.mark.parametrize("hq,hkv,lens", [(8, 8, [40000]), (16, 8, [33000, 5]), (16, 8, [9000] * 8),
                                         (16, 8, [5000] * 9)],
                         ids=["g1-one-40k", "g2-two", "g2-eight-tiles", "g2-nine-split-kv"])
def test_decode_groups_1_2_few_long_contexts(hq, hkv, lens):
    """Groups 1 and 2 with at most 8 sequences holding 32768 keys or more (num_seqs x max_context_len)
    decode on the tile kernel; nine sequences stay on the split-KV kernel: every sequence against the
    oracle."""
    _full(W.make_decode("g12-few-long", 37, lens, hq, hkv, 128, 256), f"group {hq // hkv} few long {len(lens)}")


def test_decode_group8_at_the_sequence_limit():
    """65535 sequences of 1-16 positions at group 8 (8 q / 1 kv head, block size 16): the most the tile
    kernel's work list addresses (one more is refused on the host).  Every sequence against the oracle."""
    rng = np.random.default_rng(41)
    b = W.make_decode("max-seqs", 41, rng.integers(1, 17, size=65535), 8, 1, 128, 16)
    shape = (b.num_blocks, b.block_size, b.num_kv_heads, b.head_dim)
    kc, vc = W.normal_bf16(rng, shape), W.normal_bf16(rng, shape)     # one draw each: quick to build
    db = DeviceBatch(b, kc, vc)
    db.store()
    got = host_f32(db.decode())
    assert db.err() == 0
    kc1, vc1 = oracle_store_in_place(oracle.default(), b, kc, vc)
    compare(got, oracle_decode(oracle.default(), b, kc1, vc1, threads=ORACLE_THREADS), "65535 sequences")


def test_decode_block_permutation_invariance():
    b = W.make_decode("perm", 23, [40, 700, 1200], 16, 8, 128, 64)
    db, got, kc, vc = _run(b)
    perm = np.random.default_rng(4).permutation(b.num_blocks)
    kc2, vc2 = np.empty_like(db.kc_host0), np.empty_like(db.vc_host0)
    kc2[perm], vc2[perm] = db.kc_host0, db.vc_host0
    bt2 = np.where(b.block_tables >= 0, perm[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    sm2 = np.array([perm[s // 64] * 64 + s % 64 for s in b.slot_mapping], np.int32)
    b2 = W.PagedBatch(**{**b.__dict__, "block_tables": bt2, "slot_mapping": sm2})
    db2 = DeviceBatch(b2, kc2, vc2)
    db2.store()
    got2 = host_f32(db2.decode())
    compare(got2, got, "permuted vs original")
    # the reduction order depends only on logical positions, so the result is identical
    assert np.array_equal(got2, got)


def test_decode_stale_table_entries_are_not_read():
    """Entries past the blocks a length needs hold garbage ids: nothing reads them."""
    b = W.make_decode("stale", 24, [5, 17, 33], 16, 8, 128, 16, width=8)
    bt = b.block_tables.copy()
    for i, L in enumerate(b.seq_lens):
        bt[i, W.blocks_needed(int(L), 16):] = 10 ** 6 + i
    b2 = W.PagedBatch(**{**b.__dict__, "block_tables": bt})
    db, got, kc, vc = _run(b2)
    compare(got, oracle_decode(oracle.default(), b2, kc, vc), "stale")


def test_decode_bad_block_id_is_flagged_not_faulted():
    import paged_kv_attention_store_gb300 as nv
    b = W.make_decode("badblk", 25, [40, 20], 16, 8, 128, 16)
    bt = b.block_tables.copy()
    bt[0, 1] = b.num_blocks + 7
    b2 = W.PagedBatch(**{**b.__dict__, "block_tables": bt})
    db = DeviceBatch(b2)
    db.decode()
    assert db.err() & nv.NV_DERR_BLOCK_RANGE


def test_decode_length_beyond_hint_is_flagged():
    import paged_kv_attention_store_gb300 as nv
    b = W.make_decode("len", 26, [40, 300], 16, 8, 128, 16)
    db = DeviceBatch(b)
    db.decode(max_context_len=100)
    assert db.err() & nv.NV_DERR_LENGTH


def test_decode_workspace_reused_across_batches_and_after_an_error():
    """One zero-filled workspace serves calls of different batch sizes and split counts, including one
    right after a call that flagged a bad block id: the per-sequence split counters the merge uses are
    left at zero by every call, so each call still matches the oracle."""
    import torch
    import paged_kv_attention_store_gb300 as nv
    from tests.gpu_util import oracle_cache_after_store, oracle_decode
    orc = oracle.default()
    rng = np.random.default_rng(27)
    big = W.make_decode("reuse-big", 27, rng.integers(1, 4097, 200).tolist(), 32, 8, 128, 64)
    small = W.make_decode("reuse-small", 28, [4096, 3000, 17, 2500], 32, 8, 128, 64)
    ws = torch.zeros(max(nv.nv_paged_decode_workspace_size(b.num_seqs, 32, 128, 4096) for b in (big, small)),
                     dtype=torch.uint8, device="cuda")
    bad_bt = small.block_tables.copy()
    bad_bt[1, 3] = small.num_blocks + 5
    bad = W.PagedBatch(**{**small.__dict__, "block_tables": bad_bt})
    for b, expect_err in ((big, False), (small, False), (bad, True), (small, False), (big, False)):
        db = DeviceBatch(b)
        db.store()
        got = nv.nv_paged_decode_attn(db.q, db.k_cache, db.v_cache, db.block_tables, db.seq_lens, b.scale,
                                      max_context_len=4096, workspace=ws, d_err=db.d_err)
        err = db.err()
        if expect_err:
            assert err & nv.NV_DERR_BLOCK_RANGE
            continue
        assert err == 0
        kc, vc = oracle_cache_after_store(orc, b, db.kc_host0, db.vc_host0)
        compare(host_f32(got), oracle_decode(orc, b, kc, vc), f"reused workspace {b.name}")


def test_decode_workspace_not_zero_filled_is_flagged():
    """Split counters that do not start at zero (a workspace that was not zero-filled) are reported.
    100 sequences of 1024 positions at group 2 (always the split-KV kernel) split 8 ways, so the last
    split of each merges in the kernel through the counters (above 16 splits a merge launch combines
    them, and no counter is used)."""
    import torch
    import paged_kv_attention_store_gb300 as nv
    b = W.make_decode("dirty-ws", 29, [1024] * 100, 4, 2, 128, 64)
    db = DeviceBatch(b)
    db.store()
    ws = torch.full((nv.nv_paged_decode_workspace_size(b.num_seqs, 4, 128, 1024),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    nv.nv_paged_decode_attn(db.q, db.k_cache, db.v_cache, db.block_tables, db.seq_lens, b.scale,
                            max_context_len=1024, workspace=ws, d_err=db.d_err)
    assert db.err() & nv.NV_DERR_VALUE


# ---- groups of 8 and 16 query heads per kv head: the tcgen05 tile kernel (one query row per sequence) ----

@pytest.mark.parametrize("hq,hkv,bs", [(128, 8, 256), (16, 1, 16), (64, 4, 64)], ids=["g16-hkv8", "g16-hkv1", "g16-hkv4"])
def test_decode_group16(hq, hkv, bs):
    b = W.make_decode(f"g16-{hq}-{hkv}", 30, [1, 2, 127, 128, 129, 2000, 4100], hq, hkv, 128, bs, n_pad=2,
                      poison_tail=True)
    db, got, kc, vc = _run(b)
    compare(got, oracle_decode(oracle.default(), b, kc, vc), b.name)
    assert not got[b.seq_lens == 0].any()


def test_decode_group8_length_beyond_hint_is_truncated_and_flagged():
    """As on the split-KV kernel: a context longer than the host hint attends to its first
    max_context_len keys and NV_DERR_LENGTH is set; the other rows are unaffected."""
    import paged_kv_attention_store_gb300 as nv
    b = W.make_decode("len8", 31, [40, 300, 90], 64, 8, 128, 16, n_pad=1)
    db = DeviceBatch(b)
    db.store()
    got = host_f32(db.decode(max_context_len=100))
    assert db.err() & nv.NV_DERR_LENGTH
    kc, vc = oracle_cache_after_store(oracle.default(), b, db.kc_host0, db.vc_host0)
    cut = W.PagedBatch(**{**b.__dict__, "seq_lens": np.minimum(b.seq_lens, 100).astype(np.int32)})
    compare(got, oracle_decode(oracle.default(), cut, kc, vc), "truncated")
    assert not got[3].any()


def test_decode_group8_bad_block_id_is_flagged_not_faulted():
    import paged_kv_attention_store_gb300 as nv
    b = W.make_decode("badblk8", 32, [400, 20], 64, 8, 128, 16)
    bt = b.block_tables.copy()
    bt[0, 3] = b.num_blocks + 7
    b2 = W.PagedBatch(**{**b.__dict__, "block_tables": bt})
    db = DeviceBatch(b2)
    got = host_f32(db.decode())
    assert db.err() & nv.NV_DERR_BLOCK_RANGE
    # the sequence without a bad entry is unaffected (the oracle runs on the valid tables: row 1's is
    # the same in both)
    want = oracle_decode(oracle.default(), b, db.kc_host0, db.vc_host0)
    compare(got[1:2], want[1:2], "unaffected row")


def test_decode_group8_one_long_sequence_splits_its_keys():
    """One sequence of 20000 keys at group 8 gives the tile kernel 8 (sequence, kv head) units; its keys
    are split into ranges of 1024 whose fp32 partials a merge launch combines."""
    b = W.make_decode("g8-one", 33, [20000], 64, 8, 128, 256)
    db, got, kc, vc = _run(b)
    compare(got, oracle_decode(oracle.default(), b, kc, vc), b.name)
