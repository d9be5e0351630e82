"""The seeded generator: shapes and structure of the five workloads (no GPU)."""
import numpy as np

import workloads as W


def test_bf16_rounding_is_rne():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3, 1.0 + 2 ** -8 + 2 ** -20], np.float32)
    b = W.f32_to_bf16_bits(x)
    back = W.bf16_bits_to_f32(b)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa wins (1.0)
    assert back[1] == 1.0
    # 1 + 3*2^-8 ties between 1+2^-7 and 1+2^-6: even wins (1 + 2^-6)
    assert back[2] == np.float32(1 + 2 ** -6)
    assert back[3] == -2.5
    assert back[5] == np.float32(1 + 2 ** -7)
    assert np.all(np.abs(back - x) <= np.abs(x) * 2 ** -8)


def test_tiny_shape():
    b = W.tiny()
    assert b.seq_lens.tolist() == [1, 17, 256, 300]
    assert b.num_blocks == 8 and b.block_size == 256
    used = b.used_blocks()
    assert len(used) == 5 and len(set(used)) == 5
    assert b.q.shape == (4, 16, 128) and b.k_new.shape == (4, 8, 128)


def test_qwen06_decode_padding():
    b = W.qwen06_decode()
    assert b.num_seqs == 288 and (b.seq_lens[256:] == 0).all() and (b.slot_mapping[256:] == -1).all()
    assert (b.seq_lens[:256] >= 100).all() and (b.seq_lens[:256] <= 2048).all()
    assert (b.block_tables[256:] == -1).all()


def test_qwen8_pool_is_a_permutation():
    b = W.qwen8_decode()
    assert b.num_seqs == 512 and b.num_q_heads == 32
    ids = np.concatenate([b.block_tables[s, :W.blocks_needed(int(b.seq_lens[s]), 256)] for s in range(512)])
    assert sorted(ids.tolist()) == list(range(b.num_blocks))


def test_prefill_chunk_budget():
    b = W.prefill_chunk()
    assert int(b.q_lens.sum()) == 16384 and (b.q_lens >= 1).all() and b.num_seqs == 16
    P = b.meta["prefix_lens"]
    assert ((P % 256) == 0).all() and P.max() <= 2048
    assert b.block_tables.shape[1] <= (2048 + 16384 + 255) // 256


def test_shared_prefix_tables():
    for bs in (256, 16):
        b = W.shared_prefix(block_size=bs)
        s = 3072 // bs
        assert (b.block_tables[:, :s] == b.block_tables[0, :s]).all()
        tails = b.block_tables[:, s:].reshape(-1)
        assert len(set(tails.tolist())) == tails.size
        assert b.num_blocks == s + 64 * (4096 // bs - s)


def test_cache_blocks_are_deterministic_and_subsettable():
    b = W.make_decode("d", 3, [40, 70, 5], 4, 2, 16, 16)
    kc, vc = b.cache()
    sub, ids = b.subset([1])
    kc_s, vc_s = sub.cache(ids)
    assert np.array_equal(kc_s, kc[ids]) and np.array_equal(vc_s, vc[ids])
