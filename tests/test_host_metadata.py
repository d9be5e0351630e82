"""Host-side metadata builders against the pages' worked examples (no GPU)."""
import numpy as np
import pytest

import oracle
import workloads as W
from paged_kv_attention_store_gb300 import metadata as M
from tests.oracle_pin_checks import golden


def test_prefill_examples():
    for ex in golden()["prefill"]:
        seqs = [(s["block_table"], s["num_cached_tokens"], s["num_scheduled_tokens"]) for s in ex["seqs"]]
        m = M.prepare_prefill(seqs, ex["block_size"])
        assert m.cu_seqlens_q.tolist() == ex["cu_seqlens_q"], ex["cite"]
        assert m.cu_seqlens_k.tolist() == ex["cu_seqlens_k"], ex["cite"]
        assert m.max_seqlen_q == ex["max_seqlen_q"] and m.max_seqlen_k == ex["max_seqlen_k"]
        assert m.has_prefix == ex["block_tables_passed"]
        if "slot_mapping" in ex:
            assert m.slot_mapping.tolist() == ex["slot_mapping"], ex["cite"]
            assert m.positions.tolist() == ex["positions"]
        else:
            # every new token gets a distinct slot inside its own blocks
            assert len(set(m.slot_mapping.tolist())) == m.cu_seqlens_q[-1]


def test_decode_examples():
    for ex in golden()["decode"]:
        seqs = [(s["block_table"], s["num_tokens"]) for s in ex["seqs"]]
        width = ex.get("block_table_width")
        m = M.prepare_decode(seqs, ex["block_size"], width)
        assert m.positions.tolist() == ex["positions"]
        assert m.context_lens.tolist() == ex["context_lens"]
        if "slot_mapping" in ex:
            assert m.slot_mapping.tolist() == ex["slot_mapping"]
        if width:
            assert m.block_tables.shape == (len(seqs), width)
            for i, s in enumerate(ex["seqs"]):
                n = len(s["block_table"])
                assert m.block_tables[i, :n].tolist() == s["block_table"]
                assert (m.block_tables[i, n:] == -1).all()
        if "bucket" in ex:
            assert M.graph_bucket(len(seqs)) == ex["bucket"]
            p = M.pad_decode_to_bucket(m, ex["bucket"])
            assert p.slot_mapping[len(seqs):].tolist() == [ex["bucket_slot_pad"]] * (ex["bucket"] - len(seqs))
            assert p.context_lens[len(seqs):].tolist() == [ex["bucket_context_pad"]] * (ex["bucket"] - len(seqs))


def test_graph_buckets():
    # 1, 2, 4, 8, then every multiple of 16 up to 512: 36 buckets
    assert len(M.GRAPH_BUCKETS) == 36
    assert M.graph_bucket(3) == 4 and M.graph_bucket(17) == 32 and M.graph_bucket(512) == 512
    with pytest.raises(ValueError):
        M.graph_bucket(97, max_bs=96)


@pytest.mark.parametrize("bs", [4, 16, 256])
def test_slots_for_range_matches_oracle(bs):
    rng = np.random.default_rng(bs)
    table = rng.permutation(40).astype(np.int32)
    for start, end in [(0, 1), (0, 9 * bs // 4 + 1), (bs - 1, bs + 1), (3, 3), (2 * bs, 5 * bs)]:
        got = M.slots_for_range(table, start, end, bs)
        want = [oracle.slot_of(table, p, bs) for p in range(start, end)]
        assert got == want


@pytest.mark.parametrize("make", [W.tiny, lambda: W.make_decode("d", 4, [3, 300, 17], 8, 2, 128, 16, n_pad=3),
                                  lambda: W.make_prefill("p", 5, [0, 32, 512], [20, 1, 300], 8, 4, 128, 16)])
def test_generator_slots_agree_with_oracle(make):
    """The generator's allocator bookkeeping and the oracle's slot definition agree on every token."""
    b = make()
    cu = b.cu_seqlens_q
    for s in range(b.num_seqs):
        L, nq = int(b.seq_lens[s]), int(b.q_lens[s])
        for j in range(nq):
            pos = L - nq + j
            assert b.slot_mapping[cu[s] + j] == oracle.slot_of(b.block_tables[s], pos, b.block_size)
    if b.kind == "decode":
        assert (b.slot_mapping[b.seq_lens == 0] == -1).all()
