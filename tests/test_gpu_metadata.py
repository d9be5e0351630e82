"""nv_prepare_decode / nv_prepare_prefill on the GPU: bit-exact against the oracle (integers),
on the pages' worked examples and on random batches."""
import json
import os

import numpy as np
import pytest

import oracle
import paged_kv_attention_store_gb300 as nv
import workloads as W
from tests.gpu_util import dev_i32

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "slot_examples.json")


def _host(t):
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


def _err():
    import torch
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _table(tables, width=None):
    w = width or max(len(t) for t in tables)
    bt = np.full((len(tables), w), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    return bt


def test_prepare_decode_golden():
    g = json.load(open(GOLDEN))
    for ex in g["decode"]:
        bt = _table([s["block_table"] for s in ex["seqs"]], ex.get("block_table_width"))
        lens = np.array([s["num_tokens"] for s in ex["seqs"]], np.int32)
        pad = ex.get("bucket", len(lens))
        err = _err()
        cl, pos, sm = nv.nv_prepare_decode(dev_i32(lens), dev_i32(bt), ex["block_size"], int(bt.max()) + 1, pad,
                                           d_err=err)
        ocl, opos, osm, bad = oracle.default().prepare_decode(lens, bt, ex["block_size"], pad)
        assert np.array_equal(_host(cl), ocl) and np.array_equal(_host(pos), opos) and np.array_equal(_host(sm), osm)
        assert _host(cl)[:len(lens)].tolist() == ex["context_lens"]
        if "slot_mapping" in ex:
            assert _host(sm)[:len(lens)].tolist() == ex["slot_mapping"]
        assert int(_host(err)[0]) == 0


def test_prepare_prefill_golden():
    g = json.load(open(GOLDEN))
    for ex in g["prefill"]:
        bt = _table([s["block_table"] for s in ex["seqs"]])
        nc = np.array([s["num_cached_tokens"] for s in ex["seqs"]], np.int32)
        ns = np.array([s["num_scheduled_tokens"] for s in ex["seqs"]], np.int32)
        err = _err()
        cq, ck, pos, sm, mx = nv.nv_prepare_prefill(dev_i32(nc), dev_i32(ns), dev_i32(bt), ex["block_size"],
                                                    int(bt.max()) + 1, int(ns.sum()), d_err=err)
        assert _host(cq).tolist() == ex["cu_seqlens_q"] and _host(ck).tolist() == ex["cu_seqlens_k"]
        assert tuple(_host(mx).tolist()) == (ex["max_seqlen_q"], ex["max_seqlen_k"])
        if "positions" in ex:
            assert _host(pos).tolist() == ex["positions"]
        if "slot_mapping" in ex:
            assert _host(sm).tolist() == ex["slot_mapping"]
        assert int(_host(err)[0]) == 0


@pytest.mark.parametrize("bs", [1, 16, 256])
def test_prepare_random_batches_match_oracle(bs):
    rng = np.random.default_rng(bs)
    B = 1500                                   # more than one 1024-thread scan chunk
    lens = rng.integers(1, 4000, B).astype(np.int32)
    nb = (lens + bs - 1) // bs
    bt = np.full((B, int(nb.max()) + 2), -1, np.int32)
    perm = rng.permutation(int(nb.sum())).astype(np.int32)
    k = 0
    for i, n in enumerate(nb):
        bt[i, :n] = perm[k:k + n]
        k += n
    num_blocks = int(nb.sum())
    orc = oracle.default()
    err = _err()
    cl, pos, sm = nv.nv_prepare_decode(dev_i32(lens), dev_i32(bt), bs, num_blocks, B + 37, d_err=err)
    ocl, opos, osm, _ = orc.prepare_decode(lens, bt, bs, B + 37)
    assert np.array_equal(_host(cl), ocl) and np.array_equal(_host(pos), opos) and np.array_equal(_host(sm), osm)
    cached = (rng.random(B) * lens).astype(np.int32)
    cached[::7] = 0
    sched = (lens - cached).astype(np.int32)
    sched[::11] = 0                            # sequences with nothing scheduled
    total = int(sched.sum())
    cq, ck, pos, sm, mx = nv.nv_prepare_prefill(dev_i32(cached), dev_i32(sched), dev_i32(bt), bs, num_blocks, total,
                                                d_err=err)
    ocq, ock, opos, osm, omx = orc.prepare_prefill(cached, sched, bt, bs)
    assert np.array_equal(_host(cq), ocq) and np.array_equal(_host(ck), ock)
    assert np.array_equal(_host(pos), opos) and np.array_equal(_host(sm), osm)
    assert tuple(_host(mx).tolist()) == omx
    assert int(_host(err)[0]) == 0


def test_prepare_decode_matches_the_generated_batches():
    for b in (W.qwen06_decode(), W.make_decode("m", 5, [1, 16, 17, 300], 16, 8, 128, 16, n_pad=3)):
        n_real = int((b.seq_lens > 0).sum())
        cl, pos, sm = nv.nv_prepare_decode(dev_i32(b.seq_lens[:n_real]), dev_i32(b.block_tables[:n_real]),
                                           b.block_size, b.num_blocks, b.num_seqs)
        assert np.array_equal(_host(sm), b.slot_mapping) and np.array_equal(_host(cl), b.seq_lens)


def test_prepare_errors_are_flagged():
    bt = _table([[0, 1], [2]])
    err = _err()
    cl, pos, sm = nv.nv_prepare_decode(dev_i32(np.array([0, 300], np.int32)), dev_i32(bt), 256, 3, d_err=err)
    assert int(_host(err)[0]) & nv.NV_DERR_LENGTH          # row 0 has length 0; row 1's second block is -1
    assert _host(sm).tolist() == [-1, -1] and _host(cl).tolist() == [0, 0]
    err = _err()
    nv.nv_prepare_decode(dev_i32(np.array([5, 5], np.int32)), dev_i32(_table([[0], [9]])), 256, 3, d_err=err)
    assert int(_host(err)[0]) & nv.NV_DERR_BLOCK_RANGE
    err = _err()
    nv.nv_prepare_prefill(dev_i32(np.array([0, 4], np.int32)), dev_i32(np.array([3, 2], np.int32)), dev_i32(bt), 256,
                          3, 4, d_err=err)                  # lengths add up to 5, not 4
    assert int(_host(err)[0]) & nv.NV_DERR_LENGTH
