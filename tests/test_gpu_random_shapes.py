"""Seeded random shapes for decode and prefill against the oracle: group sizes 1-16 (kv heads 1-16), every supported
block size, lengths drawn around block and tile edges (1, bs-1, bs, bs+1, 127, 128, 129, ...), padding
rows, and pools whose unused tails hold NaN patterns.  Small enough that the oracle runs every row."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gpu_util import (ORACLE_THREADS, DeviceBatch, compare, host_f32, oracle_cache_after_store, oracle_decode,
                            oracle_prefill)

pytestmark = pytest.mark.gpu

GROUPS = [(8, 8), (16, 8), (32, 8), (16, 2), (8, 1), (32, 16), (64, 8), (48, 12), (256, 16), (128, 16)]
BLOCKS = [16, 32, 64, 128, 256]


def _edge_lengths(rng, bs, n, lo=1, hi=1500):
    """n lengths mixing random draws with block- and tile-edge values."""
    edges = [1, bs - 1, bs, bs + 1, 127, 128, 129, 255, 256, 257, 2 * bs + 3]
    out = []
    for _ in range(n):
        if rng.random() < 0.5:
            out.append(int(rng.choice([e for e in edges if lo <= e <= hi])))
        else:
            out.append(int(rng.integers(lo, hi + 1)))
    return out


@pytest.mark.parametrize("seed", range(10))
def test_decode_random_shapes(seed):
    rng = np.random.default_rng([seed, 401])
    hq, hkv = GROUPS[seed % len(GROUPS)]
    bs = BLOCKS[seed % len(BLOCKS)]
    ctx = _edge_lengths(rng, bs, int(rng.integers(1, 24)))
    b = W.make_decode(f"rand-dec-{seed}", 500 + seed, ctx, hq, hkv, 128, bs, n_pad=int(rng.integers(0, 3)),
                      poison_tail=True)
    db = DeviceBatch(b)
    db.store()
    got = host_f32(db.decode())
    assert db.err() == 0
    kc, vc = oracle_cache_after_store(oracle.default(), b, db.kc_host0, db.vc_host0)
    compare(got, oracle_decode(oracle.default(), b, kc, vc), b.name)
    assert not got[b.seq_lens == 0].any()


@pytest.mark.parametrize("seed", range(10))
def test_prefill_random_shapes(seed):
    rng = np.random.default_rng([seed, 402])
    hq, hkv = GROUPS[(seed + 3) % len(GROUPS)]
    bs = BLOCKS[(seed + 1) % len(BLOCKS)]
    n = int(rng.integers(1, 7))
    chunks = _edge_lengths(rng, bs, n, hi=400)
    prefixes = [0 if rng.random() < 0.3 else int(rng.choice([bs, 2 * bs, int(rng.integers(1, 600))]))
                for _ in range(n)]
    b = W.make_prefill(f"rand-pf-{seed}", 600 + seed, prefixes, chunks, hq, hkv, 128, bs, poison_tail=True)
    db = DeviceBatch(b)
    db.store()
    got = host_f32(db.prefill())
    assert db.err() == 0
    kc, vc = oracle_cache_after_store(oracle.default(), b, db.kc_host0, db.vc_host0)
    compare(got, oracle_prefill(oracle.default(), b, kc, vc, threads=ORACLE_THREADS), b.name)
