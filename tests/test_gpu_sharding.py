"""The path shards by kv head with no exchange (the tensor-parallel split of the pages' KV pools by
head): running decode and prefill on two halves of the kv heads -- each half with its own pool and its
query heads -- and concatenating the outputs along the head axis gives the full call's result."""
import numpy as np
import pytest

import workloads as W
from tests.gpu_util import DeviceBatch, compare, host_bits, host_f32

pytestmark = pytest.mark.gpu


def _halves(db, hkv, g):
    """(q, k_cache, v_cache) for kv heads [0, hkv/2) and [hkv/2, hkv), each contiguous."""
    h = hkv // 2
    out = []
    for lo in (0, h):
        q = db.q[:, lo * g:(lo + h) * g].contiguous()
        kc = db.k_cache[:, :, lo:lo + h].contiguous()
        vc = db.v_cache[:, :, lo:lo + h].contiguous()
        out.append((q, kc, vc))
    return out


def test_decode_head_halves_concatenate_to_the_full_call():
    import torch
    import paged_kv_attention_store_gb300 as nv
    b = W.make_decode("shard-dec", 61, list(np.random.default_rng(3).integers(1, 3000, 48)), 32, 8, 128, 256)
    db = DeviceBatch(b)
    db.store()
    full = db.decode()
    g = b.num_q_heads // b.num_kv_heads
    maxc = int(b.seq_lens.max())
    parts = [nv.nv_paged_decode_attn(q, kc, vc, db.block_tables, db.seq_lens, b.scale, max_context_len=maxc,
                                     d_err=db.d_err) for q, kc, vc in _halves(db, b.num_kv_heads, g)]
    torch.cuda.synchronize()
    assert db.err() == 0
    got = torch.cat(parts, dim=1)
    compare(host_f32(got), host_f32(full), "decode head halves")


def test_prefill_head_halves_concatenate_to_the_full_call():
    import torch
    import paged_kv_attention_store_gb300 as nv
    b = W.make_prefill("shard-pf", 62, [0, 256, 512, 37], [300, 129, 64, 700], 16, 8, 128, 64)
    db = DeviceBatch(b)
    db.store()
    mq = int(b.q_lens.max())
    full = db.prefill(mq)
    g = b.num_q_heads // b.num_kv_heads
    parts = [nv.nv_paged_prefill_attn(q, kc, vc, db.cu_q, db.cu_k, db.block_tables, b.scale, max_seqlen_q=mq,
                                      d_err=db.d_err) for q, kc, vc in _halves(db, b.num_kv_heads, g)]
    torch.cuda.synchronize()
    assert db.err() == 0
    got = torch.cat(parts, dim=1)
    # every (query tile, kv head) unit is computed the same way whatever other heads the call has
    assert np.array_equal(host_bits(got), host_bits(full))
