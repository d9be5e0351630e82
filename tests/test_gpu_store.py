"""nv_store_kvcache on the GPU against the oracle: bit-exact over the whole pool."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gpu_util import DeviceBatch, dev_bf16, dev_i32, host_bits, oracle_cache_after_store

pytestmark = pytest.mark.gpu


def _check_whole_pool(batch, kc=None, vc=None):
    db = DeviceBatch(batch, kc, vc)
    db.store()
    assert db.err() == 0
    want_k, want_v = oracle_cache_after_store(oracle.default(), batch, db.kc_host0, db.vc_host0)
    assert np.array_equal(host_bits(db.k_cache), want_k)
    assert np.array_equal(host_bits(db.v_cache), want_v)


def test_store_tiny():
    _check_whole_pool(W.tiny())


def test_store_qwen06_with_graph_padding():
    b = W.qwen06_decode()
    assert (b.slot_mapping == -1).sum() == 32
    _check_whole_pool(b)


@pytest.mark.parametrize("n", [1, 2, 3, 17, 255])
def test_store_ragged_small(n):
    b = W.make_decode("ragged", 10 + n, list(range(1, n + 1)), 4, 2, 128, 16, n_pad=n % 3)
    _check_whole_pool(b)


def test_store_prefill_sized():
    """16384 new rows (the chunked-prefill budget): every stored row and the untouched rest."""
    _check_whole_pool(W.prefill_chunk())


def test_store_strided_value_view():
    """V is a view into a fused QKV output with 4096-wide rows (Qwen3-0.6B layout)."""
    torch = pytest.importorskip("torch")
    import paged_kv_attention_store_gb300 as nv
    b = W.qwen06_decode()
    n, hkv, d = b.v_new.shape
    fused = np.zeros((n, 4096), np.uint16)
    fused[:, 2048 + 1024:2048 + 2048] = b.v_new.reshape(n, -1)
    fused[:, 2048:2048 + 1024] = b.k_new.reshape(n, -1)
    fused_d = dev_bf16(fused)
    k_view = fused_d[:, 2048:3072].view(n, hkv, d)
    v_view = fused_d[:, 3072:4096].view(n, hkv, d)
    assert v_view.stride(0) == 4096
    db = DeviceBatch(b)
    nv.nv_store_kvcache(k_view, v_view, db.slot_mapping, db.k_cache, db.v_cache, d_err=db.d_err)
    assert db.err() == 0
    want_k, want_v = oracle_cache_after_store(oracle.default(), b, db.kc_host0, db.vc_host0)
    assert np.array_equal(host_bits(db.k_cache), want_k) and np.array_equal(host_bits(db.v_cache), want_v)


def test_store_out_of_range_slots_are_skipped_and_flagged():
    import paged_kv_attention_store_gb300 as nv
    b = W.make_decode("bad-slots", 3, [5, 9, 30, 2], 4, 2, 128, 16, n_pad=1)
    num_slots = b.num_blocks * b.block_size
    sm = b.slot_mapping.copy()
    sm[1] = num_slots
    sm[2] = -5
    db = DeviceBatch(b)
    nv.nv_store_kvcache(db.k_new, db.v_new, dev_i32(sm), db.k_cache, db.v_cache, d_err=db.d_err)
    assert db.err() & nv.NV_DERR_SLOT_RANGE
    kc, vc = db.kc_host0.copy(), db.vc_host0.copy()
    assert oracle.store_kvcache(b.k_new, b.v_new, sm, kc, vc) == 2
    assert np.array_equal(host_bits(db.k_cache), kc) and np.array_equal(host_bits(db.v_cache), vc)


def test_store_zero_tokens_is_a_no_op():
    torch = pytest.importorskip("torch")
    import paged_kv_attention_store_gb300 as nv
    b = W.tiny()
    db = DeviceBatch(b)
    empty = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    nv.nv_store_kvcache(empty, empty, torch.empty(0, dtype=torch.int32, device="cuda"), db.k_cache, db.v_cache)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(db.k_cache), db.kc_host0)
