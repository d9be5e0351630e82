"""The Python binding's argument checks run on the host before anything is enqueued: tensors of the
wrong shape or layout raise ValueError, whatever device they live on (CPU tensors here, no GPU)."""
import pytest

torch = pytest.importorskip("torch")

import paged_kv_attention_store_gb300 as nv  # noqa: E402


def bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


POOL = (4, 16, 8, 128)      # [num_blocks, block_size, Hkv, D]


def test_pool_shape_checks():
    kc = bf(*POOL)
    with pytest.raises(ValueError, match="caches must be"):
        nv.nv_store_kvcache(bf(3, 8, 128), bf(3, 8, 128), i32(3), kc, bf(4, 16, 4, 128))
    with pytest.raises(ValueError, match="caches must be"):
        nv.nv_store_kvcache(bf(3, 8, 128), bf(3, 8, 128), i32(3), bf(4, 16, 1024), bf(4, 16, 1024))
    with pytest.raises(ValueError, match="contiguous"):
        big = bf(4, 16, 8, 256)
        nv.nv_store_kvcache(bf(3, 8, 128), bf(3, 8, 128), i32(3), big[..., :128], big[..., 128:])


def test_store_row_checks():
    kc, vc = bf(*POOL), bf(*POOL)
    with pytest.raises(ValueError, match=r"k must be \[N, Hkv, D\]"):
        nv.nv_store_kvcache(bf(3, 8, 64), bf(3, 8, 128), i32(3), kc, vc)
    with pytest.raises(ValueError, match=r"v must be \[N, Hkv, D\]"):
        nv.nv_store_kvcache(bf(3, 8, 128), bf(2, 8, 128), i32(3), kc, vc)
    with pytest.raises(ValueError, match="heads must be contiguous"):
        wide = bf(3, 8, 256)
        nv.nv_store_kvcache(bf(3, 8, 128), wide[..., :128], i32(3), kc, vc)


def test_decode_checks():
    kc, vc = bf(*POOL), bf(*POOL)
    with pytest.raises(ValueError, match="q must be contiguous"):
        nv.nv_paged_decode_attn(bf(2, 32, 64), kc, vc, i32(2, 4), i32(2), 0.088)
    with pytest.raises(ValueError, match="block_tables must be"):
        nv.nv_paged_decode_attn(bf(2, 32, 128), kc, vc, i32(3, 4), i32(2), 0.088)
    with pytest.raises(ValueError, match="block_tables must be"):
        nv.nv_paged_decode_attn(bf(2, 32, 128), kc, vc, i32(4, 2).t(), i32(2), 0.088)


def test_fused_decode_checks():
    kc, vc = bf(*POOL), bf(*POOL)
    q, k, v = bf(2, 32, 128), bf(2, 8, 128), bf(2, 8, 128)
    with pytest.raises(ValueError, match="slot_mapping must have one entry per sequence"):
        nv.nv_store_decode_attn(q, k, v, i32(3), kc, vc, i32(2, 4), i32(2), 0.088)
    with pytest.raises(ValueError, match=r"k must be \[B, Hkv, D\]"):
        nv.nv_store_decode_attn(q, bf(2, 4, 128), v, i32(2), kc, vc, i32(2, 4), i32(2), 0.088)


def test_prefill_checks():
    kc, vc = bf(*POOL), bf(*POOL)
    with pytest.raises(ValueError, match="q must be contiguous"):
        nv.nv_paged_prefill_attn(bf(10, 16, 128)[:, ::2], kc, vc, i32(3), i32(3), i32(2, 4), 0.088)
    with pytest.raises(ValueError, match="B\\+1 entries"):
        nv.nv_paged_prefill_attn(bf(10, 16, 128), kc, vc, i32(3), i32(4), i32(2, 4), 0.088)
    with pytest.raises(ValueError, match="block_tables must be"):
        nv.nv_paged_prefill_attn(bf(10, 16, 128), kc, vc, i32(3), i32(3), i32(3, 4), 0.088)


def test_prologue_checks():
    kc, vc = bf(*POOL), bf(*POOL)
    row = (16 + 2 * 8) * 128
    w = bf(128)
    with pytest.raises(ValueError, match="too short"):
        nv.nv_qk_norm_rope_store(bf(5, row - 8), i32(5), w, w, i32(5), kc, vc, 16)
    with pytest.raises(ValueError, match="one position and slot per token"):
        nv.nv_qk_norm_rope_store(bf(5, row), i32(4), w, w, i32(5), kc, vc, 16)
    with pytest.raises(ValueError, match="norm weights"):
        nv.nv_qk_norm_rope_store(bf(5, row), i32(5), bf(64), w, i32(5), kc, vc, 16)


def test_sampler_checks():
    with pytest.raises(ValueError, match="unit column stride"):
        nv.nv_sample_exponential_race(bf(4, 100).t(), torch.ones(100), torch.ones(100, 4))
    with pytest.raises(ValueError, match="one temperature and V draws per row"):
        nv.nv_sample_exponential_race(bf(4, 100), torch.ones(3), torch.ones(4, 100))


def test_output_checks_before_anything_is_enqueued():
    """A caller's ``out`` of the wrong shape, type or layout is refused: the kernels would write the
    full [B, Hq, D] extent through its pointer."""
    kc, vc = bf(*POOL), bf(*POOL)
    q = bf(2, 32, 128)
    for entry in (nv.nv_paged_decode_attn, nv.nv_paged_decode_attn_noalloc):
        with pytest.raises(ValueError, match=r"out must be \(2, 32, 128\)"):
            entry(q, kc, vc, i32(2, 4), i32(2), 0.088, out=bf(1, 32, 128))
        with pytest.raises(ValueError, match="out must be bfloat16"):
            entry(q, kc, vc, i32(2, 4), i32(2), 0.088, out=torch.zeros(2, 32, 128))
        with pytest.raises(ValueError, match="out must be contiguous"):
            entry(q, kc, vc, i32(2, 4), i32(2), 0.088, out=bf(2, 128, 32).transpose(1, 2))
    with pytest.raises(ValueError, match=r"out must be \(10, 16, 128\)"):
        nv.nv_paged_prefill_attn(bf(10, 16, 128), kc, vc, i32(3), i32(3), i32(2, 4), 0.088, out=bf(9, 16, 128))
    with pytest.raises(ValueError, match=r"q_out must be"):
        nv.nv_qk_norm_rope_store(bf(5, (16 + 16) * 128), i32(5), bf(128), bf(128), i32(5), kc, vc, 16,
                                 q_out=bf(5, 8, 128))


def test_index_and_value_types():
    kc, vc = bf(*POOL), bf(*POOL)
    q = bf(2, 32, 128)
    with pytest.raises(ValueError, match="block_tables must be int32"):
        nv.nv_paged_decode_attn(q, kc, vc, torch.zeros(2, 4, dtype=torch.int64), i32(2), 0.088)
    with pytest.raises(ValueError, match="context_lens must be int32"):
        nv.nv_paged_decode_attn(q, kc, vc, i32(2, 4), torch.zeros(2, dtype=torch.int64), 0.088)
    with pytest.raises(ValueError, match="context_lens must have 2 entries"):
        nv.nv_paged_decode_attn(q, kc, vc, i32(2, 4), i32(3), 0.088)
    with pytest.raises(ValueError, match="q must be bfloat16"):
        nv.nv_paged_decode_attn(torch.zeros(2, 32, 128, dtype=torch.float16), kc, vc, i32(2, 4), i32(2), 0.088)
    with pytest.raises(ValueError, match="k_cache must be bfloat16"):
        nv.nv_store_kvcache(bf(3, 8, 128), bf(3, 8, 128), i32(3), torch.zeros(POOL), torch.zeros(POOL))
    with pytest.raises(ValueError, match="slot_mapping must be int32"):
        nv.nv_store_kvcache(bf(3, 8, 128), bf(3, 8, 128), torch.zeros(3, dtype=torch.int64), kc, vc)
    with pytest.raises(ValueError, match="cu_seqlens_k must be int32"):
        nv.nv_paged_prefill_attn(bf(10, 16, 128), kc, vc, i32(3), torch.zeros(3, dtype=torch.int64), i32(2, 4),
                                 0.088)
    with pytest.raises(ValueError, match="d_err must be int32"):
        nv.nv_store_kvcache(bf(3, 8, 128), bf(3, 8, 128), i32(3), kc, vc, d_err=torch.zeros(1))


def test_host_tensors_are_refused():
    """Well-formed tensors that live in host memory never reach the library: its kernels would
    dereference host addresses."""
    kc, vc = bf(*POOL), bf(*POOL)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        nv.nv_store_kvcache(bf(3, 8, 128), bf(3, 8, 128), i32(3), kc, vc)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        nv.nv_paged_decode_attn(bf(2, 32, 128), kc, vc, i32(2, 4), i32(2), 0.088, out=bf(2, 32, 128))
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        nv.nv_paged_decode_attn_noalloc(bf(2, 32, 128), kc, vc, i32(2, 4), i32(2), 0.088)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        nv.nv_paged_prefill_attn(bf(10, 16, 128), kc, vc, i32(3), i32(3), i32(2, 4), 0.088)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        nv.nv_sample_exponential_race(bf(4, 100), torch.ones(4), torch.ones(4, 100))
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        nv.nv_prepare_decode(i32(4), i32(4, 3), 16, 100)
