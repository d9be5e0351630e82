"""Every entry point runs inside a CUDA graph (the field guide's model runner replays decode through
captured graphs, padding the batch with rows of context 0 and slot -1, Step 07.8): each test captures
the calls once on static buffers, then copies two different batches into those buffers and replays,
and each replay must match the oracle.  This pins that the calls make no host synchronisation and no
allocation, read their lengths from device memory, and leave their workspaces ready for the next
replay (the split and row counters back at zero)."""
import numpy as np
import pytest

import oracle
import paged_kv_attention_store_gb300 as nv
import workloads as W
from tests.gpu_util import (compare, dev_bf16, host_bits, host_f32, oracle_cache_after_store, oracle_decode,
                            oracle_prefill)

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Run ``fn`` once (first-call set-up happens outside the capture), then capture it."""
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def _bf16_into(dst, a):
    import torch
    dst.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16))


def _i32_into(dst, a):
    import torch
    dst.copy_(torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)))


class _Static:
    """Static device buffers shaped for the largest of ``batches`` (pool, rows, tables)."""

    def __init__(self, batches, rows):
        import torch
        b0 = batches[0]
        self.nb = max(b.num_blocks for b in batches)
        self.width = max(b.block_tables.shape[1] for b in batches)
        hq, hkv, d, bs = b0.num_q_heads, b0.num_kv_heads, b0.head_dim, b0.block_size
        bf = dict(dtype=torch.bfloat16, device="cuda")
        i32 = dict(dtype=torch.int32, device="cuda")
        self.k_cache = torch.zeros((self.nb, bs, hkv, d), **bf)
        self.v_cache = torch.zeros((self.nb, bs, hkv, d), **bf)
        self.q = torch.zeros((rows, hq, d), **bf)
        self.k_new = torch.zeros((rows, hkv, d), **bf)
        self.v_new = torch.zeros((rows, hkv, d), **bf)
        self.out = torch.zeros((rows, hq, d), **bf)
        self.slots = torch.full((rows,), -1, **i32)
        seqs = max(b.num_seqs for b in batches)
        self.bt = torch.full((seqs, self.width), -1, **i32)
        self.lens = torch.zeros((seqs,), **i32)
        self.cu_q = torch.zeros((seqs + 1,), **i32)
        self.cu_k = torch.zeros((seqs + 1,), **i32)
        self.d_err = torch.zeros(1, **i32)

    def load(self, b):
        """Copy batch ``b`` in; returns its initial pool (host) for the oracle."""
        kc, vc = b.cache()
        self.k_cache.zero_()
        self.v_cache.zero_()
        _bf16_into(self.k_cache[:b.num_blocks], kc)
        _bf16_into(self.v_cache[:b.num_blocks], vc)
        n = b.q.shape[0]
        _bf16_into(self.q[:n], b.q)
        _bf16_into(self.k_new[:n], b.k_new)
        _bf16_into(self.v_new[:n], b.v_new)
        _i32_into(self.slots[:n], b.slot_mapping)
        bt = np.full((b.num_seqs, self.width), -1, np.int32)
        bt[:, :b.block_tables.shape[1]] = b.block_tables
        _i32_into(self.bt[:b.num_seqs], bt)
        _i32_into(self.lens[:b.num_seqs], b.seq_lens)
        _i32_into(self.cu_q, b.cu_seqlens_q)
        _i32_into(self.cu_k, b.cu_seqlens_k)
        self.d_err.zero_()
        return kc, vc

    def pool_bits(self, b):
        return host_bits(self.k_cache[:b.num_blocks]), host_bits(self.v_cache[:b.num_blocks])


@pytest.mark.parametrize("hq", [32, 64], ids=["group4", "group8-tiles"])
@pytest.mark.parametrize("fused", [False, True], ids=["store+decode", "fused"])
def test_decode_step_replayed_from_a_graph(fused, hq):
    """A 16-row decode bucket: one batch fills it, the other has 12 real rows and 4 padding rows.  At
    group 8 the step runs the tile kernel with the keys split and a merge launch."""
    import torch
    orc = oracle.default()
    rng = np.random.default_rng(71)
    full = W.make_decode("graph-full", 71, rng.integers(1, 3000, 16).tolist(), hq, 8, 128, 64, width=48)
    padded = W.make_decode("graph-pad", 72, rng.integers(1, 3000, 12).tolist(), hq, 8, 128, 64, n_pad=4, width=48)
    st = _Static([full, padded], rows=16)
    max_ctx = st.width * full.block_size
    ws = torch.zeros(nv.nv_paged_decode_workspace_size(16, hq, 128, max_ctx), dtype=torch.uint8, device="cuda")

    def step():
        if fused:
            nv.nv_store_decode_attn(st.q, st.k_new, st.v_new, st.slots, st.k_cache, st.v_cache, st.bt, st.lens,
                                    full.scale, out=st.out, max_context_len=max_ctx, workspace=ws, d_err=st.d_err)
        else:
            nv.nv_store_kvcache(st.k_new, st.v_new, st.slots, st.k_cache, st.v_cache, d_err=st.d_err)
            nv.nv_paged_decode_attn(st.q, st.k_cache, st.v_cache, st.bt, st.lens, full.scale, out=st.out,
                                    max_context_len=max_ctx, workspace=ws, d_err=st.d_err)

    st.load(full)
    g = _capture(step)
    for b in (full, padded, full):
        kc, vc = st.load(b)
        g.replay()
        torch.cuda.synchronize()
        assert int(st.d_err.item()) == 0, b.name
        okc, ovc = oracle_cache_after_store(orc, b, kc, vc)
        gk, gv = st.pool_bits(b)
        assert np.array_equal(gk, okc) and np.array_equal(gv, ovc), b.name
        got = host_f32(st.out)
        compare(got, oracle_decode(orc, b, okc, ovc), f"graph {b.name}")
        assert not got[b.seq_lens == 0].any()


def test_prefill_step_replayed_from_a_graph():
    """Two chunked-prefill batches with the same token budget (total_q), split differently over their
    sequences and with different cached prefixes, replayed through one captured store + prefill."""
    import torch
    orc = oracle.default()
    a = W.make_prefill("graph-pf-a", 73, [0, 256, 100], [300, 129, 83], 16, 8, 128, 64, width=16)
    b = W.make_prefill("graph-pf-b", 74, [500, 0, 64], [1, 383, 128], 16, 8, 128, 64, width=16)
    total = int(a.q_lens.sum())
    assert total == int(b.q_lens.sum())
    st = _Static([a, b], rows=total)
    ws = torch.empty(nv.nv_paged_prefill_workspace_size(3, total, total, 16, 8), dtype=torch.uint8, device="cuda")

    def step():
        nv.nv_store_kvcache(st.k_new, st.v_new, st.slots, st.k_cache, st.v_cache, d_err=st.d_err)
        nv.nv_paged_prefill_attn(st.q, st.k_cache, st.v_cache, st.cu_q, st.cu_k, st.bt, a.scale, max_seqlen_q=total,
                                 out=st.out, workspace=ws, d_err=st.d_err)

    st.load(a)
    g = _capture(step)
    for batch in (a, b, a):
        kc, vc = st.load(batch)
        g.replay()
        torch.cuda.synchronize()
        assert int(st.d_err.item()) == 0, batch.name
        okc, ovc = oracle_cache_after_store(orc, batch, kc, vc)
        gk, gv = st.pool_bits(batch)
        assert np.array_equal(gk, okc) and np.array_equal(gv, ovc), batch.name
        compare(host_f32(st.out), oracle_prefill(orc, batch, okc, ovc), f"graph {batch.name}")


def test_prologue_and_sampler_replayed_from_a_graph():
    """QK-norm + RoPE + store, and the sampler, captured once and replayed on two sets of inputs."""
    import torch
    orc = oracle.default()
    b = W.make_prefill("graph-pro", 75, [0, 64], [100, 28], 16, 8, 128, 64)
    n = int(b.q_lens.sum())
    st = _Static([b], rows=n)
    width = (16 + 2 * 8) * 128
    qkv = torch.zeros((n, width), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros((n,), dtype=torch.int32, device="cuda")
    pi0 = W.prologue_inputs(b, 0)
    qw, kw = dev_bf16(pi0.q_weight), dev_bf16(pi0.k_weight)
    q_out = torch.zeros((n, 16, 128), dtype=torch.bfloat16, device="cuda")
    R, V = 24, 5000
    logits = torch.zeros((R, V), dtype=torch.bfloat16, device="cuda")
    temps = torch.ones((R,), dtype=torch.float32, device="cuda")
    draws = torch.ones((R, V), dtype=torch.float32, device="cuda")
    tokens = torch.zeros((R,), dtype=torch.int64, device="cuda")
    sws = torch.zeros(nv.load_library().nv_sample_workspace_size(R, V), dtype=torch.uint8, device="cuda")

    def step():
        nv.nv_qk_norm_rope_store(qkv, pos, qw, kw, st.slots, st.k_cache, st.v_cache, 16, rms_eps=pi0.eps,
                                 rope_theta=pi0.theta, q_out=q_out, d_err=st.d_err)
        nv.nv_sample_exponential_race(logits, temps, draws, tokens=tokens, workspace=sws, d_err=st.d_err)

    st.load(b)
    g = _capture(step)
    for seed in (1, 2):
        kc, vc = st.load(b)
        pi = W.prologue_inputs(b, seed)
        _bf16_into(qw, pi.q_weight)
        _bf16_into(kw, pi.k_weight)
        _bf16_into(qkv, pi.qkv)
        _i32_into(pos, pi.positions)
        rng = np.random.default_rng([seed, 76])
        lg = W.f32_to_bf16_bits((rng.standard_normal((R, V)) * 3.0).astype(np.float32))
        tm = rng.uniform(0.5, 1.5, R).astype(np.float32)
        dr = rng.exponential(1.0, (R, V)).astype(np.float32)
        _bf16_into(logits, lg)
        temps.copy_(torch.from_numpy(tm))
        draws.copy_(torch.from_numpy(dr))
        g.replay()
        torch.cuda.synchronize()
        assert int(st.d_err.item()) == 0
        # prologue: the same call made directly on fresh buffers gives the same bits
        k2, v2 = dev_bf16(kc), dev_bf16(vc)
        q2 = nv.nv_qk_norm_rope_store(dev_bf16(pi.qkv), torch.from_numpy(pi.positions).cuda(), qw, kw,
                                      torch.from_numpy(b.slot_mapping).cuda(), k2, v2, 16, rms_eps=pi.eps,
                                      rope_theta=pi.theta)
        assert torch.equal(q2, q_out) and torch.equal(k2, st.k_cache[:b.num_blocks])
        assert torch.equal(v2, st.v_cache[:b.num_blocks])
        # sampler: the oracle's token on every row, up to near-ties
        want = orc.sample(lg, tm, dr, threads=4)
        assert (tokens.cpu().numpy() != want).sum() <= 1
