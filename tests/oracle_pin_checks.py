"""Pins for the CPU oracle: facts fixed by the pages or by the mathematics, not by the oracle.

Each ``check_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` on a miss.  The
same checks run against the real oracle (``test_oracle_pins.py``) and against mutated
copies of it (``test_oracle_mutants.py``), which shows that a plausible mistake in the
oracle (wrong index, dropped term, off-by-one mask, ...) fails at least one of them.
"""
from __future__ import annotations

import json
import os

import numpy as np

import workloads as W
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "slot_examples.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# slot arithmetic (worked examples printed on the pages)
# ---------------------------------------------------------------------------

def check_slot_examples(orc):
    g = golden()
    for ex in g["single_position"]:
        got = orc.slot_of(ex["block_table"], ex["position"], ex["block_size"])
        assert got == ex["slot"], (ex["cite"], got)
    for ex in g["decode"]:
        if "slot_mapping" not in ex:
            continue
        for s, pos, want in zip(ex["seqs"], ex["positions"], ex["slot_mapping"]):
            assert orc.slot_of(s["block_table"], pos, ex["block_size"]) == want, ex["cite"]
    for ex in g["prefill"]:
        if "slot_mapping" not in ex:
            continue
        got = []
        for s in ex["seqs"]:
            a = s["num_cached_tokens"]
            for pos in range(a, a + s["num_scheduled_tokens"]):
                got.append(orc.slot_of(s["block_table"], pos, ex["block_size"]))
        assert got == ex["slot_mapping"], (ex["cite"], got)


# ---------------------------------------------------------------------------
# store_kvcache
# ---------------------------------------------------------------------------

def _small_decode(seed=1, ctx=(5, 40, 64, 70, 1), hq=4, hkv=2, d=16, bs=16, n_pad=2, poison=True):
    return W.make_decode("small-decode", seed, list(ctx), hq, hkv, d, bs, n_pad=n_pad, poison_tail=poison)


def check_store_tiny(orc):
    """After the store, reading each sequence back through the 4-D pool view (no slot arithmetic)
    gives the new row at position L-1 and the old history below it; exactly one row per real
    token changed; padding rows changed nothing."""
    bt = W.tiny()
    kc0, vc0 = bt.cache()
    kc, vc = kc0.copy(), vc0.copy()
    assert orc.store_kvcache(bt.k_new, bt.v_new, bt.slot_mapping, kc, vc) == 0
    for b in range(bt.num_seqs):
        L = int(bt.seq_lens[b])
        k_seq = brute.unpage(kc, bt.block_tables[b], L)
        v_seq = brute.unpage(vc, bt.block_tables[b], L)
        assert np.array_equal(k_seq[L - 1], bt.k_new[b]) and np.array_equal(v_seq[L - 1], bt.v_new[b])
        assert np.array_equal(k_seq[:L - 1], brute.unpage(kc0, bt.block_tables[b], L)[:L - 1])
    changed = np.any((kc != kc0).reshape(-1, bt.kv_row_elems), axis=1)
    assert int(changed.sum()) == bt.num_seqs
    changed_v = np.any((vc != vc0).reshape(-1, bt.kv_row_elems), axis=1)
    assert np.array_equal(changed, changed_v)


def check_store_padding_and_range(orc):
    bt = _small_decode()
    kc0, vc0 = bt.cache()
    kc, vc = kc0.copy(), vc0.copy()
    sm = bt.slot_mapping.copy()
    num_slots = bt.num_blocks * bt.block_size
    assert (sm[-2:] == -1).all()
    sm[0] = num_slots          # one past the pool
    sm[1] = -7                 # below -1
    rejected = orc.store_kvcache(bt.k_new, bt.v_new, sm, kc, vc)
    assert rejected == 2
    flat_k, flat_k0 = kc.reshape(num_slots, -1), kc0.reshape(num_slots, -1)
    changed = np.nonzero(np.any(flat_k != flat_k0, axis=1))[0]
    want = sorted(int(s) for s in sm if 0 <= s < num_slots)
    assert changed.tolist() == want
    for i, s in enumerate(sm):
        if 0 <= s < num_slots:
            assert np.array_equal(flat_k[s], bt.k_new[i].reshape(-1))


def check_store_strided_value(orc):
    """V arrives as a view into a fused QKV row (row stride wider than Hkv*D), as in the pages'
    Qwen3 layer, where value rows are 4096 wide."""
    bt = _small_decode(poison=False)
    n, hkv, d = bt.v_new.shape
    hq = bt.num_q_heads
    fused = np.zeros((n, (hq + 2 * hkv) * d), np.uint16)
    fused[:, (hq + hkv) * d:] = bt.v_new.reshape(n, -1)
    v_view = fused[:, (hq + hkv) * d:].reshape(n, hkv, d)
    kc_a, vc_a = bt.cache()
    kc_b, vc_b = kc_a.copy(), vc_a.copy()
    orc.store_kvcache(bt.k_new, bt.v_new, bt.slot_mapping, kc_a, vc_a)
    orc.store_kvcache(bt.k_new, v_view, bt.slot_mapping, kc_b, vc_b)
    assert np.array_equal(vc_a, vc_b) and np.array_equal(kc_a, kc_b)


def check_store_roundtrip(orc):
    """Store every position of every sequence into a poisoned pool; un-paging gives back the
    contiguous source exactly."""
    lens = [37, 16, 1, 50]
    bs, hkv, d = 16, 2, 8
    rng = np.random.default_rng(5)
    tables, nblocks = W.deal_block_tables(rng, lens, bs)
    pool = np.full((nblocks, bs, hkv, d), W.BF16_NAN_SENTINEL, np.uint16)
    pool_v = pool.copy()
    src_k = [W.normal_bf16(rng, (L, hkv, d)) for L in lens]
    src_v = [W.normal_bf16(rng, (L, hkv, d)) for L in lens]
    slots = np.concatenate([W.physical_slots(tables[b], bs, L) for b, L in enumerate(lens)]).astype(np.int32)
    assert orc.store_kvcache(np.concatenate(src_k), np.concatenate(src_v), slots, pool, pool_v) == 0
    for b, L in enumerate(lens):
        assert np.array_equal(brute.unpage(pool, tables[b], L), src_k[b])
        assert np.array_equal(brute.unpage(pool_v, tables[b], L), src_v[b])


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def _stored(orc, batch):
    kc, vc = batch.cache()
    orc.store_kvcache(batch.k_new, batch.v_new, batch.slot_mapping, kc, vc)
    return kc, vc


def _decode(orc, batch, kc, vc, q=None, scale=None):
    return orc.decode_attn(batch.q if q is None else q, kc, vc, batch.block_tables, batch.context_lens,
                           batch.num_kv_heads, batch.block_size, batch.scale if scale is None else scale)


def check_single_key(orc):
    """A sequence with one key returns that key's V row exactly (softmax weight 1)."""
    bt = W.tiny()
    kc, vc = _stored(orc, bt)
    out = _decode(orc, bt, kc, vc)
    assert int(bt.seq_lens[0]) == 1
    g = bt.num_q_heads // bt.num_kv_heads
    want = W.bf16_bits_to_f32(bt.v_new[0])              # [Hkv, D]
    for h in range(bt.num_q_heads):
        assert np.array_equal(out[0, h], want[h // g])


def check_equal_scores_mean(orc):
    """q = 0 makes every score equal, so the output is the plain mean of the L value rows."""
    bt = W.tiny()
    kc, vc = _stored(orc, bt)
    q0 = np.zeros_like(bt.q)
    out = _decode(orc, bt, kc, vc, q=q0)
    g = bt.num_q_heads // bt.num_kv_heads
    for b in range(bt.num_seqs):
        L = int(bt.seq_lens[b])
        V = brute.widen(brute.unpage(vc, bt.block_tables[b], L))     # [L, Hkv, D]
        mean = V.mean(axis=0)
        for h in range(bt.num_q_heads):
            np.testing.assert_allclose(out[b, h], mean[h // g], rtol=0, atol=2e-6)


def check_two_keys_closed_form(orc):
    """Two keys: weights are the logistic function of the score gap, exactly."""
    hq = hkv = 1
    d, bs = 8, 16
    q = np.zeros((1, hq, d), np.uint16)
    q[0, 0, 0] = W.f32_to_bf16_bits(np.float32(1.0))
    k = np.zeros((1, bs, hkv, d), np.uint16)
    v = np.zeros((1, bs, hkv, d), np.uint16)
    k[0, 0, 0, 0] = W.f32_to_bf16_bits(np.float32(0.5))
    k[0, 1, 0, 0] = W.f32_to_bf16_bits(np.float32(-1.25))
    v[0, 0, 0, :] = W.f32_to_bf16_bits(np.arange(d, dtype=np.float32))
    v[0, 1, 0, :] = W.f32_to_bf16_bits(-2.0 * np.ones(d, np.float32))
    out = orc.decode_attn(q, k, v, np.array([[0]], np.int32), np.array([2], np.int32), 1, bs, 0.75)
    gap = 0.75 * (0.5 - (-1.25))
    w0 = 1.0 / (1.0 + np.exp(-gap))
    want = w0 * np.arange(d) + (1 - w0) * (-2.0)
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-6)


def check_brute_decode(orc):
    for bt in (W.tiny(), _small_decode(), _small_decode(seed=3, ctx=(33, 2, 17), hq=8, hkv=2, n_pad=0)):
        kc, vc = _stored(orc, bt)
        out = _decode(orc, bt, kc, vc)
        ref = brute.decode(bt.q, kc, vc, bt.block_tables, bt.context_lens, bt.scale)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-5)


def check_padding_rows_zero(orc):
    bt = _small_decode()
    kc, vc = _stored(orc, bt)
    out = _decode(orc, bt, kc, vc)
    pad = bt.seq_lens == 0
    assert pad.sum() == 2 and not out[pad].any()


def check_large_scores_finite(orc):
    """Scores of several hundred: a softmax without max subtraction would overflow."""
    bt = _small_decode(poison=False)
    kc, vc = _stored(orc, bt)
    out = _decode(orc, bt, kc, vc, scale=60.0)
    assert np.isfinite(out).all()
    ref = brute.decode(bt.q, kc, vc, bt.block_tables, bt.context_lens, 60.0)
    np.testing.assert_allclose(out, ref, rtol=0, atol=2e-3)


def check_block_permutation_invariance(orc):
    """Relabelling physical blocks (pool and tables together) changes nothing, bit for bit."""
    bt = _small_decode(poison=False)
    kc, vc = _stored(orc, bt)
    out = _decode(orc, bt, kc, vc)
    perm = np.random.default_rng(11).permutation(bt.num_blocks)      # new id of old block i
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    tables = np.where(bt.block_tables >= 0, perm[np.maximum(bt.block_tables, 0)], -1).astype(np.int32)
    out2 = orc.decode_attn(bt.q, kc2, vc2, tables, bt.context_lens, bt.num_kv_heads, bt.block_size, bt.scale)
    assert np.array_equal(out, out2)


def _small_prefill(seed=2, prefix=(0, 32, 48, 16), chunk=(40, 1, 70, 16), hq=4, hkv=2, d=16, bs=16, poison=True):
    return W.make_prefill("small-prefill", seed, list(prefix), list(chunk), hq, hkv, d, bs, poison_tail=poison)


def _prefill(orc, b, kc, vc, q=None, rows=None, scale=None):
    return orc.prefill_attn(b.q if q is None else q, kc, vc, b.cu_seqlens_q, b.cu_seqlens_k, b.block_tables,
                            b.num_kv_heads, b.block_size, b.scale if scale is None else scale, rows=rows)


def check_brute_prefill(orc):
    for b in (_small_prefill(), _small_prefill(seed=4, prefix=(64,), chunk=(5,), hq=2, hkv=2)):
        kc, vc = _stored(orc, b)
        out = _prefill(orc, b, kc, vc)
        ref = brute.prefill(b.q, kc, vc, b.cu_seqlens_q, b.cu_seqlens_k, b.block_tables, b.scale)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-5)


def check_chunked_equals_full(orc):
    """A prompt prefilled in one go, or as a cached prefix plus a chunk, gives the same rows
    (bit for bit): prefix caching and chunked prefill share one path."""
    hq, hkv, d, bs = 4, 2, 16, 16
    Lk, P = 90, 48
    full = W.make_prefill("full", 7, [0], [Lk], hq, hkv, d, bs)
    kc, vc = _stored(orc, full)
    out_full = _prefill(orc, full, kc, vc)
    # The same sequence as P cached tokens plus a chunk of Lk-P: same pool, same table.
    cu_q = np.array([0, Lk - P], np.int32)
    cu_k = np.array([0, Lk], np.int32)
    q_chunk = full.q[P:]
    out_chunk = orc.prefill_attn(q_chunk, kc, vc, cu_q, cu_k, full.block_tables, hkv, bs, full.scale)
    assert np.array_equal(out_chunk, out_full[P:])


def check_decode_equals_last_prefill_row(orc):
    b = _small_prefill(poison=False)
    kc, vc = _stored(orc, b)
    out = _prefill(orc, b, kc, vc)
    cu = b.cu_seqlens_q
    for s in range(b.num_seqs):
        last = int(cu[s + 1]) - 1
        dec = orc.decode_attn(b.q[last:last + 1], kc, vc, b.block_tables[s:s + 1],
                              b.seq_lens[s:s + 1], b.num_kv_heads, b.block_size, b.scale)
        assert np.array_equal(dec[0], out[last])


def check_causal_alignment_spike(orc):
    """Scores that grow by 10 per key position make each query pick its last visible key, so
    query i of a chunk after P cached tokens returns (almost exactly) V[P+i]: the mask is
    aligned bottom-right, and key P+i itself is visible."""
    hq = hkv = 1
    d, bs = 8, 16
    P, Lq = 40, 30
    Lk = P + Lq
    rng = np.random.default_rng(9)
    tables, nb = W.deal_block_tables(rng, [Lk], bs)
    kc = np.zeros((nb, bs, hkv, d), np.uint16)
    vc = W.normal_bf16(rng, (nb, bs, hkv, d))
    slots = W.physical_slots(tables[0], bs, Lk)
    flat_k = kc.reshape(nb * bs, d)
    flat_k[slots, 0] = W.f32_to_bf16_bits(np.arange(Lk, dtype=np.float32))   # exact in bf16 for < 256
    q = np.zeros((Lq, hq, d), np.uint16)
    q[:, 0, 0] = W.f32_to_bf16_bits(np.float32(1.0))
    out = orc.prefill_attn(q, kc, vc, np.array([0, Lq], np.int32), np.array([0, Lk], np.int32), tables,
                           hkv, bs, 10.0)
    V = brute.widen(vc.reshape(nb * bs, d)[slots])
    np.testing.assert_allclose(out[:, 0, :], V[P:Lk], rtol=0, atol=1e-3)


# ---------------------------------------------------------------------------
# attention prologue: QK-norm + RoPE + store
# ---------------------------------------------------------------------------

def _bf16_ulp(v):
    """One bf16 ulp at each |v| (>= the smallest normal's)."""
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def _prologue_case(n=6, hq=4, hkv=2, d=128, seed=3, positions=None):
    rng = np.random.default_rng([seed, 77])
    qkv = W.normal_bf16(rng, (n, (hq + 2 * hkv) * d))
    w = W.f32_to_bf16_bits(1.0 + 0.1 * rng.standard_normal((2, d)).astype(np.float32))
    pos = np.asarray(positions if positions is not None else rng.integers(0, 5000, n), np.int32)
    return qkv, w[0].copy(), w[1].copy(), pos


def _run_prologue(orc, qkv, qw, kw, pos, hq, hkv, slots=None, num_slots=None, eps=1e-6, theta=1e6):
    n = qkv.shape[0]
    d = qw.shape[0]
    slots = np.arange(n, dtype=np.int32) if slots is None else np.asarray(slots, np.int32)
    num_slots = n if num_slots is None else num_slots
    kc = np.full((num_slots, hkv * d), 0x7FC1, np.uint16)
    vc = np.full((num_slots, hkv * d), 0x7FC1, np.uint16)
    q, rej = orc.qk_norm_rope_store(qkv, pos, qw, kw, eps, theta, slots, hq, hkv, kc, vc)
    return q, kc, vc, rej


def check_prologue_brute_force(orc):
    """The C oracle against a float64 restatement: within one bf16 ulp, and equal nearly everywhere."""
    hq, hkv, d = 4, 2, 128
    qkv, qw, kw, pos = _prologue_case(hq=hq, hkv=hkv)
    q, kc, vc, _ = _run_prologue(orc, qkv, qw, kw, pos, hq, hkv)
    n = qkv.shape[0]
    xq = qkv[:, :hq * d].reshape(n, hq, d)
    xk = qkv[:, hq * d:(hq + hkv) * d].reshape(n, hkv, d)
    for got_bits, x, w in ((q, xq, qw), (kc.reshape(n, hkv, d), xk, kw)):
        got = brute.widen(got_bits)
        want = brute.norm_rope(x, w, 1e-6, 1e6, pos)
        diff = np.abs(got - want)
        # the pages form each angle in fp32 (position * frequency): up to pos * 2^-24 rad away from
        # the float64 angle, which moves an output by at most that times the pair's magnitude
        mag = np.abs(want).max(axis=-1, keepdims=True) * 2.0
        tol = _bf16_ulp(want) * 1.01 + mag * pos[:, None, None] * 2.0 ** -23
        assert (diff <= tol).all(), (diff - tol).max()
        assert (diff > 0).mean() < 0.05, (diff > 0).mean()
    # v is stored unchanged
    assert np.array_equal(vc, qkv[:, (hq + hkv) * d:])


def check_prologue_position_zero_is_norm_only(orc):
    """At position 0 every angle is 0: the output is the normalised, weighted input, whatever theta."""
    hq, hkv, d = 2, 1, 128
    qkv, qw, kw, _ = _prologue_case(n=3, hq=hq, hkv=hkv, positions=[0, 0, 0])
    pos = np.zeros(3, np.int32)
    a = _run_prologue(orc, qkv, qw, kw, pos, hq, hkv, theta=1e6)
    b = _run_prologue(orc, qkv, qw, kw, pos, hq, hkv, theta=10.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    x = brute.widen(qkv[:, :hq * d].reshape(3, hq, d))
    r = 1.0 / np.sqrt((x * x).mean(axis=-1, keepdims=True) + 1e-6)
    want = brute.round_bf16(brute.round_bf16(x * r) * brute.widen(qw))
    assert (np.abs(brute.widen(a[0]) - want) <= _bf16_ulp(want) * 1.01).all()


def check_prologue_rope_closed_form(orc):
    """A head vector with one nonzero value a at dim j normalises to sqrt(D) * sign(a) (weight 1),
    and RoPE turns it into (v cos phi, v sin phi) at dims (j, j + D/2), phi = pos * theta^(-2j/D)."""
    hq, hkv, d = 1, 1, 128
    theta = 1e6
    one = np.full(d, 0x3F80, np.uint16)                       # weight 1.0
    for j, pos in ((0, 1), (0, 1000), (1, 4095), (5, 77), (63, 3000)):
        qkv = np.zeros((1, 3 * d), np.uint16)
        qkv[0, j] = 0x3FC0                                     # 1.5
        q, _, _, _ = _run_prologue(orc, qkv, one, one, np.array([pos], np.int32), hq, hkv, theta=theta)
        v = float(brute.round_bf16(np.sqrt(d / (1.0 + 1e-6 * d / 2.25))))   # bf16 of the normalised value
        phi = pos * theta ** (-2.0 * j / d)
        got = brute.widen(q[0, 0])
        want = np.zeros(d)
        want[j], want[j + d // 2] = v * np.cos(phi), v * np.sin(phi)
        want = brute.round_bf16(want)
        assert (np.abs(got - want) <= _bf16_ulp(want) * 1.01 + 1e-6).all(), (j, pos, got[j], want[j])


def check_prologue_relative_position(orc):
    """RoPE makes <q(p), k(p')> depend only on p - p': shifting both positions leaves it unchanged."""
    hq, hkv, d = 1, 1, 128
    one = np.full(d, 0x3F80, np.uint16)
    rng = np.random.default_rng(5)
    qkv = W.normal_bf16(rng, (1, 3 * d))
    qkv2 = np.repeat(qkv, 4, axis=0)
    pos = np.array([700, 400, 1700, 1400], np.int32)           # pairs (700, 400) and (1700, 1400)
    q, kc, _, _ = _run_prologue(orc, qkv2, one, one, pos, hq, hkv)
    qf, kf = brute.widen(q[:, 0]), brute.widen(kc)
    d1 = float(qf[0] @ kf[1])
    d2 = float(qf[2] @ kf[3])
    assert abs(d1 - d2) <= 0.02 * (abs(d1) + 1.0), (d1, d2)
    d3 = float(qf[0] @ kf[3])                                  # a different offset changes it
    assert abs(d3 - d1) > 0.05 * (abs(d1) + 1.0)


def check_prologue_zero_vector_and_slots(orc):
    """A zero head vector stays zero (eps keeps it finite); slot -1 stores nothing but q is
    produced; slots outside the pool are counted and skipped."""
    hq, hkv, d = 2, 1, 128
    qkv, qw, kw, pos = _prologue_case(n=4, hq=hq, hkv=hkv)
    qkv[0, :] = 0
    q, kc, vc, rej = _run_prologue(orc, qkv, qw, kw, pos, hq, hkv, slots=[0, -1, 7, 1], num_slots=3)
    assert not brute.widen(q[0]).any() and np.isfinite(brute.widen(q)).all()
    assert not brute.widen(kc[0]).any()
    assert rej == 1
    assert (kc[2] == 0x7FC1).all() and (vc[2] == 0x7FC1).all()      # nothing for tokens 1 (-1) and 2 (7)
    assert brute.widen(q[1]).any()
    assert np.array_equal(vc[1], qkv[3, (hq + hkv) * d:])


# ---------------------------------------------------------------------------
# attention metadata: prepare_decode / prepare_prefill (worked examples on the pages)
# ---------------------------------------------------------------------------

def check_prepare_decode_golden(orc):
    for ex in golden()["decode"]:
        tables = [s["block_table"] for s in ex["seqs"]]
        w = ex.get("block_table_width", max(len(t) for t in tables))
        bt = np.full((len(tables), w), -1, np.int32)
        for i, t in enumerate(tables):
            bt[i, :len(t)] = t
        lens = [s["num_tokens"] for s in ex["seqs"]]
        pad = ex.get("bucket", len(lens))
        cl, pos, sm, bad = orc.prepare_decode(lens, bt, ex["block_size"], pad)
        assert bad == 0
        assert cl[:len(lens)].tolist() == ex["context_lens"], ex["cite"]
        assert pos[:len(lens)].tolist() == ex["positions"], ex["cite"]
        if "slot_mapping" in ex:
            assert sm[:len(lens)].tolist() == ex["slot_mapping"], ex["cite"]
        for i, L in enumerate(lens):          # the slot of position L-1, by the single-position rule
            assert sm[i] == orc.slot_of(tables[i], L - 1, ex["block_size"])
        if "bucket" in ex:
            assert (sm[len(lens):] == ex["bucket_slot_pad"]).all() and (cl[len(lens):] == ex["bucket_context_pad"]).all()


def check_prepare_prefill_golden(orc):
    for ex in golden()["prefill"]:
        tables = [s["block_table"] for s in ex["seqs"]]
        w = max(len(t) for t in tables)
        bt = np.full((len(tables), w), -1, np.int32)
        for i, t in enumerate(tables):
            bt[i, :len(t)] = t
        nc = [s["num_cached_tokens"] for s in ex["seqs"]]
        ns = [s["num_scheduled_tokens"] for s in ex["seqs"]]
        cq, ck, pos, sm, mx = orc.prepare_prefill(nc, ns, bt, ex["block_size"])
        assert cq.tolist() == ex["cu_seqlens_q"] and ck.tolist() == ex["cu_seqlens_k"], ex["cite"]
        assert mx == (ex["max_seqlen_q"], ex["max_seqlen_k"]), ex["cite"]
        if "positions" in ex:
            assert pos.tolist() == ex["positions"], ex["cite"]
        if "slot_mapping" in ex:
            assert sm.tolist() == ex["slot_mapping"], ex["cite"]
        # every token's slot is the slot of its position, by the single-position rule
        t = 0
        for b in range(len(tables)):
            for p_ in range(nc[b], nc[b] + ns[b]):
                assert sm[t] == orc.slot_of(tables[b], p_, ex["block_size"])
                t += 1


def check_prepare_random_consistency(orc):
    """Random batches: decode slots are the slots of position L-1, prefill slots of each position;
    a row whose length needs more blocks than its table holds is rejected."""
    rng = np.random.default_rng(9)
    for bs in (4, 16, 256):
        lens = rng.integers(1, 40 * bs // 16 + 2, 12)
        nb = (lens + bs - 1) // bs
        bt = np.full((12, int(nb.max())), -1, np.int32)
        perm = rng.permutation(int(nb.sum()))
        k = 0
        for i, n in enumerate(nb):
            bt[i, :n] = perm[k:k + n]
            k += n
        cl, pos, sm, bad = orc.prepare_decode(lens, bt, bs, 15)
        assert bad == 0 and (cl[:12] == lens).all() and (pos[:12] == lens - 1).all()
        for i in range(12):
            assert sm[i] == orc.slot_of(bt[i], int(lens[i]) - 1, bs)
        assert (sm[12:] == -1).all() and (cl[12:] == 0).all()
        cached = (rng.random(12) * lens).astype(np.int32)
        sched = (lens - cached).astype(np.int32)
        cq, ck, pos, sm, mx = orc.prepare_prefill(cached, sched, bt, bs)
        assert ck[-1] == lens.sum() and cq[-1] == sched.sum()
        t = 0
        for i in range(12):
            for p_ in range(int(cached[i]), int(lens[i])):
                assert pos[t] == p_ and sm[t] == orc.slot_of(bt[i], p_, bs)
                t += 1
        too_long = lens.copy()
        too_long[3] = bt.shape[1] * bs + 1
        assert orc.prepare_decode(too_long, bt, bs)[3] == 1


# ---------------------------------------------------------------------------
# sampler: temperature and the exponential race
# ---------------------------------------------------------------------------

def _logit_bits(vals):
    return W.f32_to_bf16_bits(np.asarray(vals, np.float32))


def check_sampler_unit_draws_is_greedy(orc):
    """With every draw equal to 1 the race is won by the most probable token: the first argmax of the
    logits, whatever the temperature."""
    rng = np.random.default_rng(11)
    lg = _logit_bits(rng.standard_normal((6, 1000)) * 3)
    lg[2, 5] = lg[2, 700] = _logit_bits([30.0])[0]           # a tie: the first index wins
    want = np.argmax(brute.widen(lg), axis=1)
    for t in (0.3, 1.0, 2.5):
        got = orc.sample(lg, np.full(6, t, np.float32), np.ones((6, 1000), np.float32))
        assert np.array_equal(got, want), (t, got, want)
    assert want[2] == 5


def check_sampler_closed_form(orc):
    """logits [2, 0], draws [1, 0.2]: p = softmax([2, 0] / T); p0 / 1 vs p1 / 0.2 -- token 0 at T = 1
    (0.881 vs 0.596), token 1 at T = 4 (0.622 vs 1.89).  Equal logits: the smallest draw wins."""
    lg = _logit_bits([[2.0, 0.0]])
    e = np.array([[1.0, 0.2]], np.float32)
    assert orc.sample(lg, np.array([1.0], np.float32), e)[0] == 0
    assert orc.sample(lg, np.array([4.0], np.float32), e)[0] == 1
    eq = _logit_bits(np.zeros((1, 9)))
    d = np.array([[3.0, 0.5, 2.0, 0.4, 0.9, 0.4, 7.0, 1.0, 0.41]], np.float32)
    assert orc.sample(eq, np.array([0.8], np.float32), d)[0] == 3


def check_sampler_large_logits_finite(orc):
    """Logits of 100 at temperature 0.5 (scores of 200) still sample the right token (the softmax is
    max-subtracted)."""
    lg = _logit_bits([[100.0, 99.0, 90.0]])
    d = np.array([[1.0, 0.1, 1.0]], np.float32)          # p1/p0 = e^-2 = 0.135 > 0.1: token 1 wins
    assert orc.sample(lg, np.array([0.5], np.float32), d)[0] == 1


def check_sampler_distribution(orc):
    """The race picks token i with probability softmax(l / T)_i: empirical frequencies over 40000
    independent draws agree within 5 standard errors."""
    lg = _logit_bits([[1.0, 0.5, -0.3, 2.0, 0.0, -1.5, 1.2, 0.8]])
    t = 0.7
    rng = np.random.default_rng(12)
    n = 40000
    draws = rng.exponential(1.0, (n, 8)).astype(np.float32)
    tok = orc.sample(np.repeat(lg, n, axis=0), np.full(n, t, np.float32), draws, threads=4)
    p = np.exp(brute.widen(lg[0]) / t)
    p /= p.sum()
    freq = np.bincount(tok, minlength=8) / n
    se = np.sqrt(p * (1 - p) / n)
    assert (np.abs(freq - p) < 5 * se + 1e-12).all(), (freq, p)


ALL_CHECKS = [
    check_sampler_unit_draws_is_greedy,
    check_sampler_closed_form,
    check_sampler_large_logits_finite,
    check_sampler_distribution,
    check_prepare_decode_golden,
    check_prepare_prefill_golden,
    check_prepare_random_consistency,
    check_prologue_brute_force,
    check_prologue_position_zero_is_norm_only,
    check_prologue_rope_closed_form,
    check_prologue_relative_position,
    check_prologue_zero_vector_and_slots,
    check_slot_examples,
    check_store_tiny,
    check_store_padding_and_range,
    check_store_strided_value,
    check_store_roundtrip,
    check_single_key,
    check_equal_scores_mean,
    check_two_keys_closed_form,
    check_brute_decode,
    check_padding_rows_zero,
    check_large_scores_finite,
    check_block_permutation_invariance,
    check_brute_prefill,
    check_chunked_equals_full,
    check_decode_equals_last_prefill_row,
    check_causal_alignment_spike,
]
