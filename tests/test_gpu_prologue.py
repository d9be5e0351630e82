"""nv_qk_norm_rope_store (QK-norm + RoPE + K/V store) on the GPU against the oracle.

The bar (derived from the arithmetic): both sides compute in fp32 and round to bf16 at the
same points; the GPU's rsqrtf and sincosf differ from the CPU's libm by an ulp or two of fp32.
That can flip the bf16 rounding of a normalised value n (one bf16 ulp of n), which the rotation
y = n_j cos - n_{j+D/2} sin carries into y at up to one ulp of the pair's larger |n| -- many ulps
of y when the two terms cancel -- and y's own rounding can flip too.  So every element must be
within 2 ulp(y) + ulp(max(|n_j|, |n_{j+D/2}|)) of the oracle, and almost all must be equal.
V is a copy: bit for bit."""
import numpy as np
import pytest

import oracle
import paged_kv_attention_store_gb300 as nv
import workloads as W
from oracle import brute
from tests.gpu_util import dev_bf16, dev_i32, host_bits

pytestmark = pytest.mark.gpu


def _ulp(v):
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def _close(got_bits, want_bits, n, what):
    """``n``: the normalised (pre-rotation) values [.., D] the outputs were rotated from."""
    got, want = brute.widen(got_bits), brute.widen(want_bits)
    assert np.isfinite(got).all(), what
    diff = np.abs(got - want)
    h = n.shape[-1] // 2
    pair = np.maximum(np.abs(n[..., :h]), np.abs(n[..., h:]))
    tol = 2.0 * _ulp(want) + 1.01 * _ulp(np.concatenate([pair, pair], axis=-1))
    assert (diff <= tol).all(), (what, float((diff - tol).max()))
    frac = float((diff > 0).mean()) if diff.size else 0.0
    assert frac < 0.05, (what, frac)
    return frac


def _run(batch, seed=0, slots=None):
    import torch
    pi = W.prologue_inputs(batch, seed)
    kc, vc = batch.cache()
    sm = batch.slot_mapping if slots is None else np.asarray(slots, np.int32)
    # oracle
    okc, ovc = kc.copy(), vc.copy()
    oq, rej = oracle.default().qk_norm_rope_store(pi.qkv, pi.positions, pi.q_weight, pi.k_weight, pi.eps, pi.theta,
                                                  sm, batch.num_q_heads, batch.num_kv_heads, okc, ovc)
    # GPU
    k_cache, v_cache = dev_bf16(kc), dev_bf16(vc)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = nv.nv_qk_norm_rope_store(dev_bf16(pi.qkv), dev_i32(pi.positions), dev_bf16(pi.q_weight),
                                 dev_bf16(pi.k_weight), dev_i32(sm), k_cache, v_cache, batch.num_q_heads,
                                 rms_eps=pi.eps, rope_theta=pi.theta, d_err=d_err)
    torch.cuda.synchronize()
    return pi, host_bits(q), host_bits(k_cache), host_bits(v_cache), oq, okc, ovc, rej, int(d_err.item()), kc, vc


def _normed(pi, batch, which):
    hq, hkv, d = batch.num_q_heads, batch.num_kv_heads, batch.head_dim
    n = pi.qkv.shape[0]
    if which == "q":
        return brute.rms_norm(pi.qkv[:, :hq * d].reshape(n, hq, d), pi.q_weight, pi.eps)
    return brute.rms_norm(pi.qkv[:, hq * d:(hq + hkv) * d].reshape(n, hkv, d), pi.k_weight, pi.eps)


def _check_batch(batch, seed=0):
    pi, q, kc, vc, oq, okc, ovc, rej, err, kc0, vc0 = _run(batch, seed)
    assert err == 0 and rej == 0
    _close(q, oq, _normed(pi, batch, "q"), "q")
    assert np.array_equal(vc, ovc)                      # v: copied bit for bit, untouched rows kept
    sel = batch.slot_mapping >= 0
    stored = batch.slot_mapping[sel]
    hkv, d = batch.num_kv_heads, batch.head_dim
    k2, ok2 = kc.reshape(-1, hkv, d), okc.reshape(-1, hkv, d)
    _close(k2[stored], ok2[stored], _normed(pi, batch, "k")[sel], "k")
    keep = np.ones(k2.shape[0], bool)
    keep[stored] = False
    assert np.array_equal(k2[keep], kc0.reshape(-1, hkv, d)[keep])


def test_prologue_tiny():
    _check_batch(W.tiny())


def test_prologue_decode_with_padding_rows():
    _check_batch(W.make_decode("pro-dec", 41, [1, 17, 300, 4000], 32, 8, 128, 16, n_pad=2))


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (8, 8), (16, 2)])
def test_prologue_prefill_shapes(hq, hkv):
    _check_batch(W.make_prefill(f"pro-pf-{hq}-{hkv}", 42, [0, 256, 1000], [5, 130, 64], hq, hkv, 128, 64))


def test_prologue_full_chunked_prefill():
    """The chunked-prefill workload's 16384 new tokens (positions up to 18k), every element."""
    _check_batch(W.prefill_chunk())


def test_prologue_qwen8_decode_step():
    _check_batch(W.qwen8_decode())


def test_prologue_bad_slot_is_flagged_and_skipped():
    b = W.make_decode("pro-bad", 43, [20, 9, 5], 16, 8, 128, 16)
    sm = b.slot_mapping.copy()
    sm[1] = b.num_blocks * 16 + 3                      # outside the pool
    sm[2] = -1                                         # nothing to store, q still produced
    pi, q, kc, vc, oq, okc, ovc, rej, err, kc0, vc0 = _run(b, slots=sm)
    assert err & nv.NV_DERR_SLOT_RANGE and rej == 1
    _close(q, oq, _normed(pi, b, "q"), "q")
    keep = np.ones(kc.reshape(-1, 1024).shape[0], bool)
    keep[sm[0]] = False
    assert np.array_equal(kc.reshape(-1, 1024)[keep], kc0.reshape(-1, 1024)[keep])
    assert np.array_equal(vc, ovc)
