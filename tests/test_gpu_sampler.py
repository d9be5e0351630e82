"""nv_sample_exponential_race on the GPU against the oracle.

The sampled index is an argmax decided in float32 on both sides, but the GPU ranks entries by
logits*log2(e)/T - log2(E) (the same order as p/E) while the oracle forms p/E after a softmax, so
the two can only disagree between entries whose p/E are within a few float32 ulps.  The test
requires the same token on every row, except that on a row whose two best entries (by a float64
recomputation) are within a relative 1e-5 of each other, either of them is accepted."""
import numpy as np
import pytest

import oracle
import paged_kv_attention_store_gb300 as nv
import workloads as W
from oracle import brute
from tests.gpu_util import dev_bf16

pytestmark = pytest.mark.gpu


def _inputs(B, V, seed, sigma=3.0):
    rng = np.random.default_rng([seed, 91])
    logits = W.f32_to_bf16_bits((rng.standard_normal((B, V)) * sigma).astype(np.float32))
    temps = rng.uniform(0.5, 1.5, B).astype(np.float32)
    draws = rng.exponential(1.0, (B, V)).astype(np.float32)
    return logits, temps, draws


def _gpu(logits, temps, draws):
    """Rows are padded to strides of 8 logits / 4 draws (the kernel's vector width); only V are used."""
    import torch
    B, V = logits.shape
    lp, dp = -(-V // 8) * 8, -(-V // 4) * 4
    lg = np.zeros((B, lp), np.uint16)
    lg[:, :V] = logits
    dr = np.ones((B, dp), np.float32)
    dr[:, :V] = draws
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok = nv.nv_sample_exponential_race(dev_bf16(lg)[:, :V], torch.from_numpy(temps).cuda(),
                                        torch.from_numpy(dr).cuda()[:, :V], d_err=err)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), int(err.item())


def _value64(logits, temps, draws):
    """float64 p_i / max(E_i, 1e-10) up to each row's positive constant."""
    l = brute.widen(logits) / temps.astype(np.float64)[:, None]
    return np.exp(l - l.max(axis=1, keepdims=True)) / np.maximum(draws.astype(np.float64), 1e-10)


def _check(logits, temps, draws, threads=8):
    got, err = _gpu(logits, temps, draws)
    assert err == 0
    want = oracle.default().sample(logits, temps, draws, threads=threads)
    diff = np.nonzero(got != want)[0]
    if diff.size:
        v = _value64(logits[diff], temps[diff], draws[diff])
        best = v.max(axis=1)
        rows = np.arange(diff.size)
        assert (got[diff] >= 0).all()
        assert (v[rows, got[diff]] >= best * (1 - 1e-5)).all(), "GPU token is not a near-tie of the best"
    return diff.size


@pytest.mark.parametrize("B,V", [(1, 8), (7, 1000), (33, 1003), (300, 4096), (5, 50000)])
def test_sampler_shapes(B, V):
    assert _check(*_inputs(B, V, B + V)) <= max(1, B // 100)


def test_sampler_full_vocab_decode_batch():
    """The decode batch's sampling step: 512 rows x 151,936 entries (the Qwen3 vocabulary)."""
    n = _check(*_inputs(512, 151936, 0))
    assert n <= 3


def test_sampler_unit_draws_is_greedy_and_first_index_on_ties():
    logits, temps, _ = _inputs(64, 3000, 5)
    logits[3, 10] = logits[3, 2000] = W.f32_to_bf16_bits(np.array([40.0], np.float32))[0]
    got, _ = _gpu(logits, temps, np.ones((64, 3000), np.float32))
    assert np.array_equal(got, np.argmax(brute.widen(logits), axis=1))
    assert got[3] == 10


def test_sampler_bad_temperature_is_flagged():
    logits, temps, draws = _inputs(4, 512, 6)
    temps[2] = 0.0
    got, err = _gpu(logits, temps, draws)
    assert err & nv.NV_DERR_VALUE and got[2] == -1
    want = oracle.default().sample(logits[[0, 1, 3]], temps[[0, 1, 3]], draws[[0, 1, 3]])
    assert np.array_equal(got[[0, 1, 3]], want)


def test_sampler_workspace_reused_across_batch_sizes():
    """One zero-filled workspace serves calls of different row counts and vocabularies: the per-row
    counters the last block of a row uses are left at zero by every call."""
    import torch
    ws = torch.zeros(max(nv.load_library().nv_sample_workspace_size(B, V) for B, V in ((300, 4096), (7, 50000))),
                     dtype=torch.uint8, device="cuda")
    orc = oracle.default()
    for B, V, seed in ((300, 4096, 1), (7, 50000, 2), (300, 4096, 3), (7, 50000, 4)):
        logits, temps, draws = _inputs(B, V, seed)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        tok = nv.nv_sample_exponential_race(dev_bf16(logits), torch.from_numpy(temps).cuda(),
                                            torch.from_numpy(draws).cuda(), workspace=ws, d_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        want = orc.sample(logits, temps, draws, threads=8)
        assert (tok.cpu().numpy() != want).sum() <= max(1, B // 100)


def test_sampler_workspace_not_zero_filled_is_flagged():
    """Row counters that do not start at zero (a workspace that was not zero-filled) are reported."""
    import torch
    logits, temps, draws = _inputs(16, 50000, 6)
    ws = torch.full((nv.load_library().nv_sample_workspace_size(16, 50000),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    nv.nv_sample_exponential_race(dev_bf16(logits), torch.from_numpy(temps).cuda(), torch.from_numpy(draws).cuda(),
                                  workspace=ws, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & nv.NV_DERR_VALUE
