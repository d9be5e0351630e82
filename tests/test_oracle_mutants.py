"""Plant plausible mistakes in copies of the oracle (on the CPU) and show the pins catch each.

Every mutant is the oracle's C source with one small edit: a wrong index, a dropped term,
an off-by-one causal bound, a swapped GQA map.  If a mutant survived every pin, the pins
could not tell that mistake from the right answer.  Each mutant runs in a child process,
because an index mistake can read outside an array and kill the process (which also
counts as caught).
"""
import os
import subprocess
import sys

import pytest

import oracle

MUTANTS = {
    "slot_offset_uses_division": ("pos % block_size;", "pos / block_size;"),
    "slot_block_index_off_by_one": ("table[pos / block_size]", "table[pos / block_size + 1]"),
    "store_skips_nothing": ("if (s == -1)\n            continue;", "if (s == -2)\n            continue;"),
    "store_uses_k_stride_for_v": ("v + i * v_row_stride", "v + i * k_row_stride"),
    "no_max_subtraction": ("expf(work[j] - m)", "expf(work[j])"),
    "no_normalisation": ("out[t] = out[t] / sum;", "out[t] = out[t];"),
    "scale_dropped": ("const float s = scale * dot;", "const float s = dot;"),
    "causal_off_by_one": ("const int32_t L = (lk - lq) + i + 1;", "const int32_t L = (lk - lq) + i;"),
    "causal_top_left": ("const int32_t L = (lk - lq) + i + 1;", "const int32_t L = i + 1;"),
    "gqa_interleaved_map": ("h / group, head_dim, scale, work, out + r);",
                            "h % num_kv_heads, head_dim, scale, work, out + r);"),
    "value_from_key_cache": ("const uint16_t *vr = v_cache +", "const uint16_t *vr = k_cache +"),
    "zero_len_not_zero": ("out[t] = 0.0f;\n        return;", "out[t] = 1.0f;\n        return;"),
    # attention prologue (QK-norm + RoPE + store)
    "rope_adjacent_pairs": ("const float x1 = n[j], x2 = n[j + half];", "const float x1 = n[2 * j], x2 = n[2 * j + 1];"),
    "rope_sign_flip": ("y[j] = round_bf16(x1 * c - x2 * s);", "y[j] = round_bf16(x1 * c + x2 * s);"),
    "rope_freq_not_inverted": ("const float inv_freq = 1.0f / powf(", "const float inv_freq = 1.0f * powf("),
    "rope_freq_index_j": ("(float)(2 * j) / (float)d", "(float)(j) / (float)d"),
    "norm_eps_dropped": ("sqrtf(var + eps)", "sqrtf(var)"),
    "norm_mean_not_divided": ("const float var = ss / (float)d;", "const float var = ss;"),
    "norm_weight_dropped": ("round_bf16(widen_bf16(cast) * widen_bf16(w[i]))", "round_bf16(widen_bf16(cast))"),
    "k_normed_with_q_weight": ("norm_rope_head(krow + (int64_t)h * head_dim, k_weight,",
                               "norm_rope_head(krow + (int64_t)h * head_dim, q_weight,"),
    "v_stored_from_k": ("memcpy(v_cache + slot * dkv, vrow,", "memcpy(v_cache + slot * dkv, krow,"),
    # attention metadata
    "decode_slot_one_past": ("slot_mapping[b] = last_block * block_size + last_block_num_tokens - 1;",
                             "slot_mapping[b] = last_block * block_size + last_block_num_tokens;"),
    "decode_position_is_len": ("positions[b] = len - 1;", "positions[b] = len;"),
    "decode_padding_not_cleared": ("        slot_mapping[b] = -1;\n        if (b >= num_seqs)",
                                   "        slot_mapping[b] = 0;\n        if (b >= num_seqs)"),
    "prefill_cu_k_counts_new_tokens": ("cu_seqlens_k[b + 1] = cu_seqlens_k[b] + end;",
                                       "cu_seqlens_k[b + 1] = cu_seqlens_k[b] + seqlen_q;"),
    "prefill_first_block_offset_dropped": ("(i == start_block ? start % block_size : 0)", "0"),
    "prefill_positions_from_zero": ("positions[n + (p - start)] = p;", "positions[n + (p - start)] = p - start;"),
    # sampler
    "sampler_temperature_multiplies": ("p[i] = widen_bf16(lr[i]) / t;", "p[i] = widen_bf16(lr[i]) * t;"),
    "sampler_draw_multiplies": ("const float v = (p[i] / sum) / e;", "const float v = (p[i] / sum) * e;"),
    "sampler_last_index_on_ties": ("if (v > best_v) {", "if (v >= best_v) {"),
    "sampler_no_max_subtraction": ("p[i] = expf(p[i] - m);", "p[i] = expf(p[i]);"),
    "sampler_draws_ignored": ("const float v = (p[i] / sum) / e;", "const float v = (p[i] / sum);"),
}

_RUNNER = r"""
import sys
sys.path.insert(0, sys.argv[2])
import oracle
from tests import oracle_pin_checks as pins
orc = oracle.Oracle(sys.argv[1])
caught = []
for check in pins.ALL_CHECKS:
    try:
        check(orc)
    except Exception:
        caught.append(check.__name__)
print("CAUGHT", ",".join(caught))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    c_path = tmp_path / f"{name}.c"
    c_path.write_text(src.replace(old, new))
    so = oracle.compile_c(str(c_path), str(tmp_path / f"lib{name}.so"))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _RUNNER, so, root], capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return      # the mutant crashed or raised outside a check: caught
    line = [l for l in r.stdout.splitlines() if l.startswith("CAUGHT")][-1]
    caught = [c for c in line[len("CAUGHT"):].strip().split(",") if c]
    assert caught, f"mutant {name} passed every pin"
