/*
 * Oracle for the paged KV attention store -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-threaded C that states what the hot path of the nano-vLLM
 * engine computes, written from the nano-vLLM field guide (Step 05 "Blocks, block
 * tables and slots"; Step 07.5-07.6 "prepare_prefill" / "prepare_decode"; Step 10.3
 * "attention.py: storing K/V and calling FlashAttention").  Only tests/, the smoke
 * check and the bench's CPU-baseline leg may load it; the product path never does.
 * It shares no code, header or table with the CUDA library.
 *
 * Conventions
 *   - bf16 values are uint16 bit patterns, widened exactly to float.
 *   - A pool of one layer is [num_blocks, block_size, Hkv, D]; one slot is a row of
 *     Hkv*D contiguous values, and slot = block_id * block_size + offset.
 *   - Attention is evaluated per query and per head by its plain definition over
 *     LOGICAL key positions j = 0..L-1:
 *         s_j = scale * sum_d q_d k_{j,d}          (float, summed in d order)
 *         p_j = exp(s_j - max_j s_j)               (float max-subtracted softmax)
 *         o_d = (sum_j p_j v_{j,d}) / (sum_j p_j)  (float, summed in j order)
 *     The output stays float, unrounded.  L == 0 gives zeros.
 *   - GQA: q head h reads kv head h / (Hq / Hkv) (contiguous head groups; the pages
 *     say only that several query heads share one KV head).
 *   - Prefill with fewer queries than keys uses the bottom-right causal alignment the
 *     field guide states for FlashAttention: query i of a chunk of Lq after P cached
 *     tokens sees keys 0..P+i, i.e. L = P + i + 1.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -shared -fPIC (no fast-math; no FMA
 * contraction, so x86-64 and aarch64 hosts give the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static float widen_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Field guide, "Blocks, block tables and slots": the block that holds position
 * `pos` is table[pos / block_size]; the slot is block_id * block_size + pos % block_size. */
int32_t oracle_slot_of(const int32_t *table, int32_t pos, int32_t block_size)
{
    return table[pos / block_size] * block_size + pos % block_size;
}

/* Field guide Step 10.3, the Triton store kernel: for each new-token row i, read
 * slot_mapping[i]; -1 marks a padding row and writes nothing; otherwise copy the
 * row's Hkv*D key values and value values into row `slot` of the flattened caches.
 * Slots the pages never produce (below -1, or past the pool) are skipped and
 * counted; the return value is that count. */
int64_t oracle_store_kvcache(const uint16_t *k, int64_t k_row_stride,
                             const uint16_t *v, int64_t v_row_stride,
                             const int32_t *slot_mapping, int64_t n_tokens,
                             uint16_t *k_cache, uint16_t *v_cache,
                             int64_t num_slots, int32_t row_elems)
{
    int64_t rejected = 0;
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s == -1)
            continue;
        if (s < -1 || s >= num_slots) {
            ++rejected;
            continue;
        }
        memcpy(k_cache + s * row_elems, k + i * k_row_stride, (size_t)row_elems * sizeof(uint16_t));
        memcpy(v_cache + s * row_elems, v + i * v_row_stride, (size_t)row_elems * sizeof(uint16_t));
    }
    return rejected;
}

/* One query vector against logical keys 0..L-1 of one sequence, read through its
 * block table.  `work` holds at least L floats. */
static void attend_one(const uint16_t *qv, int32_t L, const int32_t *table, int32_t block_size,
                       const uint16_t *k_cache, const uint16_t *v_cache, int32_t num_kv_heads,
                       int32_t kv_head, int32_t head_dim, float scale, float *work, float *out)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (L <= 0) {
        for (int32_t t = 0; t < head_dim; ++t)
            out[t] = 0.0f;
        return;
    }
    float m = -INFINITY;
    for (int32_t j = 0; j < L; ++j) {
        const int64_t slot = oracle_slot_of(table, j, block_size);
        const uint16_t *kr = k_cache + slot * row + (int64_t)kv_head * head_dim;
        float dot = 0.0f;
        for (int32_t t = 0; t < head_dim; ++t)
            dot += widen_bf16(qv[t]) * widen_bf16(kr[t]);
        const float s = scale * dot;
        work[j] = s;
        if (s > m)
            m = s;
    }
    float sum = 0.0f;
    for (int32_t j = 0; j < L; ++j) {
        const float p = expf(work[j] - m);
        work[j] = p;
        sum += p;
    }
    for (int32_t t = 0; t < head_dim; ++t)
        out[t] = 0.0f;
    for (int32_t j = 0; j < L; ++j) {
        const int64_t slot = oracle_slot_of(table, j, block_size);
        const uint16_t *vr = v_cache + slot * row + (int64_t)kv_head * head_dim;
        const float p = work[j];
        for (int32_t t = 0; t < head_dim; ++t)
            out[t] += p * widen_bf16(vr[t]);
    }
    for (int32_t t = 0; t < head_dim; ++t)
        out[t] = out[t] / sum;
}

/* Field guide Step 10.3 (decode branch) with Step 07.6: one query per sequence at
 * position L-1, where L = context_lens[b] already counts the token stored in the same
 * forward; it reads keys 0..L-1 through block_tables[b].  q and out are [B, Hq, D].
 * Sequences seq_begin..seq_end-1 are computed (the rest of `out` is untouched).
 * Returns 0, or -1 if scratch memory could not be had. */
int32_t oracle_decode_attn(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *block_tables, int32_t bt_stride, const int32_t *context_lens,
                           int32_t seq_begin, int32_t seq_end, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, float scale, float *out)
{
    const int32_t group = num_q_heads / num_kv_heads;
    int32_t max_len = 1;
    for (int32_t b = seq_begin; b < seq_end; ++b)
        if (context_lens[b] > max_len)
            max_len = context_lens[b];
    float *work = (float *)malloc(sizeof(float) * (size_t)max_len);
    if (!work)
        return -1;
    for (int32_t b = seq_begin; b < seq_end; ++b) {
        for (int32_t h = 0; h < num_q_heads; ++h) {
            const int64_t r = ((int64_t)b * num_q_heads + h) * head_dim;
            attend_one(q + r, context_lens[b], block_tables + (int64_t)b * bt_stride, block_size,
                       k_cache, v_cache, num_kv_heads, h / group, head_dim, scale, work, out + r);
        }
    }
    free(work);
    return 0;
}

/* Field guide Step 10.3 (prefill branch, prefix cache) with Step 07.5: the new tokens
 * of all sequences are packed; sequence b owns query rows cu_q[b]..cu_q[b+1]-1 and
 * Lk = cu_k[b+1]-cu_k[b] keys, of which P = Lk - Lq were cached before this chunk.
 * Query i of the chunk (absolute position P+i) sees keys 0..P+i.
 * `rows` lists the packed query rows to compute (NULL: rows 0..n_rows-1); output row
 * r of `out` ([n_rows, Hq, D]) is query row rows[r].  Returns 0, -1 on allocation
 * failure, -2 if a row is outside the batch. */
int32_t oracle_prefill_attn(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            const int32_t *block_tables, int32_t bt_stride, int32_t num_seqs,
                            const int64_t *rows, int64_t n_rows, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, float scale, float *out)
{
    const int32_t group = num_q_heads / num_kv_heads;
    int32_t max_len = 1;
    for (int32_t b = 0; b < num_seqs; ++b) {
        const int32_t lk = cu_seqlens_k[b + 1] - cu_seqlens_k[b];
        if (lk > max_len)
            max_len = lk;
    }
    float *work = (float *)malloc(sizeof(float) * (size_t)max_len);
    if (!work)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t t = rows ? rows[r] : r;
        int32_t b = 0;
        while (b < num_seqs && !(cu_seqlens_q[b] <= t && t < cu_seqlens_q[b + 1]))
            ++b;
        if (b == num_seqs) {
            free(work);
            return -2;
        }
        const int32_t lq = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        const int32_t lk = cu_seqlens_k[b + 1] - cu_seqlens_k[b];
        const int32_t i = (int32_t)(t - cu_seqlens_q[b]);
        const int32_t L = (lk - lq) + i + 1;
        for (int32_t h = 0; h < num_q_heads; ++h) {
            attend_one(q + (t * num_q_heads + h) * head_dim, L, block_tables + (int64_t)b * bt_stride,
                       block_size, k_cache, v_cache, num_kv_heads, h / group, head_dim, scale, work,
                       out + (r * num_q_heads + h) * head_dim);
        }
    }
    free(work);
    return 0;
}

/* ------------------------------------------------------------------------------------
 * QK-norm + RoPE + store (the attention layer's prologue).
 *
 * Field guide, "Qwen3Attention.forward": the fused projection output of each token is split into
 * q [Hq, D], k [Hkv, D], v [Hkv, D]; q and k go through Qwen3's QK-norm (an RMSNorm over each
 * head's D values, before RoPE), then RoPE at the token's position; k and v are then stored at
 * the token's slot (Step 10.3) and q goes on to attention.
 *   RMSNorm ("layernorm.py"): statistics in float32 -- var = mean(x^2), x * rsqrt(var + eps) --
 *   the result cast back to bf16, THEN multiplied by the bf16 weight (a bf16 product).
 *   RoPE ("rotary_embedding.py"): frequencies inv_freq_j = 1 / base^(2j / D) (float32),
 *   angle = position * inv_freq_j (float32), rotate-half layout: element j pairs with element
 *   j + D/2; y1 = x1 cos - x2 sin, y2 = x2 cos + x1 sin in float32, cast to bf16.
 * ------------------------------------------------------------------------------------ */

/* float -> bf16 bit pattern, round to nearest even (NaN kept quiet). */
static uint16_t round_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x40u);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* One head vector x (D bf16 values): RMSNorm with weight w, then RoPE at `pos`; bf16 out. */
static void norm_rope_head(const uint16_t *x, const uint16_t *w, int32_t d, float eps, float theta, int32_t pos,
                           uint16_t *y)
{
    float ss = 0.0f;
    for (int32_t i = 0; i < d; ++i) {
        const float xi = widen_bf16(x[i]);
        ss += xi * xi;
    }
    const float var = ss / (float)d;
    const float r = 1.0f / sqrtf(var + eps);
    float n[256];
    for (int32_t i = 0; i < d; ++i) {
        const uint16_t cast = round_bf16(widen_bf16(x[i]) * r);            /* x.to(orig_dtype) */
        n[i] = widen_bf16(round_bf16(widen_bf16(cast) * widen_bf16(w[i])));   /* .mul_(weight) in bf16 */
    }
    const int32_t half = d / 2;
    for (int32_t j = 0; j < half; ++j) {
        const float inv_freq = 1.0f / powf(theta, (float)(2 * j) / (float)d);
        const float angle = (float)pos * inv_freq;
        const float c = cosf(angle), s = sinf(angle);
        const float x1 = n[j], x2 = n[j + half];
        y[j] = round_bf16(x1 * c - x2 * s);
        y[j + half] = round_bf16(x2 * c + x1 * s);
    }
}

/* For each token t < n: row t of qkv holds [Hq*D q | Hkv*D k | Hkv*D v] (row_stride elements
 * apart).  q heads -> normed + roped -> q_out[t] ([Hq, D]); k heads -> normed + roped -> row
 * slot_mapping[t] of k_cache; v -> copied unchanged to row slot_mapping[t] of v_cache.  A slot of
 * -1 stores nothing (q is still produced); other slots outside [0, num_slots) are skipped and
 * counted (the return value). */
int64_t oracle_qk_norm_rope_store(const uint16_t *qkv, int64_t row_stride, const int32_t *positions,
                                  const uint16_t *q_weight, const uint16_t *k_weight, float eps, float theta,
                                  const int32_t *slot_mapping, int64_t n, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, uint16_t *q_out, uint16_t *k_cache, uint16_t *v_cache,
                                  int64_t num_slots)
{
    int64_t rejected = 0;
    const int64_t dkv = (int64_t)num_kv_heads * head_dim;
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t *row = qkv + t * row_stride;
        const int32_t pos = positions[t];
        for (int32_t h = 0; h < num_q_heads; ++h)
            norm_rope_head(row + (int64_t)h * head_dim, q_weight, head_dim, eps, theta, pos,
                           q_out + (t * num_q_heads + h) * head_dim);
        const int32_t slot = slot_mapping[t];
        if (slot == -1)
            continue;
        if (slot < -1 || slot >= num_slots) {
            ++rejected;
            continue;
        }
        const uint16_t *krow = row + (int64_t)num_q_heads * head_dim;
        const uint16_t *vrow = krow + dkv;
        for (int32_t h = 0; h < num_kv_heads; ++h)
            norm_rope_head(krow + (int64_t)h * head_dim, k_weight, head_dim, eps, theta, pos,
                           k_cache + slot * dkv + (int64_t)h * head_dim);
        memcpy(v_cache + slot * dkv, vrow, (size_t)dkv * sizeof(uint16_t));
    }
    return rejected;
}

/* ------------------------------------------------------------------------------------
 * Attention metadata (the model runner's prepare_decode / prepare_prefill).
 * ------------------------------------------------------------------------------------ */

/* Field guide Step 07.6 "prepare_decode: one token per sequence": for sequence b with len(seq) =
 * seq_lens[b] tokens (the new one included), position = len - 1, context_len = len, and the slot is
 * the last block's base slot plus last_block_num_tokens - 1, i.e. the slot of position len - 1.
 * Step 07.8 graph replay: rows num_seqs .. padded_seqs-1 get slot -1 and context 0 (position 0).
 * A row whose length is < 1 or needs a block the table does not hold gets slot -1 / context 0;
 * the count of such rows is returned. */
int64_t oracle_prepare_decode(const int32_t *seq_lens, const int32_t *block_tables, int32_t bt_stride,
                              int32_t num_seqs, int32_t padded_seqs, int32_t block_size, int32_t *context_lens,
                              int32_t *positions, int32_t *slot_mapping)
{
    int64_t bad = 0;
    for (int32_t b = 0; b < padded_seqs; ++b) {
        context_lens[b] = 0;
        positions[b] = 0;
        slot_mapping[b] = -1;
        if (b >= num_seqs)
            continue;
        const int32_t len = seq_lens[b];
        const int32_t nblocks = (len + block_size - 1) / block_size;
        if (len < 1 || nblocks > bt_stride) {
            ++bad;
            continue;
        }
        const int32_t last_block = block_tables[(int64_t)b * bt_stride + nblocks - 1];
        const int32_t last_block_num_tokens = len - (nblocks - 1) * block_size;
        context_lens[b] = len;
        positions[b] = len - 1;
        slot_mapping[b] = last_block * block_size + last_block_num_tokens - 1;
    }
    return bad;
}

/* Field guide Step 07.5 "prepare_prefill: pack a varlen batch": sequence b schedules the new
 * tokens [start, end) with start = num_cached[b], end = start + num_scheduled[b]; their positions
 * are start .. end-1; cu_seqlens_q accumulates num_scheduled, cu_seqlens_k accumulates end (the
 * keys include the cached prefix); max_seqlens = {max seqlen_q, max seqlen_k}; slot_mapping walks
 * the blocks the range touches: the first starts at start % block_size, the last ends at
 * end - i * block_size, the ones between contribute all their slots.  Returns the number of
 * tokens written (the sum of num_scheduled), or -1 when a range needs a block the table lacks. */
int64_t oracle_prepare_prefill(const int32_t *num_cached, const int32_t *num_scheduled, const int32_t *block_tables,
                               int32_t bt_stride, int32_t num_seqs, int32_t block_size, int32_t *cu_seqlens_q,
                               int32_t *cu_seqlens_k, int32_t *positions, int32_t *slot_mapping,
                               int32_t *max_seqlens)
{
    int64_t n = 0;
    cu_seqlens_q[0] = 0;
    cu_seqlens_k[0] = 0;
    max_seqlens[0] = 0;
    max_seqlens[1] = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        const int32_t start = num_cached[b];
        const int32_t seqlen_q = num_scheduled[b];
        const int32_t end = start + seqlen_q;
        cu_seqlens_q[b + 1] = cu_seqlens_q[b] + seqlen_q;
        cu_seqlens_k[b + 1] = cu_seqlens_k[b] + end;
        if (seqlen_q > max_seqlens[0])
            max_seqlens[0] = seqlen_q;
        if (end > max_seqlens[1])
            max_seqlens[1] = end;
        for (int32_t p = start; p < end; ++p)
            positions[n + (p - start)] = p;
        const int32_t start_block = start / block_size;
        const int32_t end_block = (end + block_size - 1) / block_size;
        if (end_block > bt_stride)
            return -1;
        int64_t k = n;
        for (int32_t i = start_block; i < end_block; ++i) {
            const int32_t base = block_tables[(int64_t)b * bt_stride + i] * block_size;
            const int32_t slot_start = base + (i == start_block ? start % block_size : 0);
            const int32_t slot_end = (i != end_block - 1) ? base + block_size : base + end - i * block_size;
            for (int32_t s = slot_start; s < slot_end; ++s)
                slot_mapping[k++] = s;
        }
        n += seqlen_q;
    }
    return n;
}

/* ------------------------------------------------------------------------------------
 * Sampler: temperature and the exponential race.
 *
 * Field guide, "sampler.py": logits (bf16, widened to float32) are divided by the row's temperature
 * and turned into probabilities with softmax; the sampled token is argmax_i p_i / E_i, where the
 * E_i are independent Exp(1) draws clamped below at 1e-10.  Here the draws are an input (the pages
 * draw them with torch's exponential_).  The argmax takes the first index on ties (torch's argmax
 * returns the first occurrence).  float32 throughout, as the pages compute it.
 * ------------------------------------------------------------------------------------ */
void oracle_sample_exponential_race(const uint16_t *logits, int64_t logits_stride, const float *temperatures,
                                    const float *draws, int64_t draws_stride, int32_t num_rows, int32_t vocab,
                                    int64_t *tokens)
{
    float *p = (float *)malloc(sizeof(float) * (size_t)vocab);
    for (int32_t r = 0; r < num_rows; ++r) {
        const uint16_t *lr = logits + (int64_t)r * logits_stride;
        const float *er = draws + (int64_t)r * draws_stride;
        const float t = temperatures[r];
        float m = -INFINITY;
        for (int32_t i = 0; i < vocab; ++i) {
            p[i] = widen_bf16(lr[i]) / t;
            if (p[i] > m)
                m = p[i];
        }
        float sum = 0.0f;
        for (int32_t i = 0; i < vocab; ++i) {
            p[i] = expf(p[i] - m);
            sum += p[i];
        }
        int64_t best = 0;
        float best_v = -INFINITY;
        for (int32_t i = 0; i < vocab; ++i) {
            const float e = er[i] < 1e-10f ? 1e-10f : er[i];
            const float v = (p[i] / sum) / e;
            if (v > best_v) {
                best_v = v;
                best = i;
            }
        }
        tokens[r] = best;
    }
    free(p);
}
