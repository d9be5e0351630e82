// nv_qk_norm_rope_store: the attention layer's prologue -- Qwen3 QK-norm, RoPE, and the K/V store.
//
// What it computes (nano-vLLM field guide, "Qwen3Attention.forward", "layernorm.py",
// "rotary_embedding.py" and Step 10.3): each token's fused projection row is split into q
// [Hq, D], k [Hkv, D], v [Hkv, D]; every q and k head goes through an RMSNorm over its D values
// (statistics in fp32, the normalised value cast to bf16, then multiplied by the bf16 weight),
// then RoPE at the token's position (rotate-half pairs j, j + D/2; angle = position *
// base^(-2j/D); rotation in fp32, cast to bf16); q goes to q_out for attention, and the roped k
// and the untouched v are stored at the token's slot (slot -1 stores nothing).
//
// How (GB300): a memory-bound elementwise pass with a per-head reduction.  One warp handles one
// token: lane l owns frequencies 2l and 2l+1, so the token's sines and cosines are computed once
// and shared by all its heads.  For each head vector of 128 values lane l holds dims 2l, 2l+1 and
// their rotation partners 64+2l, 64+2l+1, so the rotation needs no shuffles and every load and
// store is a coalesced 128-byte row half; the sum of squares is a 5-level butterfly.  The loads
// of kItems heads go out together before any arithmetic, to keep enough bytes in flight for HBM.
// The two bf16 roundings work on pairs: one conversion rounds two normalised values, and one
// bf16x2 multiply forms both weight products (the kernel is issue-bound, so instruction count
// matters).
// The RoPE frequencies are computed once per call on the host (64 floats, passed as a kernel
// parameter); the angle product and sincosf are fp32, as the pages compute them.
#include <cmath>

#include "nv_common.cuh"

namespace {

using namespace nvkv;

constexpr int kD = 128;
constexpr int kItems = 8;              // head vectors of a token whose loads go out together
constexpr int kWarps = 8;              // per block

struct RopeParams {
    const __nv_bfloat16 *qkv;
    const int32_t *positions;
    const __nv_bfloat16 *q_weight;
    const __nv_bfloat16 *k_weight;
    const int32_t *slot_mapping;
    __nv_bfloat16 *q_out;
    __nv_bfloat16 *k_cache;
    __nv_bfloat16 *v_cache;
    int32_t *d_err;
    int64_t row_stride;     // elements between qkv rows
    int64_t num_slots;
    int64_t n_tokens;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    float eps;
    float inv_freq[kD / 2];
};

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t v)
{
    return make_float2(bf16lo(v), bf16hi(v));
}

// bf16x2 product, rounded to nearest: the exact product of two bf16 values fits in fp32, so this
// equals rounding the fp32 product to bf16 (the pages' bf16 multiply by the norm weight)
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__global__ void __launch_bounds__(kWarps * 32) qk_norm_rope_store_kernel(const __grid_constant__ RopeParams p)
{
    const int lane = threadIdx.x & 31;
    const int heads = p.num_q_heads + 2 * p.num_kv_heads;
    const int qk_heads = p.num_q_heads + p.num_kv_heads;
    const int64_t dkv = (int64_t)p.num_kv_heads * kD;
    const int64_t warp_id = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;
    // this lane's weights (dims 2l, 2l+1 and 64+2l, 64+2l+1) and frequencies (2l, 2l+1)
    const uint32_t qw1 = __ldg(reinterpret_cast<const uint32_t *>(p.q_weight) + lane);
    const uint32_t qw2 = __ldg(reinterpret_cast<const uint32_t *>(p.q_weight) + 32 + lane);
    const uint32_t kw1 = __ldg(reinterpret_cast<const uint32_t *>(p.k_weight) + lane);
    const uint32_t kw2 = __ldg(reinterpret_cast<const uint32_t *>(p.k_weight) + 32 + lane);
    const float f0 = p.inv_freq[2 * lane], f1 = p.inv_freq[2 * lane + 1];

    // one warp per token: the token's angles are shared by all its heads
    for (int64_t t = warp_id; t < p.n_tokens; t += nwarps) {
        const uint32_t *row = reinterpret_cast<const uint32_t *>(p.qkv + t * p.row_stride);
        const float pos = (float)__ldg(p.positions + t);
        float s0, c0, s1, c1;
        sincosf(pos * f0, &s0, &c0);
        sincosf(pos * f1, &s1, &c1);
        const int sraw = __ldg(p.slot_mapping + t);
        const bool store = sraw >= 0 && sraw < p.num_slots;
        if (lane == 0 && (sraw < -1 || sraw >= p.num_slots))
            flag_error(p.d_err, NV_DERR_SLOT_RANGE);
        const int64_t slot = store ? sraw : 0;
        // the token's heads, kItems at a time: all loads first, then the arithmetic
        for (int h0 = 0; h0 < heads; h0 += kItems) {
            uint32_t a[kItems], b[kItems];
#pragma unroll
            for (int i = 0; i < kItems; ++i) {
                const int h = h0 + i;
                a[i] = b[i] = 0;
                if (h < heads && (h < p.num_q_heads || store)) {
                    a[i] = __ldg(row + h * (kD / 2) + lane);          // dims 2l, 2l+1
                    b[i] = __ldg(row + h * (kD / 2) + 32 + lane);     // dims 64+2l, 64+2l+1
                }
            }
#pragma unroll
            for (int i = 0; i < kItems; ++i) {
                const int h = h0 + i;
                if (h >= heads)
                    break;
                const bool is_q = h < p.num_q_heads;
                if (!is_q && !store)
                    continue;
                if (h >= qk_heads) {                   // v: stored unchanged
                    uint32_t *dst = reinterpret_cast<uint32_t *>(p.v_cache + slot * dkv + (int64_t)(h - qk_heads) * kD);
                    dst[lane] = a[i];
                    dst[32 + lane] = b[i];
                    continue;
                }
                // RMSNorm over the head's 128 values (fp32 statistics)
                const float2 x1 = bf16x2_to_f2(a[i]), x2 = bf16x2_to_f2(b[i]);
                float ss = x1.x * x1.x + x1.y * x1.y + x2.x * x2.x + x2.y * x2.y;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float r = rsqrtf(ss * (1.0f / kD) + p.eps);
                const uint32_t w1 = is_q ? qw1 : kw1, w2 = is_q ? qw2 : kw2;
                // cast to bf16 (two values per conversion), then the bf16 product with the weight
                const float2 na = bf16x2_to_f2(mul_bf16x2(pack_bf16x2(x1.x * r, x1.y * r), w1));
                const float2 nb = bf16x2_to_f2(mul_bf16x2(pack_bf16x2(x2.x * r, x2.y * r), w2));
                const float n0 = na.x, n1 = na.y, n2 = nb.x, n3 = nb.y;
                // RoPE, rotate-half: (n0, n2) at frequency 2l, (n1, n3) at frequency 2l+1
                const uint32_t y1 = pack_bf16x2(n0 * c0 - n2 * s0, n1 * c1 - n3 * s1);
                const uint32_t y2 = pack_bf16x2(n2 * c0 + n0 * s0, n3 * c1 + n1 * s1);
                uint32_t *dst = is_q
                    ? reinterpret_cast<uint32_t *>(p.q_out + (t * p.num_q_heads + h) * kD)
                    : reinterpret_cast<uint32_t *>(p.k_cache + slot * dkv + (int64_t)(h - p.num_q_heads) * kD);
                dst[lane] = y1;
                dst[32 + lane] = y2;
            }
        }
    }
}

}  // namespace

extern "C" int nv_qk_norm_rope_store(const void *qkv, int64_t qkv_row_stride, const int32_t *positions,
                                     const void *q_norm_weight, const void *k_norm_weight, float rms_eps,
                                     float rope_theta, const int32_t *slot_mapping, int32_t n_tokens,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, void *q_out,
                                     void *k_cache, void *v_cache, int64_t num_slots, int32_t *d_err,
                                     nv_stream_t stream)
{
    using namespace nvkv_host;
    if (n_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_slots < 0)
        return NV_ERR_SHAPE;
    if (n_tokens == 0)
        return NV_OK;
    if (!qkv || !positions || !q_norm_weight || !k_norm_weight || !slot_mapping || !q_out || !k_cache || !v_cache)
        return NV_ERR_NULL;
    if (head_dim != kD)
        return NV_ERR_UNSUPPORTED;
    const int64_t heads = (int64_t)num_q_heads + 2 * num_kv_heads;
    if (qkv_row_stride < heads * kD)
        return NV_ERR_SHAPE;
    if (qkv_row_stride % 8 != 0 || !aligned16(qkv) || !aligned16(q_out) || !aligned16(k_cache) ||
        !aligned16(v_cache) || ((uintptr_t)q_norm_weight & 3) || ((uintptr_t)k_norm_weight & 3))
        return NV_ERR_ALIGN;
    if (!(rope_theta > 1.0f) || !(rms_eps >= 0.0f))
        return NV_ERR_SHAPE;
    const int sms = sm_count();
    if (sms <= 0)
        return NV_ERR_CUDA;

    RopeParams p{};
    p.qkv = static_cast<const __nv_bfloat16 *>(qkv);
    p.positions = positions;
    p.q_weight = static_cast<const __nv_bfloat16 *>(q_norm_weight);
    p.k_weight = static_cast<const __nv_bfloat16 *>(k_norm_weight);
    p.slot_mapping = slot_mapping;
    p.q_out = static_cast<__nv_bfloat16 *>(q_out);
    p.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
    p.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
    p.d_err = d_err;
    p.row_stride = qkv_row_stride;
    p.num_slots = num_slots;
    p.n_tokens = n_tokens;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.eps = rms_eps;
    // inv_freq_j = 1 / base^(2j / D), in fp32 as the pages build their table
    for (int j = 0; j < kD / 2; ++j)
        p.inv_freq[j] = 1.0f / powf(rope_theta, (float)(2 * j) / (float)kD);

    const int64_t blocks_needed = ((int64_t)n_tokens + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)sms * 4;      // half the resident limit: measured a little faster
    const int grid = (int)(blocks_needed < cap ? blocks_needed : cap);
    qk_norm_rope_store_kernel<<<grid, kWarps * 32, 0, (cudaStream_t)stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}
