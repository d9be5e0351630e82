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
// How (GB300): a memory-bound elementwise pass with a per-head reduction, issue-bound on its
// arithmetic, so the layout is chosen for few instructions per value.  One warp handles one token
// and four of its heads at a time: 8 lanes per head, lane i of a head holding dims 8i..8i+7 and
// their rotation partners 64+8i..64+8i+7 (two 16-byte loads, two 16-byte stores), so the rotation
// needs no shuffles and the sum of squares is a 3-level butterfly inside the 8 lanes.  The token's
// sines and cosines are computed once, two frequencies per lane, and gathered to the lanes that
// use them with shuffles.  Values are held as fp32 pairs and the arithmetic uses the packed pair
// instructions (squares, the scaling by 1/rms and the rotation); the two bf16 roundings also work
// on pairs (one conversion rounds two normalised values, one bf16x2 multiply forms both weight
// products).  All of a token's heads (kBatch groups of four) are loaded before any arithmetic, and
// the next token's position and slot one token ahead, so each token costs one memory latency rather
// than three; a padding token's k and v rows are read although nothing of them is stored.
// The RoPE frequencies are computed once per call on the host (64 floats, passed as a kernel
// parameter); the angle product and sincosf are fp32, as the pages compute them.
#include <cmath>

#include "nv_common.cuh"

namespace {

using namespace nvkv;

constexpr int kD = 128;
constexpr int kGroup = 4;              // heads per warp instruction (8 lanes each)
constexpr int kBatch = 8;              // groups of four heads whose loads go out together
constexpr int kWarps = 4;              // per block
constexpr int kBlocksPerSm = 3;        // 158 registers a thread: three 128-thread blocks per SM

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

__device__ __forceinline__ uint32_t word(const uint4 &v, int m)
{
    return m == 0 ? v.x : m == 1 ? v.y : m == 2 ? v.z : v.w;
}

// RMSNorm (fp32 statistics; normalised value cast to bf16, times the bf16 weight) of 8 values
// held as 4 bf16 pairs, given 1/rms: returns the 4 fp32 pairs of the bf16 results.
__device__ __forceinline__ void norm8(const float2 (&x)[4], float r, const uint4 &w, float2 (&n)[4])
{
    const float2 r2 = make_float2(r, r);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float2 xr = __fmul2_rn(x[m], r2);
        n[m] = bf16x2_to_f2(mul_bf16x2(pack_bf16x2(xr.x, xr.y), word(w, m)));
    }
}

__global__ void __launch_bounds__(kWarps * 32, kBlocksPerSm)
    qk_norm_rope_store_kernel(const __grid_constant__ RopeParams p)
{
    const int lane = threadIdx.x & 31;
    const int gi = lane >> 3;              // head of a group of four
    const int li = lane & 7;               // dims 8li..8li+7 and 64+8li..64+8li+7
    const int heads = p.num_q_heads + 2 * p.num_kv_heads;
    const int qk_heads = p.num_q_heads + p.num_kv_heads;
    const int64_t dkv = (int64_t)p.num_kv_heads * kD;
    const int64_t warp_id = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;
    // this lane's weights (4-byte loads: the weights need only 4-byte alignment)
    const uint32_t *qwp = reinterpret_cast<const uint32_t *>(p.q_weight);
    const uint32_t *kwp = reinterpret_cast<const uint32_t *>(p.k_weight);
    const uint4 qw1 = make_uint4(__ldg(qwp + 4 * li), __ldg(qwp + 4 * li + 1), __ldg(qwp + 4 * li + 2),
                                 __ldg(qwp + 4 * li + 3));
    const uint4 qw2 = make_uint4(__ldg(qwp + 32 + 4 * li), __ldg(qwp + 33 + 4 * li), __ldg(qwp + 34 + 4 * li),
                                 __ldg(qwp + 35 + 4 * li));
    const uint4 kw1 = make_uint4(__ldg(kwp + 4 * li), __ldg(kwp + 4 * li + 1), __ldg(kwp + 4 * li + 2),
                                 __ldg(kwp + 4 * li + 3));
    const uint4 kw2 = make_uint4(__ldg(kwp + 32 + 4 * li), __ldg(kwp + 33 + 4 * li), __ldg(kwp + 34 + 4 * li),
                                 __ldg(kwp + 35 + 4 * li));
    // lane l computes the angles of frequencies 2l and 2l+1
    const float f0 = p.inv_freq[2 * lane], f1 = p.inv_freq[2 * lane + 1];

    int nxt_pos = warp_id < p.n_tokens ? __ldg(p.positions + warp_id) : 0;      // one token ahead
    int nxt_slot = warp_id < p.n_tokens ? __ldg(p.slot_mapping + warp_id) : -1;
    for (int64_t t = warp_id; t < p.n_tokens; t += nwarps) {
        const uint4 *row = reinterpret_cast<const uint4 *>(p.qkv + t * p.row_stride);
        const float pos = (float)nxt_pos;
        const int sraw = nxt_slot;
        if (t + nwarps < p.n_tokens) {
            nxt_pos = __ldg(p.positions + t + nwarps);
            nxt_slot = __ldg(p.slot_mapping + t + nwarps);
        }
        float s0, c0, s1, c1;
        sincosf(pos * f0, &s0, &c0);
        sincosf(pos * f1, &s1, &c1);
        // pair m of this lane (dims 8li+2m, 8li+2m+1) rotates at frequencies 8li+2m, 8li+2m+1,
        // computed by lane 4li+m
        float2 cs[4], sn[4], nsn[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int src = 4 * li + m;
            cs[m] = make_float2(__shfl_sync(0xffffffffu, c0, src), __shfl_sync(0xffffffffu, c1, src));
            sn[m] = make_float2(__shfl_sync(0xffffffffu, s0, src), __shfl_sync(0xffffffffu, s1, src));
            nsn[m] = make_float2(-sn[m].x, -sn[m].y);
        }
        const bool store = sraw >= 0 && sraw < p.num_slots;
        if (lane == 0 && (sraw < -1 || sraw >= p.num_slots))
            flag_error(p.d_err, NV_DERR_SLOT_RANGE);
        const int64_t slot = store ? sraw : 0;
        for (int h0 = 0; h0 < heads; h0 += kGroup * kBatch) {
            uint4 a[kBatch], b[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int h = h0 + kGroup * i + gi;
                a[i] = b[i] = make_uint4(0, 0, 0, 0);
                if (h < heads) {
                    a[i] = __ldg(row + h * (kD / 8) + li);          // dims 8li .. 8li+7
                    b[i] = __ldg(row + h * (kD / 8) + 8 + li);      // dims 64+8li .. 64+8li+7
                }
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (h0 + kGroup * i >= heads)
                    break;                                          // the same for every lane
                const int h = h0 + kGroup * i + gi;
                float2 xa[4], xb[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    xa[m] = bf16x2_to_f2(word(a[i], m));
                    xb[m] = bf16x2_to_f2(word(b[i], m));
                }
                // sum of squares over the head's 128 values: 16 here, then the 8 lanes
                float2 q2 = __fmul2_rn(xa[0], xa[0]);
#pragma unroll
                for (int m = 1; m < 4; ++m)
                    q2 = __ffma2_rn(xa[m], xa[m], q2);
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    q2 = __ffma2_rn(xb[m], xb[m], q2);
                float ss = q2.x + q2.y;
                ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (h >= heads || (h >= p.num_q_heads && !store)) {
                    // no head here, or a k / v row of a token that stores nothing
                } else if (h >= qk_heads) {                         // v: stored unchanged
                    uint4 *dst = reinterpret_cast<uint4 *>(p.v_cache + slot * dkv + (int64_t)(h - qk_heads) * kD);
                    dst[li] = a[i];
                    dst[8 + li] = b[i];
                } else {
                    const bool is_q = h < p.num_q_heads;
                    const float r = rsqrtf(ss * (1.0f / kD) + p.eps);
                    float2 na[4], nb[4];
                    norm8(xa, r, is_q ? qw1 : kw1, na);
                    norm8(xb, r, is_q ? qw2 : kw2, nb);
                    // RoPE, rotate-half: y_j = n_j cos - n_{j+64} sin, y_{j+64} = n_{j+64} cos + n_j sin
                    uint32_t y1[4], y2[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float2 u = __ffma2_rn(nb[m], nsn[m], __fmul2_rn(na[m], cs[m]));
                        const float2 v = __ffma2_rn(na[m], sn[m], __fmul2_rn(nb[m], cs[m]));
                        y1[m] = pack_bf16x2(u.x, u.y);
                        y2[m] = pack_bf16x2(v.x, v.y);
                    }
                    uint4 *dst = is_q
                        ? reinterpret_cast<uint4 *>(p.q_out + (t * p.num_q_heads + h) * kD)
                        : reinterpret_cast<uint4 *>(p.k_cache + slot * dkv + (int64_t)(h - p.num_q_heads) * kD);
                    dst[li] = make_uint4(y1[0], y1[1], y1[2], y1[3]);
                    dst[8 + li] = make_uint4(y2[0], y2[1], y2[2], y2[3]);
                }
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
    const int64_t cap = (int64_t)sms * kBlocksPerSm;   // one resident wave
    const int grid = (int)(blocks_needed < cap ? blocks_needed : cap);
    qk_norm_rope_store_kernel<<<grid, kWarps * 32, 0, (cudaStream_t)stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}
