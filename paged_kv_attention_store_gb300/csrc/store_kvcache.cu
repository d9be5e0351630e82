// nv_store_kvcache: scatter new K/V rows into their cache slots.
//
// Follows the nano-vLLM field guide, Step 10.3 ("The Triton store kernel"): each new-token
// row i goes to row slot_mapping[i] of the flattened [num_slots, Hkv*D] caches, and a slot
// of -1 (CUDA-graph padding) writes nothing.  The pages launch one program per token; here
// the work is flattened into 16-byte chunks so that consecutive threads move consecutive
// chunks of a row (fully coalesced 16-byte loads and stores), each thread keeps four
// chunks of K and four of V in flight before storing, and the grid is sized in multiples
// of the SM count.  The copy is bit-exact: no value is converted.
#include "nv_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) store_kvcache_kernel(const uint8_t *__restrict__ k, int64_t k_stride_b,
                                                                 const uint8_t *__restrict__ v, int64_t v_stride_b,
                                                                 const int32_t *__restrict__ slot_mapping,
                                                                 uint32_t total_chunks, uint32_t chunks_per_row,
                                                                 uint4 *__restrict__ k_cache,
                                                                 uint4 *__restrict__ v_cache, int64_t num_slots,
                                                                 int32_t *d_err)
{
    const uint32_t step = gridDim.x * (uint32_t)(kThreads * kUnroll);
    for (uint32_t base = blockIdx.x * (uint32_t)(kThreads * kUnroll) + threadIdx.x; base < total_chunks;
         base += step) {
        uint4 kr[kUnroll], vr[kUnroll];
        int64_t dst[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t idx = base + (uint32_t)(u * kThreads);
            dst[u] = -1;
            if (idx < total_chunks) {
                const uint32_t tok = idx / chunks_per_row;
                const uint32_t c = idx - tok * chunks_per_row;
                const int64_t s = __ldg(slot_mapping + tok);
                if (s >= 0 && s < num_slots) {
                    kr[u] = nvkv::ld_stream_u4(k + (int64_t)tok * k_stride_b + (int64_t)c * 16);
                    vr[u] = nvkv::ld_stream_u4(v + (int64_t)tok * v_stride_b + (int64_t)c * 16);
                    dst[u] = s * chunks_per_row + c;
                } else if (s != -1 && c == 0) {
                    nvkv::flag_error(d_err, NV_DERR_SLOT_RANGE);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (dst[u] >= 0) {
                k_cache[dst[u]] = kr[u];
                v_cache[dst[u]] = vr[u];
            }
        }
    }
}

}  // namespace

extern "C" int nv_store_kvcache(const void *k, int64_t k_row_stride, const void *v, int64_t v_row_stride,
                                const int32_t *slot_mapping, int32_t n_tokens, void *k_cache, void *v_cache,
                                int64_t num_slots, int32_t num_kv_heads, int32_t head_dim, int32_t *d_err,
                                nv_stream_t stream)
{
    using namespace nvkv_host;
    if (n_tokens < 0 || num_slots < 0 || num_kv_heads <= 0 || head_dim <= 0)
        return NV_ERR_SHAPE;
    if (n_tokens == 0)
        return NV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache)
        return NV_ERR_NULL;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (row % 8 != 0)
        return NV_ERR_UNSUPPORTED;
    if (k_row_stride < row || v_row_stride < row)
        return NV_ERR_SHAPE;
    if (k_row_stride % 8 || v_row_stride % 8 || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) ||
        !aligned16(v_cache))
        return NV_ERR_ALIGN;
    const uint64_t chunks_per_row = (uint64_t)row / 8;
    const uint64_t total = chunks_per_row * (uint64_t)n_tokens;
    if (total >= (1ull << 31))
        return NV_ERR_UNSUPPORTED;
    const int sms = sm_count();
    if (sms <= 0)
        return NV_ERR_CUDA;
    const uint64_t per_block = (uint64_t)kThreads * kUnroll;
    uint64_t blocks = (total + per_block - 1) / per_block;
    const uint64_t cap = (uint64_t)sms * 16;
    if (blocks > cap)
        blocks = cap;
    store_kvcache_kernel<<<(unsigned)blocks, kThreads, 0, (cudaStream_t)stream>>>(
        static_cast<const uint8_t *>(k), k_row_stride * 2, static_cast<const uint8_t *>(v), v_row_stride * 2,
        slot_mapping, (uint32_t)total, (uint32_t)chunks_per_row, static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), num_slots, d_err);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}
