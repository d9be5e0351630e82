// nv_sample_exponential_race: temperature sampling by the exponential race.
//
// What it computes (nano-vLLM field guide, "sampler.py: temperature and the exponential race"):
// for each row, p = softmax(logits / T) and the sampled token is argmax_i p_i / E_i, with E_i the
// row's Exp(1) draws clamped below at 1e-10 (first index on ties).  The draws are an input, as the
// pages draw them with torch's exponential_.
//
// How (GB300): the softmax denominator and max are common to a row, so the argmax is the same as
// argmax_i (logits_i / T - ln E_i): one pass over the row, no normalisation, HBM-bound (2 bytes of
// logits + 4 bytes of draw per vocabulary entry).  Computed in base 2 (scores scaled by log2 e, the
// draw's log2 from the special-function unit).  A row is split over a few CTAs; each thread keeps
// its best (score, index), a block reduces them as 64-bit keys (order-preserving score bits above,
// the complement of the index below, so equal scores prefer the smaller index) and writes the
// block's best key; the row's last CTA to finish (a per-row counter in the workspace) takes the best
// of the row's keys and writes the token, so no separate merge pass runs.
#include "nv_common.cuh"

namespace {

using namespace nvkv;

constexpr int kThreads = 256;
constexpr int kUnroll = 4;         // vectors per thread whose loads go out together (1: 79.8 us, 8: 75.7)
// Per-row counters sit at the start of the workspace in a region of fixed size, so a workspace reused
// for batches of different sizes keeps them in place (they are zero between calls).
constexpr int kMaxRows = 65536;
constexpr size_t kCounterBytes = (size_t)kMaxRows * sizeof(int32_t);

struct SampleParams {
    const __nv_bfloat16 *logits;
    const float *draws;
    const float *temperatures;
    unsigned long long *partial;    // [num_rows, chunks]
    int32_t *done;                  // [num_rows]: chunks finished in this call; zero between calls
    int64_t *tokens;
    int32_t *d_err;
    int64_t logits_stride;          // elements
    int64_t draws_stride;
    int32_t num_rows;
    int32_t vocab;
    int32_t chunks;
    int32_t chunk_len;              // multiple of 8
};

// score -> 32 bits that sort like the score (NaN sorts below everything)
__device__ __forceinline__ uint32_t order_bits(float s)
{
    if (s != s)
        return 0u;
    const uint32_t u = __float_as_uint(s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long make_key(float s, int idx)
{
    return ((unsigned long long)order_bits(s) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ float race_score(float logit, float draw, float scale2)
{
    // log2 of p_i / E_i up to the row's common offset: logit * log2(e) / T - log2(max(E, 1e-10))
    return logit * scale2 - __log2f(fmaxf(draw, 1e-10f));
}

__global__ void __launch_bounds__(kThreads) sample_partial_kernel(const SampleParams p)
{
    const int row = blockIdx.y;
    const int chunk = blockIdx.x;
    const float t = __ldg(p.temperatures + row);
    const int lo = chunk * p.chunk_len;
    const int hi = min(p.vocab, lo + p.chunk_len);
    unsigned long long best = 0ull;     // below every real key
    if (!(t > 0.f) || t == INFINITY) {
        if (chunk == 0 && threadIdx.x == 0)
            flag_error(p.d_err, NV_DERR_VALUE);
    } else {
        const float scale2 = kLog2e / t;
        const __nv_bfloat16 *lr = p.logits + (int64_t)row * p.logits_stride;
        const float *er = p.draws + (int64_t)row * p.draws_stride;
        float bs = -INFINITY;
        int bi = lo;
        // 8 entries per vector: 16 bytes of logits, 32 bytes of draws.  A thread takes vectors
        // v, v + kThreads, ... in increasing order, kUnroll of them loaded before any is compared, so
        // more bytes are in flight; comparing them in order keeps the first index on ties.
        const int nvec = (hi - lo) / 8;
        auto take = [&](int i0, const uint4 &lq, const float4 &e0, const float4 &e1) {
            const float l[8] = {bf16lo(lq.x), bf16hi(lq.x), bf16lo(lq.y), bf16hi(lq.y),
                                bf16lo(lq.z), bf16hi(lq.z), bf16lo(lq.w), bf16hi(lq.w)};
            const float e[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float s = race_score(l[j], e[j], scale2);
                if (s > bs) {           // strictly greater: the first index wins a tie
                    bs = s;
                    bi = i0 + j;
                }
            }
        };
        int v = threadIdx.x;
        for (; v + (kUnroll - 1) * kThreads < nvec; v += kUnroll * kThreads) {
            uint4 lq[kUnroll];
            float4 e0[kUnroll], e1[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i0 = lo + (v + u * kThreads) * 8;
                lq[u] = ld_stream_u4(lr + i0);
                e0[u] = __ldcs(reinterpret_cast<const float4 *>(er + i0));
                e1[u] = __ldcs(reinterpret_cast<const float4 *>(er + i0) + 1);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                take(lo + (v + u * kThreads) * 8, lq[u], e0[u], e1[u]);
        }
        for (; v < nvec; v += kThreads) {
            const int i0 = lo + v * 8;
            take(i0, ld_stream_u4(lr + i0), __ldcs(reinterpret_cast<const float4 *>(er + i0)),
                 __ldcs(reinterpret_cast<const float4 *>(er + i0) + 1));
        }
        for (int i = lo + nvec * 8 + threadIdx.x; i < hi; i += kThreads) {   // ragged tail
            const float s = race_score(__bfloat162float(lr[i]), er[i], scale2);
            if (s > bs) {
                bs = s;
                bi = i;
            }
        }
        if (hi > lo)
            best = make_key(bs, bi);            // an empty thread offers (-inf, chunk start)
    }
    // block reduction of the 64-bit keys
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
    }
    __shared__ unsigned long long wk[kThreads / 32];
    if ((threadIdx.x & 31) == 0)
        wk[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x < 32) {
        best = threadIdx.x < kThreads / 32 ? wk[threadIdx.x] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other > best ? other : best;
        }
        // Publish the block's key, then count the chunk as done; the row's last chunk to get here
        // reads every key of the row (from L2, past this SM's L1) and writes the token.  The fence
        // before the count makes the key visible device-wide first; on the last chunk, the fence
        // after it orders the reads after every other chunk's key.
        int last = 0;
        if (threadIdx.x == 0) {
            p.partial[(int64_t)row * p.chunks + chunk] = best;
            __threadfence();
            const int prev = atomicAdd(p.done + row, 1);
            if (prev < 0 || prev >= p.chunks)
                flag_error(p.d_err, NV_DERR_VALUE);   // the counters were not zero: workspace not zero-filled
            last = prev == p.chunks - 1;
            __threadfence();
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
            unsigned long long m = 0ull;
            for (int c = threadIdx.x; c < p.chunks; c += 32) {
                const unsigned long long k = __ldcg(p.partial + (int64_t)row * p.chunks + c);
                m = k > m ? k : m;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xffffffffu, m, o);
                m = other > m ? other : m;
            }
            if (threadIdx.x == 0) {
                p.tokens[row] = m == 0ull ? -1 : (int64_t)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFull));
                p.done[row] = 0;      // ready for the next call
            }
        }
    }
}

int sample_chunks(int32_t num_rows, int32_t vocab)
{
    // a few waves of CTAs over the whole batch, each CTA at least 4096 entries
    const int want = (1216 + num_rows - 1) / num_rows;
    const int cap = (vocab + 4095) / 4096;
    return want < 1 ? 1 : (want > cap ? (cap < 1 ? 1 : cap) : want);
}

}  // namespace

extern "C" size_t nv_sample_workspace_size(int32_t num_rows, int32_t vocab)
{
    if (num_rows <= 0 || vocab <= 0)
        return 0;
    return kCounterBytes + (size_t)num_rows * sample_chunks(num_rows, vocab) * sizeof(unsigned long long);
}

extern "C" int nv_sample_exponential_race(const void *logits, int64_t logits_stride, const float *temperatures,
                                          const float *draws, int64_t draws_stride, int32_t num_rows,
                                          int32_t vocab, int64_t *tokens, void *workspace, size_t workspace_bytes,
                                          int32_t *d_err, nv_stream_t stream)
{
    using namespace nvkv_host;
    if (num_rows < 0 || vocab <= 0 || logits_stride < vocab || draws_stride < vocab)
        return NV_ERR_SHAPE;
    if (num_rows == 0)
        return NV_OK;
    if (!logits || !temperatures || !draws || !tokens)
        return NV_ERR_NULL;
    if (num_rows > 65535)
        return NV_ERR_UNSUPPORTED;
    if (!aligned16(logits) || !aligned16(draws) || logits_stride % 8 != 0 || draws_stride % 4 != 0)
        return NV_ERR_ALIGN;
    const int chunks = sample_chunks(num_rows, vocab);
    if (!workspace || workspace_bytes < nv_sample_workspace_size(num_rows, vocab) || !aligned16(workspace))
        return NV_ERR_WORKSPACE;
    SampleParams p{};
    p.logits = static_cast<const __nv_bfloat16 *>(logits);
    p.draws = draws;
    p.temperatures = temperatures;
    p.done = static_cast<int32_t *>(workspace);
    p.partial = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(workspace) + kCounterBytes);
    p.tokens = tokens;
    p.d_err = d_err;
    p.logits_stride = logits_stride;
    p.draws_stride = draws_stride;
    p.num_rows = num_rows;
    p.vocab = vocab;
    p.chunks = chunks;
    p.chunk_len = (((vocab + chunks - 1) / chunks) + 7) / 8 * 8;
    sample_partial_kernel<<<dim3(chunks, num_rows), kThreads, 0, (cudaStream_t)stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}
