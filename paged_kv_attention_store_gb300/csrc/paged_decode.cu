// nv_paged_decode_attn: split-KV flash-decoding over a paged KV pool (GQA), CUDA cores.
//
// What it computes is the decode branch of the nano-vLLM field guide's Step 10.3: for
// sequence b with L = context_lens[b] keys (the token stored in this same forward included,
// Step 07.6) and query head h, out[b,h] = softmax_j(scale * q[b,h] . K_j) V_j over the
// kv-head h/group rows of the L logical positions, read through block_tables[b].
//
// How (GB300 design; the pages call a library kernel here):
//   * Work unit = (sequence, split of `split_tokens` consecutive positions).  One CTA takes
//     ALL kv heads of its unit, so each position's K (and V) row of Hkv*128 bf16 values is
//     one contiguous run in the pool, and T consecutive positions inside a block are one
//     contiguous run of T*Hkv*256 bytes: a single 1-D TMA bulk copy moves them into shared
//     memory, completing on an mbarrier.  A producer warp keeps three such chunks in
//     flight per CTA (two CTAs per SM), reading one block-table entry per block.
//   * Consumer warp w owns kv head w and its G = Hq/Hkv query heads, so every K/V element
//     is read from shared memory once and used G times (GQA sharing).  This kernel takes
//     G = 1, 2, 4; with G = 8 or 16 the warps would do too many FMAs per KV byte to keep up
//     with HBM, and decode runs on the tcgen05 tile kernel instead (tile_attention.cuh), as a
//     prefill of one query row per sequence; so do mid-sized group-4 batches and a few long
//     contexts at groups 1-4, where a split-KV grid fills the GPU poorly (decode_on_tiles_rule,
//     below, with the measurements behind it).  A half-warp handles
//     one position at a time, each lane 8 of the 128 dims; partial dot products are reduced
//     with a reduce-scatter over 4 shuffle levels that leaves each lane the full score of
//     one of the G heads, so the exponential is computed once per (position, head).
//   * Online softmax in base 2 with a lazy rescale: the running max only moves when a score
//     exceeds it by more than 8 (a factor 256), which keeps the rescale branch rare; the
//     weights then stay below 2^8 and the accumulation in fp32 is unaffected.
//   * HBM-bound (about 4 flop per byte of KV), so no tensor cores: fp32 FMAs on CUDA cores.
//   * A sequence split over several CTAs writes unnormalised partial outputs plus its
//     (max, sum); the sequence's last CTA to finish (a per-sequence counter in the workspace)
//     combines them and writes the bf16 output, so no separate merge pass runs -- except above
//     16 splits (small batches of long contexts), where merge_splits_kernel follows with a CTA
//     per (sequence, query head).  Single-split sequences write bf16 output directly.
//   * nv_store_decode_attn (the store of the same forward fused in; kFused): the CTA whose
//     split holds position L-1 copies the new K/V row from the inputs into its last staged
//     chunk instead of from the pool, and its consumer warps write that row to its slot.
#include <atomic>
#include <mutex>

#include "nv_common.cuh"
#include "tile_attention.cuh"

namespace {

using namespace nvkv;

constexpr int kD = 128;           // head_dim
constexpr int kT = 8;             // positions per staged chunk
constexpr float kRescaleLog2 = 8.0f;
// Split counters sit at the start of the workspace in a region of fixed size, so a workspace
// reused for batches of different sizes keeps them in place (they are zero between calls).
constexpr int kMaxCountedSeqs = 65536;
constexpr size_t kCounterBytes = (size_t)kMaxCountedSeqs * sizeof(int32_t);

struct DecodeParams {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_cache;
    const __nv_bfloat16 *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    __nv_bfloat16 *out;
    float *part_o;      // [num_seqs, max_splits, Hq, 128]
    float *part_ml;     // [num_seqs, max_splits, Hq, 2]
    int32_t *split_done;  // [num_seqs]: splits finished in this call; zero between calls
    int32_t *d_err;
    int32_t bt_stride;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t block_shift;
    int32_t num_blocks;
    int32_t max_len;    // min(max_context_len, bt_stride * block_size)
    int32_t split_tokens;
    int32_t max_splits;
    int32_t merge_in_kernel;   // 1: a sequence's last split merges; 0: merge_splits_kernel follows
    float scale_log2;   // scale * log2(e)
    // fused store (nv_store_decode_attn); k_new == nullptr for a plain decode
    const __nv_bfloat16 *k_new;     // [num_seqs, Hkv, 128], rows k_new_stride elements apart
    const __nv_bfloat16 *v_new;
    int64_t k_new_stride;
    int64_t v_new_stride;
    const int32_t *slot_mapping;    // [num_seqs]
    __nv_bfloat16 *k_cache_w;       // the pools, writable (same memory as k_cache / v_cache)
    __nv_bfloat16 *v_cache_w;
    int64_t num_slots;
};

// Reduce G per-lane partial sums over the 16 lanes of a half-warp so that each lane ends
// with the FULL sum of exactly one of the G values: lane sl holds value sl / (16 / G).
template <int G>
__device__ __forceinline__ float reduce_to_owner(const float (&x)[G], int sl)
{
    float v[G];
#pragma unroll
    for (int i = 0; i < G; ++i)
        v[i] = x[i];
    int cnt = G;
#pragma unroll
    for (int mask = 8; mask >= 1; mask >>= 1) {
        if (cnt > 1) {
            const bool hi = (sl & mask) != 0;
#pragma unroll
            for (int i = 0; i < G / 2; ++i) {
                if (i < cnt / 2) {
                    const float keep = hi ? v[cnt / 2 + i] : v[i];
                    const float send = hi ? v[i] : v[cnt / 2 + i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                }
            }
            cnt /= 2;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
        }
    }
    return v[0];
}

__device__ __forceinline__ void unpack8(const uint4 &r, float2 (&f)[4])
{
    f[0] = make_float2(bf16lo(r.x), bf16hi(r.x));
    f[1] = make_float2(bf16lo(r.y), bf16hi(r.y));
    f[2] = make_float2(bf16lo(r.z), bf16hi(r.z));
    f[3] = make_float2(bf16lo(r.w), bf16hi(r.w));
}

// Combine the partial results of a sequence that was split: o = sum_s 2^(m_s-M) o_s /
// sum_s 2^(m_s-M) l_s.  Run by the sequence's last CTA, a thread owning 4 dims of one head at a
// time.  The partials were written by other CTAs in this call: read them from L2 (.cg), past this
// SM's L1.
__device__ __forceinline__ void merge_splits(const DecodeParams &p, int b, int nsplit, int tid, int nthreads)
{
    const int items = p.num_q_heads * (kD / 4);
    for (int it = tid; it < items; it += nthreads) {
        const int h = it / (kD / 4);
        const int d4 = it % (kD / 4);
        float M = -INFINITY;
        for (int s = 0; s < nsplit; ++s)
            M = fmaxf(M, __ldcg(p.part_ml + (((size_t)b * p.max_splits + s) * p.num_q_heads + h) * 2));
        float den = 0.f, n0 = 0.f, n1 = 0.f, n2 = 0.f, n3 = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const size_t unit = (size_t)b * p.max_splits + s;
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + (unit * p.num_q_heads + h) * 2));
            const float w = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
            const float4 o = __ldcg(reinterpret_cast<const float4 *>(p.part_o + (unit * p.num_q_heads + h) * kD + d4 * 4));
            den = fmaf(w, ml.y, den);
            n0 = fmaf(w, o.x, n0);
            n1 = fmaf(w, o.y, n1);
            n2 = fmaf(w, o.z, n2);
            n3 = fmaf(w, o.w, n3);
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        uint2 w2;
        w2.x = pack_bf16x2(n0 * inv, n1 * inv);
        w2.y = pack_bf16x2(n2 * inv, n3 * inv);
        *reinterpret_cast<uint2 *>(p.out + ((size_t)b * p.num_q_heads + h) * kD + d4 * 4) = w2;
    }
}

// Sequences with more splits than this merge in merge_splits_kernel after the split launch: the
// in-kernel merge runs on one CTA, whose loop over the splits is bound by L2 latency (one 32K-token
// sequence in 512 splits of 64 positions took 275 us, nearly all of it that merge).
constexpr int kFusedMergeMaxSplits = 16;

// The split partials of sequence blockIdx.x, query head blockIdx.y, combined as in merge_splits: warp
// w takes splits w, w+4, ..., lane l dims 4l..4l+3, and the four warps' sums meet in shared memory.
__global__ void __launch_bounds__(128) merge_splits_kernel(const DecodeParams p)
{
    const int b = blockIdx.x, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int L = __ldg(p.context_lens + b);
    L = L < 0 ? 0 : (L > p.max_len ? p.max_len : L);      // as the split launch read it (it flags)
    const int nsplit = (L + p.split_tokens - 1) / p.split_tokens;
    if (nsplit <= 1)
        return;                   // written directly by its one split (zeros for L == 0)
    const float *ml = p.part_ml + ((size_t)b * p.max_splits * p.num_q_heads + h) * 2;
    const float *po = p.part_o + ((size_t)b * p.max_splits * p.num_q_heads + h) * kD + lane * 4;
    const size_t split_ml = (size_t)p.num_q_heads * 2, split_o = (size_t)p.num_q_heads * kD;
    __shared__ float s_m[4];
    __shared__ float4 s_n[4][32];
    __shared__ float s_den[4];
    float M = -INFINITY;
    for (int sp = threadIdx.x; sp < nsplit; sp += 128)
        M = fmaxf(M, ml[sp * split_ml]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0)
        s_m[warp] = M;
    __syncthreads();
    M = fmaxf(fmaxf(s_m[0], s_m[1]), fmaxf(s_m[2], s_m[3]));
    float den = 0.f;
    float4 n = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int sp = warp; sp < nsplit; sp += 4) {
        const float2 m_l = *reinterpret_cast<const float2 *>(ml + sp * split_ml);
        const float4 o = *reinterpret_cast<const float4 *>(po + sp * split_o);
        const float w = (m_l.x == -INFINITY) ? 0.f : fast_exp2(m_l.x - M);
        den = fmaf(w, m_l.y, den);
        n.x = fmaf(w, o.x, n.x);
        n.y = fmaf(w, o.y, n.y);
        n.z = fmaf(w, o.z, n.z);
        n.w = fmaf(w, o.w, n.w);
    }
    s_n[warp][lane] = n;
    if (lane == 0)
        s_den[warp] = den;
    __syncthreads();
    if (warp == 0) {
        float4 t = s_n[0][lane];
        for (int w2 = 1; w2 < 4; ++w2) {
            const float4 u = s_n[w2][lane];
            t.x += u.x;
            t.y += u.y;
            t.z += u.z;
            t.w += u.w;
        }
        const float d = s_den[0] + s_den[1] + s_den[2] + s_den[3];
        const float inv = d > 0.f ? 1.f / d : 0.f;
        uint2 w2;
        w2.x = pack_bf16x2(t.x * inv, t.y * inv);
        w2.y = pack_bf16x2(t.z * inv, t.w * inv);
        *reinterpret_cast<uint2 *>(p.out + ((size_t)b * p.num_q_heads + h) * kD + lane * 4) = w2;
    }
}

constexpr int kStages = 3;   // chunks in flight per CTA: 96 KB at 8 kv heads, two CTAs per SM

__host__ __device__ constexpr size_t decode_smem_bytes(int stages, int num_kv_heads)
{
    return (size_t)stages * 2 * kT * num_kv_heads * kD * 2 + 2 * stages * 8 + stages * 4 + 16;
}

template <int G, int MAX_KV_HEADS, bool kFused>
__global__ void __launch_bounds__((MAX_KV_HEADS + 1) * 32, MAX_KV_HEADS <= 8 ? 2 : 1)
    paged_decode_kernel(const DecodeParams p)
{
    constexpr int kS = kStages;
    extern __shared__ __align__(128) uint8_t smem[];
    const int hkv = p.num_kv_heads;
    const int dkv = hkv * kD;                        // elements per pool row
    const uint32_t chunk_bytes = (uint32_t)kT * dkv * 2;  // one K (or V) chunk
    const int b = blockIdx.x;
    const int split = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    int L = __ldg(p.context_lens + b);
    if (L < 0 || L > p.max_len) {
        if (split == 0 && threadIdx.x == 0)
            flag_error(p.d_err, NV_DERR_LENGTH);
        L = L < 0 ? 0 : p.max_len;
    }
    const int t0 = split * p.split_tokens;
    if (L == 0) {
        if (kFused && split == 0 && threadIdx.x == 0 && __ldg(p.slot_mapping + b) >= 0)
            flag_error(p.d_err, NV_DERR_SLOT_MISMATCH);   // a new row for a row with no position L-1
        if (split == 0) {   // padding row: attends to nothing, writes zeros
            uint4 *o = reinterpret_cast<uint4 *>(p.out + (size_t)b * p.num_q_heads * kD);
            for (int i = threadIdx.x; i < p.num_q_heads * kD / 8; i += blockDim.x)
                o[i] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    if (t0 >= L)
        return;
    const int t1 = min(L, t0 + p.split_tokens);
    // Fused store: the new token is position L-1; its K/V rows come straight from k_new / v_new
    // (no round trip through the pool) and this CTA also writes them to their slot.  That is only
    // done when slot_mapping[b] is the slot of position L-1 through the block table; otherwise the
    // row is not stored, position L-1 is read from the pool, and NV_DERR_SLOT_MISMATCH is set.
    int new_pos = -1;
    int64_t new_slot = 0;
    if (kFused && t1 == L) {                    // only the CTA that holds position L-1
        const int s = __ldg(p.slot_mapping + b);
        if (s >= 0) {
            const int lp = L - 1;
            const int blk = __ldg(p.block_tables + (size_t)b * p.bt_stride + (lp >> p.block_shift));
            const int64_t want = ((int64_t)blk << p.block_shift) + (lp & ((1 << p.block_shift) - 1));
            if (s < p.num_slots && blk >= 0 && blk < p.num_blocks && want == s) {
                new_pos = lp;
                new_slot = s;
            } else if (threadIdx.x == 0) {
                flag_error(p.d_err, s < p.num_slots ? NV_DERR_SLOT_MISMATCH : NV_DERR_SLOT_RANGE);
            }
        } else if (s < -1 && threadIdx.x == 0) {
            flag_error(p.d_err, NV_DERR_SLOT_RANGE);
        }
    }
    const int nsplit = (L + p.split_tokens - 1) / p.split_tokens;
    const int nchunks = (t1 - t0 + kT - 1) / kT;

    // shared memory: [kS][K chunk | V chunk], then barriers and per-stage valid counts
    const uint32_t stage_bytes = 2 * chunk_bytes;
    uint8_t *tail = smem + (size_t)kS * stage_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(tail);   // full[kS], empty[kS]
    int32_t *valid_rows = reinterpret_cast<int32_t *>(tail + 2 * kS * sizeof(uint64_t));
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t bar_base = smem_u32(bars);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(bar_base + 8 * s, 1);                    // full: producer arrive + tx bytes
            mbar_init(bar_base + 8 * (kS + s), hkv);   // empty: one arrive per consumer warp
        }
        fence_barrier_init();
    }
    // Rows a partial chunk does not copy keep stale-but-finite values (zero at first).
    for (uint32_t i = threadIdx.x; i < (uint32_t)kS * stage_bytes / 16; i += blockDim.x)
        sts_u4(smem_base + 16 * i, make_uint4(0, 0, 0, 0));
    fence_proxy_async_smem();   // the zeros must land before any bulk copy writes these bytes
    __syncthreads();

    if (warp == hkv) {
        // ---------------- producer: one lane issues the bulk copies ----------------
        if (lane == 0) {
            const int bs_mask = (1 << p.block_shift) - 1;
            const int32_t *bt = p.block_tables + (size_t)b * p.bt_stride;
            int cur_lblk = -1;
            int64_t blk_slot0 = 0;
            bool blk_ok = false;
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kS;
                if (c >= kS && !mbar_wait(bar_base + 8 * (kS + s), ((c / kS) - 1) & 1)) {
                    flag_error(p.d_err, NV_DERR_TIMEOUT);
                    break;
                }
                const int tok0 = t0 + c * kT;
                const int n = min(kT, t1 - tok0);
                const int lblk = tok0 >> p.block_shift;
                if (lblk != cur_lblk) {
                    cur_lblk = lblk;
                    const int blk = __ldg(bt + lblk);
                    blk_ok = blk >= 0 && blk < p.num_blocks;
                    if (!blk_ok)
                        flag_error(p.d_err, NV_DERR_BLOCK_RANGE);
                    blk_slot0 = (int64_t)blk << p.block_shift;
                }
                const uint32_t full = bar_base + 8 * s;
                if (blk_ok) {
                    valid_rows[s] = n;
                    const int64_t slot = blk_slot0 + (tok0 & bs_mask);
                    const uint32_t row = (uint32_t)dkv * 2;
                    mbar_arrive_expect_tx(full, 2u * (uint32_t)n * row);
                    // rows from the pool, except the new token's, which comes from k_new / v_new
                    const int from_pool = (kFused && new_pos >= tok0 && new_pos < tok0 + n) ? new_pos - tok0 : n;
                    if (from_pool > 0) {
                        bulk_g2s(smem_base + s * stage_bytes, p.k_cache + slot * dkv, (uint32_t)from_pool * row, full);
                        bulk_g2s(smem_base + s * stage_bytes + chunk_bytes, p.v_cache + slot * dkv,
                                 (uint32_t)from_pool * row, full);
                    }
                    if (from_pool < n) {
                        bulk_g2s(smem_base + s * stage_bytes + (uint32_t)from_pool * row,
                                 p.k_new + (size_t)b * p.k_new_stride, row, full);
                        bulk_g2s(smem_base + s * stage_bytes + chunk_bytes + (uint32_t)from_pool * row,
                                 p.v_new + (size_t)b * p.v_new_stride, row, full);
                    }
                } else {
                    valid_rows[s] = 0;     // keys of an out-of-pool block are treated as absent
                    mbar_arrive(full);
                }
                issued = c + 1;
            }
            // Do not leave while copies still land in this CTA's shared memory.
            for (int c = max(0, issued - kS); c < issued; ++c)
                mbar_wait(bar_base + 8 * (c % kS), (c / kS) & 1);
        }
        return;
    }

    // ---------------- consumers: warp w = kv head w and its G query heads ----------------
    const int kvh = warp;
    const int half = lane >> 4;
    const int sl = lane & 15;
    constexpr int kLanesPerHead = 16 / G;
    const int head0 = kvh * G;

    // Dims are held in pairs and the dot products and accumulations use the packed fp32 pair
    // instructions: each one does the FMAs of two dims.
    const float2 scale2 = make_float2(p.scale_log2, p.scale_log2);
    float2 qf[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 r = *reinterpret_cast<const uint4 *>(p.q + ((size_t)b * p.num_q_heads + head0 + g) * kD + sl * 8);
        unpack8(r, qf[g]);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            qf[g][i] = __fmul2_rn(qf[g][i], scale2);
    }
    float2 acc2[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            acc2[g][i] = make_float2(0.f, 0.f);
    float m_run = -INFINITY;   // running max (log2 units) of head own_g, this half's positions
    float l_run = 0.f;         // running sum of weights of head own_g

    // lane's column inside a staged row: kv head kvh, dims sl*8 .. sl*8+7
    const uint32_t col_off = (uint32_t)(kvh * kD + sl * 8) * 2;
    const uint32_t row_bytes = (uint32_t)dkv * 2;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % kS;
        if (!__all_sync(0xffffffffu, mbar_wait(bar_base + 8 * s, (c / kS) & 1))) {
            if (lane == 0)
                flag_error(p.d_err, NV_DERR_TIMEOUT);
            ok = false;
            break;
        }
        const int nvalid = valid_rows[s];
        const uint32_t kbase = smem_base + s * stage_bytes + col_off;
        const uint32_t vbase = kbase + chunk_bytes;

        float sc[kT / 2];
#pragma unroll
        for (int jj = 0; jj < kT / 2; ++jj) {
            const int j = half * (kT / 2) + jj;
            float2 kf[4];
            unpack8(lds_u4(kbase + j * row_bytes), kf);
            float part[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float2 a = __fmul2_rn(qf[g][0], kf[0]);
#pragma unroll
                for (int i = 1; i < 4; ++i)
                    a = __ffma2_rn(qf[g][i], kf[i], a);
                part[g] = a.x + a.y;
            }
            const float full = reduce_to_owner<G>(part, sl);
            sc[jj] = (j < nvalid) ? full : -INFINITY;
        }
        float mx = sc[0];
#pragma unroll
        for (int jj = 1; jj < kT / 2; ++jj)
            mx = fmaxf(mx, sc[jj]);
        const bool need = mx > m_run + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? fast_exp2(m_run - mx) : 1.f;   // m_run = -inf -> 0
            if (need)
                m_run = mx;
            l_run *= alpha;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float a = __shfl_sync(0xffffffffu, alpha, (half << 4) + g * kLanesPerHead);
                const float2 a2 = make_float2(a, a);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    acc2[g][i] = __fmul2_rn(acc2[g][i], a2);
            }
        }
        float pj[kT / 2];
#pragma unroll
        for (int jj = 0; jj < kT / 2; ++jj) {
            pj[jj] = (sc[jj] == -INFINITY) ? 0.f : fast_exp2(sc[jj] - m_run);
            l_run += pj[jj];
        }
#pragma unroll
        for (int jj = 0; jj < kT / 2; ++jj) {
            const int j = half * (kT / 2) + jj;
            float2 vf[4];
            unpack8(lds_u4(vbase + j * row_bytes), vf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pg = __shfl_sync(0xffffffffu, pj[jj], (half << 4) + g * kLanesPerHead);
                const float2 pg2 = make_float2(pg, pg);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    acc2[g][i] = __ffma2_rn(pg2, vf[i], acc2[g][i]);
            }
        }
        // fused store: this warp writes its kv head of the new row (K by lanes 0-15, V by 16-31)
        if (kFused && new_pos >= t0 + c * kT && new_pos < t0 + c * kT + kT && nvalid > 0) {
            const int tok0 = t0 + c * kT;
            const uint32_t src = (half ? vbase : kbase) + (uint32_t)(new_pos - tok0) * row_bytes;
            __nv_bfloat16 *dst = (half ? p.v_cache_w : p.k_cache_w) + new_slot * dkv + kvh * kD + sl * 8;
            *reinterpret_cast<uint4 *>(dst) = lds_u4(src);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar_base + 8 * (kS + s));
    }

    // ---- merge the two half-warps (they saw disjoint positions), then write ----
    float acc[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[g][2 * i] = acc2[g][i].x;
            acc[g][2 * i + 1] = acc2[g][i].y;
        }
    float m_g[G], l_g[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m_g[g] = __shfl_sync(0xffffffffu, m_run, (half << 4) + g * kLanesPerHead);
        l_g[g] = __shfl_sync(0xffffffffu, l_run, (half << 4) + g * kLanesPerHead);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float mo = __shfl_xor_sync(0xffffffffu, m_g[g], 16);
        const float lo = __shfl_xor_sync(0xffffffffu, l_g[g], 16);
        const float M = fmaxf(m_g[g], mo);
        const float fa = (m_g[g] == -INFINITY) ? 0.f : fast_exp2(m_g[g] - M);
        const float fb = (mo == -INFINITY) ? 0.f : fast_exp2(mo - M);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float other = __shfl_xor_sync(0xffffffffu, acc[g][i], 16);
            acc[g][i] = acc[g][i] * fa + other * fb;
        }
        m_g[g] = M;
        l_g[g] = l_g[g] * fa + lo * fb;
    }

    if (nsplit == 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if ((G == 1 && half == 0) || (G > 1 && (g & 1) == half)) {
                const float inv = l_g[g] > 0.f ? 1.f / l_g[g] : 0.f;
                uint4 w;
                w.x = pack_bf16x2(acc[g][0] * inv, acc[g][1] * inv);
                w.y = pack_bf16x2(acc[g][2] * inv, acc[g][3] * inv);
                w.z = pack_bf16x2(acc[g][4] * inv, acc[g][5] * inv);
                w.w = pack_bf16x2(acc[g][6] * inv, acc[g][7] * inv);
                *reinterpret_cast<uint4 *>(p.out + ((size_t)b * p.num_q_heads + head0 + g) * kD + sl * 8) = w;
            }
        }
    } else {
        const size_t unit = (size_t)b * p.max_splits + split;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if ((G == 1 && half == 0) || (G > 1 && (g & 1) == half)) {
                float *po = p.part_o + (unit * p.num_q_heads + head0 + g) * kD + sl * 8;
                *reinterpret_cast<float4 *>(po) = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
                *reinterpret_cast<float4 *>(po + 4) = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
                if (sl == 0)
                    *reinterpret_cast<float2 *>(p.part_ml + (unit * p.num_q_heads + head0 + g) * 2) =
                        make_float2(m_g[g], l_g[g]);
            }
        }
        if (!p.merge_in_kernel)
            return;           // many splits: merge_splits_kernel combines them after this launch
        // Count this split as done (its partials made visible first); the sequence's last split
        // to get here merges them all.  Every CTA with t0 < L reaches this point exactly once,
        // whatever happened in its loop, so the counter always reaches nsplit and is reset.
        // (The barrier orders the warps' partial stores before thread 0's fence, which makes them
        // visible device-wide before its count; on the last split, the fence after the count
        // orders the merge's reads after every other split's partials.)
        __shared__ int s_last;
        const uint32_t consumers = (uint32_t)hkv * 32u;
        asm volatile("bar.sync 1, %0;" ::"r"(consumers) : "memory");
        if (threadIdx.x == 0) {
            __threadfence();
            const int prev = atomicAdd(p.split_done + b, 1);
            s_last = prev == nsplit - 1;
            if (prev < 0 || prev >= nsplit)
                flag_error(p.d_err, NV_DERR_VALUE);   // the counters were not zero: workspace not zero-filled
            __threadfence();
        }
        asm volatile("bar.sync 1, %0;" ::"r"(consumers) : "memory");
        if (s_last) {
            merge_splits(p, b, nsplit, (int)threadIdx.x, (int)consumers);
            if (threadIdx.x == 0)
                p.split_done[b] = 0;      // ready for the next call
        }
    }
}

// Positions per split: aim for at least ~1200 work units so every SM has several, but keep
// units long enough (>= 64 positions) that the partial-output traffic stays a few percent, and
// stop at 256 positions once there are 600 units: each sequence's last split merges all of its
// partials, so on a small batch of long contexts more, shorter splits cost more than they gain
// (64 sequences x 4096: 202 us at 128 positions, 178 us at 256).
int decode_split_tokens(int num_seqs, int max_context_len)
{
    auto units = [&](int sp) { return (int64_t)num_seqs * ((max_context_len + sp - 1) / sp); };
    int split = 512;
    while (split > 64 && units(split) < 1200 && !(split <= 256 && units(split) >= 600))
        split >>= 1;
    return split;
}

// The store half of nv_store_decode_attn when its decode runs on the tile kernel: a warp per row
// writes the new K/V row of sequence b to slot_mapping[b] only when that is the slot of position
// L-1 through the block table -- the rule the fused CUDA-core kernel applies -- and flags any
// other slot the same way (the decode then reads position L-1 from the pool).
__global__ void __launch_bounds__(256) decode_store_kernel(const DecodeParams p, int num_seqs)
{
    const int b = blockIdx.x * 8 + (int)(threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= num_seqs)
        return;
    const int s = __ldg(p.slot_mapping + b);
    if (s == -1)
        return;
    int L = __ldg(p.context_lens + b);
    L = L < 0 ? 0 : (L > p.max_len ? p.max_len : L);   // as the decode reads it (it flags the length)
    if (s < -1 || s >= p.num_slots) {
        if (lane == 0)
            flag_error(p.d_err, NV_DERR_SLOT_RANGE);
        return;
    }
    const int lp = L - 1;
    const int blk = L > 0 ? __ldg(p.block_tables + (size_t)b * p.bt_stride + (lp >> p.block_shift)) : -1;
    const int64_t want = ((int64_t)blk << p.block_shift) + (lp & ((1 << p.block_shift) - 1));
    if (L == 0 || blk < 0 || blk >= p.num_blocks || want != s) {
        if (lane == 0)
            flag_error(p.d_err, NV_DERR_SLOT_MISMATCH);
        return;
    }
    const int row_u4 = p.num_kv_heads * kD / 8;
    const uint4 *kr = reinterpret_cast<const uint4 *>(p.k_new + (size_t)b * p.k_new_stride);
    const uint4 *vr = reinterpret_cast<const uint4 *>(p.v_new + (size_t)b * p.v_new_stride);
    uint4 *kd = reinterpret_cast<uint4 *>(p.k_cache_w + (int64_t)s * p.num_kv_heads * kD);
    uint4 *vd = reinterpret_cast<uint4 *>(p.v_cache_w + (int64_t)s * p.num_kv_heads * kD);
    for (int i = lane; i < row_u4; i += 32) {
        kd[i] = __ldg(kr + i);
        vd[i] = __ldg(vr + i);
    }
}

template <int G, int MAXH, bool kFused>
int launch_decode(const DecodeParams &p, int num_seqs, cudaStream_t stream)
{
    const size_t smem_bytes = decode_smem_bytes(kStages, p.num_kv_heads);
    // The shared-memory opt-in is a per-device attribute: bit d records that device d has it.
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return NV_ERR_CUDA;
    if (!((configured.load(std::memory_order_acquire) >> dev) & 1u)) {
        if (cudaFuncSetAttribute(paged_decode_kernel<G, MAXH, kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes > 200 * 1024 ? 227 * 1024 : 200 * 1024) != cudaSuccess)
            return NV_ERR_CUDA;
        configured.fetch_or(1ull << dev, std::memory_order_release);
    }
    dim3 grid(num_seqs, p.max_splits);
    paged_decode_kernel<G, MAXH, kFused><<<grid, (p.num_kv_heads + 1) * 32, smem_bytes, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

template <int MAXH, bool kFused>
int dispatch_group(int group, const DecodeParams &p, int num_seqs, cudaStream_t st)
{
    switch (group) {
    case 1: return launch_decode<1, MAXH, kFused>(p, num_seqs, st);
    case 2: return launch_decode<2, MAXH, kFused>(p, num_seqs, st);
    case 4: return launch_decode<4, MAXH, kFused>(p, num_seqs, st);
    default: return NV_ERR_UNSUPPORTED;
    }
}

int dispatch(int group, const DecodeParams &p, int num_seqs, cudaStream_t st)
{
    const bool fused = p.k_new != nullptr;
    if (p.num_kv_heads <= 8)
        return fused ? dispatch_group<8, true>(group, p, num_seqs, st)
                     : dispatch_group<8, false>(group, p, num_seqs, st);
    return fused ? dispatch_group<16, true>(group, p, num_seqs, st)
                 : dispatch_group<16, false>(group, p, num_seqs, st);
}

// The split launch; with more than kFusedMergeMaxSplits splits, then a merge launch over
// (sequence, query head).
int run_split_kv(int group, DecodeParams &p, int num_seqs, cudaStream_t st)
{
    p.merge_in_kernel = p.max_splits <= kFusedMergeMaxSplits ? 1 : 0;
    const int rc = dispatch(group, p, num_seqs, st);
    if (rc != NV_OK || p.merge_in_kernel)
        return rc;
    merge_splits_kernel<<<dim3(num_seqs, p.num_q_heads), 128, 0, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

// Decode with this many query heads per kv head or more runs on the tcgen05 tile kernel (as a
// prefill of one query row per sequence): the CUDA-core kernel's warps do G times the FMAs per KV
// byte and stop keeping up with HBM at G = 8 (measured 0.54 of the HBM roofline there, against
// about 1.0 for the tile kernel on the same batch).  Its work list sits after the split counters.
constexpr int kTileGroup = 8;

// Which kernel decodes a batch.  G >= 8: the tile kernel (above).  G = 1, 2: the split-KV kernel
// except for a few long contexts (below).  G = 4: the split-KV kernel for
// batches whose grid spans at least ten waves of the GPU (two CTAs per SM), and for batches of at
// most 16 sequences with short contexts; the tile kernel otherwise.  Measured at G = 4 (32 q / 8 kv heads, contexts
// U[1024, 4096]): the split-KV grid of a mid-sized batch ends in a partly filled last wave and
// pays each CTA's start (barriers, a pipeline refilled from HBM) per (sequence, split): 64
// sequences 149.5 us (4.3 TB/s) against 109.2 us (5.9 TB/s) on the tile kernel, whose persistent
// CTAs claim (sequence, kv head) units and split long keys into ranges; 256 sequences 437 against
// 392 us; and when most of the KV is shared and sits in L2 (64 sequences sharing 3072 of their
// 4096 positions) the split-KV consumers are bound by their own FMAs: 172 against 123 us.  The
// headline-sized batch (512 sequences, 13 waves) is HBM-bound on CUDA cores at 0.98 of the copy
// peak and stays there.  G = 1, 2 always use the split-KV kernel (G = 2, 256 sequences: 180 against
// 189 us).  Group 4, 16 sequences or fewer: the split-KV kernel is the faster one on short contexts
// (51 against 56 us at 8 of U[1024, 4096]), the tile kernel once num_seqs x max_context_len reaches 32768 keys
// (one 32K-token sequence 50 against 64 us on the split-KV kernel, one of 128K 97 against 170 us,
// four of 32K 96 against 119 us); below that the batch is a few tens of MB, latency-bound on either
// kernel, and the split-KV launch is 2-4 us quicker.  Groups 1 and 2, whose CUDA-core consumers have
// less arithmetic per byte: the tile kernel for at most 8 sequences holding 32768 keys or more (GPU
// time in a CUDA graph at group 2, split-KV against tiles: two of 16K 41.2 / 33.2 us, four of 8K
// 36.5 / 32.4, eight of 8K 60.1 / 53.1, eight of 16K 97.0 / 90.8, one of 32K 54.6 / 35.5, one of 128K
// 164 / 97); from 12 sequences the split-KV kernel is as fast or faster (twelve of 16K 125.9 / 134.8).
constexpr int64_t kTileMinKeysSmallBatch = 32768;

bool decode_on_tiles_rule(int group, int num_seqs, int max_context_len)
{
    if (group >= kTileGroup)
        return true;
    if (group < 4)
        return num_seqs <= 8 && (int64_t)num_seqs * max_context_len >= kTileMinKeysSmallBatch;
    if (num_seqs <= 16)
        return (int64_t)num_seqs * max_context_len >= kTileMinKeysSmallBatch;
    const int split = decode_split_tokens(num_seqs, max_context_len);
    const int64_t units = (int64_t)num_seqs * ((max_context_len + split - 1) / split);
    const int sms = nvkv_host::sm_count();
    return sms > 0 && units < 10 * 2 * (int64_t)sms;
}

// The tile kernel's own limits (its work list packs sequence ids and pool slots in 16 and 31 bits),
// checked before the workspace so the refusal does not depend on it.
bool tile_shape_ok(int32_t num_seqs, int32_t num_blocks, int32_t block_size)
{
    return num_seqs <= 65535 && (int64_t)num_blocks * block_size < (1ll << 31);
}

size_t tile_list_bytes(int32_t num_seqs)
{
    return nvkv_host::tile_workspace_bytes(num_seqs, num_seqs, 1, kTileGroup);
}

}  // namespace

// 256 KiB of split counters, then the partials of the split-KV kernel's splits, then room for the
// tile kernel's work list at that many entries per sequence.  The tile kernel splits a sequence
// only into ranges of at least 1024 keys, never shorter than the split-KV kernel's, so its
// partials and list fit the same space.
extern "C" size_t nv_paged_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                                 int32_t max_context_len)
{
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim != kD || max_context_len <= 0)
        return 0;
    const int split = decode_split_tokens(num_seqs, max_context_len);
    const int max_splits = (max_context_len + split - 1) / split;
    const size_t part = max_splits <= 1 ? 0 : (size_t)num_seqs * max_splits * num_q_heads * (kD + 2) * sizeof(float);
    return kCounterBytes + part + tile_list_bytes((int32_t)((int64_t)num_seqs * (max_splits > 1 ? max_splits : 1)));
}

namespace {

// Decode as a tile-kernel prefill of one query row per sequence (sequence b's query is row b, at
// position L-1): the pre-pass lists one query tile per sequence with keys and zeroes the rows of
// sequences without.
//
// The tile kernel takes a (sequence, kv head) unit's keys in one CTA, so a batch with fewer than two
// units per SM (a few long contexts) is split into key ranges: enough splits for about three units
// per SM, each at least 8 key steps (1024 keys) long.  Splits write fp32 partials, and
// merge_splits_kernel combines them as it does the split-KV kernel's.
constexpr int kTileMinSplitSteps = 8;

int tile_split_steps(int num_seqs, int num_kv_heads, int max_len)
{
    const int64_t units = (int64_t)num_seqs * num_kv_heads;
    const int sms = nvkv_host::sm_count();
    const int steps = (max_len + 127) / 128;
    if (sms <= 0 || units >= 2 * (int64_t)sms || steps <= kTileMinSplitSteps)
        return 0;
    const int64_t want = (3 * (int64_t)sms + units - 1) / units;     // splits per sequence
    int s = (int)((steps + want - 1) / want);
    if (s < kTileMinSplitSteps)
        s = kTileMinSplitSteps;
    return s >= steps ? 0 : s;
}

int decode_on_tiles(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
                    int32_t bt_stride, const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t block_size, int32_t num_blocks, int32_t max_len, float scale,
                    void *scratch, size_t scratch_bytes, int32_t *d_err, cudaStream_t stream, void *out)
{
    // scratch: [partials O][partials (max, sum)][work list]; the split grows until they fit
    int split_steps = tile_split_steps(num_seqs, num_kv_heads, max_len);
    int max_splits = 0;
    size_t part_bytes = 0;
    while (split_steps > 0) {
        max_splits = (((max_len + 127) / 128) + split_steps - 1) / split_steps;
        part_bytes = ((size_t)num_seqs * max_splits * num_q_heads * (kD + 2) * sizeof(float) + 15) & ~(size_t)15;
        if (part_bytes + tile_list_bytes((int32_t)((int64_t)num_seqs * max_splits)) <= scratch_bytes)
            break;
        split_steps *= 2;
        if (split_steps * 128 >= max_len)
            split_steps = 0;
    }
    if (split_steps == 0) {
        max_splits = 0;
        part_bytes = 0;
    }
    float *part_o = static_cast<float *>(scratch);
    float *part_ml = part_o + (size_t)num_seqs * max_splits * num_q_heads * kD;
    nvkv_host::TileAttnArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.context_lens = context_lens;
    a.block_tables = block_tables;
    a.bt_stride = bt_stride;
    a.num_seqs = num_seqs;
    a.total_q = num_seqs;
    a.max_seqlen_q = 1;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.max_len = max_len;
    a.split_steps = split_steps;
    a.max_splits = max_splits;
    a.part_o = split_steps ? part_o : nullptr;
    a.part_ml = split_steps ? part_ml : nullptr;
    a.scale = scale;
    a.out = out;
    a.workspace = static_cast<uint8_t *>(scratch) + part_bytes;
    a.workspace_bytes = scratch_bytes - part_bytes;
    a.d_err = d_err;
    a.stream = stream;
    const int rc = nvkv_host::tile_attention(a);
    if (rc != NV_OK || split_steps == 0)
        return rc;
    DecodeParams mp{};
    mp.context_lens = context_lens;
    mp.out = static_cast<__nv_bfloat16 *>(out);
    mp.part_o = part_o;
    mp.part_ml = part_ml;
    mp.num_q_heads = num_q_heads;
    mp.max_len = max_len;
    mp.split_tokens = split_steps * 128;
    mp.max_splits = max_splits;
    merge_splits_kernel<<<dim3(num_seqs, num_q_heads), 128, 0, stream>>>(mp);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

struct StoreArgs {     // the new rows of a fused store + decode (absent for a plain decode)
    const void *k;
    int64_t k_row_stride;
    const void *v;
    int64_t v_row_stride;
    const int32_t *slot_mapping;
};

int decode_entry(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
                 int32_t bt_stride, const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                 int32_t max_context_len, float scale, void *out, void *workspace, size_t workspace_bytes,
                 int32_t *d_err, nv_stream_t stream, const StoreArgs *st)
{
    using namespace nvkv_host;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || bt_stride <= 0 || num_blocks < 0 ||
        max_context_len < 0)
        return NV_ERR_SHAPE;
    if (num_seqs == 0)
        return NV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return NV_ERR_NULL;
    if (head_dim != kD)
        return NV_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0)
        return NV_ERR_SHAPE;
    const int group = num_q_heads / num_kv_heads;
    if (num_kv_heads > 16 || !(group == 1 || group == 2 || group == 4 || group == 8 || group == 16))
        return NV_ERR_UNSUPPORTED;
    if (!is_pow2(block_size) || block_size < 16 || block_size > 256)
        return NV_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return NV_ERR_ALIGN;
    if ((int64_t)num_blocks * block_size * num_kv_heads * kD >= (1ll << 40))
        return NV_ERR_UNSUPPORTED;
    if (max_context_len == 0)
        max_context_len = 1;   // every row is padding; one split writes the zeros
    const int64_t bt_cap = (int64_t)bt_stride * block_size;
    const int max_len = (int)(bt_cap < max_context_len ? bt_cap : max_context_len);

    DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_cache = static_cast<const __nv_bfloat16 *>(k_cache);
    p.v_cache = static_cast<const __nv_bfloat16 *>(v_cache);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.d_err = d_err;
    p.bt_stride = bt_stride;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_shift = ilog2(block_size);
    p.num_blocks = num_blocks;
    p.max_len = max_len;
    p.split_tokens = decode_split_tokens(num_seqs, max_context_len);
    p.max_splits = (max_len + p.split_tokens - 1) / p.split_tokens;
    p.scale_log2 = scale * nvkv::kLog2e;
    if (st) {
        const int64_t dkv = (int64_t)num_kv_heads * kD;
        if (!st->k || !st->v || !st->slot_mapping)
            return NV_ERR_NULL;
        if (st->k_row_stride < dkv || st->v_row_stride < dkv)
            return NV_ERR_SHAPE;
        if (st->k_row_stride % 8 != 0 || st->v_row_stride % 8 != 0 || !aligned16(st->k) || !aligned16(st->v))
            return NV_ERR_ALIGN;
        p.k_new = static_cast<const __nv_bfloat16 *>(st->k);
        p.v_new = static_cast<const __nv_bfloat16 *>(st->v);
        p.k_new_stride = st->k_row_stride;
        p.v_new_stride = st->v_row_stride;
        p.slot_mapping = st->slot_mapping;
        p.k_cache_w = static_cast<__nv_bfloat16 *>(const_cast<void *>(k_cache));
        p.v_cache_w = static_cast<__nv_bfloat16 *>(const_cast<void *>(v_cache));
        p.num_slots = (int64_t)num_blocks * block_size;
    }
    if (decode_on_tiles_rule(group, num_seqs, max_context_len)) {
        if (!tile_shape_ok(num_seqs, num_blocks, block_size))
            return NV_ERR_UNSUPPORTED;
        if (!workspace || workspace_bytes < kCounterBytes + tile_list_bytes(num_seqs) || !aligned16(workspace))
            return NV_ERR_WORKSPACE;
        if (st) {       // the store first, by the fused kernel's rule; then the decode reads the pool
            decode_store_kernel<<<(num_seqs + 7) / 8, 256, 0, (cudaStream_t)stream>>>(p, num_seqs);
            if (cudaGetLastError() != cudaSuccess)
                return NV_ERR_CUDA;
        }
        return decode_on_tiles(q, k_cache, v_cache, block_tables, bt_stride, context_lens, num_seqs, num_q_heads,
                               num_kv_heads, block_size, num_blocks, max_len, scale,
                               static_cast<uint8_t *>(workspace) + kCounterBytes, workspace_bytes - kCounterBytes,
                               d_err, (cudaStream_t)stream, out);
    }
    if (p.max_splits > 1) {
        const size_t need = nv_paged_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len);
        if (!workspace || workspace_bytes < need || !aligned16(workspace))
            return NV_ERR_WORKSPACE;
        if (num_seqs > kMaxCountedSeqs)
            return NV_ERR_UNSUPPORTED;
        p.split_done = static_cast<int32_t *>(workspace);
        p.part_o = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kCounterBytes);
        p.part_ml = p.part_o + (size_t)num_seqs * p.max_splits * num_q_heads * kD;
    }
    return run_split_kv(group, p, num_seqs, (cudaStream_t)stream);
}

}  // namespace

extern "C" int nv_paged_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_tables, int32_t bt_stride, const int32_t *context_lens,
                                    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t block_size, int32_t num_blocks, int32_t max_context_len, float scale,
                                    void *out, void *workspace, size_t workspace_bytes, int32_t *d_err,
                                    nv_stream_t stream)
{
    return decode_entry(q, k_cache, v_cache, block_tables, bt_stride, context_lens, num_seqs, num_q_heads,
                        num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, out, workspace,
                        workspace_bytes, d_err, stream, nullptr);
}

extern "C" int nv_store_decode_attn(const void *q, const void *k, int64_t k_row_stride, const void *v,
                                    int64_t v_row_stride, const int32_t *slot_mapping, void *k_cache, void *v_cache,
                                    const int32_t *block_tables, int32_t bt_stride, const int32_t *context_lens,
                                    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t block_size, int32_t num_blocks, int32_t max_context_len, float scale,
                                    void *out, void *workspace, size_t workspace_bytes, int32_t *d_err,
                                    nv_stream_t stream)
{
    const StoreArgs st{k, k_row_stride, v, v_row_stride, slot_mapping};
    return decode_entry(q, k_cache, v_cache, block_tables, bt_stride, context_lens, num_seqs, num_q_heads,
                        num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, out, workspace,
                        workspace_bytes, d_err, stream, &st);
}

// ---------------------------------------------------------------------------------------
// Allocation-free decode.
//
// Some callers cannot allocate device memory at the point where they run decode: an engine
// whose KV pool was sized to take all the memory its allocator may use, a host application
// that only lends the library its tensors (the library sees raw pointers and has no
// allocator of its own), or C code with no CUDA allocator at hand.  For them the split-KV
// partials live in a fixed array below, which every GPU that loads this library holds until
// the process exits.
// ---------------------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_decode_scratch[NV_DECODE_STATIC_SCRATCH_BYTES];
// split counters of the allocation-free path: zero at load, and every call leaves them zero
static __device__ int32_t g_decode_split_done[kMaxCountedSeqs];

namespace {

// Device addresses of g_decode_scratch and g_decode_split_done on the current device.  Looked
// up once per device (the host-side names are only stand-ins for the device arrays, never
// addresses to pass a kernel).
bool static_arrays(void **scratch, int32_t **split_done)
{
    static std::mutex mu;
    static void *addr[64][2];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev][0] || !addr[dev][1]) {
        void *a = nullptr, *c = nullptr;
        if (cudaGetSymbolAddress(&a, g_decode_scratch) != cudaSuccess || !a ||
            cudaGetSymbolAddress(&c, g_decode_split_done) != cudaSuccess || !c)
            return false;
        addr[dev][0] = a;
        addr[dev][1] = c;
    }
    *scratch = addr[dev][0];
    *split_done = static_cast<int32_t *>(addr[dev][1]);
    return true;
}

}  // namespace

extern "C" int nv_paged_decode_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                            const int32_t *block_tables, int32_t bt_stride,
                                            const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                            int32_t num_blocks, int32_t max_context_len, float scale, void *out,
                                            int32_t *d_err, nv_stream_t stream)
{
    using namespace nvkv_host;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || bt_stride <= 0 || num_blocks < 0 ||
        max_context_len < 0)
        return NV_ERR_SHAPE;
    if (num_seqs == 0)
        return NV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return NV_ERR_NULL;
    if (head_dim != kD)
        return NV_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0)
        return NV_ERR_SHAPE;
    const int group = num_q_heads / num_kv_heads;
    if (num_kv_heads > 16 || !(group == 1 || group == 2 || group == 4 || group == 8 || group == 16))
        return NV_ERR_UNSUPPORTED;
    if (!is_pow2(block_size) || block_size < 16 || block_size > 256)
        return NV_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return NV_ERR_ALIGN;
    if ((int64_t)num_blocks * block_size * num_kv_heads * kD >= (1ll << 40))
        return NV_ERR_UNSUPPORTED;
    if (max_context_len == 0)
        max_context_len = 1;
    const int64_t bt_cap = (int64_t)bt_stride * block_size;
    const int max_len = (int)(bt_cap < max_context_len ? bt_cap : max_context_len);
    if (decode_on_tiles_rule(group, num_seqs, max_context_len)) {   // the work list goes in the static array
        if (!tile_shape_ok(num_seqs, num_blocks, block_size))
            return NV_ERR_UNSUPPORTED;
        void *scratch = nullptr;
        int32_t *counters = nullptr;
        if (!static_arrays(&scratch, &counters))
            return NV_ERR_CUDA;
        return decode_on_tiles(q, k_cache, v_cache, block_tables, bt_stride, context_lens, num_seqs, num_q_heads,
                               num_kv_heads, block_size, num_blocks, max_len, scale, scratch,
                               (size_t)NV_DECODE_STATIC_SCRATCH_BYTES, d_err, (cudaStream_t)stream, out);
    }

    // The usual split length, doubled until the partials fit in the static array.
    int split = decode_split_tokens(num_seqs, max_context_len);
    auto need = [&](int sp) {
        const int splits = (max_len + sp - 1) / sp;
        return splits <= 1 ? (size_t)0 : (size_t)num_seqs * splits * num_q_heads * (kD + 2) * sizeof(float);
    };
    while (need(split) > (size_t)NV_DECODE_STATIC_SCRATCH_BYTES && split < 4096)
        split *= 2;
    if (need(split) > (size_t)NV_DECODE_STATIC_SCRATCH_BYTES)
        return NV_ERR_WORKSPACE;   // partials of this batch exceed the static array

    DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_cache = static_cast<const __nv_bfloat16 *>(k_cache);
    p.v_cache = static_cast<const __nv_bfloat16 *>(v_cache);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.d_err = d_err;
    p.bt_stride = bt_stride;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_shift = ilog2(block_size);
    p.num_blocks = num_blocks;
    p.max_len = max_len;
    p.split_tokens = split;
    p.max_splits = (max_len + split - 1) / split;
    p.scale_log2 = scale * nvkv::kLog2e;
    if (p.max_splits > 1) {
        if (num_seqs > kMaxCountedSeqs)
            return NV_ERR_UNSUPPORTED;
        void *scratch = nullptr;
        if (!static_arrays(&scratch, &p.split_done))
            return NV_ERR_CUDA;
        // Every partial the merge reads is written earlier in the same call, so nothing in the
        // scratch array has to start at zero; the counters are zero between calls.
        p.part_o = static_cast<float *>(scratch);
        p.part_ml = p.part_o + (size_t)num_seqs * p.max_splits * num_q_heads * kD;
    }
    return run_split_kv(group, p, num_seqs, (cudaStream_t)stream);
}
