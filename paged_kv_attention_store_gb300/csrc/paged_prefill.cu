// nv_paged_prefill_attn: varlen causal prefill over a paged prefix + new chunk, on tcgen05.
//
// What it computes is the prefill branch of the nano-vLLM field guide's Step 10.3 (with the
// packing of Step 07.5): sequence b owns packed query rows cu_q[b]..cu_q[b+1]-1 (Lq of them)
// and Lk = cu_k[b+1]-cu_k[b] keys read through its block table; the first P = Lk-Lq were
// cached before.  Query i of the chunk sees keys 0..P+i (bottom-right causal alignment).
//
// How (GB300 design; the pages call a library kernel here).  One CTA computes one 128-row
// tile of one (sequence, kv head): with G = Hq/Hkv query heads per kv head, the tile packs
// 128/G consecutive query tokens x G heads, so every K/V tile it loads serves all G heads.
//   * warp 4 (TMA producer): K and V tiles of 128 keys x 128 dims come straight from the
//     paged pool with 3-D tensor-map copies (dims: head_dim, kv head, slot) in 128-byte
//     swizzled layout -- one box per block piece, so a 128-key tile costs one table lookup
//     when block_size >= 128.  Two stages of K+V are in flight.
//   * warp 5 (MMA issuer; also owns the tensor-memory allocation): one elected lane issues
//     tcgen05.mma kind::f16 (bf16 operands from shared memory, fp32 accumulation in TMEM):
//     S = Q K^T into one of two TMEM S buffers, then O += P V into the TMEM O accumulator.
//     S(n+1) is issued before PV(n) so the tensor core works while softmax runs.
//   * warps 0-3 (softmax / correction / epilogue): thread r owns tile row r = TMEM lane r.
//     It reads its S row with tcgen05.ld, applies the causal mask only on tiles that cross
//     the diagonal, keeps an online softmax in base 2 with a lazy rescale (the running max
//     moves only when a score beats it by more than 8), writes P as bf16 into shared
//     memory in the MMA's swizzled K-major layout, and -- rarely -- rescales its O row in
//     TMEM.  At the end it normalises O and writes bf16 rows.
// Every mbarrier wait is bounded; on timeout the kernel records NV_DERR_TIMEOUT and stops.
#include <cuda.h>

#include <mutex>

#include "nv_common.cuh"

namespace {

using namespace nvkv;

constexpr int kD = 128;
constexpr int kBM = 128;            // tile rows (TMEM lanes)
constexpr int kBN = 128;            // keys per KV tile
constexpr int kStages = 2;          // K+V stages
constexpr int kThreads = 192;       // warps 0-3 softmax, 4 producer, 5 MMA
constexpr uint32_t kTmemCols = 512; // S0 [0,128), S1 [128,256), O [256,384)
constexpr float kRescaleLog2 = 8.0f;

constexpr uint32_t kHalfTile = kBM * 128;          // 128 rows x 128 bytes (64 bf16) = 16 KB
constexpr uint32_t kTileBytes = 2 * kHalfTile;     // a 128 x 128 bf16 operand tile = 32 KB
// shared memory layout (offsets from a 1024-aligned base)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kTileBytes;                    // stage s: K at +0, V at +kTileBytes
constexpr uint32_t kOffP = kOffKV + kStages * 2 * kTileBytes;
constexpr uint32_t kOffBar = kOffP + kTileBytes;
constexpr uint32_t kNumBars = 1 + 3 * kStages + 2 + 2 + 1 + 1;
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffTmemSlot + 16 + 1024;          // + slack for 1024 alignment

// barrier indices
constexpr int kBarQ = 0;
constexpr int kBarKFull = 1;                       // + stage
constexpr int kBarVFull = kBarKFull + kStages;     // + stage
constexpr int kBarKVEmpty = kBarVFull + kStages;   // + stage
constexpr int kBarSFull = kBarKVEmpty + kStages;   // + (n & 1)
constexpr int kBarSFree = kBarSFull + 2;           // + (n & 1)
constexpr int kBarPFull = kBarSFree + 2;
constexpr int kBarODone = kBarPFull + 1;

struct PrefillParams {
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *block_tables;
    int32_t *d_err;
    int32_t bt_stride;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t group;          // G
    int32_t group_shift;    // log2 G
    int32_t block_shift;    // log2 block_size
    int32_t box_rows;       // min(block_size, 128)
    int32_t num_blocks;
    int32_t max_tiles;      // gridDim.x
    float scale_log2;
};

// Offset of the 16-byte chunk `chunk` (0..7) of row `row` inside a 128-byte-swizzled
// [rows x 128 B] half tile: the chunk index is XOR-ed with the row's position in its 8-row group.
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                         const PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;     // SW128 tiles need 1024-byte alignment
    uint8_t *smem = smem_raw + (base - raw_base);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.z;
    const int kvh = blockIdx.y;

    // ---------------- per-tile geometry (uniform over the CTA) ----------------
    const int cq0 = __ldg(p.cu_q + b), cq1 = __ldg(p.cu_q + b + 1);
    const int ck0 = __ldg(p.cu_k + b), ck1 = __ldg(p.cu_k + b + 1);
    const int Lq = cq1 - cq0, Lk = ck1 - ck0;
    const int P = Lk - Lq;
    const int tq = kBM >> p.group_shift;                  // query tokens per tile
    if (Lq < 0 || P < 0 || ((Lk + (1 << p.block_shift) - 1) >> p.block_shift) > p.bt_stride) {
        if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0)
            flag_error(p.d_err, NV_DERR_LENGTH);
        return;
    }
    const int ntiles = (Lq + tq - 1) / tq;
    if (ntiles > p.max_tiles && blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0)
        flag_error(p.d_err, NV_DERR_LENGTH);
    const int tile = p.max_tiles - 1 - (int)blockIdx.x;  // heaviest tiles are dispatched first
    if (tile >= ntiles)
        return;
    const int i0 = tile * tq;
    const int nq = min(tq, Lq - i0);
    const int kv_len = P + i0 + nq;                        // keys any row of this tile can see
    const int nkv = (kv_len + kBN - 1) / kBN;
    const int first_masked = (P + i0 + 1) / kBN;           // tiles before this one need no mask

    const uint32_t bar = base + kOffBar;
    auto BAR = [&](int i) { return bar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmemSlot);

    if (threadIdx.x == 0) {
        mbar_init(BAR(kBarQ), 4);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(BAR(kBarKFull + s), 1);
            mbar_init(BAR(kBarVFull + s), 1);
            mbar_init(BAR(kBarKVEmpty + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(kBarSFull + s), 1);
            mbar_init(BAR(kBarSFree + s), 4);
        }
        mbar_init(BAR(kBarPFull), 4);
        mbar_init(BAR(kBarODone), 1);
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_o = tmem + 256;

    if (warp == 4) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            const int32_t *bt = p.block_tables + (size_t)b * p.bt_stride;
            const int bs_mask = (1 << p.block_shift) - 1;
            const int boxes = kBN / p.box_rows;
            for (int n = 0; n < nkv; ++n) {
                const int st = n % kStages;
                if (n >= kStages && !mbar_wait(BAR(kBarKVEmpty + st), ((n / kStages) - 1) & 1)) {
                    flag_error(p.d_err, NV_DERR_TIMEOUT);
                    break;
                }
                int slot0[kBN / 16];
                int nbox = 0;
                for (int k = 0; k < boxes; ++k) {
                    const int j0 = n * kBN + k * p.box_rows;
                    slot0[k] = -1;
                    if (j0 >= kv_len)
                        continue;
                    const int blk = __ldg(bt + (j0 >> p.block_shift));
                    if (blk < 0 || blk >= p.num_blocks) {
                        flag_error(p.d_err, NV_DERR_BLOCK_RANGE);
                        continue;
                    }
                    slot0[k] = (blk << p.block_shift) + (j0 & bs_mask);
                    ++nbox;
                }
                const uint32_t bytes = (uint32_t)nbox * p.box_rows * 128u * 2u;
                const uint32_t kdst = base + kOffKV + st * 2 * kTileBytes;
                const uint32_t vdst = kdst + kTileBytes;
                mbar_arrive_expect_tx(BAR(kBarKFull + st), bytes);
                for (int k = 0; k < boxes; ++k) {
                    if (slot0[k] < 0)
                        continue;
                    const uint32_t roff = (uint32_t)k * p.box_rows * 128u;
                    tma_load_3d(kdst + roff, &tmap_k, 0, kvh, slot0[k], BAR(kBarKFull + st));
                    tma_load_3d(kdst + kHalfTile + roff, &tmap_k, 64, kvh, slot0[k], BAR(kBarKFull + st));
                }
                mbar_arrive_expect_tx(BAR(kBarVFull + st), bytes);
                for (int k = 0; k < boxes; ++k) {
                    if (slot0[k] < 0)
                        continue;
                    const uint32_t roff = (uint32_t)k * p.box_rows * 128u;
                    tma_load_3d(vdst + roff, &tmap_v, 0, kvh, slot0[k], BAR(kBarVFull + st));
                    tma_load_3d(vdst + kHalfTile + roff, &tmap_v, 64, kvh, slot0[k], BAR(kBarVFull + st));
                }
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ============================ MMA issuer ============================
        constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);   // Q, K both K-major
        constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, kD, false, true);     // P K-major, V MN-major
        bool ok = __all_sync(0xffffffffu, mbar_wait(BAR(kBarQ), 0));
        tc_fence_after();
        auto issue_pv = [&](int m) {
            const int st = m % kStages;
            ok = ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarPFull), m & 1));
            ok = ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarVFull + st), (m / kStages) & 1));
            if (!ok)
                return;
            const uint32_t vtile = base + kOffKV + st * 2 * kTileBytes + kTileBytes;
            const int vrows = kv_len - m * kBN;
            if (vrows < kBN) {
                // Keys past the sequence: their P is zero, but their V rows may hold anything
                // (NaN patterns included) and 0 * NaN would poison O -- zero them.
                const int nzero = (kBN - vrows) * 2 * 8;       // 16-byte chunks over both halves
                for (int i = lane; i < nzero; i += 32) {
                    const int half = i / ((kBN - vrows) * 8);
                    const int rem = i % ((kBN - vrows) * 8);
                    const uint32_t row = vrows + rem / 8;
                    sts_u4(vtile + half * kHalfTile + row * 128u + (uint32_t)(rem % 8) * 16u, make_uint4(0, 0, 0, 0));
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t ptile = base + kOffP;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(ptile + (kk >> 2) * kHalfTile + (kk & 3) * 32, 16, 1024);
                    const uint64_t bdesc = smem_desc_sw128(vtile + kk * 16 * 128, kHalfTile, 1024);
                    mma_bf16_ss(tmem_o, a, bdesc, idesc_o, (m > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(BAR(kBarODone));
                mma_commit(BAR(kBarKVEmpty + st));
            }
            __syncwarp();
        };
        for (int n = 0; n < nkv && ok; ++n) {
            const int st = n % kStages;
            if (n >= 2)
                ok = ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarSFree + (n & 1)), ((n >> 1) - 1) & 1));
            ok = ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarKFull + st), (n / kStages) & 1));
            if (!ok)
                break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t qtile = base + kOffQ;
                const uint32_t ktile = base + kOffKV + st * 2 * kTileBytes;
                const uint32_t s_tmem = tmem + (uint32_t)(n & 1) * kBN;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalfTile + (kk & 3) * 32;
                    mma_bf16_ss(s_tmem, smem_desc_sw128(qtile + off, 16, 1024), smem_desc_sw128(ktile + off, 16, 1024),
                                idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(BAR(kBarSFull + (n & 1)));
            }
            __syncwarp();
            if (n >= 1)
                issue_pv(n - 1);
        }
        if (ok && nkv >= 1)
            issue_pv(nkv - 1);
        if (!ok && lane == 0)
            flag_error(p.d_err, NV_DERR_TIMEOUT);
    } else {
        // ================= softmax / correction / epilogue (warps 0-3) =================
        const int r = threadIdx.x;                    // tile row == TMEM lane
        const int tok = i0 + (r >> p.group_shift);    // token index inside the chunk
        const int head = kvh * p.group + (r & (p.group - 1));
        const bool valid = tok < Lq;
        const int lim = P + tok;                      // last key this row may see

        // ---- stage the Q tile (row r), 128-byte swizzled, zeros for rows past the chunk ----
        {
            const uint32_t qtile = base + kOffQ;
            const uint4 *src = reinterpret_cast<const uint4 *>(p.q + ((size_t)(cq0 + tok) * p.num_q_heads + head) * kD);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                sts_u4(qtile + (c >> 3) * kHalfTile + sw128(r, c & 7), v);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(BAR(kBarQ));
        }

        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t ptile = base + kOffP;
        float m_run = -INFINITY;   // running max of scale*log2(e)*s over this row
        float l_run = 0.f;
        bool ok = true;
        for (int n = 0; n < nkv; ++n) {
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBarSFull + (n & 1)), (n >> 1) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t s_addr = tmem + lane_base + (uint32_t)(n & 1) * kBN;
            const bool masked = n >= first_masked;
            const int kbase = n * kBN;
            // pass 1: row max of the (masked) raw scores
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(s_addr + c * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float s = __uint_as_float(v[i]);
                    const bool keep = !masked || (kbase + c * 32 + i <= lim);
                    mx = keep ? fmaxf(mx, s) : mx;
                }
            }
            const float mx2 = mx * p.scale_log2;
            const bool need = mx2 > m_run + kRescaleLog2;
            const float m_new = need ? mx2 : m_run;
            const float alpha = need ? fast_exp2(m_run - m_new) : 1.f;
            // P buffer and O are free once PV(n-1) has completed
            if (n >= 1 && !__all_sync(0xffffffffu, mbar_wait(BAR(kBarODone), (n - 1) & 1))) {
                ok = false;
                break;
            }
            // pass 2: p = 2^(s*scale*log2e - m), row sum, bf16 P into shared memory
            float rs = 0.f;
            const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(s_addr + c * 32, v);
                tmem_wait_ld();
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const bool k0 = !masked || (kbase + c * 32 + i <= lim);
                    const bool k1 = !masked || (kbase + c * 32 + i + 1 <= lim);
                    const float p0 = k0 ? fast_exp2(fmaf(__uint_as_float(v[i]), p.scale_log2, neg_m)) : 0.f;
                    const float p1 = k1 ? fast_exp2(fmaf(__uint_as_float(v[i + 1]), p.scale_log2, neg_m)) : 0.f;
                    rs += p0 + p1;
                    packed[i >> 1] = pack_bf16x2(p0, p1);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t chunk = (uint32_t)(c * 4 + k);          // 16-byte chunk of the 128-key row
                    const uint32_t addr = ptile + (chunk >> 3) * kHalfTile + sw128((uint32_t)r, chunk & 7);
                    sts_u4(addr, make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(BAR(kBarSFree + (n & 1)));
            l_run = l_run * alpha + rs;
            m_run = m_new;
            // rare: rescale this row's O accumulator (nothing to rescale before the first PV)
            if (n >= 1 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tmem_o + lane_base + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                    tmem_st32(tmem_o + lane_base + c * 32, v);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(BAR(kBarPFull));
        }
        // ---- epilogue: O / l -> bf16 rows ----
        if (ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarODone), (nkv - 1) & 1))) {
            tc_fence_after();
            const float inv = (valid && l_run > 0.f) ? 1.f / l_run : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((size_t)(cq0 + tok) * p.num_q_heads + head) * kD);
#pragma unroll
            for (int c = 0; c < kD / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem_o + lane_base + c * 32, v);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(v[8 * k + 0]) * inv, __uint_as_float(v[8 * k + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(v[8 * k + 2]) * inv, __uint_as_float(v[8 * k + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(v[8 * k + 4]) * inv, __uint_as_float(v[8 * k + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(v[8 * k + 6]) * inv, __uint_as_float(v[8 * k + 7]) * inv);
                        dst[c * 4 + k] = w;
                    }
                }
            }
        } else if (lane == 0) {
            flag_error(p.d_err, NV_DERR_TIMEOUT);
        }
    }

    // ---------------- teardown: every TMEM read is done before the free ----------------
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Pool [num_slots, Hkv, 128] bf16 seen as a 3-D tensor (dim0 = head_dim, dim1 = kv head,
// dim2 = slot); a box is 64 dims x 1 head x box_rows slots, 128-byte swizzled.
bool make_pool_map(CUtensorMap *map, const void *pool, int64_t num_slots, int num_kv_heads, int box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)num_kv_heads, (cuuint64_t)num_slots};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)num_kv_heads * kD * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int nv_paged_prefill_attn(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                     const int32_t *block_tables, int32_t bt_stride, int32_t num_seqs,
                                     int32_t total_q, int32_t max_seqlen_q, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                     float scale, void *out, int32_t *d_err, nv_stream_t stream)
{
    using namespace nvkv_host;
    if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        bt_stride <= 0 || num_blocks < 0)
        return NV_ERR_SHAPE;
    if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0)
        return NV_OK;
    if (!q || !k_cache || !v_cache || !cu_seqlens_q || !cu_seqlens_k || !block_tables || !out)
        return NV_ERR_NULL;
    if (head_dim != kD)
        return NV_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0)
        return NV_ERR_SHAPE;
    const int group = num_q_heads / num_kv_heads;
    if (!is_pow2(group) || group > 16 || num_kv_heads > 65535)
        return NV_ERR_UNSUPPORTED;
    if (!is_pow2(block_size) || block_size < 16 || block_size > 256)
        return NV_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * block_size >= (1ll << 31) || num_seqs > 65535)
        return NV_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return NV_ERR_ALIGN;
    if (num_blocks == 0)
        return NV_ERR_SHAPE;

    const int box_rows = block_size < kBN ? block_size : kBN;
    CUtensorMap tk, tv;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    if (!make_pool_map(&tk, k_cache, num_slots, num_kv_heads, box_rows) ||
        !make_pool_map(&tv, v_cache, num_slots, num_kv_heads, box_rows))
        return NV_ERR_CUDA;

    PrefillParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.block_tables = block_tables;
    p.d_err = d_err;
    p.bt_stride = bt_stride;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.group_shift = ilog2(group);
    p.block_shift = ilog2(block_size);
    p.box_rows = box_rows;
    p.num_blocks = num_blocks;
    const int tq = kBM / group;
    p.max_tiles = (max_seqlen_q + tq - 1) / tq;
    p.scale_log2 = scale * nvkv::kLog2e;

    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (attr_err != cudaSuccess)
        return NV_ERR_CUDA;
    dim3 grid(p.max_tiles, num_kv_heads, num_seqs);
    paged_prefill_kernel<<<grid, kThreads, kSmemBytes, (cudaStream_t)stream>>>(tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}
