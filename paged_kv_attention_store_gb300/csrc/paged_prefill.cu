// nv_paged_prefill_attn: varlen causal prefill over a paged prefix + new chunk, on tcgen05.
//
// What it computes is the prefill branch of the nano-vLLM field guide's Step 10.3 (with the
// packing of Step 07.5): sequence b owns packed query rows cu_q[b]..cu_q[b+1]-1 (Lq of them)
// and Lk = cu_k[b+1]-cu_k[b] keys read through its block table; the first P = Lk-Lq were
// cached before.  Query i of the chunk sees keys 0..P+i (bottom-right causal alignment).
//
// How (GB300 design; the pages call a library kernel here).  One CTA computes TWO 128-row
// query tiles of one (sequence, kv head).  With G = Hq/Hkv query heads per kv head a tile
// packs 128/G consecutive tokens x G heads, so every K/V tile loaded serves 2*G*(128/G) rows.
//   * warp 8 (TMA producer): both Q tiles with one 3-D tensor-map copy each (dims head_dim,
//     q head, token), then K and V tiles of 64 keys x 128 dims straight from the paged pool
//     (dims head_dim, kv head, slot), 128-byte swizzled, into a 6-slot ring (K0 V0 K1 V1 ...),
//     so loads run up to three key tiles ahead of the tensor core.
//   * warps 9 and 10 (MMA issuers, one per query tile; warp 9 owns the tensor-memory
//     allocation): one lane issues tcgen05.mma kind::f16 -- bf16 operands from shared
//     memory, fp32 accumulators in TMEM.  For its tile i and key tile n it issues
//     S_i(n+1) = Q_i K(n+1)^T into the other half of a double-buffered TMEM S tile BEFORE it
//     waits for P_i(n), then O_i += P_i(n) V(n).  The two tiles' streams interleave on the
//     tensor core, and each warpgroup finds its next S ready when it finishes a softmax.
//   * warps 0-3 / 4-7 (softmax warpgroups, one per query tile): thread r owns row r = TMEM
//     lane r.  It copies its 64 scores to registers with tcgen05.ld and frees the S buffer,
//     masks only on tiles that cross the diagonal, keeps a base-2 online softmax with a lazy
//     rescale (the running max moves only when a score beats it by more than 8, so O is
//     rarely touched), writes P as bf16 into shared memory in the MMA's swizzled K-major
//     layout (double-buffered), and at the end normalises O and stores bf16 rows.  A quarter
//     of the exponentials run as a cubic polynomial on the FMA pipe (see exp2_poly3) so the
//     two warpgroups do not queue on the special-function unit.
// Every mbarrier wait is bounded; on timeout the kernel records NV_DERR_TIMEOUT and stops.
#include <cuda.h>

#include <mutex>

#include "nv_common.cuh"

namespace {

using namespace nvkv;

constexpr int kD = 128;
constexpr int kBM = 128;             // rows per query tile (TMEM lanes)
constexpr int kBN = 64;              // keys per K/V tile
constexpr int kSlots = 6;            // K/V ring slots
constexpr int kThreads = 352;        // warps 0-3, 4-7 softmax; 8 producer; 9, 10 MMA
constexpr uint32_t kTmemCols = 512;  // S[i][b] at i*128 + b*64; O[i] at 256 + i*128
constexpr float kRescaleLog2 = 8.0f;

constexpr uint32_t kQHalf = kBM * 128;        // 128 rows x 64 dims bf16 = 16 KB
constexpr uint32_t kQTile = 2 * kQHalf;       // 32 KB
constexpr uint32_t kKVHalf = kBN * 128;       // 64 keys x 64 dims = 8 KB
constexpr uint32_t kKVTile = 2 * kKVHalf;     // 16 KB
constexpr uint32_t kPTile = kBM * 128;        // 128 rows x 64 keys bf16 = 16 KB

constexpr uint32_t kOffQ = 0;                                   // Q[i] at i*kQTile
constexpr uint32_t kOffP = kOffQ + 2 * kQTile;                  // P[i][b] at (2i+b)*kPTile
constexpr uint32_t kOffKV = kOffP + 4 * kPTile;                 // slot s at s*kKVTile
constexpr uint32_t kOffBar = kOffKV + kSlots * kKVTile;
// barriers
constexpr int kBarQ = 0;
constexpr int kBarKVFull = 1;                      // + slot
constexpr int kBarKVEmpty = kBarKVFull + kSlots;   // + slot
constexpr int kBarSFull = kBarKVEmpty + kSlots;    // + 2*i + b
constexpr int kBarSFree = kBarSFull + 4;           // + 2*i + b
constexpr int kBarPFull = kBarSFree + 4;           // + 2*i + b
constexpr int kBarODone = kBarPFull + 4;           // + 2*i + b
constexpr int kNumBars = kBarODone + 4;
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffTmemSlot + 16 + 1024;      // + slack for 1024-byte alignment

struct PrefillParams {
    __nv_bfloat16 *out;
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *block_tables;
    int32_t *d_err;
    int32_t bt_stride;
    int32_t num_q_heads;
    int32_t group;          // G
    int32_t group_shift;    // log2 G
    int32_t block_shift;    // log2 block_size
    int32_t box_rows;       // min(block_size, kBN)
    int32_t num_blocks;
    int32_t max_pairs;      // gridDim.z
    float scale_log2;
};

// Offset of 16-byte chunk `chunk` (0..7) of row `row` in a [rows x 128 B] 128-byte-swizzled
// operand: the chunk index is XOR-ed with the row's position inside its 8-row group.
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// 2^x on the FMA pipe, for x <= 8 (scores minus a running max).  Range reduction: adding
// 1.5 * 2^23 rounds x to the nearest integer j, held in the low mantissa bits of the sum;
// f = x - j lies in [-0.5, 0.5] and 2^f comes from a cubic fitted to minimise the relative
// error on that interval (max relative error 7.6e-5, well below the bf16 rounding of P);
// finally j is added into the exponent field.  x is clamped at -126 so masked scores
// (-inf) give a normal number of order 1e-38 instead of a wrapped exponent.
__device__ __forceinline__ float exp2_poly3(float x)
{
    constexpr float kC0 = 0.9999282882344301f, kC1 = 0.6932609081979648f;
    constexpr float kC2 = 0.24260776842531798f, kC3 = 0.05517030853684025f;
    constexpr float kRound = 12582912.0f;
    x = fmaxf(x, -126.0f);
    const float y = __fadd_rn(x, kRound);
    const float j = __fsub_rn(y, kRound);
    const float f = __fsub_rn(x, j);
    float q = fmaf(kC3, f, kC2);
    q = fmaf(q, f, kC1);
    q = fmaf(q, f, kC0);
    return __uint_as_float(__float_as_uint(q) + (__float_as_uint(y) << 23));
}

__device__ __forceinline__ void tmem_ld32x2(uint32_t taddr, uint32_t (&r)[64])
{
    uint32_t (&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
    uint32_t (&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
    tmem_ld32(taddr, a);
    tmem_ld32(taddr + 32, b);
}

__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;     // swizzled tiles need 1024-byte alignment
    uint8_t *smem = smem_raw + (base - raw_base);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kvh = blockIdx.x;
    const int b = blockIdx.y;

    // ---------------- work item geometry (uniform over the CTA) ----------------
    const int cq0 = __ldg(p.cu_q + b), cq1 = __ldg(p.cu_q + b + 1);
    const int ck0 = __ldg(p.cu_k + b), ck1 = __ldg(p.cu_k + b + 1);
    const int Lq = cq1 - cq0, Lk = ck1 - ck0;
    const int P = Lk - Lq;
    if (Lq < 0 || P < 0 || ((Lk + (1 << p.block_shift) - 1) >> p.block_shift) > p.bt_stride) {
        if (blockIdx.z == 0 && kvh == 0 && threadIdx.x == 0)
            flag_error(p.d_err, NV_DERR_LENGTH);
        return;
    }
    const int tq = kBM >> p.group_shift;                   // query tokens per tile
    const int npairs = (Lq + 2 * tq - 1) / (2 * tq);
    if (npairs > p.max_pairs && blockIdx.z == 0 && kvh == 0 && threadIdx.x == 0)
        flag_error(p.d_err, NV_DERR_LENGTH);
    const int pair = p.max_pairs - 1 - (int)blockIdx.z;    // the heaviest pairs are dispatched first
    if (pair >= npairs)
        return;
    int i0[2], nq[2], nkv[2], first_masked[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        i0[i] = pair * 2 * tq + i * tq;
        nq[i] = max(0, min(tq, Lq - i0[i]));
        nkv[i] = nq[i] > 0 ? (P + i0[i] + nq[i] + kBN - 1) / kBN : 0;
        first_masked[i] = (P + i0[i] + 1) / kBN;           // key tiles before this need no mask
    }
    const int kv_len = P + i0[nq[1] > 0 ? 1 : 0] + nq[nq[1] > 0 ? 1 : 0];   // keys any row can see
    const int nkv_all = max(nkv[0], nkv[1]);

    const uint32_t bar = base + kOffBar;
    auto BAR = [&](int i) { return bar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmemSlot);

    if (threadIdx.x == 0) {
        mbar_init(BAR(kBarQ), 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(BAR(kBarKVFull + s), 1);
            mbar_init(BAR(kBarKVEmpty + s), 2);    // one release per query tile's issuer
        }
        for (int s = 0; s < 4; ++s) {
            mbar_init(BAR(kBarSFull + s), 1);
            mbar_init(BAR(kBarSFree + s), 4);
            mbar_init(BAR(kBarPFull + s), 4);
            mbar_init(BAR(kBarODone + s), 1);
        }
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            const uint32_t qbytes = (nq[1] > 0 ? 2u : 1u) * kQTile;
            mbar_arrive_expect_tx(BAR(kBarQ), qbytes);
            for (int i = 0; i < 2; ++i) {
                if (nq[i] == 0)
                    continue;
                for (int h = 0; h < 2; ++h)
                    tma_load_3d(base + kOffQ + i * kQTile + h * kQHalf, &tmap_q, h * 64, kvh * p.group, cq0 + i0[i],
                                BAR(kBarQ));
            }
            const int32_t *bt = p.block_tables + (size_t)b * p.bt_stride;
            const int bs_mask = (1 << p.block_shift) - 1;
            const int boxes = kBN / p.box_rows;
            for (int t = 0; t < 2 * nkv_all; ++t) {
                const int n = t >> 1;
                const int slot = t % kSlots;
                if (t >= kSlots && !mbar_wait(BAR(kBarKVEmpty + slot), ((t / kSlots) - 1) & 1)) {
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
                const CUtensorMap *map = (t & 1) ? &tmap_v : &tmap_k;
                const uint32_t dst = base + kOffKV + slot * kKVTile;
                mbar_arrive_expect_tx(BAR(kBarKVFull + slot), (uint32_t)nbox * p.box_rows * 128u * 2u);
                for (int k = 0; k < boxes; ++k) {
                    if (slot0[k] < 0)
                        continue;
                    const uint32_t roff = (uint32_t)k * p.box_rows * 128u;
                    tma_load_3d(dst + roff, map, 0, kvh, slot0[k], BAR(kBarKVFull + slot));
                    tma_load_3d(dst + kKVHalf + roff, map, 64, kvh, slot0[k], BAR(kBarKVFull + slot));
                }
            }
        }
        __syncwarp();
    } else if (warp >= 9) {
        // ================== MMA issuer for query tile i = warp - 9 ==================
        constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);   // Q, K both K-major
        constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, kD, false, true);     // P K-major, V MN-major
        const int i = warp - 9;
        const int my_nkv = nkv[i];
        const uint32_t qtile = base + kOffQ + i * kQTile;
        const uint32_t o_tmem = tmem + 256 + i * 128;
        bool ok = my_nkv == 0 || __all_sync(0xffffffffu, mbar_wait(BAR(kBarQ), 0));
        auto issue_s = [&](int n) {
            const int t = 2 * n;
            const int slot = t % kSlots;
            const int bb = n & 1;
            ok = ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarKVFull + slot), (t / kSlots) & 1));
            if (n >= 2)
                ok = ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarSFree + 2 * i + bb), ((n - 2) >> 1) & 1));
            if (!ok)
                return;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t ktile = base + kOffKV + slot * kKVTile;
                const uint32_t s_tmem = tmem + i * 128 + bb * 64;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    mma_bf16_ss(s_tmem, smem_desc_sw128(qtile + (kk >> 2) * kQHalf + (kk & 3) * 32, 16, 1024),
                                smem_desc_sw128(ktile + (kk >> 2) * kKVHalf + (kk & 3) * 32, 16, 1024), idesc_s,
                                kk > 0 ? 1u : 0u);
                mma_commit(BAR(kBarSFull + 2 * i + bb));
                mma_commit(BAR(kBarKVEmpty + slot));
            }
            __syncwarp();
        };
        auto issue_pv = [&](int m) {
            const int t = 2 * m + 1;
            const int slot = t % kSlots;
            const int bb = m & 1;
            ok = ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarKVFull + slot), (t / kSlots) & 1));
            if (!ok)
                return;
            const uint32_t vtile = base + kOffKV + slot * kKVTile;
            const int vrows = kv_len - m * kBN;
            if (vrows < kBN) {
                // Keys past the sequence carry P = 0, but their V rows may hold anything (NaN
                // patterns included) and 0 * NaN would poison O: zero them.  Both issuers may
                // do this for the last tile; they write the same zeros.
                const int per_half = (kBN - vrows) * 8;        // 16-byte chunks
                for (int c = lane; c < 2 * per_half; c += 32) {
                    const int half = c / per_half;
                    const int rem = c % per_half;
                    sts_u4(vtile + half * kKVHalf + (uint32_t)(vrows + rem / 8) * 128u + (uint32_t)(rem % 8) * 16u,
                           make_uint4(0, 0, 0, 0));
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            ok = ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarPFull + 2 * i + bb), (m >> 1) & 1));
            if (!ok)
                return;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t ptile = base + kOffP + (2 * i + bb) * kPTile;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_bf16_ss(o_tmem, smem_desc_sw128(ptile + kk * 32, 16, 1024),
                                smem_desc_sw128(vtile + kk * 16 * 128, kKVHalf, 1024), idesc_o,
                                (m > 0 || kk > 0) ? 1u : 0u);
                mma_commit(BAR(kBarODone + 2 * i + bb));
                mma_commit(BAR(kBarKVEmpty + slot));
            }
            __syncwarp();
        };
        if (my_nkv > 0)
            issue_s(0);
        for (int n = 0; n < my_nkv && ok; ++n) {
            if (n + 1 < my_nkv)
                issue_s(n + 1);      // the next scores are computed while this tile's softmax runs
            issue_pv(n);
        }
        // Key tiles this query tile never needs still count toward their slot's release: wait
        // until the tile is loaded (so the arrival lands in the right phase), then arrive.
        for (int t = 2 * my_nkv; t < 2 * nkv_all && ok; ++t) {
            const int slot = t % kSlots;
            ok = __all_sync(0xffffffffu, mbar_wait(BAR(kBarKVFull + slot), (t / kSlots) & 1));
            if (ok && lane == 0)
                mbar_arrive(BAR(kBarKVEmpty + slot));
            __syncwarp();
        }
        if (!ok && lane == 0)
            flag_error(p.d_err, NV_DERR_TIMEOUT);
    } else {
        // ============ softmax / correction / epilogue: warpgroup i owns query tile i ============
        const int i = warp >> 2;
        const int r = threadIdx.x & 127;                // tile row == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_col = tmem + lane_base + i * 128;
        const uint32_t o_addr = tmem + lane_base + 256 + i * 128;
        const int tok = i0[i] + (r >> p.group_shift);   // token index inside the chunk
        const int head = (int)kvh * p.group + (r & (p.group - 1));
        const bool valid = tok < Lq;
        const int lim = P + tok;                        // last key this row may see
        float m_run = -INFINITY;                        // running max of scale*log2(e)*s
        float l_run = 0.f;
        bool ok = true;
        const int n_end = nkv[i];
        for (int n = 0; n < n_end && ok; ++n) {
            const int bb = n & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBarSFull + 2 * i + bb), (n >> 1) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[64];
            tmem_ld32x2(s_col + bb * 64, sv);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(BAR(kBarSFree + 2 * i + bb));
            float s[64];
#pragma unroll
            for (int j = 0; j < 64; ++j)
                s[j] = __uint_as_float(sv[j]);
            if (n >= first_masked[i]) {
                const int rel = lim - n * kBN;          // keys j <= rel are visible
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    s[j] = (j <= rel) ? s[j] : -INFINITY;
            }
            // row max: a tree, so the compare chain is 6 deep instead of 64
            float mx8[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                mx8[j] = fmaxf(fmaxf(fmaxf(s[j], s[j + 8]), fmaxf(s[j + 16], s[j + 24])),
                               fmaxf(fmaxf(s[j + 32], s[j + 40]), fmaxf(s[j + 48], s[j + 56])));
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float mx2 = mx * p.scale_log2;
            const bool need = mx2 > m_run + kRescaleLog2;
            const float m_new = need ? mx2 : m_run;
            const float alpha = need ? fast_exp2(m_run - m_new) : 1.f;   // m_run = -inf -> 0
            const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
            uint32_t pk[32];
            float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
                // every fourth pair on the FMA pipe, the rest on the special-function unit
                const bool poly = ((j >> 1) & 3) == 3;
                const float x0 = fmaf(s[j], p.scale_log2, neg_m);
                const float x1 = fmaf(s[j + 1], p.scale_log2, neg_m);
                const float p0 = poly ? exp2_poly3(x0) : fast_exp2(x0);
                const float p1 = poly ? exp2_poly3(x1) : fast_exp2(x1);
                rs8[(j >> 1) & 7] += p0 + p1;
                pk[j >> 1] = pack_bf16x2(p0, p1);
            }
            const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
            l_run = l_run * alpha + rs;
            m_run = m_new;
            // P buffer bb is free once PV_i(n-2) has completed
            if (n >= 2 && !__all_sync(0xffffffffu, mbar_wait(BAR(kBarODone + 2 * i + bb), ((n - 2) >> 1) & 1))) {
                ok = false;
                break;
            }
            const uint32_t ptile = base + kOffP + (2 * i + bb) * kPTile;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                sts_u4(ptile + sw128((uint32_t)r, (uint32_t)c),
                       make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
            // rare: rescale this row's O (PV_i(n-1) must be complete first; nothing to do at n = 0)
            if (n >= 1 && __any_sync(0xffffffffu, need)) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(BAR(kBarODone + 2 * i + ((n - 1) & 1)), ((n - 1) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(o_addr + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
                    tmem_st32(o_addr + c * 32, v);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(BAR(kBarPFull + 2 * i + bb));
        }
        // ---- epilogue: O / l -> bf16 rows ----
        if (n_end > 0) {
            const int last = n_end - 1;
            if (ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarODone + 2 * i + (last & 1)), (last >> 1) & 1))) {
                tc_fence_after();
                const float inv = (valid && l_run > 0.f) ? 1.f / l_run : 0.f;
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((size_t)(cq0 + tok) * p.num_q_heads + head) * kD);
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(o_addr + c * 32, v);
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
    }

    // ---------------- teardown: every TMEM access is done before the free ----------------
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
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

// A [rows, heads, 128] bf16 tensor seen as 3-D (dim0 = head_dim, dim1 = head, dim2 = row); a box
// is 64 dims x box_heads heads x box_rows rows, 128-byte swizzled.  Rows past the end read zeros.
bool make_map(CUtensorMap *map, const void *base, int64_t rows, int heads, int box_heads, int box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)heads * kD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
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
    const int tq = kBM / group;
    CUtensorMap tq_map, tk, tv;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    if (!make_map(&tq_map, q, total_q, num_q_heads, group, tq) ||
        !make_map(&tk, k_cache, num_slots, num_kv_heads, 1, box_rows) ||
        !make_map(&tv, v_cache, num_slots, num_kv_heads, 1, box_rows))
        return NV_ERR_CUDA;

    PrefillParams p{};
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.block_tables = block_tables;
    p.d_err = d_err;
    p.bt_stride = bt_stride;
    p.num_q_heads = num_q_heads;
    p.group = group;
    p.group_shift = ilog2(group);
    p.block_shift = ilog2(block_size);
    p.box_rows = box_rows;
    p.num_blocks = num_blocks;
    p.max_pairs = (max_seqlen_q + 2 * tq - 1) / (2 * tq);
    p.scale_log2 = scale * nvkv::kLog2e;
    if (p.max_pairs > 65535)
        return NV_ERR_UNSUPPORTED;

    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (attr_err != cudaSuccess)
        return NV_ERR_CUDA;
    dim3 grid(num_kv_heads, num_seqs, p.max_pairs);
    paged_prefill_kernel<<<grid, kThreads, kSmemBytes, (cudaStream_t)stream>>>(tq_map, tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}
