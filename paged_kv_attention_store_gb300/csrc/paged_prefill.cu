// nv_paged_prefill_attn: varlen causal prefill over a paged prefix + new chunk, on tcgen05.
//
// What it computes is the prefill branch of the nano-vLLM field guide's Step 10.3 (with the
// packing of Step 07.5): sequence b owns packed query rows cu_q[b]..cu_q[b+1]-1 (Lq of them)
// and Lk = cu_k[b+1]-cu_k[b] keys read through its block table; the first P = Lk-Lq were
// cached before.  Query i of the chunk sees keys 0..P+i (bottom-right causal alignment).
//
// How (GB300 design; the pages call a library kernel here).  One CTA computes one 128-row
// query tile of one (sequence, kv head); with G = Hq/Hkv query heads per kv head the tile packs
// 128/G consecutive tokens x G heads, so every K/V tile loaded serves all G heads.
//   * warp 4 (TMA producer): the Q tile with one 3-D tensor-map copy per 64-dim half (dims
//     head_dim, q head, token), then K and V tiles of 128 keys x 128 dims straight from the
//     paged pool (dims head_dim, kv head, slot), 128-byte swizzled, into a 6-slot ring
//     K0 V0 K1 V1 ...; the sequence's block-table row is held 32 entries at a time in the
//     warp's registers, so a copy never waits on a dependent table load.
//   * warp 5 (MMA issuer; owns the TMEM allocation): one lane issues tcgen05.mma kind::f16
//     with fp32 accumulators in tensor memory.  TMEM holds THREE score buffers of 128 columns
//     and the 128-column O accumulator.  S(n) = Q K(n)^T (operands in shared memory) goes to
//     buffer n % 3; the softmax writes P(n) as bf16 pairs over the first half of that buffer;
//     O += P(n) V(n) reads P from tensor memory.  S(n+2) is issued right after PV(n): its
//     buffer last held P(n-1), whose PV finished an iteration earlier, so the issuer never
//     waits on a group it has just queued and the tensor pipe stays fed while the softmax of
//     tile n+1 runs.  (Sharing one score buffer with P forces S(n+1) to wait for PV(n) to
//     complete, which drains the pipe every iteration.)
//   * warps 0-3 (softmax / correction / epilogue): thread r owns row r = TMEM lane r.  It loads
//     its 128 scores at once, masks only on tiles that cross the diagonal, keeps a base-2 online
//     softmax with a lazy rescale (the running max moves only when a score beats it by more
//     than 8; only then is O rescaled in TMEM), writes P with tcgen05.st, and at the end
//     normalises O and stores bf16 rows.
// Tile shapes follow measurements on GB300: an M=128 tcgen05.mma costs about the same for N=64
// as for N=128, so key tiles are 128 wide; a group of 8 MMAs queued behind others streams at
// ~800 cycles but costs ~1100 issued into an empty pipe.
// Every mbarrier wait is bounded; on timeout the kernel records NV_DERR_TIMEOUT and stops.
#include <cuda.h>

#include <mutex>

#include "nv_common.cuh"

namespace {

using namespace nvkv;

constexpr int kD = 128;
constexpr int kBM = 128;             // rows per query tile (TMEM lanes)
constexpr int kBN = 128;             // keys per K/V tile
constexpr int kSlots = 6;            // K/V ring slots
constexpr int kBufs = 3;             // score / P buffers in TMEM
constexpr int kThreads = 192;        // warps 0-3 softmax; 4 producer; 5 MMA
constexpr uint32_t kTmemCols = 512;  // buffer b at b*128, O at 384
constexpr uint32_t kTmemO = 384;
constexpr float kRescaleLog2 = 8.0f;
// Of every 8 score pairs, this many take the polynomial exp2 on the FMA pipe; the rest use the
// special-function unit.
#ifndef NVKV_PREFILL_POLY_PAIRS
#define NVKV_PREFILL_POLY_PAIRS 0
#endif
constexpr int kPolyPairs = NVKV_PREFILL_POLY_PAIRS;

constexpr uint32_t kHalf = 128 * 128;         // 128 rows x 64 dims bf16 (one swizzle atom wide) = 16 KB
constexpr uint32_t kTile = 2 * kHalf;         // a 128 x 128 bf16 operand = 32 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kTile;            // slot s at kOffKV + s*kTile
constexpr uint32_t kOffBar = kOffKV + kSlots * kTile;
constexpr int kBarQ = 0;
constexpr int kBarKVFull = 1;                      // + slot
constexpr int kBarKVEmpty = kBarKVFull + kSlots;   // + slot
constexpr int kBarSFull = kBarKVEmpty + kSlots;    // + buffer
constexpr int kBarPFull = kBarSFull + kBufs;       // + buffer
constexpr int kBarODone = kBarPFull + kBufs;       // + buffer (PV(n) commits to n % 3)
constexpr int kNumBars = kBarODone + kBufs;
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
    int32_t max_tiles;      // gridDim.z
    float scale_log2;
};

// ---- packed fp32x2 arithmetic (Blackwell: one instruction for two fp32 lanes) ----
__device__ __forceinline__ uint64_t f2_pack(float a, float b)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 2^x0, 2^x1 on the FMA pipe (packed fp32x2), for x <= 8 (scores minus a running max).
// Range reduction: adding 1.5 * 2^23 rounds x to the nearest integer j, held in the low
// mantissa bits of the sum; f = x - j lies in [-0.5, 0.5] and 2^f comes from a cubic fitted to
// minimise the relative error on that interval (max relative error 7.6e-5, well below the bf16
// rounding of P); finally j is added into the exponent field.  x is clamped at -126 so masked
// scores (-inf) give a normal number of order 1e-38 instead of a wrapped exponent.
__device__ __forceinline__ void exp2_poly3_x2(float x0, float x1, float &p0, float &p1)
{
    constexpr float kC0 = 0.9999282882344301f, kC1 = 0.6932609081979648f;
    constexpr float kC2 = 0.24260776842531798f, kC3 = 0.05517030853684025f;
    constexpr float kRound = 12582912.0f;
    const uint64_t x = f2_pack(fmaxf(x0, -126.0f), fmaxf(x1, -126.0f));
    const uint64_t y = f2_add(x, f2_pack(kRound, kRound));
    const uint64_t j = f2_add(y, f2_pack(-kRound, -kRound));
    const uint64_t f = f2_fma(j, f2_pack(-1.0f, -1.0f), x);
    uint64_t q = f2_fma(f2_pack(kC3, kC3), f, f2_pack(kC2, kC2));
    q = f2_fma(q, f, f2_pack(kC1, kC1));
    q = f2_fma(q, f, f2_pack(kC0, kC0));
    float q0, q1, y0, y1;
    f2_unpack(q, q0, q1);
    f2_unpack(y, y0, y1);
    p0 = __uint_as_float(__float_as_uint(q0) + (__float_as_uint(y0) << 23));
    p1 = __uint_as_float(__float_as_uint(q1) + (__float_as_uint(y1) << 23));
}

// Max of 64 scores with 3-input max (32 instructions, 4 levels deep).
__device__ __forceinline__ float max64(const float (&s)[64])
{
    float m22[22];
#pragma unroll
    for (int k = 0; k < 21; ++k)
        m22[k] = fmax3(s[3 * k], s[3 * k + 1], s[3 * k + 2]);
    m22[21] = s[63];
    float m8[8];
#pragma unroll
    for (int k = 0; k < 7; ++k)
        m8[k] = fmax3(m22[3 * k], m22[3 * k + 1], m22[3 * k + 2]);
    m8[7] = m22[21];
    return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

// p = 2^(s * scale_log2 + neg_m) for 64 scores -> 32 bf16 pairs in pk; returns the fp32 sum.
__device__ __forceinline__ float exp_pack64(const float (&s)[64], float scale_log2, float neg_m, uint32_t *pk)
{
    const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
    const uint64_t negm2 = f2_pack(neg_m, neg_m);
    uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        float x0, x1, p0, p1;
        f2_unpack(f2_fma(f2_pack(s[2 * k], s[2 * k + 1]), scale2, negm2), x0, x1);
        if ((k & 7) >= 8 - kPolyPairs) {
            exp2_poly3_x2(x0, x1, p0, p1);
        } else {
            p0 = fast_exp2(x0);
            p1 = fast_exp2(x1);
        }
        rs2[k & 3] = f2_add(rs2[k & 3], f2_pack(p0, p1));
        pk[k] = pack_bf16x2(p0, p1);
    }
    float ra, rb, rc, rd;
    f2_unpack(f2_add(rs2[0], rs2[1]), ra, rb);
    f2_unpack(f2_add(rs2[2], rs2[3]), rc, rd);
    return (ra + rb) + (rc + rd);
}

// Load 64 score columns of this thread's row and apply the causal mask (keys j > rel hidden).
__device__ __forceinline__ void load_scores(uint32_t taddr, bool masked, int rel, float (&s)[64])
{
    uint32_t v[64];
    tmem_ld64(taddr, v);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 64; ++j)
        s[j] = (!masked || j <= rel) ? __uint_as_float(v[j]) : -INFINITY;
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
    const int ntiles = (Lq + tq - 1) / tq;
    if (ntiles > p.max_tiles && blockIdx.z == 0 && kvh == 0 && threadIdx.x == 0)
        flag_error(p.d_err, NV_DERR_LENGTH);
    const int tile = p.max_tiles - 1 - (int)blockIdx.z;    // the heaviest tiles are dispatched first
    if (tile >= ntiles)
        return;
    const int i0 = tile * tq;
    const int nq = min(tq, Lq - i0);
    const int kv_len = P + i0 + nq;                        // keys any row of the tile can see
    const int nkv = (kv_len + kBN - 1) / kBN;
    const int first_masked = (P + i0 + 1) / kBN;           // key tiles before this need no mask

    const uint32_t bar = base + kOffBar;
    auto BAR = [&](int i) { return bar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmemSlot);

    if (threadIdx.x == 0) {
        mbar_init(BAR(kBarQ), 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(BAR(kBarKVFull + s), 1);
            mbar_init(BAR(kBarKVEmpty + s), 1);
        }
        for (int s = 0; s < kBufs; ++s) {
            mbar_init(BAR(kBarSFull + s), 1);
            mbar_init(BAR(kBarPFull + s), 4);
            mbar_init(BAR(kBarODone + s), 1);
        }
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

    if (warp == 4) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            mbar_arrive_expect_tx(BAR(kBarQ), kTile);
            for (int h = 0; h < 2; ++h)
                tma_load_3d(base + kOffQ + h * kHalf, &tmap_q, h * 64, kvh * p.group, cq0 + i0, BAR(kBarQ));
        }
        const int32_t *bt = p.block_tables + (size_t)b * p.bt_stride;
        const int nblk = (kv_len + (1 << p.block_shift) - 1) >> p.block_shift;   // entries this CTA reads
        const int bs_mask = (1 << p.block_shift) - 1;
        const int boxes = kBN / p.box_rows;
        int win_base = 0;
        int win = lane < nblk ? __ldg(bt + lane) : -1;
        bool ok = true;
        for (int n = 0; n < nkv && ok; ++n) {
            int slot0[kBN / 16];                    // first slot of each box; -1 = skip the box
            int nbox = 0;
            for (int k = 0; k < boxes; ++k) {
                const int j0 = n * kBN + k * p.box_rows;
                slot0[k] = -1;
                if (j0 >= kv_len)
                    continue;
                const int lb = j0 >> p.block_shift;
                if (lb >= win_base + 32) {          // advance the window (warp-uniform)
                    win_base = lb & ~31;
                    win = win_base + lane < nblk ? __ldg(bt + win_base + lane) : -1;
                }
                const int blk = __shfl_sync(0xffffffffu, win, lb - win_base);
                if (blk < 0 || blk >= p.num_blocks) {
                    if (lane == 0)
                        flag_error(p.d_err, NV_DERR_BLOCK_RANGE);
                    continue;
                }
                slot0[k] = (blk << p.block_shift) + (j0 & bs_mask);
                ++nbox;
            }
            const uint32_t bytes = (uint32_t)nbox * p.box_rows * 128u * 2u;
            for (int kv = 0; kv < 2; ++kv) {        // K(n) then V(n): tiles t = 2n, 2n+1
                const int t = 2 * n + kv;
                const int slot = t % kSlots;
                if (t >= kSlots &&
                    !__all_sync(0xffffffffu, mbar_wait(BAR(kBarKVEmpty + slot), ((t / kSlots) - 1) & 1))) {
                    if (lane == 0)
                        flag_error(p.d_err, NV_DERR_TIMEOUT);
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const CUtensorMap *map = kv ? &tmap_v : &tmap_k;
                    const uint32_t dst = base + kOffKV + slot * kTile;
                    mbar_arrive_expect_tx(BAR(kBarKVFull + slot), bytes);
                    for (int k = 0; k < boxes; ++k) {
                        if (slot0[k] < 0)
                            continue;
                        const uint32_t roff = (uint32_t)k * p.box_rows * 128u;
                        tma_load_3d(dst + roff, map, 0, kvh, slot0[k], BAR(kBarKVFull + slot));
                        tma_load_3d(dst + kHalf + roff, map, 64, kvh, slot0[k], BAR(kBarKVFull + slot));
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp == 5) {
        // ============================ MMA issuer ============================
        constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);   // Q, K both K-major
        constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, kD, false, true);     // P (TMEM), V MN-major
        bool ok = __all_sync(0xffffffffu, mbar_wait(BAR(kBarQ), 0));
        auto wait_all = [&](uint32_t b_, uint32_t parity) {
            ok = ok && __all_sync(0xffffffffu, mbar_wait(b_, parity));
            return ok;
        };
        auto issue_s = [&](int n) {
            const int t = 2 * n;
            const int slot = t % kSlots;
            const int bb = n % kBufs;
            if (!wait_all(BAR(kBarKVFull + slot), (t / kSlots) & 1))
                return;
            // buffer bb last held P(n-3): its PV must have finished (one iteration ago)
            if (n >= kBufs && !wait_all(BAR(kBarODone + bb), ((n - kBufs) / kBufs) & 1))
                return;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t ktile = base + kOffKV + slot * kTile;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                    mma_bf16_ss(tmem + bb * 128, smem_desc_sw128(base + kOffQ + off, 16, 1024),
                                smem_desc_sw128(ktile + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(BAR(kBarSFull + bb));
                mma_commit(BAR(kBarKVEmpty + slot));
            }
            __syncwarp();
        };
        auto issue_pv = [&](int n) {
            const int t = 2 * n + 1;
            const int slot = t % kSlots;
            const int bb = n % kBufs;
            if (!wait_all(BAR(kBarKVFull + slot), (t / kSlots) & 1))
                return;
            const uint32_t vtile = base + kOffKV + slot * kTile;
            const int vrows = kv_len - n * kBN;
            if (vrows < kBN) {
                // Keys past the sequence carry P = 0, but their V rows may hold anything (NaN
                // patterns included) and 0 * NaN would poison O: zero them.
                const int per_half = (kBN - vrows) * 8;        // 16-byte chunks
                for (int c = lane; c < 2 * per_half; c += 32) {
                    const int half = c / per_half;
                    const int rem = c % per_half;
                    sts_u4(vtile + half * kHalf + (uint32_t)(vrows + rem / 8) * 128u + (uint32_t)(rem % 8) * 16u,
                           make_uint4(0, 0, 0, 0));
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (!wait_all(BAR(kBarPFull + bb), (n / kBufs) & 1))
                return;
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_bf16_ts(tmem + kTmemO, tmem + bb * 128 + kk * 8,
                                smem_desc_sw128(vtile + kk * 16 * 128, kHalf, 1024), idesc_o,
                                (n > 0 || kk > 0) ? 1u : 0u);
                mma_commit(BAR(kBarODone + bb));
                mma_commit(BAR(kBarKVEmpty + slot));
            }
            __syncwarp();
        };
        issue_s(0);
        if (nkv > 1)
            issue_s(1);
        for (int n = 0; n < nkv && ok; ++n) {
            issue_pv(n);
            if (n + 2 < nkv)
                issue_s(n + 2);
        }
        if (!ok && lane == 0)
            flag_error(p.d_err, NV_DERR_TIMEOUT);
    } else {
        // ================= softmax / correction / epilogue (warps 0-3) =================
        const int r = threadIdx.x;                      // tile row == TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t o_addr = tmem + lane_base + kTmemO;
        const int tok = i0 + (r >> p.group_shift);      // token index inside the chunk
        const int head = (int)kvh * p.group + (r & (p.group - 1));
        const bool valid = tok < Lq;
        const int lim = P + tok;                        // last key this row may see
        float m_run = -INFINITY;                        // running max of scale*log2(e)*s
        float l_run = 0.f;
        bool ok = true;
        for (int n = 0; n < nkv && ok; ++n) {
            const int bb = n % kBufs;
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBarSFull + bb), (n / kBufs) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t s_addr = tmem + lane_base + bb * 128;
            const bool masked = n >= first_masked;
            const int rel = lim - n * kBN;              // keys j <= rel of this tile are visible
            float s0[64], s1[64];
            load_scores(s_addr, masked, rel, s0);
            load_scores(s_addr + 64, masked, rel - 64, s1);
            const float mx2 = fmaxf(max64(s0), max64(s1)) * p.scale_log2;
            const bool need = mx2 > m_run + kRescaleLog2;
            float alpha = 1.f;
            if (need) {
                alpha = fast_exp2(m_run - mx2);         // m_run = -inf -> 0
                m_run = mx2;
            }
            const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
            uint32_t pk[64];
            const float rs = exp_pack64(s0, p.scale_log2, neg_m, pk) + exp_pack64(s1, p.scale_log2, neg_m, pk + 32);
            l_run = l_run * alpha + rs;
            if (n >= 1 && __any_sync(0xffffffffu, need)) {
                // rare: rescale O.  PV(0..n-1) accumulate into O in order; wait for the last.
                const int pb = (n - 1) % kBufs;
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBarODone + pb), ((n - 1) / kBufs) & 1))) {
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
            }
            // P(n) as bf16 pairs over the first 64 columns of buffer bb (A operand of PV(n))
            tmem_st64(s_addr, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(BAR(kBarPFull + bb));
        }
        // ---- epilogue: O / l -> bf16 rows ----
        const int last = nkv - 1;
        if (ok && __all_sync(0xffffffffu, mbar_wait(BAR(kBarODone + last % kBufs), (last / kBufs) & 1))) {
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

    // ---------------- teardown: every TMEM access is done before the free ----------------
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
    p.max_tiles = (max_seqlen_q + tq - 1) / tq;
    p.scale_log2 = scale * nvkv::kLog2e;
    if (p.max_tiles > 65535)
        return NV_ERR_UNSUPPORTED;

    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (attr_err != cudaSuccess)
        return NV_ERR_CUDA;
    dim3 grid(num_kv_heads, num_seqs, p.max_tiles);
    paged_prefill_kernel<<<grid, kThreads, kSmemBytes, (cudaStream_t)stream>>>(tq_map, tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}
