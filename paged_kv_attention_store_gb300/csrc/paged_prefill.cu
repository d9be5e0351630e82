// nv_paged_prefill_attn: varlen causal prefill over a paged prefix + new chunk, on tcgen05.
//
// What it computes is the prefill branch of the nano-vLLM field guide's Step 10.3 (with the
// packing of Step 07.5): sequence b owns packed query rows cu_q[b]..cu_q[b+1]-1 (Lq of them)
// and Lk = cu_k[b+1]-cu_k[b] keys read through its block table; the first P = Lk-Lq were
// cached before.  Query i of the chunk sees keys 0..P+i (bottom-right causal alignment).
//
// How (GB300 design; the pages call a library kernel here).  The unit of work is one 128-row
// query tile of one (sequence, kv head); with G = Hq/Hkv query heads per kv head the tile packs
// 128/G consecutive tokens x G heads, so every K/V tile loaded serves all G heads.  The kernel
// is persistent (one CTA per SM): CTAs claim tiles, heaviest first, from a counter in the
// caller's workspace, and each CTA runs its tiles as one continuous stream of 128-key steps, so
// the next tile's first scores are computed while the current tile finishes.
//   * warp 4 (TMA producer): claims tiles and passes them to the other warps through a small
//     queue in shared memory.  Copies go out in the order they are needed: a tile's Q (one 3-D
//     tensor-map copy per 64-dim half; dims head_dim, q head, token) into one of two Q buffers,
//     K and V tiles of 128 keys x 128 dims straight from the paged pool (dims head_dim, kv
//     head, slot), 128-byte swizzled, into a 3-slot K ring and a 2-slot V ring, K running two
//     steps ahead of V as the MMAs consume them.  Lane i copies box i of a step; the block-table
//     row is held 32 entries at a time in the warp's registers.
//   * warp 5 (MMA issuer; owns the TMEM allocation): one lane issues tcgen05.mma kind::f16
//     with fp32 accumulators in tensor memory.  TMEM holds THREE score buffers of 128 columns
//     and the 128-column O accumulator.  S(n) = Q K(n)^T (operands in shared memory) goes to
//     buffer n % 3; the softmax writes P(n) as bf16 pairs over the first half of that buffer;
//     O += P(n) V(n) reads P from tensor memory.  S(n+2) is issued right after PV(n): its
//     buffer last held P(n-1), whose PV finished an iteration earlier, so the issuer never
//     waits on a group it has just queued.  Operand descriptors are precomputed per buffer.
//   * warps 0-3 (softmax / correction / epilogue): thread r owns row r = TMEM lane r.  It loads
//     its 128 scores at once, masks only on steps that cross the diagonal (a separate code
//     path), keeps a base-2 online softmax with a lazy rescale (the running max moves only when
//     a score beats it by more than 8; only then is O rescaled in TMEM), and writes P with
//     tcgen05.st.  At a tile's end it normalises O, stages the bf16 rows in the tile's Q buffer
//     (free once the last PV is done) and writes them with tensor-map stores.
// Measured on GB300: an M=128 tcgen05.mma costs about the same for N=64 as for N=128 (so key
// steps are 128 wide), the MMA issue queue is shallow (any idle time in the issuing warp idles
// the tensor pipe), and loading 128 fp32 scores from TMEM takes ~100 cycles.
// Every mbarrier wait is bounded; on timeout the kernel records NV_DERR_TIMEOUT and stops.
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "nv_common.cuh"

namespace {

using namespace nvkv;

constexpr int kD = 128;
constexpr int kBM = 128;             // rows per query tile (TMEM lanes)
constexpr int kBN = 128;             // keys per K/V tile
constexpr int kQBufs = 2;            // Q buffers: the next item's Q loads while this one runs
#ifndef NVKV_PREFILL_KSLOTS
#define NVKV_PREFILL_KSLOTS 3
#endif
constexpr int kKSlots = NVKV_PREFILL_KSLOTS;   // K ring slots
constexpr int kVSlots = 5 - kKSlots;           // V ring slots
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
constexpr uint32_t kOffQ = 0;                 // Q buffer q at q*kTile (two: the next tile's Q loads early)
constexpr uint32_t kOffK = kQBufs * kTile;    // K slot s at kOffK + s*kTile
constexpr uint32_t kOffV = kOffK + kKSlots * kTile;
constexpr uint32_t kOffBar = kOffV + kVSlots * kTile;
constexpr int kBarQFull = 0;                       // + q buffer
constexpr int kBarQEmpty = 2;                      // + q buffer
constexpr int kBarKFull = 4;                       // + K slot
constexpr int kBarKEmpty = kBarKFull + kKSlots;    // + K slot
constexpr int kBarVFull = kBarKEmpty + kKSlots;    // + V slot
constexpr int kBarVEmpty = kBarVFull + kVSlots;    // + V slot
constexpr int kBarSFull = kBarVEmpty + kVSlots;    // + buffer
constexpr int kBarPFull = kBarSFull + kBufs;       // + buffer
constexpr int kBarODone = kBarPFull + kBufs;       // + buffer (PV(n) commits to n % 3)
constexpr int kQueue = 8;                          // claimed work items in flight
constexpr int kBarItemFull = kBarODone + kBufs;    // + queue slot
constexpr int kBarItemEmpty = kBarItemFull + kQueue;
constexpr int kItemReaders = 6;                    // MMA S cursor, MMA PV cursor, 4 softmax warps
constexpr int kNumBars = kBarItemEmpty + kQueue;
constexpr uint32_t kOffItems = kOffBar + kNumBars * 8;
constexpr uint32_t kOffTmemSlot = kOffItems + kQueue * 4;
constexpr uint32_t kSmemBytes = kOffTmemSlot + 16 + 1024;      // + slack for 1024-byte alignment
static_assert(kSmemBytes <= 227u * 1024u, "shared memory per CTA");

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
    int32_t max_tiles;      // query tiles of the longest chunk
    int32_t num_kv_heads;
    int32_t num_seqs;
    int32_t *tile_counter;  // zeroed before the launch; CTAs claim work items from it
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

// One unit of work: a 128-row query tile of one (sequence, kv head).  Virtual tile v runs over
// (tile level, sequence, kv head) with the tile level slowest and counted from the LAST tile of
// the longest chunk, so the heaviest tiles (most keys) come first.  Persistent CTAs claim them
// in that order from a global counter and skip those past the end of their sequence's chunk.
struct Item {
    int v;
    int b, kvh, cq0, Lq, P, i0, nq, kv_len, nkv, first_masked;
};

__device__ __forceinline__ bool load_item(const PrefillParams &p, int v, Item &it)
{
    const int per_level = p.num_seqs * p.num_kv_heads;
    const int level = v / per_level;
    const int rem = v - level * per_level;
    it.v = v;
    it.b = rem / p.num_kv_heads;
    it.kvh = rem - it.b * p.num_kv_heads;
    it.cq0 = __ldg(p.cu_q + it.b);
    const int cq1 = __ldg(p.cu_q + it.b + 1);
    const int Lk = __ldg(p.cu_k + it.b + 1) - __ldg(p.cu_k + it.b);
    it.Lq = cq1 - it.cq0;
    it.P = Lk - it.Lq;
    if (it.Lq < 0 || it.P < 0 || ((Lk + (1 << p.block_shift) - 1) >> p.block_shift) > p.bt_stride) {
        flag_error(p.d_err, NV_DERR_LENGTH);
        return false;
    }
    const int tq = kBM >> p.group_shift;
    const int ntiles = (it.Lq + tq - 1) / tq;
    if (level == 0 && ntiles > p.max_tiles)
        flag_error(p.d_err, NV_DERR_LENGTH);
    const int tile = p.max_tiles - 1 - level;
    if (tile >= ntiles)
        return false;
    it.i0 = tile * tq;
    it.nq = min(tq, it.Lq - it.i0);
    it.kv_len = it.P + it.i0 + it.nq;
    it.nkv = (it.kv_len + kBN - 1) / kBN;
    it.first_masked = (it.P + it.i0 + 1) / kBN;
    return true;
}

// Resolve a claimed virtual tile: while it is empty (past its chunk's end), claim the next one
// from the global counter.  Returns total when none is left.  Tiles are claimed in the
// heaviest-first order as CTAs free up, which balances the load.
__device__ __forceinline__ int resolve_claim(const PrefillParams &p, int v, int total)
{
    Item it;
    while (v < total && !load_item(p, v, it))
        v = atomicAdd(p.tile_counter, 1);
    return v < total ? v : total;
}

__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_o,
                         const PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;     // swizzled tiles need 1024-byte alignment
    uint8_t *smem = smem_raw + (base - raw_base);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total = p.max_tiles * p.num_seqs * p.num_kv_heads;

    const uint32_t bar = base + kOffBar;
    auto BAR = [&](int i) { return bar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmemSlot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(kBarQFull + s), 1);
            mbar_init(BAR(kBarQEmpty + s), 1 + 4);     // last S of the item + the 4 epilogue warps
        }
        for (int s = 0; s < kKSlots; ++s) {
            mbar_init(BAR(kBarKFull + s), 1);
            mbar_init(BAR(kBarKEmpty + s), 1);
        }
        for (int s = 0; s < kVSlots; ++s) {
            mbar_init(BAR(kBarVFull + s), 1);
            mbar_init(BAR(kBarVEmpty + s), 1);
        }
        for (int s = 0; s < kBufs; ++s) {
            mbar_init(BAR(kBarSFull + s), 1);
            mbar_init(BAR(kBarPFull + s), 4);
            mbar_init(BAR(kBarODone + s), 1);
        }
        for (int s = 0; s < kQueue; ++s) {
            mbar_init(BAR(kBarItemFull + s), 1);
            mbar_init(BAR(kBarItemEmpty + s), kItemReaders);
        }
        fence_barrier_init();
    }
    // Work items pass from the producer (which claims them) to the MMA issuer's two cursors and
    // the four softmax warps through a small queue in shared memory.
    volatile int *items = reinterpret_cast<volatile int *>(smem + kOffItems);
    auto read_item = [&](int k, int &v) {            // whole warp calls; lane 0 releases the slot
        if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBarItemFull + k % kQueue), (k / kQueue) & 1)))
            return false;
        v = items[k % kQueue];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(BAR(kBarItemEmpty + k % kQueue));
        return true;
    };
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
        // Copies go out in the order the MMA issuer needs them.  S(j) is issued two key tiles
        // before PV(j), so K(j) is copied two tiles ahead of V(j): the stream is K(j) V(j-2),
        // K(j+1) V(j-1), ...  An item's Q tile goes out just before its first K tile (after the
        // V copy that precedes it: that V feeds the PV whose completion frees the Q buffer).
        // Lane kb copies box kb of a tile (box_rows keys, both 64-dim halves).
        const int bs_mask = (1 << p.block_shift) - 1;
        const int boxes = kBN / p.box_rows;
        if (lane == 0) {
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            prefetch_tmap(&tmap_o);
        }
        struct TileCopy {
            int slot;           // this lane's box: first pool slot, -1 = none
            int kvh;
            uint32_t bytes;     // whole tile
        };
        // copy one K or V tile into its ring (idx = its global key tile)
        auto copy_tile = [&](bool is_v, int idx, const TileCopy &c) {
            const int n_slots = is_v ? kVSlots : kKSlots;
            const int s_ = idx % n_slots;
            const uint32_t full = BAR((is_v ? kBarVFull : kBarKFull) + s_);
            if (idx >= n_slots &&
                !__all_sync(0xffffffffu,
                            mbar_wait(BAR((is_v ? kBarVEmpty : kBarKEmpty) + s_), ((idx / n_slots) - 1) & 1)))
                return false;
            const uint32_t dst = base + (is_v ? kOffV : kOffK) + s_ * kTile + (uint32_t)lane * p.box_rows * 128u;
            if (lane == 0)
                mbar_arrive_expect_tx(full, c.bytes);
            __syncwarp();
            if (c.slot >= 0) {
                const CUtensorMap *map = is_v ? &tmap_v : &tmap_k;
                tma_load_3d(dst, map, 0, c.kvh, c.slot, full);
                tma_load_3d(dst + kHalf, map, 64, c.kvh, c.slot, full);
            }
            return true;
        };
        bool ok = true;
        int j = 0;                                  // global key tile of the next K copy
        TileCopy v1{-1, 0, 0}, v2{-1, 0, 0};        // tiles j-1 and j-2, whose V is still to copy
        // lane 0 claims one item ahead: the counter's answer for item k+1 travels while item k's
        // copies are issued, and is resolved (empty tiles skipped) only when it is needed
        int pending = 0;
        if (lane == 0)
            pending = atomicAdd(p.tile_counter, 1);
        for (int k = 0; ok; ++k) {
            // publish item k to the other warps
            if (k >= kQueue &&
                !__all_sync(0xffffffffu, mbar_wait(BAR(kBarItemEmpty + k % kQueue), ((k / kQueue) - 1) & 1))) {
                ok = false;
                break;
            }
            int v = 0;
            if (lane == 0) {
                v = resolve_claim(p, pending, total);
                items[k % kQueue] = v;
                mbar_arrive(BAR(kBarItemFull + k % kQueue));
                if (v < total)
                    pending = atomicAdd(p.tile_counter, 1);
            }
            v = __shfl_sync(0xffffffffu, v, 0);
            if (v >= total)
                break;
            Item it;
            load_item(p, v, it);
            const int32_t *bt = p.block_tables + (size_t)it.b * p.bt_stride;
            const int nblk = (it.kv_len + (1 << p.block_shift) - 1) >> p.block_shift;
            int win_base = 0;                       // the block-table row, 32 entries at a time
            int win = lane < nblk ? __ldg(bt + lane) : -1;
            for (int n = 0; n < it.nkv && ok; ++n) {
                // this lane's box of tile n
                TileCopy cur{-1, it.kvh, 0};
                const int lb0 = (n * kBN) >> p.block_shift;
                const int lb_hi = min(lb0 + boxes - 1, nblk - 1);
                if (lb_hi >= win_base + 32) {       // warp-uniform window move
                    win_base = lb0;
                    win = win_base + lane < nblk ? __ldg(bt + win_base + lane) : -1;
                }
                const int j0 = n * kBN + lane * p.box_rows;
                const int lb = j0 >> p.block_shift;
                const int blk = __shfl_sync(0xffffffffu, win, (lb - win_base) & 31);
                if (lane < boxes && j0 < it.kv_len) {
                    if (blk < 0 || blk >= p.num_blocks)
                        flag_error(p.d_err, NV_DERR_BLOCK_RANGE);
                    else
                        cur.slot = (blk << p.block_shift) + (j0 & bs_mask);
                }
                cur.bytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, cur.slot >= 0)) * p.box_rows * 256u;
                if (n == 0) {
                    if (j >= 2 && !copy_tile(true, j - 2, v2)) {
                        ok = false;
                        break;
                    }
                    // the item's Q, into buffer k % 2 once item k-2's last S and epilogue are done
                    const int qb = k % kQBufs;
                    if (k >= kQBufs &&
                        !__all_sync(0xffffffffu, mbar_wait(BAR(kBarQEmpty + qb), ((k / kQBufs) - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(BAR(kBarQFull + qb), kTile);
                        for (int h = 0; h < 2; ++h)
                            tma_load_3d(base + kOffQ + qb * kTile + h * kHalf, &tmap_q, h * 64,
                                        it.kvh * p.group, it.cq0 + it.i0, BAR(kBarQFull + qb));
                    }
                    if (!copy_tile(false, j, cur)) {
                        ok = false;
                        break;
                    }
                } else {
                    if (!copy_tile(false, j, cur) || (j >= 2 && !copy_tile(true, j - 2, v2))) {
                        ok = false;
                        break;
                    }
                }
                v2 = v1;
                v1 = cur;
                ++j;
            }
        }
        // the last two V tiles
        if (ok && j >= 2)
            ok = copy_tile(true, j - 2, v2);
        if (ok && j >= 1)
            ok = copy_tile(true, j - 1, v1);
        if (!ok && lane == 0)
            flag_error(p.d_err, NV_DERR_TIMEOUT);
    } else if (warp == 5) {
        // ============================ MMA issuer ============================
        // Key tiles of all this CTA's work items form one global sequence g.  S(g) goes to TMEM
        // buffer g % 3; the issue order S(0) S(1) | PV(g) S(g+2) | ... runs across tile boundaries,
        // so the next tile's first scores are computed during the current tile's last softmax.
        constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);   // Q, K both K-major
        constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, kD, false, true);     // P (TMEM), V MN-major
        // Operand descriptors of Q buffer 0 and K / V slot 0; the others differ only in the start
        // address field (address / 16, 14 bits: every buffer lies below 256 KB), so a buffer's
        // descriptor is the slot-0 one plus its offset / 16.
        const uint64_t desc_q0 = smem_desc_sw128(base + kOffQ, 16, 1024);
        const uint64_t desc_k0 = smem_desc_sw128(base + kOffK, 16, 1024);
        const uint64_t desc_v0 = smem_desc_sw128(base + kOffV, kHalf, 1024);
        bool ok = true;
        auto wait_all = [&](uint32_t b_, uint32_t parity) {
            ok = ok && __all_sync(0xffffffffu, mbar_wait(b_, parity));
            return ok;
        };
        struct Cursor {
            Item it;
            int k;      // work item count
            int n;      // key tile within the item
            int g;      // global key tile
            bool have;  // it holds item k
        };
        // true when the cursor has a key tile to issue; reads its item from the queue only when
        // the cursor reaches it, so the issuer never waits for a claim it does not yet need
        auto ready = [&](Cursor &c) {
            if (!c.have) {
                int v = total;
                if (!read_item(c.k, v)) {
                    ok = false;
                    v = total;
                }
                c.it.v = v;
                if (v < total)
                    load_item(p, v, c.it);
                c.have = true;
            }
            return ok && c.it.v < total;
        };
        Cursor cs{}, cp{};                           // S cursor, PV cursor
        auto advance = [&](Cursor &c) {
            if (++c.n == c.it.nkv) {
                ++c.k;
                c.n = 0;
                c.have = false;
            }
            ++c.g;
        };
        auto issue_s = [&](Cursor &c) {
            const int g = c.g;
            const int slot = g % kKSlots;
            const int bb = g % kBufs;
            const int qb = c.k % kQBufs;
            if (c.n == 0 && !wait_all(BAR(kBarQFull + qb), (c.k / kQBufs) & 1))
                return;
            if (!wait_all(BAR(kBarKFull + slot), (g / kKSlots) & 1))
                return;
            // buffer bb last held P(g-3): its PV must have finished (one key tile ago)
            if (g >= kBufs && !wait_all(BAR(kBarODone + bb), ((g - kBufs) / kBufs) & 1))
                return;
            tc_fence_after();
            if (lane == 0) {
                const uint64_t dq = desc_q0 + (uint64_t)(qb * (kTile >> 4));
                const uint64_t dk = desc_k0 + (uint64_t)(slot * (kTile >> 4));
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    // k-step kk: 16 dims = 32 bytes into the 128-byte swizzle row, 64 dims per half
                    const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                    mma_bf16_ss(tmem + bb * 128, dq + off, dk + off, idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(BAR(kBarSFull + bb));
                mma_commit(BAR(kBarKEmpty + slot));
                if (c.n == c.it.nkv - 1)
                    mma_commit(BAR(kBarQEmpty + qb));   // the item's last use of its Q buffer
            }
            __syncwarp();
            advance(c);
        };
        auto issue_pv = [&](Cursor &c) {
            const int g = c.g;
            const int n = c.n;
            const int slot = g % kVSlots;
            const int bb = g % kBufs;
            if (!wait_all(BAR(kBarVFull + slot), (g / kVSlots) & 1))
                return;
            const uint32_t vtile = base + kOffV + slot * kTile;
            const int vrows = c.it.kv_len - n * kBN;
            if (vrows < kBN) {
                // Keys past the sequence carry P = 0, but their V rows may hold anything (NaN
                // patterns included) and 0 * NaN would poison O: zero them.
                const int per_half = (kBN - vrows) * 8;        // 16-byte chunks
                for (int c2 = lane; c2 < 2 * per_half; c2 += 32) {
                    const int half = c2 / per_half;
                    const int rem = c2 % per_half;
                    sts_u4(vtile + half * kHalf + (uint32_t)(vrows + rem / 8) * 128u + (uint32_t)(rem % 8) * 16u,
                           make_uint4(0, 0, 0, 0));
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (!wait_all(BAR(kBarPFull + bb), (g / kBufs) & 1))
                return;
            tc_fence_after();
            if (lane == 0) {
                const uint64_t dv = desc_v0 + (uint64_t)(slot * (kTile >> 4));
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)      // k-step kk: keys 16kk.. = 16 rows of 128 bytes
                    mma_bf16_ts(tmem + kTmemO, tmem + bb * 128 + kk * 8, dv + (uint64_t)(kk * 16 * 128 >> 4),
                                idesc_o, (n > 0 || kk > 0) ? 1u : 0u);
                mma_commit(BAR(kBarODone + bb));
                mma_commit(BAR(kBarVEmpty + slot));
            }
            __syncwarp();
            advance(c);
        };
        // S runs two key tiles ahead of PV
        if (ready(cs))
            issue_s(cs);
        if (ready(cs))
            issue_s(cs);
        while (ready(cp)) {
            issue_pv(cp);
            if (ready(cs))
                issue_s(cs);
        }
        if (!ok && lane == 0)
            flag_error(p.d_err, NV_DERR_TIMEOUT);
    } else {
        // ================= softmax / correction / epilogue (warps 0-3) =================
        const int r = threadIdx.x;                      // tile row == TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t o_addr = tmem + lane_base + kTmemO;
        Item it;
        bool ok = true;
        int g = 0;                                      // global key tile
        for (int k = 0; ok; ++k) {
            int v = total;
            if (!read_item(k, v)) {
                ok = false;
                break;
            }
            if (v >= total)
                break;
            load_item(p, v, it);
            const int tok = it.i0 + (r >> p.group_shift);   // token index inside the chunk
            const int head = it.kvh * p.group + (r & (p.group - 1));
            const bool valid = tok < it.Lq;
            const int lim = it.P + tok;                 // last key this row may see
            float m_run = -INFINITY;                    // running max of scale*log2(e)*s
            float l_run = 0.f;
            // One key tile; MASKED is a compile-time flag so the tiles that do not cross the
            // diagonal (nearly all) carry no per-score select.
            auto tile = [&](int n, auto masked_c) -> bool {
                constexpr bool kMasked = decltype(masked_c)::value;
                const int bb = g % kBufs;
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBarSFull + bb), (g / kBufs) & 1)))
                    return false;
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_base + bb * 128;
                uint32_t u0[64], u1[64];
                tmem_ld64(s_addr, u0);
                tmem_ld64(s_addr + 64, u1);
                tmem_wait_ld();
                float s0[64], s1[64];
                const int rel = lim - n * kBN;          // keys j <= rel of this tile are visible
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    s0[j] = (!kMasked || j <= rel) ? __uint_as_float(u0[j]) : -INFINITY;
                    s1[j] = (!kMasked || j + 64 <= rel) ? __uint_as_float(u1[j]) : -INFINITY;
                }
                const float mx2 = fmaxf(max64(s0), max64(s1)) * p.scale_log2;
                const bool need = mx2 > m_run + kRescaleLog2;
                float alpha = 1.f;
                if (need) {
                    alpha = fast_exp2(m_run - mx2);     // m_run = -inf -> 0
                    m_run = mx2;
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
                uint32_t pk[64];
                const float rs =
                    exp_pack64(s0, p.scale_log2, neg_m, pk) + exp_pack64(s1, p.scale_log2, neg_m, pk + 32);
                l_run = l_run * alpha + rs;
                if (n >= 1 && __any_sync(0xffffffffu, need)) {
                    // rare: rescale O.  The PVs of this item accumulate into O in order; wait
                    // for the last one issued (global tile g-1).
                    const int pb = (g - 1) % kBufs;
                    if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBarODone + pb), ((g - 1) / kBufs) & 1)))
                        return false;
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
                // P as bf16 pairs over the first 64 columns of buffer bb (A operand of its PV)
                tmem_st64(s_addr, pk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(BAR(kBarPFull + bb));
                return true;
            };
            for (int n = 0; n < it.nkv && ok; ++n, ++g)
                ok = n < it.first_masked ? tile(n, std::false_type{}) : tile(n, std::true_type{});
            if (!ok)
                break;
            // ---- epilogue: O / l -> bf16 rows (before this warpgroup's next P lets PV reuse O) ----
            // The last PV's completion also means every S of the item has read its Q buffer, so
            // the rows are staged there (same 128-byte swizzled layout as the Q tile: row r of
            // the tile is TMEM lane r) and each warp writes its 32 rows with one tensor store per
            // 64-dim half.  A warp whose rows run past the chunk's end (the ragged last tile)
            // stores its valid rows directly instead, so it never touches the next sequence.
            const int last = g - 1;
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBarODone + last % kBufs), (last / kBufs) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv = (valid && l_run > 0.f) ? 1.f / l_run : 0.f;
            const bool warp_full = __all_sync(0xffffffffu, valid);
            const int qb = k % kQBufs;
            const uint32_t stage = base + kOffQ + qb * kTile;
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((size_t)(it.cq0 + tok) * p.num_q_heads + head) * kD);
#pragma unroll
            for (int c = 0; c < kD / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(o_addr + c * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * inv, __uint_as_float(v[8 * j + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv, __uint_as_float(v[8 * j + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv, __uint_as_float(v[8 * j + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv, __uint_as_float(v[8 * j + 7]) * inv);
                    const int chunk = c * 4 + j;            // 16-byte chunk of the 256-byte row
                    if (warp_full)
                        sts_u4(stage + (chunk >> 3) * kHalf + (uint32_t)r * 128u +
                                   ((uint32_t)((chunk & 7) ^ (r & 7)) << 4),
                               w);
                    else if (valid)
                        dst[chunk] = w;
                }
            }
            if (warp_full) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int row0 = it.cq0 + it.i0 + ((warp * 32) >> p.group_shift);
                    for (int h = 0; h < 2; ++h)
                        tma_store_3d(&tmap_o, stage + h * kHalf + warp * 4096, h * 64, it.kvh * p.group, row0);
                    bulk_commit_group();
                    bulk_wait_group_read0();
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(BAR(kBarQEmpty + qb));
            tc_fence_before();      // O reads are ordered before the next item's first PV
        }
        if (!ok && lane == 0)
            flag_error(p.d_err, NV_DERR_TIMEOUT);
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
                                     float scale, void *out, void *workspace, size_t workspace_bytes,
                                     int32_t *d_err, nv_stream_t stream)
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
    if (!workspace || workspace_bytes < NV_PREFILL_WORKSPACE_BYTES || !aligned16(workspace))
        return NV_ERR_WORKSPACE;

    const int box_rows = block_size < kBN ? block_size : kBN;
    const int tq = kBM / group;
    CUtensorMap tq_map, tk, tv, to;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    if (!make_map(&tq_map, q, total_q, num_q_heads, group, tq) ||
        !make_map(&tk, k_cache, num_slots, num_kv_heads, 1, box_rows) ||
        !make_map(&tv, v_cache, num_slots, num_kv_heads, 1, box_rows) ||
        !make_map(&to, out, total_q, num_q_heads, group, 32 / group))
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
    p.num_kv_heads = num_kv_heads;
    p.num_seqs = num_seqs;
    p.scale_log2 = scale * nvkv::kLog2e;
    const int64_t total = (int64_t)p.max_tiles * num_seqs * num_kv_heads;
    if (total >= (1ll << 31))
        return NV_ERR_UNSUPPORTED;
    const int sms = sm_count();
    if (sms <= 0)
        return NV_ERR_CUDA;
    p.tile_counter = static_cast<int32_t *>(workspace);

    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (attr_err != cudaSuccess)
        return NV_ERR_CUDA;
    // persistent: one CTA per SM (shared memory and TMEM admit one); CTAs claim tiles of the
    // heaviest-first order from the counter in the workspace
    const int grid = (int)(total < sms ? total : sms);
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), (cudaStream_t)stream) != cudaSuccess)
        return NV_ERR_CUDA;
    paged_prefill_kernel<<<grid, kThreads, kSmemBytes, (cudaStream_t)stream>>>(tq_map, tk, tv, to, p);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}
