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
// is persistent (one CTA per SM): CTAs take tiles in work-list order (dealt round-robin, then
// claimed from a counter in the caller's workspace), and each CTA runs its tiles as one continuous
// stream of 128-key steps, so the next tile's first scores are computed while the current tile
// finishes.
//   * a one-CTA pre-pass lists the non-empty query tiles in the caller's workspace, sequence by
//     sequence (heaviest sequence first, each sequence's tiles heaviest first), so the CTAs at
//     work share a few sequences' K/V in L2.  The first three quarters of the claims are dealt
//     round-robin (CTA i takes i, i + grid, ...); the rest go to whichever CTA asks first, one
//     atomic add on a counter there each.
//   * warps 4 and 11 (TMA producers): warp 4 claims tiles and passes them to the other warps
//     through a small queue in shared memory, and copies each tile's Q (one 3-D tensor-map copy
//     per 64-dim half; dims head_dim, q head, token) into one of two Q buffers and its K tiles
//     (128 keys x 128 dims straight from the paged pool: dims head_dim, kv head, slot; 128-byte
//     swizzled) into a 3-slot K ring; warp 11 copies the V tiles into a 2-slot V ring, each as
//     soon as its slot is free, so a late K slot never holds up a V copy.  Lane i copies box i of
//     a step; the block-table row is held 32 entries at a time in the warp's registers.
//   * warps 5 and 6 (MMA issuers; warp 5 owns the TMEM allocation): one lane of warp 5 issues
//     S(n) = Q K(n)^T (operands in shared memory), one lane of warp 6 issues O += P(n) V(n)
//     (P read from tensor memory), tcgen05.mma kind::f16 with fp32 accumulators.  TMEM holds
//     THREE score buffers of 128 columns and the 128-column O accumulator; S(n) goes to buffer
//     n % 3, where the softmax then writes P(n) as bf16 pairs over the first half.  S(n) may be
//     issued as soon as PV(n-3) has freed its buffer.  The MMA issue queue is shallow, so any
//     latency in the issuing thread (barrier waits, commits, bookkeeping) idles the tensor pipe;
//     with two issuers one warp's waits overlap the other's MMAs (a single alternating issuer
//     measured 25% slower).  Operand descriptors are precomputed per buffer.
//   * warps 0-3 (softmax / correction): thread r owns row r = TMEM lane r.  It loads its 128
//     scores at once, masks only on steps that cross the diagonal (a separate code path), keeps
//     a base-2 online softmax with a lazy rescale (the running max moves only when a score beats
//     it by more than 8; only then is O rescaled in TMEM), and writes P with tcgen05.st.  At a
//     tile's end it hands the row sums to warps 7-10 and goes on with the next tile.
//   * warps 7-10 (epilogue; TMEM lane quarter = warp % 4): read O, normalise it, stage the bf16
//     rows in the tile's Q buffer (free once the last S has read it) and write them with
//     tensor-map stores.
// Measured on GB300: an M=128 K=16 tcgen05.mma fed back to back takes 64 cycles at N=128 and 48
// at N=64 (so key steps are 128 wide), and loading 128 fp32 scores from TMEM takes ~30 cycles.
// Every mbarrier wait is bounded; on timeout the kernel records NV_DERR_TIMEOUT and stops.
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "nv_common.cuh"
#include "tile_attention.cuh"

namespace {

using namespace nvkv;

constexpr int kD = 128;
constexpr int kBM = 128;             // rows per query tile (TMEM lanes)
constexpr int kBN = 128;             // keys per K/V tile
constexpr int kQBufs = 2;            // Q buffers: the next item's Q loads while this one runs
constexpr int kKSlots = 3;           // K ring slots
constexpr int kVSlots = 2;           // V ring slots
constexpr int kBufs = 3;             // score / P buffers in TMEM
// Warp roles: 0-3 softmax (warpgroup 0); 4 TMA producer of Q and K; 5 S = Q K^T issuer (owns TMEM);
// 6 O += P V issuer; 7-10 epilogue (TMEM lane quarter = warp % 4); 11 TMA producer of V.  Warpgroup 0 runs with more
// registers than the others (setmaxnreg); the split must add up to the launch budget.
constexpr int kThreads = 384;
constexpr int kWarpProducer = 4, kWarpS = 5, kWarpPV = 6, kWarpEpi0 = 7, kWarpEpiEnd = 11, kWarpVProducer = 11;
constexpr int kLaunchRegs = 168;                       // per thread at launch (checked on the host)
constexpr int kSoftmaxRegs = 200, kOtherRegs = 152;
static_assert(4 * kSoftmaxRegs + 8 * kOtherRegs == 12 * kLaunchRegs, "register split must match the launch");
constexpr uint32_t kTmemCols = 512;  // buffer b at b*128, O at 384
constexpr uint32_t kTmemO = 384;
constexpr float kRescaleLog2 = 8.0f;

constexpr uint32_t kHalf = 128 * 128;         // 128 rows x 64 dims bf16 (one swizzle atom wide) = 16 KB
constexpr uint32_t kTile = 2 * kHalf;         // a 128 x 128 bf16 operand = 32 KB
constexpr uint32_t kOffQ = 0;                 // Q buffer q at q*kTile (two: the next tile's Q loads early)
constexpr uint32_t kOffK = kQBufs * kTile;    // K slot s at kOffK + s*kTile
constexpr uint32_t kOffV = kOffK + kKSlots * kTile;
constexpr uint32_t kOffBar = kOffV + kVSlots * kTile;
constexpr int kBarQFull = 0;                       // + q buffer
constexpr int kBarQEmpty = 2;                      // + q buffer
constexpr int kBarKFull = 4;                       // + K slot
constexpr int kBarVFull = kBarKFull + kKSlots;     // + V slot
constexpr int kBarSFull = kBarVFull + kVSlots;     // + buffer (also: K slot of that S is free)
constexpr int kBarPFull = kBarSFull + kBufs;       // + buffer
constexpr int kBarODone = kBarPFull + kBufs;       // + buffer (PV(n) commits to n % 3; its V slot is free)
constexpr int kQueue = 8;                          // claimed work items in flight
constexpr int kItemInts = 12;                      // one work item in the shared-memory queue
constexpr int kBarOFree = kBarODone + kBufs;       // + item parity: the epilogue has read O (4 warps)
constexpr int kBarRowSum = kBarOFree + 2;          // + item parity: the softmax has written the row sums
constexpr int kBarItemFull = kBarRowSum + 2;       // + queue slot
constexpr int kBarItemEmpty = kBarItemFull + kQueue;
constexpr int kItemReaders = 2 + 4 + 4 + 1;        // S cursor, PV cursor, 4 softmax, 4 epilogue warps, V copies
constexpr int kBarDrain = kBarItemEmpty + kQueue;   // + issuer warp: its last MMAs, after a wait gave up
constexpr int kNumBars = kBarDrain + 2;
constexpr uint32_t kOffItems = kOffBar + kNumBars * 8;
constexpr uint32_t kOffRowSum = kOffItems + kQueue * kItemInts * 4;   // float [2 item parities][128 rows]
constexpr uint32_t kOffTmemSlot = kOffRowSum + 2 * 128 * 4;
// TMEM address, abort flag, then the copies the producers attempted (K, Q, V), for the drain
constexpr uint32_t kSmemBytes = kOffTmemSlot + 32 + 1024;      // + slack for 1024-byte alignment
static_assert(kSmemBytes <= 227u * 1024u, "shared memory per CTA");

struct PrefillParams {
    __nv_bfloat16 *out;
    const int32_t *block_tables;
    int32_t *d_err;
    int32_t bt_stride;
    int32_t num_q_heads;
    int32_t group;          // G
    int32_t group_shift;    // log2 G
    int32_t block_shift;    // log2 block_size
    int32_t box_rows;       // min(block_size, kBN)
    int32_t num_blocks;
    int32_t num_kv_heads;
    int32_t *ws;            // work list written by the pre-pass: [0] claim counter, [1] entries
    float scale_log2;
    // decode split over key ranges (split_steps > 0): an item of a sequence with more than
    // split_steps key steps writes unnormalised fp32 partials (O, and the row's max and sum in the
    // log2 domain) for a merge launch instead of bf16 rows
    int32_t split_steps;
    int32_t max_splits;
    float *part_o;          // [num_seqs, max_splits, num_q_heads, 128]
    float *part_ml;         // [num_seqs, max_splits, num_q_heads, 2]
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
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(s[2 * k], s[2 * k + 1]), scale2, negm2), x0, x1);
        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
        rs2[k & 3] = f2_add(rs2[k & 3], f2_pack(p0, p1));
        pk[k] = pack_bf16x2(p0, p1);
    }
    float ra, rb, rc, rd;
    f2_unpack(f2_add(rs2[0], rs2[1]), ra, rb);
    f2_unpack(f2_add(rs2[2], rs2[3]), rc, rd);
    return (ra + rb) + (rc + rd);
}

// One unit of work: a 128-row query tile of one (sequence, kv head).
struct Item {
    int v;                  // claim number; >= total marks the end of the work
    int b, kvh, cq0, Lq, P, i0, nq, kv_len, nkv, first_masked;
    int n0;                 // first key step (a decode split's key range starts there)
};

// ---------------------------------------------------------------------------------------
// Work list.  A one-CTA pre-pass lists every non-empty query tile of every sequence (all kv
// heads share an entry) in the workspace, validates the lengths, and sets up the claims: the first
// m rounds of grid-size claims (m = 3/4 of all claims / grid, at least 1) are static, CTA i taking
// i, i + grid, ..., i + (m-1) grid, and the counter starts at m * grid for the rest.  A claim from
// the counter is an atomic whose answer the producer warp waits for at the item boundary (~1,400
// cycles); the static rounds have none, and the dynamic last quarter still evens out the CTAs'
// finishing times, as the list runs heaviest first.
// The list runs sequence by sequence, heaviest sequence first (a counting sort on the key steps
// of its last tile), and within a sequence from its last (heaviest) tile to its first.  So the
// CTAs busy at any moment work on one or two sequences, whose K/V then stays in L2 while every
// tile of the sequence reads it (ordering all tiles by weight alone instead streamed the whole
// batch's K/V from HBM once per wave), and the lightest tiles still come last.  The main
// kernel's claim number v then names entry v / Hkv and kv head v % Hkv: a claim is at most one
// atomic add and one 32-byte record load, with no empty tiles to skip.
//   workspace ints: [0] claim counter, [1] entries, [2] static rounds m, [16 + 8e ...] entry e:
//   {b, cq0, Lq, P, i0, nq, kv_len, nkv}
// ---------------------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 8192;  // by 128-key steps; heavier tiles share the last bucket
constexpr int kPlanHeaderInts = 16;

struct PlanParams {
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *ctx;      // decode mode (cu_q, cu_k unused): context lengths, query row b = sequence b
    uint4 *out;              // decode mode: rows of sequences with no keys are zeroed here
    int32_t *ws;
    int32_t *d_err;
    int32_t num_seqs, total_q, bt_stride, block_shift, tq, max_tiles, cap;
    int32_t max_len;         // decode mode: longer contexts are truncated to this (NV_DERR_LENGTH)
    int32_t row_u4;          // decode mode: 16-byte words per output row
    int32_t split_steps;     // decode mode: key steps per entry (0: one entry per sequence)
    int32_t grid;            // CTAs of the main kernel
    int32_t num_kv_heads;    // claims per work-list entry
};

__device__ __forceinline__ bool plan_seq(const PlanParams &pp, int b, int &cq0, int &Lq, int &P, int &T)
{
    if (pp.ctx) {
        // decode: the sequence's one query (row b) sits at position L-1 and sees all L keys
        int L = pp.ctx[b];
        if (L < 0 || L > pp.max_len) {
            flag_error(pp.d_err, NV_DERR_LENGTH);
            L = L < 0 ? 0 : pp.max_len;
        }
        cq0 = b;
        Lq = L > 0 ? 1 : 0;
        P = L - Lq;
        const int steps = (L + kBN - 1) / kBN;
        T = L == 0 ? 0 : (pp.split_steps > 0 ? (steps + pp.split_steps - 1) / pp.split_steps : 1);
        return true;
    }
    cq0 = pp.cu_q[b];
    const int cq1 = pp.cu_q[b + 1];
    const int Lk = pp.cu_k[b + 1] - pp.cu_k[b];
    Lq = cq1 - cq0;
    P = Lk - Lq;
    if (Lq < 0 || P < 0 || cq0 < 0 || cq1 > pp.total_q ||
        ((Lk + (1 << pp.block_shift) - 1) >> pp.block_shift) > pp.bt_stride) {
        flag_error(pp.d_err, NV_DERR_LENGTH);
        return false;
    }
    const int nt = (Lq + pp.tq - 1) / pp.tq;
    if (nt > pp.max_tiles)
        flag_error(pp.d_err, NV_DERR_LENGTH);
    T = min(nt, pp.max_tiles);
    return true;
}

__device__ __forceinline__ int tile_steps(int P, int Lq, int i0, int tq)
{
    return (P + i0 + min(tq, Lq - i0) + kBN - 1) / kBN;
}

// A sequence's sort bucket: the key steps of its last listed tile (its heaviest); in decode mode
// the key steps of its first entry.
__device__ __forceinline__ int seq_bucket(const PlanParams &pp, int P, int Lq, int T, int tq)
{
    if (pp.ctx) {
        const int steps = (P + Lq + kBN - 1) / kBN;
        return min(pp.split_steps > 0 ? min(steps, pp.split_steps) : steps, kPlanBuckets - 1);
    }
    return min(tile_steps(P, Lq, (T - 1) * tq, tq), kPlanBuckets - 1);
}

__global__ void __launch_bounds__(kPlanThreads, 1) prefill_plan_kernel(const PlanParams pp)
{
    __shared__ int hist[kPlanBuckets];
    __shared__ int warp_tot[kPlanThreads / 32];
    __shared__ int count;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kPlanBuckets; i += kPlanThreads)
        hist[i] = 0;
    __syncthreads();
    // a thread per sequence: its tiles go to the bucket of its heaviest (last) tile's steps
    for (int b = tid; b < pp.num_seqs; b += kPlanThreads) {
        int cq0, Lq, P, T;
        if (plan_seq(pp, b, cq0, Lq, P, T) && T > 0)
            atomicAdd(&hist[seq_bucket(pp, P, Lq, T, pp.tq)], T);
    }
    __syncthreads();
    // exclusive prefix sum with the buckets in DESCENDING order: thread tid owns 8 of them
    constexpr int kPer = kPlanBuckets / kPlanThreads;
    int loc[kPer];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        loc[j] = hist[kPlanBuckets - 1 - (tid * kPer + j)];
        sum += loc[j];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        warp_tot[lane] = w;             // inclusive over warps
        if (lane == 31)
            count = w;
    }
    __syncthreads();
    int run = incl - sum + (warp > 0 ? warp_tot[warp - 1] : 0);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        hist[kPlanBuckets - 1 - (tid * kPer + j)] = run;
        run += loc[j];
    }
    __syncthreads();
    int4 *rec = reinterpret_cast<int4 *>(pp.ws + kPlanHeaderInts);
    // a warp per sequence: it takes a run of entries in its bucket and lists its tiles there, last
    // (heaviest) tile first
    for (int b = warp; b < pp.num_seqs; b += kPlanThreads / 32) {
        int cq0, Lq, P, T;
        if (!plan_seq(pp, b, cq0, Lq, P, T))
            continue;
        if (T == 0) {
            if (pp.ctx)      // decode: a row with no keys (graph padding) attends to nothing: zeros
                for (int i = lane; i < pp.row_u4; i += 32)
                    pp.out[(size_t)b * pp.row_u4 + i] = make_uint4(0, 0, 0, 0);
            continue;
        }
        int first = 0;
        if (lane == 0)
            first = atomicAdd(&hist[seq_bucket(pp, P, Lq, T, pp.tq)], T);
        first = __shfl_sync(0xffffffffu, first, 0);
        for (int t = lane; t < T; t += 32) {
            const int e = first + (T - 1 - t);
            if (e >= pp.cap)
                continue;
            rec[2 * e] = make_int4(b, cq0, Lq, P);
            if (pp.ctx && pp.split_steps > 0) {
                // decode split t: key steps n0 .. n0+nkv-1, packed as nkv | n0 << 16
                const int steps = (P + Lq + kBN - 1) / kBN;
                const int n0 = t * pp.split_steps;
                const int nkv = min(pp.split_steps, steps - n0);
                rec[2 * e + 1] = make_int4(0, 1, P + Lq, nkv | (n0 << 16));
            } else {
                const int i0 = t * pp.tq;
                const int nq = min(pp.tq, Lq - i0);
                rec[2 * e + 1] = make_int4(i0, nq, P + i0 + nq, tile_steps(P, Lq, i0, pp.tq));
            }
        }
    }
    if (tid == 0) {
        if (count > pp.cap)
            flag_error(pp.d_err, NV_DERR_LENGTH);
        const int entries = min(count, pp.cap);
        const long long claims = (long long)entries * pp.num_kv_heads;
        const int m = max(1, (int)(claims * 3 / 4 / pp.grid));
        pp.ws[0] = pp.grid * m;
        pp.ws[1] = entries;
        pp.ws[2] = m;
    }
}

// kRanges: work items may cover a range of key steps and write decode partials (the decode split);
// prefill runs the instantiation without, so none of it costs the prefill softmax anything.
template <bool kRanges>
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
    int total = 0;                                   // claims: work-list entries x kv heads (below)

    const uint32_t bar = base + kOffBar;
    auto BAR = [&](int i) { return bar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmemSlot);
    // Shared words after the TMEM address: [1] set by any warp whose bounded wait gave up (the CTA
    // then lets its copies and MMAs land before it frees tensor memory and leaves); [2..4] the copies
    // the producers attempted (K, Q, V), for that drain.  Addressed from `base`, so that no other
    // register stays live in every warp for them.
    auto word = [&](int i) { return base + kOffTmemSlot + 4u * (uint32_t)i; };
    auto st_word = [](uint32_t a, int v) { asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory"); };
    auto ld_word = [](uint32_t a) {
        int v;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
        return v;
    };
    auto give_up = [&]() {
        st_word(word(1), 1);
        flag_error(p.d_err, NV_DERR_TIMEOUT);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(kBarQFull + s), 1);
            mbar_init(BAR(kBarQEmpty + s), 1 + 4);     // last S of the item + the 4 epilogue warps
            mbar_init(BAR(kBarOFree + s), 4);
            mbar_init(BAR(kBarRowSum + s), 4);
        }
        for (int s = 0; s < kKSlots; ++s) {
            mbar_init(BAR(kBarKFull + s), 1);
        }
        for (int s = 0; s < kVSlots; ++s) {
            mbar_init(BAR(kBarVFull + s), 1);
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
        mbar_init(BAR(kBarDrain), 1);
        mbar_init(BAR(kBarDrain + 1), 1);
        for (int i = 1; i <= 4; ++i)
            st_word(word(i), 0);
        fence_barrier_init();
    }
    // Work items pass from the producer (which claims them) to the MMA issuer's two cursors and
    // the four softmax warps through a small queue in shared memory.
    volatile int *items = reinterpret_cast<volatile int *>(smem + kOffItems);
    auto read_item = [&](int k, Item &it) {          // whole warp calls; lane 0 releases the slot
        if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBarItemFull + k % kQueue), (k / kQueue) & 1)))
            return false;
        volatile int *q = items + (k % kQueue) * kItemInts;
        it.v = q[0];
        it.b = q[1];
        it.kvh = q[2];
        it.cq0 = q[3];
        it.Lq = q[4];
        it.P = q[5];
        it.i0 = q[6];
        it.nq = q[7];
        it.kv_len = q[8];
        it.nkv = q[9];
        it.first_masked = q[10];
        it.n0 = q[11];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(BAR(kBarItemEmpty + k % kQueue));
        return true;
    };
    auto first_step = [](const Item &x) {           // an item's first key step (0 without ranges)
        if constexpr (kRanges)
            return x.n0;
        else
            return 0;
    };
    if (warp == kWarpS) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The work list comes from the pre-pass launched just before; this kernel is its programmatic
    // dependent, so the setup above overlapped it.
    if (warp == kWarpProducer && lane == 0) {    // kernel parameters: fetch them during the pre-pass
        prefetch_tmap(&tmap_q);
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        prefetch_tmap(&tmap_o);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    total = p.ws[1] * p.num_kv_heads;
    if (warp < 4) {
        warpgroup_reg_alloc<kSoftmaxRegs>();
        // ======================= softmax / correction (warps 0-3) =======================
        const int r = threadIdx.x;                      // tile row == TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t o_addr = tmem + lane_base + kTmemO;
        volatile float *rowsum = reinterpret_cast<volatile float *>(smem + kOffRowSum);
        Item it;
        bool ok = true;
        int g = 0;                                      // global key tile
        for (int k = 0; ok; ++k) {
            if (!read_item(k, it)) {
                ok = false;
                break;
            }
            if (it.v >= total)
                break;
            const int tok = it.i0 + (r >> p.group_shift);   // token index inside the chunk
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
                const int rel = lim - (first_step(it) + n) * kBN;   // keys j <= rel of this tile are visible
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
                ok = first_step(it) + n < it.first_masked ? tile(n, std::false_type{}) : tile(n, std::true_type{});
            if (!ok)
                break;
            // Hand the row sums to the epilogue warps and go on with the next item at once.  The
            // sums of item k share a buffer with item k-2's, which that epilogue must have read.
            if (k >= 2 && !__all_sync(0xffffffffu, mbar_wait(BAR(kBarOFree + (k & 1)), ((k - 2) >> 1) & 1))) {
                ok = false;
                break;
            }
            rowsum[(k & 1) * 128 + r] = l_run;
            if constexpr (kRanges) {
                if (it.kv_len > p.split_steps * kBN && tok < it.Lq) {
                    // a decode split: the row's (max, sum) go straight to the partials (O follows from
                    // the epilogue)
                    const size_t unit = (size_t)it.b * p.max_splits + it.n0 / p.split_steps;
                    const int head = it.kvh * p.group + (r & (p.group - 1));
                    *reinterpret_cast<float2 *>(p.part_ml + (unit * p.num_q_heads + head) * 2) =
                        make_float2(m_run, l_run);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(BAR(kBarRowSum + (k & 1)));
        }
        if (!ok && lane == 0)
            give_up();
    } else {
        warpgroup_reg_dealloc<kOtherRegs>();
        // this lane's box of key tile n of an item (its first pool slot, -1 = none); the block-table
        // row is held 32 entries at a time in the warp's registers (win, from entry win_base)
        const int bs_mask = (1 << p.block_shift) - 1;
        const int boxes = kBN / p.box_rows;
        auto box_slot = [&](const Item &it, int n, const int32_t *bt, int nblk, int &win_base, int &win) {
            const int lb0 = ((first_step(it) + n) * kBN) >> p.block_shift;
            const int lb_hi = min(lb0 + boxes - 1, nblk - 1);
            if (lb_hi >= win_base + 32) {               // warp-uniform window move
                win_base = lb0;
                win = win_base + lane < nblk ? __ldg(bt + win_base + lane) : -1;
            }
            const int j0 = (first_step(it) + n) * kBN + lane * p.box_rows;
            const int lb = j0 >> p.block_shift;
            const int blk = __shfl_sync(0xffffffffu, win, (lb - win_base) & 31);
            int slot = -1;
            if (lane < boxes && j0 < it.kv_len) {
                if (blk < 0 || blk >= p.num_blocks)
                    flag_error(p.d_err, NV_DERR_BLOCK_RANGE);
                else
                    slot = (blk << p.block_shift) + (j0 & bs_mask);
            }
            return slot;
        };
        // copy one K or V tile (global key tile idx) into its ring; the slot's previous tile
        // (idx - slots) is free once its MMA group has completed: S for K, PV for V, whose commits
        // to the score-buffer barriers already signal that.  Lane kb copies box kb (box_rows keys,
        // both 64-dim halves).
        auto copy_tile = [&](bool is_v, int idx, int kvh, int slot) {
            const int n_slots = is_v ? kVSlots : kKSlots;
            const int s_ = idx % n_slots;
            const uint32_t full = BAR((is_v ? kBarVFull : kBarKFull) + s_);
            const int prev = idx - n_slots;
            if (prev >= 0 &&
                !__all_sync(0xffffffffu,
                            mbar_wait(BAR((is_v ? kBarODone : kBarSFull) + prev % kBufs), (prev / kBufs) & 1)))
                return false;
            const uint32_t bytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, slot >= 0)) * p.box_rows * 256u;
            const uint32_t dst = base + (is_v ? kOffV : kOffK) + s_ * kTile + (uint32_t)lane * p.box_rows * 128u;
            if (lane == 0)
                mbar_arrive_expect_tx(full, bytes);
            __syncwarp();
            if (slot >= 0) {
                const CUtensorMap *map = is_v ? &tmap_v : &tmap_k;
                tma_load_3d(dst, map, 0, kvh, slot, full);
                tma_load_3d(dst + kHalf, map, 64, kvh, slot, full);
            }
            return true;
        };
        if (warp == kWarpProducer) {
            // ====================== TMA producer: work items, Q and K ======================
            // Claims items and queues them; copies each item's Q tile (one 3-D tensor-map copy
            // per 64-dim half) into one of two Q buffers just before the item's first K tile, and
            // its K tiles into the K ring as the S issuer frees the slots.
            bool ok = true;
            int j = 0;                                  // global key tile of the next K copy
            // Item k+1's claim is known as item k starts: CTA index + (k+1) * grid for the first
            // m_static items, else the counter's answer, which lane 0 asks for then and which travels
            // while item k's copies are issued.
            const int4 *plan = reinterpret_cast<const int4 *>(p.ws + kPlanHeaderInts);
            int pending = (int)blockIdx.x;
            const int m_static = p.ws[2];
            for (int k = 0; ok; ++k) {
                // item k: its claim number, then its work-list entry (lanes 0-1 load the two halves)
                if (k >= kQueue &&
                    !__all_sync(0xffffffffu, mbar_wait(BAR(kBarItemEmpty + k % kQueue), ((k / kQueue) - 1) & 1))) {
                    ok = false;
                    break;
                }
                const int v = __shfl_sync(0xffffffffu, pending, 0);
                if (k + 1 < m_static)
                    pending = v + (int)gridDim.x;
                else if (lane == 0 && v < total)
                    pending = atomicAdd(p.ws, 1);
                Item it{};
                it.v = v < total ? v : total;
                if (v < total) {
                    const int e = v / p.num_kv_heads;
                    int4 r = make_int4(0, 0, 0, 0);
                    if (lane < 2)
                        r = plan[2 * e + lane];
                    it.b = __shfl_sync(0xffffffffu, r.x, 0);
                    it.cq0 = __shfl_sync(0xffffffffu, r.y, 0);
                    it.Lq = __shfl_sync(0xffffffffu, r.z, 0);
                    it.P = __shfl_sync(0xffffffffu, r.w, 0);
                    it.i0 = __shfl_sync(0xffffffffu, r.x, 1);
                    it.nq = __shfl_sync(0xffffffffu, r.y, 1);
                    it.kv_len = __shfl_sync(0xffffffffu, r.z, 1);
                    it.nkv = __shfl_sync(0xffffffffu, r.w, 1);
                    it.n0 = 0;
                    if constexpr (kRanges) {        // decode split: nkv | n0 << 16
                        it.n0 = it.nkv >> 16;
                        it.nkv &= 0xFFFF;
                    }
                    it.kvh = v - e * p.num_kv_heads;
                    it.first_masked = (it.P + it.i0 + 1) / kBN;
                }
                if (lane == 0) {
                    volatile int *q = items + (k % kQueue) * kItemInts;
                    q[0] = it.v;
                    q[1] = it.b;
                    q[2] = it.kvh;
                    q[3] = it.cq0;
                    q[4] = it.Lq;
                    q[5] = it.P;
                    q[6] = it.i0;
                    q[7] = it.nq;
                    q[8] = it.kv_len;
                    q[9] = it.nkv;
                    q[10] = it.first_masked;
                    q[11] = it.n0;
                    mbar_arrive(BAR(kBarItemFull + k % kQueue));
                }
                if (v >= total)
                    break;
                const int32_t *bt = p.block_tables + (size_t)it.b * p.bt_stride;
                const int nblk = (it.kv_len + (1 << p.block_shift) - 1) >> p.block_shift;
                int win_base = 0;
                int win = lane < nblk ? __ldg(bt + lane) : -1;
                for (int n = 0; n < it.nkv && ok; ++n, ++j) {
                    const int slot = box_slot(it, n, bt, nblk, win_base, win);
                    if (n == 0) {
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
                        if (lane == 0)
                            st_word(word(3), k + 1);
                    }
                    ok = copy_tile(false, j, it.kvh, slot);
                }
            }
            if (lane == 0)
                st_word(word(2), j);    // K copies attempted (after a wait gave up: one more than issued)
            if (!ok && lane == 0)
                give_up();
        } else if (warp == kWarpVProducer) {
            // ========================= TMA producer: V =========================
            // Copies each item's V tiles into the V ring as soon as the PV issuer frees a slot,
            // independently of the K stream.
            bool ok = true;
            int j = 0;                                  // global key tile of the next V copy
            Item it;
            for (int k = 0; ok; ++k) {
                if (!read_item(k, it)) {
                    ok = false;
                    break;
                }
                if (it.v >= total)
                    break;
                const int32_t *bt = p.block_tables + (size_t)it.b * p.bt_stride;
                const int nblk = (it.kv_len + (1 << p.block_shift) - 1) >> p.block_shift;
                int win_base = 0;
                int win = lane < nblk ? __ldg(bt + lane) : -1;
                for (int n = 0; n < it.nkv && ok; ++n, ++j)
                    ok = copy_tile(true, j, it.kvh, box_slot(it, n, bt, nblk, win_base, win));
            }
            if (lane == 0)
                st_word(word(4), j);    // as for K
            if (!ok && lane == 0)
                give_up();
        } else if (warp == kWarpS || warp == kWarpPV) {
            // ============================ MMA issuer(s) ============================
            // Key steps of all this CTA's work items form one global sequence g.  S(g) goes to TMEM
            // buffer g % 3 once PV(g-3) has finished with it; both streams run across tile
            // boundaries, so the next tile's first scores are computed during the current tile's last
            // softmax.
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
                    if (!read_item(c.k, c.it)) {
                        ok = false;
                        c.it.v = total;
                    }
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
                // Keys past the sequence carry P = 0, but their V rows may hold anything (NaN patterns
                // included) and 0 * NaN would poison O: zero them.  (Skipping their k-steps instead
                // measured slower.)
                const int vrows = min(c.it.kv_len - (first_step(c.it) + n) * kBN, kBN);
                if (vrows < kBN) {
                    for (int c2 = lane; c2 < (kBN - vrows) * 16; c2 += 32)     // 16-byte chunk: row, half, column
                        sts_u4(vtile + ((c2 >> 3) & 1) * kHalf + (uint32_t)(vrows + (c2 >> 4)) * 128u +
                                   (uint32_t)(c2 & 7) * 16u,
                               make_uint4(0, 0, 0, 0));
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (!wait_all(BAR(kBarPFull + bb), (g / kBufs) & 1))
                    return;
                // an item's first PV overwrites O: the previous item's epilogue must have read it
                if (n == 0 && c.k > 0 && !wait_all(BAR(kBarOFree + ((c.k - 1) & 1)), ((c.k - 1) >> 1) & 1))
                    return;
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t dv = desc_v0 + (uint64_t)(slot * (kTile >> 4));
    #pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)      // k-step kk: keys 16kk.. = 16 rows of 128 bytes
                        mma_bf16_ts(tmem + kTmemO, tmem + bb * 128 + kk * 8, dv + (uint64_t)(kk * 16 * 128 >> 4),
                                    idesc_o, (n > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(BAR(kBarODone + bb));
                }
                __syncwarp();
                advance(c);
            };
            // each warp streams its own groups; S(g) goes as soon as PV(g-3) has freed its buffer
            if (warp == kWarpS) {
                while (ready(cs))
                    issue_s(cs);
            } else {
                while (ready(cp))
                    issue_pv(cp);
            }
            if (!ok && lane == 0)
                give_up();
        } else if (warp >= kWarpEpi0 && warp < kWarpEpiEnd) {
            // ============================ epilogue (warps 7-10) ============================
            // Item by item: wait for the softmax's row sums and the item's last PV, read O from TMEM
            // (then the next item's PVs may overwrite it), normalise, round to bf16, stage the rows in
            // the item's Q buffer (every S of the item has read it by then; same 128-byte swizzled
            // layout as the Q tile, row r = TMEM lane r) and write each warp's 32 rows with one tensor
            // store per 64-dim half.  A warp whose rows run past the chunk's end (the ragged last tile)
            // stores its valid rows directly instead, so it never touches the next sequence.
            const int r = (warp & 3) * 32 + lane;           // tile row == TMEM lane
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t o_addr = tmem + lane_base + kTmemO;
            const volatile float *rowsum = reinterpret_cast<const volatile float *>(smem + kOffRowSum);
            Item it;
            bool ok = true;
            int g = 0;                                      // global key step
            for (int k = 0; ok; ++k) {
                if (!read_item(k, it)) {
                    ok = false;
                    break;
                }
                if (it.v >= total)
                    break;
                g += it.nkv;
                const int last = g - 1;
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBarRowSum + (k & 1)), (k >> 1) & 1)) ||
                    !__all_sync(0xffffffffu, mbar_wait(BAR(kBarODone + last % kBufs), (last / kBufs) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int tok = it.i0 + (r >> p.group_shift);
                const int head = it.kvh * p.group + (r & (p.group - 1));
                const bool valid = tok < it.Lq;
                const float l_row = rowsum[(k & 1) * 128 + r];
                if (kRanges && it.kv_len > p.split_steps * kBN) {
                    // a decode split: unnormalised O goes to the partials (the softmax wrote the row's
                    // max and sum)
                    const size_t unit = (size_t)it.b * p.max_splits + it.n0 / p.split_steps;
                    float *po = p.part_o + (unit * p.num_q_heads + head) * kD;
#pragma unroll
                    for (int c = 0; c < kD / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(o_addr + c * 32, v);
                        tmem_wait_ld();
                        if (valid) {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                reinterpret_cast<float4 *>(po + c * 32)[j] =
                                    make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(BAR(kBarOFree + (k & 1)));   // O and this item's row sums are read
                        mbar_arrive(BAR(kBarQEmpty + k % kQBufs));   // its Q buffer was not used for staging
                    }
                    continue;
                }
                const float inv = (valid && l_row > 0.f) ? 1.f / l_row : 0.f;
                // O -> registers as bf16 pairs, 32 columns at a time
                uint32_t ob[kD / 2];
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(o_addr + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        ob[c * 16 + j] = pack_bf16x2(__uint_as_float(v[2 * j]) * inv, __uint_as_float(v[2 * j + 1]) * inv);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(BAR(kBarOFree + (k & 1)));  // O and this item's row sums are read
                const bool warp_full = __all_sync(0xffffffffu, valid);
                const int qb = k % kQBufs;
                const uint32_t stage = base + kOffQ + qb * kTile;
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((size_t)(it.cq0 + tok) * p.num_q_heads + head) * kD);
#pragma unroll
                for (int chunk = 0; chunk < kD / 8; ++chunk) {     // 16-byte chunk of the 256-byte row
                    const uint4 w = make_uint4(ob[4 * chunk], ob[4 * chunk + 1], ob[4 * chunk + 2], ob[4 * chunk + 3]);
                    if (warp_full)
                        sts_u4(stage + (chunk >> 3) * kHalf + (uint32_t)r * 128u +
                                   ((uint32_t)((chunk & 7) ^ (r & 7)) << 4),
                               w);
                    else if (valid)
                        dst[chunk] = w;
                }
                if (warp_full) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int row0 = it.cq0 + it.i0 + (((warp & 3) * 32) >> p.group_shift);
                        for (int h = 0; h < 2; ++h)
                            tma_store_3d(&tmap_o, stage + h * kHalf + (warp & 3) * 4096, h * 64, it.kvh * p.group, row0);
                        bulk_commit_group();
                        bulk_wait_group_read0();            // the staging buffer goes back to the producer
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(BAR(kBarQEmpty + qb));
            }
            if (!ok && lane == 0)
                give_up();
        }
    }

    // ---------------- teardown: every TMEM access is done before the free ----------------
    // On the normal path every copy and MMA this CTA issued has been waited for by the warp that
    // consumes it.  After a wait gave up that no longer holds: copies may still be landing in shared
    // memory and MMAs still reading it and writing tensor memory.  So each producer waits for the
    // copies it attempted last (one per ring slot: all earlier ones were consumed, or their slot
    // reused after they landed; a copy whose slot wait gave up was never issued, and its wait here
    // just runs out), each issuing thread commits its MMAs to a barrier of its own and waits for it,
    // and only then is tensor memory freed and the CTA's shared memory released.  Every wait is
    // bounded as usual.
    tc_fence_before();
    __syncthreads();
    if (ld_word(word(1))) {
        if (lane == 0) {
            if (warp == kWarpProducer) {
                const int nk = ld_word(word(2)), nq = ld_word(word(3));
                for (int i = max(0, nk - kKSlots); i < nk; ++i)
                    mbar_wait(BAR(kBarKFull + i % kKSlots), (i / kKSlots) & 1);
                for (int i = max(0, nq - kQBufs); i < nq; ++i)
                    mbar_wait(BAR(kBarQFull + i % kQBufs), (i / kQBufs) & 1);
            } else if (warp == kWarpVProducer) {
                const int nv = ld_word(word(4));
                for (int i = max(0, nv - kVSlots); i < nv; ++i)
                    mbar_wait(BAR(kBarVFull + i % kVSlots), (i / kVSlots) & 1);
            } else if (warp == kWarpS || warp == kWarpPV) {
                mma_commit(BAR(kBarDrain + (warp - kWarpS)));
                mbar_wait(BAR(kBarDrain + (warp - kWarpS)), 0);
            }
        }
        tc_fence_before();
        __syncthreads();
    }
    if (warp == kWarpS) {
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

namespace {
// Upper bound on the work list's entries: sum_b ceil(Lq_b / tq) <= ceil(total_q / tq) + num_seqs,
// and no sequence lists more than ceil(max_seqlen_q / tq) tiles.
int64_t prefill_entries_cap(int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q, int group)
{
    const int64_t tq = kBM / group;
    const int64_t a = (total_q + tq - 1) / tq + num_seqs;
    const int64_t b = (int64_t)num_seqs * ((max_seqlen_q + tq - 1) / tq);
    return a < b ? a : b;
}
size_t prefill_workspace_bytes(int64_t cap)
{
    return (size_t)kPlanHeaderInts * 4u + (size_t)cap * 32u;
}
}  // namespace

size_t nvkv_host::tile_workspace_bytes(int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q, int group)
{
    return prefill_workspace_bytes(prefill_entries_cap(num_seqs, total_q, max_seqlen_q, group));
}

extern "C" size_t nv_paged_prefill_workspace_size(int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                                                  int32_t num_q_heads, int32_t num_kv_heads)
{
    if (num_seqs <= 0 || total_q <= 0 || max_seqlen_q <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0)
        return (size_t)kPlanHeaderInts * 4u;
    const int group = num_q_heads / num_kv_heads;
    if (group > kBM)
        return (size_t)kPlanHeaderInts * 4u;
    return prefill_workspace_bytes(prefill_entries_cap(num_seqs, total_q, max_seqlen_q, group));
}

int nvkv_host::tile_attention(const TileAttnArgs &a)
{
    using namespace nvkv_host;
    const int num_q_heads = a.num_q_heads, num_kv_heads = a.num_kv_heads, block_size = a.block_size;
    const int num_seqs = a.num_seqs, total_q = a.total_q, max_seqlen_q = a.max_seqlen_q, num_blocks = a.num_blocks;
    const int group = num_q_heads / num_kv_heads;
    if (!is_pow2(group) || group > 16 || num_kv_heads > 65535)
        return NV_ERR_UNSUPPORTED;
    if (!is_pow2(block_size) || block_size < 16 || block_size > 256)
        return NV_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * block_size >= (1ll << 31) || num_seqs > 65535)
        return NV_ERR_UNSUPPORTED;
    if (!aligned16(a.q) || !aligned16(a.k_cache) || !aligned16(a.v_cache) || !aligned16(a.out))
        return NV_ERR_ALIGN;
    if (num_blocks == 0)
        return NV_ERR_SHAPE;
    const bool split = a.context_lens && a.split_steps > 0;
    if (split && (a.split_steps >= (1 << 16) || (int64_t)a.max_splits * a.split_steps >= (1 << 15) ||
                  !a.part_o || !a.part_ml))
        return NV_ERR_UNSUPPORTED;    // an entry packs its step count and first step in 16 bits each
    const int64_t cap = split ? (int64_t)num_seqs * a.max_splits
                              : prefill_entries_cap(num_seqs, total_q, max_seqlen_q, group);
    if (cap * num_kv_heads >= (1ll << 31))
        return NV_ERR_UNSUPPORTED;
    if (!a.workspace || a.workspace_bytes < prefill_workspace_bytes(cap) || !aligned16(a.workspace))
        return NV_ERR_WORKSPACE;

    const int box_rows = block_size < kBN ? block_size : kBN;
    const int tq = kBM / group;
    CUtensorMap tq_map, tk, tv, to;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    if (!make_map(&tq_map, a.q, total_q, num_q_heads, group, tq) ||
        !make_map(&tk, a.k_cache, num_slots, num_kv_heads, 1, box_rows) ||
        !make_map(&tv, a.v_cache, num_slots, num_kv_heads, 1, box_rows) ||
        !make_map(&to, a.out, total_q, num_q_heads, group, 32 / group))
        return NV_ERR_CUDA;

    PrefillParams p{};
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.block_tables = a.block_tables;
    p.d_err = a.d_err;
    p.bt_stride = a.bt_stride;
    p.num_q_heads = num_q_heads;
    p.group = group;
    p.group_shift = ilog2(group);
    p.block_shift = ilog2(block_size);
    p.box_rows = box_rows;
    p.num_blocks = num_blocks;
    p.num_kv_heads = num_kv_heads;
    p.scale_log2 = a.scale * nvkv::kLog2e;
    p.ws = static_cast<int32_t *>(a.workspace);
    p.split_steps = split ? a.split_steps : 0;
    p.max_splits = split ? a.max_splits : 0;
    p.part_o = a.part_o;
    p.part_ml = a.part_ml;

    PlanParams pp{};
    pp.cu_q = a.cu_seqlens_q;
    pp.cu_k = a.cu_seqlens_k;
    pp.ctx = a.context_lens;
    pp.out = static_cast<uint4 *>(a.out);
    pp.ws = p.ws;
    pp.d_err = a.d_err;
    pp.num_seqs = num_seqs;
    pp.total_q = total_q;
    pp.bt_stride = a.bt_stride;
    pp.block_shift = p.block_shift;
    pp.tq = tq;
    pp.max_tiles = (max_seqlen_q + tq - 1) / tq;
    pp.cap = (int32_t)cap;
    pp.max_len = a.max_len;
    pp.row_u4 = num_q_heads * kD / 8;
    pp.split_steps = p.split_steps;
    const int sms = sm_count();
    if (sms <= 0)
        return NV_ERR_CUDA;
    // Once per device (the shared-memory opt-in is a per-device attribute): set it, and check that
    // the warpgroups' register split (setmaxnreg) adds up to exactly the launch budget -- a build
    // whose per-thread register count differs is refused rather than launched, since a warpgroup
    // would wait for registers that never come.
    static std::mutex attr_mu;
    static int attr_state[64];          // 0 not yet, 1 ready, NV_ERR_* the refusal
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return NV_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(attr_mu);
        if (attr_state[dev] == 0) {
            int st = 1;
            for (const void *f : {(const void *)paged_prefill_kernel<false>, (const void *)paged_prefill_kernel<true>}) {
                cudaFuncAttributes fa{};
                if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess ||
                    cudaFuncGetAttributes(&fa, f) != cudaSuccess) {
                    st = NV_ERR_CUDA;
                    break;
                }
                if (fa.numRegs != kLaunchRegs)
                    st = NV_ERR_UNSUPPORTED;
            }
            if (st == NV_ERR_CUDA)
                return st;              // not cached: the next call tries again
            attr_state[dev] = st;
        }
        if (attr_state[dev] != 1)
            return attr_state[dev];
    }
    // persistent: one CTA per SM (shared memory and TMEM admit one); CTAs claim the work list's
    // entries in order
    const int64_t claims = cap * num_kv_heads;
    const int grid = (int)(claims < sms ? claims : sms);
    pp.grid = grid;
    pp.num_kv_heads = num_kv_heads;
    prefill_plan_kernel<<<1, kPlanThreads, 0, a.stream>>>(pp);
    // launched as a programmatic dependent of the pre-pass: its CTAs set up (barriers, TMEM, tensor
    // maps) while the pre-pass runs, and wait for the work list with griddepcontrol.wait
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le = split ? cudaLaunchKernelEx(&cfg, paged_prefill_kernel<true>, tq_map, tk, tv, to, p)
                                 : cudaLaunchKernelEx(&cfg, paged_prefill_kernel<false>, tq_map, tk, tv, to, p);
    if (le != cudaSuccess)
        return NV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

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
    TileAttnArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.cu_seqlens_q = cu_seqlens_q;
    a.cu_seqlens_k = cu_seqlens_k;
    a.block_tables = block_tables;
    a.bt_stride = bt_stride;
    a.num_seqs = num_seqs;
    a.total_q = total_q;
    a.max_seqlen_q = max_seqlen_q;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.out = out;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.d_err = d_err;
    a.stream = (cudaStream_t)stream;
    return tile_attention(a);
}
