// nv_prepare_decode / nv_prepare_prefill: the attention metadata, built on the device.
//
// What they compute is the model runner's prepare_decode and prepare_prefill (nano-vLLM field
// guide, Steps 07.5, 07.6 and the graph-replay padding of 07.8), from per-sequence lengths and the
// block tables already on the GPU, so a step needs no host-built tensors and no pinned copies:
//   decode:  context_len = len(seq), position = len - 1, slot = the slot of position len - 1
//            (the last block's base slot + last_block_num_tokens - 1); padded rows: slot -1,
//            context 0, position 0.
//   prefill: sequence b schedules positions [num_cached, num_cached + num_scheduled);
//            cu_seqlens_q / cu_seqlens_k are running sums of num_scheduled and of the end
//            position; max_seqlens = {max seqlen_q, max seqlen_k}; each new token's slot is the
//            slot of its position (the pages walk the touched blocks; the slots are the same).
//
// How: decode is one thread per row.  Prefill is two launches: one CTA scans the lengths (running
// sums in chunks of 1024 with a warp-shuffle scan, the maxima by reduction), then one thread per
// new token finds its sequence by binary search in cu_seqlens_q and writes its position and slot.
#include "nv_common.cuh"

namespace {

using namespace nvkv;

__global__ void __launch_bounds__(256) prepare_decode_kernel(const int32_t *seq_lens, const int32_t *block_tables,
                                                             int32_t bt_stride, int32_t num_seqs, int32_t padded,
                                                             int32_t block_shift, int32_t num_blocks,
                                                             int32_t *context_lens, int32_t *positions,
                                                             int32_t *slot_mapping, int32_t *d_err)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= padded)
        return;
    int32_t cl = 0, pos = 0, slot = -1;
    if (b < num_seqs) {
        const int32_t len = __ldg(seq_lens + b);
        const int32_t bs = 1 << block_shift;
        const int32_t nblocks = len >= 1 ? ((len - 1) >> block_shift) + 1 : 0;
        if (len < 1 || nblocks > bt_stride) {
            flag_error(d_err, NV_DERR_LENGTH);
        } else {
            const int32_t blk = __ldg(block_tables + (int64_t)b * bt_stride + nblocks - 1);
            if (blk < 0 || blk >= num_blocks) {
                flag_error(d_err, NV_DERR_BLOCK_RANGE);
            } else {
                cl = len;
                pos = len - 1;
                slot = blk * bs + (len - (nblocks - 1) * bs) - 1;   // last block base + tokens in it - 1
            }
        }
    }
    context_lens[b] = cl;
    positions[b] = pos;
    slot_mapping[b] = slot;
}

// Inclusive scan of one value per thread over a 1024-thread block (warp shuffles + one smem step).
__device__ __forceinline__ int block_scan_incl(int v, int *warp_sums)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += y;
    }
    if (lane == 31)
        warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int r = v + (warp > 0 ? warp_sums[warp - 1] : 0);
    __syncthreads();            // warp_sums is reused by the next call
    return r;
}

__global__ void __launch_bounds__(1024) prepare_prefill_scan_kernel(const int32_t *num_cached,
                                                                    const int32_t *num_scheduled, int32_t num_seqs,
                                                                    int32_t *cu_seqlens_q, int32_t *cu_seqlens_k,
                                                                    int32_t *max_seqlens, int32_t *d_err)
{
    __shared__ int warp_sums[32];
    __shared__ int red[2][32];
    int carry_q = 0, carry_k = 0, mq = 0, mk = 0;
    bool bad = false;
    if (threadIdx.x == 0) {
        cu_seqlens_q[0] = 0;
        cu_seqlens_k[0] = 0;
    }
    for (int base = 0; base < num_seqs; base += 1024) {
        const int b = base + threadIdx.x;
        int sq = 0, end = 0;
        if (b < num_seqs) {
            const int start = __ldg(num_cached + b);
            sq = __ldg(num_scheduled + b);
            if (start < 0 || sq < 0) {
                bad = true;
                sq = max(sq, 0);
            }
            end = max(start, 0) + sq;
            mq = max(mq, sq);
            mk = max(mk, end);
        }
        const int iq = block_scan_incl(sq, warp_sums);
        const int ik = block_scan_incl(end, warp_sums);
        if (b < num_seqs) {
            cu_seqlens_q[b + 1] = carry_q + iq;
            cu_seqlens_k[b + 1] = carry_k + ik;
        }
        // the chunk's totals, from its last thread, to every thread
        __shared__ int tot[2];
        if (threadIdx.x == 1023) {
            tot[0] = iq;
            tot[1] = ik;
        }
        __syncthreads();
        carry_q += tot[0];
        carry_k += tot[1];
        __syncthreads();
    }
    if (bad)
        flag_error(d_err, NV_DERR_LENGTH);
    // maxima
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mq = max(mq, __shfl_xor_sync(0xffffffffu, mq, o));
        mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    }
    if ((threadIdx.x & 31) == 0) {
        red[0][threadIdx.x >> 5] = mq;
        red[1][threadIdx.x >> 5] = mk;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        mq = red[0][threadIdx.x];
        mk = red[1][threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mq = max(mq, __shfl_xor_sync(0xffffffffu, mq, o));
            mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, o));
        }
        if (threadIdx.x == 0) {
            max_seqlens[0] = mq;
            max_seqlens[1] = mk;
        }
    }
}

__global__ void __launch_bounds__(256) prepare_prefill_fill_kernel(const int32_t *num_cached,
                                                                   const int32_t *block_tables, int32_t bt_stride,
                                                                   int32_t num_seqs, int32_t total_q,
                                                                   int32_t block_shift, int32_t num_blocks,
                                                                   const int32_t *cu_seqlens_q, int32_t *positions,
                                                                   int32_t *slot_mapping, int32_t *d_err)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t == 0 && __ldg(cu_seqlens_q + num_seqs) != total_q)
        flag_error(d_err, NV_DERR_LENGTH);      // the lengths do not add up to the caller's total
    if (t >= total_q)
        return;
    int32_t pos = 0, slot = -1;
    if (t < __ldg(cu_seqlens_q + num_seqs)) {
        // the sequence whose new tokens contain t: the last b with cu_seqlens_q[b] <= t
        int lo = 0, hi = num_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(cu_seqlens_q + mid) <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int b = lo;
        pos = max(__ldg(num_cached + b), 0) + (t - __ldg(cu_seqlens_q + b));
        const int lb = pos >> block_shift;
        if (lb >= bt_stride) {
            flag_error(d_err, NV_DERR_LENGTH);
        } else {
            const int32_t blk = __ldg(block_tables + (int64_t)b * bt_stride + lb);
            if (blk < 0 || blk >= num_blocks)
                flag_error(d_err, NV_DERR_BLOCK_RANGE);
            else
                slot = (blk << block_shift) + (pos & ((1 << block_shift) - 1));
        }
    }
    positions[t] = pos;
    slot_mapping[t] = slot;
}

}  // namespace

extern "C" int nv_prepare_decode(const int32_t *seq_lens, const int32_t *block_tables, int32_t bt_stride,
                                 int32_t num_seqs, int32_t padded_seqs, int32_t block_size, int32_t num_blocks,
                                 int32_t *context_lens, int32_t *positions, int32_t *slot_mapping, int32_t *d_err,
                                 nv_stream_t stream)
{
    using namespace nvkv_host;
    if (num_seqs < 0 || padded_seqs < num_seqs || bt_stride <= 0 || num_blocks < 0)
        return NV_ERR_SHAPE;
    if (padded_seqs == 0)
        return NV_OK;
    if ((num_seqs > 0 && (!seq_lens || !block_tables)) || !context_lens || !positions || !slot_mapping)
        return NV_ERR_NULL;
    if (!is_pow2(block_size) || block_size < 1 || block_size > (1 << 20) ||
        (int64_t)num_blocks * block_size >= (1ll << 31))
        return NV_ERR_UNSUPPORTED;
    const int grid = (padded_seqs + 255) / 256;
    prepare_decode_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(seq_lens, block_tables, bt_stride, num_seqs,
                                                                 padded_seqs, ilog2(block_size), num_blocks,
                                                                 context_lens, positions, slot_mapping, d_err);
    return cudaGetLastError() == cudaSuccess ? NV_OK : NV_ERR_CUDA;
}

extern "C" int nv_prepare_prefill(const int32_t *num_cached, const int32_t *num_scheduled,
                                  const int32_t *block_tables, int32_t bt_stride, int32_t num_seqs, int32_t total_q,
                                  int32_t block_size, int32_t num_blocks, int32_t *cu_seqlens_q,
                                  int32_t *cu_seqlens_k, int32_t *positions, int32_t *slot_mapping,
                                  int32_t *max_seqlens, int32_t *d_err, nv_stream_t stream)
{
    using namespace nvkv_host;
    if (num_seqs < 0 || total_q < 0 || bt_stride <= 0 || num_blocks < 0)
        return NV_ERR_SHAPE;
    if (num_seqs == 0)
        return NV_OK;
    if (!num_cached || !num_scheduled || !block_tables || !cu_seqlens_q || !cu_seqlens_k || !max_seqlens ||
        (total_q > 0 && (!positions || !slot_mapping)))
        return NV_ERR_NULL;
    if (!is_pow2(block_size) || block_size < 1 || block_size > (1 << 20) ||
        (int64_t)num_blocks * block_size >= (1ll << 31))
        return NV_ERR_UNSUPPORTED;
    prepare_prefill_scan_kernel<<<1, 1024, 0, (cudaStream_t)stream>>>(num_cached, num_scheduled, num_seqs,
                                                                      cu_seqlens_q, cu_seqlens_k, max_seqlens,
                                                                      d_err);
    if (cudaGetLastError() != cudaSuccess)
        return NV_ERR_CUDA;
    if (total_q > 0) {
        prepare_prefill_fill_kernel<<<(total_q + 255) / 256, 256, 0, (cudaStream_t)stream>>>(
            num_cached, block_tables, bt_stride, num_seqs, total_q, ilog2(block_size), num_blocks, cu_seqlens_q,
            positions, slot_mapping, d_err);
        if (cudaGetLastError() != cudaSuccess)
            return NV_ERR_CUDA;
    }
    return NV_OK;
}
