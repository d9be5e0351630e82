// Host side of the tcgen05 tile-attention kernels (paged_prefill.cu), shared with the decode entry
// points: decode with 8 or more query heads per kv head runs as a prefill of one query row per
// sequence (its query sits at position L-1, so the causal mask keeps all L keys).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace nvkv_host {

struct TileAttnArgs {
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *cu_seqlens_q;      // prefill: [num_seqs + 1] (unused in decode mode)
    const int32_t *cu_seqlens_k;
    const int32_t *context_lens;      // decode mode when non-null: [num_seqs], query row b is sequence b
    const int32_t *block_tables;
    int32_t bt_stride;
    int32_t num_seqs;
    int32_t total_q;                  // query rows (decode mode: num_seqs)
    int32_t max_seqlen_q;             // decode mode: 1
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t num_blocks;
    int32_t max_len;                  // decode mode: contexts longer than this are truncated to it
    int32_t split_steps;              // decode mode: 128-key steps per split (0: no split); a sequence
                                      // with more writes fp32 partials for a merge launch
    int32_t max_splits;               // splits of the longest sequence
    float *part_o;                    // [num_seqs, max_splits, num_q_heads, 128]
    float *part_ml;                   // [num_seqs, max_splits, num_q_heads, 2]: log2-domain max, sum
    float scale;
    void *out;
    void *workspace;
    size_t workspace_bytes;
    int32_t *d_err;
    cudaStream_t stream;
};

// Bytes of work list the tile kernels need: a 64-byte header and 32 bytes per query tile.
size_t tile_workspace_bytes(int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q, int group);

// Checks the shapes and enqueues the pre-pass and the attention kernel on a.stream; returns an
// nv_status.  Decode mode: rows of sequences with no keys are written as zeros by the pre-pass.
int tile_attention(const TileAttnArgs &a);

}  // namespace nvkv_host
