/*
 * nv_paged_kv.h -- C ABI of the paged KV attention store for NVIDIA GB300 (sm_103a).
 *
 * The data-parallel hot path of a vLLM-style engine's attention layer, as the nano-vLLM
 * field guide walks through it (Step 10.3 "attention.py: storing K/V and calling
 * FlashAttention"): each forward first scatters the new tokens' K/V rows into a paged pool,
 * then attends over the pool through per-sequence block tables -- one query per sequence
 * in decode, a causal chunk after a cached prefix in prefill.
 *
 * Common conventions
 *   - Every pointer is a DEVICE pointer owned by the caller.  No entry point allocates,
 *     frees, synchronises or keeps state between calls, with two documented exceptions
 *     that cost nothing on the device: the first call on a device reads its SM count, and
 *     nv_paged_prefill_attn looks up the driver's tensor-map encoder once per process.
 *     Work is enqueued on `stream` and returns at once.
 *   - bf16 tensors are passed as `void*` (IEEE bfloat16 bit patterns).
 *   - One layer's pool is two tensors k_cache, v_cache of shape
 *     [num_blocks, block_size, num_kv_heads, head_dim], contiguous (the per-layer view of the
 *     field guide's Step 07.4 KV pool).  A "slot" is one row of num_kv_heads*head_dim values;
 *     slot = block_id * block_size + offset (Step 05.1).
 *   - block_tables: int32 [num_seqs, bt_stride]; row b lists sequence b's physical block ids
 *     in logical order, padded with -1 (Step 07.7).  Entries beyond the blocks a sequence's
 *     length needs are never read.
 *   - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *   - Shape limits, the same for decode and prefill unless an entry point adds its own:
 *     head_dim must be 128 and block_size a power of two in [16, 256] (else NV_ERR_UNSUPPORTED);
 *     num_q_heads a multiple of num_kv_heads (else NV_ERR_SHAPE), with a group
 *     G = num_q_heads / num_kv_heads of 1, 2, 4, 8 or 16 (else NV_ERR_UNSUPPORTED).  Decode takes
 *     num_kv_heads <= 16 and a pool of fewer than 2^40 values per tensor (num_blocks * block_size *
 *     num_kv_heads * head_dim); prefill, and decode at G = 8 or 16, take num_seqs <= 65535 and
 *     num_blocks * block_size < 2^31 (else NV_ERR_UNSUPPORTED).
 *   - Host-side argument errors return a negative nv_status before anything is enqueued.
 *     Data-dependent errors found on the device (a slot or block id outside the pool, a
 *     length beyond what the block table or the host hint allows) never fault: the offending
 *     row or key is skipped and a bit from NV_DERR_* is OR-ed into *d_err when d_err is not
 *     NULL (int32, caller-zeroed; read it after the stream has finished).
 *   - The library is safe to call from several host threads; calls on different streams
 *     may overlap on the device, except where an entry point says otherwise.
 */
#ifndef NV_PAGED_KV_H
#define NV_PAGED_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t / CUstream.  NULL means the legacy default stream. */
typedef struct CUstream_st *nv_stream_t;

typedef enum nv_status {
    NV_OK = 0,
    NV_ERR_NULL = -1,         /* a required pointer is NULL */
    NV_ERR_SHAPE = -2,        /* a size is negative, zero where it may not be, or inconsistent */
    NV_ERR_ALIGN = -3,        /* a pointer or row stride breaks the 16-byte alignment rule */
    NV_ERR_UNSUPPORTED = -4,  /* a shape outside what the kernels implement (e.g. head_dim != 128) */
    NV_ERR_WORKSPACE = -5,    /* workspace NULL or smaller than the size query returned */
    NV_ERR_CUDA = -6          /* the CUDA runtime reported an error (launch, attribute, driver entry) */
} nv_status;

/* Bits OR-ed into *d_err by the kernels. */
#define NV_DERR_SLOT_RANGE 0x1    /* slot_mapping entry < -1 or >= num_slots: row skipped */
#define NV_DERR_BLOCK_RANGE 0x2   /* a needed block-table entry outside [0, num_blocks): nothing is read
                                     from it; that sequence's output is not meaningful (the store and
                                     the split-KV decode kernel skip its keys) */
#define NV_DERR_LENGTH 0x4        /* a length exceeds the block table, the host hint, or is negative */
#define NV_DERR_TIMEOUT 0x8       /* a bounded wait on an asynchronous copy gave up */
#define NV_DERR_SLOT_MISMATCH 0x10 /* fused store + decode: a slot that is not position L-1's (row not stored) */
#define NV_DERR_VALUE 0x20         /* sampler: a temperature that is not positive and finite (token -1);
                                      decode and sampler: a counter of the workspace was not zero */

/* Human-readable name of an nv_status value (static string). */
const char *nv_status_string(int status);

/*
 * nv_store_kvcache -- scatter new K/V rows into their cache slots.
 *
 * Field guide Step 10.3, "The Triton store kernel": for every new-token row i,
 * s = slot_mapping[i]; s == -1 marks a padding row (CUDA-graph bucket padding,
 * Step 07.8) and writes nothing; otherwise row i of k (num_kv_heads*head_dim values) goes
 * to row s of the flattened k_cache, and likewise for v.  Bit-exact copy.
 *
 *   k, v          bf16 [n_tokens, num_kv_heads, head_dim]; heads contiguous (head stride
 *                 head_dim), rows k_row_stride / v_row_stride ELEMENTS apart (v may be a view
 *                 into a fused QKV output whose rows are wider).  Strides >= num_kv_heads*head_dim
 *                 and multiples of 8; base pointers 16-byte aligned.
 *   slot_mapping  int32 [n_tokens].
 *   k_cache, v_cache  bf16 [num_slots, num_kv_heads*head_dim] (any [num_blocks, block_size, ...]
 *                 pool flattened), 16-byte aligned.
 *   n_tokens      >= 0 (0 enqueues nothing).
 *   d_err         nullable; NV_DERR_SLOT_RANGE for slots outside [-1, num_slots).
 * Duplicate slots within one call are not supported (the pages never produce them).
 */
int nv_store_kvcache(const void *k, int64_t k_row_stride, const void *v, int64_t v_row_stride,
                     const int32_t *slot_mapping, int32_t n_tokens, void *k_cache, void *v_cache,
                     int64_t num_slots, int32_t num_kv_heads, int32_t head_dim, int32_t *d_err,
                     nv_stream_t stream);

/*
 * nv_qk_norm_rope_store -- the attention layer's prologue: QK-norm, RoPE, then the K/V store.
 *
 * Field guide, "Qwen3Attention.forward" with "layernorm.py" and "rotary_embedding.py", and Step
 * 10.3: each token's fused projection row is split into q [Hq, D], k [Hkv, D], v [Hkv, D].  Every
 * q and k head is RMS-normalised over its D values -- var = mean(x^2) in fp32, x * rsqrt(var +
 * eps) cast to bf16, then multiplied by the bf16 weight (q_norm_weight / k_norm_weight, [D]) as a
 * bf16 product -- and then rotated by RoPE at positions[t]: element j pairs with j + D/2
 * (rotate-half), angle = positions[t] * rope_theta^(-2j/D) in fp32, y1 = x1 cos - x2 sin,
 * y2 = x2 cos + x1 sin in fp32, rounded to bf16.  q goes to q_out; the roped k and the unchanged
 * v are written to row slot_mapping[t] of the caches (-1 = store nothing; q is still produced).
 *
 *   qkv           bf16 [n_tokens, row stride qkv_row_stride elements] holding q | k | v
 *                 (>= (Hq + 2 Hkv) * head_dim, multiple of 8); 16-byte aligned.
 *   positions     int32 [n_tokens] (< 2^24).
 *   q_norm_weight, k_norm_weight  bf16 [head_dim], 4-byte aligned.
 *   q_out         bf16 [n_tokens, Hq, head_dim] contiguous.
 *   k_cache, v_cache  as for nv_store_kvcache ([num_slots, Hkv*head_dim] flattened).
 *   rms_eps >= 0 (1e-6 in Qwen3); rope_theta > 1 (1e6 in Qwen3).
 *   d_err         nullable; NV_DERR_SLOT_RANGE for slots outside [-1, num_slots) (row not stored).
 * head_dim must be 128.  Results are within a bf16 rounding of the fp32 definition (the GPU's
 * rsqrt / sincos differ from a CPU libm by an ulp or two of fp32); v is copied bit for bit.
 */
int nv_qk_norm_rope_store(const void *qkv, int64_t qkv_row_stride, const int32_t *positions,
                          const void *q_norm_weight, const void *k_norm_weight, float rms_eps, float rope_theta,
                          const int32_t *slot_mapping, int32_t n_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, void *q_out, void *k_cache, void *v_cache, int64_t num_slots,
                          int32_t *d_err, nv_stream_t stream);

/*
 * nv_prepare_decode -- a decode step's attention metadata, built on the device.
 *
 * Field guide Step 07.6 "prepare_decode" and Step 07.8 (graph-replay padding): for sequence b with
 * len = seq_lens[b] tokens (the new one included): context_lens[b] = len, positions[b] = len - 1,
 * slot_mapping[b] = the slot of position len - 1 (the last block's base slot plus
 * last_block_num_tokens - 1).  Rows num_seqs .. padded_seqs-1 get slot -1, context 0 and position 0,
 * so a graph replayed at a larger bucket stores and attends to nothing for them.  A row whose length
 * is < 1 or needs more blocks than bt_stride (NV_DERR_LENGTH), or whose last block id lies outside
 * [0, num_blocks) (NV_DERR_BLOCK_RANGE), is written as a padding row.
 *   seq_lens int32 [num_seqs]; block_tables int32 [num_seqs, bt_stride]; outputs int32 [padded_seqs].
 *   block_size a power of two; num_blocks * block_size < 2^31.
 */
int nv_prepare_decode(const int32_t *seq_lens, const int32_t *block_tables, int32_t bt_stride, int32_t num_seqs,
                      int32_t padded_seqs, int32_t block_size, int32_t num_blocks, int32_t *context_lens,
                      int32_t *positions, int32_t *slot_mapping, int32_t *d_err, nv_stream_t stream);

/*
 * nv_prepare_prefill -- a prefill step's attention metadata, built on the device.
 *
 * Field guide Step 07.5 "prepare_prefill": sequence b schedules positions [start, end) with
 * start = num_cached[b], end = start + num_scheduled[b].  Writes cu_seqlens_q ([num_seqs + 1],
 * running sum of num_scheduled), cu_seqlens_k ([num_seqs + 1], running sum of end: the keys include
 * the cached prefix), max_seqlens ([2]: max num_scheduled, max end), and for every new token t (packed
 * in sequence order) positions[t] and slot_mapping[t] = the slot of that position through the
 * sequence's block table.  total_q is the host's count of new tokens (the scheduler knows it): the
 * outputs positions / slot_mapping have total_q entries; if the lengths add up to a different total,
 * NV_DERR_LENGTH is set and only the first min of the two are meaningful.  Tokens whose block is
 * missing or out of range get slot -1 (NV_DERR_LENGTH / NV_DERR_BLOCK_RANGE).  Two launches.
 */
int nv_prepare_prefill(const int32_t *num_cached, const int32_t *num_scheduled, const int32_t *block_tables,
                       int32_t bt_stride, int32_t num_seqs, int32_t total_q, int32_t block_size, int32_t num_blocks,
                       int32_t *cu_seqlens_q, int32_t *cu_seqlens_k, int32_t *positions, int32_t *slot_mapping,
                       int32_t *max_seqlens, int32_t *d_err, nv_stream_t stream);

/*
 * nv_sample_exponential_race -- temperature sampling by the exponential race.
 *
 * Field guide, "sampler.py: temperature and the exponential race": logits are divided by each row's
 * temperature and turned into probabilities with softmax; the token is argmax_i p_i / E_i, where the
 * E_i are independent Exp(1) draws clamped below at 1e-10 -- token i wins with probability p_i.  The
 * draws are an input (the pages draw them with torch's exponential_); the first index wins a tie.
 *   logits        bf16 [num_rows, logits_stride] (first vocab entries used; stride a multiple of 8).
 *   temperatures  float32 [num_rows], each > 0 and finite (else the row's token is -1 and
 *                 NV_DERR_VALUE is set).
 *   draws         float32 [num_rows, draws_stride] (stride a multiple of 4).  Both bases 16-byte aligned.
 *   tokens        int64 [num_rows] (out).
 *   workspace     at least nv_sample_workspace_size(num_rows, vocab) bytes, 16-byte aligned, ZERO-FILLED
 *                 before its first use.  Its first 256 KiB hold one counter per row, which every call
 *                 leaves at zero again, so one workspace, zeroed once, serves any later call (any batch
 *                 size); the rest is scratch.  Calls that share a workspace must not run concurrently.
 *                 A counter found non-zero (a workspace that was not zero-filled) sets NV_DERR_VALUE
 *                 and leaves that row's token unspecified.
 * The argmax is taken over logits_i * log2(e) / T - log2(max(E_i, 1e-10)), which orders the
 * entries exactly as p_i / E_i does; rounding can only matter between entries within a few
 * float32 ulps of each other.  One launch: a row is split over several CTAs and the row's last
 * CTA to finish writes its token.
 */
size_t nv_sample_workspace_size(int32_t num_rows, int32_t vocab);

int nv_sample_exponential_race(const void *logits, int64_t logits_stride, const float *temperatures, const float *draws,
                               int64_t draws_stride, int32_t num_rows, int32_t vocab, int64_t *tokens, void *workspace,
                               size_t workspace_bytes, int32_t *d_err, nv_stream_t stream);

/*
 * Bytes of workspace nv_paged_decode_attn needs for this batch: 256 KiB of split counters, then the
 * larger of the split-KV partials (none when one split covers max_context_len) and the tile kernel's
 * partials and work list (64 bytes + 32 per sequence and split).  Depends only on its
 * arguments, so it can be sized once for the largest batch and reused.
 */
size_t nv_paged_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                      int32_t max_context_len);

/*
 * nv_paged_decode_attn -- one query per sequence over its paged KV history (GQA).
 *
 * Field guide Step 10.3 (decode branch) and Step 07.6: sequence b has L = context_lens[b]
 * keys -- this already counts the token whose K/V nv_store_kvcache wrote in the same forward
 * -- read through block_tables[b]; the query sits at position L-1, so it sees every key.
 *   out[b, h, :] = sum_j softmax_j(scale * <q[b,h,:], K_j>) * V_j,   j = 0..L-1,
 * with K_j, V_j the kv-head (h / group) rows of slot block_tables[b][j / block_size] *
 * block_size + j % block_size.  fp32 accumulation and softmax, bf16 output rounded once.
 * A row with L == 0 (graph padding) gets zeros.
 *
 * Groups (num_q_heads / num_kv_heads) 1 and 2 (except at most 8 sequences with num_seqs x
 * max_context_len of 32768 or more), and group 4 for batches of at most 16 sequences with
 * num_seqs x max_context_len below 32768 or whose split-KV grid spans at least ten waves of the
 * GPU (the 512-sequence Qwen3-8B batch): a
 * split-KV flash-decoding kernel on CUDA cores (one launch; a second one merges the partials when a
 * sequence spans more than 16 splits).  Groups 8 and 16, and the other batches: the tcgen05 tile
 * kernel of nv_paged_prefill_attn with one query row per sequence at position L-1 (two launches: a
 * work-list pre-pass, which also zeroes the rows with L == 0, and the tile kernel; a batch with
 * fewer than two (sequence, kv head) units per SM has its keys split into ranges of at least 1024,
 * and a third launch merges them).  At group 8 the CUDA-core kernel's FMAs no longer keep up with
 * HBM (measured 0.54 of the roofline); at group 4 the tile kernel's persistent schedule fills the
 * GPU where a short split-KV grid cannot (64 sequences: 109 against 150 us; one 128K-token
 * sequence: 97 against 170 us), and it keeps up when
 * shared prefix blocks come from L2 and the CUDA-core consumers are bound by their FMAs.  The two
 * paths round differently (P is rounded to bf16 before the PV product on the tile kernel); both
 * are within the parity bar of the fp32 definition.
 *
 *   q, out        bf16 [num_seqs, num_q_heads, head_dim], contiguous, 16-byte aligned.
 *   block_tables  int32 [num_seqs, bt_stride]; context_lens int32 [num_seqs].
 *   num_blocks    pool size in blocks (block ids must lie in [0, num_blocks)).
 *   max_context_len  host-side upper bound on every context_lens[b] (sizes the split-KV
 *                 grid without reading device memory).  A sequence longer than it is
 *                 truncated to it and flagged NV_DERR_LENGTH.  <= bt_stride*block_size.
 *   scale         softmax scale (head_dim ** -0.5 in the pages).
 *   workspace     device scratch of at least nv_paged_decode_workspace_size(...) bytes, 16-byte
 *                 aligned (a batch on the split-KV kernel may pass NULL when one split covers
 *                 max_context_len; the tile kernel always needs one for its work list).  Its first 256 KiB hold
 *                 the per-sequence split counters: they must be ZERO before the first call
 *                 that uses the workspace (allocate it zero-filled), and every call leaves them
 *                 zero, whatever the batch; the rest needs no initialisation.  A counter found
 *                 outside [0, splits) sets NV_DERR_VALUE (that sequence's output is then not
 *                 trustworthy, and the workspace must be zero-filled again).  Calls that share
 *                 a workspace must not overlap on the device.  Batches of more than 65536
 *                 sequences whose contexts need several splits return NV_ERR_UNSUPPORTED.
 */
int nv_paged_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, int32_t bt_stride, const int32_t *context_lens,
                         int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int32_t num_blocks, int32_t max_context_len, float scale,
                         void *out, void *workspace, size_t workspace_bytes, int32_t *d_err,
                         nv_stream_t stream);

/*
 * nv_store_decode_attn -- nv_store_kvcache followed by nv_paged_decode_attn, in one pass.
 *
 * Field guide Step 10.3: every decode forward first stores the new token's K/V (store kernel) and
 * then attends over the history that now ends with it (decode branch); Step 07.6: the new token
 * is position context_lens[b]-1 of sequence b, and its slot is slot_mapping[b].  This call does
 * both with the same kernels as the decode: the new rows are read once from k / v, used as
 * position L-1, and written to their slot by the CTA that attends over that position, so the
 * store costs no launch and no re-read from the pool.
 *
 *   q, block_tables, context_lens, out, workspace, scale, max_context_len: as nv_paged_decode_attn
 *                 (same workspace size).
 *   k, v          bf16 [num_seqs, num_kv_heads, head_dim], one new row per sequence; heads
 *                 contiguous, rows k_row_stride / v_row_stride elements apart (>= Hkv*head_dim,
 *                 multiples of 8), base pointers 16-byte aligned.
 *   slot_mapping  int32 [num_seqs]: -1 = no new row for this sequence (graph padding; position
 *                 L-1, if any, is then read from the pool).  A slot >= 0 must be the slot of
 *                 position L-1 through block_tables[b] (as the engine builds it); any other slot is
 *                 not written, position L-1 is read from the pool, and NV_DERR_SLOT_MISMATCH is set
 *                 (NV_DERR_SLOT_RANGE when it lies outside the pool).
 * The result (cache and out) equals nv_store_kvcache then nv_paged_decode_attn with the same
 * arguments whenever the slots follow that rule.  Groups 8 and 16 (which decode on the tile kernel)
 * apply the same rule in a separate store pass before the decode's launches.  The new slots must
 * not lie in another sequence's history within the same call (they never do: a new token's slot
 * belongs to its own sequence).
 */
int nv_store_decode_attn(const void *q, const void *k, int64_t k_row_stride, const void *v, int64_t v_row_stride,
                         const int32_t *slot_mapping, void *k_cache, void *v_cache, const int32_t *block_tables,
                         int32_t bt_stride, const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                         int32_t max_context_len, float scale, void *out, void *workspace, size_t workspace_bytes,
                         int32_t *d_err, nv_stream_t stream);

/*
 * nv_paged_decode_attn_noalloc -- nv_paged_decode_attn without a caller-provided workspace.
 *
 * The source pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory when they run decode -- an engine whose KV pool already took all the
 * memory its allocator may hand out, a host application that lends the library only its
 * tensors, or C code with no CUDA allocator at hand.  It allocates nothing: the split-KV
 * partials live in a fixed device array of NV_DECODE_STATIC_SCRATCH_BYTES inside the library,
 * which every GPU that loads the library holds until the process exits.
 *
 * Arguments and results are those of nv_paged_decode_attn (same kernels, chosen the same way; a
 * batch that decodes on the tile kernel keeps its work list, and its split partials when its keys are
 * split, in the same static array, and does not split when they would not fit).  On the split-KV
 * kernel the split length is the usual one, doubled (up to 4096 positions) while the partials would
 * not fit the array; a batch whose partials still exceed it (num_seqs * splits * num_q_heads * 520
 * bytes) is rejected with NV_ERR_WORKSPACE before anything is enqueued.
 *
 * The first call on a device looks up the arrays' device addresses (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  All calls share the
 * one scratch array (it keeps the last call's contents; nothing in it needs to start at zero)
 * and one array of 65536 split counters (zero when the library loads; every call leaves them
 * zero): calls that overlap on the GPU -- on different streams, or from different threads --
 * race on them and give wrong results.  Serialise them.
 */
#define NV_DECODE_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

int nv_paged_decode_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int32_t bt_stride, const int32_t *context_lens,
                                 int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int32_t num_blocks, int32_t max_context_len, float scale,
                                 void *out, int32_t *d_err, nv_stream_t stream);

/*
 * nv_paged_prefill_attn -- varlen causal prefill over a cached prefix plus the new chunk.
 *
 * Field guide Step 10.3 (prefill branch, prefix cache) and Step 07.5: the new tokens of all
 * sequences are packed; sequence b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
 * (Lq of them) and attends to Lk = cu_seqlens_k[b+1] - cu_seqlens_k[b] keys read through
 * block_tables[b]; P = Lk - Lq keys were cached before this chunk, and the chunk's own K/V
 * must already be in the pool (store first).  With fewer queries than keys the causal mask
 * is aligned bottom-right: query i of the chunk (position P+i) sees keys 0..P+i.
 * Tensor-core (tcgen05) QK^T and PV in bf16 with fp32 accumulation; fp32 softmax; bf16 out.
 *
 *   q, out        bf16 [total_q, num_q_heads, head_dim], contiguous, 16-byte aligned.
 *   cu_seqlens_q, cu_seqlens_k  int32 [num_seqs + 1], non-decreasing, starting at 0,
 *                 with Lk >= Lq for every sequence (else NV_DERR_LENGTH; rows untouched).
 *   max_seqlen_q  host-side upper bound on every Lq (sizes the grid).  Rows of a longer
 *                 chunk beyond it are not computed and NV_DERR_LENGTH is set.
 *   total_q       cu_seqlens_q[num_seqs] (rows of q and out).
 *   k_cache, v_cache  as above; additionally num_blocks*block_size < 2^31.
 *   workspace     device scratch of at least nv_paged_prefill_workspace_size(...) bytes,
 *                 16-byte aligned, else NV_ERR_WORKSPACE.  The call first writes into it (on
 *                 `stream`, a one-CTA pre-pass) the list of query tiles -- sequence by
 *                 sequence, heaviest sequence first, each sequence's tiles heaviest first -- and
 *                 how the persistent CTAs claim them (the first three quarters dealt round-robin,
 *                 the rest from a counter), so it needs no
 *                 initialisation; calls that share a workspace must not overlap on the device.
 *                 A batch whose tiles would not fit (cu_seqlens_q inconsistent with total_q) sets
 *                 NV_DERR_LENGTH and leaves the last-listed tiles uncomputed.
 * Enqueues two kernels: the pre-pass and the attention kernel.
 */

/*
 * Bytes of workspace nv_paged_prefill_attn needs: 64 + 32 bytes per query tile of 128/G rows
 * (G = num_q_heads / num_kv_heads), for at most min(ceil(total_q*G/128) + num_seqs,
 * num_seqs * ceil(max_seqlen_q*G/128)) tiles.  Depends only on its arguments.
 */
size_t nv_paged_prefill_workspace_size(int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                                       int32_t num_q_heads, int32_t num_kv_heads);

int nv_paged_prefill_attn(const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                          const int32_t *block_tables, int32_t bt_stride, int32_t num_seqs,
                          int32_t total_q, int32_t max_seqlen_q, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                          float scale, void *out, void *workspace, size_t workspace_bytes,
                          int32_t *d_err, nv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NV_PAGED_KV_H */
