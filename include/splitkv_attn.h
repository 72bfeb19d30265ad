/*
 * splitkv_attn.h -- exact attention over a KV cache split along the sequence, with an
 * exact log-sum-exp (LSE) merge of the per-split partials.  C ABI of
 * libsplitkv_attn.so (NVIDIA GB300, sm_103a).
 *
 * The operation (cited by web page title and section):
 *   - "Helix Parallelism: Why Tensor Parallelism Hits a Wall at Million-Token
 *     Context", section "Sharding the sequence instead": the KV cache is sharded
 *     along the sequence; attention over each shard yields a partial output plus a
 *     log-sum-exp per token and query head; the fragments are merged exactly with
 *     m = max lse, den = sum exp(lse - m), o = sum o * exp(lse - m) / den.
 *   - "Context Parallelism for Scalable Million-Token Inference" (knowledge note),
 *     section "Pass-KV keeps queries local and circulates keys and values": the
 *     same merge over the N ring steps of a prefill chunk; section "A runtime
 *     heuristic chooses the ring direction": shape(Q) = [T, N_H, D_H] and
 *     shape(K) = shape(V) = [T+P, N_KV, D_H].
 *   - "现代大模型推理并行策略总览", section "Transformer 的工程实践": query heads
 *     map to KV heads in contiguous groups; section "序列布局": the causal mask is
 *     decided by original token positions.
 *
 * On one GPU the KVP shards / ring steps are the splits of one call; the merge is
 * the reduction the pages' All-to-All feeds.
 *
 * Conventions for every entry point
 *   - Device pointers are owned by the caller and must stay valid until the work
 *     queued on `stream` (a cudaStream_t, NULL = legacy default stream) completes.
 *     The library allocates no memory.  Calls are asynchronous on `stream`.
 *   - Errors are returned, never raised: argument errors are detected on the host
 *     before anything is launched; a CUDA error maps to SKV_ECUDA.  The text of
 *     the last error of the calling thread is splitkv_last_error().
 *   - Query head h reads KV head h / (Hq / Hkv).
 *   - Visibility: query row i of sequence b sees KV position t iff
 *       bounds[b][j] <= t < bounds[b][j+1]   (its split j),
 *       t < seq_lens[b]  (and t < S_max), and
 *       t <= causal_offset + i.
 *     Decode passes a causal_offset >= S_max (SKV_NO_CAUSAL) so nothing is masked;
 *     a prefill chunk whose first row sits at global position P passes P.
 *   - Split bounds are a DEVICE int32 array [B][n_split + 1] (like seq_lens), read by the
 *     kernels and never by the host, so a call needs no host-to-device copy and takes any
 *     batch size.  Each row should be non-decreasing; the kernels clip every split to
 *     [0, min(seq_lens[b], S_max)) and treat a split whose upper bound does not exceed its
 *     lower one as empty, so no row of bounds can make a kernel read outside the caches
 *     (but overlapping splits count their common tokens once per split).  The calls that
 *     merge their splits in one kernel (see gqa_decode_attn) attend over
 *     [bounds[b][0], bounds[b][n_split]).
 *   - Work decomposition: long splits are cut into chunks so that one launch fills the
 *     GPU.  The host plans for splits of about S_max / n_split tokens and every split is
 *     cut into the same number of chunks, sized on the device from the split's own length;
 *     splits of very unequal length therefore load the GPU unevenly (the result is the
 *     same).
 *   - Partials: o is normalised by its own softmax denominator and lse is the
 *     natural log of that denominator over scaled scores (softmax_scale * q.k).
 *     A split with no visible token has o = 0 and lse = -inf.
 *   - fp8-e4m3 KV: value = e4m3(code) * scale[b][kv_head][t / scale_block].  The products
 *     run on f16 tensor cores: the codes widen to fp16 exactly; the bf16 query rows of
 *     each 16-row group are multiplied by the power of two that puts their largest
 *     magnitude in [2^14, 2^15) and rounded to fp16 (exact for every element within 2^-29
 *     of that largest; the power of two is divided out of the scores), so any finite bf16
 *     query is accepted; p times the V block scale is rounded to fp16 for the PV product
 *     (finite while the V block scale stays below 65504, i.e. |V| below 2.9e7).
 *   - MLA (latent KV): Hkv = 1, dk = 576 (512 latent + 64 rope), dv = 512 and
 *     v_cache = k_cache with the same strides (V is the first 512 latent columns).
 *   - Supported shapes (anything else returns SKV_EUNSUPPORTED before launch): bf16 KV
 *     with dk = dv = 64 or 128; fp8-e4m3 KV with dk = dv = 128; the bf16 MLA latent above.
 *     Any Hq multiple of Hkv, any Tq and B; bf16 dk = dv = 128 with Hq / Hkv dividing 128
 *     and at least 128 (query row, head) rows per KV head runs on the tensor-core kernel,
 *     the MLA latent with Hq dividing 128 on the tensor-core cluster kernel.  Strides are
 *     free within the alignment rules of each call (16-byte aligned rows, 16-byte
 *     multiples for K/V strides, 8-element multiples for q strides).
 */
#ifndef SPLITKV_ATTN_H
#define SPLITKV_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SKV_OK = 0,
  SKV_EINVAL = -1,       /* invalid argument: null pointer, shape, stride, alignment, bounds */
  SKV_EUNSUPPORTED = -2, /* valid but not implemented (head dims, dtype combination) */
  SKV_ECUDA = -3,        /* CUDA error while launching; see splitkv_last_error() */
  SKV_EWORKSPACE = -4    /* workspace missing or smaller than the matching *_workspace_size */
} skv_status;

typedef enum { SKV_KV_BF16 = 0, SKV_KV_FP8_E4M3 = 1 } skv_kv_dtype;

/* causal_offset that masks nothing */
#define SKV_NO_CAUSAL ((int64_t)1 << 62)

/* Problem description shared by attn_partial and gqa_decode_attn. */
typedef struct {
  int32_t B;            /* sequences in the batch */
  int32_t Tq;           /* query rows per sequence (1 for decode) */
  int32_t Hq;           /* query heads */
  int32_t Hkv;          /* KV heads, Hq % Hkv == 0 */
  int32_t dk;           /* query/key head dim */
  int32_t dv;           /* value head dim */
  int64_t S_max;        /* KV positions allocated per (sequence, KV head), < 2^31 */
  float softmax_scale;  /* multiplies q.k (e.g. 1/sqrt(dk)) */
  int32_t kv_dtype;     /* skv_kv_dtype */
  int32_t scale_block;  /* fp8 only: tokens per scale block, a positive multiple of 64 */
  int64_t q_strides[3]; /* q: bf16, element strides of (b, query row, head); dim stride 1 */
  int64_t k_strides[3]; /* k_cache: element strides of (b, KV head, token); dim stride 1 */
  int64_t v_strides[3]; /* v_cache: same for V */
} skv_desc;

/* Library version: (major << 16) | minor. */
int32_t splitkv_version(void);

/* Text of the calling thread's last error ("" if none).  Valid until the thread's next call. */
const char* splitkv_last_error(void);

/*
 * Read and clear the device error word of the current device (blocking: waits for all
 * work on the device).  *code = 0 if no kernel gave up a bounded wait, else a bitmask
 * (1: a consumer waited too long for a tile, 2: the loader waited too long for a free
 * stage, 4: a final drain waited too long).  Every wait in the kernels has a time limit.
 */
skv_status splitkv_device_error(uint32_t* code);

/*
 * Read and clear the whole device error record (8 words, blocking): [0] the code as above,
 * [1] nonzero if the first failure was described, [2] its block index, [3] its thread
 * index, [4] the shared-memory address of the barrier it waited on, [5] the phase parity it
 * waited for | code << 8.  For diagnosing a wait that gave up.
 */
skv_status splitkv_device_error_detail(uint32_t* record);

/*
 * Kernel timing.  splitkv_kernel_timing(1) clears the record and makes every later call of
 * this library, from this host thread, record a pair of CUDA events (owned by the library)
 * on the call's stream immediately before and after its attention kernel -- the split-KV
 * partial / tensor-core kernel, not the merge -- so that the kernel's own device time can
 * be read while a caller times whole calls; splitkv_kernel_timing(0) stops recording.
 * splitkv_kernel_timing_read waits for the recorded events and returns the summed kernel
 * time in milliseconds and the number of kernel launches recorded since the last enable
 * (at most 4096 per enable; later launches are not recorded).  SKV_ECUDA on event errors.
 */
skv_status splitkv_kernel_timing(int32_t enable);
skv_status splitkv_kernel_timing_read(float* total_ms, int32_t* launches);

/*
 * attn_partial -- one partial attention output per split.
 *
 *   q            bf16, logical [B][Tq][Hq][dk] with desc->q_strides
 *   k_cache      bf16 or e4m3 codes, logical [B][Hkv][S_max][dk] with desc->k_strides
 *   v_cache      same for V ([..][dv], desc->v_strides)
 *   k_scale      fp8: fp32 [B][Hkv][ceil(S_max / scale_block)] contiguous; NULL for bf16
 *   v_scale      fp8: same layout; NULL for bf16
 *   seq_lens     DEVICE int32 [B]; 0 <= seq_lens[b] <= S_max
 *   split_bounds DEVICE int32 [B][n_split + 1], contiguous, 4-byte aligned (see Conventions)
 *   n_split      >= 1
 *   causal_offset  see Visibility above
 *   out_partial  fp32 [n_split][B][Tq][Hq][dv] contiguous, 16-byte aligned
 *   lse_partial  fp32 [n_split][B][Tq][Hq] contiguous
 *   workspace    device scratch of at least attn_partial_workspace_size() bytes (256-byte
 *                aligned); may be NULL when that size is 0.  Used when long splits are cut
 *                into chunks to fill the GPU; the chunks are merged back per split.
 * Alignment: q, k_cache, v_cache 16-byte aligned; q strides multiples of 8 elements; K/V
 * token/head/batch strides multiples of 16 bytes.
 */
skv_status attn_partial_workspace_size(const skv_desc* desc, int32_t n_split, size_t* bytes);
skv_status attn_partial(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                        const int32_t* split_bounds, int32_t n_split, int64_t causal_offset, float* out_partial,
                        float* lse_partial, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_merge_lse -- exact LSE merge of n_split partials (the merge of the pages above).
 *
 *   out_partials fp32 [n_split][B][Tq][Hq][dv], lse_partials fp32 [n_split][B][Tq][Hq] (device)
 *   out          bf16 [B][Tq][Hq][dv];  lse  fp32 [B][Tq][Hq]  (device)
 * Rows whose partials are all empty (lse = -inf) get out = 0, lse = -inf.  dv must be a
 * multiple of 4; pointers 16-byte aligned (out 8-byte).
 */
skv_status attn_merge_lse(int32_t n_split, int32_t B, int32_t Tq, int32_t Hq, int32_t dv,
                          const float* out_partials, const float* lse_partials, void* out, float* lse,
                          void* stream);

/*
 * gqa_decode_attn -- split-KV attention and the merge in one call: the exact attention of
 * every query row over the union of its splits, written as bf16 out [B][Tq][Hq][dv] and
 * fp32 lse [B][Tq][Hq] (contiguous).  Arguments as attn_partial; the per-split / per-chunk
 * partials live in the caller's workspace of at least gqa_decode_attn_workspace_size() bytes.
 * Kernels by shape: bf16 KV with dk = dv = 128, Hq / Hkv dividing 128 and at least 128
 * (query row, head) rows per KV head runs one tensor-core kernel that merges the splits
 * on the fly (workspace size 0; out must be 16-byte aligned); every other shape runs a
 * split-KV partial kernel into the workspace and the merge kernel.
 */
skv_status gqa_decode_attn_workspace_size(const skv_desc* desc, int32_t n_split, size_t* bytes);
skv_status gqa_decode_attn(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                           const int32_t* split_bounds, int32_t n_split, int64_t causal_offset, void* out,
                           float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * gqa_decode_attn_noalloc -- gqa_decode_attn for callers that cannot allocate device memory.
 *
 * No counterpart in the pages: this is a deployment convenience of this library.  Some
 * callers cannot call cudaMalloc or hand over a workspace: a plugin living inside a host
 * runtime that owns every device allocation and forbids allocating behind its back, a
 * latency-critical path where an allocation (which may synchronise the whole device) is not
 * acceptable, or a foreign-language caller that only has the C ABI and no device allocator.
 * This entry point takes the same arguments as gqa_decode_attn minus the workspace and
 * allocates nothing.
 *   - The tensor-core shapes (see gqa_decode_attn) run the same fused kernel as
 *     gqa_decode_attn, which needs no scratch at all.
 *   - Every other shape runs the same partial and merge kernels, with the per-split /
 *     per-chunk partials in a fixed scratch array of 32 MiB (33554432 bytes) compiled into
 *     the library, which every GPU that loads the library keeps reserved until the process
 *     exits.  When gqa_decode_attn's plan would need more than that, the work is planned
 *     again with as many chunks per split as the scratch holds (same result, possibly a
 *     less even load).  A part needs B * Tq * Hq * (dv + 1) * 4 bytes (each of its two
 *     arrays rounded up to 256 bytes); if even n_split parts (one chunk per split) exceed
 *     32 MiB the call returns SKV_EWORKSPACE, with both sizes in the message, before
 *     anything is launched.
 *   - The first call on each device looks up the scratch array's device address (with that
 *     device current) and caches it; make that first call before any stream capture.
 *   - Every call on a device uses the same scratch array, so calls that may overlap on the
 *     GPU (different streams, or different host threads) race and corrupt each other's
 *     results; serialise them (one stream, or events).  The scratch keeps the last call's
 *     contents; nothing in it needs to start at zero.
 */
skv_status gqa_decode_attn_noalloc(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                                   const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                                   const int32_t* split_bounds, int32_t n_split, int64_t causal_offset, void* out,
                                   float* lse, void* stream);

/*
 * attn_partial_pos / gqa_decode_attn_pos -- attn_partial and gqa_decode_attn for tokens
 * stored out of sequence order.  The causal rule is taken from original positions instead
 * of causal_offset: token t of sequence b is visible to query row i iff
 * k_pos[b * S_max + t] <= q_pos[b * Tq + i] (besides lying in its split and below
 * seq_len[b]).  This is the mask by original position of the zigzag and striped layouts
 * ("现代大模型推理并行策略总览", section "序列布局：Contiguous、Zigzag 与 Striped"; rank r of
 * a zigzag layout holds chunks r and 2N-1-r, "Context Parallelism for Scalable Million-Token
 * Inference", section "Load-balanced sharding makes causal work and memory land evenly"):
 * a ring-prefill step whose query chunk and KV shards come from such a layout passes their
 * positions here.
 *
 *   q_pos  DEVICE int32 [B][Tq], contiguous, 4-byte aligned.
 *   k_pos  DEVICE int32 [B][S_max], contiguous, 16-byte aligned, S_max a multiple of 4.
 * Every other argument, the workspace (sizes from attn_partial_workspace_size and
 * gqa_decode_attn_workspace_size), the outputs and the ownership rules are those of
 * attn_partial / gqa_decode_attn.  Fully masked tiles are still streamed (no tile
 * skipping by position).  Errors: SKV_EINVAL for NULL or misaligned positions or S_max
 * not a multiple of 4; SKV_EUNSUPPORTED for the MLA latent shape.
 */
skv_status attn_partial_pos(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                            const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                            const int32_t* split_bounds, int32_t n_split, const int32_t* q_pos,
                            const int32_t* k_pos, float* out_partial, float* lse_partial, void* workspace,
                            size_t workspace_bytes, void* stream);

skv_status gqa_decode_attn_pos(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                               const int32_t* split_bounds, int32_t n_split, const int32_t* q_pos,
                               const int32_t* k_pos, void* out, float* lse, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * Paged block KV cache.  "Attention DP", section "KV Cache", keeps each rank's
 * cache as [num_blocks, num_kv_heads, block_len, d_head]; a per-sequence block table maps
 * logical block i of sequence b (its tokens [i * block_len, (i + 1) * block_len)) to the
 * physical page that holds it, so token t of sequence b, KV head g is row t % block_len
 * of page block_table[b * max_blocks + t / block_len], head g.  Pages may be shared.
 */
typedef struct {
  int32_t block_len;           /* tokens per page: a positive multiple of 64 */
  int32_t max_blocks;          /* block-table entries per sequence */
  int64_t num_blocks;          /* pages in the caches (entries >= num_blocks read zeros) */
  const int32_t* block_table;  /* DEVICE int32 [B][max_blocks], 4-byte aligned */
} skv_paged;

/*
 * attn_partial_paged / gqa_decode_attn_paged -- attn_partial and gqa_decode_attn over a
 * paged cache.  k_cache / v_cache are the pages [num_blocks][Hkv][block_len][d] with
 * desc->k_strides / v_strides = (page, head, token) strides in elements (the MLA value
 * cache is a view of the latent pages, as for the contiguous call); desc->S_max is the
 * logical capacity of a sequence, at most max_blocks * block_len; fp8 block scales are
 * per page: [num_blocks][Hkv][block_len / scale_block] (block_len a multiple of
 * scale_block).  Split bounds, seq_lens and causal_offset are in logical tokens.  The
 * workspace sizes are those of attn_partial_workspace_size / gqa_decode_attn_workspace_size
 * for the same desc; outputs, ownership and errors as for the contiguous calls, plus
 * SKV_EINVAL for a NULL or misaligned block table, block_len not a positive multiple of
 * 64, or S_max above max_blocks * block_len.
 */
skv_status attn_partial_paged(const skv_desc* desc, const skv_paged* paged, const void* q, const void* k_cache,
                              const void* v_cache, const float* k_scale, const float* v_scale,
                              const int32_t* seq_lens, const int32_t* split_bounds, int32_t n_split,
                              int64_t causal_offset, float* out_partial, float* lse_partial, void* workspace,
                              size_t workspace_bytes, void* stream);

skv_status gqa_decode_attn_paged(const skv_desc* desc, const skv_paged* paged, const void* q, const void* k_cache,
                                 const void* v_cache, const float* k_scale, const float* v_scale,
                                 const int32_t* seq_lens, const int32_t* split_bounds, int32_t n_split,
                                 int64_t causal_offset, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * attn_ring_step -- one pass-KV ring step ("Context Parallelism for Scalable Million-Token
 * Inference", section "Pass-KV keeps queries local and circulates keys and values"): the
 * local query chunk attends over the KV block received at this step, held in its own
 * buffer, and the result is merged into a running output in place with the exact LSE
 * merge, so no step's partial is kept.
 *
 *   desc     shapes; desc->S_max = tokens in this step's block
 *   k_block, v_block  DEVICE [B][Hkv][S_max][d] with desc strides (fp8: scales as for
 *            attn_partial, indexed by position in the block)
 *   seq_lens DEVICE int32 [B]: tokens of the block that exist for each sequence
 *   causal_offset  query row i sees block token t iff t <= causal_offset + i (the chunk's
 *            offset minus the block's start; SKV_NO_CAUSAL for none)
 *   first    nonzero: o_acc / lse_acc are written, not read (the first step)
 *   o_acc    DEVICE fp32 [B][Tq][Hq][dv], lse_acc DEVICE fp32 [B][Tq][Hq]: the running
 *            normalised output and natural-log LSE, updated in place; rows that have seen
 *            no token yet hold o = 0, lse = -inf
 *   workspace  DEVICE, at least attn_ring_step_workspace_size(desc) bytes, 256-aligned
 * No bounds table: the block is one split [0, S_max).  Errors as for attn_partial; the merge
 * is the same one attn_merge_lse applies.
 */
skv_status attn_ring_step_workspace_size(const skv_desc* desc, size_t* bytes);

skv_status attn_ring_step(const skv_desc* desc, const void* q, const void* k_block, const void* v_block,
                          const float* k_scale, const float* v_scale, const int32_t* seq_lens, int64_t causal_offset,
                          int32_t first, float* o_acc, float* lse_acc, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * gqa_decode_attn_passq -- pass-Q decode over a context-parallel group of n_ranks ranks,
 * every rank emulated on this GPU ("Context Parallelism for Scalable Million-Token
 * Inference", sections "Pass-Q keeps KV stationary for cache-heavy turns" and "Pass-Q
 * decode protects capacity but can hurt TTIT").  Each rank keeps its own resident shard of
 * every request's KV cache; the one-token queries travel the ring with their batch ids and
 * attend over the shard of whichever rank they reach; the partials are permuted back to the
 * queries' owners (the All-to-All) and merged exactly by their LSE.  The result is the
 * attention of each request's query over the union of its shards.
 *
 *   desc        desc->B = requests, a multiple of n_ranks (rank r owns the queries of
 *               requests [r * B / n_ranks, (r + 1) * B / n_ranks): pad the batch to a
 *               multiple of the group size); desc->Tq = 1; desc->S_max = capacity of one
 *               rank's shard of one request; GQA shapes only (bf16 d = 64 / 128, fp8
 *               d = 128); desc strides as for attn_partial, k/v strides of one shard row
 *   n_ranks     ranks in the group, >= 1
 *   q           DEVICE bf16 [B][1][Hq][dk] with desc->q_strides
 *   k_shards, v_shards  DEVICE [n_ranks * B][Hkv][S_max][d] with desc->k/v_strides: row
 *               r * B + b is rank r's resident shard of request b.  The order of the tokens
 *               inside a shard is free (the new token follows every cached one, so it sees
 *               all of them); tokens past the shard's length are never read
 *   k_scale, v_scale  fp8 only: DEVICE fp32 [n_ranks * B][Hkv][S_max / scale_block]
 *   shard_lens  DEVICE int32 [n_ranks][B]: resident tokens of request b on rank r, 0 allowed
 *   out, lse    DEVICE bf16 [B][1][Hq][dv] and fp32 [B][1][Hq] (contiguous); a request
 *               with no resident token anywhere gets out = 0, lse = -inf
 *   workspace   DEVICE, gqa_decode_attn_passq_workspace_size() bytes, 256-byte aligned:
 *               the exchange buffer of fp32 partials [owner][source rank][part][B /
 *               n_ranks][Hq][dv] and their LSEs
 * Schedule: rank k at ring step s (s = 0 .. n_ranks - 1) holds the query block that started
 * on rank (k - s) mod n_ranks and writes its partial to that owner's slot from rank k.  One
 * partial launch covers every rank and step; one merge launch covers the exchange and the
 * merge.  Caller owns every buffer; the library allocates nothing.
 * Errors: as gqa_decode_attn, plus SKV_EINVAL for n_ranks < 1 or B not a multiple of n_ranks;
 * SKV_EUNSUPPORTED for Tq != 1 or the MLA latent shape.
 */
skv_status gqa_decode_attn_passq_workspace_size(const skv_desc* desc, int32_t n_ranks, size_t* bytes);

skv_status gqa_decode_attn_passq(const skv_desc* desc, int32_t n_ranks, const void* q, const void* k_shards,
                                 const void* v_shards, const float* k_scale, const float* v_scale,
                                 const int32_t* shard_lens, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPLITKV_ATTN_H */
