// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace skv {

// Tokens per KV tile of the GQA partial kernel (and the chunk granularity).
constexpr int kTileN = 64;

// Kernel attributes set with cudaFuncSetAttribute belong to the current device's context,
// so a launcher applies them the first time it launches on each device: `done` keeps one
// bit per device (devices past 63 set them on every launch).
template <class F>
cudaError_t once_per_device(std::atomic<uint64_t>& done, F&& set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = set();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Parameters of one split-KV partial-attention launch.
//
// Work item = (b, kv head g, split j, chunk c, row tile mt).  Split j of sequence b
// covers tokens [bounds[b][j], bounds[b][j+1]) clipped to [0, min(seq_lens[b], S_max))
// (no bounds table: the one split [0, S_max)); the table lives in device memory and is
// read by the kernels, never by the host.  From its first whole kTileN-token tile the
// split is cut into n_chunk chunks of equal tile counts, sized on the device from the
// split's own length, so every split is spread over the same number of work items
// whatever its length.  Row m of kv head g's row space (m < Tq*G) is query row
// t = m / G of query head g*G + m % G.
//
// The item writes its partial (normalised o, natural-log lse) to part
// p = j * n_chunk + c of out_o [n_part][B][Tq][Hq][dv] and out_lse [n_part][B][Tq][Hq].
struct PartialParams {
  const void* q;  // bf16 [B][Tq][Hq][dk] with strides below (elements)
  int64_t q_sb, q_st, q_sh;
  const float* k_scale;  // fp8 only: [B][Hkv][n_scale_blk]
  const float* v_scale;
  int32_t n_scale_blk;
  int32_t scale_block;
  const int32_t* seq_lens;  // device [B]
  float* out_o;
  float* out_lse;
  unsigned int* err;  // device error word
  int64_t causal_offset;
  const int32_t* q_pos;  // original positions [B][Tq] / [B][S_max] (NULL: rows at
  const int32_t* k_pos;  // causal_offset + i, tokens at their index)
  const int32_t* block_table;  // paged cache: [B][max_blocks] page of each logical block
  int32_t block_len;           //   (NULL: contiguous [B][Hkv][S_max][d]; the tensor maps'
  int32_t max_blocks;          //   outer coordinate is then the page, the token one the
  int64_t num_blocks;          //   row inside it)
  float scale_log2;  // softmax_scale * log2(e)
  int32_t B, Tq, Hq, Hkv, G;
  int32_t S_max;  // tokens at or past S_max do not exist
  int32_t n_split, n_chunk, m_tiles;
  int32_t zero_empty;  // write o = 0 for items with no visible token
  int32_t ring_n;      // pass-Q ring: ranks (0: off) and query rows each rank owns; B then
  int32_t ring_bq;     //   counts ring_n * ring_n * ring_bq work rows (rank, step, slot)
  const int32_t* bounds;  // device [B][n_split + 1], or NULL: one split [0, S_max) per row
};

#ifdef __CUDACC__
// Token range [*lo, *hi) from bound ja to bound jb of KV row b (a split: jb = ja + 1; the
// union of all splits: 0 and n_split), clipped to the row's length and to S_max.
__device__ __forceinline__ void split_range(const PartialParams& p, int b, int ja, int jb, int seq_len, int* lo,
                                            int* hi) {
  int a = 0, e = p.S_max;
  if (p.bounds) {
    const int32_t* bnd = p.bounds + static_cast<int64_t>(b) * (p.n_split + 1);
    a = __ldg(bnd + ja);
    e = __ldg(bnd + jb);
  }
  *lo = max(a, 0);
  *hi = min(min(e, seq_len), p.S_max);
}

// Tile-aligned window [*win_lo, *win_hi) of chunk c of the token range [lo, hi): from the
// tile holding lo, the range's tiles are dealt out in n_chunk runs of equal length (the
// last ones shorter or empty).  An empty range gives an empty window.
__device__ __forceinline__ void chunk_window(const PartialParams& p, int lo, int hi, int c, int* win_lo, int* win_hi) {
  const int a = (lo / kTileN) * kTileN;
  const int tiles = hi > a ? (hi - a + kTileN - 1) / kTileN : 0;
  const int ct = (tiles + p.n_chunk - 1) / p.n_chunk;
  *win_lo = a + c * ct * kTileN;
  *win_hi = *win_lo + ct * kTileN;
}

// Page holding logical token `tok` of sequence b in a paged cache (the tensor maps then
// take (tok % block_len, page) where a contiguous cache takes (tok, b)).
__device__ __forceinline__ int kv_page_of(const PartialParams& p, int b, int tok) {
  return __ldg(p.block_table + static_cast<int64_t>(b) * p.max_blocks + tok / p.block_len);
}
#endif

// Supported GQA kernel variants.
enum class GqaVariant {
  kBf16D64Decode,
  kBf16D128Decode,
  kFp8D128Decode,
  kBf16D64Prefill,
  kBf16D128Prefill,
  kFp8D128Prefill,
};

struct GqaLaunchInfo {
  int rows_per_cta;  // M rows handled by one work item
  int threads;
  int smem_bytes;
  int ctas_per_sm;    // resident CTAs per SM the variant is built for
  int ctas_per_item = 1;  // CTAs that share one work item (2: a cluster pair)
};

GqaLaunchInfo gqa_launch_info(GqaVariant v);

cudaError_t launch_gqa_partial(GqaVariant v, const PartialParams& p, const CUtensorMap& tmk,
                               const CUtensorMap& tmv, int64_t n_items, cudaStream_t stream);

// MLA latent variant (dk = 576 latent+rope, dv = 512, one shared latent "head").
// Tiles are 32 tokens; the tensor map's box is 64 elements x 32 tokens.
constexpr int kMlaTileN = 32;
GqaLaunchInfo mla_launch_info();
cudaError_t launch_mla_partial(const PartialParams& p, const CUtensorMap& tmk, int64_t n_items, cudaStream_t stream);

// Tensor-core (tcgen05) attention for query tiles of >= 128 rows (see attn_tc.cu):
// bf16 KV, dk = dv = 128, G = Hq / Hkv dividing 128.  Work item = (b, g, [split j,]
// 256-row tile); `fused` processes the union of all splits and writes the final bf16
// output and lse, otherwise one fp32 partial per split goes to p.out_o / p.out_lse.
struct TcAttnExtra {
  int32_t fused;
  void* out_bf16;
  float* out_lse;
  // partial mode with one split: merge the result into the running (out_o, out_lse) held
  // there already instead of overwriting it (a pass-KV ring step)
  int32_t accumulate = 0;
  // MLA over a contiguous latent: its base and byte strides (sequence, token), for the value
  // CTA's L2 prefetches of the score CTA's coming tiles (NULL: none)
  const uint8_t* kv = nullptr;
  int64_t kv_seq_bytes = 0, kv_tok_bytes = 0;
};
int tc_attn_rows_per_cta();
int tc_attn_kv_tile();  // tokens per K/V tile = rows of the K/V tensor-map box
cudaError_t launch_tc_attn(const PartialParams& p, const TcAttnExtra& x, const CUtensorMap& tmq,
                           const CUtensorMap& tmk, const CUtensorMap& tmv, int64_t n_items, cudaStream_t stream);

// Tensor-core MLA latent attention (see mla_tc.cu): a cluster pair per work item of the
// partial decomposition (b, split j, chunk c, 128-row tile), writing fp32 partials.
// tml: the latent as (dim, token row, head, sequence | page) with 64 x kv_tile boxes;
// tmg / tmv (contiguous caches): the latent's chunked view (64 dims, token row, 64-dim
// slice, sequence) with boxes of (64, score tile, group slices) and (64, kv tile, 8).
int mla_tc_rows_per_item();
int mla_tc_kv_tile();
int mla_tc_score_tile();
int mla_tc_group_slices();
cudaError_t launch_mla_tc(const PartialParams& p, const TcAttnExtra& x, const CUtensorMap& tmq,
                          const CUtensorMap& tml, const CUtensorMap& tmg, const CUtensorMap& tmv, int64_t n_items,
                          cudaStream_t stream);

// tcgen05 self-test GEMM (see umma_selftest.cu).
cudaError_t launch_umma_selftest(const CUtensorMap& ta, const CUtensorMap& tb, float* C, int N, bool b_mn_major,
                                 bool a_tmem, unsigned int* err, cudaStream_t stream);

// Merge n_in partials per output group: in_o [G_out][n_in][R][dv], in_lse [G_out][n_in][R]
// -> out [G_out][R][dv] (fp32 or bf16) and out_lse [G_out][R].
// acc <- exact two-way LSE merge of acc and in (rows of dv fp32 values, lse per row).
cudaError_t launch_merge_into(float* acc_o, float* acc_lse, const float* in_o, const float* in_lse, int64_t R,
                              int32_t dv, cudaStream_t stream);
cudaError_t launch_merge(const float* in_o, const float* in_lse, int32_t n_in, int32_t g_out, int64_t R,
                         int32_t dv, void* out, bool out_bf16, float* out_lse, cudaStream_t stream);

}  // namespace skv
