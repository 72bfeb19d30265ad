// C-ABI entry points of libsplitkv_attn.so: argument validation, work decomposition,
// TMA descriptor set-up and dispatch to the kernels.  See include/splitkv_attn.h for
// the contract of every call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <vector>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/splitkv_attn.h"
#include "../../include/splitkv_attn_selftest.h"
#include "skv_common.cuh"
#include "skv_internal.h"

// Device error record written by kernels whose bounded waits gave up (layout: see
// DevErrWord in skv_common.cuh).
__device__ unsigned int g_skv_device_error[skv::kDevErrWords] = {0};

namespace {

using namespace skv;

thread_local std::string t_last_error;

skv_status fail(skv_status code, const std::string& msg) {
  t_last_error = msg;
  return code;
}

skv_status cuda_fail(cudaError_t e, const char* where) {
  t_last_error = std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return SKV_ECUDA;
}

constexpr int kMaxDevices = 64;

unsigned int* device_error_word(cudaError_t* err) {
  static unsigned int* cache[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    *err = cudaGetSymbolAddress(&ptr, g_skv_device_error);
    if (*err != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned int*>(ptr);
  }
  return cache[dev];
}

// SM count and resident CTAs per SM of a kernel variant (fallback when no device is
// visible, e.g. for size queries on a build host: a GB300's 152 SMs, 2 CTAs per SM).
int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    return 152;
  }
  return sms;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn(cudaError_t* err) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  static cudaError_t once_err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    once_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (once_err == cudaSuccess && q != cudaDriverEntryPointSuccess) once_err = cudaErrorNotSupported;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  *err = once_err;
  return fn;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------------ kernel timing

// Events around the attention kernel of each call while timing is on (host-thread state;
// the events are created on first use, on the device current at that time).
struct KernelTiming {
  static constexpr int kMax = 4096;
  bool on = false;
  int n = 0;
  cudaEvent_t ev[2 * kMax] = {};
};
thread_local KernelTiming t_timing;

cudaError_t timing_mark(bool after, cudaStream_t stream) {
  KernelTiming& t = t_timing;
  if (!t.on || t.n >= KernelTiming::kMax) return cudaSuccess;
  cudaEvent_t& e = t.ev[2 * t.n + (after ? 1 : 0)];
  if (!e) {
    cudaError_t r = cudaEventCreate(&e);
    if (r != cudaSuccess) return r;
  }
  cudaError_t r = cudaEventRecord(e, stream);
  if (after) ++t.n;
  return r;
}

// ------------------------------------------------------------------ plan of a call

struct Plan {
  bool mla = false;
  GqaVariant variant;
  int rows_per_cta = 0;
  int m_tiles = 1;
  int n_chunk = 1;
  int64_t n_items = 0;
  int n_part = 0;  // n_split * n_chunk
};

bool is_mla_shape(const skv_desc* d) {
  return d->dk == 576 && d->dv == 512 && d->Hkv == 1 && d->kv_dtype == SKV_KV_BF16;
}

// The MLA latent with a head count dividing 128 runs on the tensor-core cluster kernel.
bool use_mla_tc(const skv_desc* d) {
  const int G = d->Hq / d->Hkv;
  return is_mla_shape(d) && G <= 128 && 128 % G == 0;
}

bool is_gqa_shape(const skv_desc* d) {
  if (d->dk != d->dv) return false;
  if (d->kv_dtype == SKV_KV_BF16) return d->dk == 64 || d->dk == 128;
  return d->dk == 128;
}

// Shape, dtype and stride checks of a call (the split bounds live in device memory and are
// never read on the host).
skv_status validate(const skv_desc* d, int32_t n_split) {
  if (!d) return fail(SKV_EINVAL, "desc is NULL");
  if (d->B <= 0 || d->Tq <= 0 || d->Hq <= 0 || d->Hkv <= 0 || d->dk <= 0 || d->dv <= 0)
    return fail(SKV_EINVAL, "B, Tq, Hq, Hkv, dk, dv must be positive");
  if (d->Hq % d->Hkv) return fail(SKV_EINVAL, "Hq must be a multiple of Hkv");
  if (d->S_max <= 0 || d->S_max >= (int64_t(1) << 31)) return fail(SKV_EINVAL, "S_max must be in [1, 2^31)");
  if (!std::isfinite(d->softmax_scale) || d->softmax_scale == 0.f)
    return fail(SKV_EINVAL, "softmax_scale must be finite and non-zero");
  if (d->kv_dtype != SKV_KV_BF16 && d->kv_dtype != SKV_KV_FP8_E4M3) return fail(SKV_EINVAL, "unknown kv_dtype");
  if (d->kv_dtype == SKV_KV_FP8_E4M3 && (d->scale_block <= 0 || d->scale_block % kTileN))
    return fail(SKV_EINVAL, "scale_block must be a positive multiple of 64 for fp8 KV");
  if (n_split < 1) return fail(SKV_EINVAL, "n_split must be >= 1");
  if (static_cast<int64_t>(d->B) * (n_split + 1) >= (int64_t(1) << 31))
    return fail(SKV_EINVAL, "B * (n_split + 1) must be below 2^31");
  for (int i = 0; i < 3; ++i) {
    if (d->q_strides[i] < 0 || d->k_strides[i] < 0 || d->v_strides[i] < 0)
      return fail(SKV_EINVAL, "strides must be non-negative");
    if (d->q_strides[i] % 8) return fail(SKV_EINVAL, "q strides must be multiples of 8 elements (16 bytes)");
  }
  const int esz = d->kv_dtype == SKV_KV_FP8_E4M3 ? 1 : 2;
  for (int i = 0; i < 3; ++i) {
    if ((d->k_strides[i] * esz) % 16 || (d->v_strides[i] * esz) % 16)
      return fail(SKV_EINVAL, "K/V strides must be multiples of 16 bytes");
  }
  if (d->k_strides[2] < d->dk || d->v_strides[2] < d->dv)
    return fail(SKV_EINVAL, "K/V token stride must cover a whole head row");
  if (!is_gqa_shape(d) && !is_mla_shape(d)) {
    return fail(SKV_EUNSUPPORTED, "unsupported head dims / dtype: supported are bf16 dk=dv in {64,128}, "
                                  "fp8-e4m3 dk=dv=128, and the bf16 MLA latent (Hkv=1, dk=576, dv=512)");
  }
  if (is_mla_shape(d)) {
    for (int i = 0; i < 3; ++i)
      if (d->k_strides[i] != d->v_strides[i])
        return fail(SKV_EINVAL, "MLA: v_cache must be the latent buffer itself (same strides as k_cache)");
  }
  return SKV_OK;
}

skv_status validate_ptrs(const skv_desc* d, const void* q, const void* k, const void* v, const float* ks,
                         const float* vs, const int32_t* seq_lens) {
  if (!q || !k || !v || !seq_lens) return fail(SKV_EINVAL, "q, k_cache, v_cache and seq_lens must be non-NULL");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16))
    return fail(SKV_EINVAL, "q, k_cache and v_cache must be 16-byte aligned");
  if (!aligned(seq_lens, 4)) return fail(SKV_EINVAL, "seq_lens must be 4-byte aligned");
  if (is_mla_shape(d) && k != v) return fail(SKV_EINVAL, "MLA: v_cache must equal k_cache (V is the latent)");
  if (d->kv_dtype == SKV_KV_FP8_E4M3) {
    if (!ks || !vs) return fail(SKV_EINVAL, "fp8 KV needs k_scale and v_scale");
    if (!aligned(ks, 4) || !aligned(vs, 4)) return fail(SKV_EINVAL, "scales must be 4-byte aligned");
  }
  return SKV_OK;
}

// The caller's split-bounds table: a device int32 array [B][n_split + 1].
skv_status validate_bounds(const int32_t* bounds) {
  if (!bounds) return fail(SKV_EINVAL, "split_bounds is NULL");
  if (!aligned(bounds, 4)) return fail(SKV_EINVAL, "split_bounds must be 4-byte aligned");
  return SKV_OK;
}

// Work decomposition of a partial launch.  Long splits are cut into chunks so that the grid
// fills the GPU; the host does not read the split bounds, so it plans for splits of the
// allocated S_max cut into n_split equal parts, and each item sizes its chunk from its own
// split's length on the device.  max_chunk > 0 caps the chunks per split.
Plan make_plan(const skv_desc* d, int32_t n_split, int max_chunk = 0) {
  Plan pl;
  const int G = d->Hq / d->Hkv;
  const bool fp8 = d->kv_dtype == SKV_KV_FP8_E4M3;
  const bool decode = static_cast<int64_t>(d->Tq) * G <= 16;
  pl.mla = is_mla_shape(d);
  if (fp8)
    pl.variant = decode ? GqaVariant::kFp8D128Decode : GqaVariant::kFp8D128Prefill;
  else if (d->dk == 64)
    pl.variant = decode ? GqaVariant::kBf16D64Decode : GqaVariant::kBf16D64Prefill;
  else
    pl.variant = decode ? GqaVariant::kBf16D128Decode : GqaVariant::kBf16D128Prefill;
  GqaLaunchInfo li = pl.mla ? mla_launch_info() : gqa_launch_info(pl.variant);
  if (pl.mla && use_mla_tc(d)) li = GqaLaunchInfo{mla_tc_rows_per_item(), 224, 0, 1, 2};
  pl.rows_per_cta = li.rows_per_cta;
  const int64_t rows = static_cast<int64_t>(d->Tq) * G;
  pl.m_tiles = static_cast<int>((rows + li.rows_per_cta - 1) / li.rows_per_cta);

  // expected split length in tiles: S_max cut into n_split equal splits
  const int64_t split_tok = (d->S_max + n_split - 1) / n_split;
  const int64_t max_tiles = (split_tok + kTileN - 1) / kTileN;
  const int64_t base = static_cast<int64_t>(d->B) * d->Hkv * n_split * pl.m_tiles;
  const int64_t slots =  // work items resident at once
      std::max<int64_t>(1, static_cast<int64_t>(device_sm_count()) * li.ctas_per_sm / li.ctas_per_item);
  pl.n_chunk = 1;
  if (max_tiles > 1 && base < 4 * slots && max_chunk != 1) {
    // Cut every split into n chunks so that the grid fills the GPU in whole waves;
    // cost model: waves * (tiles per chunk + per-CTA overhead of ~3 tiles).
    double best = 1e300;
    int64_t n_hi = std::min<int64_t>(max_tiles, 512);
    if (max_chunk > 0) n_hi = std::min<int64_t>(n_hi, max_chunk);
    for (int64_t n = 1; n <= n_hi; ++n) {
      const int64_t ct = (max_tiles + n - 1) / n;
      const int64_t nn = (max_tiles + ct - 1) / ct;
      const int64_t waves = (base * nn + slots - 1) / slots;
      const double cost = static_cast<double>(waves) * static_cast<double>(ct + 3);
      if (cost < best * 0.999) {
        best = cost;
        pl.n_chunk = static_cast<int>(nn);
      }
    }
  }
  pl.n_part = n_split * pl.n_chunk;
  pl.n_items = base * pl.n_chunk;
  return pl;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shapes served by the tensor-core (tcgen05) attention kernel: bf16 KV, dk = dv = 128,
// G dividing 128 and at least one full 128-row query tile per KV head.
bool use_tc(const skv_desc* d) {
  if (d->kv_dtype != SKV_KV_BF16 || d->dk != 128 || d->dv != 128) return false;
  const int G = d->Hq / d->Hkv;
  if (G > 128 || 128 % G) return false;
  return static_cast<int64_t>(d->Tq) * G >= 128;
}

size_t ws_bytes_for(const skv_desc* d, int n_part) {
  const size_t rows = static_cast<size_t>(d->B) * d->Tq * d->Hq;
  return align_up(static_cast<size_t>(n_part) * rows * d->dv * 4, 256) + align_up(static_cast<size_t>(n_part) * rows * 4, 256);
}

skv_status encode_kv_map(CUtensorMap* map, const void* base, const skv_desc* d, const int64_t* strides, int dim,
                         int box_rows, const skv_paged* pg = nullptr) {
  cudaError_t e;
  auto encode = get_encode_fn(&e);
  if (!encode) return cuda_fail(e == cudaSuccess ? cudaErrorNotSupported : e, "cuTensorMapEncodeTiled lookup");
  const bool fp8 = d->kv_dtype == SKV_KV_FP8_E4M3;
  const int esz = fp8 ? 1 : 2;
  // contiguous: (dim, token, head, sequence); paged: (dim, row in page, head, page)
  const int64_t rows = pg ? pg->block_len : d->S_max;
  const int64_t outer = pg ? pg->num_blocks : d->B;
  cuuint64_t gdim[4] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(d->Hkv), static_cast<cuuint64_t>(outer)};
  const int64_t tok_b = strides[2] * esz;
  int64_t head_b = strides[1] * esz, batch_b = strides[0] * esz;
  // a stride of a size-1 dimension is never stepped; give it any legal value
  if (d->Hkv == 1 || head_b == 0) head_b = std::max<int64_t>(head_b, tok_b * rows);
  if (outer == 1 || batch_b == 0) batch_b = std::max<int64_t>(batch_b, head_b * d->Hkv);
  cuuint64_t gstride[3] = {static_cast<cuuint64_t>(tok_b), static_cast<cuuint64_t>(head_b),
                           static_cast<cuuint64_t>(batch_b)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                      const_cast<void*>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return fail(SKV_ECUDA, buf);
  }
  return SKV_OK;
}

// The MLA latent [B][S_max][dk] viewed as (64 dims, token row, 64-dim slice, sequence): a
// box of (64, rows, slices, 1) lands in shared memory as `slices` consecutive 128-byte-
// swizzled [rows][64 dims] tiles, one copy for what would take rows/64 x slices boxes of the
// plain view.  (The slice stride, 128 bytes, is below the token stride; the map only adds the
// strides up per element.)
skv_status encode_latent_slices_map(CUtensorMap* map, const void* base, const skv_desc* d, int box_rows,
                                    int box_slices) {
  cudaError_t e;
  auto encode = get_encode_fn(&e);
  if (!encode) return cuda_fail(e == cudaSuccess ? cudaErrorNotSupported : e, "cuTensorMapEncodeTiled lookup");
  const int64_t row_b = d->k_strides[2] * 2;
  int64_t seq_b = d->k_strides[0] * 2;
  if (d->B == 1 || seq_b == 0) seq_b = std::max<int64_t>(seq_b, row_b * d->S_max);
  cuuint64_t gdim[4] = {64, static_cast<cuuint64_t>(d->S_max), static_cast<cuuint64_t>(d->dk / 64),
                        static_cast<cuuint64_t>(d->B)};
  cuuint64_t gstride[3] = {static_cast<cuuint64_t>(row_b), 128, static_cast<cuuint64_t>(seq_b)};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(box_slices), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gdim, gstride, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled (latent slices) failed (CUresult %d)", static_cast<int>(r));
    return fail(SKV_ECUDA, buf);
  }
  return SKV_OK;
}

// 2-D bf16 tensor map with 128-byte swizzle: `inner` contiguous elements per row,
// `outer` rows `row_bytes` apart, box of box_inner x box_outer.
skv_status encode_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                          uint32_t box_inner, uint32_t box_outer) {
  cudaError_t e;
  auto encode = get_encode_fn(&e);
  if (!encode) return cuda_fail(e == cudaSuccess ? cudaErrorNotSupported : e, "cuTensorMapEncodeTiled lookup");
  cuuint64_t gdim[2] = {inner, outer};
  cuuint64_t gstride[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled (2-D) failed (CUresult %d)", static_cast<int>(r));
    return fail(SKV_ECUDA, buf);
  }
  return SKV_OK;
}

// Fill the launch parameters common to every GQA partial launch.
skv_status fill_params(PartialParams* p, const skv_desc* d, const Plan& pl, const void* q, const float* ks,
                       const float* vs, const int32_t* seq_lens, const int32_t* bounds, int32_t n_split,
                       int64_t causal_offset, const int32_t* q_pos, const int32_t* k_pos, const skv_paged* pg,
                       float* out_o, float* out_lse, bool zero_empty) {
  std::memset(p, 0, sizeof(*p));
  cudaError_t e;
  p->err = device_error_word(&e);
  if (!p->err) return cuda_fail(e, "device error word");
  p->q = q;
  p->q_sb = d->q_strides[0];
  p->q_st = d->q_strides[1];
  p->q_sh = d->q_strides[2];
  p->k_scale = ks;
  p->v_scale = vs;
  p->scale_block = d->kv_dtype == SKV_KV_FP8_E4M3 ? d->scale_block : kTileN;
  p->n_scale_blk = static_cast<int32_t>((d->S_max + p->scale_block - 1) / p->scale_block);
  p->seq_lens = seq_lens;
  p->out_o = out_o;
  p->out_lse = out_lse;
  // positions replace the offset rule: no contiguous horizon to cut tiles at
  p->causal_offset = q_pos ? SKV_NO_CAUSAL : causal_offset;
  p->q_pos = q_pos;
  p->k_pos = k_pos;
  if (pg) {
    p->block_table = pg->block_table;
    p->block_len = pg->block_len;
    p->max_blocks = pg->max_blocks;
    p->num_blocks = pg->num_blocks;
  }
  p->scale_log2 = d->softmax_scale * 1.4426950408889634f;
  p->B = d->B;
  p->Tq = d->Tq;
  p->Hq = d->Hq;
  p->Hkv = d->Hkv;
  p->G = d->Hq / d->Hkv;
  p->S_max = static_cast<int32_t>(d->S_max);
  p->n_split = n_split;
  p->n_chunk = pl.n_chunk;
  p->m_tiles = pl.m_tiles;
  p->zero_empty = zero_empty ? 1 : 0;
  p->bounds = bounds;
  return SKV_OK;
}

// Query tensor map for the tensor-core kernel: dims (d, head, row, batch), box
// (64, G, 128/G, 1) so that one box is a 128-row x 128-byte K-major tile.
skv_status encode_q_map(CUtensorMap* map, const void* q, const skv_desc* d) {
  cudaError_t e;
  auto encode = get_encode_fn(&e);
  if (!encode) return cuda_fail(e == cudaSuccess ? cudaErrorNotSupported : e, "cuTensorMapEncodeTiled lookup");
  const int G = d->Hq / d->Hkv;
  cuuint64_t gdim[4] = {static_cast<cuuint64_t>(d->dk), static_cast<cuuint64_t>(d->Hq),
                        static_cast<cuuint64_t>(d->Tq), static_cast<cuuint64_t>(d->B)};
  int64_t sh = d->q_strides[2] * 2, st = d->q_strides[1] * 2, sb = d->q_strides[0] * 2;
  if (sh == 0) sh = d->dk * 2;
  if (d->Tq == 1 || st == 0) st = std::max<int64_t>(st, sh * d->Hq);
  if (d->B == 1 || sb == 0) sb = std::max<int64_t>(sb, st * d->Tq);
  cuuint64_t gstride[3] = {static_cast<cuuint64_t>(sh), static_cast<cuuint64_t>(st), static_cast<cuuint64_t>(sb)};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(128 / G), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), gdim, gstride, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled (q) failed (CUresult %d)", static_cast<int>(r));
    return fail(SKV_ECUDA, buf);
  }
  return SKV_OK;
}

// Tensor-core path: fused = one pass over every split (final bf16 out + lse), else one
// fp32 partial per split straight into out_o / out_lse.
skv_status run_tc(const skv_desc* d, const void* q, const void* k, const void* v, const int32_t* seq_lens,
                  const int32_t* bounds, int32_t n_split, int64_t causal_offset, const int32_t* q_pos,
                  const int32_t* k_pos, const skv_paged* pg, bool fused, float* out_o,
                  float* out_lse, void* out_bf16, float* lse_final, cudaStream_t stream, bool accumulate = false) {
  PartialParams p;
  Plan pl;
  pl.n_chunk = 1;
  const int rows = tc_attn_rows_per_cta();
  pl.m_tiles = static_cast<int>((static_cast<int64_t>(d->Tq) * (d->Hq / d->Hkv) + rows - 1) / rows);
  skv_status st = fill_params(&p, d, pl, q, nullptr, nullptr, seq_lens, bounds, n_split, causal_offset, q_pos,
                              k_pos, pg, out_o, out_lse, true);
  if (st != SKV_OK) return st;
  TcAttnExtra x;
  x.fused = fused ? 1 : 0;
  x.out_bf16 = out_bf16;
  x.out_lse = lse_final;
  x.accumulate = accumulate ? 1 : 0;
  CUtensorMap tmq, tmk, tmv;
  if ((st = encode_q_map(&tmq, q, d)) != SKV_OK) return st;
  // a paged cache is read in 64-token halves of a tile (pages hold multiples of 64 tokens)
  const int kv_box = pg ? tc_attn_kv_tile() / 2 : tc_attn_kv_tile();
  if ((st = encode_kv_map(&tmk, k, d, d->k_strides, d->dk, kv_box, pg)) != SKV_OK) return st;
  if ((st = encode_kv_map(&tmv, v, d, d->v_strides, d->dv, kv_box, pg)) != SKV_OK) return st;
  const int64_t n_items = static_cast<int64_t>(d->B) * d->Hkv * (fused ? 1 : n_split) * pl.m_tiles;
  cudaError_t e = timing_mark(false, stream);
  if (e == cudaSuccess) e = launch_tc_attn(p, x, tmq, tmk, tmv, n_items, stream);
  if (e == cudaSuccess) e = timing_mark(true, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core attention launch");
  return SKV_OK;
}

skv_status run_partial(const skv_desc* d, const Plan& pl, const void* q, const void* k, const void* v,
                       const float* ks, const float* vs, const int32_t* seq_lens, const int32_t* bounds,
                       int32_t n_split, int64_t causal_offset, const int32_t* q_pos, const int32_t* k_pos,
                       const skv_paged* pg, float* out_o, float* out_lse, bool zero_empty, cudaStream_t stream,
                       int32_t ring_n = 0) {
  PartialParams p;
  skv_status st = fill_params(&p, d, pl, q, ks, vs, seq_lens, bounds, n_split, causal_offset, q_pos, k_pos, pg,
                              out_o, out_lse, zero_empty);
  if (st != SKV_OK) return st;
  if (ring_n > 0) {  // pass-Q: d->B counts (rank, ring step, slot) work rows
    p.ring_n = ring_n;
    p.ring_bq = d->B / (ring_n * ring_n);
  }
  CUtensorMap tmk, tmv;
  cudaError_t e;
  if (pl.mla) {
    if (q_pos) return fail(SKV_EUNSUPPORTED, "position-masked attention is not supported for the MLA latent shape");
    if (use_mla_tc(d)) {
      // the latent is both K (all 576 dims) and V (its first 512): a per-slice map with
      // 64-dim x 64-token boxes, and over a contiguous cache the chunked view that lets one
      // copy land a whole score group (CTA 0) or value tile (CTA 1)
      CUtensorMap tmq, tmg, tmv2;
      if ((st = encode_q_map(&tmq, q, d)) != SKV_OK) return st;
      if ((st = encode_kv_map(&tmk, k, d, d->k_strides, d->dk, mla_tc_kv_tile(), pg)) != SKV_OK) return st;
      if (pg) {  // paged: the per-slice map serves every load
        tmg = tmk;
        tmv2 = tmk;
      } else {
        if ((st = encode_latent_slices_map(&tmg, k, d, mla_tc_score_tile(), mla_tc_group_slices())) != SKV_OK)
          return st;
        if ((st = encode_latent_slices_map(&tmv2, k, d, mla_tc_kv_tile(), 8)) != SKV_OK) return st;
      }
      TcAttnExtra x;
      x.fused = 0;
      x.out_bf16 = nullptr;
      x.out_lse = nullptr;
      if (!pg) {
        x.kv = static_cast<const uint8_t*>(k);
        x.kv_seq_bytes = d->k_strides[0] * 2;
        x.kv_tok_bytes = d->k_strides[2] * 2;
      }
      e = timing_mark(false, stream);
      if (e == cudaSuccess) e = launch_mla_tc(p, x, tmq, tmk, tmg, tmv2, pl.n_items, stream);
      if (e == cudaSuccess) e = timing_mark(true, stream);
      if (e != cudaSuccess) return cuda_fail(e, "MLA tensor-core attention launch");
      return SKV_OK;
    }
    // one latent map serves K (all 576 columns) and V (its first 512 columns)
    if ((st = encode_kv_map(&tmk, k, d, d->k_strides, d->dk, kMlaTileN, pg)) != SKV_OK) return st;
    e = timing_mark(false, stream);
    if (e == cudaSuccess) e = launch_mla_partial(p, tmk, pl.n_items, stream);
    if (e == cudaSuccess) e = timing_mark(true, stream);
    if (e != cudaSuccess) return cuda_fail(e, "MLA partial attention launch");
    return SKV_OK;
  }
  if ((st = encode_kv_map(&tmk, k, d, d->k_strides, d->dk, kTileN, pg)) != SKV_OK) return st;
  if ((st = encode_kv_map(&tmv, v, d, d->v_strides, d->dv, kTileN, pg)) != SKV_OK) return st;
  e = timing_mark(false, stream);
  if (e == cudaSuccess) e = launch_gqa_partial(pl.variant, p, tmk, tmv, pl.n_items, stream);
  if (e == cudaSuccess) e = timing_mark(true, stream);
  if (e != cudaSuccess) return cuda_fail(e, "partial attention launch");
  return SKV_OK;
}

}  // namespace

extern "C" {

int32_t splitkv_version(void) { return (1 << 16) | 0; }

skv_status splitkv_kernel_timing(int32_t enable) {
  t_timing.on = enable != 0;
  if (t_timing.on) t_timing.n = 0;
  return SKV_OK;
}

skv_status splitkv_kernel_timing_read(float* total_ms, int32_t* launches) {
  if (!total_ms || !launches) return fail(SKV_EINVAL, "total_ms and launches must be non-NULL");
  float sum = 0.f;
  for (int i = 0; i < t_timing.n; ++i) {
    cudaError_t e = cudaEventSynchronize(t_timing.ev[2 * i + 1]);
    if (e != cudaSuccess) return cuda_fail(e, "kernel timing event");
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, t_timing.ev[2 * i], t_timing.ev[2 * i + 1]);
    if (e != cudaSuccess) return cuda_fail(e, "kernel timing elapsed");
    sum += ms;
  }
  *total_ms = sum;
  *launches = t_timing.n;
  return SKV_OK;
}

const char* splitkv_last_error(void) { return t_last_error.c_str(); }

skv_status splitkv_device_error_detail(uint32_t* record) {
  if (!record) return fail(SKV_EINVAL, "record is NULL");
  unsigned int v[kDevErrWords] = {0}, zero[kDevErrWords] = {0};
  cudaError_t e = cudaMemcpyFromSymbol(v, g_skv_device_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "read device error record");
  e = cudaMemcpyToSymbol(g_skv_device_error, zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "clear device error record");
  for (int i = 0; i < kDevErrWords; ++i) record[i] = v[i];
  return SKV_OK;
}

skv_status splitkv_device_error(uint32_t* code) {
  if (!code) return fail(SKV_EINVAL, "code is NULL");
  uint32_t rec[kDevErrWords];
  skv_status st = splitkv_device_error_detail(rec);
  if (st != SKV_OK) return st;
  *code = rec[0];
  return SKV_OK;
}

skv_status splitkv_selftest_umma_gemm(const void* A, const void* B, float* C, int32_t N, int32_t flags,
                                      void* stream) {
  const int32_t b_mn_major = flags & 1;
  const bool a_tmem = (flags & 2) != 0;
  if (!A || !B || !C) return fail(SKV_EINVAL, "A, B and C must be non-NULL");
  if (N != 64 && N != 128) return fail(SKV_EINVAL, "N must be 64 or 128");
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16)) return fail(SKV_EINVAL, "pointers must be 16-byte aligned");
  CUtensorMap ta, tb;
  skv_status st = encode_2d_bf16(&ta, A, 64, 128, 128, 64, 128);
  if (st != SKV_OK) return st;
  if (b_mn_major)
    st = encode_2d_bf16(&tb, B, static_cast<uint64_t>(N), 64, static_cast<uint64_t>(N) * 2, 64, 64);
  else
    st = encode_2d_bf16(&tb, B, 64, static_cast<uint64_t>(N), 128, 64, static_cast<uint32_t>(N));
  if (st != SKV_OK) return st;
  cudaError_t e;
  unsigned int* err = device_error_word(&e);
  if (!err) return cuda_fail(e, "device error word");
  e = launch_umma_selftest(ta, tb, C, N, b_mn_major != 0, a_tmem, err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 self-test launch");
  return SKV_OK;
}

skv_status attn_partial_workspace_size(const skv_desc* desc, int32_t n_split, size_t* bytes) {
  if (!bytes) return fail(SKV_EINVAL, "bytes is NULL");
  skv_status st = validate(desc, n_split);
  if (st != SKV_OK) return st;
  if (use_tc(desc)) {
    *bytes = 0;
    return SKV_OK;
  }
  const Plan pl = make_plan(desc, n_split);
  *bytes = pl.n_chunk > 1 ? ws_bytes_for(desc, pl.n_part) : 0;
  return SKV_OK;
}

}  // extern "C"

namespace {

// Paged-cache description of a *_paged call.
skv_status validate_paged(const skv_desc* d, const skv_paged* pg) {
  if (!pg) return fail(SKV_EINVAL, "paged is NULL");
  if (!pg->block_table || !aligned(pg->block_table, 4)) return fail(SKV_EINVAL, "block_table NULL or misaligned");
  if (pg->block_len <= 0 || pg->block_len % kTileN)
    return fail(SKV_EINVAL, "block_len must be a positive multiple of 64");
  if (pg->max_blocks <= 0 || pg->num_blocks <= 0) return fail(SKV_EINVAL, "max_blocks and num_blocks must be positive");
  if (pg->num_blocks >= (int64_t(1) << 31)) return fail(SKV_EINVAL, "num_blocks must be below 2^31");
  if (d->S_max > static_cast<int64_t>(pg->max_blocks) * pg->block_len)
    return fail(SKV_EINVAL, "S_max must be at most max_blocks * block_len");
  if (d->kv_dtype == SKV_KV_FP8_E4M3 && pg->block_len % d->scale_block)
    return fail(SKV_EINVAL, "block_len must be a multiple of scale_block for fp8 pages");
  return SKV_OK;
}

// Positions of a *_pos call: both arrays present, aligned for the kernels' vector loads.
skv_status validate_positions(const skv_desc* d, const int32_t* q_pos, const int32_t* k_pos) {
  if (!q_pos || !k_pos) return fail(SKV_EINVAL, "q_pos and k_pos must be non-NULL");
  if (!aligned(q_pos, 4) || !aligned(k_pos, 16)) return fail(SKV_EINVAL, "q_pos must be 4-byte, k_pos 16-byte aligned");
  if (d->S_max % 4) return fail(SKV_EINVAL, "S_max must be a multiple of 4 with k_pos");
  if (is_mla_shape(d)) return fail(SKV_EUNSUPPORTED, "position-masked attention is not supported for the MLA latent shape");
  return SKV_OK;
}

// Checks shared by every public call taking a bounds table: the shape and the table pointer.
skv_status validate_call(const skv_desc* d, const int32_t* bounds, int32_t n_split) {
  skv_status st = validate(d, n_split);
  if (st != SKV_OK) return st;
  return validate_bounds(bounds);
}

// split_bounds may be NULL here (internal callers): one split [0, S_max) per sequence.
skv_status attn_partial_impl(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                             const int32_t* split_bounds, int32_t n_split, int64_t causal_offset,
                             const int32_t* q_pos, const int32_t* k_pos, const skv_paged* pg, float* out_partial,
                             float* lse_partial, void* workspace, size_t workspace_bytes, void* stream) {
  skv_status st = validate(desc, n_split);
  if (st != SKV_OK) return st;
  if ((st = validate_ptrs(desc, q, k_cache, v_cache, k_scale, v_scale, seq_lens)) != SKV_OK) return st;
  if (!out_partial || !lse_partial) return fail(SKV_EINVAL, "out_partial and lse_partial must be non-NULL");
  if (!aligned(out_partial, 16) || !aligned(lse_partial, 4)) return fail(SKV_EINVAL, "outputs misaligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (use_tc(desc)) {
    return run_tc(desc, q, k_cache, v_cache, seq_lens, split_bounds, n_split, causal_offset, q_pos, k_pos, pg, false,
                  out_partial, lse_partial, nullptr, nullptr, s);
  }
  const Plan pl = make_plan(desc, n_split);
  if (pl.n_chunk == 1) {
    return run_partial(desc, pl, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split,
                       causal_offset, q_pos, k_pos, pg, out_partial, lse_partial, true, s);
  }
  const size_t need = ws_bytes_for(desc, pl.n_part);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
    return fail(SKV_EWORKSPACE, "workspace missing, misaligned or smaller than attn_partial_workspace_size()");
  const size_t rows = static_cast<size_t>(desc->B) * desc->Tq * desc->Hq;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_l = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         align_up(static_cast<size_t>(pl.n_part) * rows * desc->dv * 4, 256));
  st = run_partial(desc, pl, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split, causal_offset,
                   q_pos, k_pos, pg, ws_o, ws_l, false, s);
  if (st != SKV_OK) return st;
  cudaError_t e = launch_merge(ws_o, ws_l, pl.n_chunk, n_split, static_cast<int64_t>(rows), desc->dv, out_partial,
                               false, lse_partial, s);
  if (e != cudaSuccess) return cuda_fail(e, "chunk merge launch");
  return SKV_OK;
}

// The fused call's partials (and their merge) in `workspace`, planned by `pl`.
skv_status decode_with_plan(const skv_desc* desc, const Plan& pl, const void* q, const void* k_cache,
                            const void* v_cache, const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                            const int32_t* split_bounds, int32_t n_split, int64_t causal_offset, const int32_t* q_pos,
                            const int32_t* k_pos, const skv_paged* pg, void* out, float* lse, void* workspace,
                            cudaStream_t s) {
  const size_t rows = static_cast<size_t>(desc->B) * desc->Tq * desc->Hq;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_l = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         align_up(static_cast<size_t>(pl.n_part) * rows * desc->dv * 4, 256));
  skv_status st = run_partial(desc, pl, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split,
                              causal_offset, q_pos, k_pos, pg, ws_o, ws_l, false, s);
  if (st != SKV_OK) return st;
  cudaError_t e = launch_merge(ws_o, ws_l, pl.n_part, 1, static_cast<int64_t>(rows), desc->dv, out, true, lse, s);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return SKV_OK;
}

skv_status gqa_decode_attn_impl(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                                const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                                const int32_t* split_bounds, int32_t n_split, int64_t causal_offset,
                                const int32_t* q_pos, const int32_t* k_pos, const skv_paged* pg, void* out,
                                float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  skv_status st = validate(desc, n_split);
  if (st != SKV_OK) return st;
  if ((st = validate_ptrs(desc, q, k_cache, v_cache, k_scale, v_scale, seq_lens)) != SKV_OK) return st;
  if (!out || !lse) return fail(SKV_EINVAL, "out and lse must be non-NULL");
  if (!aligned(out, 8) || !aligned(lse, 4)) return fail(SKV_EINVAL, "outputs misaligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (use_tc(desc)) {
    if (!aligned(out, 16)) return fail(SKV_EINVAL, "out must be 16-byte aligned for this shape");
    return run_tc(desc, q, k_cache, v_cache, seq_lens, split_bounds, n_split, causal_offset, q_pos, k_pos, pg, true,
                  nullptr, nullptr, out, lse, s);
  }
  const Plan pl = make_plan(desc, n_split);
  const size_t need = ws_bytes_for(desc, pl.n_part);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
    return fail(SKV_EWORKSPACE, "workspace missing, misaligned or smaller than gqa_decode_attn_workspace_size()");
  return decode_with_plan(desc, pl, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split,
                          causal_offset, q_pos, k_pos, pg, out, lse, workspace, s);
}

}  // namespace

extern "C" {

skv_status attn_partial(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                        const int32_t* split_bounds, int32_t n_split, int64_t causal_offset, float* out_partial,
                        float* lse_partial, void* workspace, size_t workspace_bytes, void* stream) {
  skv_status st = validate_call(desc, split_bounds, n_split);
  if (st != SKV_OK) return st;
  return attn_partial_impl(desc, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split,
                           causal_offset, nullptr, nullptr, nullptr, out_partial, lse_partial, workspace,
                           workspace_bytes, stream);
}

skv_status attn_partial_pos(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                            const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                            const int32_t* split_bounds, int32_t n_split, const int32_t* q_pos,
                            const int32_t* k_pos, float* out_partial, float* lse_partial, void* workspace,
                            size_t workspace_bytes, void* stream) {
  skv_status st = validate_call(desc, split_bounds, n_split);
  if (st != SKV_OK) return st;
  if ((st = validate_positions(desc, q_pos, k_pos)) != SKV_OK) return st;
  return attn_partial_impl(desc, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split, 0, q_pos,
                           k_pos, nullptr, out_partial, lse_partial, workspace, workspace_bytes, stream);
}

skv_status attn_merge_lse(int32_t n_split, int32_t B, int32_t Tq, int32_t Hq, int32_t dv, const float* out_partials,
                          const float* lse_partials, void* out, float* lse, void* stream) {
  if (n_split < 1 || B <= 0 || Tq <= 0 || Hq <= 0 || dv <= 0) return fail(SKV_EINVAL, "sizes must be positive");
  if (dv % 4) return fail(SKV_EINVAL, "dv must be a multiple of 4");
  if (!out_partials || !lse_partials || !out || !lse) return fail(SKV_EINVAL, "pointers must be non-NULL");
  if (!aligned(out_partials, 16) || !aligned(out, 8) || !aligned(lse_partials, 4) || !aligned(lse, 4))
    return fail(SKV_EINVAL, "pointers misaligned");
  const int64_t rows = static_cast<int64_t>(B) * Tq * Hq;
  cudaError_t e = launch_merge(out_partials, lse_partials, n_split, 1, rows, dv, out, true, lse,
                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return SKV_OK;
}

skv_status gqa_decode_attn_workspace_size(const skv_desc* desc, int32_t n_split, size_t* bytes) {
  if (!bytes) return fail(SKV_EINVAL, "bytes is NULL");
  skv_status st = validate(desc, n_split);
  if (st != SKV_OK) return st;
  if (use_tc(desc)) {  // the tensor-core path merges the splits on the fly: no partials
    *bytes = 0;
    return SKV_OK;
  }
  const Plan pl = make_plan(desc, n_split);
  *bytes = ws_bytes_for(desc, pl.n_part);
  return SKV_OK;
}

skv_status gqa_decode_attn(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                           const int32_t* split_bounds, int32_t n_split, int64_t causal_offset, void* out,
                           float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  skv_status st = validate_call(desc, split_bounds, n_split);
  if (st != SKV_OK) return st;
  return gqa_decode_attn_impl(desc, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split,
                              causal_offset, nullptr, nullptr, nullptr, out, lse, workspace, workspace_bytes, stream);
}

skv_status attn_partial_paged(const skv_desc* desc, const skv_paged* paged, const void* q, const void* k_cache,
                              const void* v_cache, const float* k_scale, const float* v_scale,
                              const int32_t* seq_lens, const int32_t* split_bounds, int32_t n_split,
                              int64_t causal_offset, float* out_partial, float* lse_partial, void* workspace,
                              size_t workspace_bytes, void* stream) {
  skv_status st = validate_call(desc, split_bounds, n_split);
  if (st != SKV_OK) return st;
  if ((st = validate_paged(desc, paged)) != SKV_OK) return st;
  return attn_partial_impl(desc, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split,
                           causal_offset, nullptr, nullptr, paged, out_partial, lse_partial, workspace,
                           workspace_bytes, stream);
}

skv_status gqa_decode_attn_paged(const skv_desc* desc, const skv_paged* paged, const void* q, const void* k_cache,
                                 const void* v_cache, const float* k_scale, const float* v_scale,
                                 const int32_t* seq_lens, const int32_t* split_bounds, int32_t n_split,
                                 int64_t causal_offset, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  skv_status st = validate_call(desc, split_bounds, n_split);
  if (st != SKV_OK) return st;
  if ((st = validate_paged(desc, paged)) != SKV_OK) return st;
  return gqa_decode_attn_impl(desc, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split,
                              causal_offset, nullptr, nullptr, paged, out, lse, workspace, workspace_bytes, stream);
}

skv_status attn_ring_step_workspace_size(const skv_desc* desc, size_t* bytes) {
  if (!bytes) return fail(SKV_EINVAL, "bytes is NULL");
  size_t part_ws = 0;
  skv_status st = attn_partial_workspace_size(desc, 1, &part_ws);
  if (st != SKV_OK) return st;
  const size_t rows = static_cast<size_t>(desc->B) * desc->Tq * desc->Hq;
  *bytes = align_up(part_ws, 256) + align_up(rows * desc->dv * 4, 256) + align_up(rows * 4, 256);
  return SKV_OK;
}

skv_status attn_ring_step(const skv_desc* desc, const void* q, const void* k_block, const void* v_block,
                          const float* k_scale, const float* v_scale, const int32_t* seq_lens, int64_t causal_offset,
                          int32_t first, float* o_acc, float* lse_acc, void* workspace, size_t workspace_bytes,
                          void* stream) {
  size_t need = 0;
  skv_status st = attn_ring_step_workspace_size(desc, &need);
  if (st != SKV_OK) return st;
  if (!o_acc || !lse_acc) return fail(SKV_EINVAL, "o_acc and lse_acc must be non-NULL");
  if (!aligned(o_acc, 16) || !aligned(lse_acc, 4)) return fail(SKV_EINVAL, "o_acc / lse_acc misaligned");
  if (desc->dv % 4) return fail(SKV_EINVAL, "dv must be a multiple of 4");
  // one split per sequence, the whole block: no bounds table (the kernels take [0, S_max))
  if (first) {  // the first block's partial is the running result
    return attn_partial_impl(desc, q, k_block, v_block, k_scale, v_scale, seq_lens, nullptr, 1, causal_offset,
                             nullptr, nullptr, nullptr, o_acc, lse_acc, workspace, workspace_bytes, stream);
  }
  if (use_tc(desc)) {  // the tensor-core kernel merges into the running output in its epilogue
    if ((st = validate_ptrs(desc, q, k_block, v_block, k_scale, v_scale, seq_lens)) != SKV_OK) return st;
    return run_tc(desc, q, k_block, v_block, seq_lens, nullptr, 1, causal_offset, nullptr, nullptr, nullptr,
                  false, o_acc, lse_acc, nullptr, nullptr, static_cast<cudaStream_t>(stream), true);
  }
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
    return fail(SKV_EWORKSPACE, "workspace missing, misaligned or smaller than attn_ring_step_workspace_size()");
  const size_t rows = static_cast<size_t>(desc->B) * desc->Tq * desc->Hq;
  size_t part_ws = 0;
  if ((st = attn_partial_workspace_size(desc, 1, &part_ws)) != SKV_OK) return st;
  char* base = static_cast<char*>(workspace);
  float* step_o = reinterpret_cast<float*>(base + align_up(part_ws, 256));
  float* step_l = reinterpret_cast<float*>(base + align_up(part_ws, 256) + align_up(rows * desc->dv * 4, 256));
  st = attn_partial_impl(desc, q, k_block, v_block, k_scale, v_scale, seq_lens, nullptr, 1, causal_offset, nullptr,
                         nullptr, nullptr, step_o, step_l, part_ws ? workspace : nullptr, part_ws, stream);
  if (st != SKV_OK) return st;
  cudaError_t e = launch_merge_into(o_acc, lse_acc, step_o, step_l, static_cast<int64_t>(rows), desc->dv,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ring-step merge launch");
  return SKV_OK;
}

skv_status gqa_decode_attn_pos(const skv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                               const int32_t* split_bounds, int32_t n_split, const int32_t* q_pos,
                               const int32_t* k_pos, void* out, float* lse, void* workspace, size_t workspace_bytes,
                               void* stream) {
  skv_status st = validate_call(desc, split_bounds, n_split);
  if (st != SKV_OK) return st;
  if ((st = validate_positions(desc, q_pos, k_pos)) != SKV_OK) return st;
  return gqa_decode_attn_impl(desc, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split, 0, q_pos,
                              k_pos, nullptr, out, lse, workspace, workspace_bytes, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// gqa_decode_attn_noalloc: the fused decode call for callers that cannot allocate
// device memory.  Its per-split / per-chunk partials live in a fixed scratch array
// compiled into this library instead of a caller-provided workspace.

namespace {

// Largest partial buffer the no-allocation entry point can use (32 MiB).  Every GPU
// that loads this library reserves it for the life of the process.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once per device
// (with that device current) and cached.  In host code the array's name only stands in
// for the symbol; only this looked-up address may be given to a kernel.
skv_status noalloc_scratch_ptr(void** out) {
  static void* cache[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SKV_EINVAL, "device index out of range");
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    if (!ptr) return fail(SKV_ECUDA, "cudaGetSymbolAddress returned NULL for the no-alloc scratch");
    cache[dev] = ptr;
  }
  *out = cache[dev];
  return SKV_OK;
}

}  // namespace

extern "C" skv_status gqa_decode_attn_noalloc(const skv_desc* desc, const void* q, const void* k_cache,
                                              const void* v_cache, const float* k_scale, const float* v_scale,
                                              const int32_t* seq_lens, const int32_t* split_bounds, int32_t n_split,
                                              int64_t causal_offset, void* out, float* lse, void* stream) {
  skv_status st = validate_call(desc, split_bounds, n_split);
  if (st != SKV_OK) return st;
  if ((st = validate_ptrs(desc, q, k_cache, v_cache, k_scale, v_scale, seq_lens)) != SKV_OK) return st;
  if (!out || !lse) return fail(SKV_EINVAL, "out and lse must be non-NULL");
  if (!aligned(out, 8) || !aligned(lse, 4)) return fail(SKV_EINVAL, "outputs misaligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (use_tc(desc)) {
    // the tensor-core shapes merge their splits inside the kernel: no partials, no scratch
    if (!aligned(out, 16)) return fail(SKV_EINVAL, "out must be 16-byte aligned for this shape");
    return run_tc(desc, q, k_cache, v_cache, seq_lens, split_bounds, n_split, causal_offset, nullptr, nullptr,
                  nullptr, true, nullptr, nullptr, out, lse, s);
  }
  Plan pl = make_plan(desc, n_split);
  if (ws_bytes_for(desc, pl.n_part) > kNoAllocScratchBytes) {
    // plan again with as many chunks per split as the scratch holds partials for
    int cap = pl.n_chunk - 1;
    while (cap >= 1 && ws_bytes_for(desc, n_split * cap) > kNoAllocScratchBytes) --cap;
    if (cap < 1) {
      char buf[320];
      snprintf(buf, sizeof buf,
               "gqa_decode_attn_noalloc: the %d split partials of this problem need %zu bytes but the built-in "
               "scratch holds %zu bytes; use gqa_decode_attn with a workspace",
               n_split, ws_bytes_for(desc, n_split), kNoAllocScratchBytes);
      return fail(SKV_EWORKSPACE, buf);
    }
    pl = make_plan(desc, n_split, cap);
  }
  void* scratch = nullptr;
  if ((st = noalloc_scratch_ptr(&scratch)) != SKV_OK) return st;
  // Nothing in the scratch has to start at zero: the partial kernel writes the lse of
  // every (part, row) slot before the merge reads it, and the merge never reads the o
  // of a slot whose lse is -inf.
  return decode_with_plan(desc, pl, q, k_cache, v_cache, k_scale, v_scale, seq_lens, split_bounds, n_split,
                          causal_offset, nullptr, nullptr, nullptr, out, lse, scratch, s);
}

// ------------------------------------------------------------------ pass-Q decode

namespace {

// A pass-Q call as one batched partial launch: the n_ranks * B work rows (rank, ring step,
// slot) and the n_ranks * B cache rows (rank, request) share one count, every cache row is
// one split [0, S_max) (no bounds table) clipped to its shard length on the device.
skv_status passq_setup(const skv_desc* d, int32_t n_ranks, skv_desc* vd) {
  if (!d) return fail(SKV_EINVAL, "desc is NULL");
  if (n_ranks < 1) return fail(SKV_EINVAL, "n_ranks must be >= 1");
  if (d->B <= 0 || d->B % n_ranks) return fail(SKV_EINVAL, "B must be a positive multiple of n_ranks");
  if (static_cast<int64_t>(n_ranks) * d->B >= (int64_t(1) << 30)) return fail(SKV_EINVAL, "n_ranks * B must be below 2^30");
  if (is_mla_shape(d)) return fail(SKV_EUNSUPPORTED, "pass-Q decode is not supported for the MLA latent shape");
  if (d->Tq != 1) return fail(SKV_EUNSUPPORTED, "pass-Q decode takes one query token per request (Tq = 1)");
  *vd = *d;
  vd->B = n_ranks * d->B;
  return validate(vd, 1);
}

}  // namespace

extern "C" {

skv_status gqa_decode_attn_passq_workspace_size(const skv_desc* desc, int32_t n_ranks, size_t* bytes) {
  if (!bytes) return fail(SKV_EINVAL, "bytes is NULL");
  skv_desc vd;
  skv_status st = passq_setup(desc, n_ranks, &vd);
  if (st != SKV_OK) return st;
  const Plan pl = make_plan(&vd, 1);
  *bytes = ws_bytes_for(&vd, pl.n_part);
  return SKV_OK;
}

skv_status gqa_decode_attn_passq(const skv_desc* desc, int32_t n_ranks, const void* q, const void* k_shards,
                                 const void* v_shards, const float* k_scale, const float* v_scale,
                                 const int32_t* shard_lens, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  skv_desc vd;
  skv_status st = passq_setup(desc, n_ranks, &vd);
  if (st != SKV_OK) return st;
  if ((st = validate_ptrs(&vd, q, k_shards, v_shards, k_scale, v_scale, shard_lens)) != SKV_OK) return st;
  if (!out || !lse) return fail(SKV_EINVAL, "out and lse must be non-NULL");
  if (!aligned(out, 8) || !aligned(lse, 4)) return fail(SKV_EINVAL, "outputs misaligned");
  const Plan pl = make_plan(&vd, 1);
  const size_t need = ws_bytes_for(&vd, pl.n_part);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
    return fail(SKV_EWORKSPACE, "workspace missing, misaligned or smaller than gqa_decode_attn_passq_workspace_size()");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(vd.B) * vd.Tq * vd.Hq;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_l = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         align_up(static_cast<size_t>(pl.n_part) * rows * vd.dv * 4, 256));
  // every rank, every ring step: partials land in the owners' exchange slots
  st = run_partial(&vd, pl, q, k_shards, v_shards, k_scale, v_scale, shard_lens, nullptr, 1, SKV_NO_CAUSAL,
                   nullptr, nullptr, nullptr, ws_o, ws_l, false, s, n_ranks);
  if (st != SKV_OK) return st;
  // the exchange delivered [owner][source rank][part] slabs: each owner merges its
  // n_ranks * n_part partials per query row
  const int64_t owner_rows = static_cast<int64_t>(desc->B / n_ranks) * desc->Tq * desc->Hq;
  cudaError_t e = launch_merge(ws_o, ws_l, n_ranks * pl.n_part, n_ranks, owner_rows, desc->dv, out, true, lse, s);
  if (e != cudaSuccess) return cuda_fail(e, "pass-Q merge launch");
  return SKV_OK;
}

}  // extern "C"
