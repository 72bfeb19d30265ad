// Exact merge of partial attention outputs by their log-sum-exp.
//
// For every output row: m = max_s lse_s, w_s = exp(lse_s - m), o = sum_s w_s o_s / sum_s w_s,
// lse = m + ln sum_s w_s -- the merge of "Helix Parallelism: Why Tensor Parallelism
// Hits a Wall at Million-Token Context" (section "Sharding the sequence instead",
// the merge after the All-to-All) and the exact-merge equation of "Context
// Parallelism for Scalable Million-Token Inference" (section "Pass-KV keeps queries
// local and circulates keys and values").  The merged lse (m + ln den) is the
// reading that makes a merged result mergeable again.  Partials with lse = -inf
// carry weight 0 and their o is never read; a row whose partials are all empty gets
// o = 0, lse = -inf.
//
// One warp per output row; each lane owns 4 consecutive output columns per pass
// (16-byte loads), so reads of the n_in partial rows are coalesced and read once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "skv_internal.h"

namespace skv {

namespace {

template <bool OUT_BF16>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ in_o, const float* __restrict__ in_lse,
                                                    int32_t n_in, int32_t g_out, int64_t R, int32_t dv,
                                                    void* __restrict__ out, float* __restrict__ out_lse) {
  // launched as a programmatic dependent of the partial kernel: wait until that grid has
  // completed and its partials are visible (a no-op for an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t row_id = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row_id >= static_cast<int64_t>(g_out) * R) return;
  const int64_t grp = row_id / R, r = row_id % R;
  const float* lse_base = in_lse + grp * n_in * R + r;  // + s*R
  const float* o_base = in_o + (grp * n_in * R + r) * dv;  // + s*R*dv

  float m = -INFINITY;
  for (int s = lane; s < n_in; s += 32) m = fmaxf(m, lse_base[static_cast<int64_t>(s) * R]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));

  float den = 0.f;
  if (m != -INFINITY) {
    for (int s = lane; s < n_in; s += 32) den += __expf(lse_base[static_cast<int64_t>(s) * R] - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  const float inv = den > 0.f ? 1.f / den : 0.f;

  const int64_t out_row = grp * R + r;
  for (int d = lane * 4; d < dv; d += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m != -INFINITY) {
      // partials in batches of 8: all loads of a batch are in flight together
      constexpr int kBatch = 8;
      for (int s0 = 0; s0 < n_in; s0 += kBatch) {
        float w[kBatch];
        float4 x[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int s = s0 + u;
          const float ls = (s < n_in) ? lse_base[static_cast<int64_t>(s) * R] : -INFINITY;
          w[u] = (ls == -INFINITY) ? 0.f : __expf(ls - m);
          x[u] = (w[u] != 0.f) ? *reinterpret_cast<const float4*>(o_base + static_cast<int64_t>(s) * R * dv + d)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          acc.x += w[u] * x[u].x;
          acc.y += w[u] * x[u].y;
          acc.z += w[u] * x[u].z;
          acc.w += w[u] * x[u].w;
        }
      }
    }
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    if constexpr (OUT_BF16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + out_row * dv + d) = u;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + out_row * dv + d) = acc;
    }
  }
  if (lane == 0) out_lse[out_row] = (den > 0.f) ? m + logf(den) : -INFINITY;
}

// Two-way merge in place: (acc_o, acc_lse) <- merge((acc_o, acc_lse), (in_o, in_lse)), the
// same formula as above for two fragments; one warp per row, 4 columns per lane per pass.
__global__ void __launch_bounds__(256) merge_into_kernel(float* __restrict__ acc_o, float* __restrict__ acc_lse,
                                                         const float* __restrict__ in_o,
                                                         const float* __restrict__ in_lse, int64_t R, int32_t dv) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= R) return;
  const float la = acc_lse[row], lb = in_lse[row];
  const float m = fmaxf(la, lb);
  if (m == -INFINITY) return;  // neither has seen a token: acc stays o = 0, lse = -inf
  const float wa = (la == -INFINITY) ? 0.f : __expf(la - m);
  const float wb = (lb == -INFINITY) ? 0.f : __expf(lb - m);
  const float inv = 1.f / (wa + wb);
  float* ao = acc_o + row * dv;
  const float* bo = in_o + row * dv;
  for (int d = lane * 4; d < dv; d += 128) {
    const float4 x = (wa != 0.f) ? *reinterpret_cast<const float4*>(ao + d) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 y = (wb != 0.f) ? *reinterpret_cast<const float4*>(bo + d) : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(ao + d) = make_float4((wa * x.x + wb * y.x) * inv, (wa * x.y + wb * y.y) * inv,
                                                     (wa * x.z + wb * y.z) * inv, (wa * x.w + wb * y.w) * inv);
  }
  __syncwarp();
  if (lane == 0) acc_lse[row] = m + logf(wa + wb);
}

}  // namespace

cudaError_t launch_merge_into(float* acc_o, float* acc_lse, const float* in_o, const float* in_lse, int64_t R,
                              int32_t dv, cudaStream_t stream) {
  if (R <= 0) return cudaSuccess;
  merge_into_kernel<<<static_cast<unsigned int>((R + 7) / 8), 256, 0, stream>>>(acc_o, acc_lse, in_o, in_lse, R, dv);
  return cudaGetLastError();
}

cudaError_t launch_merge(const float* in_o, const float* in_lse, int32_t n_in, int32_t g_out, int64_t R, int32_t dv,
                         void* out, bool out_bf16, float* out_lse, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(g_out) * R;
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;
  // programmatic dependent launch: the merge grid is set up while the partial kernel
  // before it on the stream drains; griddepcontrol.wait in the kernel keeps the order
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(blocks));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (out_bf16)
    return cudaLaunchKernelEx(&cfg, merge_kernel<true>, in_o, in_lse, n_in, g_out, R, dv, out, out_lse);
  return cudaLaunchKernelEx(&cfg, merge_kernel<false>, in_o, in_lse, n_in, g_out, R, dv, out, out_lse);
}

}  // namespace skv
