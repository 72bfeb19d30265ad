// Self-test of the tcgen05 building blocks used by the tensor-core attention kernels:
// one CTA computes C[128 x N] = A[128 x 64] * B with A K-major and B either K-major
// (C = A B^T, B stored [N][64]) or MN-major (C = A B, B stored [64][N]), operands
// loaded by TMA with 128-byte swizzle, the product accumulated in tensor memory and
// read back with tcgen05.ld.  Shapes are chosen so that every shared-memory address a
// descriptor can reach stays inside the CTA's allocation.
#include <cuda_runtime.h>

#include "skv_common.cuh"
#include "skv_internal.h"
#include "tc_common.cuh"

namespace skv {

namespace {

constexpr int kSelftestSmem = 1024 + 128 * 1024;  // generous: any descriptor reach stays inside

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(128, 1)
    umma_selftest_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, float* C,
                         int N, int b_mn_major, int a_tmem, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;               // A: one box, 128 rows x 128 B (16 KB)
  uint8_t* sb = smem + 16 * 1024;   // B: K-major N rows x 128 B, or MN-major N/64 boxes of 64 rows x 128 B
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(smem + 48 * 1024);
  uint64_t* bar_mma = bar_load + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(smem_u32(tmem_slot), 512);  // all columns: any N the MMA uses stays inside
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    const uint32_t b_bytes = static_cast<uint32_t>(N) * 128u;
    mbar_arrive_expect_tx(bar_load, 16384u + b_bytes);
    tma_load_2d(sa, &ta, bar_load, 0, 0);
    if (!b_mn_major) {
      tma_load_2d(sb, &tb, bar_load, 0, 0);
    } else {
      for (int nb = 0; nb < N / 64; ++nb) tma_load_2d(sb + nb * 8192, &tb, bar_load, nb * 64, 0);
    }
  }
  // every thread sees the loaded tiles
  const bool loaded = mbar_wait(bar_load, 0, err, kDevErrFullWait);
  const int row = warp * 32 + lane;
  const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  constexpr uint32_t kColA = 256;  // A copy in TMEM (32 columns: 64 bf16 per row)
  if (a_tmem) {
    // A row -> TMEM lane `row`: column c holds elements (2c, 2c+1) of the row
    uint32_t w[2][16];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(sa + swz128(row, c * 16));
      w[c >> 2][(c & 3) * 4 + 0] = v.x;
      w[c >> 2][(c & 3) * 4 + 1] = v.y;
      w[c >> 2][(c & 3) * 4 + 2] = v.z;
      w[c >> 2][(c & 3) * 4 + 3] = v.w;
    }
    tc::tmem_st16(taddr + kColA, w[0]);
    tc::tmem_st16(taddr + kColA + 16, w[1]);
    tc::tmem_wait_st();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (threadIdx.x == 0 && loaded) {
    const uint32_t idesc = tc::idesc_f16(128, N, true, false, b_mn_major != 0);
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t bd = b_mn_major ? tc::smem_desc_sw128(smem_u32(sb) + ks * 2048, 8192, 1024)
                                     : tc::smem_desc_sw128(smem_u32(sb) + ks * 32, 16, 1024);
      if (a_tmem) {
        tc::mma_f16_ts(tmem, tmem + kColA + ks * 8, bd, idesc, ks > 0 ? 1u : 0u);
      } else {
        const uint64_t ad = tc::smem_desc_sw128(smem_u32(sa) + ks * 32, 16, 1024);
        tc::mma_f16_ss(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
      }
    }
    tc::mma_commit(smem_u32(bar_mma));
  }
  __syncwarp();
  mbar_wait(bar_mma, 0, err, kDevErrFullWait);
  tc::fence_after_sync();
  for (int c = 0; c < N / 16; ++c) {
    uint32_t r[16];
    tc::tmem_ld16(taddr + c * 16, r);
    tc::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) C[row * N + c * 16 + e] = __uint_as_float(r[e]);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_umma_selftest(const CUtensorMap& ta, const CUtensorMap& tb, float* C, int N, bool b_mn_major,
                                 bool a_tmem, unsigned int* err, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSelftestSmem);
  if (e != cudaSuccess) return e;
  umma_selftest_kernel<<<1, 128, kSelftestSmem, stream>>>(ta, tb, C, N, b_mn_major ? 1 : 0, a_tmem ? 1 : 0,
                                                           err);
  return cudaGetLastError();
}

}  // namespace skv
