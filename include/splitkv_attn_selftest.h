/*
 * splitkv_attn_selftest.h -- hardware self-test of libsplitkv_attn.so (NVIDIA GB300, sm_103a).
 *
 * Not part of the attention method: the pages describe no such call.  It checks, on the
 * GPU at hand, the 5th-generation tensor-core path (tcgen05) that the tensor-core
 * attention kernels are built from: TMA tiles with 128-byte swizzle, shared-memory matrix
 * descriptors for K-major and MN-major operands, the kind::f16 instruction descriptor,
 * MMA into tensor memory (TMEM), commit to an mbarrier, and TMEM loads.
 */
#ifndef SPLITKV_ATTN_SELFTEST_H
#define SPLITKV_ATTN_SELFTEST_H

#include <stdint.h>

#include "splitkv_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * splitkv_selftest_umma_gemm -- C[128][N] = A[128][64] * op(B) in fp32 on one CTA.
 *   A  bf16 [128][64] row-major (device, 16-byte aligned)
 *   B  bf16; (flags & 1) == 0: [N][64] row-major and op(B) = B^T (both operands K-major);
 *            (flags & 1) != 0: [64][N] row-major and op(B) = B (B is MN-major)
 *   C  fp32 [128][N] row-major (device)
 *   N  64 or 128
 *   flags  bit 0: B MN-major; bit 1: the MMA reads A from tensor memory (copied there from
 *          the shared-memory tile) instead of from shared memory
 * Asynchronous on `stream`; returns SKV_EINVAL for bad arguments, SKV_ECUDA on launch errors.
 */
skv_status splitkv_selftest_umma_gemm(const void* A, const void* B, float* C, int32_t N, int32_t flags,
                                      void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPLITKV_ATTN_SELFTEST_H */
