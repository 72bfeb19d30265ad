// Device-side building blocks shared by the split-KV attention kernels (sm_103a).
//
// Inline PTX for: mbarrier waits with a time limit, TMA tiled bulk-tensor loads,
// ldmatrix / movmatrix fragment loads, and mma.sync tensor-core tiles.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace skv {

// Device error word (one per library, owned by api.cu).  Kernels OR a code into it
// when a bounded wait gives up; the host reads and clears it.
enum DevError : unsigned int {
  kDevErrFullWait = 1u,   // a consumer gave up waiting for a TMA tile
  kDevErrEmptyWait = 2u,  // the producer gave up waiting for a free stage
  kDevErrDrainWait = 4u,  // the final drain of in-flight copies gave up
};

// Time limit of every spin-wait in the library's kernels, in SM clock cycles (the
// per-SM cycle counter is monotonic; about 2 s at 2 GHz).
constexpr long long kWaitLimitCycles = 4000000000ll;

// Layout of the device error record (unsigned int words): [0] OR of error codes,
// [1] set once the first failure is described, [2] blockIdx.x, [3] threadIdx.x,
// [4] shared-memory address of the barrier, [5] parity | code << 8 | kernel id << 16.
enum DevErrWord : int { kErrCode = 0, kErrTaken = 1, kErrBlock = 2, kErrThread = 3, kErrBar = 4, kErrWhat = 5 };
constexpr int kDevErrWords = 8;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Record a wait that gave up: OR the code into err[0]; the first failure also records
// where it happened (block, thread, barrier address, parity / code).
__device__ __forceinline__ void record_wait_failure(unsigned int* err, unsigned int code, uint32_t bar_addr,
                                                    uint32_t parity) {
  atomicOr(err + kErrCode, code);
  if (atomicCAS(err + kErrTaken, 0u, 1u) == 0u) {
    err[kErrBlock] = blockIdx.x;
    err[kErrThread] = threadIdx.x;
    err[kErrBar] = bar_addr;
    err[kErrWhat] = parity | (code << 8);
  }
}

// Wait for the phase with the given parity to complete.  Returns false (and records the
// failure in err) if it has not completed within kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* err,
                                          unsigned int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long c0 = clock64();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 255u) == 0u && clock64() - c0 > kWaitLimitCycles) {
      record_wait_failure(err, code, smem_u32(bar), parity);
      return false;
    }
  }
}

// ----------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled load (coordinates innermost first) completing on `bar` with a byte count.
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (TMA) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- fragments

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// Four e4m3 codes (bytes b0..b3 of w) -> two fp16 pairs: lo = (b0, b1), hi = (b2, b3).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Byte permute: result byte i = byte sel_i of {b, a} (a = bytes 0..3).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Same with fp16 inputs.
__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The two bf16 values of a packed pair (pack_bf16), widened back to float exactly.  A
// softmax whose P goes through bf16 normalises O by the sum of these (the output is then an
// exact convex combination of V rows with the rounded weights) and keeps the fp32 sum of p
// for its lse.  With an optimistic running max (p up to 2^8, none exact) normalising by the
// fp32 sum instead leaves the rounding errors in the output: up to ~2^-8 max|v| for a split
// of a few tokens, about twice the error of the consistent normalisation.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The same sums of a packed pair's two rounded values without unpacking it: the
// mixed-precision adds (fp32 accumulator + bf16 operand, widened exactly, one IEEE round-
// to-nearest add each) take the pair's halves directly, so the result equals
// add_f32x2(acc, bf16_lo(w), bf16_hi(w)) bit for bit, with no integer shift / mask on the
// ALU pipe that the softmax loops saturate.
__device__ __forceinline__ uint64_t add_bf16x2_f32x2(uint64_t acc, uint32_t w) {
  uint64_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t.reg .f32 x, y;\n\t"
      "mov.b32 {lo, hi}, %2;\n\tmov.b64 {x, y}, %1;\n\t"
      "add.rn.f32.bf16 x, lo, x;\n\tadd.rn.f32.bf16 y, hi, y;\n\t"
      "mov.b64 %0, {x, y};\n\t}"
      : "=l"(r)
      : "l"(acc), "r"(w));
  return r;
}

// Two running fp32 sums in one 64-bit register, advanced by one packed add (two IEEE
// round-to-nearest adds in one instruction): the softmax row sums take one instruction per
// pair of columns.
__device__ __forceinline__ uint64_t add_f32x2(uint64_t acc, float x, float y) {
  uint64_t v, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(x), "f"(y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(acc), "l"(v));
  return r;
}
// max(a, b, c) in one instruction (NaN operands ignored, as fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}
// (x0, x1) * s + c for a pair in one packed instruction (two round-to-nearest FMAs).
__device__ __forceinline__ void fma_pair(float x0, float x1, float s, float c, float& r0, float& r1) {
  uint64_t x, sv, cv, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(sv) : "f"(s));
  asm("mov.b64 %0, {%1, %1};" : "=l"(cv) : "f"(c));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(x), "l"(sv), "l"(cv));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(r));
}
__device__ __forceinline__ float sum_f32x2(uint64_t acc) {
  float x, y;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(acc));
  return x + y;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two e4m3 codes (low byte first) -> two fp16 values (exact: every e4m3 value is an fp16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// 2^x with the SFU's approximate exponential (ex2.approx.ftz: relative error about
// 2^-22; 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of (row, byte) inside a TMA tile written with 128-byte swizzle: rows of
// 128 bytes, 16-byte chunk c of row r stored at chunk c ^ (r & 7).
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t byte_in_row) {
  return row * 128u + ((((byte_in_row >> 4) ^ (row & 7u)) << 4) | (byte_in_row & 15u));
}

}  // namespace skv
