// Split-KV partial attention for the MLA latent cache (multi-head latent attention,
// absorbed decode): every query head attends over one shared latent row per token.
//
// What it computes: the same partial (normalised o, natural-log lse) per split as the
// GQA kernel -- "Helix Parallelism: Why Tensor Parallelism Hits a Wall at
// Million-Token Context" (section "Sharding the sequence instead") -- for a cache
// with a single KV "head" (the latent): the key of token t is the whole latent row
// (512 latent + 64 rope dims = 576) and its value is the first 512 latent dims.  The
// Helix page names this case ("multi-head latent attention ... keeps a single latent
// representation shared across all query heads", section "The ceiling, in algebra").
//
// GB300 design: a CTA serves 64 query heads of one sequence (a work item of the
// split/chunk decomposition); one producer warp streams 32-token latent tiles (nine
// 128-byte TMA boxes per row, 128-byte swizzle) into a 3-stage ring; the K tile is
// also the V tile (V = its first 512 columns), so every latent byte is loaded once
// per CTA.  Sixteen consumer warps = 4 head groups (16 heads, the mma M) x 4
// quarters of the 512 value dims: each warp scores 8 of the tile's 32 tokens for its
// head group over all 576 dims (mma.sync), the head group's 4 warps exchange scores
// through shared memory, and each warp then runs the same online softmax and
// accumulates its 16 x 128 slice of O.
#include <cuda_runtime.h>

#include "skv_common.cuh"
#include "skv_internal.h"

namespace skv {

namespace {

constexpr int kDk = 576;
constexpr int kDv = 512;
constexpr int kTN = 32;  // tokens per tile
constexpr int kNStage = 3;
constexpr int kHG = 4;  // head groups of 16 per CTA
constexpr int kDQ = 4;  // value-dim quarters
constexpr int kNCW = kHG * kDQ;
constexpr int kThreads = (kNCW + 1) * 32;
constexpr int kRows = 16 * kHG;  // 64 query heads per CTA
constexpr int kNBox = kDk * 2 / 128;  // 9 boxes of 64 bf16
constexpr int kBoxBytes = kTN * 128;
constexpr int kTileBytes = kNBox * kBoxBytes;
constexpr int kRingBytes = kNStage * kTileBytes;
constexpr int kQStride = kDk + 8;  // padded row (1168 bytes): conflict-free ldmatrix
constexpr int kQBytes = kRows * kQStride * 2;
constexpr int kSBytes = 2 * kRows * kTN * 4;  // double-buffered scores
constexpr int kSmem = 1024 + kRingBytes + kQBytes + kSBytes + 2 * kNStage * 8;
static_assert(kDk % 64 == 0, "latent rows are whole 128-byte boxes");
static_assert(kSmem <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t lat_off(uint32_t tok, uint32_t byte) {
  return (byte >> 7) * kBoxBytes + swz128(tok, byte & 127u);
}

__device__ __forceinline__ uint32_t half_mask(bool lo, bool hi) {
  return (lo ? 0x0000FFFFu : 0u) | (hi ? 0xFFFF0000u : 0u);
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_partial_kernel(const __grid_constant__ PartialParams p, const __grid_constant__ CUtensorMap tmk) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem + kRingBytes);
  float* sbuf = reinterpret_cast<float*>(smem + kRingBytes + kQBytes);  // [2][kRows][kTN]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRingBytes + kQBytes + kSBytes);
  uint64_t* empty = full + kNStage;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item (same decomposition as the GQA kernel; Hkv = 1, G = Hq)
  int64_t item = blockIdx.x;
  const int mt = static_cast<int>(item % p.m_tiles);
  item /= p.m_tiles;
  const int c = static_cast<int>(item % p.n_chunk);
  item /= p.n_chunk;
  const int j = static_cast<int>(item % p.n_split);
  item /= p.n_split;
  const int b = static_cast<int>(item / p.Hkv);

  const int seq_len = p.seq_lens[b];
  int lo, hi, win_lo, win_hi;
  split_range(p, b, j, j + 1, seq_len, &lo, &hi);
  chunk_window(p, lo, hi, c, &win_lo, &win_hi);
  const int r_lo = max(lo, win_lo);
  int r_hi = min(hi, win_hi);
  const int rows_total = p.Tq * p.G;
  const int m0 = mt * kRows;
  const int m_last = min(m0 + kRows, rows_total) - 1;
  {
    const int64_t horizon = p.causal_offset + m_last / p.G;
    if (horizon < static_cast<int64_t>(r_hi) - 1) r_hi = static_cast<int>(max(horizon + 1, (int64_t)r_lo));
  }
  const int tile_begin = r_lo / kTN;
  const int n_tiles = (r_hi > r_lo) ? ((r_hi + kTN - 1) / kTN - tile_begin) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNStage; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kNCW);
    }
    fence_mbar_init();
  }
  // ---- stage Q rows of this CTA (64 heads x 576) into padded shared rows
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    for (int e = threadIdx.x * 8; e < kRows * kDk; e += kThreads * 8) {
      const int r = e / kDk, d = e % kDk;
      const int m = m0 + r;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < rows_total) {
        const int t_q = m / p.G, h = m % p.G;  // Hkv = 1
        v = *reinterpret_cast<const uint4*>(q + b * p.q_sb + t_q * p.q_st + h * p.q_sh + d);
      }
      *reinterpret_cast<uint4*>(qs + r * kQStride + d) = v;
    }
  }
  __syncthreads();

  if (warp == kNCW) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tmk);
      const uint64_t pol = l2_policy_evict_first();
      const bool paged = p.block_table != nullptr;
      int page_next = paged ? kv_page_of(p, b, tile_begin * kTN) : b;  // read one tile ahead
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kNStage;
        if (i >= kNStage && !mbar_wait(&empty[s], ((i / kNStage) - 1) & 1, p.err, kDevErrEmptyWait)) break;
        mbar_arrive_expect_tx(&full[s], kTileBytes);
        uint8_t* ks = smem + s * kTileBytes;
        const int tok = (tile_begin + i) * kTN;
        const int outer = page_next;
        const int row = paged ? tok % p.block_len : tok;
        if (paged && i + 1 < n_tiles) page_next = kv_page_of(p, b, tok + kTN);
#pragma unroll
        for (int bx = 0; bx < kNBox; ++bx) tma_load_4d(ks + bx * kBoxBytes, &tmk, &full[s], bx * 64, row, 0, outer, pol);
        issued = i + 1;
      }
      for (int i = max(0, issued - kNStage); i < issued; ++i) {
        if (!mbar_wait(&full[i % kNStage], (i / kNStage) & 1, p.err, kDevErrDrainWait)) break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumer warps
  const int hg = warp / kDQ, dq = warp % kDQ;
  const int gq = lane >> 2, tq = lane & 3;
  const int mi = lane >> 3;
  const int lr0 = hg * 16 + gq, lr1 = lr0 + 8;  // local rows (heads) of this thread
  const int mrow0 = m0 + lr0, mrow1 = m0 + lr1;
  const bool v0 = mrow0 < rows_total, v1 = mrow1 < rows_total;
  const int tq0 = v0 ? mrow0 / p.G : 0, tq1 = v1 ? mrow1 / p.G : 0;
  const int64_t hz0 = p.causal_offset + tq0, hz1 = p.causal_offset + tq1;
  const int64_t hz_min = p.causal_offset + (m0 + hg * 16) / p.G;
  const uint32_t qbase = smem_u32(qs);

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrun[2] = {-INFINITY, -INFINITY};
  float lrun[2] = {0.f, 0.f};

  for (int i = 0; i < n_tiles; ++i) {
    const int s = i % kNStage;
    const int t0 = (tile_begin + i) * kTN;
    if (!mbar_wait(&full[s], (i / kNStage) & 1, p.err, kDevErrFullWait)) break;
    const uint32_t kb = smem_u32(smem + s * kTileBytes);
    float* sb = sbuf + (i & 1) * kRows * kTN;

    // ---- scores of 8 tokens (dq*8 ..) for the head group's 16 heads, over all 576 dims
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t ktok = dq * 8 + (lane & 7);
#pragma unroll 4
    for (int ks = 0; ks < kDk / 16; ks += 2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kb + lat_off(ktok, (2 * ks + mi) * 16), b0, b1, b2, b3);
      uint32_t a[4], a2[4];
      ldsm_x4(qbase + ((hg * 16 + (mi & 1) * 8 + (lane & 7)) * kQStride + (2 * ks + (mi >> 1)) * 8) * 2, a[0], a[1],
              a[2], a[3]);
      ldsm_x4(qbase + ((hg * 16 + (mi & 1) * 8 + (lane & 7)) * kQStride + (2 * ks + 2 + (mi >> 1)) * 8) * 2, a2[0],
              a2[1], a2[2], a2[3]);
      mma_bf16(sc, a, b0, b1);
      mma_bf16(sc, a2, b2, b3);
    }
    *reinterpret_cast<float2*>(sb + lr0 * kTN + dq * 8 + 2 * tq) = make_float2(sc[0], sc[1]);
    *reinterpret_cast<float2*>(sb + lr1 * kTN + dq * 8 + 2 * tq) = make_float2(sc[2], sc[3]);
    named_bar_sync(1 + hg, kDQ * 32);

    // ---- online softmax over the tile's 32 tokens (identical in the 4 warps of the group)
    const bool in_range = (t0 >= r_lo) && (t0 + kTN <= r_hi);
    const bool need_mask = !in_range || (static_cast<int64_t>(t0) + kTN - 1 > hz_min);
    float x[2][2][4];  // [row][kk][4 values: tokens 16kk+2tq, +1, 16kk+8+2tq, +1]
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float* srow = sb + (r ? lr1 : lr0) * kTN;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const float2 u = *reinterpret_cast<const float2*>(srow + 16 * kk + 2 * tq);
        const float2 w = *reinterpret_cast<const float2*>(srow + 16 * kk + 8 + 2 * tq);
        float vals[4] = {u.x, u.y, w.x, w.y};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float y = vals[e] * p.scale_log2;
          if (need_mask) {
            const int tok = t0 + 16 * kk + (e >> 1) * 8 + 2 * tq + (e & 1);
            const bool ok = tok >= r_lo && tok < r_hi && static_cast<int64_t>(tok) <= (r ? hz1 : hz0);
            y = ok ? y : -INFINITY;
          }
          x[r][kk][e] = y;
          tmax[r] = fmaxf(tmax[r], y);
        }
      }
    }
    float base[2], alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
      const float mnew = fmaxf(mrun[r], tmax[r]);
      base[r] = (mnew == -INFINITY) ? 0.f : mnew;
      alpha[r] = fast_exp2(mrun[r] - base[r]);
      mrun[r] = mnew;
      lrun[r] *= alpha[r];
    }
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {  // a row max moved
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
    }
    uint32_t pa[2][4];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      float pr[2][4];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pr[r][e] = fast_exp2(x[r][kk][e] - base[r]);
          lrun[r] += pr[r][e];
        }
      }
      pa[kk][0] = pack_bf16(pr[0][0], pr[0][1]);
      pa[kk][1] = pack_bf16(pr[1][0], pr[1][1]);
      pa[kk][2] = pack_bf16(pr[0][2], pr[0][3]);
      pa[kk][3] = pack_bf16(pr[1][2], pr[1][3]);
    }

    // ---- O[16 x 128 (quarter dq)] += P[16 x 32] V[32 x 128]; V = latent dims 0..511
    const bool vmask = !in_range;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
      if (vmask) {
        const int ta = t0 + 16 * kk + 2 * tq, tb = ta + 8;
        mlo = half_mask(ta >= r_lo && ta < r_hi, ta + 1 >= r_lo && ta + 1 < r_hi);
        mhi = half_mask(tb >= r_lo && tb < r_hi, tb + 1 >= r_lo && tb + 1 < r_hi);
      }
      const uint32_t vtok = 16 * kk + (mi & 1) * 8 + (lane & 7);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const uint32_t chunk = dq * 16 + 2 * dp + (mi >> 1);
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(kb + lat_off(vtok, chunk * 16), r0, r1, r2, r3);
        mma_bf16(o[2 * dp], pa[kk], r0 & mlo, r1 & mhi);
        mma_bf16(o[2 * dp + 1], pa[kk], r2 & mlo, r3 & mhi);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- finish: every warp writes its 16 x 128 slice; the dq == 0 warp writes lse
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], 1);
    lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], 2);
  }
  constexpr float kLn2 = 0.6931471805599453f;
  const int part = j * p.n_chunk + c;
  const int h0 = v0 ? mrow0 % p.G : 0, h1 = v1 ? mrow1 % p.G : 0;
  const int64_t ro0 = ((static_cast<int64_t>(part) * p.B + b) * p.Tq + tq0) * p.Hq + h0;
  const int64_t ro1 = ((static_cast<int64_t>(part) * p.B + b) * p.Tq + tq1) * p.Hq + h1;
  const float inv0 = lrun[0] > 0.f ? 1.f / lrun[0] : 0.f;
  const float inv1 = lrun[1] > 0.f ? 1.f / lrun[1] : 0.f;
  const bool w0 = v0 && (lrun[0] > 0.f || p.zero_empty);
  const bool w1 = v1 && (lrun[1] > 0.f || p.zero_empty);
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int d = dq * 128 + 8 * n + 2 * tq;
    if (w0) *reinterpret_cast<float2*>(p.out_o + ro0 * kDv + d) = make_float2(o[n][0] * inv0, o[n][1] * inv0);
    if (w1) *reinterpret_cast<float2*>(p.out_o + ro1 * kDv + d) = make_float2(o[n][2] * inv1, o[n][3] * inv1);
  }
  if (dq == 0 && tq == 0) {
    if (v0) p.out_lse[ro0] = lrun[0] > 0.f ? (mrun[0] + __log2f(lrun[0])) * kLn2 : -INFINITY;
    if (v1) p.out_lse[ro1] = lrun[1] > 0.f ? (mrun[1] + __log2f(lrun[1])) * kLn2 : -INFINITY;
  }
}

}  // namespace

GqaLaunchInfo mla_launch_info() { return GqaLaunchInfo{kRows, kThreads, kSmem, 1}; }

cudaError_t launch_mla_partial(const PartialParams& p, const CUtensorMap& tmk, int64_t n_items, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e0 = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(mla_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (e0 != cudaSuccess) return e0;
  if (n_items <= 0) return cudaSuccess;
  mla_partial_kernel<<<static_cast<unsigned int>(n_items), kThreads, kSmem, stream>>>(p, tmk);
  return cudaGetLastError();
}

}  // namespace skv
