// Split-KV partial attention for grouped-query attention (GQA), bf16 or fp8-e4m3 KV.
//
// What it computes (per work item = sequence b, KV head g, split j, chunk c, row tile):
// for every query row t and query head h of KV head g's group, the softmax attention
// of q[b,t,h] over the visible tokens of the item's token range, returned as the
// normalised partial output o and its natural-log log-sum-exp -- the "partial
// attention output plus a log-sum-exp" each KVP rank emits in "Helix Parallelism:
// Why Tensor Parallelism Hits a Wall at Million-Token Context" (section "Sharding
// the sequence instead"), and each ring step emits in "Context Parallelism for
// Scalable Million-Token Inference" (section "Pass-KV keeps queries local and
// circulates keys and values").  Query heads map to KV heads in contiguous groups
// (head h reads KV head h / G).  A token t is visible to query row i when it lies in
// the range, t < seq_len[b] and t <= causal_offset + i.
//
// Pass-Q decode ("Context Parallelism for Scalable Million-Token Inference", sections
// "Pass-Q keeps KV stationary for cache-heavy turns" and "Pass-Q decode protects capacity
// but can hurt TTIT") runs through the same kernel: with ring_n ranks, each holding its
// own resident shard of every request, one launch covers every rank's every ring step; a
// work item decodes which query block has arrived at which rank and writes its partial
// straight into the exchange slot of the query's owner, so the exchange and the merge
// that follow are one merge launch.
//
// GB300 design:
//   * one producer warp streams K and V tiles (64 tokens) with TMA tiled bulk-tensor
//     copies into a multi-stage shared-memory ring (128-byte swizzle, conflict-free
//     ldmatrix), completion tracked by mbarriers; tiles are read-once, so the loads
//     carry an L2 evict-first policy;
//   * every consumer warp owns 16 rows of the item (for decode: the 16 query heads
//     of one KV head), so each K/V byte crosses HBM once per KV head and serves the
//     whole group;
//   * QK^T and PV run on mma.sync m16n8k16 tensor-core tiles with fp32 accumulation;
//     the online softmax (running max / sum, rescale) is kept in registers with
//     quad shuffles; exponentials are base-2 with log2(e) folded into the scale;
//   * decode variants spread the item's tiles over 4 (bf16 d=128: 3) consumer warps
//     and combine their (m, l, O) in shared memory at the end; prefill variants give
//     each of 4 warps its own 16 rows and share every tile.
//   * fp8: K/V codes are widened to fp16 in registers (exact), q is used in fp16,
//     the K block scale multiplies the score and the V block scale multiplies p.
#include <cuda_runtime.h>

#include <type_traits>

#include "skv_common.cuh"
#include "skv_internal.h"

namespace skv {

namespace {

template <bool FP8_, int D_, int WM_, int WN_, int NSTAGE_, int MINB_, int SUB_ = kTileN>
struct GqaCfg {
  static constexpr int SUB = SUB_;  // tokens per online-softmax step (a tile is TN / SUB steps)
  static constexpr bool FP8 = FP8_;
  static constexpr int D = D_;  // dk = dv
  static constexpr int WM = WM_;
  static constexpr int WN = WN_;
  static constexpr int NSTAGE = NSTAGE_;
  static constexpr int MINB = MINB_;
  static constexpr int TN = kTileN;
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int ROW_BYTES = D * ESZ;
  static constexpr int NBOX = ROW_BYTES / 128;  // 128-byte TMA boxes per token row
  static constexpr int BOX_ELEMS = 128 / ESZ;
  static constexpr int BOX_BYTES = TN * 128;
  static constexpr int TILE_BYTES = TN * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int NCW = WM * WN;
  static constexpr int THREADS = (NCW + 1) * 32;
  static constexpr int ROWS = 16 * WM;
  static constexpr int RING_BYTES = NSTAGE * STAGE_BYTES;
  // Full barriers are per consumer warp column, DW of them each (see full_slot).
  static constexpr int DW = (NSTAGE + WN - 1) / WN;
  static constexpr int NFULL = WN * DW;
  static constexpr int BAR_BYTES = ((NFULL + NSTAGE) * 8 + 15) / 16 * 16;
  static constexpr int ML_BYTES = WN * ROWS * 2 * 4;
  // fp8 variants keep their fp16 q fragments in shared memory ([WM][D/16][32 lanes] x 16 B)
  static constexpr int QF_BYTES = FP8 ? WM * (D / 16) * 32 * 16 : 0;
  // ... and the score scale of each warp row (the softmax scale times their q scaling)
  static constexpr int QS_BYTES = FP8 ? 16 : 0;
  static constexpr int SMEM = 1024 + RING_BYTES + BAR_BYTES + ML_BYTES + QF_BYTES + QS_BYTES;
  static_assert(ROW_BYTES % 128 == 0, "token rows must be whole 128-byte boxes");
  static_assert(WN == 1 || WN * ROWS * D * 4 <= RING_BYTES, "combine buffer must fit in the ring");
  static_assert(D % 16 == 0, "head dim must be a multiple of 16");
  static_assert(NFULL >= NSTAGE, "a full barrier is re-armed only after its previous tile was consumed");
  static_assert(kTileN % SUB_ == 0 && SUB_ % 16 == 0, "softmax step must divide the tile");
};

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Byte offset of (token row, byte in the row) in a K or V tile of the ring.
template <class C>
__device__ __forceinline__ uint32_t tile_off(uint32_t tok, uint32_t byte) {
  return (byte >> 7) * C::BOX_BYTES + swz128(tok, byte & 127u);
}

// Tile i lands in data stage i % NSTAGE but signals its own full barrier: consumer warp
// column wn = i % WN owns barriers [wn*DW, wn*DW + DW) and uses them in turn.  A parity
// wait is exact only when the barrier is at most one phase away from the awaited one.
// With one barrier per stage that fails once WN does not divide NSTAGE: the stage's
// previous tile belongs to another warp and its copy can land after this warp's own
// previous tile, so the wait would match that older phase and return early.  With
// per-column barriers the previous phase of tile i's barrier is tile i - WN*DW of the
// same warp (already observed), and the next phase (tile i + WN*DW) cannot start
// early: the producer issues tiles in order and waits, before issuing tile x, until
// tile x - NSTAGE was consumed, so by the time it reaches tile i + WN*DW >= i + NSTAGE
// tile i has been consumed.
template <class C>
__device__ __forceinline__ int full_slot(int i) {
  return (i % C::WN) * C::DW + (i / C::WN) % C::DW;
}
template <class C>
__device__ __forceinline__ uint32_t full_parity(int i) {
  return static_cast<uint32_t>((i / C::WN) / C::DW) & 1u;
}

__device__ __forceinline__ uint32_t half_mask(bool lo, bool hi) {
  return (lo ? 0x0000FFFFu : 0u) | (hi ? 0xFFFF0000u : 0u);
}

// Pass-Q ring (RING instantiation, ring_n > 0): work row b = (k * ring_n + s) * ring_bq + jj is rank k at ring
// step s, holding the query block that started on rank src = (k - s) mod ring_n; its slot
// jj carries request src * ring_bq + jj (the batch id that travels with the query), whose
// shard on rank k is cache row k * (ring_n * ring_bq) + request.
__device__ __forceinline__ void ring_rows(const PartialParams& p, int b, int* bq, int* bkv) {
  const int jj = b % p.ring_bq;
  const int ks = b / p.ring_bq;
  const int s = ks % p.ring_n, k = ks / p.ring_n;
  const int src = (k - s + p.ring_n) % p.ring_n;
  *bq = src * p.ring_bq + jj;
  *bkv = k * (p.ring_n * p.ring_bq) + *bq;
}

// Output slot of a pass-Q ring's work item: the exchange slot [owner src][from rank k]
// [part][jj] of the query's owner (the permutation before the All-to-All, done at the
// store); recomputed from the block index so that it holds no register through the loop.
__device__ __forceinline__ int64_t ring_out_slot(const PartialParams& p) {
  int64_t item = blockIdx.x / p.m_tiles;
  const int c = static_cast<int>(item % p.n_chunk);
  item /= p.n_chunk;
  const int j = static_cast<int>(item % p.n_split);
  item /= p.n_split;
  const int b = static_cast<int>(item / p.Hkv);
  const int part = j * p.n_chunk + c;
  const int jj = b % p.ring_bq;
  const int ks = b / p.ring_bq;
  const int s = ks % p.ring_n, k = ks / p.ring_n;
  const int src = (k - s + p.ring_n) % p.ring_n;
  return ((static_cast<int64_t>(src) * p.ring_n + k) * (p.n_split * p.n_chunk) + part) * p.ring_bq + jj;
}

// PAGED: K/V live in pages with a block table; POS: the causal rule comes from position
// arrays; RING: a pass-Q ring's work rows (never with PAGED or POS).  Separate
// instantiations, so the plain kernels carry none of that code (a runtime test of the
// first two cost the fp8 decode 4 %, of the third 1.3 %).
template <class C, bool PAGED, bool POS, bool RING>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
    gqa_partial_kernel(const __grid_constant__ PartialParams p, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv) {
  constexpr int D = C::D, TN = C::TN, NSTAGE = C::NSTAGE, WN = C::WN, WM = C::WM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES);  // [NFULL]
  uint64_t* empty = full + C::NFULL;                                     // [NSTAGE]
  float* ml = reinterpret_cast<float*>(smem + C::RING_BYTES + C::BAR_BYTES);  // [WN][ROWS][2]
  uint4* qfrag = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(ml) + C::ML_BYTES);  // fp8 only
  float* qscale = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(qfrag) + C::QF_BYTES);  // fp8: [WM]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item
  int64_t item = blockIdx.x;
  const int mt = static_cast<int>(item % p.m_tiles);
  item /= p.m_tiles;
  const int c = static_cast<int>(item % p.n_chunk);
  item /= p.n_chunk;
  const int j = static_cast<int>(item % p.n_split);
  item /= p.n_split;
  const int g = static_cast<int>(item % p.Hkv);
  const int b = static_cast<int>(item / p.Hkv);

  // bq: query row; bkv: KV row (sequence) of the cache
  int bq = b, bkv = b;
  if constexpr (RING) ring_rows(p, b, &bq, &bkv);

  const int seq_len = p.seq_lens[bkv];
  int lo, hi, win_lo, win_hi;
  split_range(p, bkv, j, j + 1, seq_len, &lo, &hi);
  chunk_window(p, lo, hi, c, &win_lo, &win_hi);
  static_assert(TN == kTileN, "chunks are cut in whole tiles");
  int r_lo = max(lo, win_lo);
  int r_hi = min(hi, win_hi);
  const int rows_total = p.Tq * p.G;
  const int m0 = mt * C::ROWS;
  const int m_last = min(m0 + C::ROWS, rows_total) - 1;
  {
    // no row of this tile sees a token past causal_offset + (its query row)
    const int64_t horizon = p.causal_offset + m_last / p.G;
    if (horizon < static_cast<int64_t>(r_hi) - 1) r_hi = static_cast<int>(max(horizon + 1, (int64_t)r_lo));
  }
  const int tile_begin = r_lo / TN;
  const int n_tiles = (r_hi > r_lo) ? ((r_hi + TN - 1) / TN - tile_begin) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NFULL; ++s) mbar_init(&full[s], 1);
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&empty[s], WM);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      const uint64_t pol = l2_policy_evict_first();
      // paged cache: the next tile's page is read one tile ahead, behind the stage wait
      int page_next = bkv;
      if constexpr (PAGED) page_next = kv_page_of(p, bkv, tile_begin * TN);
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % NSTAGE;
        if (i >= NSTAGE && !mbar_wait(&empty[s], ((i / NSTAGE) - 1) & 1, p.err, kDevErrEmptyWait)) break;
        uint64_t* fb = &full[full_slot<C>(i)];
        mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
        uint8_t* ks = smem + s * C::STAGE_BYTES;
        uint8_t* vs = ks + C::TILE_BYTES;
        const int tok = (tile_begin + i) * TN;
        const int outer = page_next;  // page (paged) or sequence
        int row = tok;
        if constexpr (PAGED) {
          row = tok % p.block_len;
          if (i + 1 < n_tiles) page_next = kv_page_of(p, bkv, tok + TN);
        }
#pragma unroll
        for (int bx = 0; bx < C::NBOX; ++bx) {
          tma_load_4d(ks + bx * C::BOX_BYTES, &tmk, fb, bx * C::BOX_ELEMS, row, g, outer, pol);
          tma_load_4d(vs + bx * C::BOX_BYTES, &tmv, fb, bx * C::BOX_ELEMS, row, g, outer, pol);
        }
        issued = i + 1;
      }
      // drain: every issued copy must have landed before this CTA may exit (tiles before
      // issued - NSTAGE were consumed before their stage was refilled)
      for (int i = max(0, issued - NSTAGE); i < issued; ++i) {
        if (!mbar_wait(&full[full_slot<C>(i)], full_parity<C>(i), p.err, kDevErrDrainWait)) break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumer warps
  const int wm = warp % WM, wn = warp / WM;
  const int gq = lane >> 2, tq = lane & 3;
  const int mrow0 = m0 + wm * 16 + gq, mrow1 = mrow0 + 8;
  const bool v0 = mrow0 < rows_total, v1 = mrow1 < rows_total;
  const int tq0 = v0 ? mrow0 / p.G : 0, tq1 = v1 ? mrow1 / p.G : 0;
  const int h0 = g * p.G + (v0 ? mrow0 % p.G : 0), h1 = g * p.G + (v1 ? mrow1 % p.G : 0);
  const int64_t hz0 = p.causal_offset + tq0, hz1 = p.causal_offset + tq1;
  const int64_t hz_min = p.causal_offset + (m0 + wm * 16) / p.G;
  // tokens stored out of sequence order: visible iff k_pos[t] <= q_pos[row]
  const int32_t* kpos_b = POS ? p.k_pos + static_cast<int64_t>(bkv) * p.S_max : nullptr;
  const int qp0 = POS ? __ldg(p.q_pos + bq * p.Tq + tq0) : 0;
  const int qp1 = POS ? __ldg(p.q_pos + bq * p.Tq + tq1) : 0;

  // ---- Q fragments (A operand, 16 rows x D): registers for bf16, shared memory for fp8
  uint32_t qa[C::FP8 ? 1 : D / 16][4];
  // fp8 KV: the warp's 16 q rows are multiplied by 2^-qe (their largest magnitude then
  // lies in [2^14, 2^15)) before the fp16 conversion the f16 MMA needs, and 2^qe goes back
  // into the score scale: the conversion cannot overflow, and every element within 2^-29
  // of the rows' largest converts exactly.  The scale waits in shared memory (the kernel
  // has no register to spare for it).
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* q0 = q + bq * p.q_sb + tq0 * p.q_st + h0 * p.q_sh;
    const __nv_bfloat16* q1 = q + bq * p.q_sb + tq1 * p.q_st + h1 * p.q_sh;
    float qsc = 1.f;  // 2^-qe
    if constexpr (C::FP8) {
      float amax = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int d0 = 16 * ks + 4 * tq;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (r == 0 ? v0 : v1) {
            const uint2 u = *reinterpret_cast<const uint2*>((r == 0 ? q0 : q1) + d0);
            const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
            const __nv_bfloat162 bb = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
            amax = fmaxf(fmaxf(amax, fmaxf(fabsf(__low2float(a)), fabsf(__high2float(a)))),
                         fmaxf(fabsf(__low2float(bb)), fabsf(__high2float(bb))));
          }
        }
      }
      // non-negative floats order as their bit patterns (a NaN above every number)
      amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
      int qe = 0;  // all-zero or non-finite rows keep their values
      if (amax > 0.f && amax <= 3.4e38f)
        qe = min(max(static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 14, -100), 100);
      qsc = __uint_as_float(static_cast<uint32_t>(127 - qe) << 23);
      if (wn == 0 && lane == 0) qscale[wm] = p.scale_log2 * __uint_as_float(static_cast<uint32_t>(127 + qe) << 23);
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      if constexpr (!C::FP8) {
        const int d0 = 16 * ks + 2 * tq;
        qa[ks][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + d0) : 0u;
        qa[ks][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + d0) : 0u;
        qa[ks][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + d0 + 8) : 0u;
        qa[ks][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + d0 + 8) : 0u;
      } else {
        // k-slots (2tq, 2tq+1 | 2tq+8, 2tq+9) hold d = 16ks + 4tq + (0,1 | 2,3), the
        // order in which ldmatrix delivers the e4m3 key bytes
        const int d0 = 16 * ks + 4 * tq;
        float f0[4] = {0.f, 0.f, 0.f, 0.f}, f1[4] = {0.f, 0.f, 0.f, 0.f};
        if (v0) {
          const uint2 u = *reinterpret_cast<const uint2*>(q0 + d0);
          const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
          const __nv_bfloat162 bb = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
          f0[0] = __low2float(a) * qsc; f0[1] = __high2float(a) * qsc;
          f0[2] = __low2float(bb) * qsc; f0[3] = __high2float(bb) * qsc;
        }
        if (v1) {
          const uint2 u = *reinterpret_cast<const uint2*>(q1 + d0);
          const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
          const __nv_bfloat162 bb = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
          f1[0] = __low2float(a) * qsc; f1[1] = __high2float(a) * qsc;
          f1[2] = __low2float(bb) * qsc; f1[3] = __high2float(bb) * qsc;
        }
        if (wn == 0) {
          qfrag[(wm * (D / 16) + ks) * 32 + lane] =
              make_uint4(pack_f16(f0[0], f0[1]), pack_f16(f1[0], f1[1]), pack_f16(f0[2], f0[3]),
                         pack_f16(f1[2], f1[3]));
        }
      }
    }
  }
  if constexpr (C::FP8) named_bar_sync(1, C::NCW * 32);  // q fragments and scales visible to every consumer

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrun[2] = {-INFINITY, -INFINITY};
  float lrun[2] = {0.f, 0.f};
  const float* kscale_row = nullptr;
  const float* vscale_row = nullptr;
  if constexpr (C::FP8) {
    kscale_row = p.k_scale + (static_cast<int64_t>(bkv) * p.Hkv + g) * p.n_scale_blk;
    vscale_row = p.v_scale + (static_cast<int64_t>(bkv) * p.Hkv + g) * p.n_scale_blk;
  }

  for (int i = wn; i < n_tiles; i += WN) {
    const int s = i % NSTAGE;
    const int t0 = (tile_begin + i) * TN;
    float ksc = 1.f, vsc = 1.f;
    if constexpr (C::FP8) {
      if constexpr (!PAGED) {
        ksc = __ldg(kscale_row + t0 / p.scale_block);
        vsc = __ldg(vscale_row + t0 / p.scale_block);
      } else {
        // per-page scales [num_blocks][Hkv][block_len / scale_block]; a page outside the
        // cache reads as zeros through TMA, so its scale is never fetched
        const int page = kv_page_of(p, bkv, t0);
        if (page >= 0 && page < p.num_blocks) {
          const int per = p.block_len / p.scale_block;
          const int64_t idx = (static_cast<int64_t>(page) * p.Hkv + g) * per + (t0 % p.block_len) / p.scale_block;
          ksc = __ldg(p.k_scale + idx);
          vsc = __ldg(p.v_scale + idx);
        } else {
          ksc = vsc = 0.f;
        }
      }
    }
    if (!mbar_wait(&full[full_slot<C>(i)], full_parity<C>(i), p.err, kDevErrFullWait)) break;
    const uint32_t kbase = smem_u32(smem + s * C::STAGE_BYTES);
    const uint32_t vbase = kbase + C::TILE_BYTES;
    const int mi = lane >> 3;
    constexpr int NS = C::SUB;
#pragma unroll 1
    for (int sub = 0; sub < TN / NS; ++sub) {
    const int t0s = t0 + sub * NS;
    const int tb = sub * NS;  // first token of this step inside the tile

    // ---- S = Q K^T  (16 x NS)
    float sc[NS / 8][4];
#pragma unroll
    for (int i2 = 0; i2 < NS / 8; ++i2) sc[i2][0] = sc[i2][1] = sc[i2][2] = sc[i2][3] = 0.f;
    if constexpr (!C::FP8) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < NS / 16; ++np) {
          const uint32_t tok = tb + 16 * np + (mi >> 1) * 8 + (lane & 7);
          const uint32_t byte = (2 * ks + (mi & 1)) * 16;
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kbase + tile_off<C>(tok, byte), r0, r1, r2, r3);
          mma_bf16(sc[2 * np], qa[ks], r0, r1);
          mma_bf16(sc[2 * np + 1], qa[ks], r2, r3);
        }
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < D / 16; ks += 2) {
        const uint4 qv0 = qfrag[(wm * (D / 16) + ks) * 32 + lane];
        const uint4 qv1 = qfrag[(wm * (D / 16) + ks + 1) * 32 + lane];
        const uint32_t qa0[4] = {qv0.x, qv0.y, qv0.z, qv0.w};
        const uint32_t qa1[4] = {qv1.x, qv1.y, qv1.z, qv1.w};
#pragma unroll
        for (int np = 0; np < NS / 16; ++np) {
          const uint32_t tok = tb + 16 * np + (mi >> 1) * 8 + (lane & 7);
          const uint32_t byte = (ks + (mi & 1)) * 16;
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kbase + tile_off<C>(tok, byte), r0, r1, r2, r3);
          uint32_t k0l, k0h, k1l, k1h, k2l, k2h, k3l, k3h;
          e4m3x4_to_f16x2x2(r0, k0l, k0h);
          e4m3x4_to_f16x2x2(r1, k1l, k1h);
          e4m3x4_to_f16x2x2(r2, k2l, k2h);
          e4m3x4_to_f16x2x2(r3, k3l, k3h);
          mma_f16(sc[2 * np], qa0, k0l, k0h);
          mma_f16(sc[2 * np], qa1, k1l, k1h);
          mma_f16(sc[2 * np + 1], qa0, k2l, k2h);
          mma_f16(sc[2 * np + 1], qa1, k3l, k3h);
        }
      }
    }

    // ---- scale, mask, online softmax (fp8: the q scaling undone here)
    float sl = p.scale_log2;
    if constexpr (C::FP8) sl = *reinterpret_cast<volatile const float*>(qscale + wm) * ksc;
    const bool in_range = (t0s >= r_lo) && (t0s + NS <= r_hi);
    const bool need_mask = POS || !in_range || (static_cast<int64_t>(t0s) + NS - 1 > hz_min);
    float tmax[2] = {-INFINITY, -INFINITY};
    // fp8: one instantiation per mask mode (need_mask is warp-uniform; written as one loop
    // with the test inside, the compiler evaluated it on every tile, and the fp8 decode does
    // twice the arithmetic per byte of the bf16 one).  bf16 keeps the single masked loop: its
    // kernel time moved by under 1 % either way.
    auto scale_mask = [&](auto masked) {
#pragma unroll
      for (int nt = 0; nt < NS / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = sc[nt][e] * sl;
          if constexpr (decltype(masked)::value) {
            const int tok = t0s + 8 * nt + 2 * tq + (e & 1);
            const int64_t hz = (e < 2) ? hz0 : hz1;
            bool ok = tok >= r_lo && tok < r_hi && static_cast<int64_t>(tok) <= hz;
            if constexpr (POS) ok = ok && __ldg(kpos_b + tok) <= ((e < 2) ? qp0 : qp1);
            x = ok ? x : -INFINITY;
          }
          sc[nt][e] = x;
          tmax[e >> 1] = fmaxf(tmax[e >> 1], x);
        }
      }
    };
    if (!C::FP8 || need_mask)
      scale_mask(std::true_type{});
    else
      scale_mask(std::false_type{});
    float base[2], alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
      const float mnew = fmaxf(mrun[r], tmax[r]);
      base[r] = (mnew == -INFINITY) ? 0.f : mnew;
      alpha[r] = fast_exp2(mrun[r] - base[r]);  // 0 when mrun = -inf
      mrun[r] = mnew;
      lrun[r] *= alpha[r];
    }
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {  // a row max moved
      if constexpr (!C::FP8) {
#pragma unroll
        for (int i2 = 0; i2 < D / 8; ++i2) {
          o[i2][0] *= alpha[0];
          o[i2][1] *= alpha[0];
          o[i2][2] *= alpha[1];
          o[i2][3] *= alpha[1];
        }
      } else {
        // O^T: this thread's columns are rows 2tq, 2tq+1 (+8) of the row set
        float ar[2][2];
        ar[0][0] = __shfl_sync(0xffffffffu, alpha[0], 8 * tq);
        ar[0][1] = __shfl_sync(0xffffffffu, alpha[0], 8 * tq + 4);
        ar[1][0] = __shfl_sync(0xffffffffu, alpha[1], 8 * tq);
        ar[1][1] = __shfl_sync(0xffffffffu, alpha[1], 8 * tq + 4);
#pragma unroll
        for (int i2 = 0; i2 < D / 8; ++i2) {
          const int n = i2 & 1;
          o[i2][0] *= ar[n][0];
          o[i2][1] *= ar[n][1];
          o[i2][2] *= ar[n][0];
          o[i2][3] *= ar[n][1];
        }
      }
    }
    uint32_t pa[NS / 16][4];
#pragma unroll
    for (int nt = 0; nt < NS / 8; ++nt) {
      const float p0 = fast_exp2(sc[nt][0] - base[0]);
      const float p1 = fast_exp2(sc[nt][1] - base[0]);
      const float p2 = fast_exp2(sc[nt][2] - base[1]);
      const float p3 = fast_exp2(sc[nt][3] - base[1]);
      lrun[0] += p0 + p1;
      lrun[1] += p2 + p3;
      const int kk = nt >> 1, hf = (nt & 1) * 2;
      if constexpr (!C::FP8) {
        pa[kk][hf + 0] = pack_bf16(p0, p1);
        pa[kk][hf + 1] = pack_bf16(p2, p3);
      } else {
        pa[kk][hf + 0] = pack_f16(p0 * vsc, p1 * vsc);
        pa[kk][hf + 1] = pack_f16(p2 * vsc, p3 * vsc);
      }
    }

    // ---- O += P V (the masks of V rows outside [r_lo, r_hi): as for the scores, fp8 keeps
    // them out of the instantiation for tiles that need none)
    const bool vmask = !in_range;
    auto pv = [&](auto vmasked) {
#pragma unroll
    for (int kk = 0; kk < NS / 16; ++kk) {
      if constexpr (!C::FP8) {
        uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
        if constexpr (decltype(vmasked)::value) {
          const int ta = t0s + 16 * kk + 2 * tq, tb2 = ta + 8;
          mlo = half_mask(ta >= r_lo && ta < r_hi, ta + 1 >= r_lo && ta + 1 < r_hi);
          mhi = half_mask(tb2 >= r_lo && tb2 < r_hi, tb2 + 1 >= r_lo && tb2 + 1 < r_hi);
        }
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const uint32_t tok = tb + 16 * kk + (mi & 1) * 8 + (lane & 7);
          const uint32_t byte = (2 * dp + (mi >> 1)) * 16;
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(vbase + tile_off<C>(tok, byte), r0, r1, r2, r3);
          if constexpr (decltype(vmasked)::value) {
            r0 &= mlo, r1 &= mhi, r2 &= mlo, r3 &= mhi;
          }
          mma_bf16(o[2 * dp], pa[kk], r0, r1);
          mma_bf16(o[2 * dp + 1], pa[kk], r2, r3);
        }
      } else {
        // O^T[dv x rows] += V^T[dv x tok] P^T[tok x rows]: ldmatrix.trans of the e4m3 tile
        // (16-bit view) gives each lane bytes V[2tq][2gq], V[2tq][2gq+1], V[2tq+1][2gq],
        // V[2tq+1][2gq+1]; one byte permute pairs them by dv, so the A rows gq / gq+8 of a
        // 16-dv chunk c are dv 16c+2gq / 16c+2gq+1, and P's fragments are already the B
        // operand (columns = the 16 rows).
        uint32_t m0 = 0xFFFFFFFFu, m1 = 0xFFFFFFFFu;
        if constexpr (decltype(vmasked)::value) {
          const int ta = t0s + 16 * kk + 2 * tq, tb2 = ta + 8;
          m0 = half_mask(ta >= r_lo && ta < r_hi, ta + 1 >= r_lo && ta + 1 < r_hi);
          m1 = half_mask(tb2 >= r_lo && tb2 < r_hi, tb2 + 1 >= r_lo && tb2 + 1 < r_hi);
        }
        const uint32_t b00 = pa[kk][0], b01 = pa[kk][2], b10 = pa[kk][1], b11 = pa[kk][3];
#pragma unroll
        for (int cc = 0; cc < D / 16; ++cc) {
          const uint32_t tok = tb + 16 * kk + ((lane >> 3) & 1) * 8 + (lane & 7);
          uint32_t r0, r1;
          ldsm_x2_t(vbase + tile_off<C>(tok, cc * 16), r0, r1);
          uint32_t a[4];
          if constexpr (decltype(vmasked)::value) {
            r0 &= m0, r1 &= m1;
          }
          e4m3x4_to_f16x2x2(prmt(r0, 0u, 0x3120u), a[0], a[1]);
          e4m3x4_to_f16x2x2(prmt(r1, 0u, 0x3120u), a[2], a[3]);
          mma_f16(o[2 * cc], a, b00, b01);
          mma_f16(o[2 * cc + 1], a, b10, b11);
        }
      }
    }
    };
    if (!C::FP8 || vmask)
      pv(std::true_type{});
    else
      pv(std::false_type{});
    }  // sub-steps
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- finish: normalise, combine the WN warps of a row set, store
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], 1);
    lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], 2);
  }
  constexpr float kLn2 = 0.6931471805599453f;
  int64_t oslot;
  if constexpr (RING)
    oslot = ring_out_slot(p);
  else
    oslot = static_cast<int64_t>(j * p.n_chunk + c) * p.B + b;
  auto row_out = [&](int t_q, int h) -> int64_t { return (oslot * p.Tq + t_q) * p.Hq + h; };

  if constexpr (WN == 1) {
    const float inv0 = lrun[0] > 0.f ? 1.f / lrun[0] : 0.f;
    const float inv1 = lrun[1] > 0.f ? 1.f / lrun[1] : 0.f;
    const bool w0 = v0 && (lrun[0] > 0.f || p.zero_empty);
    const bool w1 = v1 && (lrun[1] > 0.f || p.zero_empty);
    if constexpr (!C::FP8) {
      float* o0 = p.out_o + row_out(tq0, h0) * D;
      float* o1 = p.out_o + row_out(tq1, h1) * D;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        const int d = 8 * nt + 2 * tq;
        if (w0) *reinterpret_cast<float2*>(o0 + d) = make_float2(o[nt][0] * inv0, o[nt][1] * inv0);
        if (w1) *reinterpret_cast<float2*>(o1 + d) = make_float2(o[nt][2] * inv1, o[nt][3] * inv1);
      }
    } else {
      // O^T: this thread holds rows (8n + 2tq + {0,1}) at dv 16c + 2gq + {0,1}
#pragma unroll
      for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int src = 4 * (2 * tq + e);
          const float inv = __shfl_sync(0xffffffffu, n ? inv1 : inv0, src);
          const bool wr = __shfl_sync(0xffffffffu, (n ? w1 : w0) ? 1 : 0, src) != 0;
          const int tq_r = __shfl_sync(0xffffffffu, n ? tq1 : tq0, src);
          const int h_r = __shfl_sync(0xffffffffu, n ? h1 : h0, src);
          float* orow = p.out_o + row_out(tq_r, h_r) * D;
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            const float* ov = o[2 * c + n];
            if (wr) *reinterpret_cast<float2*>(orow + 16 * c + 2 * gq) = make_float2(ov[e] * inv, ov[2 + e] * inv);
          }
        }
      }
    }
    if (tq == 0) {
      if (v0) p.out_lse[row_out(tq0, h0)] = lrun[0] > 0.f ? (mrun[0] + __log2f(lrun[0])) * kLn2 : -INFINITY;
      if (v1) p.out_lse[row_out(tq1, h1)] = lrun[1] > 0.f ? (mrun[1] + __log2f(lrun[1])) * kLn2 : -INFINITY;
    }
  } else {
    constexpr int NCT = C::NCW * 32;
    named_bar_sync(1, NCT);  // every consumer is done with the ring
    const int lr0 = wm * 16 + gq, lr1 = lr0 + 8;  // local rows
    if (tq == 0) {
      ml[(wn * C::ROWS + lr0) * 2 + 0] = mrun[0];
      ml[(wn * C::ROWS + lr0) * 2 + 1] = lrun[0];
      ml[(wn * C::ROWS + lr1) * 2 + 0] = mrun[1];
      ml[(wn * C::ROWS + lr1) * 2 + 1] = lrun[1];
    }
    named_bar_sync(1, NCT);
    float f[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int lr = r ? lr1 : lr0;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < WN; ++w) M = fmaxf(M, ml[(w * C::ROWS + lr) * 2]);
      float L = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < WN; ++w) L += ml[(w * C::ROWS + lr) * 2 + 1] * fast_exp2(ml[(w * C::ROWS + lr) * 2] - M);
      }
      f[r] = (L > 0.f) ? fast_exp2(mrun[r] - M) / L : 0.f;
    }
    float* obuf = reinterpret_cast<float*>(smem);  // [WN][ROWS][D]
    if constexpr (!C::FP8) {
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        const int d = 8 * nt + 2 * tq;
        *reinterpret_cast<float2*>(obuf + (wn * C::ROWS + lr0) * D + d) =
            make_float2(o[nt][0] * f[0], o[nt][1] * f[0]);
        *reinterpret_cast<float2*>(obuf + (wn * C::ROWS + lr1) * D + d) =
            make_float2(o[nt][2] * f[1], o[nt][3] * f[1]);
      }
    } else {
#pragma unroll
      for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float fr = __shfl_sync(0xffffffffu, n ? f[1] : f[0], 4 * (2 * tq + e));
          const int lr = wm * 16 + 8 * n + 2 * tq + e;
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            const float* ov = o[2 * c + n];
            *reinterpret_cast<float2*>(obuf + (wn * C::ROWS + lr) * D + 16 * c + 2 * gq) =
                make_float2(ov[e] * fr, ov[2 + e] * fr);
          }
        }
      }
    }
    named_bar_sync(1, NCT);
    const int tid = threadIdx.x;  // < NCT
    for (int e = tid * 4; e < C::ROWS * D; e += NCT * 4) {
      const int lr = e / D, d = e % D;
      const int m = m0 + lr;
      if (m >= rows_total) continue;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < WN; ++w) M = fmaxf(M, ml[(w * C::ROWS + lr) * 2]);
      float L = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < WN; ++w) L += ml[(w * C::ROWS + lr) * 2 + 1] * fast_exp2(ml[(w * C::ROWS + lr) * 2] - M);
      }
      const int t_q = m / p.G, h = g * p.G + m % p.G;
      const int64_t ro = row_out(t_q, h);
      if (L > 0.f || p.zero_empty) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < WN; ++w) {
          const float4 x = *reinterpret_cast<const float4*>(obuf + (w * C::ROWS + lr) * D + d);
          acc.x += x.x;
          acc.y += x.y;
          acc.z += x.z;
          acc.w += x.w;
        }
        *reinterpret_cast<float4*>(p.out_o + ro * D + d) = acc;
      }
      if (d == 0) p.out_lse[ro] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
    }
  }
}

using CfgBf16D64Dec = GqaCfg<false, 64, 1, 4, 6, 2>;
using CfgBf16D128Dec = GqaCfg<false, 128, 1, 3, 3, 2>;
using CfgFp8D128Dec = GqaCfg<true, 128, 1, 4, 6, 2>;
using CfgBf16D64Pre = GqaCfg<false, 64, 4, 1, 6, 2>;
using CfgBf16D128Pre = GqaCfg<false, 128, 4, 1, 3, 2>;
using CfgFp8D128Pre = GqaCfg<true, 128, 4, 1, 5, 2>;

template <class C>
GqaLaunchInfo info_of() {
  return GqaLaunchInfo{C::ROWS, C::THREADS, C::SMEM, C::MINB};
}

template <class C>
cudaError_t launch_cfg(const PartialParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv, int64_t n_items,
                       cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};  // per variant, per device
  cudaError_t e0 = once_per_device(attr_done, [] {
    const void* fns[5] = {reinterpret_cast<const void*>(gqa_partial_kernel<C, false, false, false>),
                          reinterpret_cast<const void*>(gqa_partial_kernel<C, true, false, false>),
                          reinterpret_cast<const void*>(gqa_partial_kernel<C, false, true, false>),
                          reinterpret_cast<const void*>(gqa_partial_kernel<C, true, true, false>),
                          reinterpret_cast<const void*>(gqa_partial_kernel<C, false, false, true>)};
    for (const void* f : fns) {
      cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  });
  if (e0 != cudaSuccess) return e0;
  if (n_items <= 0) return cudaSuccess;
  const unsigned int grid = static_cast<unsigned int>(n_items);
  if (p.ring_n > 0) {
    if (p.block_table || p.k_pos) return cudaErrorInvalidValue;  // no such instantiation
    gqa_partial_kernel<C, false, false, true><<<grid, C::THREADS, C::SMEM, stream>>>(p, tmk, tmv);
  } else if (p.block_table && p.k_pos) {
    gqa_partial_kernel<C, true, true, false><<<grid, C::THREADS, C::SMEM, stream>>>(p, tmk, tmv);
  } else if (p.block_table) {
    gqa_partial_kernel<C, true, false, false><<<grid, C::THREADS, C::SMEM, stream>>>(p, tmk, tmv);
  } else if (p.k_pos) {
    gqa_partial_kernel<C, false, true, false><<<grid, C::THREADS, C::SMEM, stream>>>(p, tmk, tmv);
  } else {
    gqa_partial_kernel<C, false, false, false><<<grid, C::THREADS, C::SMEM, stream>>>(p, tmk, tmv);
  }
  return cudaGetLastError();
}

}  // namespace

GqaLaunchInfo gqa_launch_info(GqaVariant v) {
  switch (v) {
    case GqaVariant::kBf16D64Decode: return info_of<CfgBf16D64Dec>();
    case GqaVariant::kBf16D128Decode: return info_of<CfgBf16D128Dec>();
    case GqaVariant::kFp8D128Decode: return info_of<CfgFp8D128Dec>();
    case GqaVariant::kBf16D64Prefill: return info_of<CfgBf16D64Pre>();
    case GqaVariant::kBf16D128Prefill: return info_of<CfgBf16D128Pre>();
    case GqaVariant::kFp8D128Prefill: return info_of<CfgFp8D128Pre>();
  }
  return GqaLaunchInfo{0, 0, 0, 1};
}

cudaError_t launch_gqa_partial(GqaVariant v, const PartialParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                               int64_t n_items, cudaStream_t stream) {
  switch (v) {
    case GqaVariant::kBf16D64Decode: return launch_cfg<CfgBf16D64Dec>(p, tmk, tmv, n_items, stream);
    case GqaVariant::kBf16D128Decode: return launch_cfg<CfgBf16D128Dec>(p, tmk, tmv, n_items, stream);
    case GqaVariant::kFp8D128Decode: return launch_cfg<CfgFp8D128Dec>(p, tmk, tmv, n_items, stream);
    case GqaVariant::kBf16D64Prefill: return launch_cfg<CfgBf16D64Pre>(p, tmk, tmv, n_items, stream);
    case GqaVariant::kBf16D128Prefill: return launch_cfg<CfgBf16D128Pre>(p, tmk, tmv, n_items, stream);
    case GqaVariant::kFp8D128Prefill: return launch_cfg<CfgFp8D128Pre>(p, tmk, tmv, n_items, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace skv
