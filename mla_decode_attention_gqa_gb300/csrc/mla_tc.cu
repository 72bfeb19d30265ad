// Tensor-core (tcgen05) split-KV attention for the MLA latent cache: 128 query heads
// (the MMA M) attend over one shared latent row per token (576 dims = 512 latent + 64
// rope as the key; its first 512 dims as the value).
//
// What it computes: the same partial (normalised o, natural-log lse) per split as the
// other kernels -- "Helix Parallelism: Why Tensor Parallelism Hits a Wall at
// Million-Token Context" (sections "Sharding the sequence instead" and, for the single
// shared latent, "The ceiling, in algebra") -- or, fused, the exact merge of all splits
// (the online softmax over their union), written as the final bf16 output.
//
// GB300 design: a cluster of two CTAs on two SMs serves one (sequence, split, chunk)
// item.  The output O = P V of 128 heads x 512 dims in fp32 fills all 512 TMEM columns
// of one SM, and the scores need the whole 576-dim contraction, so the pair splits the
// two products instead of the dims:
//   CTA 0 (scores) keeps Q (128 x 576) -- dims 0..511 in tensor memory, the 64 rope dims
//          in shared memory -- streams the latent in tiles of 128 tokens, computes
//          S = Q K^T (M 128 heads, N 128 tokens, A from TMEM), runs the online softmax
//          (one thread per head = TMEM lane) and pushes P (bf16, already the MMA
//          operand) in two 64-token halves, with one rescale factor per head, into CTA 1's
//          shared memory with bulk DSMEM copies;
//   CTA 1 (values) streams the same tokens' first 512 dims in 64-token tiles (the second
//          read of each tile hits L2), applies the rescale factors to O in tensor memory
//          when a row maximum moved, and accumulates O += P V (A = P from shared memory,
//          B = the MN-major V tile, two N = 256 halves).
// Tensor work per 128 tokens: 36 MMAs of N = 128 on CTA 0 and 16 of N = 256 on CTA 1.
// An MMA-issuing warp runs its loop converged and lets one elected lane issue: an MMA then
// costs its issuer ~48 cycles, so N = 128 (64 cycles of tensor work) keeps the pipe busy
// from one warp, where N = 64 tiles (32 cycles) left it idle a third of the time.  CTA 0's
// latent tiles stream through a ring of 64-dim x 128-token boxes, waited for and released
// in three groups of three boxes per tile (one wait, fence and commit per twelve MMAs).
// Only bf16 P (32 KB per 128 tokens) crosses between the SMs, one way.
// Warp roles per CTA: TMA producer, MMA issuer, four row warps (softmax on CTA 0;
// rescale, boundary-row zeroing and the epilogue on CTA 1).  Every wait is bounded.
#include <cuda_runtime.h>

#include "skv_common.cuh"
#include "skv_internal.h"
#include "tc_common.cuh"

namespace skv {

namespace {

constexpr int kTN = 64;          // tokens per value tile (CTA 1) and per P half
constexpr int kTS = 128;         // tokens per score tile (CTA 0): two value tiles
constexpr int kRows = 128;       // heads per item (MMA M)
constexpr int kThreads = 6 * 32;
constexpr int kKBoxes = 9;       // 64-dim boxes of the 576-dim key
constexpr int kVBoxes = 8;       // 64-dim boxes of the 512-dim value
constexpr int kBoxBytes = kTN * 128;     // 64 tokens x 64 dims (one TMA box)
constexpr int kSBoxBytes = kTS * 128;    // 128 tokens x 64 dims (a CTA 0 ring slot, two TMA boxes)
constexpr int kQBoxBytes = kRows * 128;  // 128 heads x 64 dims
// CTA 0 (scores): Q staging, then a ring of kNBox0 box slots in the same bytes, filled and
// released in groups of kGrp consecutive boxes of the stream (one wait and one release per
// group: per box, the issuing warp's wait, fence and commit cost as much as its four MMAs)
constexpr int kNBox0 = 10;
constexpr int kGrp = 3;                // three groups per score tile, one ring slot each
constexpr int kNGrp0 = kKBoxes / kGrp;  // group slots (the tenth box slot stays unused)
constexpr int kOffPStage = kNBox0 * kSBoxBytes;      // 160 KB: P staging, 2 halves x 16 KB
constexpr int kPBytes = kRows * 128;                 // 128 heads x 64 tokens bf16
constexpr int kOffAStage = kOffPStage + 2 * kPBytes;  // rescale factors, 2 slots x 512 B
constexpr int kOffLStage = kOffAStage + 2 * kRows * 4;  // final row sums, 512 B
constexpr int kOffQRope = 198656;  // Q dims 512..575 (the rope part), 16 KB, kept in shared memory
constexpr int kQTmemBoxes = 8;     // Q dims 0..511 live in TMEM
// CTA 1 (values): a 3-stage ring of 512-dim tiles, P / factor / row-sum receive buffers
constexpr int kNStage1 = 3;
constexpr int kPfAhead = 6;  // value tiles (64 tokens) between CTA 1's load and its L2 prefetch
constexpr int kStage1Bytes = kVBoxes * kBoxBytes;  // 64 KB
constexpr int kOffPRecv = kNStage1 * kStage1Bytes;  // 192 KB
constexpr int kOffARecv = kOffPRecv + 2 * kPBytes;
constexpr int kOffLRecv = kOffARecv + 2 * kRows * 4;
constexpr int kOffBar = kOffLRecv + kRows * 4;
constexpr int kSmem = 1024 + kOffBar + 512;
static_assert(kQTmemBoxes * kQBoxBytes <= kNBox0 * kSBoxBytes, "Q staging reuses the ring bytes");
static_assert(kOffQRope % 1024 == 0 && kOffQRope >= kOffLStage + kRows * 4 && kOffQRope + kQBoxBytes <= kOffBar,
              "CTA 0's rope Q sits between its staging buffers and the barriers");
static_assert(kOffLStage + kRows * 4 <= kOffBar, "CTA 0 layout fits below the barriers");
static_assert(kOffPStage % 1024 == 0 && kOffPRecv % 1024 == 0, "P tiles need 1024-byte swizzle atoms");
static_assert(kSmem <= 227 * 1024, "shared memory budget");
static_assert(kNBox0 > kKBoxes, "the ring holds a whole score tile and the start of the next");
static_assert(kKBoxes % kGrp == 0 && kNGrp0 * kGrp <= kNBox0, "whole groups of a tile's boxes per ring slot");
constexpr uint32_t kTmemCols = 512;
// CTA 0: S buffer b (128 x 128 fp32) at columns 128 b; Q dims 0..511 at 256.. (two bf16 per column)
constexpr uint32_t kColS = 0;
constexpr uint32_t kColQ = 256;
constexpr uint32_t kColO = 0;    // CTA 1: O, 512 columns
constexpr uint32_t kPMsgBytes = 4 * (32 * 128 + 32 * 4);  // P rows + factors of one half, four warps
constexpr float kRescaleThreshold = 8.0f;

// One barrier block at the same offset in both CTAs (remote arrivals address a peer's
// barrier by this CTA's own offset).
struct MlaBars {
  // CTA 0
  uint64_t q_full;        // Q staged in shared memory
  uint64_t q_moved;       // Q copied into TMEM by the four row warps; staging bytes free
  uint64_t grp_full[kNGrp0];   // the boxes of a group landed
  uint64_t grp_empty[kNGrp0];  // the MMAs that read a group completed
  uint64_t s_full[2];     // S of score tile T in TMEM buffer T & 1
  uint64_t s_free[2];     // the row warps have read S buffer b
  uint64_t p_empty[2];    // CTA 1 finished PV with P slot b (arrived by CTA 1's MMA commit)
  // CTA 1
  uint64_t kv_full1[kNStage1];
  uint64_t kv_empty1[kNStage1];
  uint64_t p_full[2];     // P slot b and its factors landed (bulk copies from CTA 0)
  uint64_t o_ready[2];    // rescale / boundary zeroing for tile i done (slot i & 1)
  uint64_t pv_done;       // every PV issued so far completed
  uint64_t o_final;       // the last PV completed
  uint64_t l_full;        // the final row sums landed
  uint32_t tmem_base;
};
static_assert(sizeof(MlaBars) <= 512, "barrier block");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_addr), "r"(rank));
  return d;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bulk copy from this CTA's shared memory into a peer's, completing on the peer's barrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                                  uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(src_cta), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

// One arrive, on the barrier at this offset in every CTA of cta_mask, when all MMAs this
// thread issued so far have completed.
__device__ __forceinline__ void mma_commit_multicast(uint32_t mbar_smem_addr, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          mbar_smem_addr),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_plain(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                                  int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// Bulk copy of `bytes` contiguous shared-memory bytes to global memory (this thread's bulk
// group), and the waits for this thread's groups: sources read / copies complete.
__device__ __forceinline__ void bulk_store_global(void* dst, uint32_t src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\tcp.async.bulk.commit_group;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(src_smem), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// A warp's wait: every lane polls, and the warp leaves together.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned int* err) {
  const bool ok = mbar_wait(bar, parity, err, kDevErrFullWait);
  return __all_sync(0xffffffffu, ok);
}

// Page (paged cache) or sequence (contiguous) and row coordinate of the 64-token tile that
// starts at token `tok`.  A tile at or past S_max holds only masked tokens; over a paged
// cache it reads the page of the last tile inside S_max instead of a block-table entry past
// the sequence's row.
template <bool PAGED>
__device__ __forceinline__ void tile_coords(const PartialParams& p, int b, int tok, int* outer, int* row) {
  if constexpr (PAGED) {
    const int t = tok < p.S_max ? tok : ((p.S_max - 1) / kTN) * kTN;
    *outer = kv_page_of(p, b, t);
    *row = t % p.block_len;
  } else {
    *outer = b;
    *row = tok;
  }
}

// PAGED: the latent lives in pages with a block table (kept out of the contiguous
// instantiation: the extra producer code alone slowed it by a tenth)
template <bool PAGED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_tc_kernel(const __grid_constant__ PartialParams p, const __grid_constant__ TcAttnExtra x,
                  const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tml,
                  const __grid_constant__ CUtensorMap tmg, const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  MlaBars* bars = reinterpret_cast<MlaBars*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();

  // ---- work item of the pair: (b, [split j,] chunk c, row tile mt)
  int64_t item = blockIdx.x >> 1;
  const int mt = static_cast<int>(item % p.m_tiles);
  item /= p.m_tiles;
  const int c = static_cast<int>(item % p.n_chunk);
  item /= p.n_chunk;
  int j = 0;
  if (!x.fused) {
    j = static_cast<int>(item % p.n_split);
    item /= p.n_split;
  }
  const int b = static_cast<int>(item);
  const int seq_len = p.seq_lens[b];
  int lo, hi, win_lo, win_hi;
  split_range(p, b, x.fused ? 0 : j, x.fused ? p.n_split : j + 1, seq_len, &lo, &hi);
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
  // value tiles (64 tokens) from tile_begin; score tiles pair them, so the value CTA runs
  // an even count (a last value tile past r_hi holds only masked tokens)
  const int tile_begin = r_lo / kTN;
  const int n64 = (r_hi > r_lo) ? ((r_hi + kTN - 1) / kTN - tile_begin) : 0;
  const int n_score = (n64 + 1) / 2;
  const int n_tiles = 2 * n_score;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_moved, 4);
    for (int s = 0; s < kNGrp0; ++s) {
      mbar_init(&bars->grp_full[s], 1);
      mbar_init(&bars->grp_empty[s], 1);
    }
    for (int s = 0; s < kNStage1; ++s) {
      mbar_init(&bars->kv_full1[s], 1);
      mbar_init(&bars->kv_empty1[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars->s_full[k], 1);
      mbar_init(&bars->s_free[k], 4);
      mbar_init(&bars->p_empty[k], 1);
      mbar_init(&bars->p_full[k], 1);
      mbar_init(&bars->o_ready[k], 4);
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_final, 1);
    mbar_init(&bars->l_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive or copy
  const uint32_t tmem = bars->tmem_base;
  const int lgrp = warp & 3;         // row warps 2..5 -> TMEM lane groups 2, 3, 0, 1
  const int row = lgrp * 32 + lane;  // head row of the item (row warps)
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(lgrp * 32) << 16);

  if (rank == 0) {
    // ================================================================ CTA 0: scores
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      // box bx (dims 64 bx ..) of every score tile sits in ring box slot bx; group g = boxes 3g .. 3g + 2
      if (lane == 0 && n_score > 0) {
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(PAGED ? &tml : &tmg);
        mbar_arrive_expect_tx(&bars->q_full, kKBoxes * kQBoxBytes);
        const int t_start = m0 / p.G;
        for (int bx = 0; bx < kKBoxes; ++bx)
          tma_load_4d_plain(smem + (bx < kQTmemBoxes ? bx * kQBoxBytes : kOffQRope), &tmq, &bars->q_full, bx * 64, 0,
                            t_start, b);
        bool ok = mbar_wait(&bars->q_moved, 0, p.err, kDevErrEmptyWait);  // the ring bytes are free
        int outer0 = b, row0 = 0, outer1 = b, row1 = 0;
        int issued = 0;  // groups issued
        for (int T = 0; T < n_score && ok; ++T) {
          const int tok = (tile_begin + 2 * T) * kTN;
          tile_coords<PAGED>(p, b, tok, &outer0, &row0);
          tile_coords<PAGED>(p, b, tok + kTN, &outer1, &row1);
          for (int g = 0; g < kNGrp0; ++g) {  // group g of tile T goes to slot g
            if (T >= 1 && !mbar_wait(&bars->grp_empty[g], (T - 1) & 1, p.err, kDevErrEmptyWait)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->grp_full[g], kGrp * kSBoxBytes);
            if constexpr (!PAGED) {
              // the group's three 64-dim slices of the tile's 128 tokens in one copy: the
              // chunked view's box lands as [slice][token][128 B], the ring's own layout
              tma_load_4d_plain(smem + g * kGrp * kSBoxBytes, &tmg, &bars->grp_full[g], 0, row0, g * kGrp, outer0);
            } else {
              for (int e = 0; e < kGrp; ++e) {
                const int bx = g * kGrp + e;
                uint8_t* st = smem + bx * kSBoxBytes;
                tma_load_4d_plain(st, &tml, &bars->grp_full[g], bx * 64, row0, 0, outer0);
                tma_load_4d_plain(st + kBoxBytes, &tml, &bars->grp_full[g], bx * 64, row1, 0, outer1);
              }
            }
            ++issued;
          }
        }
        for (int gi = max(0, issued - kNGrp0); gi < issued; ++gi) {
          if (!mbar_wait(&bars->grp_full[gi % kNGrp0], (gi / kNGrp0) & 1, p.err, kDevErrDrainWait)) break;
        }
        if (!ok) mbar_wait(&bars->q_full, 0, p.err, kDevErrDrainWait);  // Q copy still in flight
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer: S = Q K^T
      // Per score tile: for each 64-dim box, four k-steps (M 128, N 128 tokens, K 16; A = Q
      // from TMEM, the rope box's from shared memory), then the box is released.  The warp
      // runs the loop and its waits together; one elected lane issues and commits.
      if (n_score > 0) {
        const uint32_t idesc_s = tc::idesc_f16(128, kTS, true, false, false);
        const uint32_t ring = smem_u32(smem);
        const uint64_t qrope_d0 = tc::smem_desc_sw128(smem_u32(smem + kOffQRope), 16, 1024);
        bool ok = warp_wait(&bars->q_moved, 0, p.err);
        // Every MMA operand is a compile-time offset from per-CTA bases (box bx of a tile
        // always sits in ring box slot bx): the unrolled tile body issues at the tensor
        // pipe's pace.  Only the S buffer alternates between tiles.
        const uint64_t bd_ring = tc::smem_desc_sw128(ring, 16, 1024);
        for (int T = 0; T < n_score && ok; ++T) {
          if (T >= 2) {  // S buffer T & 1 was read by the softmax of tile T - 2
            ok = warp_wait(&bars->s_free[T & 1], ((T >> 1) - 1) & 1, p.err);
            if (!ok) break;
          }
          const uint32_t d = tmem + kColS + 128 * (T & 1);
#pragma unroll
          for (int g = 0; g < kNGrp0; ++g) {
            ok = warp_wait(&bars->grp_full[g], T & 1, p.err);
            if (!ok) break;
            tc::fence_after_sync();
            if (tc::elect_one()) {
#pragma unroll
              for (int e = 0; e < kGrp; ++e) {
                const int bx = g * kGrp + e;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t bd = bd_ring + static_cast<uint64_t>((bx * kSBoxBytes + k * 32) >> 4);
                  if (bx < kQTmemBoxes)
                    tc::mma_f16_ts(d, tmem + kColQ + 32 * bx + 8 * k, bd, idesc_s, (bx | k) ? 1u : 0u);
                  else
                    tc::mma_f16_ss(d, qrope_d0 + static_cast<uint64_t>((k * 32) >> 4), bd, idesc_s, 1u);
                }
              }
              tc::mma_commit(smem_u32(&bars->grp_empty[g]));
              if (g == kNGrp0 - 1) tc::mma_commit(smem_u32(&bars->s_full[T & 1]));
            }
            __syncwarp();
          }
        }
      }
    } else {
      // ---------------------------------------------------------- row warps: softmax
      const int m = m0 + row;
      const bool valid = m < rows_total;
      const int t_q = valid ? m / p.G : 0;
      const int h = valid ? m % p.G : 0;
      const int64_t hz = p.causal_offset + t_q;
      const int64_t hz_min = p.causal_offset + (m0 + lgrp * 32) / p.G;
      const uint32_t peer_p_full0 = map_to_rank(smem_u32(&bars->p_full[0]), 1);
      const uint32_t peer_p_full1 = map_to_rank(smem_u32(&bars->p_full[1]), 1);
      const uint32_t peer_precv = map_to_rank(smem_u32(smem + kOffPRecv), 1);
      const uint32_t peer_arecv = map_to_rank(smem_u32(smem + kOffARecv), 1);
      // l_sum: the fp32 row sum (for the lse); l_pv: the sum of the bf16-rounded p that PV
      // uses, sent to CTA 1 to normalise O (an exact convex combination of V rows then; with
      // the optimistic max no p is exact)
      float m_used = -INFINITY, l_sum = 0.f, l_pv = 0.f;
      bool ok = true;

      if (n_score > 0) {
        // Q row, dims 0..511 -> TMEM columns kColQ + 32 bx + (0..31): the A operand of the
        // TMEM-fed S MMAs
        ok = warp_wait(&bars->q_full, 0, p.err);
        if (ok) {
#pragma unroll 1
          for (int bx = 0; bx < kQTmemBoxes; ++bx) {
            const uint8_t* qb = smem + bx * kQBoxBytes;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t w[16];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint4 v = *reinterpret_cast<const uint4*>(qb + swz128(row, (hf * 4 + u) * 16));
                w[4 * u] = v.x;
                w[4 * u + 1] = v.y;
                w[4 * u + 2] = v.z;
                w[4 * u + 3] = v.w;
              }
              tc::tmem_st16(t_lane + kColQ + 32 * bx + 16 * hf, w);
            }
          }
          tc::tmem_wait_st();
        }
        fence_proxy_async_smem();  // the staging reads come before the ring's TMA writes
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->q_moved);
      }

      const float sl = p.scale_log2;
      for (int T = 0; T < n_score && ok; ++T) {
        const int t0 = (tile_begin + 2 * T) * kTN;
        ok = warp_wait(&bars->s_full[T & 1], (T >> 1) & 1, p.err);
        if (!ok) break;
        tc::fence_after_sync();
        float sv[kTS];
        {
          uint32_t r[8][16];
          const uint32_t sc = t_lane + kColS + 128 * (T & 1);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) tc::tmem_ld16(sc + 16 * cc, r[cc]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
#pragma unroll
            for (int e = 0; e < 16; ++e) sv[16 * cc + e] = __uint_as_float(r[cc][e]);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[T & 1]);

        // ---- mask, running maximum (moved only when it rises by more than 2^8)
        const bool in_range = (t0 >= r_lo) && (t0 + kTS <= r_hi);
        const bool need_mask = !in_range || (static_cast<int64_t>(t0) + kTS - 1 > hz_min);
        if (need_mask) {
          const int c_lo = min(max(r_lo - t0, 0), kTS);
          const int c_hi = static_cast<int>(
              min(max(min(static_cast<int64_t>(r_hi), hz + 1) - t0, (int64_t)0), (int64_t)kTS));
          const unsigned span = static_cast<unsigned>(max(c_hi - c_lo, 0));
#pragma unroll
          for (int cc = 0; cc < kTS; ++cc) sv[cc] = (static_cast<unsigned>(cc - c_lo) < span) ? sv[cc] : -INFINITY;
        }
        float mx[4] = {fmaxf(sv[0], sv[4]), fmaxf(sv[1], sv[5]), fmaxf(sv[2], sv[6]), fmaxf(sv[3], sv[7])};
#pragma unroll
        for (int cc = 8; cc < kTS; cc += 8) {  // columns cc .. cc + 7
          mx[0] = fmax3(mx[0], sv[cc], sv[cc + 4]);
          mx[1] = fmax3(mx[1], sv[cc + 1], sv[cc + 5]);
          mx[2] = fmax3(mx[2], sv[cc + 2], sv[cc + 6]);
          mx[3] = fmax3(mx[3], sv[cc + 3], sv[cc + 7]);
        }
        const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl;
        float alpha = 1.f;  // factor CTA 1 applies to O before adding the first half's P V
        if ((tmax != -INFINITY) && (m_used == -INFINITY || tmax > m_used + kRescaleThreshold)) {
          const float m_new = fmaxf(m_used, tmax);
          alpha = (T > 0) ? fast_exp2(m_used - m_new) : 1.f;
          l_sum *= alpha;
          l_pv *= alpha;
          m_used = m_new;
        }
        const float base = (m_used == -INFINITY) ? 0.f : m_used;

        // ---- P of the two 64-token halves into staging slots 0 and 1 (SW128 K-major rows);
        // a slot's previous copy has landed once CTA 1 finished PV with it (half 2T - 2 + hf)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (T >= 1) {
            ok = warp_wait(&bars->p_empty[hf], (T - 1) & 1, p.err);
            if (!ok) break;
          }
          uint8_t* pst = smem + kOffPStage + hf * kPBytes;
          uint64_t ls[2] = {0ull, 0ull};  // fp32 pair sums of p (0 bits = +0.0f)
#pragma unroll
          for (int ch = 0; ch < kTN / 8; ++ch) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float p0 = fast_exp2(fmaf(sv[hf * kTN + 8 * ch + 2 * e], sl, -base));
              const float p1 = fast_exp2(fmaf(sv[hf * kTN + 8 * ch + 2 * e + 1], sl, -base));
              ls[e & 1] = add_f32x2(ls[e & 1], p0, p1);
              w[e] = pack_bf16(p0, p1);
            }
            *reinterpret_cast<uint4*>(pst + swz128(row, ch * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          l_sum += sum_f32x2(ls[0]) + sum_f32x2(ls[1]);
          float* ast = reinterpret_cast<float*>(smem + kOffAStage + hf * kRows * 4);
          ast[row] = hf == 0 ? alpha : 1.f;
          fence_proxy_async_smem();  // generic writes before the bulk copy reads them
          __syncwarp();
          if (lane == 0) {
            const uint32_t bar = hf ? peer_p_full1 : peer_p_full0;
            const uint32_t off = static_cast<uint32_t>(hf * kPBytes + lgrp * 32 * 128);
            bulk_copy_to_peer(peer_precv + off, smem_u32(smem + kOffPStage + off), 32 * 128, bar);
            const uint32_t aoff = static_cast<uint32_t>(hf * kRows * 4 + lgrp * 32 * 4);
            bulk_copy_to_peer(peer_arecv + aoff, smem_u32(smem + kOffAStage + aoff), 32 * 4, bar);
          }
          // the sum of the rounded weights, off the path to the copy: re-read the staged row
          // (the copy only reads it too; the slot is rewritten only after this PV is done)
          uint64_t lr[2] = {0ull, 0ull};
#pragma unroll
          for (int ch = 0; ch < kTN / 8; ++ch) {
            const uint4 q = *reinterpret_cast<const uint4*>(pst + swz128(row, ch * 16));
            lr[0] = add_f32x2(lr[0], bf16_lo(q.x), bf16_hi(q.x));
            lr[1] = add_f32x2(lr[1], bf16_lo(q.y), bf16_hi(q.y));
            lr[0] = add_f32x2(lr[0], bf16_lo(q.z), bf16_hi(q.z));
            lr[1] = add_f32x2(lr[1], bf16_lo(q.w), bf16_hi(q.w));
          }
          l_pv += sum_f32x2(lr[0]) + sum_f32x2(lr[1]);
        }
      }

      // ---- final row sums to CTA 1 (it normalises O); lse from here
      float* lst = reinterpret_cast<float*>(smem + kOffLStage);
      lst[row] = l_pv;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        bulk_copy_to_peer(map_to_rank(smem_u32(smem + kOffLRecv + lgrp * 32 * 4), 1), smem_u32(lst + lgrp * 32),
                          32 * 4, map_to_rank(smem_u32(&bars->l_full), 1));
      }
      constexpr float kLn2 = 0.6931471805599453f;
      const float lse = l_sum > 0.f ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
      if (valid) {
        if (x.fused) {
          x.out_lse[(static_cast<int64_t>(b) * p.Tq + t_q) * p.Hq + h] = lse;
        } else {
          const int part = j * p.n_chunk + c;
          p.out_lse[((static_cast<int64_t>(part) * p.B + b) * p.Tq + t_q) * p.Hq + h] = lse;
        }
      }
    }
  } else {
    // ================================================================ CTA 1: values
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0 && n_tiles > 0) {
        tma_prefetch_desc(PAGED ? &tml : &tmv);
        int outer = b, row_c = 0;
        int issued = 0;
        for (int i = 0; i < n_tiles; ++i) {
          const int s = i % kNStage1;
          if (i >= kNStage1 && !mbar_wait(&bars->kv_empty1[s], ((i / kNStage1) - 1) & 1, p.err, kDevErrEmptyWait))
            break;
          tile_coords<PAGED>(p, b, (tile_begin + i) * kTN, &outer, &row_c);
          mbar_arrive_expect_tx(&bars->kv_full1[s], kStage1Bytes);
          uint8_t* st = smem + s * kStage1Bytes;
          if constexpr (!PAGED) {  // the tile's eight 64-dim slices in one copy
            tma_load_4d_plain(st, &tmv, &bars->kv_full1[s], 0, row_c, 0, outer);
            // this CTA's copy engine warms L2 with a coming score tile of CTA 0 (whose own
            // engine is the busier one): the item's own tokens only
            const int pf_tok = (tile_begin + i + kPfAhead) * kTN;
            if ((i & 1) == 0 && x.kv != nullptr && pf_tok < r_hi) {
              const int n = min(kTS, r_hi - pf_tok);
              const uint8_t* src = x.kv + b * x.kv_seq_bytes + static_cast<int64_t>(pf_tok) * x.kv_tok_bytes;
              const uint32_t bytes = static_cast<uint32_t>((n - 1) * x.kv_tok_bytes + kKBoxes * 128);
              asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)),
                           "r"(bytes)
                           : "memory");
            }
          } else {
            for (int bx = 0; bx < kVBoxes; ++bx)
              tma_load_4d_plain(st + bx * kBoxBytes, &tml, &bars->kv_full1[s], bx * 64, row_c, 0, outer);
          }
          issued = i + 1;
        }
        for (int i = max(0, issued - kNStage1); i < issued; ++i) {
          if (!mbar_wait(&bars->kv_full1[i % kNStage1], (i / kNStage1) & 1, p.err, kDevErrDrainWait)) break;
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer: O += P V
      // (the whole warp runs the loop and waits; one elected lane arrives, issues, commits)
      {
        if (tc::elect_one()) mbar_arrive_expect_tx(&bars->l_full, kRows * 4);
        __syncwarp();
        const uint32_t idesc_pv = tc::idesc_f16(128, 256, true, false, true);
        const uint32_t ring = smem_u32(smem);
        const uint32_t precv = smem_u32(smem + kOffPRecv);
        static_assert((kOffBar + 1024) < (1 << 18), "descriptor start addresses (>> 4) fit 14 bits");
        bool ok = true;
        for (int i = 0; i < n_tiles && ok; ++i) {
          const int s = i % kNStage1;
          if (tc::elect_one()) mbar_arrive_expect_tx(&bars->p_full[i & 1], kPMsgBytes);
          __syncwarp();
          ok = warp_wait(&bars->kv_full1[s], (i / kNStage1) & 1, p.err);
          if (ok) ok = warp_wait(&bars->p_full[i & 1], (i >> 1) & 1, p.err);
          if (ok) ok = warp_wait(&bars->o_ready[i & 1], (i >> 1) & 1, p.err);
          if (!ok) break;
          tc::fence_after_sync();
          const uint64_t vd0 = tc::smem_desc_sw128(ring + s * kStage1Bytes, kBoxBytes, 1024);
          const uint64_t ad0 = tc::smem_desc_sw128(precv + (i & 1) * kPBytes, 16, 1024);
          if (tc::elect_one()) {
#pragma unroll
            for (int ks = 0; ks < kTN / 16; ++ks) {
              const uint64_t ad = ad0 + static_cast<uint64_t>((ks * 32) >> 4);
              const uint32_t acc = (i > 0 || ks > 0) ? 1u : 0u;
              tc::mma_f16_ss(tmem + kColO, ad, vd0 + static_cast<uint64_t>((ks * 2048) >> 4), idesc_pv, acc);
              tc::mma_f16_ss(tmem + kColO + 256, ad, vd0 + static_cast<uint64_t>((4 * kBoxBytes + ks * 2048) >> 4),
                             idesc_pv, acc);
            }
            tc::mma_commit(smem_u32(&bars->pv_done));
            tc::mma_commit(smem_u32(&bars->kv_empty1[s]));
            // CTA 0 may refill P slot i & 1 (it waits for this only when a tile i + 2 exists)
            if (i + 2 < n_tiles) mma_commit_multicast(smem_u32(&bars->p_empty[i & 1]), 0x1);
            if (i == n_tiles - 1) tc::mma_commit(smem_u32(&bars->o_final));
          }
          __syncwarp();
        }
      }
    } else {
      // ---------------------------------------------------------- row warps
      const int m = m0 + row;
      const bool valid = m < rows_total;
      const int t_q = valid ? m / p.G : 0;
      const int h = valid ? m % p.G : 0;
      const float* arecv = reinterpret_cast<const float*>(smem + kOffARecv);
      bool ok = true;
      for (int i = 0; i < n_tiles && ok; ++i) {
        const int s = i % kNStage1;
        const int t0 = (tile_begin + i) * kTN;
        ok = warp_wait(&bars->kv_full1[s], (i / kNStage1) & 1, p.err);
        if (ok) ok = warp_wait(&bars->p_full[i & 1], (i >> 1) & 1, p.err);
        if (!ok) break;
        const float alpha = arecv[(i & 1) * kRows + row];
        if (__any_sync(0xffffffffu, alpha != 1.f) && i > 0) {
          // O rows of this warp *= alpha once PV(i - 1) has completed (PV(i - 2) has: P(i)
          // was sent only after it)
          ok = warp_wait(&bars->pv_done, (i - 1) & 1, p.err);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll 1
          for (int cc = 0; cc < 512 / 16; cc += 2) {
            uint32_t r[2][16];
            tc::tmem_ld16(t_lane + kColO + 16 * cc, r[0]);
            tc::tmem_ld16(t_lane + kColO + 16 * (cc + 1), r[1]);
            tc::tmem_wait_ld();
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
              for (int e = 0; e < 16; ++e) r[h2][e] = __float_as_uint(__uint_as_float(r[h2][e]) * alpha);
            tc::tmem_st16(t_lane + kColO + 16 * cc, r[0]);
            tc::tmem_st16(t_lane + kColO + 16 * (cc + 1), r[1]);
          }
          tc::tmem_wait_st();
        }
        if (!((t0 >= r_lo) && (t0 + kTN <= r_hi))) {
          // tokens outside [r_lo, r_hi) may hold anything (NaN past the end of a sequence):
          // zero their V rows so that p = 0 contributes nothing
          if (row < kTN) {
            const int tok = t0 + row;
            if (tok < r_lo || tok >= r_hi) {
              uint8_t* vt = smem + s * kStage1Bytes;
              for (int bx = 0; bx < kVBoxes; ++bx)
                for (int q = 0; q < 8; ++q)
                  *reinterpret_cast<uint4*>(vt + bx * kBoxBytes + row * 128 + q * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_ready[i & 1]);
      }

      // ---- epilogue: O / l for all 512 dims of this CTA's rows
      if (ok && n_tiles > 0) {
        ok = warp_wait(&bars->o_final, 0, p.err);
        tc::fence_after_sync();
      }
      const bool got_l = warp_wait(&bars->l_full, 0, p.err);
      // the sum of the bf16 weights PV used (CTA 0's l_pv)
      const float l_pv = got_l ? reinterpret_cast<const float*>(smem + kOffLRecv)[row] : 0.f;
      const float inv = l_pv > 0.f ? 1.f / l_pv : 0.f;
      const bool have_o = ok && n_tiles > 0;
      constexpr int kDv = 512;
      if (x.fused) {
        __nv_bfloat16* orow =
            static_cast<__nv_bfloat16*>(x.out_bf16) + ((static_cast<int64_t>(b) * p.Tq + t_q) * p.Hq + h) * kDv;
#pragma unroll 1
        for (int cc = 0; cc < kDv / 16; ++cc) {
          uint32_t r[16];
          if (have_o) {
            tc::tmem_ld16(t_lane + kColO + 16 * cc, r);
            tc::tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = 0u;
          }
          if (valid) {
            uint4 w0, w1;
            w0.x = pack_bf16(__uint_as_float(r[0]) * inv, __uint_as_float(r[1]) * inv);
            w0.y = pack_bf16(__uint_as_float(r[2]) * inv, __uint_as_float(r[3]) * inv);
            w0.z = pack_bf16(__uint_as_float(r[4]) * inv, __uint_as_float(r[5]) * inv);
            w0.w = pack_bf16(__uint_as_float(r[6]) * inv, __uint_as_float(r[7]) * inv);
            w1.x = pack_bf16(__uint_as_float(r[8]) * inv, __uint_as_float(r[9]) * inv);
            w1.y = pack_bf16(__uint_as_float(r[10]) * inv, __uint_as_float(r[11]) * inv);
            w1.z = pack_bf16(__uint_as_float(r[12]) * inv, __uint_as_float(r[13]) * inv);
            w1.w = pack_bf16(__uint_as_float(r[14]) * inv, __uint_as_float(r[15]) * inv);
            *reinterpret_cast<uint4*>(orow + 16 * cc) = w0;
            *reinterpret_cast<uint4*>(orow + 16 * cc + 8) = w1;
          }
        }
      } else {
        // fp32 partial rows (2 KB each): staged through the ring's bytes (free once the last PV
        // has completed and every load has landed) and written by one bulk copy per half row,
        // so global memory sees whole contiguous rows rather than 16-byte pieces of 32 rows
        // per store instruction.  Row pitch 1040 B keeps the staging stores conflict-free.
        const int part = j * p.n_chunk + c;
        const int64_t ro = ((static_cast<int64_t>(part) * p.B + b) * p.Tq + t_q) * p.Hq + h;
        float* orow = p.out_o + ro * kDv;
        const bool write_o = valid && (l_pv > 0.f || p.zero_empty);
        constexpr int kHalf = kDv / 2;              // 256 floats, 1 KB
        constexpr uint32_t kPitch = kHalf * 4 + 16;  // staging row pitch
        static_assert(kRows * kPitch <= kNStage1 * kStage1Bytes, "staging fits in the ring bytes");
        float* stage = reinterpret_cast<float*>(smem + row * kPitch);
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          if (half == 1 && write_o) bulk_wait_read();  // the first half's copy has read the row
#pragma unroll 1
          for (int c4 = 0; c4 < kHalf / 64; ++c4) {  // four 16-column loads per TMEM wait
            uint32_t r[4][16];
            if (have_o) {
#pragma unroll
              for (int u = 0; u < 4; ++u) tc::tmem_ld16(t_lane + kColO + half * kHalf + 64 * c4 + 16 * u, r[u]);
              tc::tmem_wait_ld();
            } else {
#pragma unroll
              for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int e = 0; e < 16; ++e) r[u][e] = 0u;
            }
            if (write_o) {
#pragma unroll
              for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                  *reinterpret_cast<float4*>(stage + 64 * c4 + 16 * u + e) =
                      make_float4(__uint_as_float(r[u][e]) * inv, __uint_as_float(r[u][e + 1]) * inv,
                                  __uint_as_float(r[u][e + 2]) * inv, __uint_as_float(r[u][e + 3]) * inv);
            }
          }
          if (write_o) {
            fence_proxy_async_smem();  // the staging writes before the bulk copy reads them
            bulk_store_global(orow + half * kHalf, smem_u32(stage), kHalf * 4);
          }
        }
        if (write_o) bulk_wait_all();
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();  // no copy or remote arrive into the peer is still pending
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

int mla_tc_rows_per_item() { return kRows; }
int mla_tc_kv_tile() { return kTN; }
int mla_tc_score_tile() { return kTS; }
int mla_tc_group_slices() { return kGrp; }

cudaError_t launch_mla_tc(const PartialParams& p, const TcAttnExtra& x, const CUtensorMap& tmq,
                          const CUtensorMap& tml, const CUtensorMap& tmg, const CUtensorMap& tmv, int64_t n_items,
                          cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e0 = once_per_device(attr_done, [] {
    cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mla_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    return e;
  });
  if (e0 != cudaSuccess) return e0;
  if (n_items <= 0) return cudaSuccess;
  if (p.block_table)
    mla_tc_kernel<true><<<static_cast<unsigned int>(2 * n_items), kThreads, kSmem, stream>>>(p, x, tmq, tml, tmg, tmv);
  else
    mla_tc_kernel<false><<<static_cast<unsigned int>(2 * n_items), kThreads, kSmem, stream>>>(p, x, tmq, tml, tmg, tmv);
  return cudaGetLastError();
}

}  // namespace skv
