// Tensor-core (tcgen05) split-KV attention for query tiles of 128+ rows: the ring
// pass-KV prefill chunk and any GQA call with Tq * G >= 128 rows per KV head.
//
// What it computes: for each row (query row t, query head h of KV head g), exact softmax
// attention over the visible tokens of a range, as a normalised output plus its
// natural-log LSE -- per split ("Context Parallelism for Scalable Million-Token
// Inference", section "Pass-KV keeps queries local and circulates keys and values": each
// ring step's partial attention keeps a log-sum-exp), or over the union of all splits
// at once, which equals their exact LSE merge (the same page's merge equation: the online
// softmax below performs that merge tile by tile).  Causal visibility is by original
// position ("现代大模型推理并行策略总览", section "序列布局"): row t sees token p iff
// p <= causal_offset + t.
//
// GB300 design (one CTA per SM):
//   * a CTA owns 256 rows = two 128-row query tiles of one KV head; rows are (query row,
//     head) pairs, so a K/V tile read once serves the whole GQA group and both tiles;
//   * warp 0: TMA producer (Q tiles once, 128-token K/V tiles into a 2-stage ring);
//     warp 1: allocates 512 TMEM columns and issues every tcgen05.mma from one thread;
//     warps 2-5 and 6-9: softmax for query tile 0 and 1, one thread per row (the TMEM lane
//     of its row), so row max / sum need no shuffles;
//   * TMEM: S0 | S1 (128 x 128 fp32 each) | O0 | O1 (128 x 128 fp32 each); P (bf16) is
//     written over the first 64 columns of its S and read from TMEM as the A operand of
//     P V, so P never touches shared memory;
//   * MMA order per KV tile: PV0(i), S0(i+1), PV1(i), S1(i+1), so each softmax group works
//     while the tensor core serves the other group.  MMAs from one thread run in order, so
//     when S_k(i) has landed, PV_k(i-1) is complete: O_k may be rescaled and P_k rewritten;
//   * optimistic softmax: p = 2^(s - m_used) against the running max; O is rescaled (TMEM
//     load / scale / store) and the tile redone only on a row's first visible tile or when
//     the tile's p sum exceeds 2^16 (a score rose far above m_used), so no max is taken on
//     the common path and every p stays <= 2^16, fine for bf16 P and the fp32 sums.
#include <climits>
#include <cuda_runtime.h>

#include <type_traits>

#include "skv_common.cuh"
#include "skv_internal.h"
#include "tc_common.cuh"

namespace skv {

namespace {

// The softmax pass's mask mode, a compile-time flag (std::true_type / std::false_type): the
// unmasked instantiation has no test in its unrolled column loop.
template <bool B>
__device__ __forceinline__ constexpr bool mask_on(std::integral_constant<bool, B>) {
  return B;
}

constexpr int kD = 128;         // dk = dv
constexpr int kTN = 128;        // tokens per K/V tile
constexpr int kNStage = 2;      // K/V ring depth
constexpr int kRowsTile = 128;  // rows per query tile (MMA M)
constexpr int kThreads = 10 * 32;
constexpr int kQTileBytes = kRowsTile * kD * 2;  // 32 KB (two 16 KB boxes)
constexpr int kKVBoxBytes = kTN * 128;           // 16 KB: 128 tokens x 64 dims
constexpr int kKTileBytes = 2 * kKVBoxBytes;     // 32 KB
constexpr int kStageBytes = 2 * kKTileBytes;     // K + V
constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + 2 * kQTileBytes;
constexpr int kOffBar = kOffRing + kNStage * kStageBytes;
// position mode: the item's tiles that some row can see, listed once per CTA
constexpr int kMaxListTiles = 1024;  // items with more tiles keep every tile
constexpr int kOffList = kOffBar + 256;                  // int32 tile index [kMaxListTiles]
constexpr int kOffKmin = kOffList + 4 * kMaxListTiles;   // int32 min position of a tile's tokens
constexpr int kOffKmax = kOffKmin + 4 * kMaxListTiles;   // int32 max position
constexpr int kOffMisc = kOffKmax + 4 * kMaxListTiles;   // [0] the CTA's largest row position, [1] tiles kept
constexpr int kSmem = 1024 + kOffMisc + 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S_k (and P_k over its first 64 columns) at kColS + 128 k
constexpr uint32_t kColO = 256;  // O_k at kColO + 128 k
// The optimistic softmax redoes a tile (new running max, O and l rescaled) only when the
// tile's p sum exceeds this: then every p <= 2^16, fine for bf16 P and the fp32 sums.
constexpr float kTileSumLimit = 65536.0f;
static_assert(kSmem <= 227 * 1024, "shared memory budget");

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[kNStage];
  uint64_t kv_empty[kNStage];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint32_t tmem_base;
};

__device__ __forceinline__ void tma_load_4d_nohint(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                                   int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}


// POS: the causal rule comes from position arrays (tokens stored out of sequence order)
// PAGED: K/V live in pages with a block table (read in 64-token halves)
template <bool POS, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
    tc_attn_kernel(const __grid_constant__ PartialParams p, const __grid_constant__ TcAttnExtra x,
                   const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: (b, g, [split j,] 256-row tile mt)
  // Row tiles are handed out last-first across all (b, g, split): a causal chunk's later
  // rows see more keys, so the heaviest CTAs start first and the last wave is light.
  int64_t item = blockIdx.x;
  const int64_t per_tile = static_cast<int64_t>(p.B) * p.Hkv * (x.fused ? 1 : p.n_split);
  const int mt = p.m_tiles - 1 - static_cast<int>(item / per_tile);
  item %= per_tile;
  int j = 0;
  if (!x.fused) {
    j = static_cast<int>(item % p.n_split);
    item /= p.n_split;
  }
  const int g = static_cast<int>(item % p.Hkv);
  const int b = static_cast<int>(item / p.Hkv);
  const int G = p.G;
  const int seq_len = p.seq_lens[b];
  int lo, hi;
  split_range(p, b, x.fused ? 0 : j, x.fused ? p.n_split : j + 1, seq_len, &lo, &hi);
  const int rows_total = p.Tq * G;
  const int m0 = mt * 2 * kRowsTile;
  const int m_last = min(m0 + 2 * kRowsTile, rows_total) - 1;
  {
    const int64_t horizon = p.causal_offset + m_last / G;
    if (horizon < static_cast<int64_t>(hi) - 1) hi = static_cast<int>(max(horizon + 1, (int64_t)lo));
  }
  const int r_lo = lo, r_hi = hi;
  const int tile_begin = r_lo / kTN;
  const int n_tiles = (r_hi > r_lo) ? ((r_hi + kTN - 1) / kTN - tile_begin) : 0;

  // ---- position mode: list the tiles holding a token some row of this CTA can see.
  // Every role walks the same list, so a tile that no row sees is never loaded, multiplied
  // or masked; stages and barrier phases follow the position in the list.
  int n_used = n_tiles;
  bool listed = false;
  const int* lidx = reinterpret_cast<const int*>(smem + kOffList);
  const int* lkmin = reinterpret_cast<const int*>(smem + kOffKmin);
  const int* lkmax = reinterpret_cast<const int*>(smem + kOffKmax);
  if constexpr (POS) {
    int* misc = reinterpret_cast<int*>(smem + kOffMisc);
    listed = n_tiles <= kMaxListTiles;
    if (threadIdx.x == 0) misc[0] = INT_MIN;
    __syncthreads();
    int qm = INT_MIN;  // largest position of the CTA's query rows
    for (int t = m0 / G + static_cast<int>(threadIdx.x); t <= m_last / G; t += kThreads)
      qm = max(qm, __ldg(p.q_pos + b * p.Tq + t));
    qm = __reduce_max_sync(0xffffffffu, qm);
    if (lane == 0) atomicMax(&misc[0], qm);
    if (listed) {
      int* kmin_w = reinterpret_cast<int*>(smem + kOffKmin);
      int* kmax_w = reinterpret_cast<int*>(smem + kOffKmax);
      for (int i = warp; i < n_tiles; i += kThreads / 32) {
        const int t = (tile_begin + i) * kTN + 4 * lane;
        // S_max and t are multiples of 4: the four positions exist together or not at all
        const int4 kp = (t < p.S_max) ? __ldg(reinterpret_cast<const int4*>(p.k_pos + static_cast<int64_t>(b) * p.S_max + t))
                                      : make_int4(0, 0, 0, 0);
        int mn = INT_MAX, mx = INT_MIN;
        const int v4[4] = {kp.x, kp.y, kp.z, kp.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (t + u >= r_lo && t + u < r_hi) {  // only tokens of the item's range count
            mn = min(mn, v4[u]);
            mx = max(mx, v4[u]);
          }
        }
        mn = __reduce_min_sync(0xffffffffu, mn);
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (lane == 0) {
          kmin_w[i] = mn;
          kmax_w[i] = mx;
        }
      }
    }
    __syncthreads();
    if (listed && warp == 0) {
      const int qmax_cta = misc[0];
      int* lidx_w = reinterpret_cast<int*>(smem + kOffList);
      int c = 0;
      for (int base = 0; base < n_tiles; base += 32) {
        const int i = base + lane;
        const bool keep = i < n_tiles && lkmin[i] <= qmax_cta;
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (keep) lidx_w[c + __popc(bal & ((1u << lane) - 1u))] = i;
        c += __popc(bal);
      }
      if (lane == 0) misc[1] = c;
    }
    __syncthreads();
    if (listed) n_used = misc[1];
  }
  auto tile_of = [&](int c) -> int {
    if constexpr (POS) return listed ? lidx[c] : c;
    return c;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kNStage; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars->s_full[k], 1);
      mbar_init(&bars->p_full[k], kRowsTile);
      mbar_init(&bars->pv_done[k], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_used > 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      mbar_arrive_expect_tx(&bars->q_full, 2 * kQTileBytes);
      for (int k = 0; k < 2; ++k) {
        const int t_start = (m0 + k * kRowsTile) / G;
        for (int bx = 0; bx < 2; ++bx)
          tma_load_4d_nohint(smem + kOffQ + k * kQTileBytes + bx * (kQTileBytes / 2), &tmq, &bars->q_full, bx * 64,
                             g * G, t_start, b);
      }
      // a paged cache is read in 64-token halves (a page holds a multiple of 64 tokens),
      // each half's page read one tile ahead, behind the stage wait
      // (a half that starts at or past S_max only holds masked tokens: it reuses the first
      // half's page instead of reading past the sequence's block-table row)
      auto pages_of = [&](int t, int& a, int& c) {
        a = kv_page_of(p, b, t);
        c = (t + kTN / 2 < p.S_max) ? kv_page_of(p, b, t + kTN / 2) : a;
      };
      int pg0 = 0, pg1 = 0;
      if constexpr (PAGED) pages_of((tile_begin + tile_of(0)) * kTN, pg0, pg1);
      int issued = 0;
      for (int i = 0; i < n_used; ++i) {
        const int s = i % kNStage;
        if (i >= kNStage && !mbar_wait(&bars->kv_empty[s], ((i / kNStage) - 1) & 1, p.err, kDevErrEmptyWait)) break;
        mbar_arrive_expect_tx(&bars->kv_full[s], kStageBytes);
        uint8_t* st = smem + kOffRing + s * kStageBytes;
        const int tok = (tile_begin + tile_of(i)) * kTN;
        if constexpr (!PAGED) {
          for (int bx = 0; bx < 2; ++bx) {
            tma_load_4d_nohint(st + bx * kKVBoxBytes, &tmk, &bars->kv_full[s], bx * 64, tok, g, b);
            tma_load_4d_nohint(st + kKTileBytes + bx * kKVBoxBytes, &tmv, &bars->kv_full[s], bx * 64, tok, g, b);
          }
        } else {
          const int cur[2] = {pg0, pg1};
          if (i + 1 < n_used) pages_of((tile_begin + tile_of(i + 1)) * kTN, pg0, pg1);
          for (int hf = 0; hf < 2; ++hf) {
            const int row = (tok + hf * (kTN / 2)) % p.block_len;
            for (int bx = 0; bx < 2; ++bx) {
              const int off = bx * kKVBoxBytes + hf * (kKVBoxBytes / 2);  // rows 64 hf.. of box bx
              tma_load_4d_nohint(st + off, &tmk, &bars->kv_full[s], bx * 64, row, g, cur[hf]);
              tma_load_4d_nohint(st + kKTileBytes + off, &tmv, &bars->kv_full[s], bx * 64, row, g, cur[hf]);
            }
          }
        }
        issued = i + 1;
      }
      for (int i = max(0, issued - kNStage); i < issued; ++i) {
        if (!mbar_wait(&bars->kv_full[i % kNStage], (i / kNStage) & 1, p.err, kDevErrDrainWait)) break;
      }
      mbar_wait(&bars->q_full, 0, p.err, kDevErrDrainWait);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and waits; one elected lane issues the MMAs and commits
    // (a lone lane-0 loop pays about twice as much per wait and more per MMA).
    if (n_used > 0) {
      const uint32_t idesc_s = tc::idesc_f16(128, kTN, true, false, false);
      const uint32_t idesc_pv = tc::idesc_f16(128, kD, true, false, true);
      const uint32_t q_base = smem_u32(smem + kOffQ);
      const uint32_t ring = smem_u32(smem + kOffRing);
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.err, kDevErrFullWait));
      };
      bool ok = wait_all(&bars->q_full, 0);
      // Every MMA operand is a compile-time offset from per-CTA descriptor bases: the loop
      // over K/V tiles is unrolled by the ring depth, so a tile's stage is a constant too
      // (a stage index computed at run time raised each MMA's issue cost by a half).
      const uint64_t qd_base = tc::smem_desc_sw128(q_base, 16, 1024);
      const uint64_t kd_base = tc::smem_desc_sw128(ring, 16, 1024);
      const uint64_t vd_base = tc::smem_desc_sw128(ring + kKTileBytes, kKVBoxBytes, 1024);
      auto issue_s = [&](int k, int stage) {  // S_k = Q_k K^T  (M 128, N 128 tokens, K 128)
        const uint32_t d = tmem + kColS + 128 * k;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint64_t ad =
              qd_base + static_cast<uint64_t>((k * kQTileBytes + (ks >> 2) * (kQTileBytes / 2) + (ks & 3) * 32) >> 4);
          const uint64_t bd =
              kd_base + static_cast<uint64_t>((stage * kStageBytes + (ks >> 2) * kKVBoxBytes + (ks & 3) * 32) >> 4);
          tc::mma_f16_ss(d, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int k, int stage, uint32_t acc0) {  // O_k += P_k V  (M 128, N 128, K 128; P_k from TMEM)
        const uint32_t d = tmem + kColO + 128 * k;
        const uint32_t a = tmem + kColS + 128 * k;
#pragma unroll
        for (int ks = 0; ks < kTN / 16; ++ks) {
          tc::mma_f16_ts(d, a + ks * 8, vd_base + static_cast<uint64_t>((stage * kStageBytes + ks * 2048) >> 4),
                         idesc_pv, ks > 0 ? 1u : acc0);
        }
      };
      // one K/V tile i in stage ST (= i % kNStage): PV0(i), S0(i+1), PV1(i), S1(i+1)
      auto tile = [&](auto stage_c, int i) {
        constexpr int ST = decltype(stage_c)::value;
        constexpr int NX = (ST + 1) % kNStage;
        ok = wait_all(&bars->p_full[0], i & 1);
        if (!ok) return;
        tc::fence_after_sync();
        if (tc::elect_one()) {
          issue_pv(0, ST, i > 0 ? 1u : 0u);
          tc::mma_commit(smem_u32(&bars->pv_done[0]));
        }
        __syncwarp();
        if (i + 1 < n_used) {
          ok = wait_all(&bars->kv_full[NX], ((i + 1) / kNStage) & 1);
          if (!ok) return;
          tc::fence_after_sync();
          if (tc::elect_one()) {
            issue_s(0, NX);
            tc::mma_commit(smem_u32(&bars->s_full[0]));
          }
          __syncwarp();
        }
        ok = wait_all(&bars->p_full[1], i & 1);
        if (!ok) return;
        tc::fence_after_sync();
        if (tc::elect_one()) {
          issue_pv(1, ST, i > 0 ? 1u : 0u);
          tc::mma_commit(smem_u32(&bars->pv_done[1]));
          tc::mma_commit(smem_u32(&bars->kv_empty[ST]));
          if (i + 1 < n_used) {
            issue_s(1, NX);
            tc::mma_commit(smem_u32(&bars->s_full[1]));
          }
        }
        __syncwarp();
      };
      static_assert(kNStage == 2, "the tile loop is unrolled by the ring depth");
      if (ok) ok = wait_all(&bars->kv_full[0], 0);
      if (ok) {
        tc::fence_after_sync();
        if (tc::elect_one()) {
          issue_s(0, 0);
          tc::mma_commit(smem_u32(&bars->s_full[0]));
          issue_s(1, 0);
          tc::mma_commit(smem_u32(&bars->s_full[1]));
        }
        __syncwarp();
        for (int i = 0; i < n_used && ok; i += 2) {
          tile(std::integral_constant<int, 0>{}, i);
          if (ok && i + 1 < n_used) tile(std::integral_constant<int, 1>{}, i + 1);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax groups
    const int k = (warp - 2) >> 2;                 // query tile 0 or 1
    const int lgrp = warp & 3;                     // TMEM lane group of this warp
    const int row = lgrp * 32 + lane;              // row inside the query tile
    const int m = m0 + k * kRowsTile + row;        // row of KV head g's row space
    const bool valid = m < rows_total;
    const int t_q = valid ? m / G : 0;
    const int h = g * G + (valid ? m % G : 0);
    const int64_t hz = p.causal_offset + t_q;
    const int64_t hz_min = p.causal_offset + (m0 + k * kRowsTile + lgrp * 32) / G;  // smallest in this warp
    // tokens stored out of sequence order: column t is visible iff k_pos[t] <= q_pos[row]
    const int32_t* kpos_b = POS ? p.k_pos + static_cast<int64_t>(b) * p.S_max : nullptr;
    const int qp = (POS && valid) ? __ldg(p.q_pos + b * p.Tq + t_q) : 0;
    // position range of this warp's rows: a listed tile entirely at or below it needs no
    // mask, one entirely above it is invisible to the warp
    int qmin_w = INT_MAX, qmax_w = INT_MIN;
    if constexpr (POS) {
      qmin_w = __reduce_min_sync(0xffffffffu, valid ? qp : INT_MAX);
      qmax_w = __reduce_max_sync(0xffffffffu, valid ? qp : INT_MIN);
    }
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(lgrp * 32) << 16);
    // l_sum: the fp32 row sum (for the lse); l_pv: the sum of the bf16-rounded p that PV
    // uses (for normalising O: the output is then an exact convex combination of V rows with
    // those weights; with the optimistic max no p is exact, and normalising by the fp32 sum
    // left up to ~2^-8 max|v| of error in a split of a few tokens)
    float m_used = -INFINITY, l_sum = 0.f, l_pv = 0.f;
    bool ok = true;

    for (int i = 0; i < n_used && ok; ++i) {
      const int ti = tile_of(i);  // the tile; i is its place in the (listed) sequence
      const int t0 = (tile_begin + ti) * kTN;
      ok = mbar_wait(&bars->s_full[k], i & 1, p.err, kDevErrFullWait);
      if (!ok) break;
      tc::fence_after_sync();
      const bool in_range = (t0 >= r_lo) && (t0 + kTN <= r_hi);
      bool need_mask = !in_range || (static_cast<int64_t>(t0) + kTN - 1 > hz_min);
      bool none_visible = false;
      if constexpr (POS) {
        need_mask = !(listed && in_range && lkmax[ti] <= qmin_w);
        none_visible = listed && lkmin[ti] > qmax_w;
      }
      // visible columns of this row: [c_lo, c_lo + span)
      const int c_lo = min(max(r_lo - t0, 0), kTN);
      const int c_hi = static_cast<int>(
          min(max(min(static_cast<int64_t>(r_hi), hz + 1) - t0, (int64_t)0), (int64_t)kTN));
      const unsigned span = static_cast<unsigned>(max(c_hi - c_lo, 0));
      // position mode: bit c of vis[c / 32] = column c visible (in range and k_pos <= q_pos);
      // the tile's positions are the same for every lane (L1 broadcast)
      uint32_t vis[kTN / 32] = {0u, 0u, 0u, 0u};
      if constexpr (POS) {
        if (need_mask && !none_visible) {
#pragma unroll
        for (int w4 = 0; w4 < kTN / 32; ++w4) {
          uint32_t bits = 0u;
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const int col = 32 * w4 + 4 * q4;
            // S_max and t0 are multiples of 4: the four positions exist together or not at all
            const int4 kp = (t0 + col < p.S_max) ? __ldg(reinterpret_cast<const int4*>(kpos_b + t0 + col))
                                                 : make_int4(INT_MAX, INT_MAX, INT_MAX, INT_MAX);
            bits |= static_cast<uint32_t>(kp.x <= qp && static_cast<unsigned>(col - c_lo) < span) << (4 * q4);
            bits |= static_cast<uint32_t>(kp.y <= qp && static_cast<unsigned>(col + 1 - c_lo) < span) << (4 * q4 + 1);
            bits |= static_cast<uint32_t>(kp.z <= qp && static_cast<unsigned>(col + 2 - c_lo) < span) << (4 * q4 + 2);
            bits |= static_cast<uint32_t>(kp.w <= qp && static_cast<unsigned>(col + 3 - c_lo) < span) << (4 * q4 + 3);
          }
          vis[w4] = bits;
        }
        }
      }
      auto visible = [&](int col) -> bool {
        if constexpr (POS) return ((vis[col >> 5] >> (col & 31)) & 1u) != 0u;
        return static_cast<unsigned>(col - c_lo) < span;
      };
      const uint32_t s_col = t_lane + kColS + 128 * k;
      const float sl = p.scale_log2;

      // Optimistic pass: p = 2^(scale*s - m_used) with the running max; P stays packed in
      // registers until the tile's sum shows it is fine (no max is taken here: the redo
      // below finds it when needed).
      uint32_t pk[kTN / 2];
      uint64_t ls[2] = {0ull, 0ull};  // fp32 pair sums of p (0 bits = +0.0f)
      uint64_t lr[2] = {0ull, 0ull};  // the same of the bf16-rounded p
      const float base0 = (m_used == -INFINITY) ? 0.f : m_used;
      // masked: a compile-time constant, one instantiation per mask mode (need_mask is warp-
      // uniform), so that the tiles away from the diagonal and the split ends -- nearly all of
      // them -- carry no per-column visibility test (in position mode the two copies spill a
      // few registers and are still faster)
      auto pass = [&](auto masked) {
#pragma unroll
        for (int cc = 0; cc < kTN / 32; ++cc) {
          uint32_t r[2][16];
          tc::tmem_ld16(s_col + 32 * cc, r[0]);
          tc::tmem_ld16(s_col + 32 * cc + 16, r[1]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int col = 32 * cc + 2 * e;
            float v0 = __uint_as_float(r[e >> 3][(2 * e) & 15]);
            float v1 = __uint_as_float(r[e >> 3][(2 * e + 1) & 15]);
            if (mask_on(masked)) {
              v0 = visible(col) ? v0 : -INFINITY;
              v1 = visible(col + 1) ? v1 : -INFINITY;
            }
            // pairwise: one packed FMA and packed adds per column pair
            float a0, a1;
            fma_pair(v0, v1, sl, -base0, a0, a1);
            const float p0 = fast_exp2(a0);
            const float p1 = fast_exp2(a1);
            ls[e & 1] = add_f32x2(ls[e & 1], p0, p1);
            pk[16 * cc + e] = pack_bf16(p0, p1);
            lr[e & 1] = add_bf16x2_f32x2(lr[e & 1], pk[16 * cc + e]);
          }
        }
      };
      if (need_mask)
        pass(std::true_type{});
      else
        pass(std::false_type{});
      // Redo when this is the row's first visible tile, or when its p grew past the limit
      // (then some score rose far above m_used; every p <= the tile sum <= 2^16 otherwise).
      const float tile_sum = sum_f32x2(ls[0]) + sum_f32x2(ls[1]);
      bool row_vis = true;  // the row sees some column of this tile
      if (need_mask) {
        if constexpr (POS)
          row_vis = (vis[0] | vis[1] | vis[2] | vis[3]) != 0u;
        else
          row_vis = span > 0u;
      }
      const bool need = row_vis && (m_used == -INFINITY || !(tile_sum <= kTileSumLimit));
      if (__any_sync(0xffffffffu, need)) {
        // rare: rescale O and l to the tile's true max and redo this tile's P from S (still
        // in TMEM); the max comes from one pass over S (every lane of the warp takes part)
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int cc = 0; cc < kTN / 32; ++cc) {
          uint32_t r[2][16];
          tc::tmem_ld16(s_col + 32 * cc, r[0]);
          tc::tmem_ld16(s_col + 32 * cc + 16, r[1]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int col = 32 * cc + 2 * e;
            float v0 = __uint_as_float(r[e >> 3][(2 * e) & 15]);
            float v1 = __uint_as_float(r[e >> 3][(2 * e + 1) & 15]);
            if (need_mask) {
              v0 = visible(col) ? v0 : -INFINITY;
              v1 = visible(col + 1) ? v1 : -INFINITY;
            }
            mx[e & 3] = fmax3(mx[e & 3], v0, v1);
          }
        }
        // scores are scaled after the max (the scale is positive)
        const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl;
        const float m_new = need ? fmaxf(m_used, tmax) : m_used;
        if (i > 0) {
          // PV_k(i-1) ran before S_k(i) on the in-order tensor pipe, so O_k is final here
          const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < kD / 16; c += 2) {
            uint32_t r[2][16];
            tc::tmem_ld16(t_lane + kColO + 128 * k + 16 * c, r[0]);
            tc::tmem_ld16(t_lane + kColO + 128 * k + 16 * (c + 1), r[1]);
            tc::tmem_wait_ld();
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
              for (int e = 0; e < 16; ++e) r[h2][e] = __float_as_uint(__uint_as_float(r[h2][e]) * alpha);
            tc::tmem_st16(t_lane + kColO + 128 * k + 16 * c, r[0]);
            tc::tmem_st16(t_lane + kColO + 128 * k + 16 * (c + 1), r[1]);
          }
          tc::tmem_wait_st();
          l_sum *= alpha;
          l_pv *= alpha;
        } else {
          l_sum = 0.f;
          l_pv = 0.f;
        }
        m_used = m_new;
        const float base = (m_used == -INFINITY) ? 0.f : m_used;
        ls[0] = ls[1] = 0ull;
        lr[0] = lr[1] = 0ull;
#pragma unroll 1
        for (int cc = 0; cc < kTN / 32; ++cc) {
          uint32_t r[2][16];
          tc::tmem_ld16(s_col + 32 * cc, r[0]);
          tc::tmem_ld16(s_col + 32 * cc + 16, r[1]);
          tc::tmem_wait_ld();
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int col = 32 * cc + 2 * e;
            float v0 = __uint_as_float(r[e >> 3][(2 * e) & 15]);
            float v1 = __uint_as_float(r[e >> 3][(2 * e + 1) & 15]);
            if (need_mask) {
              v0 = visible(col) ? v0 : -INFINITY;
              v1 = visible(col + 1) ? v1 : -INFINITY;
            }
            const float p0 = fast_exp2(fmaf(v0, sl, -base));
            const float p1 = fast_exp2(fmaf(v1, sl, -base));
            ls[e & 1] = add_f32x2(ls[e & 1], p0, p1);
            w[e] = pack_bf16(p0, p1);
            lr[e & 1] = add_bf16x2_f32x2(lr[e & 1], w[e]);
          }
          tc::tmem_st16(s_col + 16 * cc, w);  // S columns 32cc.. were read before P 16cc.. is written
        }
      } else {
        // common case: the optimistic P is exact; S is fully read, so P may overwrite it
#pragma unroll
        for (int cc = 0; cc < kTN / 32; ++cc) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = pk[16 * cc + e];
          tc::tmem_st16(s_col + 16 * cc, w);
        }
      }
      tc::tmem_wait_st();
      l_sum += sum_f32x2(ls[0]) + sum_f32x2(ls[1]);
      l_pv += sum_f32x2(lr[0]) + sum_f32x2(lr[1]);
      if (k == 0 && !in_range) {
        // tokens outside [r_lo, r_hi) may hold anything (NaN past the end of a sequence):
        // zero their V rows so that p = 0 really contributes nothing
        const int tid = lgrp * 32 + lane;
        const int s_idx = i % kNStage;
        mbar_wait(&bars->kv_full[s_idx], (i / kNStage) & 1, p.err, kDevErrFullWait);
        if (tid < kTN) {
          const int tok = t0 + tid;
          if (tok < r_lo || tok >= r_hi) {
            uint8_t* vt = smem + kOffRing + s_idx * kStageBytes + kKTileBytes;
            for (int bx = 0; bx < 2; ++bx)
              for (int cc = 0; cc < 8; ++cc)
                *reinterpret_cast<uint4*>(vt + bx * kKVBoxBytes + tid * 128 + cc * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
      }
      tc::fence_before_sync();
      mbar_arrive(&bars->p_full[k]);
    }

    // ---- epilogue: O / l and lse
    if (n_used > 0 && ok) {
      ok = mbar_wait(&bars->pv_done[k], (n_used - 1) & 1, p.err, kDevErrFullWait);
      tc::fence_after_sync();
    }
    const float inv = l_pv > 0.f ? 1.f / l_pv : 0.f;
    constexpr float kLn2 = 0.6931471805599453f;
    const float lse = l_sum > 0.f ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
    if (x.fused) {
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(x.out_bf16) +
                            ((static_cast<int64_t>(b) * p.Tq + t_q) * p.Hq + h) * kD;
#pragma unroll 2
      for (int c = 0; c < kD / 16; ++c) {
        uint32_t r[16];
        if (n_used > 0) {
          tc::tmem_ld16(t_lane + kColO + 128 * k + 16 * c, r);
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
          *reinterpret_cast<uint4*>(orow + 16 * c) = w0;
          *reinterpret_cast<uint4*>(orow + 16 * c + 8) = w1;
        }
      }
      if (valid) x.out_lse[(static_cast<int64_t>(b) * p.Tq + t_q) * p.Hq + h] = lse;
    } else {
      const int64_t ro = ((static_cast<int64_t>(j) * p.B + b) * p.Tq + t_q) * p.Hq + h;
      float* orow = p.out_o + ro * kD;
      bool write_o = valid && (l_sum > 0.f || p.zero_empty);
      // accumulate: o <- (w_acc o_acc + w o / l) / (w_acc + w) with w_x = e^{lse_x - max},
      // the exact two-way merge; a row this item saw nothing of keeps its running value
      float a_acc = 0.f, a_new = inv;
      float lse_out = lse;
      if (x.accumulate) {
        const float lse_acc = valid ? p.out_lse[ro] : -INFINITY;
        const float mx = fmaxf(lse_acc, lse);
        write_o = valid && l_sum > 0.f;
        if (write_o) {
          const float wa = (lse_acc == -INFINITY) ? 0.f : __expf(lse_acc - mx);
          const float wb = __expf(lse - mx);
          const float den = 1.f / (wa + wb);
          a_acc = wa * den;
          a_new = wb * den * inv;
          lse_out = mx + logf(wa + wb);
        }
      }
#pragma unroll 1
      for (int c = 0; c < kD / 16; ++c) {
        uint32_t r[16];
        if (n_used > 0) {
          tc::tmem_ld16(t_lane + kColO + 128 * k + 16 * c, r);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = 0u;
        }
        if (write_o) {
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            float4 v = make_float4(__uint_as_float(r[e]) * a_new, __uint_as_float(r[e + 1]) * a_new,
                                   __uint_as_float(r[e + 2]) * a_new, __uint_as_float(r[e + 3]) * a_new);
            if (a_acc != 0.f) {
              const float4 o0 = *reinterpret_cast<const float4*>(orow + 16 * c + e);
              v.x += a_acc * o0.x;
              v.y += a_acc * o0.y;
              v.z += a_acc * o0.z;
              v.w += a_acc * o0.w;
            }
            *reinterpret_cast<float4*>(orow + 16 * c + e) = v;
          }
        }
      }
      if (valid && (!x.accumulate || write_o)) p.out_lse[ro] = lse_out;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

int tc_attn_rows_per_cta() { return 2 * kRowsTile; }
int tc_attn_kv_tile() { return kTN; }

cudaError_t launch_tc_attn(const PartialParams& p, const TcAttnExtra& x, const CUtensorMap& tmq,
                           const CUtensorMap& tmk, const CUtensorMap& tmv, int64_t n_items, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e0 = once_per_device(attr_done, [] {
    cudaError_t e = cudaFuncSetAttribute(tc_attn_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tc_attn_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tc_attn_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tc_attn_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    return e;
  });
  if (e0 != cudaSuccess) return e0;
  if (n_items <= 0) return cudaSuccess;
  const unsigned int grid = static_cast<unsigned int>(n_items);
  if (p.k_pos && p.block_table)
    tc_attn_kernel<true, true><<<grid, kThreads, kSmem, stream>>>(p, x, tmq, tmk, tmv);
  else if (p.k_pos)
    tc_attn_kernel<true, false><<<grid, kThreads, kSmem, stream>>>(p, x, tmq, tmk, tmv);
  else if (p.block_table)
    tc_attn_kernel<false, true><<<grid, kThreads, kSmem, stream>>>(p, x, tmq, tmk, tmv);
  else
    tc_attn_kernel<false, false><<<grid, kThreads, kSmem, stream>>>(p, x, tmq, tmk, tmv);
  return cudaGetLastError();
}

}  // namespace skv
