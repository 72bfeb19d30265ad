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
// item.  The output O = P V of 128 heads x 512 dims in fp32 would fill all 512 TMEM
// columns of one SM, so the pair splits the latent's dims:
//   CTA 0 holds dims [0, 256): its slice of Q, its slice of every latent tile, and
//          accumulates O[:, 0:256);
//   CTA 1 holds dims [256, 576): its slice of Q and of every latent tile, and
//          accumulates O[:, 256:512) (V dims 256..511 lie inside its slice).
// Every latent byte is therefore loaded exactly once.  Each CTA computes a partial score
// S_r = Q_r K_r^T (M 128, N 64 tokens, K 256 / 320) into TMEM; the partials are swapped
// through distributed shared memory (DSMEM) and both CTAs run the same online softmax on
// S = S_0 + S_1 (identical in both: fp32 addition commutes), write P (bf16) into TMEM
// and accumulate their half of O with tcgen05.mma (A = P from TMEM, B = the MN-major V
// slice, N = 256).  Warp roles per CTA: TMA producer, one MMA-issuing thread, four
// softmax warps (one thread per head = TMEM lane).  S is double-buffered so S(i+1)
// overlaps the softmax of tile i.  Every wait is bounded.
#include <cuda_runtime.h>

#include "skv_common.cuh"
#include "skv_internal.h"
#include "tc_common.cuh"

namespace skv {

namespace {

constexpr int kDk = 576;
constexpr int kHalfDv = 256;   // value dims per CTA
constexpr int kTN = 64;        // tokens per latent tile
constexpr int kNStage = 2;
constexpr int kRows = 128;     // heads per item (MMA M)
constexpr int kThreads = 6 * 32;
constexpr int kBoxBytes = kTN * 128;       // 64 tokens x 64 dims
constexpr int kQBoxBytes = kRows * 128;    // 128 heads x 64 dims
constexpr int kMaxBoxes = 5;               // CTA 1 holds 320 dims
constexpr int kStageBytes = kMaxBoxes * kBoxBytes;  // 40 KB
constexpr int kXBytes = kRows * kTN * 4;            // one S partial, 32 KB
constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + kMaxBoxes * kQBoxBytes;  // 80 KB
constexpr int kOffX = kOffRing + kNStage * kStageBytes;   // +80 KB
constexpr int kOffBar = kOffX + kXBytes;                  // +32 KB
constexpr int kSmem = 1024 + kOffBar + 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S buffer b at kColS + 64 b (b = 0, 1)
constexpr uint32_t kColP = 128;  // P buffer b at kColP + 32 b (bf16 pairs)
constexpr uint32_t kColO = 256;  // O half: 256 columns
constexpr float kRescaleThreshold = 8.0f;
static_assert(kSmem <= 227 * 1024, "shared memory budget");

struct MlaBars {
  uint64_t q_full;
  uint64_t kv_full[kNStage];
  uint64_t kv_empty[kNStage];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done;
  uint64_t x_full;   // the peer's S partial has landed in this CTA's exchange buffer
  uint64_t x_empty;  // the peer has read its exchange buffer: this CTA may write it again
  uint32_t tmem_base;
};

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

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void arrive_remote(uint32_t cluster_bar_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar_addr) : "memory");
}

__device__ __forceinline__ void fence_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on a barrier that the peer CTA arrives on (cluster-scope acquire).
__device__ __forceinline__ bool wait_cluster(uint64_t* bar, uint32_t parity, unsigned int* err) {
  if (try_wait_cluster(bar, parity)) return true;
  const long long c0 = clock64();
  uint32_t spins = 0;
  while (true) {
    if (try_wait_cluster(bar, parity)) return true;
    if ((++spins & 255u) == 0u && clock64() - c0 > kWaitLimitCycles) {
      record_wait_failure(err, kDevErrFullWait, smem_u32(bar), parity);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_4d_plain(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                                  int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_tc_kernel(const __grid_constant__ PartialParams p, const __grid_constant__ TcAttnExtra x,
                  const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tml) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  MlaBars* bars = reinterpret_cast<MlaBars*>(smem + kOffBar);
  float* xbuf = reinterpret_cast<float*>(smem + kOffX);  // [128 rows][64 tokens]: the peer's S partial
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int nbox = rank == 0 ? 4 : 5;  // 64-dim boxes of this CTA's latent slice
  const int dim0 = rank == 0 ? 0 : 256;

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
  const int* bnd = p.bounds + b * (p.n_split + 1);
  const int lo = max(x.fused ? bnd[0] : bnd[j], 0);
  const int hi = min(min(x.fused ? bnd[p.n_split] : bnd[j + 1], seq_len), p.S_max);
  const int win_lo = (lo / kTileN) * kTileN + c * p.chunk_tiles * kTileN;
  const int win_hi = win_lo + p.chunk_tiles * kTileN;
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
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kNStage; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars->s_full[k], 1);
      mbar_init(&bars->p_full[k], kRows);
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->x_full, kRows);  // one arrive per softmax thread of the peer
    mbar_init(&bars->x_empty, kRows);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tml);
      mbar_arrive_expect_tx(&bars->q_full, nbox * kQBoxBytes);
      const int t_start = m0 / p.G;  // G = Hq = 128 rows per query row
      for (int bx = 0; bx < nbox; ++bx)
        tma_load_4d_plain(smem + kOffQ + bx * kQBoxBytes, &tmq, &bars->q_full, dim0 + bx * 64, 0, t_start, b);
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kNStage;
        if (i >= kNStage && !mbar_wait(&bars->kv_empty[s], ((i / kNStage) - 1) & 1, p.err, kDevErrEmptyWait)) break;
        mbar_arrive_expect_tx(&bars->kv_full[s], nbox * kBoxBytes);
        uint8_t* st = smem + kOffRing + s * kStageBytes;
        const int tok = (tile_begin + i) * kTN;
        for (int bx = 0; bx < nbox; ++bx)
          tma_load_4d_plain(st + bx * kBoxBytes, &tml, &bars->kv_full[s], dim0 + bx * 64, tok, 0, b);
        issued = i + 1;
      }
      for (int i = max(0, issued - kNStage); i < issued; ++i) {
        if (!mbar_wait(&bars->kv_full[i % kNStage], (i / kNStage) & 1, p.err, kDevErrDrainWait)) break;
      }
      mbar_wait(&bars->q_full, 0, p.err, kDevErrDrainWait);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      const uint32_t idesc_s = tc::idesc_f16(128, kTN, true, false, false);
      const uint32_t idesc_pv = tc::idesc_f16(128, kHalfDv, true, false, true);
      const uint32_t q_base = smem_u32(smem + kOffQ);
      const uint32_t ring = smem_u32(smem + kOffRing);
      const int ksteps = nbox * 4;  // 16 elements per step
      auto issue_s = [&](int i) {  // S_r(i) = Q_r K_r(i)^T into S buffer i & 1
        const uint32_t kt = ring + (i % kNStage) * kStageBytes;
        for (int ks = 0; ks < ksteps; ++ks) {
          const uint64_t ad = tc::smem_desc_sw128(q_base + (ks >> 2) * kQBoxBytes + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = tc::smem_desc_sw128(kt + (ks >> 2) * kBoxBytes + (ks & 3) * 32, 16, 1024);
          tc::mma_f16_ss(tmem + kColS + 64 * (i & 1), ad, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int i) {  // O_r += P(i) V_r(i)   (M 128, N 256, K 64)
        const uint32_t vt = ring + (i % kNStage) * kStageBytes;  // V = the first 4 boxes of the slice
        for (int ks = 0; ks < kTN / 16; ++ks) {
          const uint64_t bd = tc::smem_desc_sw128(vt + ks * 2048, kBoxBytes, 1024);
          tc::mma_f16_ts(tmem + kColO, tmem + kColP + 32 * (i & 1) + ks * 8, bd, idesc_pv,
                         (i > 0 || ks > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(&bars->q_full, 0, p.err, kDevErrFullWait);
      if (ok) ok = mbar_wait(&bars->kv_full[0], 0, p.err, kDevErrFullWait);
      if (ok) {
        tc::fence_after_sync();
        issue_s(0);
        tc::mma_commit(smem_u32(&bars->s_full[0]));
      }
      for (int i = 0; i < n_tiles && ok; ++i) {
        if (i + 1 < n_tiles) {  // S(i+1) overlaps the softmax of tile i
          ok = mbar_wait(&bars->kv_full[(i + 1) % kNStage], ((i + 1) / kNStage) & 1, p.err, kDevErrFullWait);
          if (!ok) break;
          tc::fence_after_sync();
          issue_s(i + 1);
          tc::mma_commit(smem_u32(&bars->s_full[(i + 1) & 1]));
        }
        ok = mbar_wait(&bars->p_full[i & 1], (i >> 1) & 1, p.err, kDevErrFullWait);
        if (!ok) break;
        tc::fence_after_sync();
        issue_pv(i);
        tc::mma_commit(smem_u32(&bars->pv_done));
        tc::mma_commit(smem_u32(&bars->kv_empty[i % kNStage]));
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int lgrp = warp & 3;          // warps 2..5 -> TMEM lane groups 2, 3, 0, 1
    const int row = lgrp * 32 + lane;   // head row of the item
    const int m = m0 + row;
    const bool valid = m < rows_total;
    const int t_q = valid ? m / p.G : 0;
    const int h = valid ? m % p.G : 0;
    const int64_t hz = p.causal_offset + t_q;
    const int64_t hz_min = p.causal_offset + (m0 + lgrp * 32) / p.G;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(lgrp * 32) << 16);
    const uint32_t x_row_local = smem_u32(xbuf + row * kTN);
    const uint32_t x_row_peer = map_to_rank(x_row_local, peer);
    const uint32_t peer_x_full = map_to_rank(smem_u32(&bars->x_full), peer);
    const uint32_t peer_x_empty = map_to_rank(smem_u32(&bars->x_empty), peer);
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;

    for (int i = 0; i < n_tiles && ok; ++i) {
      const int t0 = (tile_begin + i) * kTN;
      ok = mbar_wait(&bars->s_full[i & 1], (i >> 1) & 1, p.err, kDevErrFullWait);
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t s_col = t_lane + kColS + 64 * (i & 1);
      float sv[kTN];
      {
        uint32_t r[4][16];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tc::tmem_ld16(s_col + 16 * cc, r[cc]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int e = 0; e < 16; ++e) sv[16 * cc + e] = __uint_as_float(r[cc][e]);
      }
      // swap partial scores with the peer: my partial -> its buffer, its partial <- mine
      if (i > 0) ok = wait_cluster(&bars->x_empty, (i - 1) & 1, p.err);  // the peer read its buffer
      if (!ok) break;
#pragma unroll
      for (int q4 = 0; q4 < kTN / 4; ++q4)
        st_cluster_v4(x_row_peer + 16 * q4, sv[4 * q4], sv[4 * q4 + 1], sv[4 * q4 + 2], sv[4 * q4 + 3]);
      arrive_remote(peer_x_full);  // release: this thread's row is visible to the peer
      ok = wait_cluster(&bars->x_full, i & 1, p.err);
      if (!ok) break;
      const float* xr = xbuf + row * kTN;
#pragma unroll
      for (int q4 = 0; q4 < kTN / 4; ++q4) {
        const float4 v = *reinterpret_cast<const float4*>(xr + 4 * q4);
        sv[4 * q4] += v.x;
        sv[4 * q4 + 1] += v.y;
        sv[4 * q4 + 2] += v.z;
        sv[4 * q4 + 3] += v.w;
      }
      arrive_remote(peer_x_empty);  // this thread's row of my buffer may be written again

      // ---- softmax on S = S_0 + S_1 (identical in both CTAs)
      const bool in_range = (t0 >= r_lo) && (t0 + kTN <= r_hi);
      const bool need_mask = !in_range || (static_cast<int64_t>(t0) + kTN - 1 > hz_min);
      if (need_mask) {
        const int c_lo = min(max(r_lo - t0, 0), kTN);
        const int c_hi = static_cast<int>(
            min(max(min(static_cast<int64_t>(r_hi), hz + 1) - t0, (int64_t)0), (int64_t)kTN));
        const unsigned span = static_cast<unsigned>(max(c_hi - c_lo, 0));
#pragma unroll
        for (int cc = 0; cc < kTN; ++cc) sv[cc] = (static_cast<unsigned>(cc - c_lo) < span) ? sv[cc] : -INFINITY;
      }
      float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
      for (int cc = 4; cc < kTN; cc += 4) {
        mx[0] = fmaxf(mx[0], sv[cc]);
        mx[1] = fmaxf(mx[1], sv[cc + 1]);
        mx[2] = fmaxf(mx[2], sv[cc + 2]);
        mx[3] = fmaxf(mx[3], sv[cc + 3]);
      }
      const float sl = p.scale_log2;
      const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl;
      const bool need = (tmax != -INFINITY) && (m_used == -INFINITY || tmax > m_used + kRescaleThreshold);
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? fmaxf(m_used, tmax) : m_used;
        if (i > 0) {
          ok = mbar_wait(&bars->pv_done, (i - 1) & 1, p.err, kDevErrFullWait);  // O final up to tile i-1
          tc::fence_after_sync();
          const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < kHalfDv / 16; cc += 2) {
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
          l_sum *= alpha;
        } else {
          l_sum = 0.f;
        }
        m_used = m_new;
      }
      const float base = (m_used == -INFINITY) ? 0.f : m_used;
      // P(i) goes to P buffer i & 1; its previous user PV(i-2) finished before S(i) ran
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int cc = 0; cc < kTN / 32; ++cc) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = fast_exp2(fmaf(sv[32 * cc + 2 * e], sl, -base));
          const float p1 = fast_exp2(fmaf(sv[32 * cc + 2 * e + 1], sl, -base));
          ls[(2 * e) & 3] += p0;
          ls[(2 * e + 1) & 3] += p1;
          w[e] = pack_bf16(p0, p1);
        }
        tc::tmem_st16(t_lane + kColP + 32 * (i & 1) + 16 * cc, w);
      }
      tc::tmem_wait_st();
      l_sum += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      if (!in_range) {
        // tokens outside [r_lo, r_hi) may hold anything (NaN past the end of a sequence):
        // zero their rows of this CTA's V slice so that p = 0 contributes nothing
        const int s_idx = i % kNStage;
        mbar_wait(&bars->kv_full[s_idx], (i / kNStage) & 1, p.err, kDevErrFullWait);
        if (row < kTN) {
          const int tok = t0 + row;
          if (tok < r_lo || tok >= r_hi) {
            uint8_t* vt = smem + kOffRing + s_idx * kStageBytes;
            for (int bx = 0; bx < 4; ++bx)
              for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4*>(vt + bx * kBoxBytes + row * 128 + q * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
      }
      tc::fence_before_sync();
      mbar_arrive(&bars->p_full[i & 1]);
    }

    // ---- epilogue: this CTA's 256 dims of O / l; CTA 0 writes lse
    if (n_tiles > 0 && ok) {
      ok = mbar_wait(&bars->pv_done, (n_tiles - 1) & 1, p.err, kDevErrFullWait);
      tc::fence_after_sync();
    }
    const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
    constexpr float kLn2 = 0.6931471805599453f;
    const float lse = l_sum > 0.f ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
    const int dv_total = 2 * kHalfDv;
    if (x.fused) {
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(x.out_bf16) +
                            ((static_cast<int64_t>(b) * p.Tq + t_q) * p.Hq + h) * dv_total + rank * kHalfDv;
#pragma unroll 1
      for (int cc = 0; cc < kHalfDv / 16; ++cc) {
        uint32_t r[16];
        if (n_tiles > 0) {
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
      if (valid && rank == 0) x.out_lse[(static_cast<int64_t>(b) * p.Tq + t_q) * p.Hq + h] = lse;
    } else {
      const int part = j * p.n_chunk + c;
      const int64_t ro = ((static_cast<int64_t>(part) * p.B + b) * p.Tq + t_q) * p.Hq + h;
      float* orow = p.out_o + ro * dv_total + rank * kHalfDv;
      const bool write_o = valid && (l_sum > 0.f || p.zero_empty);
#pragma unroll 1
      for (int cc = 0; cc < kHalfDv / 16; ++cc) {
        uint32_t r[16];
        if (n_tiles > 0) {
          tc::tmem_ld16(t_lane + kColO + 16 * cc, r);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = 0u;
        }
        if (write_o) {
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(orow + 16 * cc + e) =
                make_float4(__uint_as_float(r[e]) * inv, __uint_as_float(r[e + 1]) * inv,
                            __uint_as_float(r[e + 2]) * inv, __uint_as_float(r[e + 3]) * inv);
        }
      }
      if (valid && rank == 0) p.out_lse[ro] = lse;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer no longer touches this CTA's shared memory
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

int mla_tc_rows_per_item() { return kRows; }
int mla_tc_kv_tile() { return kTN; }

cudaError_t launch_mla_tc(const PartialParams& p, const TcAttnExtra& x, const CUtensorMap& tmq,
                          const CUtensorMap& tml, int64_t n_items, cudaStream_t stream) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  if (n_items <= 0) return cudaSuccess;
  mla_tc_kernel<<<static_cast<unsigned int>(2 * n_items), kThreads, kSmem, stream>>>(p, x, tmq, tml);
  return cudaGetLastError();
}

}  // namespace skv
