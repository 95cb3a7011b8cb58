// Selective LM head fused with the confidence + commit step, for sm_103a.
//
// Source: JetEngine notes (CLAUDE.md), "ModelRunner" (selective logits for DENOISING
// sequences), "Optimization History" (opt23: LM head only on masked rows) and "Remaining
// Optimization Avenues" (a fused postprocess kernel); the confidence and the commit rules as
// in the commit kernels (JetEngine notes, "Remasking Strategies"; dInfer blog, "Algorithmic
// Innovations").
//
// The logits of the scored rows are reduced to (max, sum of exponentials, first argmax) while
// they leave tensor memory, so they are never written to HBM and read back: the step moves W
// once and a few MB of rows and partials instead of W plus twice the logits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "confidence.cuh"
#include "kernels.h"
#include "lm_common.cuh"
#include "ptx.cuh"

namespace bdlm {
namespace {

using namespace lm;

// The same GEMM computed the other way round, for the fused LM head + confidence step: a tile
// is up to 256 active rows (two UMMAs of M = 128, the row sub-tiles) by 256 vocabulary
// columns (N = 256: the two 128-row W boxes of a stage lie side by side and form one K-major
// operand).  A tensor-memory lane is then one active row and its columns run along the
// vocabulary, so each epilogue thread reduces its own row's logits with no cross-lane
// shuffles: it rounds them to bf16 (the logits the unfused path would store), optionally
// stores them, and folds them into a running (max, sum of exponentials, first index of the
// max).  The row's logits never have to be read back.
//
// Work split: with rt row tiles (256 active rows each), CTA c < (grid / rt) * rt keeps row tile
// c % rt for its whole life and walks the vocabulary tiles c / rt, c / rt + grid / rt, ...; the
// CTAs that run together hold the same W tiles for the different row tiles, so W streams from
// HBM about once.  When its CTA is done, each row's four column shares are merged in shared
// memory (the rings are idle by then) into one partial per (row, CTA); a per-block kernel
// merges a row's partials.
constexpr int kConfWS = 4, kConfHS = 3;     // W and row stages, 32 KB each
constexpr int kConfN = kSub * kBM;          // vocabulary columns per tile (UMMA N)
constexpr int kConfShares = kEpiWarps / 4;  // epilogue warps per tensor-memory lane quadrant
constexpr int kConfShareCols = kConfN / kConfShares;
static_assert(kConfShareCols == 64, "each epilogue thread folds two groups of 32 logits");

struct LmConfParams {
  const int32_t* active_idx;
  const int32_t* n_active_dev;   // active-row count on the device (<= n_active)
  uint16_t* logits;              // may be null: the logits are then not stored
  CommitPartial* part;           // [n_active][slots]
  int* err;
  int n_active, n_rows, H, V, m_tiles, k_blocks, slots;
  float c;                       // log2(e) / temperature
};

// Loads `boxes` boxes of kBM rows (box_bytes each, kWBox apart) at row0(j) = first +
// j * step + b * kBM, every K step of jobs j < n_jobs, into a ring of NSTAGES stages.
template <int NSTAGES, int STRIDE>
__device__ bool produce_jobs(const CUtensorMap* tm, uint8_t* ring, uint64_t* full, uint64_t* empty,
                             int n_jobs, int first, int step, int boxes, int k_blocks,
                             int* abort_flag) {
  tma_prefetch_desc(tm);
  RingPos pos;
  bool ok = true;
  for (int j = 0; j < n_jobs && ok; ++j) {
    const int row0 = first + j * step;
    for (int kb = 0; kb < k_blocks; ++kb) {
      if (!(ok = mbar_wait(&empty[pos.slot], pos.phase ^ 1, abort_flag))) break;
      mbar_arrive_expect_tx(&full[pos.slot], static_cast<uint32_t>(boxes) * kWBox);
      for (int b = 0; b < boxes; ++b)   // boxes past the tensor read as zeros
        tma_load_2d(ring + pos.slot * STRIDE + b * kWBox, tm, &full[pos.slot], kb * kBK,
                    row0 + b * kBM);
      pos.advance(NSTAGES);
    }
  }
  if (!ok) {
    int dummy = 0;
    for (int s = 0; s < NSTAGES; ++s)
      mbar_wait(&full[s], pos.phase ^ (s < pos.slot ? 0u : 1u), &dummy);
  }
  return ok;
}

// Folds 32 logits (16 packed bf16 pairs, indices base .. base + 31 in order) into a row's
// running state; a strictly larger group max moves the max and its first index.  ENT: also the
// exponent-weighted sum (for the entropy).
template <bool ENT>
__device__ __forceinline__ void fold32(Acc& a, const uint32_t (&w)[16], int base, float c) {
  const float gm = group_max(w);
  if (gm > a.m) {
    if (a.m == -CUDART_INF_F) {
      a.s = 0.f;
      a.a = 0.f;
    } else {
      acc_rebase(a.s, a.a, a.m, gm, c);
    }
    a.m = gm;
    int first = 0x7FFFFFFF;
#pragma unroll
    for (int e = 31; e >= 0; --e) {
      const float x = (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
      if (x == gm) first = base + e;
    }
    a.idx = first;
  }
  if (a.m == -CUDART_INF_F) return;  // nothing but padding so far
  exp_sum32<ENT>(w, c, a.m * c, a.s, a.a);
}

template <bool ENT>
__global__ void __launch_bounds__(kThreads, 1)
lm_conf_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
               const LmConfParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* wring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t* hring = wring + kConfWS * kWBytes;
  __shared__ uint64_t w_full[kConfWS], w_empty[kConfWS], h_full[kConfHS], h_empty[kConfHS];
  __shared__ uint64_t acc_full, acc_empty, bar_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kConfWS; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 1);
    }
    for (int s = 0; s < kConfHS; ++s) {
      mbar_init(&h_full[s], 1);
      mbar_init(&h_empty[s], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kEpiThreads);
    mbar_init(&bar_done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  const uint32_t tmem = tmem_base;
  const int n_act = min(max(*p.n_active_dev, 0), p.n_active);
  const int rt = (n_act + kConfN - 1) / kConfN;          // row tiles
  const int per_tile = rt > 0 ? static_cast<int>(gridDim.x) / rt : 0;  // CTAs per row tile
  const int cta = blockIdx.x;
  const bool working = rt > 0 && cta < per_tile * rt;
  const int n = working ? cta % rt : 0;
  const int m_first = working ? cta / rt : 0;
  const int n_jobs = (working && m_first < p.m_tiles)
                         ? (p.m_tiles - m_first + per_tile - 1) / per_tile : 0;
  const int n_sub = working ? min(kSub, (n_act - n * kConfN + kBM - 1) / kBM) : 0;

  if (warp == 0) {
    if (lane == 0) {
      produce_jobs<kConfWS, kWBytes>(&tm_w, wring, w_full, w_empty, n_jobs, m_first * kConfN,
                                     per_tile * kConfN, kSub, p.k_blocks, &abort_flag);
      griddep_launch_dependents();
    }
  } else if (warp == kRowWarp) {
    if (lane == 0)
      produce_jobs<kConfHS, kWBytes>(&tm_h, hring, h_full, h_empty, n_jobs, n * kConfN, 0, n_sub,
                                     p.k_blocks, &abort_flag);
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, kConfN, false, false);
      const uint32_t w0 = smem_u32(wring), h0 = smem_u32(hring);
      RingPos wp, hp;
      bool ok = true;
      for (int j = 0; j < n_jobs && ok; ++j) {
        if (!(ok = mbar_wait(&acc_empty, (j & 1) ^ 1, &abort_flag))) break;
        tc_fence_after();
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!(ok = mbar_wait(&w_full[wp.slot], wp.phase, &abort_flag))) break;
          if (!(ok = mbar_wait(&h_full[hp.slot], hp.phase, &abort_flag))) break;
          tc_fence_after();
          const uint32_t sw = w0 + wp.slot * kWBytes;
          const uint32_t sh = h0 + hp.slot * kWBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t bd = smem_desc(sw + kk * 32, 16, 1024);
#pragma unroll
            for (int s = 0; s < kSub; ++s)
              if (s < n_sub) {
                const uint64_t ad = smem_desc(sh + s * kWBox + kk * 32, 16, 1024);
                umma_bf16(tmem + s * kConfN, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
              }
          }
          umma_commit(&w_empty[wp.slot]);
          umma_commit(&h_empty[hp.slot]);
          wp.advance(kConfWS);
          hp.advance(kConfHS);
        }
        if (!ok) break;
        umma_commit(&acc_full);
      }
      umma_commit(&bar_done);
    }
  } else {
    const int q4 = warp & 3;                 // tensor-memory lanes 32*q4 .. 32*q4+31
    const int share = (warp - 2) >> 2;       // columns share*64 .. share*64+63 of a sub-tile
    const int x = (q4 << 5) | lane;          // row within a sub-tile
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int col0 = share * kConfShareCols;
    int arow[kSub], lrow[kSub];
    Acc acc[kSub];
#pragma unroll
    for (int s = 0; s < kSub; ++s) {
      arow[s] = n * kConfN + s * kBM + x;    // active index
      const bool valid = s < n_sub && arow[s] < n_act;
      lrow[s] = -1;                          // logits row to store (-1: none)
      if (valid && p.logits != nullptr) {
        const int r = __ldg(p.active_idx + arow[s]);
        lrow[s] = (r >= 0 && r < p.n_rows) ? r : -1;   // a bad id is flagged by the gather
      }
      if (!valid) arow[s] = -1;
      acc[s] = acc_init();
    }
    bool ok = true;
    for (int j = 0; j < n_jobs; ++j) {
      if (!ok || !(ok = mbar_wait_warp(&acc_full, j & 1, &abort_flag))) break;
      tc_fence_after();
      const int vbase = (m_first + j * per_tile) * kConfN + col0;
      // Sub-tile by sub-tile (the registers hold one row's 64 logits at a time): read the
      // share's columns, round to bf16 pairs, store them if asked, fold them.  Tensor memory
      // is released after the last sub-tile; meanwhile the rings keep filling.
#pragma unroll
      for (int s = 0; s < kSub; ++s) {
        if (s >= n_sub) continue;
        __syncwarp();         // the tensor-memory loads below are warp-collective
        uint32_t wv[2][16];   // the share's 64 logits of the row as bf16 pairs
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t r[16];
          tmem_ld16(tmem + lane_off + static_cast<uint32_t>(s * kConfN + col0 + g * 16), r);
          tmem_wait_ld();
          tmem_regs_ready(r);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const __nv_bfloat162 h =
                __floats2bfloat162_rn(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]));
            wv[g >> 1][(g & 1) * 8 + k] = *reinterpret_cast<const uint32_t*>(&h);
          }
        }
        if (arow[s] < 0) continue;
        if (vbase + kConfShareCols > p.V) {
          // the last vocabulary tile: logits past V take no part
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int v = vbase + h * 32 + 2 * e;
              uint32_t t = wv[h][e];
              if (v >= p.V) t = (t & 0xFFFF0000u) | 0xFF80u;
              if (v + 1 >= p.V) t = (t & 0x0000FFFFu) | 0xFF800000u;
              wv[h][e] = t;
            }
        }
        if (lrow[s] >= 0) {
          uint4* dst =
              reinterpret_cast<uint4*>(p.logits + static_cast<size_t>(lrow[s]) * p.V + vbase);
#pragma unroll
          for (int q = 0; q < 8; ++q)   // V % 8 == 0: a group of 8 is inside V or past it
            if (vbase + 8 * q < p.V)
              dst[q] = make_uint4(wv[q >> 2][(q & 3) * 4], wv[q >> 2][(q & 3) * 4 + 1],
                                  wv[q >> 2][(q & 3) * 4 + 2], wv[q >> 2][(q & 3) * 4 + 3]);
        }
        fold32<ENT>(acc[s], wv[0], vbase, p.c);
        fold32<ENT>(acc[s], wv[1], vbase + 32, p.c);
      }
      tc_fence_before();
      mbar_arrive(&acc_empty);   // tensor memory is free for the next tile's MMAs
    }
    // the four shares of each row, merged in the (now idle) W ring: [share][sub-tile][row]
    float* sh_m = reinterpret_cast<float*>(wring);
    float* sh_s = sh_m + kConfShares * kSub * kBM;
    float* sh_a = sh_s + kConfShares * kSub * kBM;
    int* sh_i = reinterpret_cast<int*>(sh_a + kConfShares * kSub * kBM);
#pragma unroll
    for (int s = 0; s < kSub; ++s) {
      const int at = (share * kSub + s) * kBM + x;
      sh_m[at] = acc[s].m;
      sh_s[at] = acc[s].s;
      sh_a[at] = acc[s].a;
      sh_i[at] = acc[s].idx;
    }
    named_barrier(1, kEpiThreads);
    if (share == 0) {
      const int slot = cta / max(rt, 1);
#pragma unroll
      for (int s = 0; s < kSub; ++s) {
        if (arow[s] < 0) continue;
        Acc t = acc[s];
        for (int o = 1; o < kConfShares; ++o) {
          const int at = (o * kSub + s) * kBM + x;
          t = merge(t, Acc{sh_m[at], sh_s[at], sh_a[at], sh_i[at]}, p.c);
        }
        p.part[static_cast<size_t>(arow[s]) * p.slots + slot] = CommitPartial{t.m, t.s, t.idx, t.a};
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      int dummy = 0;
      mbar_wait(&bar_done, 0, &dummy);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && abort_flag) atomicOr(p.err, BDLM_DEVERR_TIMEOUT);
}

size_t lm_conf_smem() { return 1024 + static_cast<size_t>(kConfWS + kConfHS) * kWBytes; }

// ------------------------------------------------------------------ CTA-pair variant
// Above 128 scored rows the same GEMM runs on CTA pairs (clusters of two, tcgen05
// cta_group::2): a pair tile is 256 scored rows (128 per CTA, the two halves of one M = 256
// UMMA) by up to 256 vocabulary columns, and per K step each CTA stages its own 128 rows and
// its half of the tile's W rows.  A CTA's accumulator is then 128 lanes x 256 columns, half
// of tensor memory, so two tiles' accumulators alternate and the epilogue of one tile
// overlaps the MMAs of the next (the single-CTA tile of 256 x 256 fills tensor memory and
// must be drained first).  Shared-memory fill per MMA FLOP is that of the single-CTA kernel,
// and each W tile is fetched once per pair.
//
// With rt row tiles, pair q < (pairs / rt) * rt keeps row tile q % rt and owns an equal,
// contiguous share of the vocabulary (slot q / rt of pairs / rt, in units of 16 columns),
// walked in tiles of 256 columns; the last tile is narrower (the UMMA's N is set per tile),
// so every pair streams the same number of W bytes.  Each CTA writes one partial per (row,
// pair).  The even CTA's W and row barriers count both CTAs' bytes; its MMA thread issues
// every UMMA, and its commits release the stages and signal the accumulators in both CTAs.
#ifndef BDLM_PAIR_KW
#define BDLM_PAIR_KW 2
#endif
#ifndef BDLM_PAIR_KH
#define BDLM_PAIR_KH 2
#endif
#ifndef BDLM_PAIR_WS
#define BDLM_PAIR_WS 4
#endif
#ifndef BDLM_PAIR_HS
#define BDLM_PAIR_HS 3
#endif
// 64-wide K boxes per W and per row stage: a W stage reads 128 * KW contiguous bytes of each
// of its rows, which the memory system serves better than one box at a time.
constexpr int kPairKW = BDLM_PAIR_KW, kPairKH = BDLM_PAIR_KH;
constexpr int kPairWS = BDLM_PAIR_WS, kPairHS = BDLM_PAIR_HS;   // W and row stages
constexpr int kPairWStage = kPairKW * kWBox, kPairHStage = kPairKH * kWBox;   // bytes per CTA
static_assert(kPairKW % kPairKH == 0 || kPairKH % kPairKW == 0, "stage boxes must nest");
constexpr uint32_t kPairCols = 256;              // tensor-memory columns per accumulator
constexpr int kPairUnit = 16;                    // vocabulary columns per unit of work

// The vocabulary share of one pair: units [u_lo, u_hi) of 16 columns, in tiles of 256.
struct PairJobs {
  int u_lo = 0, u_hi = 0, n_jobs = 0;
  __device__ int col0(int j) const { return (u_lo + j * (kConfN / kPairUnit)) * kPairUnit; }
  __device__ int width(int j) const {   // a multiple of 16, 16 .. 256
    return min(kConfN, (u_hi - u_lo - j * (kConfN / kPairUnit)) * kPairUnit);
  }
};

// Streams the stages of every job into a ring: W (rows of the tile's half) or the row tile.
// The even CTA arms each stage's full barrier with both CTAs' bytes; both CTAs' copies
// complete on that barrier.
template <int NSTAGES, int KS, bool IS_W>
__device__ void produce_pair(const CUtensorMap* tm, uint8_t* ring, uint64_t* full, uint64_t* empty,
                             bool leader, uint32_t rank, const PairJobs& jobs, int row_tile0,
                             int k_boxes, int* abort_flag) {
  constexpr int kStage = KS * kWBox;
  const int k_stages = (k_boxes + KS - 1) / KS;
  tma_prefetch_desc(tm);
  RingPos pos;
  bool ok = true;
  for (int j = 0; j < jobs.n_jobs && ok; ++j) {
    const int row0 = IS_W ? jobs.col0(j) + static_cast<int>(rank) * (jobs.width(j) >> 1)
                          : row_tile0 + static_cast<int>(rank) * kBM;
    for (int ks = 0; ks < k_stages; ++ks) {
      if (!(ok = mbar_wait(&empty[pos.slot], pos.phase ^ 1, abort_flag))) break;
      if (leader) mbar_arrive_expect_tx(&full[pos.slot], 2 * kStage);
      const uint32_t bar = cluster_map(&full[pos.slot], 0);
#pragma unroll
      for (int b = 0; b < KS; ++b)   // boxes past the tensor read as zeros
        tma_load_2d_pair(ring + pos.slot * kStage + b * kWBox, tm, bar, (ks * KS + b) * kBK,
                         row0);
      pos.advance(NSTAGES);
    }
  }
  if (!ok) {
    // after a failed wait: copies already issued land within microseconds; give them 200 us
    // before this CTA may exit (the even CTA's barriers may never see the odd CTA's bytes)
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
}

template <bool ENT>
__global__ void __launch_bounds__(kThreads, 1)
lm_conf_pair_kernel(const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ CUtensorMap tm_h, const LmConfParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* wring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t* hring = wring + kPairWS * kPairWStage;
  __shared__ uint64_t w_full[kPairWS], w_empty[kPairWS], h_full[kPairHS], h_empty[kPairHS];
  __shared__ uint64_t acc_full[2], acc_empty[2], bar_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairWS; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 1);
    }
    for (int s = 0; s < kPairHS; ++s) {
      mbar_init(&h_full[s], 1);
      mbar_init(&h_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * kEpiWarps);   // one arrival per epilogue warp of each CTA
    }
    mbar_init(&bar_done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();   // both CTAs' barriers exist before either CTA signals the other's
  tc_fence_after();
  griddep_wait();
  const uint32_t tmem = tmem_base;
  const int n_act = min(max(*p.n_active_dev, 0), p.n_active);
  const int pairs = static_cast<int>(gridDim.x) >> 1;
  const int pair = static_cast<int>(blockIdx.x) >> 1;
  const int rt = (n_act + kConfN - 1) / kConfN;           // row tiles of 256
  const int per_tile = rt > 0 ? pairs / rt : 0;           // pairs per row tile
  const bool working = rt > 0 && pair < per_tile * rt;
  const int n = working ? pair % rt : 0;
  const int slot = working ? pair / rt : 0;
  PairJobs jobs;
  if (working) {
    const long long units = (p.V + kPairUnit - 1) / kPairUnit;
    jobs.u_lo = static_cast<int>(units * slot / per_tile);
    jobs.u_hi = static_cast<int>(units * (slot + 1) / per_tile);
    jobs.n_jobs = (jobs.u_hi - jobs.u_lo + kConfN / kPairUnit - 1) / (kConfN / kPairUnit);
  }
  const int n_jobs = jobs.n_jobs;
  // K in boxes of 64, rounded up to whole stages of both rings (boxes past H read as zeros)
  constexpr int kLcm = kPairKW > kPairKH ? kPairKW : kPairKH;
  const int k_boxes = (p.k_blocks + kLcm - 1) / kLcm * kLcm;

  if (warp == 0) {
    if (lane == 0) {
      produce_pair<kPairWS, kPairKW, true>(&tm_w, wring, w_full, w_empty, leader, rank, jobs, 0,
                                           k_boxes, &abort_flag);
      griddep_launch_dependents();
    }
  } else if (warp == kRowWarp) {
    if (lane == 0)
      produce_pair<kPairHS, kPairKH, false>(&tm_h, hring, h_full, h_empty, leader, rank, jobs,
                                            n * kConfN, k_boxes, &abort_flag);
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      const uint32_t w0 = smem_u32(wring), h0 = smem_u32(hring);
      RingPos wp, hp;
      bool ok = true;
      for (int j = 0; j < n_jobs && ok; ++j) {
        const int buf = j & 1;
        const uint32_t idesc = idesc_bf16_f32(2 * kBM, jobs.width(j), false, false);
        if (!(ok = mbar_wait_cluster(&acc_empty[buf], ((j >> 1) & 1) ^ 1, &abort_flag))) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(buf) * kPairCols;
        for (int kb = 0; kb < k_boxes; ++kb) {
          const int bw = kb % kPairKW, bh = kb % kPairKH;   // box within the W / row stage
          if (bw == 0 && !(ok = mbar_wait_cluster(&w_full[wp.slot], wp.phase, &abort_flag))) break;
          if (bh == 0 && !(ok = mbar_wait_cluster(&h_full[hp.slot], hp.phase, &abort_flag))) break;
          tc_fence_after();
          const uint32_t sw = w0 + wp.slot * kPairWStage + bw * kWBox;
          const uint32_t sh = h0 + hp.slot * kPairHStage + bh * kWBox;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_pair(d, smem_desc(sh + kk * 32, 16, 1024), smem_desc(sw + kk * 32, 16, 1024),
                           idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          if (bw == kPairKW - 1) {
            umma_commit_pair(&w_empty[wp.slot], 3);
            wp.advance(kPairWS);
          }
          if (bh == kPairKH - 1) {
            umma_commit_pair(&h_empty[hp.slot], 3);
            hp.advance(kPairHS);
          }
        }
        if (!ok) break;
        umma_commit_pair(&acc_full[buf], 3);
      }
      umma_commit_pair(&bar_done, 3);
    }
  } else {
    const int q4 = warp & 3;                 // tensor-memory lanes 32*q4 .. 32*q4+31
    const int share = (warp - 2) >> 2;       // columns share*64 .. share*64+63 of a tile
    const int x = (q4 << 5) | lane;          // row within this CTA's half of the tile
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int col0 = share * kConfShareCols;
    const uint32_t empty0 = cluster_map(&acc_empty[0], 0), empty1 = cluster_map(&acc_empty[1], 0);
    int arow = n * kConfN + static_cast<int>(rank) * kBM + x;   // active index
    const bool valid = working && arow < n_act;
    int lrow = -1;                                               // logits row to store
    if (valid && p.logits != nullptr) {
      const int r = __ldg(p.active_idx + arow);
      lrow = (r >= 0 && r < p.n_rows) ? r : -1;   // a bad id is flagged by the gather
    }
    if (!valid) arow = -1;
    Acc acc = acc_init();
    bool ok = true;
    for (int j = 0; j < n_jobs; ++j) {
      const int buf = j & 1;
      if (!ok || !(ok = mbar_wait_warp(&acc_full[buf], (j >> 1) & 1, &abort_flag))) break;
      tc_fence_after();
      const int vbase = jobs.col0(j) + col0;
      const int vend = min(jobs.col0(j) + jobs.width(j), p.V);   // the tile's last column + 1
      __syncwarp();         // the tensor-memory loads below are warp-collective
      uint32_t wv[2][16];   // the share's 64 logits of the row as bf16 pairs
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_off + static_cast<uint32_t>(buf) * kPairCols +
                      static_cast<uint32_t>(col0 + g * 16), r);
        tmem_wait_ld();
        tmem_regs_ready(r);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const __nv_bfloat162 h =
              __floats2bfloat162_rn(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]));
          wv[g >> 1][(g & 1) * 8 + k] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      // this warp's columns are in registers: the accumulator may take the tile after next (a
      // tensor-memory hand-off, ordered by the tcgen05 fences: CTA-scope release suffices)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote_cta(buf ? empty1 : empty0);
      if (arow < 0) continue;
      if (vbase + kConfShareCols > vend) {
        // a narrow tile or the end of V: columns past the tile take no part
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int v = vbase + h * 32 + 2 * e;
            uint32_t t = wv[h][e];
            if (v >= vend) t = (t & 0xFFFF0000u) | 0xFF80u;
            if (v + 1 >= vend) t = (t & 0x0000FFFFu) | 0xFF800000u;
            wv[h][e] = t;
          }
      }
      if (lrow >= 0) {
        uint4* dst = reinterpret_cast<uint4*>(p.logits + static_cast<size_t>(lrow) * p.V + vbase);
#pragma unroll
        for (int q = 0; q < 8; ++q)   // tile ends and V are multiples of 8
          if (vbase + 8 * q < vend)
            dst[q] = make_uint4(wv[q >> 2][(q & 3) * 4], wv[q >> 2][(q & 3) * 4 + 1],
                                wv[q >> 2][(q & 3) * 4 + 2], wv[q >> 2][(q & 3) * 4 + 3]);
      }
      fold32<ENT>(acc, wv[0], vbase, p.c);
      fold32<ENT>(acc, wv[1], vbase + 32, p.c);
    }
    // the four shares of each row, merged in the (now idle) W ring: [share][row]
    float* sh_m = reinterpret_cast<float*>(wring);
    float* sh_s = sh_m + kConfShares * kBM;
    float* sh_a = sh_s + kConfShares * kBM;
    int* sh_i = reinterpret_cast<int*>(sh_a + kConfShares * kBM);
    sh_m[share * kBM + x] = acc.m;
    sh_s[share * kBM + x] = acc.s;
    sh_a[share * kBM + x] = acc.a;
    sh_i[share * kBM + x] = acc.idx;
    named_barrier(1, kEpiThreads);
    if (share == 0 && arow >= 0) {
      Acc t = acc;
      for (int o = 1; o < kConfShares; ++o)
        t = merge(t, Acc{sh_m[o * kBM + x], sh_s[o * kBM + x], sh_a[o * kBM + x],
                         sh_i[o * kBM + x]}, p.c);
      p.part[static_cast<size_t>(arow) * p.slots + slot] =
          CommitPartial{t.m, t.s, t.idx, t.a};
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1 && lane == 0) {
    int dummy = 0;
    mbar_wait(&bar_done, 0, &dummy);   // every UMMA writing this CTA's tensor memory is done
  }
  tc_fence_before();
  cluster_sync();   // neither CTA exits or frees tensor memory while the other may signal it
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && abort_flag) atomicOr(p.err, BDLM_DEVERR_TIMEOUT);
}

size_t lm_conf_pair_smem() {
  return 1024 + static_cast<size_t>(kPairWS) * kPairWStage + static_cast<size_t>(kPairHS) * kPairHStage;
}

// ------------------------------------------------------------------ scored rows
// Row r = b * L + i is scored when mask[r] != 0 and (den is null or den[b] != 0).  CTA r counts
// the scored rows before r; if row r is scored it copies hidden[r] to gathered[idx] and records
// act[idx] = r, idx being that count.  CTA 0 also writes the total to *n_act.  (The row list of
// bdlm_active_rows and the gather of the LM head in one launch.)
__global__ void __launch_bounds__(256)
scored_gather_kernel(const uint16_t* __restrict__ hidden, const uint8_t* __restrict__ mask,
                     const uint8_t* __restrict__ den, int R, int L, int H,
                     uint16_t* __restrict__ gathered, int32_t* __restrict__ act,
                     int32_t* __restrict__ n_act) {
  __shared__ int s_warp[8];
  griddep_wait();
  griddep_launch_dependents();
  const int r = blockIdx.x;
  auto is_scored = [&](int q) -> int {
    return mask[q] != 0 && (den == nullptr || den[q / L] != 0);
  };
  const int mine = is_scored(r);
  if (!mine && r != 0) return;
  const int limit = r == 0 ? R : r;   // CTA 0 counts every row
  int before = 0, total = 0;
  for (int q = threadIdx.x; q < limit; q += blockDim.x) {
    const int sc = is_scored(q);
    total += sc;
    before += q < r ? sc : 0;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, off);
    total += __shfl_xor_sync(0xffffffffu, total, off);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (lane == 0) s_warp[warp] = r == 0 ? total : before;
  __syncthreads();
  int cnt = 0;
  for (int w = 0; w < nw; ++w) cnt += s_warp[w];
  if (r == 0 && threadIdx.x == 0) *n_act = cnt;
  if (!mine) return;
  const int idx = r == 0 ? 0 : cnt;
  if (threadIdx.x == 0) act[idx] = r;
  const uint4* src = reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(r) * H);
  uint4* dst = reinterpret_cast<uint4*>(gathered + static_cast<size_t>(idx) * H);
  for (int v = threadIdx.x; v < H / 8; v += blockDim.x) dst[v] = __ldg(src + v);
}

// ------------------------------------------------------------------ per-block finalize
struct LmCommitArgs {
  const uint8_t* mask;
  const uint8_t* den;        // may be null: every sequence is denoising
  int R, L;
  const CommitPartial* part; // [scored row][slots]
  int slots;                 // slots allocated per scored row
  int lm_grid, shares;       // LM head workers (CTAs or CTA pairs), partials each writes per row
  float c, threshold;
  int rule, k;
  int32_t* tok_out;
  float* conf_out;
  float* ent_out;            // may be null
  uint8_t* commit_out;
};

constexpr int kFinThreads = 1024;

__device__ __forceinline__ int scored(const LmCommitArgs& a, int r) {
  return a.mask[r] != 0 && (a.den == nullptr || a.den[r / a.L] != 0);
}

// One CTA per block b.  The scored rows (masked, in a denoising sequence) are numbered in row
// order, as the active-row list of the LM head numbers them; with rt = ceil(scored / 256) row
// tiles, the LM head ran lm_grid / rt workers (CTAs, or CTA pairs) per row tile and each wrote
// `shares` partials per row.
// Up to 32 rows at a time, 32 / rows warps per row merge a row's partials; then warp 0
// decides the block over its scored positions.
__global__ void __launch_bounds__(kFinThreads)
lm_commit_finalize_kernel(const LmCommitArgs a) {
  __shared__ int s_wsum[2][kFinThreads / 32];
  __shared__ int s_before, s_total;
  __shared__ Acc s_acc[kFinThreads / 32];
  __shared__ float s_stat[64];
  __shared__ int s_order[64];
  const int b = blockIdx.x, L = a.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int before = 0, total = 0;
  for (int r = tid; r < a.R; r += kFinThreads) {
    const int sc = scored(a, r);
    total += sc;
    before += (r < b * L) ? sc : 0;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, off);
    total += __shfl_xor_sync(0xffffffffu, total, off);
  }
  if (lane == 0) {
    s_wsum[0][warp] = before;
    s_wsum[1][warp] = total;
  }
  __syncthreads();
  if (tid == 0) {
    int sb = 0, st = 0;
    for (int i = 0; i < kFinThreads / 32; ++i) {
      sb += s_wsum[0][i];
      st += s_wsum[1][i];
    }
    s_before = sb;
    s_total = st;
  }
  uint64_t cand = 0;
  for (int i = 0; i < L; ++i) cand |= static_cast<uint64_t>(scored(a, b * L + i)) << i;
  __syncthreads();
  griddep_wait();   // the LM head's partials are complete and visible
  griddep_launch_dependents();
  const int rt = (s_total + 255) / 256;
  const int n_slots = rt > 0 ? (a.lm_grid / rt) * a.shares : 0;
  for (int i0 = 0; i0 < L; i0 += 32) {
    const int nr = min(32, L - i0);
    const int wpr = 32 / nr;   // warps per row
    const int i = i0 + warp / wpr;
    Acc q = acc_init();
    if (warp < nr * wpr && ((cand >> i) & 1)) {
      const int ai = s_before + __popcll(cand & ((1ull << i) - 1ull));
      const CommitPartial* pr = a.part + static_cast<size_t>(ai) * a.slots;
      for (int j = (warp % wpr) * 32 + lane; j < n_slots; j += wpr * 32) {
        const CommitPartial t = pr[j];
        q = merge(q, Acc{t.m, t.s, t.a, t.idx}, a.c);
      }
      q = warp_merge(q, a.c);
    }
    if (lane == 0) s_acc[warp] = q;
    __syncthreads();
    if (tid < nr) {
      const int ii = i0 + tid;
      const int r = b * L + ii;
      float conf = -CUDART_INF_F, ent = CUDART_INF_F;
      int tok = -1;
      if ((cand >> ii) & 1) {
        Acc f = acc_init();
        for (int w = tid * wpr; w < (tid + 1) * wpr; ++w) f = merge(f, s_acc[w], a.c);
        conf = acc_conf(f);
        ent = acc_entropy(f);
        tok = f.idx;
      }
      a.tok_out[r] = tok;
      a.conf_out[r] = conf;
      if (a.ent_out) a.ent_out[r] = ent;
      s_stat[ii] = a.rule == BDLM_COMMIT_ENTROPY_BOUNDED ? ent : conf;
    }
    __syncthreads();
  }
  if (warp == 0) {
    const uint64_t sel = decide_block_warp(a.rule, a.k, a.threshold, L, cand, s_stat, s_order,
                                           lane);
    uint8_t* co = a.commit_out + static_cast<size_t>(b) * L;
    for (int i = lane; i < L; i += 32) co[i] = static_cast<uint8_t>((sel >> i) & 1);
  }
}

}  // namespace

namespace {

// Clusters of two pair-kernel CTAs that fit the current device at once (0: none, or the
// query failed), queried once per device.
int pair_capacity() {
  constexpr int kMaxDev = 64;
  static int cap[kMaxDev];
  static bool known[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  if (!known[dev]) {
    int n = 0;
    const size_t smem = lm_conf_pair_smem();
    if (cudaFuncSetAttribute(lm_conf_pair_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) == cudaSuccess &&
        cudaFuncSetAttribute(lm_conf_pair_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, lm_conf_pair_kernel<false>, &cfg) != cudaSuccess)
        n = 0;
    }
    cudaGetLastError();   // a failed query leaves no sticky error: the single-CTA kernel runs
    cap[dev] = n;
    known[dev] = true;
  }
  return cap[dev];
}

}  // namespace

LmConfPlan plan_lm_conf(int max_rows, int H, int V, int num_sms) {
  LmConfPlan pl;
  pl.grid = num_sms > 0 ? num_sms : 1;
  pl.units = pl.grid;
  pl.slots = pl.grid;
  pl.m_tiles = (V + kConfN - 1) / kConfN;
  pl.max_row_tiles = (max_rows + kConfN - 1) / kConfN;
  pl.smem_bytes = lm_conf_smem();
  if (max_rows > kBM) {
    const int pairs = min(pair_capacity(), pl.grid / 2);
    if (pairs >= 1) {
      pl.pair = true;
      pl.grid = 2 * pairs;
      pl.units = pairs;
      pl.smem_bytes = lm_conf_pair_smem();
    }
  }
  pl.gather_bytes = static_cast<size_t>(max_rows) * H * 2;
  pl.part_bytes = static_cast<size_t>(max_rows) * pl.slots * sizeof(CommitPartial);
  return pl;
}

cudaError_t launch_lm_conf(const CUtensorMap& tm_w, const CUtensorMap& tm_h,
                           const int32_t* active_idx, const int32_t* n_active_dev, int max_rows,
                           int n_rows, int H, int V, float temperature, uint16_t* logits,
                           CommitPartial* part, const LmConfPlan& plan, int* err,
                           cudaStream_t stream, bool ent) {
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t ea = once_per_device(attr_done, [] {
    cudaError_t r = cudaFuncSetAttribute(lm_conf_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(lm_conf_smem()));
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(lm_conf_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(lm_conf_smem()));
  });
  if (ea != cudaSuccess) return ea;
  LmConfParams prm;
  prm.active_idx = active_idx;
  prm.n_active_dev = n_active_dev;
  prm.logits = logits;
  prm.part = part;
  prm.err = err;
  prm.n_active = max_rows;
  prm.n_rows = n_rows;
  prm.H = H;
  prm.V = V;
  prm.m_tiles = plan.m_tiles;
  prm.k_blocks = (H + kBK - 1) / kBK;
  prm.slots = plan.slots;
  prm.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  if (plan.pair) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return ent ? cudaLaunchKernelEx(&cfg, lm_conf_pair_kernel<true>, tm_w, tm_h, prm)
               : cudaLaunchKernelEx(&cfg, lm_conf_pair_kernel<false>, tm_w, tm_h, prm);
  }
  return ent ? launch_pdl(lm_conf_kernel<true>, dim3(plan.grid), dim3(kThreads), plan.smem_bytes,
                          stream, tm_w, tm_h, prm)
             : launch_pdl(lm_conf_kernel<false>, dim3(plan.grid), dim3(kThreads),
                          plan.smem_bytes, stream, tm_w, tm_h, prm);
}

cudaError_t launch_scored_gather(const uint16_t* hidden, const uint8_t* mask,
                                 const uint8_t* denoising, int B, int L, int H,
                                 uint16_t* gathered, int32_t* act, int32_t* n_act,
                                 cudaStream_t stream) {
  return launch_pdl(scored_gather_kernel, dim3(static_cast<unsigned>(B * L)), dim3(256), 0,
                    stream, hidden, mask, denoising, B * L, L, H, gathered, act, n_act);
}

cudaError_t launch_lm_commit_finalize(const uint8_t* mask, const uint8_t* denoising, int B, int L,
                                      const CommitPartial* part, const LmConfPlan& plan,
                                      float temperature, int rule, int k, float threshold,
                                      int32_t* tok_out, float* conf_out, float* ent_out,
                                      uint8_t* commit_out, cudaStream_t stream) {
  LmCommitArgs a;
  a.mask = mask;
  a.den = denoising;
  a.R = B * L;
  a.L = L;
  a.part = part;
  a.slots = plan.slots;
  a.lm_grid = plan.units;
  a.shares = 1;
  a.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  a.threshold = threshold;
  a.rule = rule;
  a.k = k;
  a.tok_out = tok_out;
  a.conf_out = conf_out;
  a.ent_out = ent_out;
  a.commit_out = commit_out;
  return launch_pdl(lm_commit_finalize_kernel, dim3(B), dim3(kFinThreads), 0, stream, a);
}

}  // namespace bdlm
