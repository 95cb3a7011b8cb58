// Selective LM head for sm_103a: logits[r, :] = hidden[r, :] . W^T for the active rows only.
//
// Source: JetEngine notes (CLAUDE.md), "ModelRunner" (selective logits: the LM head runs
// only for DENOISING sequences, "saving ~25% of the largest GEMM") and "Optimization
// History" (opt23: LM head only on masked positions).
//
// Design:
//  * The active rows are first gathered into a contiguous [n_active, H] buffer (a few MB,
//    L2-resident), so both GEMM operands can be streamed by TMA tiles.
//  * The GEMM is computed transposed, logits^T tile = W_tile . Hg^T.  A CTA tile is 256
//    vocabulary rows of W (two UMMAs of M = 128 that share one staged block of gathered
//    rows) by up to 256 gathered rows on N (the rows split evenly over as few N tiles as fit,
//    rounded to 16), fp32 accumulation in tensor memory, 64-wide K steps staged by TMA with
//    128-byte swizzle.  Sharing the row block between two W sub-tiles halves the L2 -> SM
//    traffic of the rows, which is what held the W stream below HBM speed.
//  * W (the HBM stream) and the gathered rows (L2-resident) have separate shared-memory
//    rings with their own producers, so the W ring can be deep: HBM needs tens of KB in
//    flight per SM.
//  * Persistent CTAs (one per SM) walk the tiles vocabulary-tile-major, so the CTAs that run
//    together share W tiles and W streams from HBM about once.
//  * Tensor memory holds the two sub-tile accumulators of one tile (N <= 256), or of two
//    tiles (N <= 128) so that the epilogue of one tile overlaps the MMAs of the next.  The
//    epilogue rounds once (round-to-nearest-even) to bf16 and scatters each column to its
//    row's own slot of the logits.
//  * Threads: warp 0 W loads, warp 1 tensor memory + MMA issue, then the epilogue warps
//    (several per tensor-memory lane quadrant, each draining a share of the columns), then
//    the gathered-row loads.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "lm_common.cuh"
#include "ptx.cuh"

namespace bdlm {
namespace {

using namespace lm;

// Per largest tile width: W stages of 32 KB, row stages of BN_MAX x 128 B (225 KB of shared
// memory in each case), and the tensor-memory columns of one sub-tile accumulator (kCols)
// with the number of tiles whose accumulators fit at once (kBufs).
template <int BN_MAX> struct Cfg;
template <> struct Cfg<64> { static constexpr int kW = 6, kH = 4, kCols = 128, kBufs = 2; };
template <> struct Cfg<128> { static constexpr int kW = 5, kH = 4, kCols = 128, kBufs = 2; };
template <> struct Cfg<256> { static constexpr int kW = 4, kH = 3, kCols = 256, kBufs = 1; };

struct LmParams {
  const int32_t* active_idx;
  const int32_t* n_active_dev;  // if set: the active-row count, read on the device (<= n_active)
  uint16_t* logits;
  int* err;
  int n_active, n_rows, H, V, bn, m_tiles, n_tiles, k_blocks;
};

// Active rows of this launch: the device-side count when there is one (clamped to the
// planned maximum), else the planned count.  Read after the grid dependency is resolved.
__device__ __forceinline__ int active_rows(const LmParams& p) {
  if (p.n_active_dev == nullptr) return p.n_active;
  return min(max(*p.n_active_dev, 0), p.n_active);
}

__global__ void gather_rows_kernel(const uint16_t* __restrict__ hidden,
                                   const int32_t* __restrict__ active_idx, int n_active,
                                   const int32_t* __restrict__ n_active_dev, int n_rows, int H,
                                   uint16_t* __restrict__ gathered, int* __restrict__ err) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.y;
  if (n_active_dev != nullptr && i >= min(max(*n_active_dev, 0), n_active)) return;
  const int r = active_idx[i];
  const bool bad = r < 0 || r >= n_rows;
  if (bad && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, BDLM_DEVERR_ROW);
  const int nv = H / 8;
  const uint4* src = reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(bad ? 0 : r) * H);
  uint4* dst = reinterpret_cast<uint4*>(gathered + static_cast<size_t>(i) * H);
  for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < nv; v += gridDim.x * blockDim.x)
    dst[v] = bad ? make_uint4(0, 0, 0, 0) : __ldg(src + v);
}

// Producer of one ring: loads box (kb * kBK, row0(t)) of `tm` (`box_bytes` each) into slots
// STRIDE bytes apart, for every tile and K step.  After a timeout it waits (bounded) for the
// copies it already issued, then returns false.
// For W, a stage is the kSub boxes of the tile's sub-tiles (box_bytes each, kWBox apart).
template <int NSTAGES, int STRIDE, bool IS_W>
__device__ bool produce(const CUtensorMap* tm, uint8_t* ring, uint32_t box_bytes,
                        uint64_t* full, uint64_t* empty, const LmParams& p, int n_tiles,
                        int n_tiles_total, int* abort_flag) {
  tma_prefetch_desc(tm);
  RingPos pos;
  bool ok = true;
  constexpr int kBoxes = IS_W ? kSub : 1;
  for (int t = blockIdx.x; t < n_tiles_total && ok; t += gridDim.x) {
    const int row0 = IS_W ? (t / n_tiles) * (kSub * kBM) : (t % n_tiles) * p.bn;
    for (int kb = 0; kb < p.k_blocks; ++kb) {
      if (!(ok = mbar_wait(&empty[pos.slot], pos.phase ^ 1, abort_flag))) break;
      mbar_arrive_expect_tx(&full[pos.slot], kBoxes * box_bytes);
#pragma unroll
      for (int b = 0; b < kBoxes; ++b)   // boxes past the vocabulary read as zeros
        tma_load_2d(ring + pos.slot * STRIDE + b * kWBox, tm, &full[pos.slot], kb * kBK,
                    row0 + b * kBM);
      pos.advance(NSTAGES);
    }
  }
  if (!ok) {
    // slots below pos.slot were last filled in the current phase, the others in the previous
    int dummy = 0;
    for (int s = 0; s < NSTAGES; ++s)
      mbar_wait(&full[s], pos.phase ^ (s < pos.slot ? 0u : 1u), &dummy);
  }
  return ok;
}

template <int BN_MAX>
__global__ void __launch_bounds__(kThreads, 1)
lm_head_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
               const LmParams p) {
  constexpr int kWS = Cfg<BN_MAX>::kW;
  constexpr int kHS = Cfg<BN_MAX>::kH;
  constexpr int kCols = Cfg<BN_MAX>::kCols;
  constexpr int kBufs = Cfg<BN_MAX>::kBufs;
  constexpr int kHStage = BN_MAX * kBK * 2;
  static_assert(kSub * kCols * kBufs <= static_cast<int>(kTmemCols), "tensor memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* wring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t* hring = wring + kWS * kWBytes;
  __shared__ uint64_t w_full[kWS], w_empty[kWS], h_full[kHS], h_empty[kHS];
  __shared__ uint64_t acc_full[kBufs], acc_empty[kBufs], bar_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int s_rows[256];   // logits row of each column of the current tile (-1: none)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t h_bytes = static_cast<uint32_t>(p.bn) * kBK * 2;   // one box of rows

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWS; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 1);
    }
    for (int s = 0; s < kHS; ++s) {
      mbar_init(&h_full[s], 1);
      mbar_init(&h_empty[s], 1);
    }
    for (int a = 0; a < kBufs; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiThreads);
    }
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
  // tiles of the N tiles that hold active rows only
  const int n_act = active_rows(p);
  const int n_tiles = (n_act + p.bn - 1) / p.bn;
  const int n_tiles_total = p.m_tiles * n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      produce<kWS, kWBytes, true>(&tm_w, wring, kWBox, w_full, w_empty, p, n_tiles,
                                  n_tiles_total, &abort_flag);
      griddep_launch_dependents();  // every W tile of this CTA is being loaded
    }
  } else if (warp == kRowWarp) {
    if (lane == 0)
      produce<kHS, kHStage, false>(&tm_h, hring, h_bytes, h_full, h_empty, p, n_tiles,
                                   n_tiles_total, &abort_flag);
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, p.bn, false, false);
      const uint32_t w0 = smem_u32(wring), h0 = smem_u32(hring);
      RingPos wp, hp;
      bool ok = true;
      int i = 0;
      for (int t = blockIdx.x; t < n_tiles_total && ok; t += gridDim.x, ++i) {
        const int acc = i % kBufs;
        if (!(ok = mbar_wait(&acc_empty[acc], ((i / kBufs) & 1) ^ 1, &abort_flag))) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * (kSub * kCols);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!(ok = mbar_wait(&w_full[wp.slot], wp.phase, &abort_flag))) break;
          if (!(ok = mbar_wait(&h_full[hp.slot], hp.phase, &abort_flag))) break;
          tc_fence_after();
          const uint32_t sa = w0 + wp.slot * kWBytes;
          const uint32_t sb = h0 + hp.slot * kHStage;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t bd = smem_desc(sb + kk * 32, 16, 1024);
#pragma unroll
            for (int sub = 0; sub < kSub; ++sub) {
              const uint64_t ad = smem_desc(sa + sub * kWBox + kk * 32, 16, 1024);
              umma_bf16(d + sub * kCols, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            }
          }
          umma_commit(&w_empty[wp.slot]);
          umma_commit(&h_empty[hp.slot]);
          wp.advance(kWS);
          hp.advance(kHS);
        }
        if (!ok) break;
        umma_commit(&acc_full[acc]);
      }
      umma_commit(&bar_done);
    }
  } else {
    const int q4 = warp & 3;          // tensor-memory lanes 32*q4 .. 32*q4+31
    const int part = (warp - 2) >> 2;  // which share of the column groups this warp drains
    const int et = (warp - 2) * 32 + lane;
    const int x = (q4 << 5) | lane;  // tensor-memory lane = vocabulary row within a sub-tile
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int n_groups = p.bn / 16;
    const int cg_begin = n_groups * part / (kEpiWarps / 4);
    const int cg_end = n_groups * (part + 1) / (kEpiWarps / 4);
    // Every epilogue warp runs every tile iteration (after a timeout without work), so the
    // named barriers below always see every epilogue warp.
    bool ok = true;
    int i = 0;
    for (int t = blockIdx.x; t < n_tiles_total; t += gridDim.x, ++i) {
      const int m = t / n_tiles;
      const int n = t % n_tiles;
      const int acc = i % kBufs;
      const int r0 = n * p.bn;
      // the tile's logits rows, read once (rows past n_active or out of range: -1, skipped;
      // an out-of-range id is flagged by the gather)
      named_barrier(1, kEpiThreads);   // the previous tile's readers are done
      for (int j = et; j < p.bn; j += kEpiThreads) {
        const int rr = r0 + j;
        const int row = rr < n_act ? __ldg(p.active_idx + rr) : -1;
        s_rows[j] = (row >= 0 && row < p.n_rows) ? row : -1;
      }
      named_barrier(1, kEpiThreads);
      if (!ok || !(ok = mbar_wait_warp(&acc_full[acc], (i / kBufs) & 1, &abort_flag))) continue;
      tc_fence_after();
      const int v0 = m * (kSub * kBM) + x;       // sub-tile 0; sub-tile 1 is kBM further
      const bool ok0 = v0 < p.V, ok1 = v0 + kBM < p.V;
      const uint32_t d = tmem + acc * (kSub * kCols) + lane_off;
#pragma unroll 1
      for (int cg = cg_begin; cg < cg_end; ++cg) {
        uint32_t r[kSub][16];
        tmem_ld16(d + cg * 16, r[0]);
        tmem_ld16(d + kCols + cg * 16, r[1]);
        tmem_wait_ld();
        tmem_regs_ready(r[0]);
        tmem_regs_ready(r[1]);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int row = s_rows[cg * 16 + k];
          if (row < 0) continue;
          uint16_t* dst = p.logits + static_cast<size_t>(row) * p.V + v0;
          if (ok0) dst[0] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[0][k])));
          if (ok1)
            dst[kBM] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[1][k])));
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);
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

template <int BN_MAX>
size_t lm_smem() {
  return 1024 + static_cast<size_t>(Cfg<BN_MAX>::kW) * kWBytes +
         static_cast<size_t>(Cfg<BN_MAX>::kH) * BN_MAX * kBK * 2;
}

template <int BN_MAX>
cudaError_t launch_bn(const CUtensorMap& tw, const CUtensorMap& th, const LmParams& prm, int grid,
                      cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  const size_t smem = lm_smem<BN_MAX>();
  cudaError_t e = once_per_device(attr_done, [smem] {
    return cudaFuncSetAttribute(lm_head_kernel<BN_MAX>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem));
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(lm_head_kernel<BN_MAX>, dim3(grid), dim3(kThreads), smem, stream, tw, th,
                    prm);
}

}  // namespace

LmHeadPlan plan_lm_head(int n_active, int H, int V, int num_sms) {
  LmHeadPlan pl;
  // as few N tiles of at most 256 rows as cover the rows, split evenly, multiple of 16
  pl.n_tiles = (n_active + 255) / 256;
  if (pl.n_tiles < 1) pl.n_tiles = 1;
  const int per = (n_active + pl.n_tiles - 1) / pl.n_tiles;
  pl.bn = per <= 16 ? 16 : (per + 15) / 16 * 16;
  pl.bn_max = pl.bn <= 64 ? 64 : pl.bn <= 128 ? 128 : 256;
  pl.m_tiles = (V + kSub * kBM - 1) / (kSub * kBM);   // CTA tiles of 256 vocabulary rows
  const int tiles = pl.m_tiles * pl.n_tiles;
  pl.grid = tiles < num_sms ? tiles : num_sms;
  pl.smem_bytes = pl.bn_max == 64 ? lm_smem<64>() : pl.bn_max == 128 ? lm_smem<128>()
                                                                     : lm_smem<256>();
  pl.gather_bytes = static_cast<size_t>(n_active) * H * 2;
  return pl;
}

cudaError_t launch_gather_rows(const uint16_t* hidden, const int32_t* active_idx, int n_active,
                               const int32_t* n_active_dev, int n_rows, int H,
                               uint16_t* gathered, int* err, cudaStream_t stream) {
  const int nv = H / 8;
  const int threads = nv < 256 ? ((nv + 31) / 32) * 32 : 256;
  dim3 grid((nv + threads - 1) / threads, n_active);
  return launch_pdl(gather_rows_kernel, grid, dim3(threads), 0, stream, hidden, active_idx,
                    n_active, n_active_dev, n_rows, H, gathered, err);
}

cudaError_t launch_lm_head(const CUtensorMap& tm_w, const CUtensorMap& tm_h,
                           const int32_t* active_idx, int n_active,
                           const int32_t* n_active_dev, int n_rows, int H, int V,
                           uint16_t* logits, const LmHeadPlan& plan, int* err,
                           cudaStream_t stream) {
  LmParams prm;
  prm.active_idx = active_idx;
  prm.n_active_dev = n_active_dev;
  prm.logits = logits;
  prm.err = err;
  prm.n_active = n_active;
  prm.n_rows = n_rows;
  prm.H = H;
  prm.V = V;
  prm.bn = plan.bn;
  prm.m_tiles = plan.m_tiles;
  prm.n_tiles = plan.n_tiles;
  prm.k_blocks = (H + kBK - 1) / kBK;
  switch (plan.bn_max) {
    case 64: return launch_bn<64>(tm_w, tm_h, prm, plan.grid, stream);
    case 128: return launch_bn<128>(tm_w, tm_h, prm, plan.grid, stream);
    default: return launch_bn<256>(tm_w, tm_h, prm, plan.grid, stream);
  }
}

}  // namespace bdlm
