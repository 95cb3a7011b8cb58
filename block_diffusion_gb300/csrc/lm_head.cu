// Selective LM head for sm_103a: logits[r, :] = hidden[r, :] . W^T for the active rows only.
//
// Source: JetEngine notes (CLAUDE.md), "ModelRunner" (selective logits: the LM head runs
// only for DENOISING sequences, "saving ~25% of the largest GEMM") and "Optimization
// History" (opt23: LM head only on masked positions).
//
// Design:
//  * The active rows are first gathered into a contiguous [n_active, H] buffer (a few MB,
//    L2-resident), so both GEMM operands can be streamed by TMA tiles.
//  * The GEMM is computed transposed, logits^T tile = W_tile . Hg^T: 128 vocabulary rows of
//    W on the UMMA M side and up to 256 gathered rows on N, fp32 accumulation in tensor
//    memory, 64-wide K steps staged by TMA with 128-byte swizzle.
//  * Persistent CTAs (one per SM) walk the tiles vocabulary-tile-major, so the CTAs that run
//    together share W tiles and W streams from HBM about once.
//  * Two accumulators in tensor memory (2 x 256 columns) let the epilogue of one tile overlap
//    the MMAs of the next.  The epilogue rounds once (round-to-nearest-even) to bf16 and
//    scatters each column to its row's own slot of the logits.
//  * Threads: warp 0 TMA, warp 1 tensor memory + MMA issue, warps 2-5 epilogue.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;         // vocabulary rows per tile
constexpr int kBK = 64;          // K per stage (one 128-byte swizzle atom)
constexpr int kStages = 4;
constexpr uint32_t kTmemCols = 512;
constexpr int kEpiThreads = 128;

struct LmParams {
  const int32_t* active_idx;
  uint16_t* logits;
  int* err;
  int n_active, n_rows, H, V, bn, m_tiles, n_tiles, k_blocks;
};

__global__ void gather_rows_kernel(const uint16_t* __restrict__ hidden,
                                   const int32_t* __restrict__ active_idx, int n_active,
                                   int n_rows, int H, uint16_t* __restrict__ gathered,
                                   int* __restrict__ err) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.y;
  const int r = active_idx[i];
  const bool bad = r < 0 || r >= n_rows;
  if (bad && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, BDLM_DEVERR_ROW);
  const int nv = H / 8;
  const uint4* src = reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(bad ? 0 : r) * H);
  uint4* dst = reinterpret_cast<uint4*>(gathered + static_cast<size_t>(i) * H);
  for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < nv; v += gridDim.x * blockDim.x)
    dst[v] = bad ? make_uint4(0, 0, 0, 0) : __ldg(src + v);
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
lm_head_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
               const LmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int kABytes = kBM * kBK * 2;   // 16 KB
  constexpr int kBBytes = BN * kBK * 2;    // up to 32 KB
  constexpr int kStageBytes = kABytes + kBBytes;
  __shared__ uint64_t bar_full[kStages], bar_empty[kStages], bar_acc_full[2], bar_acc_empty[2];
  __shared__ uint64_t bar_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles_total = p.m_tiles * p.n_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bar_acc_full[a], 1);
      mbar_init(&bar_acc_empty[a], kEpiThreads);
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

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_h);
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles_total && ok; t += gridDim.x) {
        const int m = t / p.n_tiles;
        const int n = t % p.n_tiles;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!(ok = mbar_wait(&bar_empty[st], ph ^ 1, &abort_flag))) break;
          uint8_t* sa = base + st * kStageBytes;
          mbar_arrive_expect_tx(&bar_full[st], kStageBytes);
          tma_load_2d(sa, &tm_w, &bar_full[st], kb * kBK, m * kBM);
          tma_load_2d(sa + kABytes, &tm_h, &bar_full[st], kb * kBK, n * BN);
          if (++st == kStages) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      griddep_launch_dependents();  // every tile of this CTA is being loaded
      if (!ok) {
        int dummy = 0;
        for (int s = 0; s < kStages; ++s) mbar_wait(&bar_full[s], ph ^ (s < st ? 0 : 1), &dummy);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN, false, false);
      const uint32_t smem0 = smem_u32(base);
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      int i = 0;
      for (int t = blockIdx.x; t < n_tiles_total && ok; t += gridDim.x, ++i) {
        const int acc = i & 1;
        if (!(ok = mbar_wait(&bar_acc_empty[acc], ((i >> 1) & 1) ^ 1, &abort_flag))) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * 256;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!(ok = mbar_wait(&bar_full[st], ph, &abort_flag))) break;
          tc_fence_after();
          const uint32_t sa = smem0 + st * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc(sa + kABytes + kk * 32, 16, 1024);
            umma_bf16(d, ad, bd, kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bar_empty[st]);
          if (++st == kStages) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&bar_acc_full[acc]);
      }
      umma_commit(&bar_done);
    }
  } else {
    const int q4 = warp & 3;
    const int x = (q4 << 5) | lane;  // tensor-memory lane = vocabulary row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    bool ok = true;
    int i = 0;
    for (int t = blockIdx.x; t < n_tiles_total && ok; t += gridDim.x, ++i) {
      const int m = t / p.n_tiles;
      const int n = t % p.n_tiles;
      const int acc = i & 1;
      if (!(ok = mbar_wait(&bar_acc_full[acc], (i >> 1) & 1, &abort_flag))) break;
      tc_fence_after();
      const int v = m * kBM + x;
      const bool v_ok = v < p.V;
      const uint32_t d = tmem + acc * 256 + lane_off;
      const int r0 = n * BN;
#pragma unroll 1
      for (int cg = 0; cg < BN / 16; ++cg) {
        uint32_t r[16];
        tmem_ld16(d + cg * 16, r);
        tmem_wait_ld();
        tmem_regs_ready(r);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int rr = r0 + cg * 16 + k;
          if (rr < p.n_active && v_ok) {
            const int row = __ldg(p.active_idx + rr);
            if (row < 0 || row >= p.n_rows) continue;  // flagged by the gather
            p.logits[static_cast<size_t>(row) * p.V + v] =
                __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[k])));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_acc_empty[acc]);
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

template <int BN>
size_t lm_smem() {
  return 1024 + static_cast<size_t>(kStages) * (kBM * kBK * 2 + BN * kBK * 2);
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap& tw, const CUtensorMap& th, const LmParams& prm, int grid,
                      cudaStream_t stream) {
  static bool attr_set = false;
  const size_t smem = lm_smem<BN>();
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(lm_head_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(lm_head_kernel<BN>, dim3(grid), dim3(kThreads), smem, stream, tw, th, prm);
}

}  // namespace

LmHeadPlan plan_lm_head(int n_active, int H, int V, int num_sms) {
  LmHeadPlan pl;
  pl.bn = n_active <= 64 ? 64 : n_active <= 128 ? 128 : 256;
  pl.m_tiles = (V + kBM - 1) / kBM;
  pl.n_tiles = (n_active + pl.bn - 1) / pl.bn;
  const int tiles = pl.m_tiles * pl.n_tiles;
  pl.grid = tiles < num_sms ? tiles : num_sms;
  pl.smem_bytes = pl.bn == 64 ? lm_smem<64>() : pl.bn == 128 ? lm_smem<128>() : lm_smem<256>();
  pl.gather_bytes = static_cast<size_t>(n_active) * H * 2;
  return pl;
}

cudaError_t launch_gather_rows(const uint16_t* hidden, const int32_t* active_idx, int n_active,
                               int n_rows, int H, uint16_t* gathered, int* err,
                               cudaStream_t stream) {
  const int nv = H / 8;
  const int threads = nv < 256 ? ((nv + 31) / 32) * 32 : 256;
  dim3 grid((nv + threads - 1) / threads, n_active);
  return launch_pdl(gather_rows_kernel, grid, dim3(threads), 0, stream, hidden, active_idx,
                    n_active, n_rows, H, gathered, err);
}

cudaError_t launch_lm_head(const CUtensorMap& tm_w, const CUtensorMap& tm_h,
                           const int32_t* active_idx, int n_active, int n_rows, int H, int V,
                           uint16_t* logits, const LmHeadPlan& plan, int* err,
                           cudaStream_t stream) {
  LmParams prm;
  prm.active_idx = active_idx;
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
  switch (plan.bn) {
    case 64: return launch_bn<64>(tm_w, tm_h, prm, plan.grid, stream);
    case 128: return launch_bn<128>(tm_w, tm_h, prm, plan.grid, stream);
    default: return launch_bn<256>(tm_w, tm_h, prm, plan.grid, stream);
  }
}

}  // namespace bdlm
