// Confidence + commit of one denoising step: one pass over the vocabulary.
//
// Source: JetEngine notes (CLAUDE.md), "Remasking Strategies" (low_confidence_dynamic) and
// "Remaining Optimization Avenues" (a fused postprocess kernel); dInfer blog, "Algorithmic
// Innovations" (threshold decoding).  Per masked row: argmax token (lowest index on ties),
// max softmax probability at temperature T; per block: commit every masked position at or
// above the threshold, else the single most confident one.
//
// Layout of the work: each row of logits is cut into S items of kItem elements; warps take
// items from a global atomic counter (any order, so the load balances whatever the mask),
// stream the item with 16-byte loads keeping a running (max, sum of exp, first argmax) per
// lane, merge the lanes with shuffles and write one partial.  The last warp to finish a row
// (atomic counter) merges the row's S partials in item order, writes tok/conf, and the last
// row to finish a block decides the block's commit.  Nothing waits on another warp; every
// counter is reset by whoever consumed it, the work counter by the last warp to leave.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;   // 16-byte vectors in flight per lane
constexpr int kItem = 8192;  // logits per work item (a multiple of 8)

struct Acc {
  float m;    // running max (raw logit)
  float s;    // sum of exp2((x - m) * c)
  int idx;    // first index of the max
};

__device__ __forceinline__ Acc merge(Acc a, Acc b, float c) {
  if (b.m == -CUDART_INF_F) return a;
  if (a.m == -CUDART_INF_F) return b;
  Acc o;
  o.m = fmaxf(a.m, b.m);
  o.s = a.s * exp2f((a.m - o.m) * c) + b.s * exp2f((b.m - o.m) * c);
  const int ia = (a.m == o.m) ? a.idx : 0x7FFFFFFF;
  const int ib = (b.m == o.m) ? b.idx : 0x7FFFFFFF;
  o.idx = min(ia, ib);
  return o;
}

// Adds elements x[0..n) (first index `base`) to the accumulator.
__device__ __forceinline__ void absorb(Acc& a, const float* x, int n, int base, float c) {
  float lm = x[0];
  int li = 0;
#pragma unroll
  for (int k = 1; k < n; ++k) {
    if (x[k] > lm) { lm = x[k]; li = k; }
  }
  if (lm > a.m) {
    a.s = (a.m == -CUDART_INF_F) ? 0.f : a.s * exp2f((a.m - lm) * c);
    a.m = lm;
    a.idx = base + li;
  }
  const float mc = a.m * c;
  float t = 0.f;
#pragma unroll
  for (int k = 0; k < n; ++k) t += exp2f(fmaf(x[k], c, -mc));
  a.s += t;
}

__device__ __forceinline__ float bf16f(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// The last row of block b to finish decides the block's commit (one lane).
__device__ void decide_block(int b, int L, const uint8_t* __restrict__ mask, const float* conf_out,
                             uint8_t* __restrict__ commit_out, int* __restrict__ blk_cnt,
                             float threshold) {
  __threadfence();
  const volatile float* cf = conf_out + static_cast<size_t>(b) * L;
  const uint8_t* mk = mask + static_cast<size_t>(b) * L;
  uint8_t* co = commit_out + static_cast<size_t>(b) * L;
  int any_masked = 0, any_commit = 0, best = -1;
  float best_c = 0.f;
  for (int i = 0; i < L; ++i) {
    uint8_t cm = 0;
    if (mk[i]) {
      const float ci = cf[i];
      any_masked = 1;
      if (ci >= threshold) { cm = 1; any_commit = 1; }
      if (best < 0 || ci > best_c) { best = i; best_c = ci; }
    }
    co[i] = cm;
  }
  if (any_masked && !any_commit) co[best] = 1;
  blk_cnt[b] = 0;
}

__device__ __forceinline__ Acc warp_merge(Acc a, float c) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Acc o;
    o.m = __shfl_xor_sync(0xffffffffu, a.m, off);
    o.s = __shfl_xor_sync(0xffffffffu, a.s, off);
    o.idx = __shfl_xor_sync(0xffffffffu, a.idx, off);
    a = merge(a, o, c);
  }
  return a;
}

__global__ void __launch_bounds__(kThreads)
commit_kernel(const uint16_t* __restrict__ logits, const uint8_t* __restrict__ mask, int L,
              int V, int S, int total_items, int total_warps, float threshold, float c,
              int32_t* __restrict__ tok_out, float* __restrict__ conf_out,
              uint8_t* __restrict__ commit_out, CommitPartial* __restrict__ part,
              int* __restrict__ row_cnt, int* __restrict__ blk_cnt, int* __restrict__ work) {
  const int lane = threadIdx.x & 31;
  int item = 0;
  if (lane == 0) item = atomicAdd(work, 1);
  item = __shfl_sync(0xffffffffu, item, 0);
  while (item < total_items) {
    int next = 0;
    if (lane == 0) next = atomicAdd(work, 1);  // the next grab overlaps this item
    const int r = item / S;
    const int s = item - r * S;
    const int b = r / L;
    if (!mask[r]) {
      if (s == 0 && lane == 0) {
        tok_out[r] = -1;
        conf_out[r] = -CUDART_INF_F;
        __threadfence();
        if (atomicAdd(blk_cnt + b, 1) == L - 1)
          decide_block(b, L, mask, conf_out, commit_out, blk_cnt, threshold);
      }
    } else {
      Acc a{-CUDART_INF_F, 0.f, 0x7FFFFFFF};
      const int e0 = s * kItem;
      const int e1 = min(V, e0 + kItem);
      const uint16_t* row = logits + static_cast<size_t>(r) * V;
      // scalar head up to a 16-byte boundary, vector body, scalar tail
      const uintptr_t addr0 = reinterpret_cast<uintptr_t>(row + e0);
      int head = static_cast<int>(((16 - (addr0 & 15)) & 15) >> 1);
      head = min(head, e1 - e0);
      const int vb = e0 + head;
      const int nvec = (e1 - vb) >> 3;
      const int tail0 = vb + nvec * 8;
      if (lane < head) {
        float x = bf16f(row[e0 + lane]);
        absorb(a, &x, 1, e0 + lane, c);
      }
      const uint4* vp = reinterpret_cast<const uint4*>(row + vb);
      for (int v0 = 0; v0 < nvec; v0 += kUnroll * 32) {
        uint4 w[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) w[u] = __ldcs(vp + v);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) {
            float x[8];
            x[0] = bf16_lo(w[u].x); x[1] = bf16_hi(w[u].x);
            x[2] = bf16_lo(w[u].y); x[3] = bf16_hi(w[u].y);
            x[4] = bf16_lo(w[u].z); x[5] = bf16_hi(w[u].z);
            x[6] = bf16_lo(w[u].w); x[7] = bf16_hi(w[u].w);
            absorb(a, x, 8, vb + v * 8, c);
          }
        }
      }
      if (tail0 + lane < e1) {
        float x = bf16f(row[tail0 + lane]);
        absorb(a, &x, 1, tail0 + lane, c);
      }
      a = warp_merge(a, c);
      int last = 0;
      if (lane == 0) {
        part[static_cast<size_t>(r) * S + s] = CommitPartial{a.m, a.s, a.idx, 0};
        __threadfence();
        last = (atomicAdd(row_cnt + r, 1) == S - 1);
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        // merge the row's partials in a fixed order (lanes then tree) -> deterministic
        __threadfence();
        const volatile CommitPartial* pr = part + static_cast<size_t>(r) * S;
        Acc f{-CUDART_INF_F, 0.f, 0x7FFFFFFF};
        for (int k0 = 0; k0 < S; k0 += 32) {
          Acc q{-CUDART_INF_F, 0.f, 0x7FFFFFFF};
          if (k0 + lane < S) q = Acc{pr[k0 + lane].m, pr[k0 + lane].s, pr[k0 + lane].idx};
          q = warp_merge(q, c);
          f = merge(f, q, c);
        }
        if (lane == 0) {
          tok_out[r] = f.idx;
          conf_out[r] = 1.0f / f.s;
          row_cnt[r] = 0;
          __threadfence();
          if (atomicAdd(blk_cnt + b, 1) == L - 1)
            decide_block(b, L, mask, conf_out, commit_out, blk_cnt, threshold);
        }
      }
    }
    item = __shfl_sync(0xffffffffu, next, 0);
  }
  // the last warp to leave resets the work counter for the next launch
  if (lane == 0) {
    __threadfence();
    if (atomicAdd(work + 1, 1) == total_warps - 1) {
      work[0] = 0;
      work[1] = 0;
    }
  }
}

__global__ void apply_commit_kernel(uint8_t* __restrict__ mask, const uint8_t* __restrict__ commit,
                                    int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n && commit[i]) mask[i] = 0;
}

}  // namespace

CommitPlan plan_commit(int B, int L, int V, int num_sms) {
  CommitPlan p;
  const long rows = static_cast<long>(B) * L;
  p.S = (V + kItem - 1) / kItem;
  p.chunk = kItem;
  p.total_items = static_cast<long long>(rows) * p.S;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, commit_kernel, kThreads, 0) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  long long grid = static_cast<long long>(num_sms) * per_sm;
  const long long warps_needed = (p.total_items + 0) / 1;
  if (grid * (kThreads / 32) > warps_needed)
    grid = (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
  if (grid < 1) grid = 1;
  p.grid = static_cast<int>(grid);
  p.part_bytes = static_cast<size_t>(rows) * p.S * sizeof(CommitPartial);
  p.row_cnt_bytes = static_cast<size_t>(rows) * sizeof(int);
  p.blk_cnt_bytes = static_cast<size_t>(B) * sizeof(int);
  p.work_bytes = 2 * sizeof(int);
  return p;
}

cudaError_t launch_commit(const uint16_t* logits, const uint8_t* mask, int B, int L, int V,
                          float threshold, float temperature, int32_t* tok_out, float* conf_out,
                          uint8_t* commit_out, const CommitPlan& plan, CommitPartial* part,
                          int* row_cnt, int* blk_cnt, int* work, cudaStream_t stream) {
  (void)B;
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  commit_kernel<<<plan.grid, kThreads, 0, stream>>>(
      logits, mask, L, V, plan.S, static_cast<int>(plan.total_items), plan.grid * (kThreads / 32),
      threshold, c, tok_out, conf_out, commit_out, part, row_cnt, blk_cnt, work);
  return cudaGetLastError();
}

cudaError_t launch_apply_commit(uint8_t* mask, const uint8_t* commit, int n, cudaStream_t stream) {
  apply_commit_kernel<<<(n + 255) / 256, 256, 0, stream>>>(mask, commit, n);
  return cudaGetLastError();
}

}  // namespace bdlm
