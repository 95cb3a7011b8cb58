// Confidence + commit of one denoising step: one pass over the vocabulary.
//
// Source: JetEngine notes (CLAUDE.md), "Remasking Strategies" (low_confidence_dynamic) and
// "Remaining Optimization Avenues" (a fused postprocess kernel); dInfer blog, "Algorithmic
// Innovations" (threshold decoding).  Per masked row: argmax token (lowest index on ties),
// max softmax probability at temperature T; per block: commit every masked position at or
// above the threshold, else the single most confident one.
//
// Layout of the work: grid (B*L, S).  CTA (r, s) streams elements [s*chunk, (s+1)*chunk)
// of logits row r with 16-byte loads, keeping a running (max, sum of exp, first argmax)
// per thread; the CTA merges its threads and writes one partial.  The last CTA to finish
// a row (atomic counter) merges the row's S partials in split order, writes tok/conf, and
// the last row to finish a block decides the block's commit.  Nothing waits on another
// CTA; counters are reset by the CTA that consumed them.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 16-byte vectors in flight per thread per iteration

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

__global__ void __launch_bounds__(kThreads)
commit_kernel(const uint16_t* __restrict__ logits, const uint8_t* __restrict__ mask, int L,
              int V, int S, int chunk, float threshold, float c, int32_t* __restrict__ tok_out,
              float* __restrict__ conf_out, uint8_t* __restrict__ commit_out,
              CommitPartial* __restrict__ part, int* __restrict__ row_cnt,
              int* __restrict__ blk_cnt) {
  const int r = blockIdx.x;
  const int s = blockIdx.y;
  const int b = r / L;
  const int tid = threadIdx.x;
  __shared__ Acc red[kThreads / 32];
  __shared__ int last_flag;

  if (!mask[r]) {
    if (s != 0) return;
    if (tid == 0) {
      tok_out[r] = -1;
      conf_out[r] = -CUDART_INF_F;
      __threadfence();
      last_flag = (atomicAdd(blk_cnt + b, 1) == L - 1);
    }
    __syncthreads();
    if (!last_flag) return;
  } else {
    Acc a{-CUDART_INF_F, 0.f, 0x7FFFFFFF};
    const int e0 = s * chunk;
    const int e1 = min(V, e0 + chunk);
    const uint16_t* row = logits + static_cast<size_t>(r) * V;
    // scalar head up to a 16-byte boundary, vector body, scalar tail
    const uintptr_t addr0 = reinterpret_cast<uintptr_t>(row + e0);
    int head = static_cast<int>(((16 - (addr0 & 15)) & 15) >> 1);
    head = min(head, e1 - e0);
    const int vb = e0 + head;                 // first element of the vector body
    const int nvec = (e1 - vb) >> 3;          // 8 elements per vector
    const int tail0 = vb + nvec * 8;
    if (tid < head) {
      float x = bf16f(row[e0 + tid]);
      absorb(a, &x, 1, e0 + tid, c);
    }
    const uint4* vp = reinterpret_cast<const uint4*>(row + vb);
    int v = tid;
    for (; v + (kUnroll - 1) * kThreads < nvec; v += kUnroll * kThreads) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) w[u] = __ldcs(vp + v + u * kThreads);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        float x[8];
        x[0] = bf16_lo(w[u].x); x[1] = bf16_hi(w[u].x);
        x[2] = bf16_lo(w[u].y); x[3] = bf16_hi(w[u].y);
        x[4] = bf16_lo(w[u].z); x[5] = bf16_hi(w[u].z);
        x[6] = bf16_lo(w[u].w); x[7] = bf16_hi(w[u].w);
        absorb(a, x, 8, vb + (v + u * kThreads) * 8, c);
      }
    }
    for (; v < nvec; v += kThreads) {
      const uint4 w = __ldcs(vp + v);
      float x[8];
      x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x);
      x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
      x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z);
      x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
      absorb(a, x, 8, vb + v * 8, c);
    }
    if (tail0 + tid < e1) {
      float x = bf16f(row[tail0 + tid]);
      absorb(a, &x, 1, tail0 + tid, c);
    }
    // warp merge, then CTA merge
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      Acc o;
      o.m = __shfl_xor_sync(0xffffffffu, a.m, off);
      o.s = __shfl_xor_sync(0xffffffffu, a.s, off);
      o.idx = __shfl_xor_sync(0xffffffffu, a.idx, off);
      a = merge(a, o, c);
    }
    if ((tid & 31) == 0) red[tid >> 5] = a;
    __syncthreads();
    if (tid == 0) {
      Acc t = red[0];
      for (int w = 1; w < kThreads / 32; ++w) t = merge(t, red[w], c);
      part[static_cast<size_t>(r) * S + s] = CommitPartial{t.m, t.s, t.idx, 0};
      __threadfence();
      int row_last = (atomicAdd(row_cnt + r, 1) == S - 1);
      int blk_last = 0;
      if (row_last) {
        __threadfence();
        Acc f{-CUDART_INF_F, 0.f, 0x7FFFFFFF};
        const volatile CommitPartial* pr = part + static_cast<size_t>(r) * S;
        for (int k = 0; k < S; ++k) {
          Acc q{pr[k].m, pr[k].s, pr[k].idx};
          f = merge(f, q, c);
        }
        tok_out[r] = f.idx;
        conf_out[r] = 1.0f / f.s;
        row_cnt[r] = 0;
        __threadfence();
        blk_last = (atomicAdd(blk_cnt + b, 1) == L - 1);
      }
      last_flag = blk_last;
    }
    __syncthreads();
    if (!last_flag) return;
  }
  // The last row of block b to finish decides the block's commit.
  if (tid == 0) {
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
}

__global__ void apply_commit_kernel(uint8_t* __restrict__ mask, const uint8_t* __restrict__ commit,
                                    int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n && commit[i]) mask[i] = 0;
}

}  // namespace

CommitPlan plan_commit(int B, int L, int V) {
  CommitPlan p;
  const long rows = static_cast<long>(B) * L;
  long S = (2048 + rows - 1) / rows;
  const long max_s = (V + 8191) / 8192;
  if (S > max_s) S = max_s;
  if (S < 1) S = 1;
  long chunk = (V + S - 1) / S;
  chunk = (chunk + 7) / 8 * 8;
  S = (V + chunk - 1) / chunk;
  p.S = static_cast<int>(S);
  p.chunk = static_cast<int>(chunk);
  p.part_bytes = static_cast<size_t>(rows) * S * sizeof(CommitPartial);
  p.row_cnt_bytes = static_cast<size_t>(rows) * sizeof(int);
  p.blk_cnt_bytes = static_cast<size_t>(B) * sizeof(int);
  return p;
}

cudaError_t launch_commit(const uint16_t* logits, const uint8_t* mask, int B, int L, int V,
                          float threshold, float temperature, int32_t* tok_out, float* conf_out,
                          uint8_t* commit_out, const CommitPlan& plan, CommitPartial* part,
                          int* row_cnt, int* blk_cnt, cudaStream_t stream) {
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  dim3 grid(static_cast<unsigned>(B) * L, plan.S);
  commit_kernel<<<grid, kThreads, 0, stream>>>(logits, mask, L, V, plan.S, plan.chunk, threshold,
                                               c, tok_out, conf_out, commit_out, part, row_cnt,
                                               blk_cnt);
  return cudaGetLastError();
}

cudaError_t launch_apply_commit(uint8_t* mask, const uint8_t* commit, int n, cudaStream_t stream) {
  apply_commit_kernel<<<(n + 255) / 256, 256, 0, stream>>>(mask, commit, n);
  return cudaGetLastError();
}

}  // namespace bdlm
