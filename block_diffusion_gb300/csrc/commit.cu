// Confidence + commit of one denoising step: one pass over the vocabulary.
//
// Source: JetEngine notes (CLAUDE.md), "Remasking Strategies" (low_confidence_dynamic) and
// "Remaining Optimization Avenues" (a fused postprocess kernel); dInfer blog, "Algorithmic
// Innovations" (threshold decoding).  Per masked row: argmax token (lowest index on ties),
// max softmax probability at temperature T; per block: commit every masked position at or
// above the threshold, else the single most confident one.
//
// Layout of the work: the masked rows, laid end to end, form one sequence of T = n_masked * V
// logits that is cut evenly across every warp of a persistent grid (each CTA first counts the
// mask to learn n_masked and where each masked row sits).  A warp streams its range through a
// private ring of two 4 KB shared-memory stages filled by bulk copies (one instruction per
// stage), keeping a running (max, sum of exp, first argmax) per lane, and at the end of each
// row segment merges its lanes with shuffles into one partial: that is all it writes.  A second
// kernel, one CTA per block, then merges each masked row's partials in warp order, writes
// tok/conf and decides the block's commit after a single round of loads: no counters, fences
// or atomics sit on the streaming warps' path.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "confidence.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kRing = 2;              // shared-memory stages per warp
constexpr int kChunkBytes = 4096;     // bytes per stage
constexpr int kChunk = kChunkBytes / 2;
constexpr int kUnroll = 4;            // 16-byte vectors per lane per group of 32 logits
constexpr int kMaskSmem = 8192;       // masks of up to this many rows are copied to smem

// A lane's running state over one row segment.  The position of the max is found lazily:
// when a group of 32 logits raises the max, the lane keeps a copy of that group (its 16
// packed words and where it starts) and locates the first occurrence only when the segment
// ends, instead of scanning every group that raises it.
struct LaneAcc {
  float m;            // running max (raw logit)
  float s;            // sum of 2^((x - m) c)
  int idx;            // first index of the max, or -1 while it lies in the saved group
  int gbase;          // saved group: vector q covers logits gbase + 256 q .. + 7
  uint32_t gw[16];    // saved group's packed bf16 pairs
};

__device__ __forceinline__ void lane_reset(LaneAcc& a) {
  a.m = -CUDART_INF_F;
  a.s = 0.f;
  a.idx = 0x7FFFFFFF;
}

// Adds the 32 logits of one group (vector q = words 4q .. 4q+3, starting at logit
// gbase + 256 q).  A lane sees its logits in increasing index order, so a strictly larger
// max keeps the first occurrence.
__device__ __forceinline__ void absorb32(LaneAcc& a, const uint32_t (&w)[16], int gbase, float c) {
  const float gm = group_max(w);
  if (gm > a.m) {
    a.s = (a.m == -CUDART_INF_F) ? 0.f : a.s * ex2((a.m - gm) * c);
    a.m = gm;
    a.idx = -1;
    a.gbase = gbase;
#pragma unroll
    for (int i = 0; i < 16; ++i) a.gw[i] = w[i];
  }
  if (a.m == -CUDART_INF_F) return;  // nothing but padding so far
  a.s += exp_sum32(w, c, a.m * c);
}

// Adds one logit x with index i.
__device__ __forceinline__ void absorb1(LaneAcc& a, float x, int i, float c) {
  if (x > a.m) {
    a.s = (a.m == -CUDART_INF_F) ? 0.f : a.s * ex2((a.m - x) * c);
    a.m = x;
    a.idx = i;
  }
  a.s += ex2(fmaf(x, c, -a.m * c));
}

// The lane's (max, sum, first index of the max) with the saved group's position resolved.
__device__ __forceinline__ Acc lane_result(const LaneAcc& a) {
  int idx = a.idx;
  if (idx < 0) {
    idx = 0x7FFFFFFF;
#pragma unroll
    for (int e = 31; e >= 0; --e) {
      const float x = (e & 1) ? bf16_hi(a.gw[e >> 1]) : bf16_lo(a.gw[e >> 1]);
      if (x == a.m) idx = a.gbase + (e >> 3) * 256 + (e & 7);
    }
  }
  return Acc{a.m, a.s, idx};
}

struct ChunkMeta {
  int r;         // row id
  int k;         // masked-row index
  int g0, g1;    // logits [g0, g1) of the row in this stage
  int i0, i1;    // the 16-byte aligned interior [i0, i1) that the bulk copy brought in
  int last;      // last stage of this row segment
  int pad;
};

struct CommitArgs {
  const uint16_t* logits;
  const uint8_t* mask;
  int R, L, V;
  float threshold, c;
  int32_t* tok_out;
  float* conf_out;
  uint8_t* commit_out;
  CommitPartial* part;
  int* err;  // device error word (may be null)
  int rule, k;  // block decision: BDLM_COMMIT_* and positions per block
};

// First logit (in the masked concatenation) of warp w out of W; a multiple of 8.
__device__ __forceinline__ long long range_start(long long T, int W, int w) {
  if (w >= W) return T;
  return ((T * w) / W) & ~7ll;
}
// The warp whose range holds element e (an estimate from the even split, then corrected for
// the rounding of range starts down to multiples of 8).
__device__ __forceinline__ int warp_of(long long e, long long T, int W) {
  int w = static_cast<int>((e * W) / T);
  if (w >= W) w = W - 1;
  while (w > 0 && range_start(T, W, w) > e) --w;
  while (w + 1 < W && range_start(T, W, w + 1) <= e) ++w;
  return w;
}

// Streams warp w's range [e0, e1) of the masked concatenation (T logits, W warps) through
// the warp's ring and finalizes the rows whose element count it completes.
__device__ __forceinline__ void stream_range(const CommitArgs& a, long long T, int W, int w,
                                          long long e0, long long e1, int per,
                                          const int* s_pref, const uint8_t* s_mask,
                                          uint8_t* ring, uint64_t* bars, ChunkMeta* meta,
                                          int lane) {
  // row id of masked index k: binary search over the per-thread counts, then a byte scan
  auto row_of = [&](long long k) -> int {
    int lo = 0, hi = kThreads - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pref[mid] <= k) lo = mid; else hi = mid - 1;
    }
    int left = static_cast<int>(k - s_pref[lo]);
    int r = min(a.R, lo * per);
    for (;; ++r)
      if ((s_mask ? s_mask[r] : a.mask[r]) && left-- == 0) break;
    return r;
  };

  // producer cursor (lane 0): masked row k, offset in that row, logits left in the range
  long long left = e1 - e0;
  int cur_k = static_cast<int>(e0 / a.V);
  int cur_off = static_cast<int>(e0 - static_cast<long long>(cur_k) * a.V);
  int cur_r = -1;
  int issued = 0;
  auto issue = [&](int slot) -> bool {  // lane 0; false when the range is exhausted
    if (left <= 0) return false;
    if (cur_r < 0) cur_r = row_of(cur_k);
    const int seg_end = static_cast<int>(min(static_cast<long long>(a.V), cur_off + left));
    const int q1 = min(seg_end, cur_off + kChunk);
    ChunkMeta m;
    m.r = cur_r;
    m.k = cur_k;
    m.g0 = cur_off;
    m.g1 = q1;
    const uint16_t* row = a.logits + static_cast<size_t>(cur_r) * a.V;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(row + m.g0);
    const uintptr_t b1 = reinterpret_cast<uintptr_t>(row + m.g1);
    const uintptr_t al0 = (b0 + 15) & ~static_cast<uintptr_t>(15);
    const uintptr_t al1 = b1 & ~static_cast<uintptr_t>(15);
    if (al1 > al0) {
      m.i0 = m.g0 + static_cast<int>((al0 - b0) >> 1);
      m.i1 = m.g0 + static_cast<int>((al1 - b0) >> 1);
    } else {
      m.i0 = m.i1 = m.g1;  // no aligned interior: lanes read the few logits directly
    }
    m.last = q1 == seg_end;
    meta[slot] = m;
    const uint32_t bytes = static_cast<uint32_t>((m.i1 - m.i0) * 2);
    if (bytes) {
      mbar_arrive_expect_tx(&bars[slot], bytes);
      bulk_load(ring + slot * kChunkBytes, row + m.i0, bytes, &bars[slot]);
    } else {
      mbar_arrive(&bars[slot]);
    }
    left -= q1 - cur_off;
    cur_off = q1;
    if (cur_off == a.V) {
      ++cur_k;
      cur_off = 0;
      cur_r = -1;
    }
    return true;
  };
  if (lane == 0) {
    for (int i = 0; i < kRing; ++i)
      if (issue(i)) ++issued;
  }
  issued = __shfl_sync(0xffffffffu, issued, 0);

  int abort_flag = 0;
  LaneAcc acc;
  lane_reset(acc);
  for (int u = 0; u < issued; ++u) {
    const int slot = u % kRing;
    // every lane waits on its own clock; the warp then agrees on the outcome, so no lane
    // leaves for the drain while the others go on to the full-warp shuffles below
    const bool landed = mbar_wait(&bars[slot], (u / kRing) & 1, &abort_flag);
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0 && a.err) atomicOr(a.err, BDLM_DEVERR_TIMEOUT);
      break;
    }
    const ChunkMeta m = meta[slot];
    const uint16_t* row = a.logits + static_cast<size_t>(m.r) * a.V;
    const uint4* vp = reinterpret_cast<const uint4*>(ring + slot * kChunkBytes);
    const int nvec = (m.i1 - m.i0) >> 3;
    // logits before the aligned interior (at most 7) come first: each lane then sees its
    // logits in increasing index order
    if (m.g0 + lane < m.i0) absorb1(acc, bf16f(row[m.g0 + lane]), m.g0 + lane, a.c);
    if (nvec == kChunk / 8) {
      // a full stage: no bounds checks
#pragma unroll
      for (int v0 = 0; v0 < kChunk / 8; v0 += 32 * kUnroll) {
        uint32_t wv[16];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
          const uint4 t = vp[v0 + q * 32 + lane];
          wv[4 * q] = t.x;
          wv[4 * q + 1] = t.y;
          wv[4 * q + 2] = t.z;
          wv[4 * q + 3] = t.w;
        }
        absorb32(acc, wv, m.i0 + (v0 + lane) * 8, a.c);
      }
    } else {
      for (int v0 = 0; v0 < nvec; v0 += 32 * kUnroll) {
        uint32_t wv[16];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
          const int v = v0 + q * 32 + lane;
          uint4 t = make_uint4(kBf16NegInfPair, kBf16NegInfPair, kBf16NegInfPair,
                               kBf16NegInfPair);
          if (v < nvec) t = vp[v];
          wv[4 * q] = t.x;
          wv[4 * q + 1] = t.y;
          wv[4 * q + 2] = t.z;
          wv[4 * q + 3] = t.w;
        }
        absorb32(acc, wv, m.i0 + (v0 + lane) * 8, a.c);
      }
    }
    // logits after the aligned interior (at most 7)
    if (m.i1 + lane < m.g1) absorb1(acc, bf16f(row[m.i1 + lane]), m.i1 + lane, a.c);
    __syncwarp();
    if (lane == 0 && issue(slot)) ++issued;  // refill the stage just read
    issued = __shfl_sync(0xffffffffu, issued, 0);
    if (!m.last) continue;
    // ---- end of a row segment: one partial per (warp, row) at slot w + k (the ranges are
    // ordered and contiguous, so the slots are distinct)
    Acc t = warp_merge(lane_result(acc), a.c);
    lane_reset(acc);
    if (lane == 0) a.part[w + m.k] = CommitPartial{t.m, t.s, t.idx, 0};
  }
  // drain: nothing may still be landing in this warp's stages when it exits
  if (lane == 0) {
    for (int u = max(0, issued - kRing); u < issued; ++u) {
      int dummy = 0;
      mbar_wait(&bars[u % kRing], (u / kRing) & 1, &dummy);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
commit_kernel(const CommitArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring_base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                                  ~static_cast<uintptr_t>(127));
  __shared__ uint64_t s_bar[kWarps][kRing];
  __shared__ ChunkMeta s_meta[kWarps][kRing];
  __shared__ int s_pref[kThreads + 1];
  __shared__ int s_wsum[kWarps];
  __shared__ uint8_t s_mask[kMaskSmem];   // copy of the mask when it fits
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_wait();
  griddep_launch_dependents();

  // ---- count the mask: s_pref[t] = masked rows before thread t's byte range
  const int per = (a.R + kThreads - 1) / kThreads;
  const int r_lo = min(a.R, tid * per), r_hi = min(a.R, r_lo + per);
  const bool mask_in_smem = a.R <= kMaskSmem;
  int cnt = 0;
  for (int r = r_lo; r < r_hi; ++r) {
    const uint8_t mk = a.mask[r];
    cnt += mk != 0;
    if (mask_in_smem) s_mask[r] = mk;
  }
  int incl = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_wsum[warp] = incl;
  if (tid < kWarps * kRing) mbar_init(&s_bar[tid / kRing][tid % kRing], 1);
  fence_mbar_init();
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += s_wsum[w];
  s_pref[tid] = wbase + incl - cnt;
  if (tid == kThreads - 1) s_pref[kThreads] = wbase + incl;
  __syncthreads();
  const long long n_masked = s_pref[kThreads];

  // ---- this warp's range of the masked concatenation
  const long long T = n_masked * a.V;
  const long long Wcap = static_cast<long long>(gridDim.x) * kWarps;
  const int W = static_cast<int>(max(1ll, min(Wcap, T / kChunk)));
  const int w = blockIdx.x * kWarps + warp;
  const long long e0 = range_start(T, W, w);
  const long long e1 = range_start(T, W, w + 1);
  if (w < W && T > 0 && e0 < e1)
    stream_range(a, T, W, w, e0, e1, per, s_pref, mask_in_smem ? s_mask : nullptr,
                 ring_base + warp * (kRing * kChunkBytes), s_bar[warp], s_meta[warp], lane);

}

// One CTA per block b, min(L, 32) warps: the masked index of each row (from the mask, an input
// that is complete before the streaming kernel lets this one start), then, once the streaming
// kernel has finished, one warp per row merges the row's partials in warp order; thread 0
// decides the block: every masked position with conf >= threshold, else the single most
// confident one (lowest position on ties).  Unmasked rows get tok = -1, conf = -inf.
__global__ void __launch_bounds__(1024)
commit_finalize_kernel(const CommitArgs a, int stream_grid) {
  __shared__ int s_wsum[32];
  __shared__ int s_blk_before, s_total;
  __shared__ float s_conf[64];
  const int b = blockIdx.x, L = a.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  // masked rows before this block, and in all
  int before = 0, total = 0;
  for (int r = tid; r < a.R; r += blockDim.x) {
    const int mk = a.mask[r] != 0;
    total += mk;
    before += (r < b * L) ? mk : 0;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, off);
    total += __shfl_xor_sync(0xffffffffu, total, off);
  }
  if (lane == 0) s_wsum[warp] = before;
  __syncthreads();
  if (tid == 0) {
    int sb = 0;
    for (int i = 0; i < nw; ++i) sb += s_wsum[i];
    s_blk_before = sb;
  }
  __syncthreads();
  if (lane == 0) s_wsum[warp] = total;
  __syncthreads();
  if (tid == 0) {
    int st = 0;
    for (int i = 0; i < nw; ++i) st += s_wsum[i];
    s_total = st;
  }
  __syncthreads();
  const long long T = static_cast<long long>(s_total) * a.V;
  const long long Wcap = static_cast<long long>(stream_grid) * kWarps;
  const int W = static_cast<int>(max(1ll, min(Wcap, T / kChunk)));
  griddep_wait();  // the streaming kernel's partials are complete and visible
  griddep_launch_dependents();
  const uint8_t* mk = a.mask + static_cast<size_t>(b) * L;
  for (int i = warp; i < L; i += nw) {
    const int r = b * L + i;
    if (!mk[i]) {
      if (lane == 0) {
        a.tok_out[r] = -1;
        a.conf_out[r] = -CUDART_INF_F;
        s_conf[i] = -CUDART_INF_F;
      }
      continue;
    }
    int k = s_blk_before;
    for (int j = 0; j < i; ++j) k += mk[j] != 0;
    const long long kv = static_cast<long long>(k) * a.V;
    const int first_w = warp_of(kv, T, W);
    const int n_w = warp_of(min(kv + a.V, T) - 1, T, W) - first_w + 1;
    const CommitPartial* pr = a.part + first_w + k;
    Acc f{-CUDART_INF_F, 0.f, 0x7FFFFFFF};
    for (int j0 = 0; j0 < n_w; j0 += 32) {
      Acc q{-CUDART_INF_F, 0.f, 0x7FFFFFFF};
      if (j0 + lane < n_w) {
        const CommitPartial c = pr[j0 + lane];
        q = Acc{c.m, c.s, c.idx};
      }
      f = merge(f, warp_merge(q, a.c), a.c);
    }
    if (lane == 0) {
      const float conf = 1.0f / f.s;
      a.tok_out[r] = f.idx;
      a.conf_out[r] = conf;
      s_conf[i] = conf;
    }
  }
  __syncthreads();
  if (tid == 0) {
    uint64_t cand = 0;
    for (int i = 0; i < L; ++i) cand |= static_cast<uint64_t>(mk[i] != 0) << i;
    const uint64_t sel = decide_block(a.rule, a.k, a.threshold, L, cand, s_conf);
    uint8_t* co = a.commit_out + static_cast<size_t>(b) * L;
    for (int i = 0; i < L; ++i) co[i] = static_cast<uint8_t>((sel >> i) & 1);
  }
}

__global__ void apply_commit_kernel(uint8_t* __restrict__ mask, const uint8_t* __restrict__ commit,
                                    int n) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n && commit[i]) mask[i] = 0;
}

}  // namespace

CommitPlan plan_commit(int B, int L, int V, int num_sms) {
  CommitPlan p;
  const long long rows = static_cast<long long>(B) * L;
  p.grid = num_sms > 0 ? num_sms : 1;
  p.total_items = rows;
  p.smem_bytes = static_cast<size_t>(kWarps) * kRing * kChunkBytes + 128;
  // one partial per (warp, masked row segment): slots w + k < warps + rows
  p.part_bytes = static_cast<size_t>(p.grid * kWarps + rows) * sizeof(CommitPartial);
  p.fin_threads = (L < 32 ? L : 32) * 32;
  (void)V;
  return p;
}

cudaError_t launch_commit(const uint16_t* logits, const uint8_t* mask, int B, int L, int V,
                          float threshold, float temperature, int32_t* tok_out, float* conf_out,
                          uint8_t* commit_out, const CommitPlan& plan, CommitPartial* part,
                          int* err, cudaStream_t stream, bool programmatic, int rule, int k) {
  static std::atomic<unsigned long long> attr_done{0};
  const int smem_bytes = static_cast<int>(plan.smem_bytes);  // the same for every plan
  cudaError_t ea = once_per_device(attr_done, [smem_bytes] {
    return cudaFuncSetAttribute(commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_bytes);
  });
  if (ea != cudaSuccess) return ea;
  CommitArgs args;
  args.logits = logits;
  args.mask = mask;
  args.R = B * L;
  args.L = L;
  args.V = V;
  args.threshold = threshold;
  args.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  args.tok_out = tok_out;
  args.conf_out = conf_out;
  args.commit_out = commit_out;
  args.part = part;
  args.err = err;
  args.rule = rule;
  args.k = k;
  cudaError_t e;
  if (!programmatic) {
    commit_kernel<<<plan.grid, kThreads, plan.smem_bytes, stream>>>(args);
    e = cudaGetLastError();
  } else {
    e = launch_pdl(commit_kernel, dim3(plan.grid), dim3(kThreads), plan.smem_bytes, stream, args);
  }
  if (e != cudaSuccess) return e;
  return launch_pdl(commit_finalize_kernel, dim3(B), dim3(plan.fin_threads), 0, stream, args,
                    plan.grid);
}

cudaError_t launch_apply_commit(uint8_t* mask, const uint8_t* commit, int n, cudaStream_t stream) {
  return launch_pdl(apply_commit_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, mask,
                    commit, n);
}

}  // namespace bdlm
