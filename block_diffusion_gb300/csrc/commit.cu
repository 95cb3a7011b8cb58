// Confidence + commit of one denoising step: one pass over the vocabulary, in one launch.
//
// Source: JetEngine notes (CLAUDE.md), "Remasking Strategies" (low_confidence_dynamic, top-k,
// sequential orders, entropy_bounded) and "Remaining Optimization Avenues" (a fused
// postprocess kernel); dInfer blog, "Algorithmic Innovations" (threshold decoding).  Per
// masked row: argmax token (lowest index on ties), max softmax probability and entropy at
// temperature T; per block: the commit rule over the block's masked positions.
//
// Layout of the work: the masked rows, laid end to end, form one sequence of T = n_masked * V
// logits that is cut evenly across every warp of a persistent grid (each CTA first counts the
// mask to learn n_masked and where each masked row sits).  A warp streams its range through a
// private ring of two 4 KB shared-memory stages filled by bulk copies (one instruction per
// stage), keeping a running (max, sum of exponentials, first argmax, and for the entropy the
// exponent-weighted sum) per lane, and at the end of each row segment merges its lanes with
// shuffles into one partial: that is all it writes.  A second kernel, one CTA per block and
// launched dependent on the first, merges each masked row's partials (one lane per row), writes
// tok/conf/entropy and decides the block's commit with one warp: no counters, fences or atomics
// sit on the streaming warps' path.  (A single-kernel variant in which the warp completing a
// row or block finalizes it through acquire-release counters was measured slower: the counter
// round trips lengthened the tail, and same-address arrivals serialised.)
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
  float a;            // sum of 2^((x - m) c) * (x - m) c
  int idx;            // first index of the max, or -1 while it lies in the saved group
  int gbase;          // saved group: vector q covers logits gbase + 256 q .. + 7
  uint32_t gw[16];    // saved group's packed bf16 pairs
};

__device__ __forceinline__ void lane_reset(LaneAcc& x) {
  x.m = -CUDART_INF_F;
  x.s = 0.f;
  x.a = 0.f;
  x.idx = 0x7FFFFFFF;
}

// Adds the 32 logits of one group (vector q = words 4q .. 4q+3, starting at logit
// gbase + 256 q).  A lane sees its logits in increasing index order, so a strictly larger
// max keeps the first occurrence.  ENT: also the exponent-weighted sum (for the entropy).
template <bool ENT>
__device__ __forceinline__ void absorb32(LaneAcc& x, const uint32_t (&w)[16], int gbase, float c) {
  const float gm = group_max(w);
  if (gm > x.m) {
    if (x.m == -CUDART_INF_F) {
      x.s = 0.f;
      x.a = 0.f;
    } else {
      acc_rebase(x.s, x.a, x.m, gm, c);
    }
    x.m = gm;
    x.idx = -1;
    x.gbase = gbase;
#pragma unroll
    for (int i = 0; i < 16; ++i) x.gw[i] = w[i];
  }
  if (x.m == -CUDART_INF_F) return;  // nothing but padding so far
  exp_sum32<ENT>(w, c, x.m * c, x.s, x.a);
}

// Adds one logit v with index i.
template <bool ENT>
__device__ __forceinline__ void absorb1(LaneAcc& x, float v, int i, float c) {
  if (v > x.m) {
    if (x.m == -CUDART_INF_F) {
      x.s = 0.f;
      x.a = 0.f;
    } else {
      acc_rebase(x.s, x.a, x.m, v, c);
    }
    x.m = v;
    x.idx = i;
  }
  if (x.m == -CUDART_INF_F) return;
  const float y = fmaf(v, c, -x.m * c);
  const float e = ex2(y);
  x.s += e;
  if constexpr (ENT) x.a = fmaf(e, y, x.a);
}

// The lane's state with the saved group's position resolved.
__device__ __forceinline__ Acc lane_result(const LaneAcc& x) {
  int idx = x.idx;
  if (idx < 0) {
    idx = 0x7FFFFFFF;
#pragma unroll
    for (int e = 31; e >= 0; --e) {
      const float v = (e & 1) ? bf16_hi(x.gw[e >> 1]) : bf16_lo(x.gw[e >> 1]);
      if (v == x.m) idx = x.gbase + (e >> 3) * 256 + (e & 7);
    }
  }
  return Acc{x.m, x.s, x.a, idx};
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
  float* ent_out;      // may be null
  uint8_t* commit_out;
  CommitPartial* part; // one per (warp, masked row segment): slot w + k
  int* err;            // device error word (may be null)
  int rule, k;         // block decision: BDLM_COMMIT_* and positions per block
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

__device__ __forceinline__ uint8_t mask_at(const CommitArgs& a, const uint8_t* s_mask, int r) {
  return s_mask ? s_mask[r] : a.mask[r];
}

// Outputs of the positions of block b that are not candidates, and its commit mask.
__device__ __forceinline__ void write_block(const CommitArgs& a, int b, uint64_t cand,
                                            uint64_t sel, int lane) {
  for (int i = lane; i < a.L; i += 32) {
    const size_t r = static_cast<size_t>(b) * a.L + i;
    a.commit_out[r] = static_cast<uint8_t>((sel >> i) & 1);
    if (!((cand >> i) & 1)) {
      a.tok_out[r] = -1;
      a.conf_out[r] = -CUDART_INF_F;
      if (a.ent_out) a.ent_out[r] = CUDART_INF_F;
    }
  }
}

// Streams warp w's range [e0, e1) of the masked concatenation (T logits, W warps) through
// the warp's ring; at the end of each row segment it stores the warp's partial.
template <bool ENT>
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
      if (mask_at(a, s_mask, r) && left-- == 0) break;
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
    if (m.g0 + lane < m.i0) absorb1<ENT>(acc, bf16f(row[m.g0 + lane]), m.g0 + lane, a.c);
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
        absorb32<ENT>(acc, wv, m.i0 + (v0 + lane) * 8, a.c);
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
        absorb32<ENT>(acc, wv, m.i0 + (v0 + lane) * 8, a.c);
      }
    }
    // logits after the aligned interior (at most 7)
    if (m.i1 + lane < m.g1) absorb1<ENT>(acc, bf16f(row[m.i1 + lane]), m.i1 + lane, a.c);
    __syncwarp();
    if (lane == 0 && issue(slot)) ++issued;  // refill the stage just read
    issued = __shfl_sync(0xffffffffu, issued, 0);
    if (!m.last) continue;
    // ---- end of a row segment: one partial per (warp, row) at slot w + k (the ranges are
    // ordered and contiguous, so the slots are distinct)
    Acc t = warp_merge(lane_result(acc), a.c);
    lane_reset(acc);
    if (lane == 0) a.part[w + m.k] = CommitPartial{t.m, t.s, t.idx, t.a};
  }
  // drain: nothing may still be landing in this warp's stages when it exits
  if (lane == 0) {
    for (int u = max(0, issued - kRing); u < issued; ++u) {
      int dummy = 0;
      mbar_wait(&bars[u % kRing], (u / kRing) & 1, &dummy);
    }
  }
}

// ENT: the entropies are wanted (an entropy output or the entropy rule).
template <bool ENT>
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
  const uint8_t* smask = mask_in_smem ? s_mask : nullptr;

  // ---- this warp's range of the masked concatenation
  const long long T = n_masked * a.V;
  const long long Wcap = static_cast<long long>(gridDim.x) * kWarps;
  const int W = static_cast<int>(max(1ll, min(Wcap, T / kChunk)));
  const int w = blockIdx.x * kWarps + warp;
  const long long e0 = range_start(T, W, w);
  const long long e1 = range_start(T, W, w + 1);
  if (w < W && T > 0 && e0 < e1)
    stream_range<ENT>(a, T, W, w, e0, e1, per, s_pref, smask,
                 ring_base + warp * (kRing * kChunkBytes), s_bar[warp], s_meta[warp], lane);
}

// One CTA of min(L, 32) warps per block b.  Before the streaming kernel is done: the masked
// rows before block b and in all (from the mask, which is complete before the streaming kernel
// starts), hence every warp's range.  Then warp x merges the partials of the block's masked rows
// x, x + warps, ...: lane j loads partial j (the row's warps in order), a shuffle tree merges
// them (lowest index on max ties), and lane 0 writes tok / conf / entropy; warp 0 then decides
// the block's commit.  Positions that are not masked get tok = -1, conf = -inf, entropy = +inf,
// commit = 0.
__global__ void __launch_bounds__(1024)
commit_finalize_kernel(const CommitArgs a, int stream_grid) {
  __shared__ int s_wsum[2][32];
  __shared__ int s_before, s_total;
  __shared__ float s_stat[64];
  __shared__ int s_order[64];
  const int b = blockIdx.x, L = a.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
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
  if (lane == 0) {
    s_wsum[0][warp] = before;
    s_wsum[1][warp] = total;
  }
  __syncthreads();
  if (tid == 0) {
    int sb = 0, st = 0;
    for (int i = 0; i < nw; ++i) {
      sb += s_wsum[0][i];
      st += s_wsum[1][i];
    }
    s_before = sb;
    s_total = st;
  }
  __syncthreads();
  const long long T = static_cast<long long>(s_total) * a.V;
  const long long Wcap = static_cast<long long>(stream_grid) * kWarps;
  const int W = static_cast<int>(max(1ll, min(Wcap, T / kChunk)));
  const uint8_t* mk = a.mask + static_cast<size_t>(b) * L;
  const uint64_t cand =
      (static_cast<uint64_t>(__ballot_sync(0xffffffffu, lane + 32 < L && mk[lane + 32] != 0))
       << 32) |
      __ballot_sync(0xffffffffu, lane < L && mk[lane] != 0);
  griddep_wait();  // the streaming kernel's partials are complete and visible
  griddep_launch_dependents();
  const bool ent_rule = a.rule == BDLM_COMMIT_ENTROPY_BOUNDED;
  for (int i = warp; i < L; i += nw) {
    if (!((cand >> i) & 1)) continue;
    const int k = s_before + __popcll(cand & ((1ull << i) - 1ull));
    const long long kv = static_cast<long long>(k) * a.V;
    const int first_w = warp_of(kv, T, W);
    const int n_w = warp_of(min(kv + a.V, T) - 1, T, W) - first_w + 1;
    const CommitPartial* pr = a.part + first_w + k;
    Acc f = acc_init();
    for (int j0 = 0; j0 < n_w; j0 += 32) {
      Acc q = acc_init();
      if (j0 + lane < n_w) {
        const CommitPartial t = pr[j0 + lane];
        q = Acc{t.m, t.s, t.a, t.idx};
      }
      f = merge(f, warp_merge(q, a.c), a.c);
    }
    if (lane == 0) {
      const size_t r = static_cast<size_t>(b) * L + i;
      const float conf = acc_conf(f), ent = acc_entropy(f);
      a.tok_out[r] = f.idx;
      a.conf_out[r] = conf;
      if (a.ent_out) a.ent_out[r] = ent;
      s_stat[i] = ent_rule ? ent : conf;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const uint64_t sel = decide_block_warp(a.rule, a.k, a.threshold, L, cand, s_stat, s_order,
                                           lane);
    write_block(a, b, cand, sel, lane);
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
  (void)B;
  (void)V;
  return p;
}

cudaError_t launch_commit(const uint16_t* logits, const uint8_t* mask, int B, int L, int V,
                          float threshold, float temperature, int32_t* tok_out, float* conf_out,
                          float* ent_out, uint8_t* commit_out, const CommitPlan& plan,
                          CommitPartial* part, int* err, cudaStream_t stream, int rule, int k) {
  static std::atomic<unsigned long long> attr_done{0};
  const int smem_bytes = static_cast<int>(plan.smem_bytes);  // the same for every plan
  cudaError_t ea = once_per_device(attr_done, [smem_bytes] {
    cudaError_t r = cudaFuncSetAttribute(commit_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(commit_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  args.ent_out = ent_out;
  args.commit_out = commit_out;
  args.part = part;
  args.err = err;
  args.rule = rule;
  args.k = k;
  const bool ent = ent_out != nullptr || rule == BDLM_COMMIT_ENTROPY_BOUNDED;
  cudaError_t e = ent ? launch_pdl(commit_kernel<true>, dim3(plan.grid), dim3(kThreads),
                                   plan.smem_bytes, stream, args)
                      : launch_pdl(commit_kernel<false>, dim3(plan.grid), dim3(kThreads),
                                   plan.smem_bytes, stream, args);
  if (e != cudaSuccess) return e;
  return launch_pdl(commit_finalize_kernel, dim3(B), dim3((L < 32 ? L : 32) * 32), 0, stream,
                    args, plan.grid);
}

cudaError_t launch_apply_commit(uint8_t* mask, const uint8_t* commit, int n, cudaStream_t stream) {
  return launch_pdl(apply_commit_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, mask,
                    commit, n);
}

}  // namespace bdlm
