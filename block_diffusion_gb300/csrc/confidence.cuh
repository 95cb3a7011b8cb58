// Confidence arithmetic shared by the commit kernels and the LM head's fused epilogue: a
// running (max, sum of exponentials, first index of the max) over bf16 logits, merges of such
// partial states, and the per-block commit decision.
//
// Source: JetEngine notes (CLAUDE.md), "Remasking Strategies" (low_confidence_dynamic: the
// confidence of a position is its max softmax probability; every masked position at or above
// the threshold is committed, else the most confident one) and "Sampling and Remasking"
// (top-k and left/right-to-right orders); dInfer blog, "Algorithmic Innovations" (threshold
// decoding).  With m the row maximum and c = log2(e) / T, conf = 1 / sum_v 2^((l_v - m) c).
#pragma once
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "../../include/bdlm.h"
#include "ptx.cuh"

namespace bdlm {

struct Acc {
  float m;    // running max (raw logit)
  float s;    // sum of 2^((x - m) * c)
  int idx;    // first index of the max
};

// The state of the union of two disjoint sets of logits; on equal maxima the lower index.
__device__ __forceinline__ Acc merge(Acc a, Acc b, float c) {
  if (b.m == -CUDART_INF_F) return a;
  if (a.m == -CUDART_INF_F) return b;
  Acc o;
  o.m = fmaxf(a.m, b.m);
  o.s = a.s * ex2((a.m - o.m) * c) + b.s * ex2((b.m - o.m) * c);
  const int ia = (a.m == o.m) ? a.idx : 0x7FFFFFFF;
  const int ib = (b.m == o.m) ? b.idx : 0x7FFFFFFF;
  o.idx = min(ia, ib);
  return o;
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

constexpr uint32_t kBf16NegInfPair = 0xFF80FF80u;

__device__ __forceinline__ float bf16f(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Max of the 32 logits held as 16 packed bf16 pairs (a tree of packed maxima).
__device__ __forceinline__ float group_max(const uint32_t (&w)[16]) {
  __nv_bfloat162 m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    m[i] = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w[2 * i]),
                   *reinterpret_cast<const __nv_bfloat162*>(&w[2 * i + 1]));
#pragma unroll
  for (int n = 4; n > 0; n >>= 1)
#pragma unroll
    for (int i = 0; i < n; ++i) m[i] = __hmax2(m[2 * i], m[2 * i + 1]);
  return fmaxf(__low2float(m[0]), __high2float(m[0]));
}

// Sum of 2^(x c - mc) over the 32 logits: the scaling runs two logits per packed FMA, the
// exponentials are independent and the sum is a tree of packed adds.
__device__ __forceinline__ float exp_sum32(const uint32_t (&w)[16], float c, float mc) {
  const float2 cc = make_float2(c, c), nm = make_float2(-mc, -mc);
  float2 e[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 y = __ffma2_rn(make_float2(bf16_lo(w[i]), bf16_hi(w[i])), cc, nm);
    e[i] = make_float2(ex2(y.x), ex2(y.y));
  }
#pragma unroll
  for (int step = 1; step < 16; step <<= 1)
#pragma unroll
    for (int i = 0; i < 16; i += 2 * step) e[i] = __fadd2_rn(e[i], e[i + step]);
  return e[0].x + e[0].y;
}

// The positions a block commits (bit i: position i), from the confidences of its candidate
// positions (bit i of `cand`: position i is masked and was scored) under one rule:
//  * THRESHOLD: every candidate with conf >= threshold, else the single most confident one
//    (lowest position on ties);
//  * TOPK: the min(k, candidates) most confident (lowest position on ties);
//  * SEQUENTIAL / ANTI_SEQUENTIAL: the first / last min(k, candidates) candidates.
__device__ __forceinline__ uint64_t decide_block(int rule, int k, float threshold, int L,
                                                 uint64_t cand, const float* conf) {
  uint64_t sel = 0;
  const int n_cand = __popcll(cand);
  if (rule == BDLM_COMMIT_THRESHOLD) {
    int best = -1;
    float best_c = 0.f;
    for (int i = 0; i < L; ++i) {
      if (!((cand >> i) & 1)) continue;
      const float ci = conf[i];
      if (ci >= threshold) sel |= 1ull << i;
      if (best < 0 || ci > best_c) {
        best = i;
        best_c = ci;
      }
    }
    if (n_cand && !sel) sel = 1ull << best;  // at least the most confident position
  } else if (rule == BDLM_COMMIT_TOPK) {
    const int n = min(k, n_cand);
    for (int c = 0; c < n; ++c) {  // the most confident candidate not yet chosen
      int best = -1;
      float best_c = 0.f;
      for (int i = 0; i < L; ++i) {
        if (!((cand >> i) & 1) || ((sel >> i) & 1)) continue;
        if (best < 0 || conf[i] > best_c) {
          best = i;
          best_c = conf[i];
        }
      }
      sel |= 1ull << best;
    }
  } else {
    const bool left = rule == BDLM_COMMIT_SEQUENTIAL;
    int n = min(k, n_cand);
    for (int j = 0; j < L && n > 0; ++j) {
      const int i = left ? j : L - 1 - j;
      if (!((cand >> i) & 1)) continue;
      sel |= 1ull << i;
      --n;
    }
  }
  return sel;
}

}  // namespace bdlm
