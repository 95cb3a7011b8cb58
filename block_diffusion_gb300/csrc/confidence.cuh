// Confidence arithmetic shared by the commit kernel and the LM head's fused epilogue: a
// running (max, sum of exponentials, exponent-weighted sum, first index of the max) over bf16
// logits, merges of such partial states, and the per-block commit decision.
//
// Source: JetEngine notes (CLAUDE.md), "Remasking Strategies" (low_confidence_dynamic: the
// confidence of a position is its max softmax probability; every masked position at or above
// the threshold is committed, else the most confident one; low_confidence_static: top-k;
// sequential orders; entropy_bounded: unmask by a cumulative entropy budget) and "Key Config
// Parameters" (eb_threshold); dInfer blog, "Algorithmic Innovations" (threshold decoding).
//
// With m the row maximum, c = log2(e) / T and y_v = (l_v - m) c <= 0 (base-2 exponents):
//     s = sum_v 2^y_v,   a = sum_v 2^y_v y_v,
//     conf = 1 / s (the largest softmax probability),
//     H = -sum_v p_v ln p_v = ln s - ln 2 * a / s   (nats; p_v = 2^y_v / s).
// When the reference maximum rises by d = (m' - m) c, 2^y scales by 2^-d and y drops by d, so
// s' = 2^-d s and a' = 2^-d (a - d s): that rescale is also the merge of two partial states.
#pragma once
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "../../include/bdlm.h"
#include "ptx.cuh"

namespace bdlm {

struct Acc {
  float m;    // running max (raw logit)
  float s;    // sum of 2^((x - m) c)
  float a;    // sum of 2^((x - m) c) * (x - m) c
  int idx;    // first index of the max
};

__device__ __forceinline__ Acc acc_init() { return Acc{-CUDART_INF_F, 0.f, 0.f, 0x7FFFFFFF}; }

// (s, a) brought from reference max m to a larger one mn: d = (mn - m) c >= 0.
__device__ __forceinline__ void acc_rebase(float& s, float& a, float m, float mn, float c) {
  const float d = (mn - m) * c;
  const float f = ex2(-d);
  a = f * fmaf(-d, s, a);
  s = f * s;
}

// The state of the union of two disjoint sets of logits; on equal maxima the lower index.
__device__ __forceinline__ Acc merge(Acc x, Acc y, float c) {
  if (y.m == -CUDART_INF_F) return x;
  if (x.m == -CUDART_INF_F) return y;
  Acc o;
  o.m = fmaxf(x.m, y.m);
  acc_rebase(x.s, x.a, x.m, o.m, c);
  acc_rebase(y.s, y.a, y.m, o.m, c);
  o.s = x.s + y.s;
  o.a = x.a + y.a;
  const int ix = (x.m == o.m) ? x.idx : 0x7FFFFFFF;
  const int iy = (y.m == o.m) ? y.idx : 0x7FFFFFFF;
  o.idx = min(ix, iy);
  return o;
}

__device__ __forceinline__ Acc warp_merge(Acc x, float c) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Acc o;
    o.m = __shfl_xor_sync(0xffffffffu, x.m, off);
    o.s = __shfl_xor_sync(0xffffffffu, x.s, off);
    o.a = __shfl_xor_sync(0xffffffffu, x.a, off);
    o.idx = __shfl_xor_sync(0xffffffffu, x.idx, off);
    x = merge(x, o, c);
  }
  return x;
}

// Confidence and entropy (nats) of a merged row state.
__device__ __forceinline__ float acc_conf(const Acc& x) { return 1.0f / x.s; }
__device__ __forceinline__ float acc_entropy(const Acc& x) {
  return fmaxf(0.f, logf(x.s) - 0.69314718055994531f * (x.a / x.s));
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

// Adds the 32 logits' 2^y (and, with ENT, 2^y * y) to s (and a), y = x c - mc: the scaling runs
// two logits per packed FMA, the exponentials are independent, and the sums are trees of packed
// adds.  Padding logits (-inf) contribute 0 to both (2^-inf = 0, and 0 * -inf is avoided by
// flushing y to a finite value first).
template <bool ENT>
__device__ __forceinline__ void exp_sum32(const uint32_t (&w)[16], float c, float mc, float& s,
                                          float& a) {
  const float2 cc = make_float2(c, c), nm = make_float2(-mc, -mc);
  float2 e[16], ey[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float2 y = __ffma2_rn(make_float2(bf16_lo(w[i]), bf16_hi(w[i])), cc, nm);
    e[i] = make_float2(ex2(y.x), ex2(y.y));
    if constexpr (ENT) {
      y.x = fmaxf(y.x, -1e30f);
      y.y = fmaxf(y.y, -1e30f);
      ey[i] = __fmul2_rn(e[i], y);
    }
  }
#pragma unroll
  for (int step = 1; step < 16; step <<= 1)
#pragma unroll
    for (int i = 0; i < 16; i += 2 * step) {
      e[i] = __fadd2_rn(e[i], e[i + step]);
      if constexpr (ENT) ey[i] = __fadd2_rn(ey[i], ey[i + step]);
    }
  s += e[0].x + e[0].y;
  if constexpr (ENT) a += ey[0].x + ey[0].y;
}

// Rank of position i among the candidates by its statistic: the number of candidates j that
// come before it, in decreasing order of stat (DESC) or increasing order (ascending), lower
// position first among equal values.  Lanes hold stat of positions lane and lane + 32.  Every
// lane of the warp must call it (it shuffles with a full mask).
__device__ __forceinline__ int stat_rank(uint64_t cand, int L, float v_lo, float v_hi, int i,
                                         float vi, bool desc) {
  int r = 0;
  for (int j = 0; j < L; ++j) {
    const float vj = __shfl_sync(0xffffffffu, j < 32 ? v_lo : v_hi, j & 31);
    if (!((cand >> j) & 1) || j == i) continue;
    const bool before = desc ? (vj > vi || (vj == vi && j < i)) : (vj < vi || (vj == vi && j < i));
    r += before;
  }
  return r;
}

// The positions a block commits (bit i: position i), decided by one warp (every lane gets the
// result).  Bit i of `cand`: position i is masked and was scored.  stat[i] (shared memory,
// L <= 64 entries) is the confidence of candidate i, or its entropy for the entropy rule.
//  * THRESHOLD: every candidate with conf >= threshold, else the single most confident one
//    (lowest position on ties);
//  * TOPK: the min(k, candidates) most confident (lowest position on ties);
//  * SEQUENTIAL / ANTI_SEQUENTIAL: the first / last min(k, candidates) candidates;
//  * ENTROPY_BOUNDED: candidates in increasing order of entropy (lowest position on ties),
//    as long as the running float32 sum of their entropies, added in that order, stays
//    <= threshold (the budget); always at least the first.
// s_order: shared scratch of 64 ints.
__device__ __forceinline__ uint64_t decide_block_warp(int rule, int k, float threshold, int L,
                                                      uint64_t cand, const float* stat,
                                                      int* s_order, int lane) {
  const int i0 = lane, i1 = lane + 32;
  const bool c0 = i0 < L && ((cand >> i0) & 1), c1 = i1 < L && ((cand >> i1) & 1);
  const float v0 = c0 ? stat[i0] : 0.f, v1 = c1 ? stat[i1] : 0.f;
  const int n_cand = __popcll(cand);
  uint64_t sel = 0;
  if (n_cand == 0) return 0;
  if (rule == BDLM_COMMIT_THRESHOLD) {
    const uint32_t lo = __ballot_sync(0xffffffffu, c0 && v0 >= threshold);
    const uint32_t hi = __ballot_sync(0xffffffffu, c1 && v1 >= threshold);
    sel = (static_cast<uint64_t>(hi) << 32) | lo;
    if (!sel) {
      // the single most confident candidate, lowest position on ties
      float bv = -CUDART_INF_F;
      int bi = 0x7FFFFFFF;
      if (c0) { bv = v0; bi = i0; }
      if (c1 && (v1 > bv || bi == 0x7FFFFFFF)) { bv = v1; bi = i1; }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (oi != 0x7FFFFFFF && (bi == 0x7FFFFFFF || ov > bv || (ov == bv && oi < bi))) {
          bv = ov;
          bi = oi;
        }
      }
      sel = 1ull << bi;
    }
  } else if (rule == BDLM_COMMIT_TOPK) {
    const int n = min(k, n_cand);
    // every lane computes both ranks: stat_rank shuffles across the whole warp
    const int r0 = stat_rank(cand, L, v0, v1, i0, v0, true);
    const int r1 = stat_rank(cand, L, v0, v1, i1, v1, true);
    const bool s0 = c0 && r0 < n, s1 = c1 && r1 < n;
    sel = (static_cast<uint64_t>(__ballot_sync(0xffffffffu, s1)) << 32) |
          __ballot_sync(0xffffffffu, s0);
  } else if (rule == BDLM_COMMIT_ENTROPY_BOUNDED) {
    const int r0 = stat_rank(cand, L, v0, v1, i0, v0, false);
    const int r1 = stat_rank(cand, L, v0, v1, i1, v1, false);
    if (c0) s_order[r0] = i0;
    if (c1) s_order[r1] = i1;
    __syncwarp();
    uint64_t chosen = 0;
    if (lane == 0) {
      float run = 0.f;
      for (int r = 0; r < n_cand; ++r) {
        const int i = s_order[r];
        const float next = run + stat[i];
        if (r > 0 && !(next <= threshold)) break;
        run = next;
        chosen |= 1ull << i;
      }
    }
    sel = __shfl_sync(0xffffffffu, chosen, 0);
    __syncwarp();
  } else {
    // sequential orders: the candidates before position i (left) or after it (right)
    const bool left = rule == BDLM_COMMIT_SEQUENTIAL;
    const int n = min(k, n_cand);
    const uint64_t below0 = cand & ((1ull << i0) - 1ull);
    const uint64_t below1 = i1 < 64 ? (cand & ((1ull << i1) - 1ull)) : cand;
    const int before0 = left ? __popcll(below0) : n_cand - 1 - __popcll(below0);
    const int before1 = left ? __popcll(below1) : n_cand - 1 - __popcll(below1);
    const bool s0 = c0 && before0 < n, s1 = c1 && before1 < n;
    sel = (static_cast<uint64_t>(__ballot_sync(0xffffffffu, s1)) << 32) |
          __ballot_sync(0xffffffffu, s0);
  }
  return sel;
}

}  // namespace bdlm
