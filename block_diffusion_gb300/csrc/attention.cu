// Block attention of one denoising round over a paged KV cache, for sm_103a.
//
// Source: JetEngine notes (CLAUDE.md), "ModelRunner" and "Optimization History" (opt18,
// opt24: paged-KV attention for the denoise forward); JetEngine README, "Block Diffusion
// Decoding".  For sequence b, block position i and query head h:
//     out = softmax_j(scale * q . K[j]) V[j]   over every j < prefix_len + L
// (full prefix, bidirectional inside the block), KV head = h / (Hq/Hkv).
//
// Design (one CTA = one (sequence, KV head, KV split, query-row group)):
//  * GQA packing: the G*L query rows that share a KV head are one UMMA operand, so each K/V
//    page is read once per KV head.  The product is computed transposed, S^T = K Q^T, with
//    128 KV tokens on the UMMA M side and the (few) query rows on N, so a 4-token block
//    still fills a 128-row tensor-core tile.
//  * TMA streams K and V pages (one 16-slot x 64-dim box per page and half) into a ring of
//    32 KB stages with 128-byte swizzle; tcgen05.mma reads them straight from shared memory.
//  * Softmax in two phases over a chunk of tiles held in tensor memory: all S^T tiles of the
//    chunk are computed first, the exact column maximum is taken once, then P^T = exp(S^T - m)
//    is written to shared memory (bf16) and O^T += V^T P^T accumulates in tensor memory.
//    Chunks after the first rescale O^T once per chunk.
//  * Long sequences are split across CTAs; each split writes (O, m, l) and the last split to
//    arrive (atomic counter) merges them.  Nothing waits on another CTA.
//  * Threads: warp 0 issues TMA, warp 1 owns tensor memory and issues the MMAs, warps 2-5
//    (128 threads, one per tensor-memory lane) do the softmax and the epilogue.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int kTile = 128;            // KV tokens per tile
constexpr int kPage = 16;             // tokens per page
constexpr int kStageBytes = 32768;    // one K or V tile: 2 halves x 8 pages x 16 x 128 B
constexpr int kHalfBytes = 16384;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr int kSoftmaxThreads = 128;

struct AttnParams {
  const int32_t* page_table;
  const int32_t* prefix_lens;
  uint16_t* out;
  float* part;
  int* cnt;
  int* err;
  int L, Hq, Hkv, G, max_pages, num_pages;
  int lsub, row_groups, rows_per_group, split_tokens, max_splits, chunk_tiles;
  float scale_log2;  // sm_scale * log2(e)
};

__device__ __forceinline__ void record_error(int* err, int bits) { atomicOr(err, bits); }

// Waits with its own time limit, ignoring the CTA's abort flag (used while draining).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  int dummy = 0;
  mbar_wait(bar, parity, &dummy);
}

template <int N, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = base;                          // 2 halves x N rows x 128 B
  uint8_t* sKV = sQ + N * 256;                 // STAGES x 32 KB
  uint8_t* sP = sKV + STAGES * kStageBytes;    // 2 buffers x (2 K-atoms x N rows x 128 B)

  __shared__ uint64_t bar_q, bar_full[STAGES], bar_empty[STAGES], bar_sfull, bar_sfree;
  __shared__ uint64_t bar_pfull[2], bar_pempty[2], bar_oready, bar_ofull, bar_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int s_last;
  __shared__ float s_m[N], s_mc[N], s_alpha[N], s_l[N];
  __shared__ float s_red[4][N];

  // ---- work item
  int item = blockIdx.x;
  const int rg = item % p.row_groups;
  item /= p.row_groups;
  const int split = item % p.max_splits;
  item /= p.max_splits;
  const int kvh = item % p.Hkv;
  const int b = item / p.Hkv;
  const int prefix = p.prefix_lens[b];
  const long long max_tok = static_cast<long long>(p.max_pages) * kPage;
  long long kvl = static_cast<long long>(prefix < 0 ? 0 : prefix) + p.L;
  const bool len_bad = prefix < 0 || kvl > max_tok;
  if (kvl > max_tok) kvl = max_tok;
  const int kv_len = static_cast<int>(kvl);
  const int t_begin = split * p.split_tokens;
  if (len_bad && split == 0 && rg == 0 && threadIdx.x == 0) record_error(p.err, BDLM_DEVERR_LENGTH);
  if (t_begin >= kv_len) return;
  const int t_end = min(kv_len, t_begin + p.split_tokens);
  const int n_splits = (kv_len + p.split_tokens - 1) / p.split_tokens;
  const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;
  const int n_chunks = (n_tiles + p.chunk_tiles - 1) / p.chunk_tiles;
  const int rows = p.rows_per_group;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- setup
  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_sfull, 1);
    mbar_init(&bar_sfree, kSoftmaxThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_pfull[i], kSoftmaxThreads);
      mbar_init(&bar_pempty[i], 1);
    }
    mbar_init(&bar_oready, kSoftmaxThreads);
    mbar_init(&bar_ofull, 1);
    mbar_init(&bar_done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    // zero the padding rows of the Q operand (rows >= rows_per_group)
    const int t = threadIdx.x - 64;
    const int pad_bytes = (N - rows) * 128;
    for (int o = t * 16; o < pad_bytes; o += kSoftmaxThreads * 16) {
      *reinterpret_cast<uint4*>(sQ + rows * 128 + o) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sQ + N * 128 + rows * 128 + o) = make_uint4(0, 0, 0, 0);
    }
    const int x = ((warp & 3) << 5) | lane;
    if (x < N) s_m[x] = -CUDART_INF_F;
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t tS = tmem;
  const uint32_t tO = tmem + static_cast<uint32_t>(p.chunk_tiles * N);

  if (warp == 0) {
    // =================================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&bar_q, 2u * 128u * static_cast<uint32_t>(p.G * p.lsub));
      for (int h = 0; h < 2; ++h)
        tma_load_3d(sQ + h * N * 128, &tm_q, &bar_q, h * 64, kvh * p.G, b * p.L + rg * p.lsub);
      const int32_t* pt = p.page_table + static_cast<size_t>(b) * p.max_pages;
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int c = 0; c < n_chunks && ok; ++c) {
        const int j0 = c * p.chunk_tiles;
        const int j1 = min(n_tiles, j0 + p.chunk_tiles);
        for (int pass = 0; pass < 2 && ok; ++pass) {
          const CUtensorMap* tm = pass == 0 ? &tm_k : &tm_v;
          for (int j = j0; j < j1; ++j) {
            if (!(ok = mbar_wait(&bar_empty[st], ph ^ 1, &abort_flag))) break;
            const int tok0 = t_begin + j * kTile;
            const int npg = min(kTile / kPage, (t_end - tok0 + kPage - 1) / kPage);
            int pid[kTile / kPage];
            uint32_t bytes = 0;
            for (int q = 0; q < npg; ++q) {
              int id = pt[tok0 / kPage + q];
              if (id < 0 || id >= p.num_pages) {
                if (pass == 0) record_error(p.err, BDLM_DEVERR_PAGE);
                id = -1;
              } else {
                bytes += 2 * 2048;
              }
              pid[q] = id;
            }
            uint8_t* stage = sKV + st * kStageBytes;
            if (bytes)
              mbar_arrive_expect_tx(&bar_full[st], bytes);
            else
              mbar_arrive(&bar_full[st]);
            for (int q = 0; q < npg; ++q) {
              if (pid[q] < 0) continue;
              tma_load_4d(stage + q * 2048, tm, &bar_full[st], 0, kvh, 0, pid[q]);
              tma_load_4d(stage + kHalfBytes + q * 2048, tm, &bar_full[st], 64, kvh, 0, pid[q]);
            }
            if (++st == STAGES) {
              st = 0;
              ph ^= 1;
            }
          }
        }
      }
      if (!ok) {
        // drain: every stage's most recent load must land before the CTA exits
        for (int s = 0; s < STAGES; ++s) mbar_wait_drain(&bar_full[s], ph ^ (s < st ? 0 : 1));
      }
    }
  } else if (warp == 1) {
    // =================================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, N, false, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(128, N, true, false);
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t kv_addr = smem_u32(sKV);
      const uint32_t p_addr = smem_u32(sP);
      bool ok = mbar_wait(&bar_q, 0, &abort_flag);
      int st = 0;
      uint32_t ph = 0;
      int pcount = 0;
      for (int c = 0; c < n_chunks && ok; ++c) {
        const int j0 = c * p.chunk_tiles;
        const int j1 = min(n_tiles, j0 + p.chunk_tiles);
        if (c > 0 && !(ok = mbar_wait(&bar_sfree, (c - 1) & 1, &abort_flag))) break;
        tc_fence_after();
        // S^T[tile] = K[tile] . Q^T, K over the 128 head dims in 8 steps of 16
        for (int j = j0; j < j1; ++j) {
          if (!(ok = mbar_wait(&bar_full[st], ph, &abort_flag))) break;
          tc_fence_after();
          const uint32_t ka = kv_addr + st * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = smem_desc(ka + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc(q_addr + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
            umma_bf16(tS + (j - j0) * N, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bar_empty[st]);
          if (++st == STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&bar_sfull);
        // O^T += V^T[tile] . P^T[tile], K over the tile's pages (16 tokens each)
        for (int j = j0; j < j1; ++j) {
          const int pb = pcount & 1;
          if (!(ok = mbar_wait(&bar_full[st], ph, &abort_flag))) break;
          if (!(ok = mbar_wait(&bar_pfull[pb], (pcount >> 1) & 1, &abort_flag))) break;
          if (c > 0 && j == j0 && !(ok = mbar_wait(&bar_oready, (c - 1) & 1, &abort_flag))) break;
          tc_fence_after();
          const int tok0 = t_begin + j * kTile;
          const int valid = min(kTile, t_end - tok0);
          const int npg = (valid + kPage - 1) / kPage;
          const int tail = valid - (npg - 1) * kPage;
          uint8_t* stage = sKV + st * kStageBytes;
          if (tail < kPage) {
            // slots past the sequence end may hold anything (NaN): 0 * NaN would poison O
            for (int h = 0; h < 2; ++h) {
              uint4* z = reinterpret_cast<uint4*>(stage + h * kHalfBytes + (npg - 1) * 2048 +
                                                  tail * 128);
              for (int o = 0; o < (kPage - tail) * 8; ++o) z[o] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          const uint32_t va = kv_addr + st * kStageBytes;
          const uint32_t pa = p_addr + pb * (N * 256);
          for (int q = 0; q < npg; ++q) {
            const uint64_t ad = smem_desc(va + q * 2048, kHalfBytes, 1024);
            const uint64_t bd = smem_desc(pa + (q >> 2) * (N * 128) + (q & 3) * 32, 16, 1024);
            umma_bf16(tO, ad, bd, kIdescO, (c > 0 || j > j0 || q > 0) ? 1u : 0u);
          }
          umma_commit(&bar_empty[st]);
          umma_commit(&bar_pempty[pb]);
          ++pcount;
          if (++st == STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&bar_ofull);
      }
      umma_commit(&bar_done);
    }
  } else {
    // =================================================================== softmax/epilogue
    const int q4 = warp & 3;
    const int x = (q4 << 5) | lane;  // tensor-memory lane: KV token of a tile, or head dim
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const float cs = p.scale_log2;
    float l[N];
#pragma unroll
    for (int n = 0; n < N; ++n) l[n] = 0.f;
    bool ok = true;
    int pcount = 0;
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int j0 = c * p.chunk_tiles;
      const int j1 = min(n_tiles, j0 + p.chunk_tiles);
      if (!(ok = mbar_wait(&bar_sfull, c & 1, &abort_flag))) break;
      tc_fence_after();
      // phase A: exact column maxima over the chunk
#pragma unroll
      for (int cg = 0; cg < N / 16; ++cg) {
        float mx[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) mx[k] = -CUDART_INF_F;
        for (int j = j0; j < j1; ++j) {
          uint32_t r[16];
          tmem_ld16(tS + lane_off + (j - j0) * N + cg * 16, r);
          tmem_wait_ld();
          tmem_regs_ready(r);
          const bool valid = t_begin + j * kTile + x < t_end;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (valid) mx[k] = fmaxf(mx[k], __uint_as_float(r[k]));
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
            mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], off));
        }
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < 16; ++k) s_red[q4][cg * 16 + k] = mx[k];
        }
      }
      named_barrier(1, kSoftmaxThreads);
      if (x < N) {
        const float mc = fmaxf(fmaxf(s_red[0][x], s_red[1][x]), fmaxf(s_red[2][x], s_red[3][x]));
        const float mo = s_m[x];
        const float mn = fmaxf(mo, mc);
        s_alpha[x] = (mo == -CUDART_INF_F) ? 0.f : exp2f((mo - mn) * cs);
        s_m[x] = mn;
        s_mc[x] = mn * cs;
      }
      named_barrier(1, kSoftmaxThreads);
      if (c > 0) {
        // rescale the running O^T columns (and l) to the new maxima
        if (!(ok = mbar_wait(&bar_ofull, (c - 1) & 1, &abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int cg = 0; cg < N / 16; ++cg) {
          uint32_t r[16];
          tmem_ld16(tO + lane_off + cg * 16, r);
          tmem_wait_ld();
          tmem_regs_ready(r);
#pragma unroll
          for (int k = 0; k < 16; ++k)
            r[k] = __float_as_uint(__uint_as_float(r[k]) * s_alpha[cg * 16 + k]);
          tmem_st16(tO + lane_off + cg * 16, r);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_oready);
#pragma unroll
        for (int n = 0; n < N; ++n) l[n] *= s_alpha[n];
      }
      // phase B: P^T = exp(S^T - m) to shared memory, tile by tile
      for (int j = j0; j < j1 && ok; ++j) {
        const int pb = pcount & 1;
        if (!(ok = mbar_wait(&bar_pempty[pb], ((pcount >> 1) & 1) ^ 1, &abort_flag))) break;
        uint8_t* pbuf = sP + pb * (N * 256) + (x >> 6) * (N * 128);
        const bool valid = t_begin + j * kTile + x < t_end;
        const uint32_t xc = (x & 63) >> 3;
        const uint32_t xb = (x & 7) * 2;
#pragma unroll
        for (int cg = 0; cg < N / 16; ++cg) {
          uint32_t r[16];
          tmem_ld16(tS + lane_off + (j - j0) * N + cg * 16, r);
          tmem_wait_ld();
          tmem_regs_ready(r);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int n = cg * 16 + k;
            const float pv = valid ? exp2f(fmaf(__uint_as_float(r[k]), cs, -s_mc[n])) : 0.f;
            l[n] += pv;
            const uint32_t off = n * 128 + ((xc ^ (n & 7)) << 4) + xb;
            *reinterpret_cast<__nv_bfloat16*>(pbuf + off) = __float2bfloat16_rn(pv);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar_pfull[pb]);
        ++pcount;
      }
      if (!ok) break;
      tc_fence_before();
      mbar_arrive(&bar_sfree);
    }
    // ---- epilogue
    if (ok) ok = mbar_wait(&bar_ofull, (n_chunks - 1) & 1, &abort_flag);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int n = 0; n < N; ++n) {
        float v = l[n];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        l[n] = v;
      }
      if (lane == 0) {
#pragma unroll
        for (int n = 0; n < N; ++n) s_red[q4][n] = l[n];
      }
      named_barrier(1, kSoftmaxThreads);
      if (x < N) s_l[x] = (s_red[0][x] + s_red[1][x]) + (s_red[2][x] + s_red[3][x]);
      named_barrier(1, kSoftmaxThreads);
      const size_t head_base = static_cast<size_t>(kvh) * p.G;
      if (n_splits == 1) {
#pragma unroll
        for (int cg = 0; cg < N / 16; ++cg) {
          uint32_t r[16];
          tmem_ld16(tO + lane_off + cg * 16, r);
          tmem_wait_ld();
          tmem_regs_ready(r);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int n = cg * 16 + k;
            if (n >= rows) continue;
            const int i = rg * p.lsub + n / p.G;
            if (i >= p.L) continue;
            const size_t o = ((static_cast<size_t>(b) * p.L + i) * p.Hq + head_base + n % p.G) * 128 + x;
            p.out[o] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[k]) / s_l[n]));
          }
        }
      } else {
        const size_t unit = static_cast<size_t>(N) * 130;
        const size_t grp = (static_cast<size_t>(b) * p.Hkv + kvh) * p.row_groups + rg;
        float* mine = p.part + (grp * p.max_splits + split) * unit;
#pragma unroll
        for (int cg = 0; cg < N / 16; ++cg) {
          uint32_t r[16];
          tmem_ld16(tO + lane_off + cg * 16, r);
          tmem_wait_ld();
          tmem_regs_ready(r);
#pragma unroll
          for (int k = 0; k < 16; ++k) mine[(cg * 16 + k) * 128 + x] = __uint_as_float(r[k]);
        }
        if (x < N) {
          mine[N * 128 + x] = s_m[x];
          mine[N * 128 + N + x] = s_l[x];
        }
        __threadfence();
        named_barrier(1, kSoftmaxThreads);
        if (x == 0) s_last = (atomicAdd(p.cnt + grp, 1) == n_splits - 1);
        named_barrier(1, kSoftmaxThreads);
        if (s_last) {
          __threadfence();
          const float* all = p.part + grp * p.max_splits * unit;
          for (int n = 0; n < rows; ++n) {
            const int i = rg * p.lsub + n / p.G;
            if (i >= p.L) break;
            float M = -CUDART_INF_F;
            for (int s = 0; s < n_splits; ++s) M = fmaxf(M, __ldcg(all + s * unit + N * 128 + n));
            float num = 0.f, den = 0.f;
            for (int s = 0; s < n_splits; ++s) {
              const float w = exp2f((__ldcg(all + s * unit + N * 128 + n) - M) * cs);
              num += w * __ldcg(all + s * unit + n * 128 + x);
              den += w * __ldcg(all + s * unit + N * 128 + N + n);
            }
            const size_t o = ((static_cast<size_t>(b) * p.L + i) * p.Hq + head_base + n % p.G) * 128 + x;
            p.out[o] = __bfloat16_as_ushort(__float2bfloat16_rn(num / den));
          }
          if (x == 0) p.cnt[grp] = 0;
        }
      }
    }
  }

  // ---- teardown: all MMAs retired before tensor memory is released
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) mbar_wait_drain(&bar_done, 0);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && abort_flag) record_error(p.err, BDLM_DEVERR_TIMEOUT);
}

template <int N, int STAGES>
size_t smem_bytes() {
  return 1024 + static_cast<size_t>(N) * 256 + static_cast<size_t>(STAGES) * kStageBytes +
         static_cast<size_t>(2) * N * 256;
}

template <int N, int STAGES>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const AttnParams& prm, int grid, cudaStream_t stream) {
  const size_t smem = smem_bytes<N, STAGES>();
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<N, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  attn_kernel<N, STAGES><<<grid, kThreads, smem, stream>>>(tq, tk, tv, prm);
  return cudaGetLastError();
}

}  // namespace

AttnPlan plan_attention(int B, int L, int Hq, int Hkv, int max_pages, int page_size) {
  AttnPlan pl;
  if (page_size != kPage || Hkv <= 0 || Hq % Hkv != 0) {
    pl.n_mma = 0;
    return pl;
  }
  pl.G = Hq / Hkv;
  pl.rows = pl.G * L;
  if (pl.rows <= 128) {
    pl.lsub = L;
    pl.row_groups = 1;
  } else {
    pl.lsub = 128 / pl.G;
    pl.row_groups = (L + pl.lsub - 1) / pl.lsub;
  }
  const int rpg = pl.G * pl.lsub;
  pl.n_mma = rpg <= 16 ? 16 : rpg <= 32 ? 32 : rpg <= 64 ? 64 : 128;
  pl.chunk_tiles = (static_cast<int>(kTmemCols) - pl.n_mma) / pl.n_mma;
  pl.split_tokens = pl.n_mma <= 32 ? 1024 : 2048;
  const long long max_tok = static_cast<long long>(max_pages) * kPage;
  pl.max_splits = static_cast<int>((max_tok + pl.split_tokens - 1) / pl.split_tokens);
  pl.tmem_cols = kTmemCols;
  const size_t groups = static_cast<size_t>(B) * Hkv * pl.row_groups;
  pl.part_bytes = groups * pl.max_splits * static_cast<size_t>(pl.n_mma) * 130 * sizeof(float);
  pl.cnt_bytes = groups * sizeof(int);
  return pl;
}

cudaError_t launch_attention(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const int32_t* page_table,
                             const int32_t* prefix_lens, uint16_t* out, int B, int L, int Hq,
                             int Hkv, int max_pages, int num_pages, float sm_scale,
                             const AttnPlan& plan, float* part, int* cnt, int* err,
                             cudaStream_t stream) {
  AttnParams prm;
  prm.page_table = page_table;
  prm.prefix_lens = prefix_lens;
  prm.out = out;
  prm.part = part;
  prm.cnt = cnt;
  prm.err = err;
  prm.L = L;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = plan.G;
  prm.max_pages = max_pages;
  prm.num_pages = num_pages;
  prm.lsub = plan.lsub;
  prm.row_groups = plan.row_groups;
  prm.rows_per_group = plan.G * plan.lsub;
  prm.split_tokens = plan.split_tokens;
  prm.max_splits = plan.max_splits;
  prm.chunk_tiles = plan.chunk_tiles;
  prm.scale_log2 = sm_scale * 1.4426950408889634f;
  const long long grid_ll = static_cast<long long>(B) * Hkv * plan.max_splits * plan.row_groups;
  if (grid_ll > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(grid_ll);
  switch (plan.n_mma) {
    case 16: return launch_t<16, 3>(tm_q, tm_k, tm_v, prm, grid, stream);
    case 32: return launch_t<32, 2>(tm_q, tm_k, tm_v, prm, grid, stream);
    case 64: return launch_t<64, 4>(tm_q, tm_k, tm_v, prm, grid, stream);
    case 128: return launch_t<128, 3>(tm_q, tm_k, tm_v, prm, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace bdlm
