// Definitions of the block-attention kernels (attention.cu): tile and page geometry, kernel
// parameters, the work item and its decoding, and the softmax helpers.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {

namespace {

constexpr int kTile = 128;          // KV tokens per tile (UMMA M)
constexpr int kPage = 16;           // tokens per page
constexpr int kStageBytes = 32768;  // one K or V tile: 2 halves x 8 pages x 16 slots x 128 B
constexpr int kHalfBytes = 16384;
constexpr int kSoftmaxThreads = 128;   // transposed mode: warps 2-5, after producer and MMA
// the rows-on-M kernel: two softmax warps per tensor-memory lane quadrant
constexpr int kRowSoftmaxThreads = 256;
// threads of a CTA: the transposed mode has warps 0-1 (producer, MMA) and 4 softmax warps; with
// rows on M 8 softmax warps per sub-group (two per lane quadrant) and a second K/V copy issuer
__host__ __device__ constexpr int attn_softmax_threads(bool rows, bool two) {
  return rows ? kRowSoftmaxThreads * (two ? 2 : 1) : kSoftmaxThreads;
}
__host__ __device__ constexpr int attn_threads(bool rows, bool two) {
  return 64 + attn_softmax_threads(rows, two) + (rows ? 32 : 0);
}
constexpr int kMaxSplitTokens = 2048;
// Page ids staged per item: a split of up to kMaxSplitTokens, or a whole sequence of up to
// kMaxItemPages pages when sequences are processed whole (two CTAs per SM at N = 16 leave
// no room for more).  The rows-on-M kernels (one CTA per SM) stage up to kMaxItemPagesRows
// pages, for splits of up to kMaxSplitTokensRows.
constexpr int kMaxItemPages = kMaxSplitTokens / kPage;
static_assert(kMaxItemPages >= kMaxSplitTokens / kPage, "a split must fit the page-id buffer");
constexpr int kMaxSplitTokensRows = 8192;
constexpr int kMaxItemPagesRows = kMaxSplitTokensRows / kPage;
// Longest KV split of the rows-on-M kernels: one 128-row sub-group, two sub-groups.
constexpr int kSplitTokensRows = 3072;
constexpr int kSplitTokensTwo = 4096;
static_assert(kSplitTokensRows <= kMaxSplitTokensRows && kSplitTokensTwo <= kMaxSplitTokensRows &&
                  kSplitTokensRows % kTile == 0 && kSplitTokensTwo % kTile == 0,
              "a split is whole tiles and fits the page-id buffer");
// Whole sequences, longest first, replace KV splits when there are at least this many
// (sequence, KV head, row group) items per CTA and up to kMaxOrderSeqs sequences.
constexpr int kWholeItemsPerCta = 2;
constexpr int kMaxOrderSeqs = 1024;
// A chunk moves a column's running softmax max only when it raises it by more than this
// (log2 units of the scaled scores), so P never exceeds 2^kLazyRescale.
constexpr float kLazyRescale = 8.0f;
constexpr int kItemRing = 4;

}  // namespace

struct AttnParams {
  const int32_t* page_table;
  const int32_t* prefix_lens;
  // the block's new K/V [B, L, Hkv, D] and the pools to write them into (null: the block's K/V
  // are already in the cache)
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_pool;
  uint16_t* v_pool;
  uint16_t* out;
  float* part;
  int* err;
  int* work;  // [0] next item, [1] CTAs finished
  const int* order;  // whole-sequence mode: sequences by decreasing KV length, else null
  int B, L, Hq, Hkv, G, max_pages, num_pages;
  int table_div;     // sequence b uses page-table row b / table_div (prompt blocks share a row)
  int lsub, row_groups, rows_per_group, split_tokens, max_splits, chunk_tiles;
  int even_splits;   // cut each sequence into equal splits of at most split_tokens
  int rank_major;    // items sequence by sequence in `order`, all splits of one together
  int total_items;
  int mask_block;    // > 0: query i of a sequence sees keys < prefix + (i / mask_block + 1) * mask_block
  float scale_log2;  // sm_scale * log2(e)
};

// What the second copy issuer of the rows-on-M kernel needs for one ring stage.
struct StageInfo {
  int pass, kvh, end;
  int id[kTile / kPage];   // page ids of the tile (-1: past the sequence)
};

struct Item {
  int b, kvh, split, rg;
  int t_begin, t_end, n_splits;
  int q0;  // key position of the sequence's first query (its prefix length)
  int n_tiles, n_chunks;
  int end;
  int wr;  // the producer writes the block's new K/V into the cache before reading it
};

namespace {

__device__ __forceinline__ void record_error(int* err, int bits) { atomicOr(err, bits); }

// Waits with its own time limit, ignoring the CTA's abort flag (used while draining).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  int dummy = 0;
  mbar_wait(bar, parity, &dummy);
}

// KV tokens per split of a sequence of kv_len tokens: split_tokens, or with even splits the
// sequence cut into as many splits as split_tokens needs, of equal length rounded up to whole
// tiles (at most split_tokens, so a split still fits the page-id buffer; the last one takes
// what is left), so that no split is a short remainder.
__device__ __forceinline__ int split_len(int kv_len, const AttnParams& p) {
  if (!p.even_splits || kv_len <= 0) return p.split_tokens;
  const int ns = (kv_len + p.split_tokens - 1) / p.split_tokens;
  return ((kv_len + ns - 1) / ns + kTile - 1) / kTile * kTile;
}

// Item index -> work item; items are enumerated split-major so that the short last splits
// of long sequences come at the end of the schedule, or (rank_major) sequence by sequence in
// the order of `order`.  Returns false for an empty split.
__device__ __forceinline__ bool decode_item(int idx, const AttnParams& p, Item& it) {
  it.rg = idx % p.row_groups;
  idx /= p.row_groups;
  it.kvh = idx % p.Hkv;
  idx /= p.Hkv;
  if (p.rank_major) {
    // even splits, sequences by decreasing split length, all splits of one together
    it.split = idx % p.max_splits;
    it.b = __ldg(p.order + idx / p.max_splits);
  } else {
    it.b = idx % p.B;
    it.split = idx / p.B;
    if (p.order) it.b = __ldg(p.order + it.b);  // whole sequences, longest first
  }
  const int prefix = p.prefix_lens[it.b];
  const long long max_tok = static_cast<long long>(p.max_pages) * kPage;
  long long kvl = static_cast<long long>(prefix < 0 ? 0 : prefix) + p.L;
  if (kvl > max_tok) kvl = max_tok;
  const int kv_len = static_cast<int>(kvl);
  const int per = split_len(kv_len, p);
  it.t_begin = it.split * per;
  if (it.t_begin >= kv_len) return false;
  it.q0 = kv_len - p.L;
  it.t_end = min(kv_len, it.t_begin + per);
  it.n_splits = (kv_len + per - 1) / per;
  it.n_tiles = (it.t_end - it.t_begin + kTile - 1) / kTile;
  it.n_chunks = (it.n_tiles + p.chunk_tiles - 1) / p.chunk_tiles;
  it.end = 0;
  const bool len_ok = prefix >= 0 && static_cast<long long>(prefix) + p.L <= max_tok;
  it.wr = p.k_new != nullptr && len_ok;
  if (it.split == 0 && it.rg == 0 && it.kvh == 0 && !len_ok)
    record_error(p.err, BDLM_DEVERR_LENGTH);
  return true;
}

// Writes 128 bytes per lane to global memory (lane l: w, the 32 words of its row piece; dst,
// where they go, or null for nothing) through a 1 KB shared-memory staging buffer, 8 rows at a
// time, so that each global store instruction writes four whole 128-byte row pieces instead of
// 16 bytes of each of 32 rows.  Chunk c of staged row r sits at 16 * (c ^ r) within the row, so
// neither the writes of 8 rows nor the reads fall on one bank.  Whole warp.
__device__ __forceinline__ void store_rows_128b(const uint32_t (&w)[32], void* dst,
                                                uint8_t* stage, int lane) {
  const unsigned long long dptr = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
  for (int p8 = 0; p8 < 4; ++p8) {
    if ((lane >> 3) == p8) {
      const int r = lane & 7;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(stage + r * 128 + ((c ^ r) << 4)) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = (lane >> 3) + 4 * h, c = lane & 7;
      const unsigned long long d = __shfl_sync(0xffffffffu, dptr, p8 * 8 + r);
      const uint4 v = *reinterpret_cast<const uint4*>(stage + r * 128 + ((c ^ r) << 4));
      if (d) reinterpret_cast<uint4*>(d)[c] = v;
    }
    __syncwarp();
  }
}

// Rows on M, two sub-groups: 32 scores of a half-row (keys base .. base + 31 of its 64).
// FULL: all of them are keys the row sees; otherwise keys at or past nvalid read as -inf.
template <bool FULL>
__device__ __forceinline__ float max32(const uint32_t (&r)[32], int base, int nvalid) {
  float v[32];
#pragma unroll
  for (int k = 0; k < 32; ++k)
    v[k] = FULL || base + k < nvalid ? __uint_as_float(r[k]) : -CUDART_INF_F;
  // a tree of three-input maxima: 32 -> 11 -> 4 -> 1 (17 instructions)
  float t[11];
#pragma unroll
  for (int k = 0; k < 10; ++k) t[k] = fmax3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
  t[10] = fmaxf(v[30], v[31]);
  const float u0 = fmax3(t[0], t[1], t[2]), u1 = fmax3(t[3], t[4], t[5]);
  const float u2 = fmax3(t[6], t[7], t[8]), u3 = fmaxf(t[9], t[10]);
  return fmaxf(fmax3(u0, u1, u2), u3);
}

// p = 2^(s cs - m cs) of the same 32 scores, packed as bf16 pairs into pk; returns their sum.
template <bool FULL>
__device__ __forceinline__ float exp_pack32(const uint32_t (&r)[32], int base, int nvalid,
                                            float2 cs2, float2 nm2, uint32_t (&pk)[16]) {
  float2 e[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float a = FULL || base + 2 * k < nvalid ? __uint_as_float(r[2 * k]) : -CUDART_INF_F;
    const float b =
        FULL || base + 2 * k + 1 < nvalid ? __uint_as_float(r[2 * k + 1]) : -CUDART_INF_F;
    const float2 y = __ffma2_rn(make_float2(a, b), cs2, nm2);
    e[k] = make_float2(ex2(y.x), ex2(y.y));
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(e[k].x, e[k].y);
    pk[k] = *reinterpret_cast<const uint32_t*>(&h2);
  }
#pragma unroll
  for (int w = 8; w > 0; w >>= 1)
#pragma unroll
    for (int k = 0; k < w; ++k) e[k] = __fadd2_rn(e[k], e[k + w]);
  return e[0].x + e[0].y;
}

}  // namespace
}  // namespace bdlm
