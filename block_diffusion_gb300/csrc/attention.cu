// Block attention of one denoising round over a paged KV cache, for sm_103a.
//
// Source: JetEngine notes (CLAUDE.md), "ModelRunner" and "Optimization History" (opt18,
// opt24: paged-KV attention for the denoise forward); JetEngine README, "Block Diffusion
// Decoding".  For sequence b, block position i and query head h:
//     out = softmax_j(scale * q . K[j]) V[j]   over every j < prefix_len + L
// (full prefix, bidirectional inside the block), KV head = h / (Hq/Hkv).
//
// Design.
//  * Work item = (sequence, KV head, KV split, query-row group).  GQA packing: the G*L query
//    rows that share a KV head form one UMMA operand, so each K/V page is read once per KV
//    head.  The product is computed transposed, S^T = K Q^T, with 128 KV tokens on the UMMA
//    M side and the query rows on N, so a 4-token block still fills a 128-row tile.
//  * Persistent CTAs take items from a global counter.  Warp 0 streams K and V pages with
//    TMA (one 16-slot x 64-dim box per page and half, 128-byte swizzle) into a ring of 32 KB
//    stages; warp 1 issues tcgen05.mma from shared memory into tensor memory; warps 2-5 (one
//    thread per tensor-memory lane) run the softmax and the epilogue.
//  * An item is cut into chunks of tiles whose S^T fits in tensor memory.  Softmax per chunk
//    in two phases: all S^T tiles first, the exact column maximum once, then P^T = exp(S^T-m)
//    (bf16, shared memory) and O^T += V^T P^T in tensor memory; a later chunk moves the
//    running max (and rescales O^T) only when it raises it by more than 2^kLazyRescale.  The
//    ring carries K of chunk u+1 ahead of V of chunk u and S^T is double-buffered, so the
//    softmax of one chunk overlaps the K stream of the next and the pipeline never drains
//    between items.
//  * Either whole sequences, longest first (when there are enough items), or splits of a
//    long sequence that write (O, m, l) partials merged by a small second kernel; no CTA
//    ever waits on another one, and every wait inside a CTA is bounded.
//  * More than 32 query rows per KV head (ROWS): S = Q K^T with 128 query rows on M, a row per
//    tensor-memory lane, two softmax threads per row (half a row each); P is written over the
//    S columns it came from and is the PV MMA's A operand in tensor memory.  With one 128-row
//    sub-group Q is copied into tensor memory too (tcgen05.cp) and the ring has five stages;
//    with two sub-groups (TWO, up to 256 rows) both share every K/V stage and sixteen softmax
//    warps work on both at once.  The block-causal prefill mask (MASKED) applies per row.
//    These kernels cut a sequence into equal splits (each item reloads Q and writes a large
//    partial, so no split is a short remainder), hand the items out longest splits first,
//    stage the epilogue's stores through shared memory (whole 128-byte rows per store
//    instruction), and wait with a suspend-time hint (fewer re-tries taking issue slots).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "attention_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

template <int N, int STAGES, int CTAS_PER_SM, bool MASKED, bool ROWS, bool TWO>
__global__ void __launch_bounds__(attn_threads(ROWS, TWO), CTAS_PER_SM)
attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  constexpr uint32_t kTmemCols = 512 / CTAS_PER_SM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // With rows on M an item has one or two (TWO) sub-groups of 128 query rows; they share every
  // K/V stage, each with its own S and O in tensor memory.
  constexpr int kSub = TWO ? 2 : 1;
  constexpr int kRowsItem = N * kSub;          // query rows of an item
  // One Q buffer: 4 KB at N = 16 in the transposed mode, 64 KB for two sub-groups; with rows on
  // M and one sub-group it only stages Q, which the MMA issuer copies into tensor memory (the S
  // MMA's A operand) as the item starts, so the next item's Q can land during this item
  constexpr int kQBufs = 1;
  constexpr bool kQTmem = ROWS && !TWO;
  uint8_t* sQ = base;                          // 2 halves x kRowsItem rows x 128 B
  uint8_t* sKV = sQ + kQBufs * kRowsItem * 256;   // STAGES x 32 KB
  uint8_t* sP = sKV + STAGES * kStageBytes;    // transposed mode: 2 buffers x (2 K-atoms x N rows x 128 B)

  __shared__ uint64_t bar_qfull[kQBufs], bar_qempty[kQBufs], bar_full[STAGES], bar_empty[STAGES];
  __shared__ uint64_t bar_sfull[2], bar_sfree[2], bar_pfull[2], bar_pempty[2];
  __shared__ uint64_t bar_oready, bar_ofull[2], bar_done;  // bar_ofull: PV of chunk u, by parity
  __shared__ uint64_t bar_ifull[kItemRing], bar_iempty[kItemRing];
  __shared__ Item s_item[kItemRing];
  __shared__ int s_pid[3][ROWS ? kMaxItemPagesRows : kMaxItemPages];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  constexpr int kCols = ROWS ? 1 : N;   // per-column state of the transposed softmax
  __shared__ float s_m[kCols], s_mc[kCols], s_alpha[kCols], s_l[kCols];
  __shared__ int s_need[2];   // chunk u (parity): some column's max rose enough to rescale O^T
  __shared__ int s_pflag[2];  // P buffer: its tile starts a chunk whose PV waits for a rescale
  __shared__ float s_red[4][kCols];
  // rows on M: a 1 KB staging buffer per softmax warp for the epilogue's global stores
  __shared__ __align__(16) uint8_t
      s_stage[ROWS ? attn_softmax_threads(ROWS, TWO) / 32 : 1][ROWS ? 1024 : 16];
  // the two halves of a row exchange maxima and sums, by exchange parity and sub-group; their
  // mbarriers are per (sub-group, lane quadrant)
  __shared__ float s_hmax[ROWS ? 2 : 1][TWO ? 2 : 1][2][ROWS ? N : 1];
  __shared__ float s_hsum[ROWS ? 2 : 1][TWO ? 2 : 1][2][ROWS ? N : 1];
  __shared__ uint64_t bar_pair[ROWS ? (TWO ? 8 : 4) : 1][2], bar_pair_end[ROWS ? (TWO ? 8 : 4) : 1];
  // rows on M: the producer issues half 0 of each stage's page boxes and hands the stage to a
  // second issuer warp for half 1 (one warp's copies issue at about 1 us per 16 boxes)
  __shared__ StageInfo s_sinfo[ROWS ? STAGES : 1];
  __shared__ uint64_t bar_sready[ROWS ? STAGES : 1];
  constexpr int kSoftmax = attn_softmax_threads(ROWS, TWO);
  constexpr int kIssueWarp = 2 + kSoftmax / 32;   // rows on M: the second K/V copy issuer
  // P buffers: the transposed softmax double-buffers P^T in shared memory; with rows on M, P is
  // written over the S columns it came from (the PV MMA's A operand; the tensor pipe executes
  // one thread's MMAs in issue order, so the next S into those columns, issued after that PV,
  // cannot overwrite P before the PV has read it).  Tensor memory with rows on M: S buffers
  // 0-255, O 256-383 and Q 384-447 (one sub-group); S_0, S_1, O_0, O_1 (two sub-groups).
  constexpr bool kPTmem = ROWS && !TWO;
  constexpr int kPBufs = 2;
  constexpr uint32_t kQCol = 384;   // first tensor-memory column of Q (kQTmem)
  static_assert(!MASKED || ROWS, "the block-causal mask is applied by the row-per-thread softmax");
  static_assert(!ROWS || N == 128, "rows on M: one UMMA of 128 query rows");
  static_assert(!TWO || ROWS, "two sub-groups only with rows on M");
  static_assert(ROWS || N <= 32, "keys on M: at most 32 query rows on N");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- setup
  if (threadIdx.x == 0) {
    for (int b = 0; b < kQBufs; ++b) {
      mbar_init(&bar_qfull[b], 1);
      mbar_init(&bar_qempty[b], 1);
    }
    for (int s = 0; s < STAGES; ++s) {
      // rows on M: the producer's arming arrival and the second issuer's, so that a stage with
      // no valid page cannot complete (and be refilled) before the issuer has read it
      mbar_init(&bar_full[s], ROWS ? 2 : 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_sfull[i], 1);
      mbar_init(&bar_sfree[i], kSoftmax);
      mbar_init(&bar_pfull[i], TWO ? kSoftmax / 2 : kSoftmax);   // TWO: one per sub-group
      mbar_init(&bar_pempty[i], 1);
    }
    mbar_init(&bar_oready, kSoftmaxThreads);
    mbar_init(&bar_ofull[0], 1);
    mbar_init(&bar_ofull[1], 1);
    mbar_init(&bar_done, 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&bar_ifull[i], 1);
      // the MMA warp, and one softmax thread (every softmax thread with rows on M)
      mbar_init(&bar_iempty[i], ROWS ? 1 + kSoftmax : 2);
    }
    if constexpr (ROWS) {
      for (int s = 0; s < STAGES; ++s) mbar_init(&bar_sready[s], 1);
      for (int q = 0; q < (TWO ? 8 : 4); ++q) {
        mbar_init(&bar_pair[q][0], 64);
        mbar_init(&bar_pair[q][1], 64);
        mbar_init(&bar_pair_end[q], 64);
      }
    }
    abort_flag = 0;
    s_need[0] = s_need[1] = 0;
    s_pflag[0] = s_pflag[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2 && warp < 2 + kSoftmax / 32) {
    // zero the padding rows of the Q operand (rows >= rows_per_group); TMA never writes them
    const int rows = p.rows_per_group;
    const int t = threadIdx.x - 64;
    for (int o = t * 16; o < (kRowsItem - rows) * 128; o += kSoftmax * 16) {
      for (int b = 0; b < kQBufs; ++b) {
        *reinterpret_cast<uint4*>(sQ + b * kRowsItem * 256 + rows * 128 + o) =
            make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sQ + b * kRowsItem * 256 + kRowsItem * 128 + rows * 128 + o) =
            make_uint4(0, 0, 0, 0);
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();  // inputs written by the previous grid on the stream are visible from here
  const uint32_t tmem = tmem_base;
  const uint32_t tO = tmem + static_cast<uint32_t>(2 * p.chunk_tiles * N);

  if (warp == 0) {
    // =================================================================== TMA producer
    int st = 0;
    uint32_t ph = 0;
    bool ok = true;
    int seq = -1;  // sequence number of the most recently published item
    // Publishes `it` to the item ring (lane 0).
    auto publish = [&](const Item& it) {
      const int rs = seq % kItemRing;
      if (ok) ok = mbar_wait<ROWS>(&bar_iempty[rs], ((seq / kItemRing) & 1) ^ 1, &abort_flag);
      s_item[rs] = it;
      mbar_arrive(&bar_ifull[rs]);
    };
    // Takes the next non-empty item from the global counter, publishes it to the item ring
    // and loads its page ids (whole warp).  When the work is done it publishes the end marker
    // at once (the MMA warp needs it before it can finish the current item) and returns false.
    auto grab = [&](Item& it) -> bool {
      while (true) {
        int idx = 0;
        if (lane == 0) idx = atomicAdd(p.work, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx >= p.total_items) {
          ++seq;
          if (lane == 0) {
            Item e{};
            e.end = 1;
            publish(e);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          return false;
        }
        if (decode_item(idx, p, it)) break;
      }
      ++seq;
      int* pid = s_pid[seq % 3];
      const int32_t* pt =
          p.page_table + static_cast<size_t>(it.b / p.table_div) * p.max_pages + it.t_begin / kPage;
      const int np = (it.t_end - it.t_begin + kPage - 1) / kPage;
      int bad = 0;
      for (int q = lane; q < np; q += 32) {
        int id = pt[q];
        if (id < 0 || id >= p.num_pages) {
          bad = 1;
          id = -1;
        }
        pid[q] = id;
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(p.err, BDLM_DEVERR_PAGE);
      __syncwarp();
      if (it.wr && max(it.t_begin, it.q0) < it.t_end) {
        // With the block's K/V-cache write fused in: the new K and V rows of the block tokens
        // this item reads go to their cache slots now, a batch of 16-byte chunks per lane at a
        // time (loads first, then stores), and a proxy fence orders the stores before the
        // item's page boxes read them.  The item is taken one ahead, while the ring is full,
        // so this work is off the copy stream.  Every item that reads a token writes it (row
        // groups store the same bytes), so no item depends on another CTA.
        const int w0 = max(it.t_begin, it.q0), n = (it.t_end - w0) * 32;
        constexpr int kBatch = 4;
        for (int c0 = 0; c0 < n; c0 += 32 * kBatch) {
          uint4 v[kBatch];
          uint4* dst[kBatch];
#pragma unroll
          for (int x = 0; x < kBatch; ++x) {
            const int c = c0 + x * 32 + lane;
            dst[x] = nullptr;
            if (c >= n) continue;
            const int t = w0 + c / 32, kv = (c / 16) & 1, q = c % 16;
            const int id = pid[(t - it.t_begin) / kPage];
            if (id < 0) continue;   // a bad page id (flagged above): its rows are skipped
            const size_t row = (static_cast<size_t>(it.b) * p.L + (t - it.q0)) * p.Hkv + it.kvh;
            v[x] = __ldg(reinterpret_cast<const uint4*>((kv ? p.v_new : p.k_new) + row * 128) + q);
            dst[x] = reinterpret_cast<uint4*>(
                         (kv ? p.v_pool : p.k_pool) +
                         ((static_cast<size_t>(id) * kPage + t % kPage) * p.Hkv + it.kvh) * 128) + q;
          }
#pragma unroll
          for (int x = 0; x < kBatch; ++x)
            if (dst[x] != nullptr) *dst[x] = v[x];
        }
        fence_proxy_async_global();
        __syncwarp();
      }
      if (lane == 0) publish(it);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      return true;
    };
    // K/V pages are read exactly once: first to leave L2, so that the split partials (and Q)
    // stay resident for the merge
    const uint64_t kv_policy = l2_policy_evict_first();
    // Loads the Q tile of item `it` (sequence number s) into Q buffer s % kQBufs once the item
    // that used it before is done with it (its last S MMA, or with Q in tensor memory the copy
    // out of the buffer).  Lane 0.
    int q_loads = 0;
    auto load_q = [&](const Item& it, int s) {
      const int b = s % kQBufs;
      if (ok) ok = mbar_wait<ROWS>(&bar_qempty[b], ((s / kQBufs) & 1) ^ 1, &abort_flag);
      if (!ok) return;
      mbar_arrive_expect_tx(&bar_qfull[b], 2u * 128u * static_cast<uint32_t>(p.G * p.lsub));
      for (int h = 0; h < 2; ++h)
        tma_load_3d(sQ + b * kRowsItem * 256 + h * kRowsItem * 128, &tm_q, &bar_qfull[b], h * 64,
                    it.kvh * p.G, it.b * p.L + it.rg * p.lsub);
      ++q_loads;
    };
    // Streams the K (pass 0) or V (pass 1) tiles of chunk c of item `it` (page ids in
    // s_pid[pbuf]).  Whole warp: lane 0 waits for a free stage and posts the byte count, then
    // lanes 0-15 issue the stage's 16 boxes (two halves of 8 pages), one each.
    auto emit = [&](const Item& it, int c, int pbuf, int pass, Item* gi = nullptr,
                    bool* gh = nullptr, int* gs = nullptr) {
      const CUtensorMap* tm = pass == 0 ? &tm_k : &tm_v;
      const int j0 = c * p.chunk_tiles;
      const int j1 = min(it.n_tiles, j0 + p.chunk_tiles);
      for (int j = j0; j < j1 && ok; ++j) {
        if (gi != nullptr && j == j0 + STAGES) {
          // the ring is full of this chunk's tiles: take the next item now, while waiting
          *gh = grab(*gi);
          *gs = seq;
          gi = nullptr;
          if (!ok) break;
        }
        const int tok0 = it.t_begin + j * kTile;
        if (lane == 0) ok = mbar_wait<ROWS>(&bar_empty[st], ph ^ 1, &abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int npg = min(kTile / kPage, (it.t_end - tok0 + kPage - 1) / kPage);
        // lane q < 16 copies half q / 8 of page q % 8 of the tile: one box per lane, so the
        // stage's 16 copies issue in parallel (a thread's copies issue one after another)
        const int pg = lane & 7, hf = ROWS ? 0 : (lane >> 3) & 1;
        const int id = (lane < (ROWS ? 8 : 16) && pg < npg) ? s_pid[pbuf][j * (kTile / kPage) + pg]
                                                            : -1;
        const uint32_t have = __ballot_sync(0xffffffffu, lane < 8 && id >= 0);
        uint8_t* stage = sKV + st * kStageBytes;
        if constexpr (ROWS) {
          if (lane < 8) s_sinfo[st].id[lane] = id;
          if (lane == 0) {
            s_sinfo[st].pass = pass;
            s_sinfo[st].kvh = it.kvh;
            s_sinfo[st].end = 0;
          }
          __syncwarp();
        }
        if (lane == 0) {
          if (have)
            mbar_arrive_expect_tx(&bar_full[st], static_cast<uint32_t>(__popc(have)) * 4096u);
          else
            mbar_arrive(&bar_full[st]);
          if constexpr (ROWS) mbar_arrive(&bar_sready[st]);   // half 1 to the second issuer
        }
        __syncwarp();
        if (id >= 0)
          tma_load_4d_hint(stage + hf * kHalfBytes + pg * 2048, tm, &bar_full[st], hf * 64, it.kvh,
                           0, id, kv_policy);
        if (++st == STAGES) {
          st = 0;
          ph ^= 1;
        }
      }
      if (gi != nullptr && ok) {
        *gh = grab(*gi);
        *gs = seq;
      }
    };
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    // Ring order: K of chunk u+1, then V of chunk u.  One item of look-ahead (`pend`) is
    // grabbed and published early, so the MMA warp always knows what follows the current
    // chunk; the next look-ahead is grabbed once the ring is full of V tiles waiting for the
    // softmax, so the scheduler's latency stays off the stream (three page-id buffers: cur,
    // pend, new pend).
    Item cur, pend, pend2;
    bool have = grab(cur);
    int cur_seq = seq, pend_seq = seq;
    bool have_pend = false;
    if (have) {
      if (lane == 0) load_q(cur, cur_seq);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      emit(cur, 0, cur_seq % 3, 0);
      have_pend = grab(pend);
      pend_seq = seq;
    }
    int c = 0;
    while (have && ok) {
      const bool same = c + 1 < cur.n_chunks;
      const bool has_next = same || have_pend;
      bool have_pend2 = false;
      int pend2_seq = 0;
      // K of the next chunk, then V of this one, in the order the MMA issuer consumes them
      // (S(u + 1) before PV(u); with two sub-groups PV(u) before S(u + 1))
      auto emit_next_k = [&]() {
        if (same) {
          emit(cur, c + 1, cur_seq % 3, 0);
        } else if (have_pend) {
          if (lane == 0) load_q(pend, pend_seq);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          emit(pend, 0, pend_seq % 3, 0);
        }
      };
      if constexpr (!TWO) emit_next_k();
      if (!same && have_pend)
        emit(cur, c, cur_seq % 3, 1, &pend2, &have_pend2, &pend2_seq);
      else
        emit(cur, c, cur_seq % 3, 1);
      if constexpr (TWO) emit_next_k();
      if (!has_next) break;
      if (same) {
        ++c;
      } else {
        cur = pend;
        cur_seq = pend_seq;
        c = 0;
        pend = pend2;
        pend_seq = pend2_seq;
        have_pend = have_pend2;
      }
    }
    if constexpr (ROWS) {
      // tell the second issuer that no stage follows (once the next stage is free)
      if (lane == 0 && ok && mbar_wait<ROWS>(&bar_empty[st], ph ^ 1, &abort_flag)) {
        s_sinfo[st].end = 1;
        mbar_arrive(&bar_sready[st]);
      }
      __syncwarp();
    }
    if (lane == 0) {
      griddep_launch_dependents();  // this CTA takes no more work
      // the last CTA to finish taking work resets the counter for the next launch
      __threadfence();
      if (atomicAdd(p.work + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        p.work[0] = 0;
        p.work[1] = 0;
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s) mbar_wait_drain(&bar_full[s], ph ^ (s < st ? 0 : 1));
        for (int s = max(0, q_loads - kQBufs); s < q_loads; ++s)
          mbar_wait_drain(&bar_qfull[s % kQBufs], (s / kQBufs) & 1);
      }
    }
  } else if (ROWS && warp == kIssueWarp) {
    // ================================================= second K/V copy issuer (rows on M)
    // Follows the ring stage by stage: once the producer has armed a stage and described it,
    // lanes 0-7 copy half 1 (head dims 64-127) of its pages.
    const uint64_t kv_policy = l2_policy_evict_first();
    int st = 0;
    uint32_t ph = 0;
    while (mbar_wait_warp<ROWS>(&bar_sready[st], ph, &abort_flag)) {
      const StageInfo& si = s_sinfo[st];
      if (si.end) break;
      if (lane < kTile / kPage) {
        const int id = si.id[lane];
        if (id >= 0)
          tma_load_4d_hint(sKV + st * kStageBytes + kHalfBytes + lane * 2048,
                           si.pass == 0 ? &tm_k : &tm_v, &bar_full[st], 64, si.kvh, 0, id,
                           kv_policy);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_full[st]);   // this stage's descriptor is read
      if (++st == STAGES) {
        st = 0;
        ph ^= 1;
      }
    }
  } else if (warp == 1) {
    // =================================================================== MMA issuer
    if (lane == 0) {
      // S^T = K Q^T and O^T += V^T P^T (keys / head dims on M), or with ROWS S = Q K^T and
      // O += P V (query rows on M): the same shared-memory operands, A and B swapped
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, N, false, false);
      constexpr uint32_t kIdescO = ROWS ? idesc_bf16_f32(128, 128, false, true)
                                        : idesc_bf16_f32(128, N, true, false);
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t kv_addr = smem_u32(sKV);
      const uint32_t p_addr = smem_u32(sP);
      bool ok = true;
      int st = 0;
      uint32_t ph = 0;
      int pcount = 0, ocount = 0;
      // S of chunk `c` of `it` (global chunk number u): into S buffer u & 1, or with two
      // sub-groups into sub-group x's buffer x (one tile per chunk)
      auto do_s = [&](const Item& it, int c, int u, int seq) {
        if constexpr (!TWO)
          if (!(ok = ok && mbar_wait<ROWS>(&bar_sfree[u & 1], ((u >> 1) & 1) ^ 1,
                                           &abort_flag)))
            return;
        const int qb = seq % kQBufs;
        if (c == 0 && !(ok = mbar_wait<ROWS>(&bar_qfull[qb], (seq / kQBufs) & 1,
                                             &abort_flag)))
          return;
        tc_fence_after();
        if (kQTmem && c == 0) {
          // the item's Q into tensor memory, 16 head dims (8 columns) per copy, behind the last
          // S of the previous item; the staging buffer is free once the copies are done
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tmem_cp_128x256b(tmem + kQCol + static_cast<uint32_t>(kk * 8),
                             smem_desc(q_addr + (kk >> 2) * (kRowsItem * 128) + (kk & 3) * 32, 16,
                                       1024));
          umma_commit(&bar_qempty[qb]);
        }
        const int j0 = c * p.chunk_tiles;
        const int j1 = min(it.n_tiles, j0 + p.chunk_tiles);
        for (int j = j0; j < j1; ++j) {
          if (!(ok = mbar_wait<ROWS>(&bar_full[st], ph, &abort_flag))) return;
          tc_fence_after();
          const uint32_t ka = kv_addr + st * kStageBytes;
          for (int x = 0; x < kSub; ++x) {
            const int sb = kSub == 1 ? (u & 1) : x;
            // (two sub-groups: S(u) holds P(u) once the softmax is done with it, and PV(u) was
            // issued before this S(u + 1), so the in-order tensor pipe reads P first)
            const uint32_t tS = tmem + static_cast<uint32_t>(sb * p.chunk_tiles * N);
            const uint32_t qa = q_addr + qb * kRowsItem * 256 + x * N * 128;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t ad =
                  smem_desc(ka + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
              const uint64_t bd =
                  smem_desc(qa + (kk >> 2) * (kRowsItem * 128) + (kk & 3) * 32, 16, 1024);
              if constexpr (kQTmem)
                umma_bf16_ts(tS + (j - j0) * N, tmem + kQCol + static_cast<uint32_t>(kk * 8), ad,
                             kIdescS, kk > 0 ? 1u : 0u);
              else if constexpr (ROWS)
                umma_bf16(tS + (j - j0) * N, bd, ad, kIdescS, kk > 0 ? 1u : 0u);
              else
                umma_bf16(tS + (j - j0) * N, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
            }
            if constexpr (TWO) umma_commit(&bar_sfull[sb]);   // this sub-group's S is ready
          }
          umma_commit(&bar_empty[st]);
          if (++st == STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
        if constexpr (!TWO) umma_commit(&bar_sfull[u & 1]);
        if (!kQTmem && c == it.n_chunks - 1) umma_commit(&bar_qempty[qb]);  // Q no longer needed
      };
      // O^T += V^T P^T (O += P V) over the tiles of chunk `c`, for each sub-group
      auto do_pv = [&](const Item& it, int c, int u) {
        const int j0 = c * p.chunk_tiles;
        const int j1 = min(it.n_tiles, j0 + p.chunk_tiles);
        for (int j = j0; j < j1; ++j) {
          if (!(ok = mbar_wait<ROWS>(&bar_full[st], ph, &abort_flag))) return;
          const int tok0 = it.t_begin + j * kTile;
          const int valid = min(kTile, it.t_end - tok0);
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
          for (int x = 0; x < kSub; ++x) {
            const int pb = TWO ? x : pcount % kPBufs;
            const uint32_t pph = TWO ? (u & 1) : ((pcount / kPBufs) & 1);
            if (!(ok = mbar_wait<ROWS>(&bar_pfull[pb], pph, &abort_flag))) return;
            if constexpr (!ROWS) {
              if (c > 0 && j == j0 && s_pflag[pb]) {  // the softmax rescales O^T first
                if (!(ok = mbar_wait<ROWS>(&bar_oready, ocount & 1, &abort_flag))) return;
                ++ocount;
              }
            }
            tc_fence_after();
            const uint32_t pa = p_addr + pb * (N * 256);
            for (int q = 0; q < npg; ++q) {
              const uint64_t ad = smem_desc(va + q * 2048, kHalfBytes, 1024);
              const uint32_t acc = (c > 0 || j > j0 || q > 0) ? 1u : 0u;
              if constexpr (kPTmem) {
                // A = P over S buffer u & 1: keys 64h .. 64h+63 as columns 64h .. 64h+31
                const uint32_t pc =
                    static_cast<uint32_t>((u & 1) * N + (q >> 2) * 64 + (q & 3) * 8);
                umma_bf16_ts(tO, tmem + pc, ad, kIdescO, acc);
              } else if constexpr (TWO) {
                // A = P in sub-group x's S columns: keys 64h .. 64h+63 as columns 64h .. 64h+31
                const uint32_t pc = static_cast<uint32_t>(x * N + (q >> 2) * 64 + (q & 3) * 8);
                umma_bf16_ts(tO + x * N, tmem + pc, ad, kIdescO, acc);
              } else {
                const uint64_t bd =
                    smem_desc(pa + (q >> 2) * (N * 128) + (q & 3) * 32, 16, 1024);
                if constexpr (ROWS)
                  umma_bf16(tO + x * N, bd, ad, kIdescO, acc);
                else
                  umma_bf16(tO, ad, bd, kIdescO, acc);
              }
            }
            if constexpr (!ROWS) umma_commit(&bar_pempty[pb]);
            ++pcount;
          }
          umma_commit(&bar_empty[st]);
          if (++st == STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
        umma_commit(&bar_ofull[u & 1]);
      };
      // Two sub-groups: PV(u) and S(u + 1) interleaved by sub-group (PV_0, S_0, PV_1, S_1) with
      // V(u) and K(u + 1) both staged, so sub-group 0's softmax of u + 1 runs while sub-group
      // 1's PV(u) and S(u + 1) execute.  S_x(u + 1) overwrites the P_x(u) that PV_x(u) reads;
      // the tensor pipe executes one thread's MMAs in issue order.
      // S_x = Q_x K^T from the K stage at ka, into sub-group x's S columns
      auto issue_s = [&](uint32_t ka, int qb, int x) {
        const uint32_t tS = tmem + static_cast<uint32_t>(x * N);
        const uint32_t qa = q_addr + qb * kRowsItem * 256 + x * N * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = smem_desc(ka + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t bd =
              smem_desc(qa + (kk >> 2) * (kRowsItem * 128) + (kk & 3) * 32, 16, 1024);
          umma_bf16(tS, bd, ad, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bar_sfull[x]);
      };
      auto do_pv_s = [&](const Item& it, int c, int u, const Item& nx, int nc, int nseq,
                         bool has_next) {
        const int stv = st;
        if (!(ok = mbar_wait<ROWS>(&bar_full[stv], ph, &abort_flag))) return;
        if (++st == STAGES) {
          st = 0;
          ph ^= 1;
        }
        const int tok0 = it.t_begin + c * kTile;
        const int valid = min(kTile, it.t_end - tok0);
        const int npg = (valid + kPage - 1) / kPage;
        const int tail = valid - (npg - 1) * kPage;
        if (tail < kPage) {
          // slots past the sequence end may hold anything (NaN): 0 * NaN would poison O
          uint8_t* stage = sKV + stv * kStageBytes;
          for (int h = 0; h < 2; ++h) {
            uint4* z = reinterpret_cast<uint4*>(stage + h * kHalfBytes + (npg - 1) * 2048 +
                                                tail * 128);
            for (int o = 0; o < (kPage - tail) * 8; ++o) z[o] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        const int stk = st;
        const uint32_t phk = ph;
        const int qb = nseq % kQBufs;
        if (has_next && ++st == STAGES) {
          st = 0;
          ph ^= 1;
        }
        const uint32_t va = kv_addr + stv * kStageBytes;
        const uint32_t ka = kv_addr + stk * kStageBytes;
        // at an item boundary S(u + 1) waits for the next item's Q: both PVs first
        const bool inter = has_next && nc > 0;
        for (int x = 0; x < 2; ++x) {
          if (!(ok = mbar_wait<ROWS>(&bar_pfull[x], u & 1, &abort_flag))) return;
          tc_fence_after();
          for (int q = 0; q < npg; ++q) {
            // A = P in sub-group x's S columns: keys 64h .. 64h+63 as columns 64h .. 64h+31
            const uint64_t ad = smem_desc(va + q * 2048, kHalfBytes, 1024);
            const uint32_t pc = static_cast<uint32_t>(x * N + (q >> 2) * 64 + (q & 3) * 8);
            umma_bf16_ts(tO + x * N, tmem + pc, ad, kIdescO, (c > 0 || q > 0) ? 1u : 0u);
          }
          if (x == 1) {
            umma_commit(&bar_empty[stv]);
            umma_commit(&bar_ofull[u & 1]);
          }
          if (!inter) continue;
          if (x == 0) {   // K(u + 1) only now: PV_0(u) does not need it
            if (!(ok = mbar_wait<ROWS>(&bar_full[stk], phk, &abort_flag))) return;
            tc_fence_after();
          }
          issue_s(ka, qb, x);
        }
        if (has_next && !inter) {
          if (!(ok = mbar_wait<ROWS>(&bar_full[stk], phk, &abort_flag))) return;
          if (!(ok = mbar_wait<ROWS>(&bar_qfull[qb], (nseq / kQBufs) & 1, &abort_flag))) return;
          tc_fence_after();
          issue_s(ka, qb, 0);
          issue_s(ka, qb, 1);
        }
        if (has_next) {
          umma_commit(&bar_empty[stk]);
          if (nc == nx.n_chunks - 1) umma_commit(&bar_qempty[qb]);  // Q no longer needed
        }
      };
      int seq = 0;
      Item cur, nxt;
      ok = mbar_wait<ROWS>(&bar_ifull[0], 0, &abort_flag);
      cur = s_item[0];
      if (ok && !cur.end) {
        int c = 0, u = 0;
        do_s(cur, 0, 0, 0);
        while (ok) {
          bool has_next;
          int nc = 0, nseq = seq;
          if (c + 1 < cur.n_chunks) {
            has_next = true;
            nc = c + 1;
            nxt = cur;
          } else {
            nseq = seq + 1;
            const int rs = nseq % kItemRing;
            if (!(ok = mbar_wait<ROWS>(&bar_ifull[rs], (nseq / kItemRing) & 1, &abort_flag))) break;
            nxt = s_item[rs];
            has_next = !nxt.end;
          }
          // S(u + 1) ahead of PV(u), so the softmax can start the next tile while PV runs
          if constexpr (!TWO) {
            if (has_next) do_s(nxt, nc, u + 1, nseq);
            if (!ok) break;
          }
          if constexpr (TWO)
            do_pv_s(cur, c, u, nxt, nc, nseq, has_next);
          else
            do_pv(cur, c, u);
          if (!ok) break;
          if (c == cur.n_chunks - 1) mbar_arrive(&bar_iempty[seq % kItemRing]);
          if (!has_next) break;
          cur = nxt;
          c = nc;
          seq = nseq;
          ++u;
        }
      }
      umma_commit(&bar_done);
    }
  } else if constexpr (ROWS && TWO) {
    // ======================== softmax/epilogue, two sub-groups in parallel, a row per 2 threads
    // Warps 2-9 take sub-group 0, warps 10-17 sub-group 1: query row x * 128 + n of the item is
    // lane n of sub-group x's S and O; half 0 takes columns 0-63, half 1 columns 64-127.  A
    // half reads its 64 scores 32 at a time (a max pass, then an exponent pass) and writes its
    // P over the first 32 of its own S columns, the PV MMA's A operand.
    const int x = (warp - 2) >> 3;
    const int half = ((warp - 2) >> 2) & 1;
    const int q4 = warp & 3;
    const int n = (q4 << 5) | lane;
    const int pq = x * 4 + q4;   // the two halves' exchange barriers
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(half * 64);
    const uint32_t tSx = tmem + lane_off + static_cast<uint32_t>(x * N) + col0;
    const uint32_t tOx = tO + lane_off + static_cast<uint32_t>(x * N) + col0;
    const float cs = p.scale_log2;
    bool ok = true;
    int u = 0, pe = 0, pair_ends = 0;
    for (int seq = 0; ok; ++seq) {
      const int rs = seq % kItemRing;
      if (!(ok = mbar_wait_warp<ROWS>(&bar_ifull[rs], (seq / kItemRing) & 1, &abort_flag))) break;
      const Item it = s_item[rs];
      mbar_arrive(&bar_iempty[rs]);   // the descriptor is in registers: its slot may be reused
      if (it.end) break;
      const int r_item = x * N + n;                  // row of the item
      const int i_row = it.rg * p.lsub + r_item / p.G;
      int lim = 0x7FFFFFFF;                           // keys past q0 the row may see
      if constexpr (MASKED) lim = (i_row / p.mask_block + 1) * p.mask_block;
      float m_run = -CUDART_INF_F, l_run = 0.f;       // l_run: this half's sum
      for (int c = 0; c < it.n_chunks && ok; ++c, ++u) {
        if (!(ok = mbar_wait_warp<ROWS>(&bar_sfull[x], u & 1, &abort_flag))) break;
        tc_fence_after();
        const int key0 = it.t_begin + c * kTile;
        int nvalid = min(kTile, it.t_end - key0);
        if constexpr (MASKED) nvalid = min(nvalid, lim - (key0 - it.q0));
        nvalid -= half * 64;   // of this half's columns
        const bool full = nvalid >= 64;   // every score of this half-row is a key the row sees
        // pass 1: the half-row max, 32 scores at a time; then the row max
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
          uint32_t r[32];
          tmem_ld16(tSx + g2 * 32, *reinterpret_cast<uint32_t(*)[16]>(r));
          tmem_ld16(tSx + g2 * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
          tmem_wait_ld();
          tmem_regs_ready(*reinterpret_cast<uint32_t(*)[16]>(r));
          tmem_regs_ready(*reinterpret_cast<uint32_t(*)[16]>(r + 16));
          mx = fmaxf(mx, full ? max32<true>(r, 0, 0) : max32<false>(r, g2 * 32, nvalid));
        }
        s_hmax[pe & 1][x][half][n] = mx;
        mbar_arrive(&bar_pair[pq][pe & 1]);
        if (!(ok = mbar_wait_warp<ROWS>(&bar_pair[pq][pe & 1], (pe >> 1) & 1, &abort_flag))) break;
        mx = fmaxf(s_hmax[pe & 1][x][0][n], s_hmax[pe & 1][x][1][n]);
        ++pe;
        // the running max moves only when the tile raises it by more than 2^kLazyRescale
        float alpha = 1.f;
        bool resc = false;
        if (m_run == -CUDART_INF_F) {
          m_run = mx;
        } else if ((mx - m_run) * cs > kLazyRescale) {
          alpha = ex2((m_run - mx) * cs);
          m_run = mx;
          resc = true;
        }
        const float mc = m_run == -CUDART_INF_F ? 0.f : m_run * cs;
        const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(-mc, -mc);
        // pass 2: p = 2^(s cs - m cs), 32 at a time; P (bf16 pairs) over columns already read
        float sum = 0.f;
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
          uint32_t r[32];
          tmem_ld16(tSx + g2 * 32, *reinterpret_cast<uint32_t(*)[16]>(r));
          tmem_ld16(tSx + g2 * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
          tmem_wait_ld();
          tmem_regs_ready(*reinterpret_cast<uint32_t(*)[16]>(r));
          tmem_regs_ready(*reinterpret_cast<uint32_t(*)[16]>(r + 16));
          uint32_t pk[16];
          sum += full ? exp_pack32<true>(r, 0, 0, cs2, nm2, pk)
                      : exp_pack32<false>(r, g2 * 32, nvalid, cs2, nm2, pk);
          tmem_st16(tSx + g2 * 16, pk);   // keys 64h + 32 g2 .. + 31 as 16 columns
        }
        l_run = l_run * alpha + sum;
        if (__any_sync(0xffffffffu, resc)) {
          // bring this warp's half of its rows of O to the new maxima once the previous
          // tile's PV is done
          if (!(ok = mbar_wait_warp<ROWS>(&bar_ofull[(u - 1) & 1], ((u - 1) >> 1) & 1,
                                          &abort_flag)))
            break;
          tc_fence_after();
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t o[16];
            tmem_ld16(tOx + g * 16, o);
            tmem_wait_ld();
            tmem_regs_ready(o);
#pragma unroll
            for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st16(tOx + g * 16, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_pfull[x]);
        if (c != it.n_chunks - 1) continue;
        // ---- epilogue of the item: this half of the row of O, divided by the row's sum or as
        // a split partial
        if (!(ok = mbar_wait_warp<ROWS>(&bar_ofull[u & 1], (u >> 1) & 1, &abort_flag))) break;
        tc_fence_after();
        s_hsum[pair_ends & 1][x][half][n] = l_run;
        mbar_arrive(&bar_pair_end[pq]);
        if (!(ok = mbar_wait_warp<ROWS>(&bar_pair_end[pq], pair_ends & 1, &abort_flag))) break;
        const float l_row = s_hsum[pair_ends & 1][x][0][n] + s_hsum[pair_ends & 1][x][1][n];
        ++pair_ends;
        const bool live = r_item < p.rows_per_group && i_row < p.L;
        const size_t grp = (static_cast<size_t>(it.b) * p.Hkv + it.kvh) * p.row_groups + it.rg;
        float* mine =
            p.part + (grp * p.max_splits + it.split) * static_cast<size_t>(kRowsItem) * 130;
        uint16_t* dst = live ? p.out + ((static_cast<size_t>(it.b) * p.L + i_row) * p.Hq +
                                        static_cast<size_t>(it.kvh) * p.G + r_item % p.G) * 128 + col0
                             : p.out;
        const float inv = 1.f / l_row;
        uint8_t* stage = s_stage[warp - 2];
        if (it.n_splits == 1) {
          // this half of the row as bf16: 128 bytes per lane
          uint32_t w[32];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t o[16];
            tmem_ld16(tOx + g * 16, o);
            tmem_wait_ld();
            tmem_regs_ready(o);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[2 * k]) * inv,
                                                              __uint_as_float(o[2 * k + 1]) * inv);
              w[8 * g + k] = *reinterpret_cast<const uint32_t*>(&h2);
            }
          }
          store_rows_128b(w, live ? dst : nullptr, stage, lane);
        } else {
          // fp32 partial: 32 columns (128 bytes) per lane at a time
#pragma unroll
          for (int g2 = 0; g2 < 2; ++g2) {
            uint32_t o[32];
            tmem_ld16(tOx + g2 * 32, *reinterpret_cast<uint32_t(*)[16]>(o));
            tmem_ld16(tOx + g2 * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(o + 16));
            tmem_wait_ld();
            tmem_regs_ready(*reinterpret_cast<uint32_t(*)[16]>(o));
            tmem_regs_ready(*reinterpret_cast<uint32_t(*)[16]>(o + 16));
            store_rows_128b(o, live ? mine + r_item * 128 + col0 + g2 * 32 : nullptr, stage,
                            lane);
          }
        }
        if (live && it.n_splits > 1 && half == 0) {
          mine[kRowsItem * 128 + r_item] = m_run;
          mine[kRowsItem * 128 + kRowsItem + r_item] = l_row;
        }
        tc_fence_before();   // O is read: the next item's first PV (after its P) may overwrite it
      }
    }
  } else if constexpr (ROWS) {
    // ====================================================== softmax/epilogue, a row per 2 threads
    // Query row x * 128 + n of the item (sub-group x) is tensor-memory lane n of sub-group x's
    // S and O.  Two warps share each lane quadrant, so each row has two threads: half 0 takes
    // columns 0-63, half 1 columns 64-127 (of S, then of O).  They exchange the half-row maxima
    // every tile and the half sums at the end.  One tile per chunk; with two sub-groups the
    // threads take sub-group 0, then 1, of every tile.
    const int q4 = warp & 3;
    const int half = (warp - 2) >> 2;
    const int n = (q4 << 5) | lane;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(half * 64);
    const float cs = p.scale_log2;
    bool ok = true;
    int pcount = 0, u = 0, pe = 0, pair_ends = 0;   // pe, pair_ends: exchanges so far
    for (int seq = 0; ok; ++seq) {
      const int rs = seq % kItemRing;
      if (!(ok = mbar_wait_warp<ROWS>(&bar_ifull[rs], (seq / kItemRing) & 1, &abort_flag))) break;
      const Item it = s_item[rs];
      mbar_arrive(&bar_iempty[rs]);   // the descriptor is in registers: its slot may be reused
      if (it.end) break;
      int i_row[kSub], lim[kSub];   // block position of the row; keys past q0 it may see
      float m_run[kSub], l_run[kSub];   // l_run: this half's sum
#pragma unroll
      for (int x = 0; x < kSub; ++x) {
        i_row[x] = it.rg * p.lsub + (x * N + n) / p.G;
        lim[x] = 0x7FFFFFFF;
        if constexpr (MASKED) lim[x] = (i_row[x] / p.mask_block + 1) * p.mask_block;
        m_run[x] = -CUDART_INF_F;
        l_run[x] = 0.f;
      }
      for (int c = 0; c < it.n_chunks && ok; ++c, ++u) {
        const int key0 = it.t_begin + c * kTile;
#pragma unroll
        for (int x = 0; x < kSub; ++x) {
          const int sb = kSub == 1 ? (u & 1) : x;
          const uint32_t sph = kSub == 1 ? ((u >> 1) & 1) : (u & 1);
          const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(sb * N) + col0;
          if (!(ok = mbar_wait_warp<ROWS>(&bar_sfull[sb], sph, &abort_flag))) break;
          tc_fence_after();
          uint32_t r[64];
#pragma unroll
          for (int g = 0; g < 4; ++g)
            tmem_ld16(tS + g * 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16 * g));
          tmem_wait_ld();
#pragma unroll
          for (int g = 0; g < 4; ++g)
            tmem_regs_ready(*reinterpret_cast<uint32_t(*)[16]>(r + 16 * g));
          tc_fence_before();
          mbar_arrive(&bar_sfree[sb]);   // S is in registers: the buffer may take the next S
          // keys of the tile the row sees: a prefix of it (sequence end, block-causal limit);
          // the others read as -inf
          int nvalid = min(kTile, it.t_end - key0);
          if constexpr (MASKED) nvalid = min(nvalid, lim[x] - (key0 - it.q0));
          nvalid -= half * 64;   // of this half's columns
          if (nvalid < 64) {
#pragma unroll
            for (int k = 0; k < 64; ++k)
              if (k >= nvalid) r[k] = 0xFF800000u;
          }
          // half-row max (trees of three-input maxima over the masked scores), then the row max
          const float hmax =
              fmaxf(max32<true>(*reinterpret_cast<const uint32_t(*)[32]>(r), 0, 0),
                    max32<true>(*reinterpret_cast<const uint32_t(*)[32]>(r + 32), 0, 0));
          s_hmax[pe & 1][0][half][n] = hmax;
          mbar_arrive(&bar_pair[q4][pe & 1]);
          if (!(ok = mbar_wait_warp<ROWS>(&bar_pair[q4][pe & 1], (pe >> 1) & 1,
                                          &abort_flag)))
            break;
          const float mx = fmaxf(s_hmax[pe & 1][0][0][n], s_hmax[pe & 1][0][1][n]);
          ++pe;
          // the running max moves only when the tile raises it by more than 2^kLazyRescale
          // (both halves of a row take the same decision)
          float alpha = 1.f;
          bool resc = false;
          if (m_run[x] == -CUDART_INF_F) {
            m_run[x] = mx;
          } else if ((mx - m_run[x]) * cs > kLazyRescale) {
            alpha = ex2((m_run[x] - mx) * cs);
            m_run[x] = mx;
            resc = true;
          }
          // p = 2^(s cs - m cs): scaling two scores per packed FMA, the exponentials
          // independent, the sum a tree of packed adds (a row that has seen no key yet has
          // m = -inf: p = 0)
          const float mc = m_run[x] == -CUDART_INF_F ? 0.f : m_run[x] * cs;
          const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(-mc, -mc);
          float2 e[32];
          uint32_t pk[32];   // this half of the row's P as bf16 pairs
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float2 y = __ffma2_rn(
                make_float2(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1])), cs2, nm2);
            e[k] = make_float2(ex2(y.x), ex2(y.y));
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(e[k].x, e[k].y);
            pk[k] = *reinterpret_cast<const uint32_t*>(&h2);
          }
#pragma unroll
          for (int w = 16; w > 0; w >>= 1)
#pragma unroll
            for (int k = 0; k < w; ++k) e[k] = __fadd2_rn(e[k], e[k + w]);
          l_run[x] = l_run[x] * alpha + (e[0].x + e[0].y);
          if (__any_sync(0xffffffffu, resc)) {
            // bring this warp's half of its rows of O to the new maxima once the previous
            // tile's PV is done
            if (!(ok = mbar_wait_warp<ROWS>(&bar_ofull[(u - 1) & 1], ((u - 1) >> 1) & 1,
                                            &abort_flag)))
              break;
            tc_fence_after();
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint32_t o[16];
              tmem_ld16(tO + lane_off + x * N + col0 + g * 16, o);
              tmem_wait_ld();
              tmem_regs_ready(o);
#pragma unroll
              for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st16(tO + lane_off + x * N + col0 + g * 16, o);
            }
            tmem_wait_st();
          }
          const int pb = pcount % kPBufs;   // = u & 1, the S buffer
          // this half of P row n over the first 32 of this half's S columns (already in
          // registers): keys 64h + 2k, 64h + 2k + 1 in column 64h + k, the PV MMA's A operand
          tmem_st16(tS, *reinterpret_cast<const uint32_t(*)[16]>(pk));
          tmem_st16(tS + 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16));
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bar_pfull[pb]);
          ++pcount;
        }
        if (!ok || c != it.n_chunks - 1) continue;
        // ---- epilogue of the item: this half of each row of O, divided by the row's sum or
        // as a split partial
        if (!(ok = mbar_wait_warp<ROWS>(&bar_ofull[u & 1], (u >> 1) & 1, &abort_flag))) break;
        tc_fence_after();
        const size_t grp = (static_cast<size_t>(it.b) * p.Hkv + it.kvh) * p.row_groups + it.rg;
        float* mine =
            p.part + (grp * p.max_splits + it.split) * static_cast<size_t>(kRowsItem) * 130;
#pragma unroll
        for (int x = 0; x < kSub; ++x) {
          s_hsum[pair_ends & 1][0][half][n] = l_run[x];
          mbar_arrive(&bar_pair_end[q4]);
          if (!(ok = mbar_wait_warp<ROWS>(&bar_pair_end[q4], pair_ends & 1, &abort_flag))) break;
          const float l_row = s_hsum[pair_ends & 1][0][0][n] + s_hsum[pair_ends & 1][0][1][n];
          ++pair_ends;
          const int r_item = x * N + n;   // row of the item
          const bool live = r_item < p.rows_per_group && i_row[x] < p.L;
          uint16_t* dst =
              live ? p.out + ((static_cast<size_t>(it.b) * p.L + i_row[x]) * p.Hq +
                              static_cast<size_t>(it.kvh) * p.G + r_item % p.G) * 128 + col0
                   : p.out;
          const float inv = 1.f / l_row;
          uint8_t* stage = s_stage[warp - 2];
          const uint32_t tOr = tO + lane_off + x * N + col0;
          if (it.n_splits == 1) {
            // this half of the row as bf16: 128 bytes per lane
            uint32_t w[32];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint32_t o[16];
              tmem_ld16(tOr + g * 16, o);
              tmem_wait_ld();
              tmem_regs_ready(o);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(
                    __uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
                w[8 * g + k] = *reinterpret_cast<const uint32_t*>(&h2);
              }
            }
            store_rows_128b(w, live ? dst : nullptr, stage, lane);
          } else {
            // fp32 partial: 32 columns (128 bytes) per lane at a time
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
              uint32_t o[32];
              tmem_ld16(tOr + g2 * 32, *reinterpret_cast<uint32_t(*)[16]>(o));
              tmem_ld16(tOr + g2 * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(o + 16));
              tmem_wait_ld();
              tmem_regs_ready(*reinterpret_cast<uint32_t(*)[16]>(o));
              tmem_regs_ready(*reinterpret_cast<uint32_t(*)[16]>(o + 16));
              store_rows_128b(o, live ? mine + r_item * 128 + col0 + g2 * 32 : nullptr, stage,
                              lane);
            }
          }
          if (live && it.n_splits > 1 && half == 0) {
            mine[kRowsItem * 128 + r_item] = m_run[x];
            mine[kRowsItem * 128 + kRowsItem + r_item] = l_row;
          }
        }
        tc_fence_before();   // O is read: the next item's first PV (after its P) may overwrite it
      }
    }
  } else {
    // =================================================================== softmax/epilogue
    const int q4 = warp & 3;
    const int x = (q4 << 5) | lane;  // tensor-memory lane: KV token of a tile, or head dim
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const float cs = p.scale_log2;
    const int rows = p.rows_per_group;
    float l[N];
    bool ok = true;
    int pcount = 0, u = 0;
    for (int seq = 0; ok; ++seq) {
      const int rs = seq % kItemRing;
      if (!(ok = mbar_wait_warp<ROWS>(&bar_ifull[rs], (seq / kItemRing) & 1, &abort_flag))) break;
      const Item it = s_item[rs];
      if (it.end) break;
#pragma unroll
      for (int n = 0; n < N; ++n) l[n] = 0.f;
      if (x < N) s_m[x] = -CUDART_INF_F;
      for (int c = 0; c < it.n_chunks && ok; ++c, ++u) {
        const int j0 = c * p.chunk_tiles;
        const int j1 = min(it.n_tiles, j0 + p.chunk_tiles);
        const uint32_t tS = tmem + lane_off + static_cast<uint32_t>((u & 1) * p.chunk_tiles * N);
        if (!(ok = mbar_wait_warp<ROWS>(&bar_sfull[u & 1], (u >> 1) & 1, &abort_flag))) break;
        tc_fence_after();
        // phase A: exact column maxima over the chunk
#pragma unroll
        for (int cg = 0; cg < N / 16; ++cg) {
          float mx[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) mx[k] = -CUDART_INF_F;
          for (int j = j0; j < j1; ++j) {
            uint32_t r[16];
            tmem_ld16(tS + (j - j0) * N + cg * 16, r);
            tmem_wait_ld();
            tmem_regs_ready(r);
            const bool valid = it.t_begin + j * kTile + x < it.t_end;
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
        if (x == 0) s_need[(u + 1) & 1] = 0;  // every reader of that slot is past this barrier
        if (x < N) {
          // The running max only moves when the chunk raises it by more than kLazyRescale
          // (log2 units): below that the exponentials use the older max, P stays below
          // 2^kLazyRescale, and O^T and l need no rescale at this chunk boundary.
          const float mc = fmaxf(fmaxf(s_red[0][x], s_red[1][x]), fmaxf(s_red[2][x], s_red[3][x]));
          const float mo = s_m[x];
          float mn = mo, alpha = 1.f;
          if (mo == -CUDART_INF_F) {
            mn = mc;
            alpha = 0.f;
          } else if ((mc - mo) * cs > kLazyRescale) {
            mn = mc;
            alpha = exp2f((mo - mn) * cs);
            s_need[u & 1] = 1;
          }
          s_alpha[x] = alpha;
          s_m[x] = mn;
          s_mc[x] = mn * cs;
        }
        named_barrier(1, kSoftmaxThreads);
        const bool need = s_need[u & 1] != 0;
        if (c > 0 && need) {
          // rescale the running O^T columns (and l) to the new maxima
          if (!(ok = mbar_wait_warp<ROWS>(&bar_ofull[(u - 1) & 1], ((u - 1) >> 1) & 1,
                                          &abort_flag)))
            break;
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
        {
          // narrow N: maxima in registers, the next tile's S^T read from tensor memory
          // while this one is exponentiated
          float mcr[N];
  #pragma unroll
          for (int n = 0; n < N; ++n) mcr[n] = s_mc[n];
          uint32_t r[N];
  #pragma unroll
          for (int cg = 0; cg < N / 16; ++cg) {
            uint32_t (&rg)[16] = *reinterpret_cast<uint32_t(*)[16]>(r + cg * 16);
            tmem_ld16(tS + cg * 16, rg);
          }
          for (int j = j0; j < j1 && ok; ++j) {
            tmem_wait_ld();
  #pragma unroll
            for (int cg = 0; cg < N / 16; ++cg)
              tmem_regs_ready(*reinterpret_cast<uint32_t(*)[16]>(r + cg * 16));
            float pv[N];
            const bool valid = it.t_begin + j * kTile + x < it.t_end;
  #pragma unroll
            for (int n = 0; n < N; ++n)
              pv[n] = valid ? exp2f(fmaf(__uint_as_float(r[n]), cs, -mcr[n])) : 0.f;
            if (j + 1 < j1) {
  #pragma unroll
              for (int cg = 0; cg < N / 16; ++cg) {
                uint32_t (&rg)[16] = *reinterpret_cast<uint32_t(*)[16]>(r + cg * 16);
                tmem_ld16(tS + (j + 1 - j0) * N + cg * 16, rg);
              }
            }
            const int pb = pcount & 1;
            if (!(ok = mbar_wait_warp<ROWS>(&bar_pempty[pb], ((pcount >> 1) & 1) ^ 1,
                                            &abort_flag)))
              break;
            uint8_t* pbuf = sP + pb * (N * 256) + (x >> 6) * (N * 128);
            const uint32_t xc = (x & 63) >> 3;
            const uint32_t xb = (x & 7) * 2;
  #pragma unroll
            for (int n = 0; n < N; ++n) {
              l[n] += pv[n];
              const uint32_t off = n * 128 + ((xc ^ (n & 7)) << 4) + xb;
              *reinterpret_cast<__nv_bfloat16*>(pbuf + off) = __float2bfloat16_rn(pv[n]);
            }
            if (x == 0) s_pflag[pb] = (j == j0) && need;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar_pfull[pb]);
            ++pcount;
          }
          if (!ok) tmem_wait_ld();
        }
        if (!ok) break;
        tc_fence_before();
        mbar_arrive(&bar_sfree[u & 1]);
        if (c != it.n_chunks - 1) continue;
        // ---- epilogue of the item
        if (!(ok = mbar_wait_warp<ROWS>(&bar_ofull[u & 1], (u >> 1) & 1, &abort_flag))) break;
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
        const size_t head_base = static_cast<size_t>(it.kvh) * p.G;
        if (it.n_splits == 1) {
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
              const int i = it.rg * p.lsub + n / p.G;
              if (i >= p.L) continue;
              const size_t o =
                  ((static_cast<size_t>(it.b) * p.L + i) * p.Hq + head_base + n % p.G) * 128 + x;
              p.out[o] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[k]) / s_l[n]));
            }
          }
        } else {
          // one split of a longer sequence: write (O, m, l); attn_merge_kernel combines them
          const size_t unit = static_cast<size_t>(N) * 130;
          const size_t grp = (static_cast<size_t>(it.b) * p.Hkv + it.kvh) * p.row_groups + it.rg;
          float* mine = p.part + (grp * p.max_splits + it.split) * unit;
          const uint64_t keep = l2_policy_evict_last();  // read back by the merge soon
#pragma unroll
          for (int cg = 0; cg < N / 16; ++cg) {
            uint32_t r[16];
            tmem_ld16(tO + lane_off + cg * 16, r);
            tmem_wait_ld();
            tmem_regs_ready(r);
#pragma unroll
            for (int k = 0; k < 16; ++k)
              st_global_hint(mine + (cg * 16 + k) * 128 + x, __uint_as_float(r[k]), keep);
          }
          if (x < N) {
            st_global_hint(mine + N * 128 + x, s_m[x], keep);
            st_global_hint(mine + N * 128 + N + x, s_l[x], keep);
          }
        }
        // O^T and the item descriptor are free for the next item
        tc_fence_before();
        named_barrier(1, kSoftmaxThreads);
        if (x == 0) mbar_arrive(&bar_iempty[rs]);
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


// Sequences by decreasing item length, so that the persistent attention CTAs take the longest
// items first and the last items handed out are the shortest: the CTAs then finish close
// together.  Whole-sequence mode ranks by KV length (a sequence fits the page-id staging buffer
// there, so at most kMaxItemPages * kPage tokens); with even KV splits, by the length of the
// sequence's splits in tiles (at most kMaxSplitTokensRows / kTile), and the items then go out
// sequence by sequence in that order, all splits of one before the next.  A counting sort in
// one CTA (B <= blockDim.x = kMaxOrderSeqs): every sequence counts its key, a scan of the
// counts from the largest key down gives each key's first slot, and each sequence takes a slot
// in its key's range (equal keys in no particular order).
constexpr int kOrderBuckets = kMaxItemPages * kPage + 1;   // keys 0 .. 2048
constexpr int kOrderPerThread = (kOrderBuckets + kMaxOrderSeqs - 1) / kMaxOrderSeqs;
static_assert(kMaxSplitTokensRows / kTile < kOrderBuckets, "split lengths in tiles fit the keys");

__global__ void __launch_bounds__(kMaxOrderSeqs)
attn_order_kernel(const AttnParams p, bool whole, int* __restrict__ order) {
  __shared__ int s_cnt[kOrderBuckets];
  __shared__ int s_warp[kMaxOrderSeqs / 32];
  griddep_wait();
  griddep_launch_dependents();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int i = t; i < kOrderBuckets; i += kMaxOrderSeqs) s_cnt[i] = 0;
  __syncthreads();
  int len = 0, pos = 0;
  if (t < p.B) {
    const int prefix = p.prefix_lens[t];
    const long long max_tok = static_cast<long long>(p.max_pages) * kPage;
    long long l = static_cast<long long>(prefix < 0 ? 0 : prefix) + p.L;
    if (l > max_tok) l = max_tok;
    if (!whole) l = split_len(static_cast<int>(l), p) / kTile;
    if (l > kOrderBuckets - 1) l = kOrderBuckets - 1;   // not reached (see above)
    len = static_cast<int>(l);
    pos = atomicAdd(&s_cnt[len], 1);
  }
  __syncthreads();
  // thread t owns the kOrderPerThread lengths just below kOrderBuckets - 1 - t * kOrderPerThread
  int cnt[kOrderPerThread], sum = 0;
#pragma unroll
  for (int k = 0; k < kOrderPerThread; ++k) {
    const int bucket = kOrderBuckets - 1 - (t * kOrderPerThread + k);
    cnt[k] = bucket >= 0 ? s_cnt[bucket] : 0;
    sum += cnt[k];
  }
  int incl = sum;   // inclusive scan over the threads (longest lengths first)
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += s_warp[w];
  int start = before + incl - sum;   // sequences longer than this thread's lengths
#pragma unroll
  for (int k = 0; k < kOrderPerThread; ++k) {
    const int bucket = kOrderBuckets - 1 - (t * kOrderPerThread + k);
    if (bucket >= 0) s_cnt[bucket] = start;
    start += cnt[k];
  }
  __syncthreads();
  if (t < p.B) order[s_cnt[len] + pos] = t;
}

// Merges the splits of every (sequence, KV head, row group) whose KV range was cut into more
// than one item: out = sum_s w_s O_s with w_s = exp(m_s - M) / sum_s exp(m_s - M) l_s.
// One warp per (group, query row): lane s fetches split s's (m, l), the weights come from
// warp shuffles, and each lane then sums a float4 of head dims over the splits with
// independent loads (two round trips to memory in all).
// Grid: x = group (sequence, KV head, row group), y = blocks of 8 warps x kMergeRows query
// rows; 32-bit index math only (the kernel is issue-bound when every warp decomposes a 64-bit
// index).  A warp merges kMergeRows rows of one group at once, so the loads of both rows are in
// flight together and the grid fits the GPU in one wave.
constexpr int kMergeRows = 2;

__global__ void __launch_bounds__(256)
attn_merge_kernel(const AttnParams p, int N) {
  const int lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();
  const int n0 = (static_cast<int>(blockIdx.y) * 8 + (threadIdx.x >> 5)) * kMergeRows;
  if (n0 >= p.rows_per_group) return;
  const unsigned grp = blockIdx.x;
  const int rg = static_cast<int>(grp % static_cast<unsigned>(p.row_groups));
  const unsigned bk = grp / static_cast<unsigned>(p.row_groups);
  const int kvh = static_cast<int>(bk % static_cast<unsigned>(p.Hkv));
  const int b = static_cast<int>(bk / static_cast<unsigned>(p.Hkv));
  bool valid[kMergeRows];
#pragma unroll
  for (int r = 0; r < kMergeRows; ++r) {
    const int n = n0 + r;
    valid[r] = n < p.rows_per_group && rg * p.lsub + n / p.G < p.L;
  }
  if (!valid[0]) return;   // rows of a group are in block order: no later row is valid either
  const size_t unit = static_cast<size_t>(N) * 130;
  const float* all = p.part + static_cast<size_t>(grp) * p.max_splits * unit;
  // lane s fetches split s's (m, l) of each row together with the prefix length (slots of
  // splits that turn out not to exist are ignored), so the split count costs no extra round trip
  float ml[kMergeRows], ll[kMergeRows];
#pragma unroll
  for (int r = 0; r < kMergeRows; ++r) {
    ml[r] = -CUDART_INF_F;
    ll[r] = 0.f;
    if (valid[r] && lane < p.max_splits) {
      ml[r] = __ldcg(all + lane * unit + N * 128 + n0 + r);
      ll[r] = __ldcg(all + lane * unit + N * 128 + N + n0 + r);
    }
  }
  const int prefix = p.prefix_lens[b];
  const long long max_tok = static_cast<long long>(p.max_pages) * kPage;
  long long kvl = static_cast<long long>(prefix < 0 ? 0 : prefix) + p.L;
  if (kvl > max_tok) kvl = max_tok;
  const int per = split_len(static_cast<int>(kvl), p);
  const int ns = static_cast<int>((kvl + per - 1) / per);
  if (ns <= 1) return;
  float4 acc[kMergeRows];
#pragma unroll
  for (int r = 0; r < kMergeRows; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (ns <= 32) {
    // the rows' maxima and normalisers over all splits: lane s holds split s's (m, l)
    float wl[kMergeRows];
#pragma unroll
    for (int r = 0; r < kMergeRows; ++r) {
      if (lane >= ns) {
        ml[r] = -CUDART_INF_F;
        ll[r] = 0.f;
      }
      float M = ml[r];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      const float e = lane < ns ? exp2f((ml[r] - M) * p.scale_log2) : 0.f;
      float den = e * ll[r];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
      wl[r] = valid[r] ? e / den : 0.f;
    }
#pragma unroll 4
    for (int j = 0; j < ns; ++j) {
#pragma unroll
      for (int r = 0; r < kMergeRows; ++r) {
        const float wj = __shfl_sync(0xffffffffu, wl[r], j);
        if (!valid[r]) continue;
        const float4 o =
            __ldcg(reinterpret_cast<const float4*>(all + j * unit + (n0 + r) * 128) + lane);
        acc[r].x += wj * o.x;
        acc[r].y += wj * o.y;
        acc[r].z += wj * o.z;
        acc[r].w += wj * o.w;
      }
    }
  } else {
    // beyond 32 splits the lanes walk the list in steps of 32, one row at a time
#pragma unroll
    for (int r = 0; r < kMergeRows; ++r) {
      if (!valid[r]) continue;
      const int n = n0 + r;
      float M = -CUDART_INF_F;
      for (int s0 = 0; s0 < ns; s0 += 32)
        if (s0 + lane < ns) M = fmaxf(M, __ldcg(all + (s0 + lane) * unit + N * 128 + n));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      float den = 0.f;
      for (int s0 = 0; s0 < ns; s0 += 32)
        if (s0 + lane < ns) {
          const float* pm = all + (s0 + lane) * unit + N * 128;
          den += exp2f((__ldcg(pm + n) - M) * p.scale_log2) * __ldcg(pm + N + n);
        }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
      const float inv = 1.0f / den;
      for (int s0 = 0; s0 < ns; s0 += 32) {
        const int cnt = min(32, ns - s0);
        float wl = 0.f;
        if (lane < cnt)
          wl = exp2f((__ldcg(all + (s0 + lane) * unit + N * 128 + n) - M) * p.scale_log2) * inv;
        for (int j = 0; j < cnt; ++j) {
          const float wj = __shfl_sync(0xffffffffu, wl, j);
          const float4 o =
              __ldcg(reinterpret_cast<const float4*>(all + (s0 + j) * unit + n * 128) + lane);
          acc[r].x += wj * o.x;
          acc[r].y += wj * o.y;
          acc[r].z += wj * o.z;
          acc[r].w += wj * o.w;
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kMergeRows; ++r) {
    if (!valid[r]) continue;
    const int n = n0 + r;
    const int i = rg * p.lsub + n / p.G;
    const size_t o = ((static_cast<size_t>(b) * p.L + i) * p.Hq + static_cast<size_t>(kvh) * p.G +
                      n % p.G) * 128 + 4 * lane;
    const uint32_t lo =
        __bfloat16_as_ushort(__float2bfloat16_rn(acc[r].x)) |
        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[r].y))) << 16);
    const uint32_t hi =
        __bfloat16_as_ushort(__float2bfloat16_rn(acc[r].z)) |
        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[r].w))) << 16);
    *reinterpret_cast<uint2*>(p.out + o) = make_uint2(lo, hi);
  }
}

template <int N, int STAGES, bool ROWS, bool TWO>
constexpr size_t smem_bytes() {
  // the Q buffer (as the kernel: one of the item's rows), K/V stages, P buffers in shared memory
  // (none with rows on M: P is in tensor memory)
  const size_t q = static_cast<size_t>(TWO ? 2 : 1) * N * 256;
  const size_t pbufs = ROWS ? 0 : 2;
  return 1024 + q + static_cast<size_t>(STAGES) * kStageBytes + pbufs * N * 256;
}

template <int N, int STAGES, int CPS, bool MASKED, bool ROWS, bool TWO>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const AttnParams& prm, int num_sms, cudaStream_t stream) {
  constexpr size_t smem = smem_bytes<N, STAGES, ROWS, TWO>();
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [] {
    cudaError_t r = cudaFuncSetAttribute(attn_kernel<N, STAGES, CPS, MASKED, ROWS, TWO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(attn_kernel<N, STAGES, CPS, MASKED, ROWS, TWO>,
                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_kernel<N, STAGES, CPS, MASKED, ROWS, TWO>, dim3(num_sms * CPS),
                    dim3(attn_threads(ROWS, TWO)), smem,
                    stream, tq, tk, tv, prm);
}

}  // namespace

namespace {
// Prompt chunk j (L queries) of sequence b becomes sequence b * nb + j of the attention: its
// prefix is the cached prefix plus the j chunks before it.
__global__ void prompt_prefix_kernel(const int32_t* __restrict__ prefix_lens, int B, int nb, int L,
                                     int32_t* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * nb) return;
  const int p = prefix_lens[i / nb];
  out[i] = p < 0 ? p : p + (i % nb) * L;
}
}  // namespace

cudaError_t launch_prompt_prefix(const int32_t* prefix_lens, int B, int nb, int L, int32_t* out,
                                 cudaStream_t stream) {
  const int n = B * nb;
  return launch_pdl(prompt_prefix_kernel, dim3((n + 255) / 256), dim3(256), 0, stream,
                    prefix_lens, B, nb, L, out);
}

AttnPlan plan_attention(int B, int L, int Hq, int Hkv, int max_pages, int page_size,
                        int num_sms) {
  AttnPlan pl;
  if (page_size != kPage || Hkv <= 0 || Hq % Hkv != 0) {
    pl.n_mma = 0;
    return pl;
  }
  pl.G = Hq / Hkv;
  pl.rows = pl.G * L;
  // one item takes up to 256 query rows (two sub-groups of 128 sharing the K/V); more rows
  // are cut into row groups of 256 that each read the K/V
  if (pl.rows <= 256) {
    pl.lsub = L;
    pl.row_groups = 1;
  } else {
    pl.lsub = 256 / pl.G;
    pl.row_groups = (L + pl.lsub - 1) / pl.lsub;
  }
  const int rpg = pl.G * pl.lsub;
  // up to 32 query rows: S^T = K Q^T with the rows on N; more: S = Q K^T, 128 rows on M per
  // sub-group (n_mma = 256: two sub-groups)
  pl.n_mma = rpg <= 16 ? 16 : rpg <= 32 ? 32 : rpg <= 128 ? 128 : 256;
  // tensor memory per CTA holds two S^T chunks and O^T (rows on N), two S tiles and O (one
  // sub-group), or S and O of each of two sub-groups
  const int ctas_per_sm = pl.n_mma <= 32 ? 2 : 1;
  pl.tmem_cols = 512 / ctas_per_sm;
  pl.chunk_tiles = pl.n_mma >= 128 ? 1 : (pl.tmem_cols - pl.n_mma) / (2 * pl.n_mma);
  const int chunks_per_split = pl.n_mma == 16 ? 1 : pl.n_mma == 32 ? 3 : 16;
  pl.split_tokens = pl.chunk_tiles * kTile * chunks_per_split;
  if (pl.split_tokens > kMaxSplitTokens) pl.split_tokens = kMaxSplitTokens;
  if (pl.n_mma >= 128) {
    // rows on M: every item reloads its Q and writes a partial, so splits are long and cut
    // evenly (no short remainder split pays those costs for a tile or two)
    pl.even = true;
    pl.split_tokens = pl.n_mma == 256 ? kSplitTokensTwo : kSplitTokensRows;
  }
  const long long max_tok = static_cast<long long>(max_pages) * kPage;
  const size_t groups = static_cast<size_t>(B) * Hkv * pl.row_groups;
  const long long ctas = static_cast<long long>(num_sms) * ctas_per_sm;
  pl.whole = B <= kMaxOrderSeqs && max_pages <= kMaxItemPages &&
             static_cast<long long>(groups) >= kWholeItemsPerCta * ctas;
  if (pl.whole) {
    // every item is a whole sequence: no partials, no merge; the workspace holds the order
    pl.even = false;
    pl.split_tokens = static_cast<int>((max_tok + kTile - 1) / kTile * kTile);
    pl.max_splits = 1;
    pl.part_bytes = static_cast<size_t>(B) * sizeof(int);
    pl.cnt_bytes = 2 * sizeof(int);
    return pl;
  }
  pl.max_splits = static_cast<int>((max_tok + pl.split_tokens - 1) / pl.split_tokens);
  pl.part_bytes = groups * pl.max_splits * static_cast<size_t>(pl.n_mma) * 130 * sizeof(float);
  if (pl.even && B <= kMaxOrderSeqs) {
    // items longest first: the sequence order goes after the partials
    pl.ranked = true;
    pl.order_offset = pl.part_bytes;
    pl.part_bytes += static_cast<size_t>(B) * sizeof(int);
  }
  pl.cnt_bytes = 2 * sizeof(int);  // the scheduler's next-item and finished-CTA counters
  return pl;
}

cudaError_t launch_attention(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const int32_t* page_table,
                             const int32_t* prefix_lens, uint16_t* out, int B, int L, int Hq,
                             int Hkv, int max_pages, int num_pages, float sm_scale,
                             const AttnPlan& plan, float* part, int* cnt, int* err, int num_sms,
                             cudaStream_t stream, int table_div, int mask_block,
                             const BlockKvWrite* kv_write) {
  AttnParams prm;
  prm.mask_block = mask_block > 0 ? mask_block : 0;
  prm.k_new = kv_write ? kv_write->k_new : nullptr;
  prm.v_new = kv_write ? kv_write->v_new : nullptr;
  prm.k_pool = kv_write ? kv_write->k_pages : nullptr;
  prm.v_pool = kv_write ? kv_write->v_pages : nullptr;
  if (kv_write && mask_block > 0) return cudaErrorInvalidValue;   // prefill writes separately
  prm.page_table = page_table;
  prm.table_div = table_div < 1 ? 1 : table_div;
  prm.prefix_lens = prefix_lens;
  prm.out = out;
  prm.part = part;
  prm.work = cnt;  // two words of scheduler state
  prm.order = nullptr;
  prm.err = err;
  prm.B = B;
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
  prm.even_splits = plan.even ? 1 : 0;
  prm.max_splits = plan.max_splits;
  prm.chunk_tiles = plan.chunk_tiles;
  prm.scale_log2 = sm_scale * 1.4426950408889634f;
  const long long items = static_cast<long long>(B) * Hkv * plan.max_splits * plan.row_groups;
  if (items > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  prm.total_items = static_cast<int>(items);
  prm.rank_major = 0;
  cudaError_t e;
  if (plan.whole) {
    int* order = reinterpret_cast<int*>(part);
    e = launch_pdl(attn_order_kernel, dim3(1), dim3(kMaxOrderSeqs), 0, stream, prm, true, order);
    if (e != cudaSuccess) return e;
    prm.order = order;
    prm.part = nullptr;
  } else if (plan.ranked) {
    // even splits, sequences by decreasing split length: the order follows the partials
    int* order = reinterpret_cast<int*>(reinterpret_cast<char*>(part) + plan.order_offset);
    e = launch_pdl(attn_order_kernel, dim3(1), dim3(kMaxOrderSeqs), 0, stream, prm, false, order);
    if (e != cudaSuccess) return e;
    prm.order = order;
    prm.rank_major = 1;
  }
  switch (plan.n_mma) {
    case 16:
      if (mask_block > 0) return cudaErrorInvalidValue;   // the mask needs rows on M
      e = launch_t<16, 3, 2, false, false, false>(tm_q, tm_k, tm_v, prm, num_sms, stream);
      break;
    case 32:
      if (mask_block > 0) return cudaErrorInvalidValue;
      e = launch_t<32, 2, 2, false, false, false>(tm_q, tm_k, tm_v, prm, num_sms, stream);
      break;
    case 128:
      e = mask_block > 0
              ? launch_t<128, 5, 1, true, true, false>(tm_q, tm_k, tm_v, prm, num_sms, stream)
              : launch_t<128, 5, 1, false, true, false>(tm_q, tm_k, tm_v, prm, num_sms, stream);
      break;
    case 256:   // two sub-groups of 128 query rows sharing the K/V
      e = mask_block > 0
              ? launch_t<128, 4, 1, true, true, true>(tm_q, tm_k, tm_v, prm, num_sms, stream)
              : launch_t<128, 4, 1, false, true, true>(tm_q, tm_k, tm_v, prm, num_sms, stream);
      break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess || plan.max_splits <= 1) return e;
  const long long groups = static_cast<long long>(B) * Hkv * plan.row_groups;
  const int row_blocks = (plan.G * plan.lsub + 8 * kMergeRows - 1) / (8 * kMergeRows);
  e = launch_pdl(attn_merge_kernel, dim3(static_cast<unsigned>(groups), row_blocks), dim3(256), 0,
                 stream, prm, plan.n_mma);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace bdlm
