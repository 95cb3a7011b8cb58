// Internal interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/bdlm.h"

namespace bdlm {

// Launches `kernel` with a programmatic dependency on the previous work of `stream`: its
// CTAs may start while the predecessor drains, and wait (griddepcontrol.wait) before they
// read anything the predecessor writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Runs `set` (a kernel-attribute setter) once per device: function attributes belong to a
// device's context, so a flag per process would leave a second device without them.  Two
// threads may both run `set` the first time; it is idempotent.  Devices past 63 run it on
// every call.
template <typename F>
cudaError_t once_per_device(std::atomic<unsigned long long>& done, F&& set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = set();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// ------------------------------------------------------------------ commit
// A partial row state: (max, sum of exponentials, first argmax, exponent-weighted sum); see
// confidence.cuh.
struct CommitPartial {
  float m;
  float s;
  int idx;
  float a;
};

struct CommitPlan {
  long long total_items = 0;  // rows
  int grid = 1;               // CTAs (one per SM, persistent)
  size_t smem_bytes = 0;
  size_t part_bytes = 0;      // one partial per (warp, masked row segment)
};

CommitPlan plan_commit(int B, int L, int V, int num_sms);
// The streaming kernel and the per-block finalize kernel; ent_out may be null.
cudaError_t launch_commit(const uint16_t* logits, const uint8_t* mask, int B, int L, int V,
                          float threshold, float temperature, int32_t* tok_out, float* conf_out,
                          float* ent_out, uint8_t* commit_out, const CommitPlan& plan,
                          CommitPartial* part, int* err, cudaStream_t stream,
                          int rule = BDLM_COMMIT_THRESHOLD, int k = 1);
cudaError_t launch_apply_commit(uint8_t* mask, const uint8_t* commit, int n, cudaStream_t stream);
// The error word of bdlm_confidence_commit_noalloc's fixed array on device `dev`, read and
// cleared (0 if the array was never set up there); allocates nothing.
int noalloc_take_error(int dev, int* bits);

// ------------------------------------------------------------------ attention
struct AttnPlan {
  int G = 1;             // query heads per KV head
  int rows = 0;          // query rows of one (sequence, KV head): G * L
  int row_groups = 1;    // CTAs splitting those rows (<= 128 rows each)
  int lsub = 0;          // block positions per row group
  int n_mma = 16;        // UMMA N: rows per group rounded up to a multiple of 16
  int split_tokens = 0;  // KV tokens per split (multiple of 128)
  int max_splits = 1;    // splits of the longest possible sequence
  int chunk_tiles = 1;   // 128-token tiles per S chunk held in tensor memory
  int tmem_cols = 0;     // tensor-memory columns allocated per CTA
  bool whole = false;    // whole sequences, longest first, instead of KV splits
  bool even = false;     // each sequence cut into equal splits of at most split_tokens
  bool ranked = false;   // even splits handed out sequence by sequence, longest splits first
  size_t order_offset = 0;   // ranked: byte offset of the sequence order in the workspace
  size_t smem_bytes = 0;
  size_t part_bytes = 0, cnt_bytes = 0;
};

AttnPlan plan_attention(int B, int L, int Hq, int Hkv, int max_pages, int page_size,
                        int num_sms);
// The block's new K/V [B, L, Hkv, D] and the pools they go to: the attention writes them into
// the cache itself, before it reads them.
struct BlockKvWrite {
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_pages;
  uint16_t* v_pages;
};
// Sequence b uses page-table row b / table_div.  mask_block > 0 makes the queries of a
// sequence block-causal: query i sees the prefix and the sequence's keys up to the end of its
// own block of mask_block queries (chunked prefill); else every query sees all L.  kv_write
// (may be null; not with mask_block) fuses the block's K/V-cache write into the attention.
cudaError_t launch_attention(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const int32_t* page_table,
                             const int32_t* prefix_lens, uint16_t* out, int B, int L, int Hq,
                             int Hkv, int max_pages, int num_pages, float sm_scale,
                             const AttnPlan& plan, float* part, int* cnt, int* err, int num_sms,
                             cudaStream_t stream, int table_div = 1, int mask_block = 0,
                             const BlockKvWrite* kv_write = nullptr);

// ------------------------------------------------------------------ LM head
struct LmHeadPlan {
  int bn = 256;          // UMMA N (gathered rows per tile), a multiple of 16
  int bn_max = 256;      // shared-memory ring layout: 64, 128 or 256 rows per row stage
  int m_tiles = 0, n_tiles = 0, grid = 0;
  size_t smem_bytes = 0;
  size_t gather_bytes = 0;
};

LmHeadPlan plan_lm_head(int n_active, int H, int V, int num_sms);
cudaError_t launch_gather_rows(const uint16_t* hidden, const int32_t* active_idx, int n_active,
                               const int32_t* n_active_dev, int n_rows, int H,
                               uint16_t* gathered, int* err, cudaStream_t stream);
// n_active_dev (may be null): the active-row count in device memory, at most n_active (the
// count the launch is planned for); rows of active_idx past it are ignored.
cudaError_t launch_lm_head(const CUtensorMap& tm_w, const CUtensorMap& tm_h,
                           const int32_t* active_idx, int n_active,
                           const int32_t* n_active_dev, int n_rows, int H, int V,
                           uint16_t* logits, const LmHeadPlan& plan, int* err,
                           cudaStream_t stream);

// LM head fused with the confidence step: partials of (max, sum of exponentials, first
// argmax, and with `ent` the exponent-weighted sum the entropy needs) per (active row, slot); a
// per-block kernel merges them and decides the commit.
struct LmConfPlan {
  int grid = 0;            // persistent CTAs (one per SM)
  int units = 0;           // workers: CTA pairs of the pair kernel, else CTAs
  bool pair = false;       // the CTA-pair kernel (more than 128 rows planned)
  int slots = 0;           // partial slots per active row (one per worker, at most)
  int m_tiles = 0;         // vocabulary tiles of 256
  int max_row_tiles = 0;   // row tiles of 256 at the planned maximum of active rows
  size_t smem_bytes = 0;
  size_t gather_bytes = 0;
  size_t part_bytes = 0;
};

LmConfPlan plan_lm_conf(int max_rows, int H, int V, int num_sms);
cudaError_t launch_lm_conf(const CUtensorMap& tm_w, const CUtensorMap& tm_h,
                           const int32_t* active_idx, const int32_t* n_active_dev, int max_rows,
                           int n_rows, int H, int V, float temperature, uint16_t* logits,
                           CommitPartial* part, const LmConfPlan& plan, int* err,
                           cudaStream_t stream, bool ent = false);
// The scored rows (masked, in a denoising sequence) listed in act / *n_act and their hidden
// rows gathered, in one launch of B * L CTAs.
cudaError_t launch_scored_gather(const uint16_t* hidden, const uint8_t* mask,
                                 const uint8_t* denoising, int B, int L, int H,
                                 uint16_t* gathered, int32_t* act, int32_t* n_act,
                                 cudaStream_t stream);
// One CTA per block: tok/conf of the block's scored positions (masked, and in a denoising
// sequence when `denoising` is given) from their partials, then the block's commit.
cudaError_t launch_lm_commit_finalize(const uint8_t* mask, const uint8_t* denoising, int B, int L,
                                      const CommitPartial* part, const LmConfPlan& plan,
                                      float temperature, int rule, int k, float threshold,
                                      int32_t* tok_out, float* conf_out, float* ent_out,
                                      uint8_t* commit_out, cudaStream_t stream);

// Prompt chunk j of sequence b -> attention sequence b * nb + j with prefix prefix[b] + j * L.
cudaError_t launch_prompt_prefix(const int32_t* prefix_lens, int B, int nb, int L, int32_t* out,
                                 cudaStream_t stream);

// Device-side round pieces (round.cu).
struct StepCopy {  // per-step inputs: slice s of src[j] (n_vec[j] 16-byte vectors) -> dst[j]
  static constexpr int kMax = 4;
  const uint4* src[kMax];
  uint4* dst[kMax];
  long long n_vec[kMax];
};
cudaError_t launch_select_step(const StepCopy& c, const int* step, int n_steps,
                               cudaStream_t stream);
// out_s (may be null): per-step copies of out (out_vec 16-byte vectors per step).
cudaError_t launch_record_step(const int* step, int n_steps, int R, const int32_t* tok,
                               const float* conf, const uint8_t* commit, int32_t* tok_s,
                               float* conf_s, uint8_t* commit_s, const uint4* out, uint4* out_s,
                               long long out_vec, cudaStream_t stream);
// One CTA whose bounded wait runs out after limit_ns, recorded as BDLM_DEVERR_TIMEOUT in *err.
cudaError_t launch_wait_timeout(int* err, unsigned long long limit_ns, cudaStream_t stream);
cudaError_t launch_loop_condition(cudaGraphConditionalHandle handle, const uint8_t* mask, int R,
                                  int* step, int n_steps, int* steps_done, cudaStream_t stream);
cudaError_t launch_active_rows(const uint8_t* mask, const uint8_t* denoising, int B, int L,
                               int32_t* active_idx, int32_t* n_active, cudaStream_t stream);
cudaError_t launch_write_block_kv(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_pages,
                                  uint16_t* v_pages, const int32_t* page_table,
                                  const int32_t* prefix_lens, int B, int L, int Hkv,
                                  int max_pages, int num_pages, int* err, cudaStream_t stream);

}  // namespace bdlm
