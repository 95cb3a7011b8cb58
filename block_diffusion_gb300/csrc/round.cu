// Device-side pieces that let a whole denoising round run without the host: the list of
// active rows computed from the mask on the device, and the write of a block's new K/V into
// the paged cache.
//
// Source: JetEngine notes (CLAUDE.md), "ModelRunner" (selective logits: the LM head runs for
// the rows still being denoised), "Important Patterns" (the block's K/V live in the paged
// cache at the slots after the prefix; a finished block's K/V are written by a SAVING pass)
// and "Optimization History" (opt18/opt24: the KV-cache write of the block combined with the
// paged attention); dlmrt page, "Highlights" (a block's rounds run inside one CUDA graph).
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int kScanThreads = 1024;

// Row r = b * L + i is active when mask[r] != 0 and (no flags, or denoising[b] != 0).  The
// active rows in increasing order go to active_idx and their number to *n_active.  One CTA:
// a block-wide scan over chunks of kScanThreads rows.
__global__ void __launch_bounds__(kScanThreads)
active_rows_kernel(const uint8_t* __restrict__ mask, const uint8_t* __restrict__ denoising,
                   int R, int L, int32_t* __restrict__ active_idx, int32_t* __restrict__ n_active) {
  __shared__ int s_warp[kScanThreads / 32];
  __shared__ int s_base;
  griddep_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_base = 0;
  __syncthreads();
  for (int r0 = 0; r0 < R; r0 += kScanThreads) {
    const int r = r0 + tid;
    int a = 0;
    if (r < R) a = mask[r] != 0 && (denoising == nullptr || denoising[r / L] != 0);
    const unsigned bal = __ballot_sync(0xffffffffu, a);
    if (lane == 0) s_warp[warp] = __popc(bal);
    __syncthreads();
    int before = s_base;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    if (a) active_idx[before + __popc(bal & ((1u << lane) - 1u))] = r;
    __syncthreads();
    if (tid == 0) {
      int total = 0;
      for (int w = 0; w < kScanThreads / 32; ++w) total += s_warp[w];
      s_base += total;
    }
    __syncthreads();
  }
  if (tid == 0) *n_active = s_base;
  griddep_launch_dependents();
}

// k_new, v_new [B, L, Hkv, D=128] -> the cache slots prefix_len .. prefix_len + L - 1 of each
// sequence.  A token's Hkv * D values are contiguous both in k_new / v_new and in its page slot
// ([page, slot, Hkv, D]), so one warp per token row (b, i) copies two contiguous runs of
// Hkv * 256 bytes in 16-byte vectors, all of a pass's loads before its stores.  Page ids and
// lengths are checked; a bad one skips the row and sets the device error word.
constexpr int kKvWarps = 8;      // token rows per CTA
constexpr int kKvVecLane = 4;    // 16-byte vectors per lane and tensor in one pass
__global__ void __launch_bounds__(kKvWarps * 32)
write_block_kv_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                      uint16_t* __restrict__ k_pages, uint16_t* __restrict__ v_pages,
                      const int32_t* __restrict__ page_table,
                      const int32_t* __restrict__ prefix_lens, int B, int L, int Hkv,
                      int max_pages, int num_pages, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int t = blockIdx.x * kKvWarps + (threadIdx.x >> 5);  // token row b * L + i
  const int lane = threadIdx.x & 31;
  if (t >= B * L) return;
  const int b = t / L, i = t - b * L;
  const int prefix = prefix_lens[b];
  if (prefix < 0 || static_cast<long long>(prefix) + L > static_cast<long long>(max_pages) * 16) {
    if (lane == 0 && i == 0) atomicOr(err, BDLM_DEVERR_LENGTH);
    return;
  }
  const int tok = prefix + i;
  const int page = page_table[static_cast<size_t>(b) * max_pages + tok / 16];
  if (page < 0 || page >= num_pages) {
    if (lane == 0) atomicOr(err, BDLM_DEVERR_PAGE);
    return;
  }
  const int nvec = Hkv * 16;  // 16-byte vectors in a token row
  const uint4* ks = reinterpret_cast<const uint4*>(k_new) + static_cast<size_t>(t) * nvec;
  const uint4* vs = reinterpret_cast<const uint4*>(v_new) + static_cast<size_t>(t) * nvec;
  const size_t slot = static_cast<size_t>(page) * 16 + tok % 16;
  uint4* kd = reinterpret_cast<uint4*>(k_pages) + slot * nvec;
  uint4* vd = reinterpret_cast<uint4*>(v_pages) + slot * nvec;
  for (int v0 = 0; v0 < nvec; v0 += 32 * kKvVecLane) {
    uint4 kr[kKvVecLane], vr[kKvVecLane];
#pragma unroll
    for (int q = 0; q < kKvVecLane; ++q) {
      const int v = v0 + q * 32 + lane;
      if (v < nvec) {
        kr[q] = ks[v];
        vr[q] = vs[v];
      }
    }
#pragma unroll
    for (int q = 0; q < kKvVecLane; ++q) {
      const int v = v0 + q * 32 + lane;
      if (v < nvec) {
        kd[v] = kr[q];
        vd[v] = vr[q];
      }
    }
  }
}

// Copies step *step's slice of up to four per-step inputs into their working buffers.
__global__ void select_step_kernel(StepCopy c, const int* __restrict__ step, int n_steps) {
  griddep_wait();
  griddep_launch_dependents();
  long long s = *step;
  if (s < 0) s = 0;
  if (s >= n_steps) s = n_steps - 1;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
#pragma unroll
  for (int j = 0; j < StepCopy::kMax; ++j) {
    if (c.dst[j] == nullptr) continue;
    const uint4* src = c.src[j] + s * c.n_vec[j];
    for (long long v = tid; v < c.n_vec[j]; v += stride) c.dst[j][v] = src[v];
  }
}

// Stores this step's tok/conf/commit (and, when out_s is given, the attention output: out_vec
// 16-byte vectors) into slice *step of the per-step outputs.
__global__ void record_step_kernel(const int* __restrict__ step, int n_steps, int R,
                                   const int32_t* __restrict__ tok, const float* __restrict__ conf,
                                   const uint8_t* __restrict__ commit, int32_t* __restrict__ tok_s,
                                   float* __restrict__ conf_s, uint8_t* __restrict__ commit_s,
                                   const uint4* __restrict__ out, uint4* __restrict__ out_s,
                                   long long out_vec) {
  griddep_wait();
  griddep_launch_dependents();
  const int s = *step;
  if (s < 0 || s >= n_steps) return;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < R; r += gridDim.x * blockDim.x) {
    const size_t o = static_cast<size_t>(s) * R + r;
    tok_s[o] = tok[r];
    conf_s[o] = conf[r];
    commit_s[o] = commit[r];
  }
  if (out_s == nullptr) return;
  uint4* dst = out_s + s * out_vec;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < out_vec;
       v += stride)
    dst[v] = out[v];
}

// End of a round: counts it, and repeats the loop while some position is still masked and
// fewer than n_steps rounds have run.  One CTA.
__global__ void __launch_bounds__(kScanThreads)
loop_condition_kernel(cudaGraphConditionalHandle handle, const uint8_t* __restrict__ mask, int R,
                      int* __restrict__ step, int n_steps, int* __restrict__ steps_done) {
  griddep_wait();
  int any = 0;
  for (int r = threadIdx.x; r < R && !any; r += blockDim.x) any = mask[r] != 0;
  any = __syncthreads_or(any);
  if (threadIdx.x == 0) {
    const int s = *step + 1;
    *step = s;
    *steps_done = s;
    cudaGraphSetConditional(handle, (any && s < n_steps) ? 1u : 0u);
  }
}

}  // namespace

cudaError_t launch_select_step(const StepCopy& c, const int* step, int n_steps,
                               cudaStream_t stream) {
  long long most = 0;
  for (int j = 0; j < StepCopy::kMax; ++j)
    if (c.dst[j] && c.n_vec[j] > most) most = c.n_vec[j];
  const long long blocks = (most + 255) / 256;
  const unsigned grid = static_cast<unsigned>(blocks < 1 ? 1 : (blocks > 1216 ? 1216 : blocks));
  return launch_pdl(select_step_kernel, dim3(grid), dim3(256), 0, stream, c, step, n_steps);
}

namespace {
// One thread waits, through the kernels' bounded wait, on an mbarrier that nothing arrives on,
// and records the timeout in the device error word as a kernel's failed wait does.
__global__ void wait_timeout_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  abort_flag = 0;
  if (!mbar_wait(&bar, 0, &abort_flag, limit_ns)) atomicOr(err, BDLM_DEVERR_TIMEOUT);
}
}  // namespace

cudaError_t launch_wait_timeout(int* err, unsigned long long limit_ns, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_record_step(const int* step, int n_steps, int R, const int32_t* tok,
                               const float* conf, const uint8_t* commit, int32_t* tok_s,
                               float* conf_s, uint8_t* commit_s, const uint4* out, uint4* out_s,
                               long long out_vec, cudaStream_t stream) {
  long long blocks = (R + 255) / 256;
  if (out_s != nullptr) {
    const long long ob = (out_vec + 255) / 256;
    if (ob > blocks) blocks = ob > 1216 ? 1216 : ob;
  }
  const unsigned grid = static_cast<unsigned>(blocks < 1 ? 1 : blocks);
  return launch_pdl(record_step_kernel, dim3(grid), dim3(256), 0, stream, step, n_steps, R, tok,
                    conf, commit, tok_s, conf_s, commit_s, out, out_s, out_vec);
}

cudaError_t launch_loop_condition(cudaGraphConditionalHandle handle, const uint8_t* mask, int R,
                                  int* step, int n_steps, int* steps_done, cudaStream_t stream) {
  return launch_pdl(loop_condition_kernel, dim3(1), dim3(kScanThreads), 0, stream, handle, mask,
                    R, step, n_steps, steps_done);
}

cudaError_t launch_active_rows(const uint8_t* mask, const uint8_t* denoising, int B, int L,
                               int32_t* active_idx, int32_t* n_active, cudaStream_t stream) {
  return launch_pdl(active_rows_kernel, dim3(1), dim3(kScanThreads), 0, stream, mask, denoising,
                    B * L, L, active_idx, n_active);
}

cudaError_t launch_write_block_kv(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_pages,
                                  uint16_t* v_pages, const int32_t* page_table,
                                  const int32_t* prefix_lens, int B, int L, int Hkv,
                                  int max_pages, int num_pages, int* err, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * L;  // token rows (callers keep it < 2^31)
  const unsigned grid = static_cast<unsigned>((rows + kKvWarps - 1) / kKvWarps);
  return launch_pdl(write_block_kv_kernel, dim3(grid), dim3(kKvWarps * 32), 0, stream, k_new, v_new,
                    k_pages, v_pages, page_table, prefix_lens, B, L, Hkv, max_pages, num_pages,
                    err);
}

}  // namespace bdlm
