// bdlm_confidence_commit_noalloc: the confidence/commit step without any device allocation.
//
// Some callers cannot let this library call cudaMalloc: a serving engine that reserved the
// GPU's memory up front for its own pools (model weights, the paged KV cache) and hands
// out nothing else, or a latency-critical decode loop where an allocation's implicit device
// synchronisation is not acceptable.  This entry point runs the same kernel as
// bdlm_confidence_commit, but its scratch (per-warp partial results and an error word) lives
// in a fixed file-scope device array that is part of the loaded module, so no call allocates or
// frees anything.
//
// Limits and behaviour (also stated in include/bdlm.h):
//  * B * L <= kNoAllocMaxRows (2048) and V <= kNoAllocMaxVocab (262144); larger problems are
//    rejected with BDLM_ERR_UNSUPPORTED before anything is launched.
//  * The array (about 96 KiB) stays resident on every GPU that loads the library until the
//    process exits.
//  * The first call on a device looks the array's device address up (cudaGetSymbolAddress)
//    with that device current; make that first call before any stream capture.
//  * Every call shares the one array: calls that overlap on the GPU (different streams, or
//    different host threads without ordering) race and give wrong results.
//  * A device error of the kernel (a bounded wait that gave up) is recorded in the error word
//    at the head of the array.  bdlm_device_error() reads and clears it together with the
//    workspace's word, and allocates nothing either; the calls never clear it themselves, so a
//    recorded error stays until it is read.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/bdlm.h"
#include "kernels.h"

namespace {

constexpr int kNoAllocMaxRows = 2048;
constexpr int kNoAllocMaxVocab = 262144;
constexpr int kNoAllocMaxWarps = 16 * 256;  // the commit kernel runs 16 warps per SM
// layout: [error word] padded to 256 bytes, then the per-(warp, row segment) partials
constexpr size_t kCounterBytes = 256;
constexpr size_t kPartialBytes =
    static_cast<size_t>(kNoAllocMaxWarps + kNoAllocMaxRows) * sizeof(bdlm::CommitPartial);
constexpr size_t kScratchBytes = kCounterBytes + kPartialBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};
int g_noalloc_sms[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void** out, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BDLM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BDLM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return BDLM_ERR_CUDA;
    if (major != 10 || minor != 3) return BDLM_ERR_UNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return BDLM_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
    g_noalloc_sms[dev] = sms;
  }
  *out = g_noalloc_ptr[dev];
  *num_sms = g_noalloc_sms[dev];
  return BDLM_OK;
}

}  // namespace

namespace bdlm {
// Reads and clears the fixed array's device error word on device `dev` into *bits (0 when no
// call has set the array up on that device).  Allocates nothing.
int noalloc_take_error(int dev, int* bits) {
  *bits = 0;
  if (dev < 0 || dev >= kMaxDevices) return BDLM_OK;
  void* p = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    p = g_noalloc_ptr[dev];
  }
  if (p == nullptr) return BDLM_OK;
  if (cudaMemcpy(bits, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return BDLM_ERR_CUDA;
  if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return BDLM_ERR_CUDA;
  return BDLM_OK;
}
}  // namespace bdlm

extern "C" int bdlm_confidence_commit_noalloc(const bdlm_bf16* logits, const uint8_t* mask, int B,
                                              int L, int V, float threshold, float temperature,
                                              int32_t* tok_out, float* conf_out,
                                              uint8_t* commit_out, bdlm_stream stream) {
  if (B < 0 || L < 1 || L > 64 || V < 1) return BDLM_ERR_INVALID;
  if (!(temperature > 0.f) || !isfinite(temperature)) return BDLM_ERR_INVALID;
  if (!(threshold >= 0.f && threshold <= 1.f)) return BDLM_ERR_INVALID;
  if (B == 0) return BDLM_OK;
  if (!logits || !mask || !tok_out || !conf_out || !commit_out) return BDLM_ERR_INVALID;
  if (static_cast<long long>(B) * L > kNoAllocMaxRows || V > kNoAllocMaxVocab)
    return BDLM_ERR_UNSUPPORTED;  // beyond the fixed scratch array
  void* base = nullptr;
  int sms = 0;
  int rc = scratch_address(&base, &sms);
  if (rc) return rc;
  const bdlm::CommitPlan plan = bdlm::plan_commit(B, L, V, sms);
  if (plan.part_bytes > kPartialBytes) return BDLM_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* p = static_cast<unsigned char*>(base);
  int* err = reinterpret_cast<int*>(p);
  auto* part = reinterpret_cast<bdlm::CommitPartial*>(p + kCounterBytes);
  cudaError_t e = bdlm::launch_commit(logits, mask, B, L, V, threshold, temperature, tok_out,
                                      conf_out, nullptr, commit_out, plan, part, err, s);
  return e == cudaSuccess ? BDLM_OK : BDLM_ERR_CUDA;
}
