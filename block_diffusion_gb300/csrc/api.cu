// C-ABI of the bdlm library: argument validation, the per-device workspace, TMA tensor
// maps and kernel launches.  See include/bdlm.h for the contract of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/bdlm.h"
#include "kernels.h"

namespace {

using bdlm::AttnPlan;
using bdlm::CommitPlan;
using bdlm::LmHeadPlan;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool checked = false;
  bool supported = false;
  int num_sms = 0;
  int* err = nullptr;            // device error word
  int* attn_cnt = nullptr;       // attention scheduler counters (zero between calls)
  size_t attn_cnt_cap = 0;
  void* data = nullptr;          // split / commit partials, gathered rows, sequence order
  size_t data_cap = 0;
  void* aux = nullptr;           // prompt-block prefix lengths of a prefill
  size_t aux_cap = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
// Bumped whenever a workspace is reallocated or freed: CUDA graphs that captured the old
// buffers are re-captured before their next launch.
unsigned g_workspace_gen = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int current_device(DeviceState** st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BDLM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BDLM_ERR_UNSUPPORTED;
  DeviceState& s = g_dev[dev];
  if (!s.checked) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return BDLM_ERR_CUDA;
    s.supported = (major == 10 && minor == 3);
    s.num_sms = sms;
    s.checked = true;
    if (s.supported) {
      if (cudaMalloc(&s.err, 256) != cudaSuccess) return BDLM_ERR_NOMEM;
      if (cudaMemset(s.err, 0, 256) != cudaSuccess) return BDLM_ERR_CUDA;
    }
  }
  if (!s.supported) return BDLM_ERR_UNSUPPORTED;
  *st = &s;
  return BDLM_OK;
}

// Grows a zero-initialised buffer; growing waits for the device to be idle first.
int ensure(void** ptr, size_t* cap, size_t need, bool zero) {
  if (need <= *cap) return BDLM_OK;
  size_t n = need + need / 4 + 4096;
  ++g_workspace_gen;
  if (*ptr) {
    if (cudaDeviceSynchronize() != cudaSuccess) return BDLM_ERR_CUDA;
    cudaFree(*ptr);
    *ptr = nullptr;
    *cap = 0;
  }
  if (cudaMalloc(ptr, n) != cudaSuccess) {
    *ptr = nullptr;
    return BDLM_ERR_NOMEM;
  }
  if (zero && cudaMemset(*ptr, 0, n) != cudaSuccess) return BDLM_ERR_CUDA;
  *cap = n;
  return BDLM_OK;
}

int get_encoder() {
  if (g_encode) return BDLM_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return BDLM_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return BDLM_OK;
}

// bf16 tensor map, 128-byte swizzle; dims/strides innermost first, strides in bytes.
int encode(CUtensorMap* tm, const void* base, int rank, const cuuint64_t* dims,
           const cuuint64_t* strides, const cuuint32_t* box) {
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base),
                        dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BDLM_OK : BDLM_ERR_INVALID;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Arguments of a commit rule: the threshold rule wants 0 <= threshold <= 1, the entropy rule a
// finite budget >= 0 (in `threshold`), the others k >= 1.
bool rule_ok(int rule, int k, float threshold) {
  switch (rule) {
    case BDLM_COMMIT_THRESHOLD: return threshold >= 0.f && threshold <= 1.f;
    case BDLM_COMMIT_ENTROPY_BOUNDED: return threshold >= 0.f && isfinite(threshold);
    case BDLM_COMMIT_TOPK:
    case BDLM_COMMIT_SEQUENTIAL:
    case BDLM_COMMIT_ANTI_SEQUENTIAL: return k >= 1;
    default: return false;
  }
}

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// Workspace of the fused LM head + commit: gathered rows | partials | scored-row list | count.
struct LmCommitLayout {
  size_t off_part, off_act, off_n, total;
};
LmCommitLayout lm_commit_layout(const bdlm::LmConfPlan& plan, int rows) {
  LmCommitLayout l;
  l.off_part = align256(plan.gather_bytes);
  l.off_act = l.off_part + align256(plan.part_bytes);
  l.off_n = l.off_act + align256(static_cast<size_t>(rows) * sizeof(int32_t));
  l.total = l.off_n + 256;
  return l;
}

int attention_impl(DeviceState* st, const bdlm_attn_desc& d, const bdlm_bf16* q,
                   const bdlm_bf16* k_pages, const bdlm_bf16* v_pages, const int32_t* page_table,
                   const int32_t* prefix_lens, bdlm_bf16* out, bdlm_stream stream,
                   int table_div, int mask_block = 0,
                   const bdlm::BlockKvWrite* kv_write = nullptr);

}  // namespace

extern "C" {

const char* bdlm_status_string(int status) {
  switch (status) {
    case BDLM_OK: return "ok";
    case BDLM_ERR_INVALID: return "invalid argument";
    case BDLM_ERR_CUDA: return "CUDA error";
    case BDLM_ERR_UNSUPPORTED: return "unsupported device or shape";
    case BDLM_ERR_NOMEM: return "workspace allocation failed";
    default: return "unknown status";
  }
}

int bdlm_device_error(int* bits_out) {
  if (!bits_out) return BDLM_ERR_INVALID;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BDLM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BDLM_ERR_UNSUPPORTED;
  if (cudaDeviceSynchronize() != cudaSuccess) return BDLM_ERR_CUDA;
  int v = 0;
  {
    // the workspace's word exists once an allocating call has run on this device
    std::lock_guard<std::mutex> lk(g_mu);
    const DeviceState& s = g_dev[dev];
    if (s.err) {
      if (cudaMemcpy(&v, s.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return BDLM_ERR_CUDA;
      if (cudaMemset(s.err, 0, sizeof(int)) != cudaSuccess) return BDLM_ERR_CUDA;
    }
  }
  int w = 0;
  const int rc = bdlm::noalloc_take_error(dev, &w);  // bdlm_confidence_commit_noalloc's word
  if (rc) return rc;
  *bits_out = v | w;
  return BDLM_OK;
}

int bdlm_selftest_wait_timeout(int limit_us, bdlm_stream stream) {
  if (limit_us < 1 || limit_us > 2000000) return BDLM_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  const int rc = current_device(&st);
  if (rc) return rc;
  const cudaError_t e = bdlm::launch_wait_timeout(
      st->err, static_cast<unsigned long long>(limit_us) * 1000ull,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BDLM_OK : BDLM_ERR_CUDA;
}

int bdlm_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st);
  if (rc) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return BDLM_ERR_CUDA;
  ++g_workspace_gen;
  cudaFree(st->attn_cnt);
  cudaFree(st->data);
  cudaFree(st->aux);
  st->attn_cnt = nullptr;
  st->data = nullptr;
  st->aux = nullptr;
  st->attn_cnt_cap = st->data_cap = st->aux_cap = 0;
  return BDLM_OK;
}

int bdlm_confidence_commit(const bdlm_bf16* logits, const uint8_t* mask, int B, int L, int V,
                           float threshold, float temperature, int32_t* tok_out,
                           float* conf_out, uint8_t* commit_out, bdlm_stream stream) {
  return bdlm_confidence_commit_rule(logits, mask, B, L, V, BDLM_COMMIT_THRESHOLD, 1, threshold,
                                     temperature, tok_out, conf_out, nullptr, commit_out, stream);
}

int bdlm_confidence_commit_rule(const bdlm_bf16* logits, const uint8_t* mask, int B, int L, int V,
                                int rule, int k, float threshold, float temperature,
                                int32_t* tok_out, float* conf_out, float* entropy_out,
                                uint8_t* commit_out, bdlm_stream stream) {
  if (B < 0 || L < 1 || L > 64 || V < 1) return BDLM_ERR_INVALID;
  if (!(temperature > 0.f) || !isfinite(temperature)) return BDLM_ERR_INVALID;
  if (!rule_ok(rule, k, threshold)) return BDLM_ERR_INVALID;
  if (B == 0) return BDLM_OK;
  if (!logits || !mask || !tok_out || !conf_out || !commit_out) return BDLM_ERR_INVALID;
  if (static_cast<long long>(B) * L > 0x7FFFFFFFll) return BDLM_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st);
  if (rc) return rc;
  const CommitPlan plan = bdlm::plan_commit(B, L, V, st->num_sms);
  if (plan.total_items > 0x7FFFFFFFll) return BDLM_ERR_INVALID;
  rc = ensure(&st->data, &st->data_cap, plan.part_bytes, false);
  if (rc) return rc;
  cudaError_t e = bdlm::launch_commit(logits, mask, B, L, V, threshold, temperature, tok_out,
                                      conf_out, entropy_out, commit_out, plan,
                                      static_cast<bdlm::CommitPartial*>(st->data), st->err,
                                      static_cast<cudaStream_t>(stream), rule, k);
  return e == cudaSuccess ? BDLM_OK : BDLM_ERR_CUDA;
}

int bdlm_apply_commit(uint8_t* mask, const uint8_t* commit, int n, bdlm_stream stream) {
  if (n < 0) return BDLM_ERR_INVALID;
  if (n == 0) return BDLM_OK;
  if (!mask || !commit) return BDLM_ERR_INVALID;
  cudaError_t e = bdlm::launch_apply_commit(mask, commit, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BDLM_OK : BDLM_ERR_CUDA;
}

int bdlm_block_attention(const bdlm_attn_desc* desc, const bdlm_bf16* q,
                         const bdlm_bf16* k_pages, const bdlm_bf16* v_pages,
                         const int32_t* page_table, const int32_t* prefix_lens, int L,
                         bdlm_bf16* out, bdlm_stream stream) {
  if (!desc) return BDLM_ERR_INVALID;
  const bdlm_attn_desc d = *desc;
  if (d.B < 0 || L != d.L || d.L < 1 || d.L > 64 || d.Hq < 1 || d.Hkv < 1 ||
      d.Hq % d.Hkv != 0 || d.Hq / d.Hkv > 16 || d.D != 128 || d.page_size != 16 ||
      d.max_pages_per_seq < 1 || d.num_pages < 1 || !isfinite(d.sm_scale))
    return BDLM_ERR_INVALID;
  if (d.B == 0) return BDLM_OK;
  if (!q || !k_pages || !v_pages || !page_table || !prefix_lens || !out) return BDLM_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
    return BDLM_ERR_INVALID;
  if (static_cast<long long>(d.B) * d.L * d.Hq > 0x7FFFFFFFll ||
      static_cast<long long>(d.B) * d.max_pages_per_seq > 0x7FFFFFFFll ||
      static_cast<long long>(d.max_pages_per_seq) * d.page_size > 0x7FFFFFFFll)
    return BDLM_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st);
  if (rc) return rc;
  return attention_impl(st, d, q, k_pages, v_pages, page_table, prefix_lens, out, stream, 1);
}

int bdlm_block_attention_kv(const bdlm_attn_desc* desc, const bdlm_bf16* q,
                            const bdlm_bf16* k_new, const bdlm_bf16* v_new, bdlm_bf16* k_pages,
                            bdlm_bf16* v_pages, const int32_t* page_table,
                            const int32_t* prefix_lens, int L, bdlm_bf16* out,
                            bdlm_stream stream) {
  if (!desc) return BDLM_ERR_INVALID;
  const bdlm_attn_desc d = *desc;
  if (d.B < 0 || L != d.L || d.L < 1 || d.L > 64 || d.Hq < 1 || d.Hkv < 1 ||
      d.Hq % d.Hkv != 0 || d.Hq / d.Hkv > 16 || d.D != 128 || d.page_size != 16 ||
      d.max_pages_per_seq < 1 || d.num_pages < 1 || !isfinite(d.sm_scale))
    return BDLM_ERR_INVALID;
  if (d.B == 0) return BDLM_OK;
  if (!q || !k_new || !v_new || !k_pages || !v_pages || !page_table || !prefix_lens || !out)
    return BDLM_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) ||
      !aligned16(v_pages) || !aligned16(out))
    return BDLM_ERR_INVALID;
  if (static_cast<long long>(d.B) * d.L * d.Hq > 0x7FFFFFFFll ||
      static_cast<long long>(d.B) * d.max_pages_per_seq > 0x7FFFFFFFll ||
      static_cast<long long>(d.max_pages_per_seq) * d.page_size > 0x7FFFFFFFll)
    return BDLM_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st);
  if (rc) return rc;
  const bdlm::BlockKvWrite kw{k_new, v_new, k_pages, v_pages};
  return attention_impl(st, d, q, k_pages, v_pages, page_table, prefix_lens, out, stream, 1, 0,
                        &kw);
}

int bdlm_prefill_attention(const bdlm_attn_desc* desc, int prompt_len, const bdlm_bf16* q,
                           const bdlm_bf16* k_new, const bdlm_bf16* v_new, bdlm_bf16* k_pages,
                           bdlm_bf16* v_pages, const int32_t* page_table,
                           const int32_t* prefix_lens, bdlm_bf16* out, bdlm_stream stream) {
  if (!desc) return BDLM_ERR_INVALID;
  const bdlm_attn_desc d = *desc;
  if (d.B < 0 || d.L < 1 || d.L > 64 || d.Hq < 1 || d.Hkv < 1 || d.Hq % d.Hkv != 0 ||
      d.Hq / d.Hkv > 16 || d.D != 128 || d.page_size != 16 || d.max_pages_per_seq < 1 ||
      d.num_pages < 1 || !isfinite(d.sm_scale))
    return BDLM_ERR_INVALID;
  if (prompt_len < 1 || prompt_len % d.L != 0) return BDLM_ERR_INVALID;
  if (d.B == 0) return BDLM_OK;
  if (!q || !k_new || !v_new || !k_pages || !v_pages || !page_table || !prefix_lens || !out)
    return BDLM_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) ||
      !aligned16(v_pages) || !aligned16(out))
    return BDLM_ERR_INVALID;
  // Queries go to the attention in chunks of Lq positions (a multiple of L dividing the prompt,
  // Lq * G <= 256 query rows per KV head, the most one attention item takes) with the
  // block-causal mask inside a chunk, so each chunk reads the K/V before it once; chunks of
  // one block (Lq = L) need no mask.  Narrow chunks (Lq * G <= 32 rows) stay one block per
  // attention sequence.
  const int G = d.Hq / d.Hkv;
  int Lq = d.L;
  for (int c = d.L; c * G <= 256 && c <= prompt_len; c += d.L)
    if (prompt_len % c == 0) Lq = c;
  if (Lq * G <= 32) Lq = d.L;
  const int nb = prompt_len / Lq;
  if (static_cast<long long>(d.B) * prompt_len * d.Hq > 0x7FFFFFFFll ||
      static_cast<long long>(d.B) * d.max_pages_per_seq > 0x7FFFFFFFll ||
      static_cast<long long>(d.max_pages_per_seq) * d.page_size > 0x7FFFFFFFll)
    return BDLM_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st);
  if (rc) return rc;
  rc = ensure(&st->aux, &st->aux_cap, static_cast<size_t>(d.B) * nb * sizeof(int32_t), false);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the prompt's K/V into the cache, then one attention sequence per chunk of Lq queries
  if (bdlm::launch_write_block_kv(k_new, v_new, k_pages, v_pages, page_table, prefix_lens, d.B,
                                  prompt_len, d.Hkv, d.max_pages_per_seq, d.num_pages, st->err,
                                  s) != cudaSuccess)
    return BDLM_ERR_CUDA;
  int32_t* pre = static_cast<int32_t*>(st->aux);
  if (bdlm::launch_prompt_prefix(prefix_lens, d.B, nb, Lq, pre, s) != cudaSuccess)
    return BDLM_ERR_CUDA;
  bdlm_attn_desc dv = d;
  dv.B = d.B * nb;
  dv.L = Lq;
  return attention_impl(st, dv, q, k_pages, v_pages, page_table, pre, out, stream, nb,
                        Lq > d.L ? d.L : 0);
}
}  // extern "C"

namespace {

// Block attention of d.B sequences (the caller holds g_mu and has validated d); sequence b
// uses page-table row b / table_div; mask_block > 0 makes each sequence's queries
// block-causal in blocks of mask_block.
int attention_impl(DeviceState* st, const bdlm_attn_desc& d, const bdlm_bf16* q,
                   const bdlm_bf16* k_pages, const bdlm_bf16* v_pages, const int32_t* page_table,
                   const int32_t* prefix_lens, bdlm_bf16* out, bdlm_stream stream,
                   int table_div, int mask_block, const bdlm::BlockKvWrite* kv_write) {
  int rc = get_encoder();
  if (rc) return rc;
  const AttnPlan plan = bdlm::plan_attention(d.B, d.L, d.Hq, d.Hkv, d.max_pages_per_seq,
                                             d.page_size, st->num_sms);
  if (plan.n_mma == 0) return BDLM_ERR_UNSUPPORTED;
  rc = ensure(reinterpret_cast<void**>(&st->attn_cnt), &st->attn_cnt_cap, plan.cnt_bytes, true);
  if (rc) return rc;
  rc = ensure(&st->data, &st->data_cap, plan.part_bytes, false);
  if (rc) return rc;
  // q viewed as [B*L rows][Hq heads][D]; box = 64 dims x G heads x lsub rows
  CUtensorMap tm_q, tm_k, tm_v;
  {
    cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(d.Hq), static_cast<cuuint64_t>(d.B) * d.L};
    cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(d.Hq) * 256};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(plan.G), static_cast<cuuint32_t>(plan.lsub)};
    if ((rc = encode(&tm_q, q, 3, dims, strides, box))) return rc;
  }
  {
    // pools viewed as [num_pages][page_size][Hkv][D]; box = 64 dims x 1 head x 16 slots
    cuuint64_t dims[4] = {128, static_cast<cuuint64_t>(d.Hkv), 16,
                          static_cast<cuuint64_t>(d.num_pages)};
    cuuint64_t strides[3] = {256, static_cast<cuuint64_t>(d.Hkv) * 256,
                             static_cast<cuuint64_t>(d.Hkv) * 256 * 16};
    cuuint32_t box[4] = {64, 1, 16, 1};
    if ((rc = encode(&tm_k, k_pages, 4, dims, strides, box))) return rc;
    if ((rc = encode(&tm_v, v_pages, 4, dims, strides, box))) return rc;
  }
  const float scale = d.sm_scale > 0.f ? d.sm_scale : 1.0f / sqrtf(128.0f);
  cudaError_t e = bdlm::launch_attention(tm_q, tm_k, tm_v, page_table, prefix_lens, out, d.B,
                                         d.L, d.Hq, d.Hkv, d.max_pages_per_seq, d.num_pages,
                                         scale, plan, static_cast<float*>(st->data),
                                         st->attn_cnt, st->err, st->num_sms,
                                         static_cast<cudaStream_t>(stream), table_div,
                                         mask_block, kv_write);
  return e == cudaSuccess ? BDLM_OK : BDLM_ERR_CUDA;
}

// The LM head planned for n_active rows; n_active_dev (may be null) holds the count the
// kernels use, read on the device (at most n_active).
int lm_head_impl(const bdlm_bf16* hidden, const bdlm_bf16* w, const int32_t* active_idx,
                 int n_active, const int32_t* n_active_dev, int n_rows, int H, int V,
                 bdlm_bf16* logits, bdlm_stream stream) {
  if (n_active < 0 || n_rows < 0 || H < 8 || V < 8 || H % 8 != 0 || V % 8 != 0 ||
      n_active > n_rows)
    return BDLM_ERR_INVALID;
  if (n_active == 0) return BDLM_OK;
  if (!hidden || !w || !active_idx || !logits) return BDLM_ERR_INVALID;
  if (!aligned16(hidden) || !aligned16(w)) return BDLM_ERR_INVALID;
  if (static_cast<long long>(n_rows) * V > (1ll << 40)) return BDLM_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st);
  if (rc) return rc;
  if ((rc = get_encoder())) return rc;
  const LmHeadPlan plan = bdlm::plan_lm_head(n_active, H, V, st->num_sms);
  rc = ensure(&st->data, &st->data_cap, plan.gather_bytes, false);
  if (rc) return rc;
  uint16_t* gathered = static_cast<uint16_t*>(st->data);
  CUtensorMap tm_w, tm_h;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(V)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[2] = {64, 128};
    if ((rc = encode(&tm_w, w, 2, dims, strides, box))) return rc;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(n_active)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(plan.bn)};
    if ((rc = encode(&tm_h, gathered, 2, dims, strides, box))) return rc;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = bdlm::launch_gather_rows(hidden, active_idx, n_active, n_active_dev, n_rows, H,
                                           gathered, st->err, s);
  if (e != cudaSuccess) return BDLM_ERR_CUDA;
  e = bdlm::launch_lm_head(tm_w, tm_h, active_idx, n_active, n_active_dev, n_rows, H, V, logits,
                           plan, st->err, s);
  return e == cudaSuccess ? BDLM_OK : BDLM_ERR_CUDA;
}

}  // namespace

extern "C" {

int bdlm_lm_head(const bdlm_bf16* hidden, const bdlm_bf16* w, const int32_t* active_idx,
                 int n_active, int n_rows, int H, int V, bdlm_bf16* logits, bdlm_stream stream) {
  return lm_head_impl(hidden, w, active_idx, n_active, nullptr, n_rows, H, V, logits, stream);
}

int bdlm_lm_head_device_count(const bdlm_bf16* hidden, const bdlm_bf16* w,
                              const int32_t* active_idx, const int32_t* n_active_dev,
                              int max_active, int n_rows, int H, int V, bdlm_bf16* logits,
                              bdlm_stream stream) {
  if (!n_active_dev) return BDLM_ERR_INVALID;
  return lm_head_impl(hidden, w, active_idx, max_active, n_active_dev, n_rows, H, V, logits,
                      stream);
}

int bdlm_active_rows(const uint8_t* mask, const uint8_t* denoising, int B, int L,
                     int32_t* active_idx, int32_t* n_active_dev, bdlm_stream stream) {
  if (B < 0 || L < 1 || L > 64 || static_cast<long long>(B) * L > 0x7FFFFFFFll)
    return BDLM_ERR_INVALID;
  if (!mask || !active_idx || !n_active_dev) return BDLM_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st);
  if (rc) return rc;
  cudaError_t e = bdlm::launch_active_rows(mask, denoising, B, L, active_idx, n_active_dev,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BDLM_OK : BDLM_ERR_CUDA;
}

int bdlm_write_block_kv(const bdlm_attn_desc* desc, const bdlm_bf16* k_new,
                        const bdlm_bf16* v_new, bdlm_bf16* k_pages, bdlm_bf16* v_pages,
                        const int32_t* page_table, const int32_t* prefix_lens, bdlm_stream stream) {
  if (!desc) return BDLM_ERR_INVALID;
  const bdlm_attn_desc d = *desc;
  if (d.B < 0 || d.L < 1 || d.L > 64 || d.Hkv < 1 || d.D != 128 || d.page_size != 16 ||
      d.max_pages_per_seq < 1 || d.num_pages < 1)
    return BDLM_ERR_INVALID;
  if (d.B == 0) return BDLM_OK;
  if (!k_new || !v_new || !k_pages || !v_pages || !page_table || !prefix_lens)
    return BDLM_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
    return BDLM_ERR_INVALID;
  if (static_cast<long long>(d.B) * d.L * d.Hkv > 0x7FFFFFFFll ||
      static_cast<long long>(d.B) * d.max_pages_per_seq > 0x7FFFFFFFll)
    return BDLM_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st);
  if (rc) return rc;
  cudaError_t e = bdlm::launch_write_block_kv(k_new, v_new, k_pages, v_pages, page_table,
                                              prefix_lens, d.B, d.L, d.Hkv, d.max_pages_per_seq,
                                              d.num_pages, st->err,
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BDLM_OK : BDLM_ERR_CUDA;
}

int bdlm_lm_head_commit(const bdlm_bf16* hidden, const bdlm_bf16* w, const uint8_t* mask,
                        const uint8_t* denoising, int B, int L, int H, int V, int rule, int k,
                        float threshold, float temperature, int32_t* tok_out, float* conf_out,
                        float* entropy_out, uint8_t* commit_out, bdlm_bf16* logits,
                        bdlm_stream stream) {
  if (B < 0 || L < 1 || L > 64 || H < 8 || V < 8 || H % 8 != 0 || V % 8 != 0)
    return BDLM_ERR_INVALID;
  if (!(temperature > 0.f) || !isfinite(temperature)) return BDLM_ERR_INVALID;
  if (!rule_ok(rule, k, threshold)) return BDLM_ERR_INVALID;
  if (B == 0) return BDLM_OK;
  if (!hidden || !w || !mask || !tok_out || !conf_out || !commit_out) return BDLM_ERR_INVALID;
  if (!aligned16(hidden) || !aligned16(w) || (logits && !aligned16(logits)))
    return BDLM_ERR_INVALID;
  const long long R = static_cast<long long>(B) * L;
  if (R > 0x7FFFFFFFll || R * V > (1ll << 40)) return BDLM_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st);
  if (rc) return rc;
  if ((rc = get_encoder())) return rc;
  const int rows = static_cast<int>(R);
  const bdlm::LmConfPlan plan = bdlm::plan_lm_conf(rows, H, V, st->num_sms);
  if (plan.max_row_tiles > plan.units) return BDLM_ERR_UNSUPPORTED;
  const LmCommitLayout lay = lm_commit_layout(plan, rows);
  rc = ensure(&st->data, &st->data_cap, lay.total, false);
  if (rc) return rc;
  uint8_t* base = static_cast<uint8_t*>(st->data);
  uint16_t* gathered = reinterpret_cast<uint16_t*>(base);
  bdlm::CommitPartial* part = reinterpret_cast<bdlm::CommitPartial*>(base + lay.off_part);
  int32_t* act = reinterpret_cast<int32_t*>(base + lay.off_act);
  int32_t* n_act = reinterpret_cast<int32_t*>(base + lay.off_n);
  CUtensorMap tm_w, tm_h;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(V)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[2] = {64, 128};
    if ((rc = encode(&tm_w, w, 2, dims, strides, box))) return rc;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[2] = {64, 128};
    if ((rc = encode(&tm_h, gathered, 2, dims, strides, box))) return rc;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = bdlm::launch_scored_gather(hidden, mask, denoising, B, L, H, gathered, act,
                                             n_act, s);
  if (e == cudaSuccess)
    e = bdlm::launch_lm_conf(tm_w, tm_h, act, n_act, rows, rows, H, V, temperature, logits, part,
                             plan, st->err, s,
                             entropy_out != nullptr || rule == BDLM_COMMIT_ENTROPY_BOUNDED);
  if (e == cudaSuccess)
    e = bdlm::launch_lm_commit_finalize(mask, denoising, B, L, part, plan, temperature, rule, k,
                                        threshold, tok_out, conf_out, entropy_out, commit_out, s);
  return e == cudaSuccess ? BDLM_OK : BDLM_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------------------------ device-side round loop
struct bdlm_round_loop {
  bdlm_round_loop_desc d;
  int device = 0;
  void* scratch = nullptr;
  bdlm_bf16 *q_w = nullptr, *k_w = nullptr, *v_w = nullptr, *h_w = nullptr;
  bdlm_bf16* attn_out = nullptr;
  int32_t* tok = nullptr;
  float* conf = nullptr;
  uint8_t* com = nullptr;
  int* step = nullptr;
  cudaStream_t cap = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  unsigned gen = 0;
};

namespace {

// Sizes the library workspaces for one round of the loop (nothing may be allocated while the
// round is being captured).
int reserve_round(const bdlm_round_loop_desc& d) {
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st);
  if (rc) return rc;
  const bdlm_attn_desc& a = d.attn;
  const AttnPlan ap = bdlm::plan_attention(a.B, a.L, a.Hq, a.Hkv, a.max_pages_per_seq,
                                           a.page_size, st->num_sms);
  if (ap.n_mma == 0) return BDLM_ERR_UNSUPPORTED;
  const int R = a.B * a.L;
  const bdlm::LmConfPlan cp = bdlm::plan_lm_conf(R, d.H, d.V, st->num_sms);
  if (cp.max_row_tiles > cp.units) return BDLM_ERR_UNSUPPORTED;
  size_t data = ap.part_bytes;
  const size_t fused = lm_commit_layout(cp, R).total;
  if (fused > data) data = fused;
  if ((rc = ensure(reinterpret_cast<void**>(&st->attn_cnt), &st->attn_cnt_cap, ap.cnt_bytes,
                   true)))
    return rc;
  if ((rc = ensure(&st->data, &st->data_cap, data, false))) return rc;
  return get_encoder();
}

void drop_graph(bdlm_round_loop* lp) {
  if (lp->exec) cudaGraphExecDestroy(lp->exec);
  if (lp->graph) cudaGraphDestroy(lp->graph);
  lp->exec = nullptr;
  lp->graph = nullptr;
}

// Builds the graph: step counter := 0, then WHILE(condition) { one round }.
int capture_round_loop(bdlm_round_loop* lp) {
  const bdlm_round_loop_desc& d = lp->d;
  const bdlm_attn_desc& a = d.attn;
  const int R = a.B * a.L;
  int rc = reserve_round(d);
  if (rc) return rc;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    lp->gen = g_workspace_gen;
  }
  drop_graph(lp);
  if (cudaGraphCreate(&lp->graph, 0) != cudaSuccess) return BDLM_ERR_CUDA;
  cudaMemsetParams ms = {};
  ms.dst = lp->step;
  ms.value = 0;
  ms.elementSize = 4;
  ms.width = 1;
  ms.height = 1;
  cudaGraphNode_t init;
  if (cudaGraphAddMemsetNode(&init, lp->graph, nullptr, 0, &ms) != cudaSuccess) return BDLM_ERR_CUDA;
  cudaGraphConditionalHandle handle;
  if (cudaGraphConditionalHandleCreate(&handle, lp->graph, 1, cudaGraphCondAssignDefault) !=
      cudaSuccess)
    return BDLM_ERR_CUDA;
  cudaGraphNodeParams np = {};
  np.type = cudaGraphNodeTypeConditional;
  np.conditional.handle = handle;
  np.conditional.type = cudaGraphCondTypeWhile;
  np.conditional.size = 1;
  cudaGraphNode_t loop;
  if (cudaGraphAddNode(&loop, lp->graph, &init, nullptr, 1, &np) != cudaSuccess) return BDLM_ERR_CUDA;
  cudaGraph_t body = np.conditional.phGraph_out[0];
  if (cudaStreamBeginCaptureToGraph(lp->cap, body, nullptr, nullptr, 0,
                                    cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    return BDLM_ERR_CUDA;
  bdlm_stream s = lp->cap;
  bdlm::StepCopy c = {};
  c.src[0] = reinterpret_cast<const uint4*>(d.q_steps);
  c.dst[0] = reinterpret_cast<uint4*>(lp->q_w);
  c.n_vec[0] = static_cast<long long>(R) * a.Hq * a.D * 2 / 16;
  c.src[1] = reinterpret_cast<const uint4*>(d.k_new_steps);
  c.dst[1] = reinterpret_cast<uint4*>(lp->k_w);
  c.n_vec[1] = static_cast<long long>(R) * a.Hkv * a.D * 2 / 16;
  c.src[2] = reinterpret_cast<const uint4*>(d.v_new_steps);
  c.dst[2] = reinterpret_cast<uint4*>(lp->v_w);
  c.n_vec[2] = c.n_vec[1];
  c.src[3] = reinterpret_cast<const uint4*>(d.hidden_steps);
  c.dst[3] = reinterpret_cast<uint4*>(lp->h_w);
  c.n_vec[3] = static_cast<long long>(R) * d.H * 2 / 16;
  int r2 = BDLM_OK;
  if (bdlm::launch_select_step(c, lp->step, d.steps, lp->cap) != cudaSuccess) r2 = BDLM_ERR_CUDA;
  if (!r2) r2 = bdlm_block_attention_kv(&a, lp->q_w, lp->k_w, lp->v_w, d.k_pages, d.v_pages,
                                        d.page_table, d.prefix_lens, a.L, lp->attn_out, s);
  if (!r2) r2 = bdlm_lm_head_commit(lp->h_w, d.w, d.mask, d.denoising, a.B, a.L, d.H, d.V, d.rule,
                                    d.k, d.threshold, d.temperature, lp->tok, lp->conf, nullptr,
                                    lp->com, nullptr, s);
  if (!r2 && bdlm::launch_record_step(lp->step, d.steps, R, lp->tok, lp->conf, lp->com,
                                      d.tok_steps, d.conf_steps, d.commit_steps,
                                      reinterpret_cast<const uint4*>(lp->attn_out),
                                      reinterpret_cast<uint4*>(d.attn_out_steps),
                                      static_cast<long long>(R) * a.Hq * a.D * 2 / 16,
                                      lp->cap) != cudaSuccess)
    r2 = BDLM_ERR_CUDA;
  if (!r2) r2 = bdlm_apply_commit(d.mask, lp->com, R, s);
  if (!r2 && bdlm::launch_loop_condition(handle, d.mask, R, lp->step, d.steps, d.steps_done,
                                         lp->cap) != cudaSuccess)
    r2 = BDLM_ERR_CUDA;
  cudaGraph_t captured = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(lp->cap, &captured);
  if (r2) return r2;
  if (ec != cudaSuccess) return BDLM_ERR_CUDA;
  if (cudaGraphInstantiate(&lp->exec, lp->graph, 0) != cudaSuccess) return BDLM_ERR_CUDA;
  return BDLM_OK;
}

}  // namespace

extern "C" {

int bdlm_round_loop_create(const bdlm_round_loop_desc* desc, bdlm_round_loop** out) {
  if (!desc || !out) return BDLM_ERR_INVALID;
  *out = nullptr;
  const bdlm_round_loop_desc& d = *desc;
  const bdlm_attn_desc& a = d.attn;
  if (a.B < 1 || a.L < 1 || a.L > 64 || a.Hq < 1 || a.Hkv < 1 || a.Hq % a.Hkv != 0 ||
      a.D != 128 || a.page_size != 16 || a.max_pages_per_seq < 1 || a.num_pages < 1)
    return BDLM_ERR_INVALID;
  if (d.steps < 1 || d.H < 8 || d.H % 8 != 0 || d.V < 8 || d.V % 8 != 0) return BDLM_ERR_INVALID;
  if (!rule_ok(d.rule, d.k, d.threshold)) return BDLM_ERR_INVALID;
  if (!(d.temperature > 0.f) || !isfinite(d.temperature)) return BDLM_ERR_INVALID;
  if (!d.q_steps || !d.k_new_steps || !d.v_new_steps || !d.hidden_steps || !d.k_pages ||
      !d.v_pages || !d.page_table || !d.prefix_lens || !d.w || !d.mask || !d.tok_steps ||
      !d.conf_steps || !d.commit_steps || !d.steps_done)
    return BDLM_ERR_INVALID;
  if (d.attn_out_steps && !aligned16(d.attn_out_steps)) return BDLM_ERR_INVALID;
  const long long R = static_cast<long long>(a.B) * a.L;
  if (R * a.Hq > 0x7FFFFFFFll || R * d.V > (1ll << 40)) return BDLM_ERR_INVALID;
  auto* lp = new bdlm_round_loop();
  lp->d = d;
  cudaGetDevice(&lp->device);
  // owned scratch: one step's inputs, the attention output, this step's tok/conf/commit and
  // the step counter (the logits never leave the fused LM head)
  const size_t q_b = align256(R * a.Hq * a.D * 2), kv_b = align256(R * a.Hkv * a.D * 2);
  const size_t h_b = align256(R * d.H * 2);
  const size_t r4 = align256(R * 4), r1 = align256(R);
  const size_t total = 2 * q_b + 2 * kv_b + h_b + 2 * r4 + r1 + 256;
  if (cudaMalloc(&lp->scratch, total) != cudaSuccess) {
    delete lp;
    return BDLM_ERR_NOMEM;
  }
  uint8_t* p = static_cast<uint8_t*>(lp->scratch);
  lp->q_w = reinterpret_cast<bdlm_bf16*>(p);      p += q_b;
  lp->attn_out = reinterpret_cast<bdlm_bf16*>(p); p += q_b;
  lp->k_w = reinterpret_cast<bdlm_bf16*>(p);      p += kv_b;
  lp->v_w = reinterpret_cast<bdlm_bf16*>(p);      p += kv_b;
  lp->h_w = reinterpret_cast<bdlm_bf16*>(p);      p += h_b;
  lp->tok = reinterpret_cast<int32_t*>(p);        p += r4;
  lp->conf = reinterpret_cast<float*>(p);         p += r4;
  lp->com = p;                                    p += r1;
  lp->step = reinterpret_cast<int*>(p);
  if (cudaStreamCreateWithFlags(&lp->cap, cudaStreamNonBlocking) != cudaSuccess) {
    cudaFree(lp->scratch);
    delete lp;
    return BDLM_ERR_CUDA;
  }
  const int rc = capture_round_loop(lp);
  if (rc) {
    bdlm_round_loop_destroy(lp);
    return rc;
  }
  *out = lp;
  return BDLM_OK;
}

int bdlm_round_loop_launch(bdlm_round_loop* loop, bdlm_stream stream) {
  if (!loop) return BDLM_ERR_INVALID;
  unsigned gen = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    gen = g_workspace_gen;
  }
  if (gen != loop->gen || !loop->exec) {
    const int rc = capture_round_loop(loop);  // a workspace moved since the capture
    if (rc) return rc;
  }
  return cudaGraphLaunch(loop->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? BDLM_OK
             : BDLM_ERR_CUDA;
}

int bdlm_round_loop_destroy(bdlm_round_loop* loop) {
  if (!loop) return BDLM_OK;
  drop_graph(loop);
  if (loop->cap) cudaStreamDestroy(loop->cap);
  if (loop->scratch) cudaFree(loop->scratch);
  delete loop;
  return BDLM_OK;
}

}  // extern "C"
