/*
 * bdlm — one denoising round of block-diffusion LLM decoding on NVIDIA GB300 (sm_103a).
 *
 * A round (JetEngine README, "Block Diffusion Decoding"; JetEngine notes (CLAUDE.md),
 * "Important Patterns"): every sequence of a batch holds a committed prefix in a paged
 * KV cache and a block of L positions (L = 1..64), some of which are still masked.  One
 * round runs block attention, the LM head for the rows still being denoised, and the
 * confidence commit that unmasks positions; the caller then clears the committed
 * positions from the mask (bdlm_apply_commit) and runs the next round.
 *
 * Conventions shared by every call:
 *  - Pointers are DEVICE pointers on the current CUDA device, owned by the caller, unless
 *    a parameter says otherwise.  bf16 data are raw bfloat16 bits (bdlm_bf16).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream).  A call validates its host-side arguments and returns before any launch on
 *    error.  Faults inside a kernel surface at the caller's next synchronisation.
 *  - Kernels never trust device-resident indices: a page id outside [0, num_pages), a
 *    prefix length that does not fit the page table, or an out-of-range row index is
 *    skipped (zero data / no write) and recorded in a device error word that
 *    bdlm_device_error() reads and clears.  Every wait inside a kernel is bounded; a
 *    wait that gives up is recorded the same way.
 *  - Scratch (split-KV and commit partial results, scheduler counters, the gathered LM-head rows)
 *    lives in a per-device workspace that the library allocates on first need and grows
 *    when a larger problem arrives (growing synchronises the device).  Calls that share
 *    a device must not run concurrently on different streams: they share that
 *    workspace.  bdlm_release() frees it.
 *  - Return value: BDLM_OK (0) or a negative BDLM_ERR_* code; bdlm_status_string() names it.
 */
#ifndef BDLM_H
#define BDLM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t bdlm_bf16;  /* raw bfloat16 bits */
typedef void* bdlm_stream;   /* cudaStream_t */

enum {
  BDLM_OK = 0,
  BDLM_ERR_INVALID = -1,     /* bad shape, null pointer, parameter out of range */
  BDLM_ERR_CUDA = -2,        /* a CUDA runtime call or launch failed */
  BDLM_ERR_UNSUPPORTED = -3, /* no sm_103 device, or a shape outside the kernels' limits */
  BDLM_ERR_NOMEM = -4        /* the workspace could not be allocated */
};

/* Device error word bits (bdlm_device_error). */
enum {
  BDLM_DEVERR_PAGE = 1,      /* page id outside [0, num_pages): that page read as zeros */
  BDLM_DEVERR_LENGTH = 2,    /* prefix_len < 0 or prefix_len + L > max_pages_per_seq*P */
  BDLM_DEVERR_TIMEOUT = 4,   /* a bounded wait inside a kernel gave up */
  BDLM_DEVERR_ROW = 8        /* an active row index outside [0, n_rows) was skipped */
};

/*
 * Shapes of block attention.
 *   B                   sequences in the batch
 *   L                   block length (1..64)
 *   Hq, Hkv             query / KV heads; Hq % Hkv == 0, Hq/Hkv <= 16
 *   D                   head dimension; must be 128
 *   page_size           tokens per KV page; must be 16
 *   max_pages_per_seq   columns of page_table
 *   num_pages           pages in the K and V pools
 *   sm_scale            softmax scale; <= 0 selects 1/sqrt(D)
 */
typedef struct {
  int B, L, Hq, Hkv, D, page_size, max_pages_per_seq, num_pages;
  float sm_scale;
} bdlm_attn_desc;

/*
 * Block attention of one denoising round over the paged KV cache.
 * Source: JetEngine notes, "ModelRunner" (paged-KV attention for denoise; the pages'
 * engines use FlashAttention-3 / flashinfer for it) and "Important Patterns" (a block of
 * L positions on top of the committed prefix); dlmrt page, "Highlights" (every forward
 * denoises a whole block).
 *
 * For sequence b, block position i and query head h, with kv_len = prefix_lens[b] + L:
 *     out[b,i,h,:] = softmax_j( sm_scale * q[b,i,h,:] . K_b[j, g(h), :] ) V_b[j, g(h), :]
 * over j = 0..kv_len-1: the whole prefix plus the whole block (bidirectional inside the
 * block), g(h) = h / (Hq/Hkv) (grouped-query attention).  Token j of sequence b is slot
 * j % page_size of page page_table[b][j / page_size]; the block's own K/V must already
 * sit at positions prefix_len .. prefix_len+L-1.
 *
 * Layouts (row-major, contiguous):
 *   q            [B, L, Hq, D]                         bf16
 *   k_pages      [num_pages, page_size, Hkv, D]        bf16 (16-byte aligned)
 *   v_pages      [num_pages, page_size, Hkv, D]        bf16 (16-byte aligned)
 *   page_table   [B, max_pages_per_seq]                int32 (unused entries are ignored)
 *   prefix_lens  [B]                                   int32
 *   out          [B, L, Hq, D]                         bf16 (16-byte aligned; fp32
 *                                                      accumulation, one rounding)
 * `L` must equal desc->L (it is the block length of this round).
 * Slots past kv_len in a sequence's last page are never used, whatever they hold.
 */
int bdlm_block_attention(const bdlm_attn_desc* desc, const bdlm_bf16* q,
                         const bdlm_bf16* k_pages, const bdlm_bf16* v_pages,
                         const int32_t* page_table, const int32_t* prefix_lens, int L,
                         bdlm_bf16* out, bdlm_stream stream);

/*
 * Block attention with the block's K/V-cache write fused in: the block's new K/V are written
 * into the paged cache and attended to by the same kernel, with no separate write launch.
 * Source: JetEngine notes, "Optimization History" (opt24: the KV-cache write of the block
 * combined with the paged attention in one kernel) and "Current Profile (H200, bs=128, opt24)".
 *
 * Results as bdlm_write_block_kv followed by bdlm_block_attention: k_new, v_new [B, L, Hkv, D]
 * bf16 (16-byte aligned) go to the slots prefix_lens[b] .. prefix_lens[b]+L-1 of sequence b,
 * and out is the block attention over the updated cache.  Inside the kernel, every work item
 * that reads one of the block's tokens first stores that token's new K (or V) row into its page
 * slot and then loads its tile; items that share tokens (query-row groups) store identical
 * bytes.  A page id outside [0, num_pages) or a prefix length that does not fit the page table
 * skips the writes it concerns and sets a device error bit, as the unfused calls do.  Other
 * arguments, layouts and limits as bdlm_block_attention; k_pages and v_pages are written.
 */
int bdlm_block_attention_kv(const bdlm_attn_desc* desc, const bdlm_bf16* q,
                            const bdlm_bf16* k_new, const bdlm_bf16* v_new, bdlm_bf16* k_pages,
                            bdlm_bf16* v_pages, const int32_t* page_table,
                            const int32_t* prefix_lens, int L, bdlm_bf16* out,
                            bdlm_stream stream);

/*
 * Block prefill: the prompt's K/V written into the cache and block-causal attention over the
 * prompt, so that the rounds that follow find the prompt in the paged cache.
 * Source: JetEngine notes, "Kernels" (block prefill attention and the KV-cache store) and
 * "ModelRunner" (prefill and denoise have different attention patterns); SDAR page, "What is
 * SDAR?" (autoregression across blocks, diffusion inside a block).
 *
 * The prompt of sequence b is prompt_len tokens (a multiple of desc->L, the block length),
 * placed after prefix_lens[b] tokens already in the cache (0 for a fresh prompt).  Token t of
 * the prompt, in prompt block j = t / L, attends to every cached token before the prompt,
 * every prompt token of blocks before j and every token of block j:
 *     out[b,t,h,:] = softmax_k(sm_scale * q[b,t,h,:] . K_b[k]) V_b[k],
 *                    k < prefix_lens[b] + (j+1) * L,  KV head as bdlm_block_attention.
 * Layouts: q, out [B, prompt_len, Hq, D]; k_new, v_new [B, prompt_len, Hkv, D] (written to
 * the slots prefix_lens[b] .. + prompt_len - 1); pools, page_table, prefix_lens as
 * bdlm_block_attention; prefix_lens[b] + prompt_len must fit the page table.  bf16 pointers
 * 16-byte aligned.  Runs as the K/V write followed by the block attention over chunks of Lq
 * prompt tokens (the largest multiple of L dividing prompt_len with Lq * Hq / Hkv <= 256 query
 * rows, or L), each chunk reading the K/V before its end once with the block-causal mask
 * applied inside it; the chunks share their sequence's page-table row.
 */
int bdlm_prefill_attention(const bdlm_attn_desc* desc, int prompt_len, const bdlm_bf16* q,
                           const bdlm_bf16* k_new, const bdlm_bf16* v_new, bdlm_bf16* k_pages,
                           bdlm_bf16* v_pages, const int32_t* page_table,
                           const int32_t* prefix_lens, bdlm_bf16* out, bdlm_stream stream);

/*
 * Selective LM head.
 * Source: JetEngine notes, "ModelRunner" (selective logits: the LM head runs only for
 * DENOISING sequences) and "Optimization History" (opt23: LM head only on masked rows).
 *
 *     logits[r, v] = sum_k hidden[r, k] * w[v, k]     for r in active_idx, v in [0, V)
 *
 * Layouts: hidden [n_rows, H] bf16; w [V, H] bf16 (one vocabulary row per output);
 * active_idx [n_active] int32 (distinct row ids in [0, n_rows)); logits [n_rows, V] bf16.
 * Only the active rows of `logits` are written (fp32 accumulation, one round-to-nearest-
 * even to bf16); other rows keep whatever they held.  H % 8 == 0, V % 8 == 0
 * (16-byte row alignment).  n_active == 0 is a no-op.
 */
int bdlm_lm_head(const bdlm_bf16* hidden, const bdlm_bf16* w, const int32_t* active_idx,
                 int n_active, int n_rows, int H, int V, bdlm_bf16* logits, bdlm_stream stream);

/*
 * bdlm_lm_head with the active-row count in device memory, for rounds that run without the
 * host (the count comes from bdlm_active_rows).  The launch is planned for max_active rows
 * (0 < max_active <= n_rows); *n_active_dev (int32, device, read when the kernels run) is
 * clamped to [0, max_active], and only that many leading entries of active_idx are used.
 * Otherwise as bdlm_lm_head.
 */
int bdlm_lm_head_device_count(const bdlm_bf16* hidden, const bdlm_bf16* w,
                              const int32_t* active_idx, const int32_t* n_active_dev,
                              int max_active, int n_rows, int H, int V, bdlm_bf16* logits,
                              bdlm_stream stream);

/*
 * The rows a step's LM head must compute, on the device.
 * Source: JetEngine notes, "ModelRunner" (selective logits: DENOISING sequences only) and
 * "Optimization History" (opt23: only the still-masked rows).
 *
 * Row r = b*L + i is active when mask[r] != 0 and (denoising is NULL or denoising[b] != 0).
 * active_idx [B*L] int32 receives the active rows in increasing order; *n_active_dev (int32,
 * device) their number.  mask [B, L] uint8; denoising [B] uint8 or NULL.  1 <= L <= 64.
 */
int bdlm_active_rows(const uint8_t* mask, const uint8_t* denoising, int B, int L,
                     int32_t* active_idx, int32_t* n_active_dev, bdlm_stream stream);

/*
 * Writes a block's new K/V into the paged cache: k_new, v_new [B, L, Hkv, D] bf16 go to the
 * slots prefix_lens[b] .. prefix_lens[b]+L-1 of sequence b (token j in page
 * page_table[b][j / page_size], slot j % page_size), the slots bdlm_block_attention reads the
 * block's own K/V from.  Used every step while the block is denoised and once more after it
 * is fully committed (the SAVING pass).
 * Source: JetEngine notes, "Important Patterns" and "Optimization History" (opt18/opt24: the
 * KV-cache write of the block combined with the paged attention).
 * desc as bdlm_block_attention (Hq and sm_scale unused); all pointers device, 16-byte aligned
 * k_new/v_new/k_pages/v_pages.  A page id outside [0, num_pages) or a length that does not fit
 * the page table skips the rows it concerns and sets a device error bit.
 */
int bdlm_write_block_kv(const bdlm_attn_desc* desc, const bdlm_bf16* k_new,
                        const bdlm_bf16* v_new, bdlm_bf16* k_pages, bdlm_bf16* v_pages,
                        const int32_t* page_table, const int32_t* prefix_lens, bdlm_stream stream);

/*
 * Confidence and commit of one denoising step (threshold / low_confidence_dynamic rule).
 * Source: JetEngine notes, "Remasking Strategies" (low_confidence_dynamic: unmask above a
 * threshold); dInfer blog, "Algorithmic Innovations" (threshold decoding); SDAR page,
 * "Reported Performance" (dynamic decoding); JetEngine README, example `SamplingParams`
 * (temperature, dynamic_threshold).
 *
 * For each masked position (mask[b,i] != 0), from logits row b*L+i, in one pass:
 *     tok_out[b,i]  = argmax_v logits[v]              (lowest index on ties)
 *     conf_out[b,i] = 1 / sum_v exp((logits[v] - max) / temperature)   (max probability)
 * Then per block b: commit_out[b,i] = 1 for every masked i with conf >= threshold; if no
 * masked position reaches the threshold and the block has one, the single most confident
 * masked position is committed (lowest i on ties).  Confidences are compared as float32.
 * Unmasked positions get tok_out = -1, conf_out = -inf, commit_out = 0; their logits rows
 * are never read.
 *
 * Layouts: logits [B*L, V] bf16 (finite in masked rows); mask, commit_out [B, L] uint8;
 * tok_out [B, L] int32; conf_out [B, L] float.  1 <= L <= 64; V >= 1.
 * temperature > 0; 0 <= threshold <= 1.
 */
int bdlm_confidence_commit(const bdlm_bf16* logits, const uint8_t* mask, int B, int L, int V,
                           float threshold, float temperature, int32_t* tok_out,
                           float* conf_out, uint8_t* commit_out, bdlm_stream stream);

/* Commit rules of bdlm_confidence_commit_rule. */
enum {
  BDLM_COMMIT_THRESHOLD = 0,       /* low_confidence_dynamic: as bdlm_confidence_commit */
  BDLM_COMMIT_TOPK = 1,            /* low_confidence_static: the k most confident */
  BDLM_COMMIT_SEQUENTIAL = 2,      /* the k leftmost masked positions */
  BDLM_COMMIT_ANTI_SEQUENTIAL = 3, /* the k rightmost masked positions */
  BDLM_COMMIT_ENTROPY_BOUNDED = 4  /* lowest entropies first, within an entropy budget */
};

/*
 * Confidence, entropy and commit with a selectable rule.
 * Source: JetEngine notes, "Remasking Strategies" (sequential: unmask left to right;
 * low_confidence_static: unmask the top-k by confidence; low_confidence_dynamic: unmask above
 * a threshold; entropy_bounded: unmask by a cumulative entropy budget; anti_sequential is named
 * beside sequential in the notes' scheduler tree) and "Key Config Parameters" (eb_threshold).
 *
 * tok_out and conf_out are those of bdlm_confidence_commit for every rule.  entropy_out [B, L]
 * float (device, or NULL when not wanted) receives, for every masked position, the entropy in
 * nats of its softmax at temperature T,
 *     H = -sum_v p_v ln p_v,   p_v = exp((l_v - max) / T) / sum_u exp((l_u - max) / T),
 * computed in the same pass; unmasked positions get +inf.  Per block:
 *   BDLM_COMMIT_THRESHOLD        exactly bdlm_confidence_commit (k ignored);
 *   BDLM_COMMIT_TOPK             the min(k, masked) masked positions of highest confidence
 *                                (compared as float32; lower position first among equals);
 *   BDLM_COMMIT_SEQUENTIAL       the min(k, masked) leftmost masked positions;
 *   BDLM_COMMIT_ANTI_SEQUENTIAL  the min(k, masked) rightmost masked positions;
 *   BDLM_COMMIT_ENTROPY_BOUNDED  the masked positions in increasing order of entropy (lower
 *                                position first among equals), as long as the running float32
 *                                sum of their entropies, added in that order, stays <= threshold
 *                                (the entropy budget, eb_threshold, in nats); at least one.
 * k >= 1 for the top-k and sequential rules (e.g. L / denoising steps); 0 <= threshold <= 1 for
 * the threshold rule; a finite threshold >= 0 for the entropy rule.  Layouts, limits and errors
 * as bdlm_confidence_commit; an unknown rule or an argument out of its range returns
 * BDLM_ERR_INVALID.  Scratch (the partial results) comes from the library workspace.
 */
int bdlm_confidence_commit_rule(const bdlm_bf16* logits, const uint8_t* mask, int B, int L, int V,
                                int rule, int k, float threshold, float temperature,
                                int32_t* tok_out, float* conf_out, float* entropy_out,
                                uint8_t* commit_out, bdlm_stream stream);

/*
 * bdlm_confidence_commit without any device allocation (the pages have no counterpart of
 * this entry point; it exists for callers that cannot let the library allocate: an engine
 * that reserved the GPU's memory up front for its own pools, or a latency-critical loop that
 * cannot afford an allocation's implicit synchronisation).
 *
 * Same arguments, layouts and results as bdlm_confidence_commit.  Its scratch lives in a
 * fixed device array of about 96 KiB inside the library, resident on every GPU that loads
 * it until the process exits; nothing is allocated or freed per call.
 *  - Limits: B*L <= 2048 and V <= 262144; larger problems return BDLM_ERR_UNSUPPORTED
 *    before any launch.
 *  - The first call on a device looks up the array's address with that device current;
 *    make that first call before any stream capture.
 *  - All calls share the array, which keeps the last call's contents; calls that overlap on
 *    the GPU race.
 *  - A device error of this call (a bounded wait inside a kernel that gave up) is recorded
 *    in an error word at the head of the array; bdlm_device_error() reads and clears it
 *    (it allocates nothing either).  The calls themselves never clear it.
 */
int bdlm_confidence_commit_noalloc(const bdlm_bf16* logits, const uint8_t* mask, int B, int L,
                                   int V, float threshold, float temperature, int32_t* tok_out,
                                   float* conf_out, uint8_t* commit_out, bdlm_stream stream);

/*
 * Selective LM head fused with the confidence and commit step: the logits of a step's scored
 * rows are reduced to (token, confidence) as they leave the tensor cores, so they never have
 * to be stored and read back.
 * Source: JetEngine notes, "ModelRunner" (selective logits for DENOISING sequences),
 * "Optimization History" (opt23: LM head only on masked rows) and "Remaining Optimization
 * Avenues" (a fused postprocess kernel); the rules as bdlm_confidence_commit_rule.
 *
 * Scored rows: r = b*L + i with mask[r] != 0 and (denoising NULL or denoising[b] != 0), the
 * rows bdlm_active_rows lists.  For each scored row the results are those of
 *     bdlm_lm_head (hidden, w, scored rows) followed by bdlm_confidence_commit_rule (rule, k,
 *     threshold, temperature) over those bf16 logits,
 * with `mask` restricted to the scored rows: tok_out is the argmax of the row's bf16-rounded
 * logits (lowest index on ties), conf_out its max probability (the same value up to float32
 * summation order), and each block commits among its scored positions by the rule.  Positions
 * that are not scored (unmasked, or in a SAVING sequence) get tok_out = -1, conf_out = -inf,
 * entropy_out = +inf, commit_out = 0.  entropy_out (NULL when not wanted) receives the scored
 * positions' entropies as bdlm_confidence_commit_rule defines them, from the same bf16 logits.
 *
 * Layouts: hidden [B*L, H] bf16 (row b*L+i); w [V, H] bf16; mask [B, L] uint8; denoising [B]
 * uint8 or NULL; tok_out [B, L] int32; conf_out, entropy_out [B, L] float; commit_out [B, L]
 * uint8; logits
 * [B*L, V] bf16 or NULL: when given, the scored rows' logits are stored as bdlm_lm_head would
 * store them (other rows untouched).  H % 8 == 0, V % 8 == 0, 1 <= L <= 64,
 * B*L <= 256 * (SM count); temperature > 0; rule arguments as bdlm_confidence_commit_rule.
 * Scratch (the scored-row list, gathered rows, partials) comes from the library workspace.
 */
int bdlm_lm_head_commit(const bdlm_bf16* hidden, const bdlm_bf16* w, const uint8_t* mask,
                        const uint8_t* denoising, int B, int L, int H, int V, int rule, int k,
                        float threshold, float temperature, int32_t* tok_out, float* conf_out,
                        float* entropy_out, uint8_t* commit_out, bdlm_bf16* logits,
                        bdlm_stream stream);

/*
 * Mask update between denoising steps: mask[i] = 0 wherever commit[i] != 0.
 * Source: JetEngine notes, "Important Patterns" (each denoising step moves positions from
 * masked to unmasked).  mask, commit: [n] uint8.  n == 0 is a no-op.
 */
int bdlm_apply_commit(uint8_t* mask, const uint8_t* commit, int n, bdlm_stream stream);

/*
 * A whole block's denoising on the device: rounds repeat inside one CUDA graph, with a
 * conditional WHILE node, until no position of any block is masked or `steps` rounds have
 * run; the host only launches the graph.
 * Source: dlmrt page, "Highlights" (a block = one CUDA graph with WHILE(not done){round});
 * JetEngine notes, "Important Patterns" (denoising steps until the block is committed).
 *
 * One round (step s, counted on the device):
 *   the step's inputs: slice s of q_steps [S, B, L, Hq, D], k_new_steps / v_new_steps
 *   [S, B, L, Hkv, D] and hidden_steps [S, B*L, H] (the model's outputs for that step, which
 *   this library does not compute) -> bdlm_block_attention_kv (the block's K/V written into the
 *   cache and attended in one kernel) -> bdlm_lm_head_commit (mask, denoising, rule, k, threshold,
 *   temperature; no logits stored) -> tok/conf/commit stored into slice s of tok_steps,
 *   conf_steps, commit_steps [S, B, L] -> bdlm_apply_commit on mask.
 * After the last round *steps_done holds the number of rounds run, and slices at or past it
 * are untouched.  The attention output is kept in the loop's own scratch (a model would feed
 * it to its next layer); when attn_out_steps [S, B, L, Hq, D] bf16 is given, each round also
 * copies it into slice s.
 *
 * All pointers are device pointers owned by the caller and must stay valid while the loop
 * exists.  bdlm_round_loop_create allocates the loop's scratch (one step's inputs, the
 * attention output, small per-row arrays) and captures the graph; it sizes
 * the library workspace first, since nothing may be allocated inside the capture.  If a later
 * call grows or releases the library workspace, the next launch captures the graph again.
 * Shapes and limits as the calls it is made of.
 */
typedef struct bdlm_round_loop bdlm_round_loop;
typedef struct {
  bdlm_attn_desc attn;        /* B, L, Hq, Hkv, D, page_size, max_pages_per_seq, num_pages */
  int steps;                  /* S: rounds at most, and slices of the per-step arrays */
  int H, V;                   /* LM head */
  int rule, k;                /* BDLM_COMMIT_* and positions per block (see _rule) */
  float threshold, temperature;
  const bdlm_bf16* q_steps;
  const bdlm_bf16* k_new_steps;
  const bdlm_bf16* v_new_steps;
  const bdlm_bf16* hidden_steps;
  bdlm_bf16* k_pages;
  bdlm_bf16* v_pages;
  const int32_t* page_table;
  const int32_t* prefix_lens;
  const bdlm_bf16* w;         /* [V, H] */
  uint8_t* mask;              /* [B, L], updated in place */
  const uint8_t* denoising;   /* [B] or NULL */
  int32_t* tok_steps;
  float* conf_steps;
  uint8_t* commit_steps;
  int32_t* steps_done;        /* one int32 */
  bdlm_bf16* attn_out_steps;  /* [S, B, L, Hq, D] or NULL */
} bdlm_round_loop_desc;

int bdlm_round_loop_create(const bdlm_round_loop_desc* desc, bdlm_round_loop** loop_out);
/* Enqueues the whole loop on `stream` (asynchronous; one graph launch). */
int bdlm_round_loop_launch(bdlm_round_loop* loop, bdlm_stream stream);
/* Frees the loop (the device must be done with it). */
int bdlm_round_loop_destroy(bdlm_round_loop* loop);

/* Human-readable name of a BDLM_* status code (a static string). */
const char* bdlm_status_string(int status);

/*
 * Reads and clears the device error words of the current device (BDLM_DEVERR_* bits) into
 * *bits_out (a HOST pointer): the workspace's word, written by every call except
 * bdlm_confidence_commit_noalloc, ORed with the word of that call's fixed array.  Allocates
 * nothing (a word that no call has set up yet reads as 0).  Synchronises the device.
 * Returns BDLM_OK or an error.
 */
int bdlm_device_error(int* bits_out);

/*
 * Self-test of the failure path every kernel shares: launches one CTA whose thread waits,
 * through the same bounded wait the kernels use, on an mbarrier that nothing ever arrives on.
 * The wait gives up after limit_us microseconds (1 .. 2,000,000) and the kernel records
 * BDLM_DEVERR_TIMEOUT in the device error word, as a kernel whose wait runs out does; it
 * faults nothing, so the context stays usable and bdlm_device_error() then reports the bit.
 * Asynchronous on `stream`.  Returns BDLM_OK, BDLM_ERR_INVALID for a limit out of range, or
 * an error of the device setup.
 */
int bdlm_selftest_wait_timeout(int limit_us, bdlm_stream stream);

/* Frees the workspace of the current device.  The device must be idle. */
int bdlm_release(void);

#ifdef __cplusplus
}
#endif

#endif /* BDLM_H */
