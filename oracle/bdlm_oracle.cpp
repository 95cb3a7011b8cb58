// Oracle for one block-diffusion denoising round: plain fp64 CPU code.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU
// baseline call this file.  It shares no code, header, table or helper with the CUDA
// library, and the product path never loads it.
//
// Every value is computed from its definition, in fp64, with plain loops (OpenMP over
// independent sequences / rows only; no blocking, no fusion, no reordering of a sum
// beyond the definition's own order).  bf16 inputs are raw uint16 bits, widened exactly.
//
// Sources (page title, section):
//  * JetEngine README, "Block Diffusion Decoding" and JetEngine notes (CLAUDE.md),
//    "Important Patterns": a block of L positions is denoised on top of a committed prefix.
//  * JetEngine notes, "ModelRunner" and "Optimization History" (opt18, opt24): denoise
//    attention runs over a paged KV cache (block table per sequence).
//  * JetEngine notes, "ModelRunner": selective logits, LM head only for DENOISING rows.
//  * JetEngine notes, "Remasking Strategies" (low_confidence_dynamic), dInfer blog
//    "Algorithmic Innovations" (threshold decoding), SDAR page "Reported Performance"
//    (dynamic decoding): commit every masked position whose confidence clears a threshold.
// Readings where the pages are silent are listed beside each function.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

double bf16_to_f64(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, sizeof(f));
    return static_cast<double>(f);
}

}  // namespace

extern "C" {

// Block attention of one denoising round over a paged KV cache.
//
// For sequence b, block position i (0..L-1) and query head h:
//     kv_len = prefix_lens[b] + L
//     s_j    = sm_scale * sum_d q[b,i,h,d] * K_b[j, h/(Hq/Hkv), d]      j = 0..kv_len-1
//     o      = sum_j exp(s_j - max_j s) V_b[j, ...] / sum_j exp(s_j - max_j s)
// where token j of sequence b lives in page page_table[b][j / P], slot j % P.
// Readings: the block's own K/V sit at slots prefix_len .. prefix_len+L-1; the block
// attends to every prefix token and to all of its own tokens (bidirectional inside the
// block, nothing of later blocks exists); query head h uses KV head h / (Hq/Hkv).
// Layouts: q [B,L,Hq,D]; k_pages, v_pages [num_pages,P,Hkv,D]; page_table [B,max_pages];
// out [B,L,Hq,D] fp64.  seq_list (n_seq entries) selects the sequences computed; NULL
// computes all B.  Returns 0, or -1 on an argument error (including a negative prefix or a
// page id of a needed token outside [0, num_pages): that sequence is left untouched).
int oracle_block_attention(int B, int L, int Hq, int Hkv, int D, int P, int max_pages,
                           int num_pages, const uint16_t* q, const uint16_t* k_pages,
                           const uint16_t* v_pages, const int32_t* page_table,
                           const int32_t* prefix_lens, double sm_scale, const int32_t* seq_list,
                           int n_seq, double* out) {
    if (B < 0 || L <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0 || Hq % Hkv != 0) return -1;
    const int G = Hq / Hkv;
    const int count = seq_list ? n_seq : B;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) collapse(2) reduction(| : bad)
    for (int sidx = 0; sidx < count; ++sidx) {
        for (int h = 0; h < Hq; ++h) {
            const int b = seq_list ? seq_list[sidx] : sidx;
            const long kv_len = static_cast<long>(prefix_lens[b]) + L;
            if (prefix_lens[b] < 0 || kv_len > static_cast<long>(max_pages) * P) {
                bad = 1;
                continue;
            }
            int bad_page = 0;
            for (long pg = 0; pg < (kv_len + P - 1) / P; ++pg) {
                const long id = page_table[static_cast<long>(b) * max_pages + pg];
                if (id < 0 || id >= num_pages) bad_page = 1;
            }
            if (bad_page) { bad = 1; continue; }
            const int kvh = h / G;
            std::vector<double> kk(static_cast<size_t>(kv_len) * D), vv(static_cast<size_t>(kv_len) * D);
            for (long j = 0; j < kv_len; ++j) {
                const long page = page_table[static_cast<long>(b) * max_pages + j / P];
                const long slot = j % P;
                const size_t base = ((static_cast<size_t>(page) * P + slot) * Hkv + kvh) * D;
                for (int d = 0; d < D; ++d) {
                    kk[static_cast<size_t>(j) * D + d] = bf16_to_f64(k_pages[base + d]);
                    vv[static_cast<size_t>(j) * D + d] = bf16_to_f64(v_pages[base + d]);
                }
            }
            std::vector<double> s(static_cast<size_t>(kv_len));
            for (int i = 0; i < L; ++i) {
                const size_t qb = ((static_cast<size_t>(b) * L + i) * Hq + h) * D;
                double smax = -std::numeric_limits<double>::infinity();
                for (long j = 0; j < kv_len; ++j) {
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += bf16_to_f64(q[qb + d]) * kk[static_cast<size_t>(j) * D + d];
                    s[j] = dot * sm_scale;
                    if (s[j] > smax) smax = s[j];
                }
                double z = 0.0;
                for (long j = 0; j < kv_len; ++j) {
                    s[j] = std::exp(s[j] - smax);
                    z += s[j];
                }
                double* o = out + qb;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (long j = 0; j < kv_len; ++j) {
                    const double p = s[j] / z;
                    for (int d = 0; d < D; ++d) o[d] += p * vv[static_cast<size_t>(j) * D + d];
                }
            }
        }
    }
    return bad ? -1 : 0;
}

// Softmax weights of one (sequence, position, head) of the attention above, written to
// probs[0..kv_len-1]; used to check that each row sums to one.
int oracle_attention_probs(int L, int Hq, int Hkv, int D, int P, int max_pages, int num_pages,
                           const uint16_t* q, const uint16_t* k_pages, const int32_t* page_table,
                           const int32_t* prefix_lens, double sm_scale, int b, int i, int h,
                           double* probs) {
    if (Hq % Hkv != 0) return -1;
    const int kvh = h / (Hq / Hkv);
    const long kv_len = static_cast<long>(prefix_lens[b]) + L;
    if (prefix_lens[b] < 0 || kv_len > static_cast<long>(max_pages) * P) return -1;
    for (long pg = 0; pg < (kv_len + P - 1) / P; ++pg) {
        const long id = page_table[static_cast<long>(b) * max_pages + pg];
        if (id < 0 || id >= num_pages) return -1;
    }
    const size_t qb = ((static_cast<size_t>(b) * L + i) * Hq + h) * D;
    double smax = -std::numeric_limits<double>::infinity();
    for (long j = 0; j < kv_len; ++j) {
        const long page = page_table[static_cast<long>(b) * max_pages + j / P];
        const size_t base = ((static_cast<size_t>(page) * P + j % P) * Hkv + kvh) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_f64(q[qb + d]) * bf16_to_f64(k_pages[base + d]);
        probs[j] = dot * sm_scale;
        if (probs[j] > smax) smax = probs[j];
    }
    double z = 0.0;
    for (long j = 0; j < kv_len; ++j) { probs[j] = std::exp(probs[j] - smax); z += probs[j]; }
    for (long j = 0; j < kv_len; ++j) probs[j] /= z;
    return 0;
}

// Selective LM head: logits[r, v] = sum_k hidden[r, k] * W[v, k] for the selected rows.
// Reading: W is stored [V, H] (one vocabulary row per output); rows are the DENOISING
// rows the caller lists (JetEngine notes, "ModelRunner": selective logits).
// rows (n_sel_rows), cols (n_sel_cols; NULL = all V) select what is computed;
// out is [n_sel_rows, n_sel_cols] fp64.
int oracle_lm_head(int n_rows, int H, int V, const uint16_t* hidden, const uint16_t* w,
                   const int32_t* rows, int n_sel_rows, const int32_t* cols, int n_sel_cols,
                   double* out) {
    if (H <= 0 || V <= 0) return -1;
    const int nc = cols ? n_sel_cols : V;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int ri = 0; ri < n_sel_rows; ++ri) {
        const int r = rows[ri];
        if (r < 0 || r >= n_rows) { bad = 1; continue; }
        std::vector<double> hrow(H);
        for (int k = 0; k < H; ++k) hrow[k] = bf16_to_f64(hidden[static_cast<size_t>(r) * H + k]);
        for (int ci = 0; ci < nc; ++ci) {
            const int v = cols ? cols[ci] : ci;
            double acc = 0.0;
            const uint16_t* wr = w + static_cast<size_t>(v) * H;
            for (int k = 0; k < H; ++k) acc += hrow[k] * bf16_to_f64(wr[k]);
            out[static_cast<size_t>(ri) * nc + ci] = acc;
        }
    }
    return bad ? -1 : 0;
}

// Confidence and commit of one denoising step.
//
// For every masked position i of block b, from row b*L+i of the logits:
//     tok  = argmax_v l_v                (first index of the maximum)
//     m    = l_tok
//     conf = 1 / sum_v exp((l_v - m) / T)   (the largest softmax probability at temperature T)
// Unmasked positions give tok = -1, conf = -inf, commit = 0.  Per block, by rule
// (JetEngine notes, "Remasking Strategies"):
//   0 threshold (low_confidence_dynamic): commit = { masked i : conf_i >= threshold }; if that
//     set is empty and the block has a masked position, the single most confident masked i
//     (lowest i on ties).  Readings: "at or above"; the fallback commits the most confident
//     position (the notes fall back to left-to-right order instead).
//   1 top-k (low_confidence_static): the k masked positions of highest confidence (lowest i
//     first among equal confidences), or every masked position if there are fewer than k.
//   2 sequential: the k leftmost masked positions (left-to-right unmasking).
//   3 anti-sequential: the k rightmost masked positions.
//   4 entropy-bounded (entropy_bounded, budget eb_threshold = `threshold`, notes "Key Config
//     Parameters"): the masked positions in increasing order of entropy (lowest i first among
//     equal entropies), as long as the running sum of their entropies stays <= the budget;
//     at least one.  Reading: the budget bounds the total entropy of the positions committed
//     in one step, lowest entropy first (the notes name the rule and its parameter only).
// Per masked position also the entropy of its softmax at temperature T, in nats:
//     H = -sum_v p_v ln p_v,   p_v = exp((l_v - m) / T) / sum_u exp((l_u - m) / T)
// (+inf for unmasked positions).
// Confidences and entropies are compared after rounding to float32, the precision the GPU
// reports them in; the entropy rule's running sum is a float32 sum in the rule's order.
// near: bit 0 = a decision at the threshold or budget that may legitimately differ:
// |conf - threshold| <= 1e-5 * threshold (rule 0), or a running entropy sum within the
// entropy tolerance (1e-4 + 1e-5 H per term) of the budget (rule 4); bit 1 = a near-tie
// decided the position: confidences within 1e-5 relative for the fallback's top two (rule 0)
// or the last chosen and first unchosen (rule 1), entropies within the entropy tolerance of
// each other at neighbouring places of the order (rule 4).
// blocks (n_blocks; NULL = all B) selects the blocks computed.  ent / ent32 may be NULL.
int oracle_confidence_commit_rule(int B, int L, int V, const uint16_t* logits,
                                  const uint8_t* mask, int rule, int k, double threshold,
                                  double temperature, const int32_t* blocks, int n_blocks,
                                  int32_t* tok, double* conf, float* conf32, uint8_t* commit,
                                  uint8_t* near, double* ent, float* ent32) {
    if (L <= 0 || V <= 0 || !(temperature > 0.0)) return -1;
    if (rule < 0 || rule > 4 || ((rule == 1 || rule == 2 || rule == 3) && k < 1)) return -1;
    if (rule == 4 && !(threshold >= 0.0 && std::isfinite(threshold))) return -1;
    std::vector<double> ent_buf;
    std::vector<float> ent32_buf;
    if (rule == 4 && (ent == nullptr || ent32 == nullptr)) {
        ent_buf.resize(static_cast<size_t>(B) * L);
        ent32_buf.resize(static_cast<size_t>(B) * L);
        ent = ent_buf.data();
        ent32 = ent32_buf.data();
    }
    const int count = blocks ? n_blocks : B;
    const float thr32 = static_cast<float>(threshold);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bi = 0; bi < count; ++bi) {
        const int b = blocks ? blocks[bi] : bi;
        const size_t r0 = static_cast<size_t>(b) * L;
        for (int i = 0; i < L; ++i) {
            const size_t r = r0 + i;
            near[r] = 0;
            commit[r] = 0;
            if (!mask[r]) {
                tok[r] = -1;
                conf[r] = -std::numeric_limits<double>::infinity();
                conf32[r] = -std::numeric_limits<float>::infinity();
                if (ent) {
                    ent[r] = std::numeric_limits<double>::infinity();
                    ent32[r] = std::numeric_limits<float>::infinity();
                }
                continue;
            }
            const uint16_t* row = logits + r * static_cast<size_t>(V);
            int best = 0;
            double m = bf16_to_f64(row[0]);
            for (int v = 1; v < V; ++v) {
                const double x = bf16_to_f64(row[v]);
                if (x > m) { m = x; best = v; }
            }
            double z = 0.0;
            for (int v = 0; v < V; ++v) z += std::exp((bf16_to_f64(row[v]) - m) / temperature);
            tok[r] = best;
            conf[r] = 1.0 / z;
            conf32[r] = static_cast<float>(conf[r]);
            if (ent) {
                // H = -sum_v p_v ln p_v over the probabilities, term by term
                double h = 0.0;
                for (int v = 0; v < V; ++v) {
                    const double p = std::exp((bf16_to_f64(row[v]) - m) / temperature) / z;
                    if (p > 0.0) h -= p * std::log(p);
                }
                ent[r] = h;
                ent32[r] = static_cast<float>(h);
            }
            if (rule == 0 && std::fabs(conf[r] - threshold) <= 1e-5 * threshold) near[r] |= 1;
        }
        std::vector<int> masked;
        for (int i = 0; i < L; ++i)
            if (mask[r0 + i]) masked.push_back(i);
        if (masked.empty()) continue;
        if (rule == 0) {
            bool any_commit = false;
            for (int i : masked)
                if (conf32[r0 + i] >= thr32) { commit[r0 + i] = 1; any_commit = true; }
            if (!any_commit) {
                int arg = -1;
                for (int i : masked)
                    if (arg < 0 || conf32[r0 + i] > conf32[r0 + arg]) arg = i;
                commit[r0 + arg] = 1;
                const double top = conf[r0 + arg];
                for (int i : masked) {
                    if (i == arg) continue;
                    if (std::fabs(conf[r0 + i] - top) <= 1e-5 * top) {
                        near[r0 + i] |= 2;
                        near[r0 + arg] |= 2;
                    }
                }
            }
        } else if (rule == 1) {
            // selection by confidence: repeatedly the most confident unchosen position
            const int n = std::min<int>(k, static_cast<int>(masked.size()));
            std::vector<char> chosen(L, 0);
            int last = -1;
            for (int c = 0; c < n; ++c) {
                int arg = -1;
                for (int i : masked)
                    if (!chosen[i] && (arg < 0 || conf32[r0 + i] > conf32[r0 + arg])) arg = i;
                chosen[arg] = 1;
                commit[r0 + arg] = 1;
                last = arg;
            }
            for (int i : masked) {
                if (chosen[i]) continue;
                const double lc = conf[r0 + last];
                if (std::fabs(conf[r0 + i] - lc) <= 1e-5 * lc) {
                    near[r0 + i] |= 2;
                    near[r0 + last] |= 2;
                }
            }
        } else if (rule == 4) {
            // increasing entropy (float32), lowest position first among equals
            std::vector<int> order(masked);
            std::stable_sort(order.begin(), order.end(),
                             [&](int x, int y) { return ent32[r0 + x] < ent32[r0 + y]; });
            const float budget32 = static_cast<float>(threshold);
            float run = 0.f;
            double tol = 0.0;
            for (size_t c = 0; c < order.size(); ++c) {
                const int i = order[c];
                const float next = run + ent32[r0 + i];
                tol += 1e-4 + 1e-5 * ent[r0 + i];
                if (std::fabs(static_cast<double>(next) - threshold) <= tol)
                    for (int j : masked) near[r0 + j] |= 1;
                if (c > 0 && !(next <= budget32)) break;
                run = next;
                commit[r0 + i] = 1;
            }
            for (size_t c = 0; c + 1 < order.size(); ++c) {
                const int i = order[c], j = order[c + 1];
                const double hi = ent[r0 + i], hj = ent[r0 + j];
                if (std::fabs(hi - hj) <= 1e-4 + 1e-5 * std::max(hi, hj)) {
                    near[r0 + i] |= 2;
                    near[r0 + j] |= 2;
                }
            }
        } else {
            const int n = std::min<int>(k, static_cast<int>(masked.size()));
            for (int c = 0; c < n; ++c) {
                const int i = rule == 2 ? masked[c] : masked[masked.size() - 1 - c];
                commit[r0 + i] = 1;
            }
        }
    }
    return 0;
}

// The threshold rule (low_confidence_dynamic): oracle_confidence_commit_rule with rule 0.
int oracle_confidence_commit(int B, int L, int V, const uint16_t* logits, const uint8_t* mask,
                             double threshold, double temperature, const int32_t* blocks,
                             int n_blocks, int32_t* tok, double* conf, float* conf32,
                             uint8_t* commit, uint8_t* near) {
    return oracle_confidence_commit_rule(B, L, V, logits, mask, 0, 1, threshold, temperature,
                                         blocks, n_blocks, tok, conf, conf32, commit, near,
                                         nullptr, nullptr);
}

// Mask update between steps: mask &= ~commit (JetEngine notes, "Important Patterns":
// each step moves committed positions from masked to unmasked).
void oracle_apply_commit(int n, uint8_t* mask, const uint8_t* commit) {
    for (int i = 0; i < n; ++i) if (commit[i]) mask[i] = 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

// Sets the OpenMP thread count of later oracle calls (n >= 1).
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

}  // extern "C"
