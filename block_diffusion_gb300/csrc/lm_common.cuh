// Pieces shared by the two LM head kernels (lm_head.cu: logits to memory; lm_conf.cu: fused
// with the confidence step): tile constants, the thread layout and the ring cursor.
#pragma once
#include <stdint.h>

namespace bdlm {
namespace lm {

constexpr int kBM = 128;         // rows of one TMA box and of one UMMA sub-tile (M = 128)
constexpr int kSub = 2;          // sub-tiles per CTA tile: two boxes per 256-row stage
constexpr int kBK = 64;          // K per stage (one 128-byte swizzle atom)
constexpr int kWBox = kBM * kBK * 2;       // 16 KB: one box
constexpr int kWBytes = kSub * kWBox;      // 32 KB: a stage of two boxes
constexpr uint32_t kTmemCols = 512;
constexpr int kEpiWarps = 16;   // a multiple of 4: kEpiWarps / 4 per tensor-memory lane quadrant
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kRowWarp = 2 + kEpiWarps;   // producer of the gathered-row ring
constexpr int kThreads = (kRowWarp + 1) * 32;

// One ring of TMA stages: `n` slots, the slot and phase of the next use.
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ void advance(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1;
    }
  }
};

}  // namespace lm
}  // namespace bdlm
