// Heavy-hitter candidates handed from a decode step to the H2O select that
// follows it (sm_103a).
//
// The H2O score only grows between two selections (every step adds
// probabilities), and the k slots kept by a selection stay candidates, so
// the k-th largest score of a row never falls below the threshold T that
// the previous selection found.  The decode step therefore collects, while
// it writes the new scores, every slot of a row whose new score is >= that
// row's last T; the select kernel finds the exact top-k among those alone
// and scans the whole row only when the list is unusable (no threshold yet,
// too few or too many entries).
//
// Layout, at the start of the H2O evict workspace (after the status block),
// for R = batch * num_kv_heads rows:
//   hint   uint32 [R]            order key of the row's last threshold (0: none)
//   count  uint32 [R]            entries collected by the last decode step
//   key    uint32 [R][kLinkCap]  order keys of the collected scores
//   pos    int32  [R][kLinkCap]  their slots
// The decode step clears `count` before collecting; the select kernel clears
// it after reading, so a list is used at most once.
#pragma once

#include "common.cuh"

namespace kvsel {

constexpr int kLinkCap = 16384;

struct H2OLink {
  uint32_t* hint;
  uint32_t* count;
  uint32_t* key;
  int32_t* pos;
};

__host__ __forceinline__ size_t link_bytes(int rows) {
  size_t off = kStatusBytes;
  off += (size_t(rows) * 4 + 255) / 256 * 256;                // hint
  off += (size_t(rows) * 4 + 255) / 256 * 256;                // count
  off += (size_t(rows) * kLinkCap * 4 + 255) / 256 * 256;     // key
  off += (size_t(rows) * kLinkCap * 4 + 255) / 256 * 256;     // pos
  return off;
}

__host__ __forceinline__ H2OLink link_layout(void* ws, int rows) {
  uint8_t* p = static_cast<uint8_t*>(ws) + kStatusBytes;
  H2OLink L;
  L.hint = reinterpret_cast<uint32_t*>(p);
  p += (size_t(rows) * 4 + 255) / 256 * 256;
  L.count = reinterpret_cast<uint32_t*>(p);
  p += (size_t(rows) * 4 + 255) / 256 * 256;
  L.key = reinterpret_cast<uint32_t*>(p);
  p += (size_t(rows) * kLinkCap * 4 + 255) / 256 * 256;
  L.pos = reinterpret_cast<int32_t*>(p);
  return L;
}

}  // namespace kvsel
