// The per-token row list shared by the two streaming kernels: which rows a token reads, in the order
// the definition consumes them, compacted by a warp ballot (flashinfer PR #6631, Test changes: -1 routes
// contribute nothing; one bound check per route).
#pragma once

#include "mfr_device.cuh"

namespace mfr {

constexpr uint32_t kTagPartial = 0xffu;
constexpr uint32_t kTagShared = 0x100u;    // the partial's shared row
constexpr uint32_t kTagResidual = 0x200u;  // the residual row (closes a pass)
constexpr uint32_t kTagLast = 0x400u;      // the partial's last row: round it into the rank sum after

// One listed row of a token: where it starts, its scale and its tag.
struct RowEntry {
  const uint8_t* src;
  float scale;
  uint32_t tag;
};

// Slot s of a token's row list, in list order: partial by partial, routes k = 0..K-1 then the
// partial's shared row (if it has one).  Returns the partial and k (-1 for the shared row).
__device__ __forceinline__ void slot_in_list_order(const KParams& p, int s, int& r, int& k) {
  int base = 0;
  for (r = 0; r < p.R - 1; ++r) {
    const int n = p.K + static_cast<int>((p.shared_mask >> r) & 1u);
    if (s < base + n) break;
    base += n;
  }
  k = s - base;
  if (k >= p.K) k = -1;
}

// The routing warp's list for token t: valid routes in order and the partial's shared row, compacted
// with a warp ballot, each partial's last row tagged, then the residual row.  Returns the number of
// entries (at least 1).
__device__ __forceinline__ int build_row_list(const KParams& p, int t, RowEntry* list, int lane) {
  int n = 0;
  for (int base = 0; base < p.nslots; base += 32) {
    const int s = base + lane;
    bool valid = false;
    RowEntry row;
    if (s < p.nslots) {
      int r, k;
      slot_in_list_order(p, s, r, k);
      const KPartial& P = p.part[r];
      if (k < 0) {
        row.src = P.shared + static_cast<int64_t>(t) * p.H * 2;
        row.scale = 1.0f;
        row.tag = static_cast<uint32_t>(r) | kTagShared;
        valid = true;
      } else {
        // flashinfer PR #6631, Test changes: -1 routes contribute nothing; one bound check per route.
        const int64_t ei = static_cast<int64_t>(t) * p.K + k;
        const int32_t idx = P.perm[ei];
        valid = idx >= 0 && static_cast<int64_t>(idx) < P.rows;
        if (valid) {
          row.src = P.gemm2 + static_cast<int64_t>(idx) * p.H * 2;
          row.scale = load_scale(P.scale, ei, p.scale_dtype);
          row.tag = static_cast<uint32_t>(r);
        }
      }
    }
    const uint32_t ballot = __ballot_sync(0xffffffffu, valid);
    if (valid) list[n + __popc(ballot & ((1u << lane) - 1u))] = row;
    n += __popc(ballot);
  }
  __syncwarp();
  // An entry is its partial's last row when the next entry belongs to another partial (or there is
  // none).  All reads of a round happen before its writes.
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const uint32_t tag = (i < n) ? list[i].tag : 0u;
    const bool last = (i < n) && (i + 1 == n || (list[i + 1].tag & kTagPartial) != (tag & kTagPartial));
    __syncwarp();
    if (last) list[i].tag = tag | kTagLast;
    __syncwarp();
  }
  if (lane == 0) {
    RowEntry res;
    res.src = p.fin_only ? nullptr : p.residual + static_cast<int64_t>(t) * p.H * 2;  // nothing to read
    res.scale = 1.0f;
    res.tag = kTagResidual;
    list[n] = res;
  }
  return n + 1;
}

}  // namespace mfr
