// tiles.cuh -- device-side view of the routing triple: validation and the
// mapping from a flat tile index to (group, slot, first row, rows).
//
// Group g covers sorted-batch rows [offs[g], offs[g+1]) and uses slot
// lora_ids[g] ("max.pipelines.lora.LoRAManagerV3", get_lora_graph_inputs).
// Each group is cut into ceil(len / tile_rows) tiles; tiles are numbered
// group by group.  A launch may work on a class of groups only (lengths in
// [seg_lo, seg_hi)): the other groups then have no tiles.  Every CTA scans
// the whole (small: G <= max_num_loras) triple, so every CTA of a launch
// reaches the same outcome on validity and an invalid triple makes the whole
// launch skip its work.
#pragma once

#include "internal.h"

namespace lora {

struct Tile {
  int g;
  int slot;
  int row0;
  int rows;
};

__device__ __forceinline__ unsigned warp_or(unsigned v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Executed by one full warp.  Returns true on every lane iff the routing is
// valid and `tile` exists; `out` is then valid on every lane.  Records
// LORA_DEV_* flags in p.status on a violation.  With what the launch knows of
// a host copy of the triple (hr, G > 0) the device triple's digest must also
// equal the host copy's (else LORA_DEV_BAD_OFFSETS).
__device__ __forceinline__ bool warp_locate_tile(const ProblemDesc& p, int tile_rows, long long tile,
                                                 Tile& out, const HostRouting* hr = nullptr) {
  const int lane = threadIdx.x & 31;
  unsigned bad = 0;
  if (lane == 0) {
    if (p.offs[0] != 0) bad |= LORA_DEV_BAD_OFFSETS;
    if (p.offs[p.G] != p.end) bad |= LORA_DEV_BAD_END;
  }
  long long base = 0;
  int found_lane_data[4] = {0, 0, 0, 0};
  bool found = false;
  unsigned long long digest = 0;
  for (int c = 0; c < p.G; c += 32) {
    const int g = c + lane;
    long long nt = 0;
    int o0 = 0, o1 = 0, id = 0;
    if (g < p.G) {
      o0 = p.offs[g];
      o1 = p.offs[g + 1];
      id = p.lora_ids[g];
      if (o1 < o0) bad |= LORA_DEV_BAD_OFFSETS;
      // offs[G] is checked against end on both sides, so offsets 0..G-1
      // and the slots decide equality
      if (hr && hr->G > 0) digest += routing_digest_term(g, o0, id);
      if (id < 0 || id >= p.S) bad |= LORA_DEV_BAD_SLOT;
      const long long len = (long long)o1 - (long long)o0;
      nt = (len > 0 && len >= p.seg_lo && len < p.seg_hi) ? (len + tile_rows - 1) / tile_rows : 0;
    }
    long long incl = nt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    const long long excl = incl - nt;
    if (nt > 0 && tile >= base + excl && tile < base + incl) {
      const int row0 = o0 + (int)((tile - base - excl) * tile_rows);
      found_lane_data[0] = g;
      found_lane_data[1] = id;
      found_lane_data[2] = row0;
      found_lane_data[3] = min(tile_rows, o1 - row0);
      found = true;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (hr && hr->G > 0) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) digest += __shfl_xor_sync(0xffffffffu, digest, d);
    if (hr->G != p.G || digest != hr->digest) bad |= LORA_DEV_BAD_OFFSETS;
  }
  bad = warp_or(bad);
  if (bad) {
    if (lane == 0) atomicOr(p.status, bad);
    return false;
  }
  const unsigned who = __ballot_sync(0xffffffffu, found);
  if (!who) return false;
  const int src = __ffs(who) - 1;
  out.g = __shfl_sync(0xffffffffu, found_lane_data[0], src);
  out.slot = __shfl_sync(0xffffffffu, found_lane_data[1], src);
  out.row0 = __shfl_sync(0xffffffffu, found_lane_data[2], src);
  out.rows = __shfl_sync(0xffffffffu, found_lane_data[3], src);
  return true;
}

// Executed by one full warp: validity of the whole triple (no tile lookup).
__device__ __forceinline__ bool warp_check_routing(const ProblemDesc& p) {
  Tile t;
  const int lane = threadIdx.x & 31;
  unsigned bad = 0;
  if (lane == 0) {
    if (p.offs[0] != 0) bad |= LORA_DEV_BAD_OFFSETS;
    if (p.offs[p.G] != p.end) bad |= LORA_DEV_BAD_END;
  }
  for (int g = lane; g < p.G; g += 32) {
    if (p.offs[g + 1] < p.offs[g]) bad |= LORA_DEV_BAD_OFFSETS;
    const int id = p.lora_ids[g];
    if (id < 0 || id >= p.S) bad |= LORA_DEV_BAD_SLOT;
  }
  (void)t;
  bad = warp_or(bad);
  if (bad && lane == 0) atomicOr(p.status, bad);
  return bad == 0;
}

// Rank columns of slot `slot` that can be non-zero: ceil16 of its true rank
// when the problem carries slot_ranks (clamped to [0, R]), else R.
__device__ __forceinline__ int slot_kmax(const ProblemDesc& p, int slot) {
  if (!p.slot_ranks) return p.R;
  int r = p.slot_ranks[slot];
  r = r < 0 ? 0 : r;
  r = (r + 15) & ~15;
  return r < p.R ? r : p.R;
}

// Group of routed row t (binary search; routing already validated).
__device__ __forceinline__ int group_of_row(const ProblemDesc& p, int t) {
  int lo = 0, hi = p.G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.offs[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

}  // namespace lora
