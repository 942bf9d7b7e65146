// internal.h -- descriptors and launcher declarations shared by the
// library's translation units (not part of the public C ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/lora_sgmv.h"

namespace lora {

// One slice, as the kernels see it (same meaning as lora_slice_t).
struct SliceDesc {
  const void* A;
  long long A_slot_stride;
  const void* B;
  long long B_slot_stride;
  int out_dim;
  void* y;
  long long y_row_stride;
  const void* bias;  // [S, out_dim] at bias + s * bias_slot_stride, or nullptr
  long long bias_slot_stride;
};

// A validated problem plus its routing, passed by value to every kernel.
struct ProblemDesc {
  int dtype;  // lora_dtype_t
  int num_tokens;
  int in_dim;
  int S;  // max_num_loras
  int R;  // max_lora_rank
  int n_slices;
  const void* x;
  long long x_row_stride;
  SliceDesc sl[LORA_MAX_SLICES];
  const int* lora_ids;  // device [G]
  const int* offs;      // device [G + 1]
  int G;
  int end;
  const int* token_rows;  // device [end] or nullptr (row i of the sorted order is row i)
  const int* slot_ranks;  // device [S] true ranks, or nullptr (all R)
  unsigned* status;  // device status word (LORA_DEV_* flags)
  // Groups this launch works on: those of seg_lo <= routed rows < seg_hi
  // (the others have no tiles).  0 and INT_MAX: every group.
  int seg_lo, seg_hi;
};

// Records a successful kernel launch of the current entry-point call
// (LORA_PATH_* bits; see lora_last_call_path).  Defined in api.cu.
void note_launch(unsigned path_bits);
// Returns e, recording the launch when it succeeded.
inline cudaError_t noted(cudaError_t e, unsigned path_bits) {
  if (e == cudaSuccess) note_launch(path_bits);
  return e;
}

// Streaming multiprocessors of the current device (cached per device; 0 if
// the query fails, which makes the split heuristics fall back to no split).
int device_sm_count();
// The workspace bound (lora_workspace_bytes) depends on shapes only, so
// where a split count grows with the SM count it is bounded assuming this
// many SMs; launches use the device's own count, which is at most this.
constexpr int kMaxSmsForWorkspace = 256;

// One group's term of the routing digest: SplitMix64's finalizer (Steele,
// Lea and Flood, "Fast splittable pseudorandom number generators", 2014)
// applied to (offset, slot) offset by a Weyl step per group index.  The
// digest of a triple is the sum of its groups' terms modulo 2^64; the host
// computes it from its copy, the kernels from the device arrays.
__host__ __device__ __forceinline__ unsigned long long routing_digest_term(int g, int offset, int slot) {
  unsigned long long z = ((unsigned long long)(unsigned)slot << 32 | (unsigned)offset) +
                         (unsigned long long)(g + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// What a launch knows of the routing triple's host copy (G == 0: nothing):
// the group count and the digest of (grouped_offsets[g], lora_ids[g]) over
// its groups.  Two uniform kernel parameters, so checking the device triple
// against the host copy costs each lane its own groups' terms and a warp sum.
struct HostRouting {
  int G;
  unsigned long long digest;
};

// The tiles of one launch, made on the host from a HostRouting: tile i is
// t[i] = {first row, slot << 8 | rows}.  A CTA reads its own entry, one
// address for all its threads (a constant-bank broadcast), so it knows its
// tile without any global load.  n == 0: none.
constexpr int kHostTilesMax = 128;
struct HostTiles {
  int n;
  int2 t[kHostTilesMax];
};

// Token rows per tile of the bf16 SGMV kernels.
constexpr int kTileRows = 64;

// Host launchers (return a cudaError_t from the launch).
cudaError_t launch_shrink_simple(const ProblemDesc& p, float* u, cudaStream_t s);
cudaError_t launch_expand_simple(const ProblemDesc& p, const float* u, cudaStream_t s, bool pdl);
cudaError_t launch_set_slot(const ProblemDesc& p, int slice, int slot, int r, float scale,
                            const void* A_raw, const void* B_raw, int raw_dtype, cudaStream_t s);
// Failure-path self test (lora_selftest_wait_timeout).
cudaError_t launch_selftest_timeout(unsigned* status, uint32_t limit, cudaStream_t s);
cudaError_t launch_set_bias(const ProblemDesc& p, int slice, int slot, const void* bias_raw, int raw_dtype,
                            cudaStream_t s);

// bf16 fast path (mma.sync tensor cores, 16-byte async copies, clusters for
// lora_shrink's reduction).  `fast_path_ok`
// tells whether a problem meets its alignment / size preconditions.
bool fast_path_ok(const ProblemDesc& p, const void* u);
// launch_shrink_bf16 writes the final u (cluster reduction);
// launch_shrink_partial_bf16 writes apply_splits(...) partial planes of u,
// plane c at u + c * end * n * R, which launch_expand_bf16 sums (nsplit).
// r (optional): a routing whose host copies of the triple were validated.
// The shrink then takes a table of its tiles made from them (no read of the
// device triple before its loads).  hr (optional): the expand checks the
// device triple's digest against the host copy's (a difference:
// LORA_DEV_BAD_OFFSETS, the launch skips its work).
cudaError_t launch_shrink_bf16(const ProblemDesc& p, float* u, cudaStream_t s);
// *splits (if given) receives the partial planes written (the expand's nsplit).
cudaError_t launch_shrink_partial_bf16(const ProblemDesc& p, float* u, cudaStream_t s,
                                       const lora_routing_t* r = nullptr, int* splits = nullptr);
cudaError_t launch_expand_bf16(const ProblemDesc& p, const float* u, cudaStream_t s, bool pdl, int nsplit,
                               const HostRouting* hr = nullptr);
// Upper bound on the partial planes the apply's shrink uses for this shape
// (1..16); shapes only (it sizes the workspace).
int apply_splits(int end, int in_dim, int nR);
// The split the apply's partial-plane shrink actually uses (and its expand
// sums): from the group count and CTA occupancy, at most apply_splits(...);
// *short_ring tells whether the shrink runs its 4-stage ring.
int apply_splits_for(const ProblemDesc& p, bool* short_ring = nullptr, long long exact_tiles = -1);

// The base projection with the delta fused in (sgmv_base.cu).  Per slice,
// the base weight W0_j [out_j, in] (row stride in elements).
struct BaseWeights {
  const void* W0[LORA_MAX_SLICES];
  long long row_stride[LORA_MAX_SLICES];
};
// tcgen05 path: bf16, the fast-path shapes, no token_rows, aligned weights.
bool base_tc_ok(const ProblemDesc& p, const BaseWeights& wts);
// Whether the tensor maps of launch_base_gemm can be encoded (checked before
// anything is launched).
bool base_maps_ok(const ProblemDesc& p, const BaseWeights& wts);
// u: nsplit fp32 planes from a shrink launched just before (after_shrink),
// or unused when end == 0.  Returns cudaErrorNotSupported, having launched
// nothing, when the tensor maps cannot be encoded.
cudaError_t launch_base_gemm(const ProblemDesc& p, const BaseWeights& wts, const float* u, int nsplit,
                             bool after_shrink, cudaStream_t s);
// Any shape / type: one thread per output, u one fp32 plane (generic shrink).
cudaError_t launch_base_gemm_simple(const ProblemDesc& p, const BaseWeights& wts, const float* u,
                                    bool after_shrink, cudaStream_t s);


// tcgen05 shrink for long groups (TMA tensor loads, TMEM accumulator): writes
// nsplit partial planes like launch_shrink_partial_bf16.  tc_shrink_ok says
// whether the shape and routing suit it; tc_shrink_splits(end, in, sms) is
// its plane count for a device of `sms` SMs (shapes and SM count only).  Returns cudaErrorNotSupported when the tensor
// maps cannot be encoded (nothing launched).
bool tc_shrink_ok(const ProblemDesc& p);
// The shape conditions of the tcgen05 kernels without the group-length
// criterion (for a launch restricted to long groups).
bool tc_shapes_ok(const ProblemDesc& p);
bool tc_expand_shapes_ok(const ProblemDesc& p);
int tc_shrink_splits(int end, int in_dim, int sms);
cudaError_t launch_tc_shrink(const ProblemDesc& p, float* u, cudaStream_t s, int nsplit);
// tcgen05 expand for long groups with R = 64 or 128 (sums nsplit planes of u).
bool tc_expand_ok(const ProblemDesc& p);
cudaError_t launch_tc_expand(const ProblemDesc& p, const float* u, cudaStream_t s, bool pdl, int nsplit);
// The apply on tensor cores when tc_expand_ok: the shrink writes u packed as
// the expand's bf16 hi|lo operand image per (128-row tile, slice) into the
// workspace (tc_packed_bytes(S, end, n, R) bytes; 0 unless R is 64 or 128)
// and the expand copies it in whole.  Returns cudaErrorNotSupported, having
// launched nothing, when the tensor maps cannot be encoded.
size_t tc_packed_bytes(int S, int end, int n_slices, int R);
cudaError_t launch_tc_apply_packed(const ProblemDesc& p, void* workspace, cudaStream_t s);

}  // namespace lora
