// sgmv_tc.cu -- SGMV shrink on the 5th-generation tensor cores (tcgen05) for
// long groups (prefill), bf16, sm_103a.
//
//   u[t, j*R+k] = sum_i A_j[s, k, i] x[t, i]      for the routed rows t of a group
// ("vLLM LoRA 实现深度解析" sections 1 and 6; routing triple of the
// "max.pipelines.lora.LoRAManagerV3" page, get_lora_graph_inputs).
//
// Shrink: one CTA per (128-row tile of a group, column part, K split).
// Warp-specialised:
//   warp 0  TMA producer: per 64-wide K stage, one box of the tile's x rows
//           (128 x 64) and the slot's A rows of the CTA's columns (R-row,
//           64-row or 16-row boxes), 128-byte swizzle, into a ring of stages;
//   warp 1  TMEM owner and MMA issuer: tcgen05.mma M=128, N = the CTA's
//           columns (two MMAs of N/2 when N > 256), K=16 per instruction,
//           accumulating in TMEM; a tcgen05.commit per stage hands the slot
//           back to the producer;
//   warps 2-5  epilogue: tcgen05.ld of their 32 TMEM lanes (= rows) and
//           stores of u: fp32 rows (a K split's plane), or for the apply on
//           ranks 64/128 the packed intermediate (bf16 hi + lo in the
//           expand's swizzled operand layout, see pack_u16).  For gathered
//           batches (token_rows) they first copy the tile's scattered x
//           rows into the stages (16-byte async copies, 32 rows each) in
//           place of the producer's x boxes.
// Expand (further down): persistent, one CTA per SM over (tile, slice,
// 128-column block) units, TMEM accumulators, 8 epilogue warps.
// Rows of the 128-row box past the group are other groups' rows (read, never
// stored) or rows at or past `end`, which the tensor maps zero-fill: base
// rows are never read.
// Every mbarrier wait is bounded; on expiry the CTA records LORA_DEV_TIMEOUT,
// skips its stores and still releases its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tiles.cuh"

namespace lora {

namespace {

constexpr int TM = 128;       // rows per tile (MMA M)
constexpr int TK = 64;        // K per stage (one 128-byte swizzle row)
constexpr int TTHREADS = 192; // 6 warps

template <int NR>
struct TcCfg {
  static constexpr int NH = NR > 256 ? 2 : 1;  // MMAs per K step
  static constexpr int NB = NR / NH;           // N per MMA
  static_assert(NB % 16 == 0 && NB >= 16 && NB <= 256, "MMA N");
  static constexpr int X_BYTES = TM * TK * 2;  // 16 KB
  static constexpr int A_BYTES = NR * TK * 2;
  static constexpr int STAGE = X_BYTES + ((A_BYTES + 1023) / 1024) * 1024;
  // As deep a ring as ~208 KB holds (up to 8 stages): with one CTA per SM the
  // bytes in flight per SM are what sets the streaming rate.
  static constexpr int NSTAGE = (208 * 1024) / STAGE >= 8 ? 8 : (208 * 1024) / STAGE;
  static constexpr int SMEM = NSTAGE * STAGE + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = NR <= 32 ? 32 : NR <= 64 ? 64 : NR <= 128 ? 128 : NR <= 256 ? 256 : 512;
};

// Byte offset of bf16 element (row r, k) in a K-major operand made of
// [128 rows x 64] blocks with the 128-byte swizzle (16-byte chunk c of row r
// stored at chunk c ^ (r % 8)).
__device__ __forceinline__ uint32_t sw128_offset(int r, int k) {
  const int kb = k >> 6, kk = k & 63;
  return (uint32_t)(kb * TM * 128 + r * 128 + ((((kk >> 3) ^ (r & 7))) << 4) + ((kk & 7) << 1));
}

// Packed u: for every (tile, slice) the expand's A operand as it sits in
// shared memory, 2R/64 swizzled [128 rows x 64] bf16 blocks holding u's hi
// part (k < R) and lo part (k >= R), u = hi + lo to 16 significant bits.
// Row r's 16 values k0 .. k0+15 of one slice go to `blk` (that slice's image).
__device__ __forceinline__ void pack_u16(uint8_t* blk, int R, int r, int k0, const float* v) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_hi_lo_bf16x2(v[8 * h + 2 * e], v[8 * h + 2 * e + 1], hi[e], lo[e]);
    const int k = k0 + 8 * h;
    *reinterpret_cast<uint4*>(blk + sw128_offset(r, k)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(blk + sw128_offset(r, R + k)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

}  // namespace

// Gathered batches (token_rows): the x / y row of every position of tile t;
// positions past the tile's rows repeat its first row (their results are
// never stored).  Executed by one full warp; false on every lane (and
// LORA_DEV_BAD_ROW recorded) if an entry is out of range.
__device__ __forceinline__ bool warp_tile_rows(const ProblemDesc& p, const Tile& t, int* rows) {
  const int lane = threadIdx.x & 31;
  int bad = 0;
  const int first = p.token_rows[t.row0];
  for (int r = lane; r < TM; r += 32) {
    const int v = r < t.rows ? p.token_rows[t.row0 + r] : first;
    if (v < 0 || v >= p.num_tokens) bad = 1;
    rows[r] = v;
  }
  bad = __any_sync(0xffffffffu, bad);
  if (bad && lane == 0) atomicOr(p.status, LORA_DEV_BAD_ROW);
  return !bad;
}

struct TcMaps {
  CUtensorMap x;                     // [T rows, in] bf16, box 64 x 128
  CUtensorMap a[LORA_MAX_SLICES];    // per slice [S, R, in] bf16, box 64 x R x 1 (full rank)
  CUtensorMap a64[LORA_MAX_SLICES];  // same tensor, box 64 x 64 x 1 (slots below full rank)
  CUtensorMap a16[LORA_MAX_SLICES];  // same tensor, box 64 x 16 x 1
};

// grid.x = tiles * nsn * nsplit.  CTA (tile, column part cn, K split ks)
// computes columns [cn * NR, +NR) of u (n*R columns in all) over input range
// ks of nsplit.  Output: fp32 plane ks of u (plane_stride apart), or, with
// PACK (nsplit == 1), packed u (see pack_u16) at upk, tile-major.
template <int NR, bool PACK>
__global__ void __launch_bounds__(TTHREADS, 1) sgmv_tc_shrink_kernel(const __grid_constant__ ProblemDesc p,
                                                                    const __grid_constant__ TcMaps maps,
                                                                    float* __restrict__ u, int nsplit,
                                                                    long long plane_stride, int nsn,
                                                                    uint8_t* __restrict__ upk) {
  using Cfg = TcCfg<NR>;
  constexpr int NSTAGE = Cfg::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[NSTAGE];
  __shared__ __align__(8) uint64_t empty[NSTAGE];
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t s_tmem;
  __shared__ Tile s_tile;
  __shared__ int s_ok;
  __shared__ int s_fail;
  __shared__ int s_kmax;
  __shared__ int s_rows[TM];  // gathered batches: the x row of each tile position

  // 1024-byte aligned ring (the 128-byte swizzle repeats every 1024 bytes).
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  // Launched as a programmatic dependent of whatever kernel precedes it: no
  // global memory is touched before that kernel has completed.
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = (int)(blockIdx.x % (unsigned)nsplit);
  const int cn = (int)((blockIdx.x / (unsigned)nsplit) % (unsigned)nsn);
  const long long tile = blockIdx.x / (unsigned)(nsplit * nsn);
  const int n_base = cn * NR;  // first u column of this CTA
  const bool gathered = p.token_rows != nullptr;
  if (warp == 0) {
    Tile t{};
    bool ok = warp_locate_tile(p, TM, tile, t);
    if (ok && gathered) ok = warp_tile_rows(p, t, s_rows);  // a bad entry skips the tile
    if (lane == 0) {
      s_tile = t;
      s_ok = ok;
      s_fail = 0;
      s_kmax = ok ? slot_kmax(p, t.slot) : 0;
      for (int i = 0; i < NSTAGE; ++i) {
        // gathered: one arrival for the A boxes' bytes, one from each of the
        // four gathering warps once its copies of the stage's x rows landed
        mbar_init(&full[i], gathered ? 1 + 4 : 1);
        mbar_init(&empty[i], 1);
      }
      mbar_init(&done, 1);
      fence_mbar_init();
    }
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Dependents (the expand) may start only once this CTA holds its TMEM, so
  // a waiting expand CTA can never hold columns this shrink still needs.
  pdl_launch_dependents();
  const uint32_t tmem = s_tmem;
  const Tile t = s_tile;
  const bool ok = s_ok != 0;
  const int R = p.R;
  const int kmax = s_kmax;  // A rows past this (per slice) are not loaded
  const int kc = p.in_dim / nsplit;
  const int k0 = split * kc;
  const int nst = kc / TK;

  if (ok && warp == 0 && lane == 0 && gathered) {
    // ---- producer, gathered batch: the A rows by TMA; the x rows are
    // copied by warps 2-5 (below), which join each stage's full barrier.
    const uint64_t pol_keep = policy_evict_last();
    uint32_t a_bytes = 0;
    for (int j = 0; j < p.n_slices; ++j) {
      const int klo = max(0, n_base - j * R), khi = min(min(R, n_base + NR - j * R), kmax);
      if (khi > klo) a_bytes += (uint32_t)((khi - klo) * TK * 2);
    }
    for (int s = 0; s < nst; ++s) {
      const int slot = s % NSTAGE;
      if (s >= NSTAGE && !mbar_wait(&empty[slot], (uint32_t)(((s / NSTAGE) - 1) & 1))) {
        atomicOr(&s_fail, 1);
        break;
      }
      uint8_t* as = smem + slot * Cfg::STAGE + Cfg::X_BYTES;
      const int kk = k0 + s * TK;
      mbar_arrive_expect_tx(&full[slot], a_bytes);
      for (int j = 0; j < p.n_slices; ++j) {
        const int klo = max(0, n_base - j * R), khi = min(min(R, n_base + NR - j * R), kmax);
        if (khi <= klo) continue;
        uint8_t* dst = as + (j * R - n_base) * TK * 2;
        if (klo == 0 && khi == R) {
          tma_load_3d_hint(dst, &maps.a[j], kk, 0, t.slot, &full[slot], pol_keep);
        } else {
          int kb = klo;
          for (; kb + 64 <= khi; kb += 64)
            tma_load_3d_hint(dst + kb * TK * 2, &maps.a64[j], kk, kb, t.slot, &full[slot], pol_keep);
          for (; kb < khi; kb += 16)
            tma_load_3d_hint(dst + kb * TK * 2, &maps.a16[j], kk, kb, t.slot, &full[slot], pol_keep);
        }
      }
    }
  } else if (ok && warp == 0 && lane == 0) {
    // ---- producer (x streams through L2 once; the slot's A rows are re-read
    // by every tile of the group, so they are kept)
    const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
    uint32_t a_bytes = Cfg::X_BYTES;
    for (int j = 0; j < p.n_slices; ++j) {
      const int klo = max(0, n_base - j * R), khi = min(min(R, n_base + NR - j * R), kmax);
      if (khi > klo) a_bytes += (uint32_t)((khi - klo) * TK * 2);
    }
    for (int s = 0; s < nst; ++s) {
      const int slot = s % NSTAGE;
      if (s >= NSTAGE && !mbar_wait(&empty[slot], (uint32_t)(((s / NSTAGE) - 1) & 1))) {
        atomicOr(&s_fail, 1);
        break;
      }
      uint8_t* xs = smem + slot * Cfg::STAGE;
      uint8_t* as = xs + Cfg::X_BYTES;
      mbar_arrive_expect_tx(&full[slot], a_bytes);
      const int kk = k0 + s * TK;
      tma_load_2d_hint(xs, &maps.x, kk, t.row0, &full[slot], pol_stream);
      for (int j = 0; j < p.n_slices; ++j) {
        // Rows [klo, khi) of slice j fall in this CTA's columns (and the rank).
        const int klo = max(0, n_base - j * R), khi = min(min(R, n_base + NR - j * R), kmax);
        if (khi <= klo) continue;
        uint8_t* dst = as + (j * R - n_base) * TK * 2;
        if (klo == 0 && khi == R) {  // one box per slice (few large TMA requests)
          tma_load_3d_hint(dst, &maps.a[j], kk, 0, t.slot, &full[slot], pol_keep);
        } else {  // 64-row boxes, then 16-row boxes
          int kb = klo;
          for (; kb + 64 <= khi; kb += 64)
            tma_load_3d_hint(dst + kb * TK * 2, &maps.a64[j], kk, kb, t.slot, &full[slot], pol_keep);
          for (; kb < khi; kb += 16)
            tma_load_3d_hint(dst + kb * TK * 2, &maps.a16[j], kk, kb, t.slot, &full[slot], pol_keep);
        }
      }
    }
  } else if (ok && warp == 1 && lane == 0) {
    // ---- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(TM, Cfg::NB);
    for (int s = 0; s < nst; ++s) {
      const int slot = s % NSTAGE;
      if (!mbar_wait(&full[slot], (uint32_t)((s / NSTAGE) & 1))) {
        atomicOr(&s_fail, 1);
        break;
      }
      tc_fence_after_sync();
      const uint32_t xs = smem_addr(smem + slot * Cfg::STAGE);
      const uint32_t as = xs + Cfg::X_BYTES;
#pragma unroll
      for (int ks = 0; ks < TK / 16; ++ks) {
        const uint64_t adesc = sw128_desc(xs + ks * 32);
#pragma unroll
        for (int h = 0; h < Cfg::NH; ++h) {
          const uint64_t bdesc = sw128_desc(as + h * Cfg::NB * 128 + ks * 32);
          tc_mma_bf16(tmem + h * Cfg::NB, adesc, bdesc, idesc, (s > 0 || ks > 0) ? 1u : 0u);
        }
      }
      tc_commit(&empty[slot]);  // slot free once these MMAs have read it
    }
    tc_commit(&done);  // accumulator complete
  } else if (ok && warp >= 2) {
    if (gathered) {
      // ---- gathered batch: warp w copies x rows 32*(w % 4) .. +31 of every
      // stage (scattered through token_rows) with 16-byte async copies into
      // the stage's 128-byte-swizzled layout, eight lanes per row, as many
      // stages deep as the ring, and arrives on each stage's full barrier
      // once its copies have landed.
      const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(p.x);
      const int rb = (warp & 3) * 32;
      int signalled = 0;
      bool gbad = false;
      for (int s = 0; s < nst; ++s) {
        const int slot = s % NSTAGE;
        bool free_ok = true;
        if (s >= NSTAGE && lane == 0) free_ok = mbar_wait(&empty[slot], (uint32_t)(((s / NSTAGE) - 1) & 1));
        if (!__shfl_sync(0xffffffffu, (int)free_ok, 0)) {
          gbad = true;
          break;
        }
        uint8_t* xs = smem + slot * Cfg::STAGE;
        const int kk = k0 + s * TK;
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // row rb + e / 8, 16-byte chunk e % 8
          const int e = lane + 32 * i, r = rb + (e >> 3), c = e & 7;
          cp_async16(xs + r * 128 + ((c ^ (r & 7)) << 4), xg + (long long)s_rows[r] * p.x_row_stride + kk + c * 8);
        }
        cp_async_commit();
        if (s - signalled >= NSTAGE - 1) {  // the oldest stage in flight has landed
          cp_async_wait<NSTAGE - 1>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[signalled % NSTAGE]);
          ++signalled;
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (gbad) atomicOr(&s_fail, 1);
        for (; signalled < nst; ++signalled) mbar_arrive(&full[signalled % NSTAGE]);
      }
    }
    // ---- epilogue: warp w reads TMEM lanes 32*(w % 4) .. +31 (= tile rows)
    const bool got = __all_sync(0xffffffffu, mbar_wait(&done, 0));  // warp-uniform for tcgen05.ld
    tc_fence_after_sync();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int nR = p.n_slices * R;
    const bool live = row < t.rows;
    const int uimg = 4 * R * TM;  // bytes of one (tile, slice) packed image
    if (!got) {
      atomicOr(&s_fail, 1);
    } else {
      float* up = u + split * plane_stride + (long long)(t.row0 + row) * nR + n_base;
      for (int c = 0; c < NR; c += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
        // Columns past the slot's rank came from rows never loaded: 0.
        const int col = n_base + c, j = col / R, k = col - j * R;
        const bool keep = k < kmax;
        if (PACK) {  // rows past the group: zeros
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = (keep && live) ? v[e] : 0.f;
          pack_u16(upk + ((long long)tile * p.n_slices + j) * uimg, R, row, k, v);
        } else if (live) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(up + c + i) =
                keep ? make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    if (s_fail) {
      // Give MMAs still in flight a bounded chance to finish before release.
      (void)mbar_wait(&done, 0);
      if (lane == 0) atomicOr(p.status, LORA_DEV_TIMEOUT);
    }
    tc_fence_after_sync();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// The apply's shrink with the input dimension split over a cluster of CL
// CTAs (2 or 4) per 128-row tile, for batches with too few tiles to fill
// the GPU one CTA per tile.  Each CTA streams its K range of the tile's x rows
// (so each column part reads x once) and of the slot's A rows for its NR
// columns (all n*R, or one of nsn column parts); the CL partial accumulators
// are then exchanged through distributed shared memory: CTA q owns columns
// [q*NR/CL, (q+1)*NR/CL) of the part, receives the other CTAs' partials of
// those columns into its (then idle) stage ring, sums the CL partials in rank
// order (the same order on every CTA: deterministic) and stores them packed
// (pack_u16).  Two cluster barriers: before the exchange (every CTA's MMAs
// have drained its ring) and after it.  NST: ring depth -- a shallow ring
// lets two CTAs share an SM when the grid has more CTAs than SMs.  Gathered
// batches: warps 2-5 copy the scattered x rows of the CTA's K range, as in
// the one-CTA shrink.
template <int NR, int CL, int NST>
__global__ void __launch_bounds__(TTHREADS, 1) sgmv_tc_shrink_ksplit_kernel(const __grid_constant__ ProblemDesc p,
                                                                           const __grid_constant__ TcMaps maps,
                                                                           uint8_t* __restrict__ upk, int nsn) {
  using Cfg = TcCfg<NR>;
  constexpr int NSTAGE = NST;
  constexpr int NRC = NR / CL;  // columns each CTA sums and stores
  static_assert(NRC % 16 == 0, "column share");
  static_assert((CL - 1) * TM * NRC * 4 <= NSTAGE * Cfg::STAGE, "exchange buffer must fit in the ring");
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[NSTAGE];
  __shared__ __align__(8) uint64_t empty[NSTAGE];
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t s_tmem;
  __shared__ Tile s_tile;
  __shared__ int s_ok;
  __shared__ int s_fail;
  __shared__ int s_kmax;
  __shared__ int s_rows[TM];  // gathered batches: the x row of each tile position

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = (int)(blockIdx.x % (unsigned)CL);  // rank in the cluster (cluster dims CL x 1 x 1)
  const int cn = (int)((blockIdx.x / (unsigned)CL) % (unsigned)nsn);
  const long long tile = blockIdx.x / (unsigned)(CL * nsn);
  const int n_base = cn * NR;  // first u column of this cluster's part
  const bool gathered = p.token_rows != nullptr;
  if (warp == 0) {
    Tile t{};
    bool ok = warp_locate_tile(p, TM, tile, t);
    if (ok && gathered) ok = warp_tile_rows(p, t, s_rows);  // the same outcome on every CTA of the cluster
    if (lane == 0) {
      s_tile = t;
      s_ok = ok;
      s_fail = 0;
      s_kmax = ok ? slot_kmax(p, t.slot) : 0;
      for (int i = 0; i < NSTAGE; ++i) {
        mbar_init(&full[i], gathered ? 1 + 4 : 1);  // gathered: + one arrival per x-copying warp
        mbar_init(&empty[i], 1);
      }
      mbar_init(&done, 1);
      fence_mbar_init();
    }
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  pdl_launch_dependents();
  const uint32_t tmem = s_tmem;
  const Tile t = s_tile;
  const bool ok = s_ok != 0;  // the same on every CTA of the cluster (same tile)
  const int R = p.R;
  const int kmax = s_kmax;
  const int kc = p.in_dim / CL;
  const int k0 = crank * kc;
  const int nst = kc / TK;

  if (ok && warp == 0 && lane == 0) {
    const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
    uint32_t a_bytes = gathered ? 0 : Cfg::X_BYTES;
    for (int j = 0; j < p.n_slices; ++j) {
      const int klo = max(0, n_base - j * R), khi = min(min(R, n_base + NR - j * R), kmax);
      if (khi > klo) a_bytes += (uint32_t)((khi - klo) * TK * 2);
    }
    for (int s = 0; s < nst; ++s) {
      const int slot = s % NSTAGE;
      if (s >= NSTAGE && !mbar_wait(&empty[slot], (uint32_t)(((s / NSTAGE) - 1) & 1))) {
        atomicOr(&s_fail, 1);
        break;
      }
      uint8_t* xs = smem + slot * Cfg::STAGE;
      uint8_t* as = xs + Cfg::X_BYTES;
      mbar_arrive_expect_tx(&full[slot], a_bytes);
      const int kk = k0 + s * TK;
      if (!gathered) tma_load_2d_hint(xs, &maps.x, kk, t.row0, &full[slot], pol_stream);
      for (int j = 0; j < p.n_slices; ++j) {
        // Rows [klo, khi) of slice j fall in this part's columns (and the rank).
        const int klo = max(0, n_base - j * R), khi = min(min(R, n_base + NR - j * R), kmax);
        if (khi <= klo) continue;
        uint8_t* dst = as + (j * R - n_base) * TK * 2;
        if (klo == 0 && khi == R) {
          tma_load_3d_hint(dst, &maps.a[j], kk, 0, t.slot, &full[slot], pol_keep);
        } else {
          int kb = klo;
          for (; kb + 64 <= khi; kb += 64)
            tma_load_3d_hint(dst + kb * TK * 2, &maps.a64[j], kk, kb, t.slot, &full[slot], pol_keep);
          for (; kb < khi; kb += 16)
            tma_load_3d_hint(dst + kb * TK * 2, &maps.a16[j], kk, kb, t.slot, &full[slot], pol_keep);
        }
      }
    }
  } else if (ok && warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(TM, Cfg::NB);
    for (int s = 0; s < nst; ++s) {
      const int slot = s % NSTAGE;
      if (!mbar_wait(&full[slot], (uint32_t)((s / NSTAGE) & 1))) {
        atomicOr(&s_fail, 1);
        break;
      }
      tc_fence_after_sync();
      const uint32_t xs = smem_addr(smem + slot * Cfg::STAGE);
      const uint32_t as = xs + Cfg::X_BYTES;
#pragma unroll
      for (int ks = 0; ks < TK / 16; ++ks) {
        const uint64_t adesc = sw128_desc(xs + ks * 32);
#pragma unroll
        for (int h = 0; h < Cfg::NH; ++h) {
          const uint64_t bdesc = sw128_desc(as + h * Cfg::NB * 128 + ks * 32);
          tc_mma_bf16(tmem + h * Cfg::NB, adesc, bdesc, idesc, (s > 0 || ks > 0) ? 1u : 0u);
        }
      }
      tc_commit(&empty[slot]);
    }
    tc_commit(&done);
  } else if (ok && warp >= 2 && gathered) {
    // ---- gathered batch: warps 2-5 copy the tile's scattered x rows of
    // this CTA's K range (32 rows each), as in the one-CTA shrink.
    const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(p.x);
    const int rb = (warp & 3) * 32;
    int signalled = 0;
    bool gbad = false;
    for (int s = 0; s < nst; ++s) {
      const int slot = s % NSTAGE;
      bool free_ok = true;
      if (s >= NSTAGE && lane == 0) free_ok = mbar_wait(&empty[slot], (uint32_t)(((s / NSTAGE) - 1) & 1));
      if (!__shfl_sync(0xffffffffu, (int)free_ok, 0)) {
        gbad = true;
        break;
      }
      uint8_t* xs = smem + slot * Cfg::STAGE;
      const int kk = k0 + s * TK;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i, r = rb + (e >> 3), c = e & 7;
        cp_async16(xs + r * 128 + ((c ^ (r & 7)) << 4), xg + (long long)s_rows[r] * p.x_row_stride + kk + c * 8);
      }
      cp_async_commit();
      if (s - signalled >= NSTAGE - 1) {
        cp_async_wait<NSTAGE - 1>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[signalled % NSTAGE]);
        ++signalled;
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (gbad) atomicOr(&s_fail, 1);
      for (; signalled < nst; ++signalled) mbar_arrive(&full[signalled % NSTAGE]);
    }
  }
  // Every thread: the accumulator is complete (or the CTA failed), and so is
  // every other CTA's of the cluster, whose rings are then free.
  bool got = true;
  if (ok && warp >= 2) got = __all_sync(0xffffffffu, mbar_wait(&done, 0));
  if (!got) atomicOr(&s_fail, 1);
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();
  const int q = warp & 3;
  const int row = q * 32 + lane;
  // [CL - 1][TM][NRC]: the other ranks' partials of this CTA's columns, rank
  // order (a sender of rank c lands in slot c, or c - 1 past the receiver).
  float* recv = reinterpret_cast<float*>(smem);
  if (ok && warp >= 2 && got) {
    // Send the partials of the other ranks' columns.
    for (int dst = 0; dst < CL; ++dst) {
      if (dst == crank) continue;
      const int slot_at_dst = crank < dst ? crank : crank - 1;
      const uint32_t base = smem_addr(recv + ((size_t)slot_at_dst * TM + row) * NRC);
      const uint32_t remote = map_shared_rank(base, (uint32_t)dst);
      for (int c = 0; c < NRC; c += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(dst * NRC + c), v);
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote + (uint32_t)((c + e) * 4)),
                       "f"(v[e]), "f"(v[e + 1]), "f"(v[e + 2]), "f"(v[e + 3])
                       : "memory");
      }
    }
  }
  tc_fence_before_sync();
  cluster_sync();  // every partial has landed
  tc_fence_after_sync();
  if (ok && warp >= 2 && got && !s_fail) {
    const bool live = row < t.rows;
    const int uimg = 4 * R * TM;
    for (int c = 0; c < NRC; c += 16) {
      float own[16];
      tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(crank * NRC + c), own);
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = 0.f;
      for (int src = 0; src < CL; ++src) {  // rank order
        if (src == crank) {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = src == 0 ? own[e] : v[e] + own[e];
        } else {
          const float* rp = recv + ((size_t)(src < crank ? src : src - 1) * TM + row) * NRC + c;
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(rp + e);
            v[e] = src == 0 ? w4.x : v[e] + w4.x;
            v[e + 1] = src == 0 ? w4.y : v[e + 1] + w4.y;
            v[e + 2] = src == 0 ? w4.z : v[e + 2] + w4.z;
            v[e + 3] = src == 0 ? w4.w : v[e + 3] + w4.w;
          }
        }
      }
      const int col = n_base + crank * NRC + c, j = col / R, k = col - j * R;
      const bool keep = k < kmax;  // columns past the slot's rank read no A rows: 0
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = (keep && live) ? v[e] : 0.f;
      pack_u16(upk + ((long long)tile * p.n_slices + j) * uimg, R, row, k, v);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    if (s_fail) {
      (void)mbar_wait(&done, 0);
      if (lane == 0) atomicOr(p.status, LORA_DEV_TIMEOUT);
    }
    tc_fence_after_sync();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host

namespace {

std::mutex g_tc_mu;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lk(g_tc_mu);
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

bool encode_maps(const ProblemDesc& p, TcMaps* m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  {
    // The map ends at row `end`: boxes reaching past it are zero-filled, so
    // base rows are never read.
    const cuuint64_t dims[2] = {(cuuint64_t)p.in_dim, (cuuint64_t)p.end};
    const cuuint64_t strides[1] = {(cuuint64_t)p.x_row_stride * 2};
    const cuuint32_t box[2] = {(cuuint32_t)TK, (cuuint32_t)TM};
    if (enc(&m->x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  for (int j = 0; j < p.n_slices; ++j) {
    const cuuint64_t dims[3] = {(cuuint64_t)p.in_dim, (cuuint64_t)p.R, (cuuint64_t)p.S};
    const cuuint64_t strides[2] = {(cuuint64_t)p.in_dim * 2, (cuuint64_t)p.sl[j].A_slot_stride * 2};
    const cuuint32_t box[3] = {(cuuint32_t)TK, (cuuint32_t)p.R, 1};
    const cuuint32_t box16[3] = {(cuuint32_t)TK, 16, 1};
    const cuuint32_t box64[3] = {(cuuint32_t)TK, (cuuint32_t)(p.R < 64 ? p.R : 64), 1};
    if (enc(&m->a[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.sl[j].A), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
    if (enc(&m->a64[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.sl[j].A), dims, strides, box64,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
    if (enc(&m->a16[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.sl[j].A), dims, strides, box16,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

template <int NR, bool PACK>
cudaError_t launch_tc_t(const ProblemDesc& p, const TcMaps& maps, float* u, cudaStream_t s, int nsplit, int nsn,
                        uint8_t* upk) {
  auto kernel = sgmv_tc_shrink_kernel<NR, PACK>;
  static unsigned long long done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(g_tc_mu);
    if (!(done & (1ull << (dev & 63)))) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<NR>::SMEM);
      if (e != cudaSuccess) return e;
      done |= 1ull << (dev & 63);
    }
  }
  const long long tiles = (long long)p.G + p.end / TM;
  const long long plane_stride = nsplit > 1 ? (long long)p.end * p.n_slices * p.R : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * nsplit * nsn));
  cfg.blockDim = dim3(TTHREADS);
  cfg.dynamicSmemBytes = TcCfg<NR>::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];  // overlap the launch with the previous kernel's tail
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return noted(cudaLaunchKernelEx(&cfg, kernel, p, maps, u, nsplit, plane_stride, nsn, upk), LORA_PATH_TC_SHRINK);
}

template <int NR>
cudaError_t launch_tc_nr(const ProblemDesc& p, const TcMaps& maps, float* u, cudaStream_t s, int nsplit, int nsn,
                         uint8_t* upk) {
  return upk ? launch_tc_t<NR, true>(p, maps, u, s, nsplit, nsn, upk)
             : launch_tc_t<NR, false>(p, maps, u, s, nsplit, nsn, nullptr);
}

}  // namespace

int tc_shrink_splits(int end, int in_dim, int sms) {
  // Split K (1, 2 or 4 planes) while a lower bound on the tiles times the
  // split stays within one CTA per SM and each split is whole stages.
  if (end <= 0 || in_dim % TK != 0) return 1;
  const long long tiles = (end + TM - 1) / TM;
  int n = 1;
  while (n < 4 && tiles * n * 2 <= sms && (in_dim / TK) % (n * 2) == 0) n *= 2;
  return n;
}

bool tc_shapes_ok(const ProblemDesc& p) {
  const int nR = p.n_slices * p.R;
  switch (nR) {
    case 16: case 32: case 48: case 64: case 96: case 128: case 192: case 256: case 384: break;
    default: return false;
  }
  return p.R % 8 == 0 && p.in_dim % TK == 0 && p.G > 0;
}

bool tc_shrink_ok(const ProblemDesc& p) {
  // Long groups only: on average at least 96 routed rows per group.
  return tc_shapes_ok(p) && p.end >= 96LL * p.G;
}

namespace {

// N (columns per CTA) = n*R / nsn.
cudaError_t launch_tc_shrink_maps(const ProblemDesc& p, const TcMaps& maps, float* u, cudaStream_t s, int nsplit,
                                  int nsn, uint8_t* upk) {
  switch (p.n_slices * p.R / nsn) {
    case 16: return launch_tc_nr<16>(p, maps, u, s, nsplit, nsn, upk);
    case 32: return launch_tc_nr<32>(p, maps, u, s, nsplit, nsn, upk);
    case 48: return launch_tc_nr<48>(p, maps, u, s, nsplit, nsn, upk);
    case 64: return launch_tc_nr<64>(p, maps, u, s, nsplit, nsn, upk);
    case 96: return launch_tc_nr<96>(p, maps, u, s, nsplit, nsn, upk);
    case 128: return launch_tc_nr<128>(p, maps, u, s, nsplit, nsn, upk);
    case 192: return launch_tc_nr<192>(p, maps, u, s, nsplit, nsn, upk);
    case 256: return launch_tc_nr<256>(p, maps, u, s, nsplit, nsn, upk);
    case 384: return launch_tc_nr<384>(p, maps, u, s, nsplit, nsn, upk);
  }
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_tc_shrink(const ProblemDesc& p, float* u, cudaStream_t s, int nsplit) {
  TcMaps maps;
  if (!encode_maps(p, &maps)) return cudaErrorNotSupported;
  return launch_tc_shrink_maps(p, maps, u, s, nsplit, 1, nullptr);
}

}  // namespace lora

// ===========================================================================
// Expand on tcgen05 for long groups (R = 64 or 128):
//   y_j[t, o] = rn(y_j[t, o] + sum_k B_j[s, o, k] u[t, j*R+k])
// Persistent: one CTA per SM.  The work is the list of units (128-row tile,
// slice j, output block of 128 columns), tile-major; CTA c takes the c-th of
// gridDim.x equal contiguous ranges, so no SM idles through a partial last
// wave and the pipeline runs across unit boundaries.  Consecutive units of
// one (tile, slice) form a segment sharing the A operand u.  Warp 0 streams
// each unit's y (two 64-column boxes) and B (R/64 boxes of 128 rows) through
// NSLOT smem slots with TMA; warp 1 issues tcgen05.mma M=128 N=128 K=2R into
// one of two TMEM buffers; warps 2-5 sum the u planes of a segment into the
// u buffer as bf16 hi | lo (K = 2R, 128-byte-swizzled K-major, one row per
// thread), then add the TMEM delta of each unit to its swizzled y block,
// round once and store the routed rows (16-byte stores; rows past the group
// are never written).  With two u buffers (R = 64) the next segment's u is
// loaded while the current one is multiplied.
// ===========================================================================
namespace lora {

namespace {

constexpr int XB = 128;         // output columns per unit (MMA N)
constexpr int XEPI = 8;         // epilogue warps: XEPI / 4 per TMEM lane quarter
constexpr int XNH = XEPI / 4;   // ... each taking XB / XNH columns of a unit
constexpr int XTHREADS = 32 * (2 + XEPI);
constexpr int RC_MAX_G = 128;   // groups cached in shared memory

// Shared memory of the expand: one u buffer, a ring of y tiles and a ring of
// B blocks.  The rings are separate because their slots live for different
// spans: a B block is free once the unit's MMAs complete, a y tile only once
// the epilogue has stored it.  The y ring (the HBM stream) gets the depth
// first -- more y loads in flight per SM is what the expand's time follows
// (a third y/B slot took the R = 64 fused-qkv apply from 108 to 98.6 us) --
// then the B ring whatever is left.  A second u buffer measured no faster
// than one.
template <int R>
struct TxCfg {
  static constexpr int KB = 2 * R / 64;                 // 64-wide K blocks of the hi|lo operand
  static constexpr int U_BYTES = KB * TM * 128;         // A operand (u hi|lo) of one segment
  static constexpr int Y_BYTES = (XB / 64) * TM * 128;  // 64-column y boxes
  static constexpr int B_BYTES = (R / 64) * XB * 128;   // R/64 boxes of XB rows x 64
  // Dynamic shared memory, the 1 KB alignment slack included; with the
  // static arrays (about 1.7 KB) within the 227 KB a CTA may hold.
  static constexpr int BUDGET = 225 * 1024;
  static constexpr int NUB = 1;
  static constexpr int fits(int ny, int nb) { return U_BYTES + ny * Y_BYTES + nb * B_BYTES + 1024 <= BUDGET; }
  static constexpr int NYS = fits(4, 2) ? 4 : (fits(3, 2) ? 3 : 2);  // y ring depth
  static constexpr int NBS = fits(NYS, 4) && NYS >= 4 ? 4 : (fits(NYS, 3) && NYS >= 3 ? 3 : 2);  // B ring
  static constexpr int SMEM = NUB * U_BYTES + NYS * Y_BYTES + NBS * B_BYTES + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * XB;
  static_assert(SMEM <= BUDGET, "expand pipeline exceeds shared memory");
};

// The routing triple as cached in shared memory: group g's rows
// [offs[g], offs[g+1]), slot ids[g], first tile tstart[g] (tstart[G] = tiles).
struct RouteCache {
  int offs[RC_MAX_G + 1];
  int ids[RC_MAX_G];
  int tstart[RC_MAX_G + 1];
};

// Tile `tile` (< tstart[G]) of the cached routing: the last group whose first
// tile is <= tile, which is never an empty group.
__device__ __forceinline__ Tile rc_tile(const RouteCache& rc, int G, int tile) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (rc.tstart[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  Tile t;
  t.g = lo;
  t.slot = rc.ids[lo];
  t.row0 = rc.offs[lo] + (tile - rc.tstart[lo]) * TM;
  t.rows = min(TM, rc.offs[lo + 1] - t.row0);
  return t;
}

}  // namespace

struct TxMaps {
  CUtensorMap y[LORA_MAX_SLICES];  // [T rows, out_j] bf16, box 64 x 128
  CUtensorMap b[LORA_MAX_SLICES];  // [S, out_j, R] bf16, box 64 x 128 x 1
};

struct TxWork {
  int nbt;                             // output blocks per tile, all slices
  int blk_begin[LORA_MAX_SLICES + 1];  // first block of each slice
  int nsplit;                          // partial planes of u
  long long plane_stride;
};

// Unit -> (tile, slice, first output column).
struct Unit {
  int tile, j, o0;
};
__device__ __forceinline__ Unit tx_unit(const TxWork& w, int n_slices, long long un) {
  Unit x;
  x.tile = (int)(un / w.nbt);
  const int b = (int)(un - (long long)x.tile * w.nbt);
  x.j = 0;
  if (n_slices > 1 && b >= w.blk_begin[1]) x.j = 1;
  if (n_slices > 2 && b >= w.blk_begin[2]) x.j = 2;
  x.o0 = (b - (x.j == 0 ? 0 : (x.j == 1 ? w.blk_begin[1] : w.blk_begin[2]))) * XB;
  return x;
}

// PACKED: u arrives packed (the tcgen05 shrink's image per (tile, slice),
// see pack_u16) and warp 0 copies each segment's image into its u buffer;
// otherwise u is fp32 [end, n*R] (nsplit planes) and the epilogue warps
// convert it.  GATHER: the batch has token_rows (the epilogue warps copy
// their blocks of the scattered y rows into the slots themselves and store
// them back through token_rows); the sorted instantiation compiles
// none of that.
template <int R, bool PACKED, bool GATHER>
__global__ void __launch_bounds__(XTHREADS, 1) sgmv_tc_expand_kernel(const __grid_constant__ ProblemDesc p,
                                                                    const __grid_constant__ TxMaps maps,
                                                                    const __grid_constant__ TxWork w,
                                                                    const float* __restrict__ u,
                                                                    const uint8_t* __restrict__ upk) {
  using Cfg = TxCfg<R>;
  constexpr int NYS = Cfg::NYS, NBS = Cfg::NBS, NUB = Cfg::NUB;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t yfull[NYS], yempty[NYS], bfull[NBS], bempty[NBS], tfull[2], tempty[2],
      uready[NUB], ufree[NUB];
  __shared__ uint32_t s_tmem;
  __shared__ RouteCache rc;
  __shared__ int s_ok, s_fail;
  __shared__ long long s_u0, s_u1;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* yring = smem + NUB * Cfg::U_BYTES;
  uint8_t* bring = yring + NYS * Cfg::Y_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;

  if (warp == 0) {
    // Validate the triple, cache it and number the tiles group by group.
    const bool valid = warp_check_routing(p);
    int base = 0;
    for (int c = 0; valid && c < G; c += 32) {
      const int g = c + lane;
      int nt = 0;
      if (g < G) {
        const int o0 = p.offs[g], o1 = p.offs[g + 1];
        rc.offs[g] = o0;
        rc.ids[g] = p.lora_ids[g];
        const int len = o1 - o0;
        nt = (len >= p.seg_lo && len < p.seg_hi) ? (len + TM - 1) / TM : 0;
      }
      int incl = nt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      if (g < G) rc.tstart[g] = base + incl - nt;
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      rc.offs[G] = p.end;
      rc.tstart[G] = base;
      // This CTA's contiguous share of the unit list.
      const long long units = valid ? (long long)base * w.nbt : 0;
      s_u0 = units * blockIdx.x / gridDim.x;
      s_u1 = units * (blockIdx.x + 1) / gridDim.x;
      s_ok = valid;
      s_fail = 0;
      for (int i = 0; i < NYS; ++i) {
        mbar_init(&yfull[i], 1);
        mbar_init(&yempty[i], XEPI);
      }
      for (int i = 0; i < NBS; ++i) {
        mbar_init(&bfull[i], 1);
        mbar_init(&bempty[i], 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&tfull[i], 1);
        mbar_init(&tempty[i], XEPI);
      }
      for (int i = 0; i < NUB; ++i) {
        mbar_init(&uready[i], PACKED ? 1 : XEPI * 32);
        mbar_init(&ufree[i], 1);
      }
      fence_mbar_init();
    }
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;
  const bool ok = s_ok != 0;
  const long long u0 = s_u0, u1 = s_u1;

  if (ok && warp == 0 && lane == 0) {
    // ---- producer: unit i's y tile into y slot i % NYS and its B block
    // into B slot i % NBS (independent of the shrink, so the first slots
    // are filled before the dependency wait); with PACKED also each
    // segment's u image into buffer seg % NUB.
    const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
    int ycur = -1, bcur = -1, nbbox = 0;
    Tile yt{}, bt{};
    auto issue_y = [&](int i, const Unit& x) {
      if (x.tile != ycur) {
        ycur = x.tile;
        yt = rc_tile(rc, G, x.tile);
      }
      uint64_t* bar = &yfull[i % NYS];
      uint8_t* ys = yring + (i % NYS) * Cfg::Y_BYTES;
      // Gathered batches: the epilogue warps copy the y rows (scattered).
      mbar_arrive_expect_tx(bar, GATHER ? 0u : (uint32_t)Cfg::Y_BYTES);
      if (!GATHER)
        for (int yb = 0; yb < XB / 64; ++yb)
          tma_load_2d_hint(ys + yb * TM * 128, &maps.y[x.j], x.o0 + yb * 64, yt.row0, bar, pol_stream);
    };
    auto issue_b = [&](int i, const Unit& x) {
      if (x.tile != bcur) {
        bcur = x.tile;
        bt = rc_tile(rc, G, x.tile);
        nbbox = (slot_kmax(p, bt.slot) + 63) / 64;
      }
      uint64_t* bar = &bfull[i % NBS];
      uint8_t* bs = bring + (i % NBS) * Cfg::B_BYTES;
      mbar_arrive_expect_tx(bar, (uint32_t)(nbbox * XB * 128));
      for (int kb = 0; kb < nbbox; ++kb)
        tma_load_3d_hint(bs + kb * XB * 128, &maps.b[x.j], kb * 64, x.o0, bt.slot, bar, pol_keep);
    };
    // Slots free at the start.
    const int pre_y = (int)min((long long)NYS, u1 - u0), pre_b = (int)min((long long)NBS, u1 - u0);
    if (PACKED) {
      for (int i = 0; i < pre_y; ++i) issue_y(i, tx_unit(w, p.n_slices, u0 + i));
      for (int i = 0; i < pre_b; ++i) issue_b(i, tx_unit(w, p.n_slices, u0 + i));
      pdl_wait();  // the packed u comes from the shrink grid
    }
    int seg = -1, seg_tile = -1, seg_j = -1;
    int i = 0;
    for (long long un = u0; un < u1; ++un, ++i) {
      const Unit x = tx_unit(w, p.n_slices, un);
      if (!PACKED || i >= pre_y) {  // the slot's previous tile has been stored
        if (i >= NYS && !mbar_wait(&yempty[i % NYS], (uint32_t)(((i / NYS) - 1) & 1))) {
          atomicOr(&s_fail, 1);
          break;
        }
        issue_y(i, x);
      }
      if (!PACKED || i >= pre_b) {  // the slot's previous block has been multiplied
        if (i >= NBS && !mbar_wait(&bempty[i % NBS], (uint32_t)(((i / NBS) - 1) & 1))) {
          atomicOr(&s_fail, 1);
          break;
        }
        issue_b(i, x);
      }
      if (PACKED && (x.tile != seg_tile || x.j != seg_j)) {
        seg_tile = x.tile;
        seg_j = x.j;
        ++seg;
        const int ub = seg % NUB;
        // The buffer's previous segment must be fully multiplied.
        if (seg >= NUB && !mbar_wait(&ufree[ub], (uint32_t)(((seg / NUB) - 1) & 1))) {
          atomicOr(&s_fail, 1);
          break;
        }
        const uint8_t* src = upk + ((long long)x.tile * p.n_slices + x.j) * Cfg::U_BYTES;
        mbar_arrive_expect_tx(&uready[ub], (uint32_t)Cfg::U_BYTES);
        for (int kb = 0; kb < Cfg::KB; ++kb)
          bulk_g2s(smem + ub * Cfg::U_BYTES + kb * TM * 128, src + kb * TM * 128, TM * 128, &uready[ub]);
      }
    }
  } else if (ok && warp == 1 && lane == 0) {
    // ---- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(TM, XB);
    int cur_tile = -1, cur_j = -1, seg = -1, kmax = 0;
    int i = 0;
    for (long long un = u0; un < u1; ++un, ++i) {
      const Unit x = tx_unit(w, p.n_slices, un);
      if (x.tile != cur_tile || x.j != cur_j) {  // new segment: wait for its u
        cur_tile = x.tile;
        cur_j = x.j;
        ++seg;
        kmax = slot_kmax(p, rc_tile(rc, G, x.tile).slot);
        if (!mbar_wait(&uready[seg % NUB], (uint32_t)((seg / NUB) & 1))) {
          atomicOr(&s_fail, 1);
          break;
        }
      }
      const int bslot = i % NBS, buf = i & 1;
      if (!mbar_wait(&bfull[bslot], (uint32_t)((i / NBS) & 1)) ||
          (i >= 2 && !mbar_wait(&tempty[buf], (uint32_t)(((i >> 1) - 1) & 1)))) {
        atomicOr(&s_fail, 1);
        break;
      }
      tc_fence_after_sync();
      const uint32_t ua = smem_addr(smem + (seg % NUB) * Cfg::U_BYTES);
      const uint32_t bs = smem_addr(bring + bslot * Cfg::B_BYTES);
      uint32_t acc = 0;
#pragma unroll
      for (int ks = 0; ks < 2 * R / 16; ++ks) {
        const int kbk = (ks * 16) % R;  // the lo half reuses B's K columns
        if (kbk >= kmax) continue;      // past the slot's rank
        const uint64_t adesc = sw128_desc(ua + (ks >> 2) * TM * 128 + (ks & 3) * 32);
        const uint64_t bdesc = sw128_desc(bs + (kbk >> 6) * XB * 128 + ((kbk & 63) >> 4) * 32);
        tc_mma_bf16(tmem + buf * XB, adesc, bdesc, idesc, acc);
        acc = 1;
      }
      tc_commit(&bempty[bslot]);  // the B slot is free once these MMAs complete
      tc_commit(&tfull[buf]);
      if (PACKED) {  // last unit of the segment: its u buffer is free once these MMAs finish
        const long long seg_end = x.j + 1 < p.n_slices ? (long long)x.tile * w.nbt + w.blk_begin[x.j + 1]
                                                       : (long long)(x.tile + 1) * w.nbt;
        if (un + 1 == min(seg_end, u1)) tc_commit(&ufree[seg % NUB]);
      }
    }
  } else if (warp >= 2) {
    // ---- epilogue warps: thread = one tile row = one TMEM lane; warps w,
    // w + 4, ... share lane quarter w % 4, warp w taking column part hf
    const int q = warp & 3;
    const int hf = (warp - 2) >> 2;  // 0 .. XNH-1
    const int row = q * 32 + lane;
    const int nR = p.n_slices * R;
    if (ok) {
      if (!PACKED) pdl_wait();  // u comes from the shrink grid
      // A warp whose wait expired keeps walking the barrier protocol (doing
      // no work) so the other roles never block on it.
      bool bad = false;
      // fp32 u of segment s -> bf16 hi | lo in buffer s % NUB, in two steps.
      // stage_u: 16-byte async copies put the fp32 values of columns
      // k .. k+7 of this thread's row where their hi chunk (k .. k+3) and lo
      // chunk (k+4 .. k+7) will live, so finish_u converts every 8-column
      // group in place.  finish_u adds planes 1.. (plane order), converts and
      // arrives on uready.
      auto stage_u = [&](int s, const Tile& ts, int js) {
        uint8_t* Ub = smem + (s % NUB) * Cfg::U_BYTES;
        if (!bad && row < ts.rows) {
          const float* ur = u + (long long)(ts.row0 + row) * nR + (long long)js * R;
#pragma unroll
          for (int m = hf * R / (8 * XNH); m < (hf + 1) * R / (8 * XNH); ++m) {
            cp_async16(Ub + sw128_offset(row, 8 * m), ur + 8 * m);
            cp_async16(Ub + sw128_offset(row, R + 8 * m), ur + 8 * m + 4);
          }
        }
        cp_async_commit();
      };
      auto finish_u = [&](int s, const Tile& ts, int js) {
        uint8_t* Ub = smem + (s % NUB) * Cfg::U_BYTES;
        const bool live = !bad && row < ts.rows;
        const float* ur = u + (long long)(ts.row0 + (live ? row : 0)) * nR + (long long)js * R;
        for (int m = hf * R / (8 * XNH); m < (hf + 1) * R / (8 * XNH); ++m) {
          uint4* ph = reinterpret_cast<uint4*>(Ub + sw128_offset(row, 8 * m));
          uint4* pl = reinterpret_cast<uint4*>(Ub + sw128_offset(row, R + 8 * m));
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
          if (live) {
            a = *reinterpret_cast<const float4*>(ph);
            b = *reinterpret_cast<const float4*>(pl);
            for (int sp = 1; sp < w.nsplit; ++sp) {
              const float4 c = __ldcg(reinterpret_cast<const float4*>(ur + sp * w.plane_stride + 8 * m));
              const float4 d = __ldcg(reinterpret_cast<const float4*>(ur + sp * w.plane_stride + 8 * m + 4));
              a.x += c.x;
              a.y += c.y;
              a.z += c.z;
              a.w += c.w;
              b.x += d.x;
              b.y += d.y;
              b.z += d.z;
              b.w += d.w;
            }
          }
          const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_hi_lo_bf16x2(v[2 * e], v[2 * e + 1], hi[e], lo[e]);
          *ph = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *pl = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        fence_proxy_async_smem();  // generic writes -> visible to the tensor cores
        mbar_arrive(&uready[s % NUB]);
      };

      const uint64_t pol_stream = policy_evict_first();
      constexpr bool gathered = GATHER;
      int cur_tile = -1, cur_j = -1, seg = -1, kmax = 0;
      int yrow = 0;            // gathered: the y row of this thread's tile position
      bool tile_skip = false;  // gathered: the tile has an out-of-range entry
      Tile t{};
      // Gathered: each warp copies its own block of a unit's y tile (32 rows
      // x XB / XNH columns, eight lanes per row, 16-byte async copies into
      // the slot's swizzled layout) two units ahead, one copy group per unit;
      // rows past the tile or out of range are not copied (such a tile is
      // skipped below).  The slot's previous unit (NYS >= 3 units back) was
      // stored by this same warp.
      // The y rows this lane copies (tile positions 32 q + lane / 8 + 4 it) are
      // looked up once per tile.
      int gtile = -1;
      int grow[8];
#pragma unroll
      for (int it = 0; it < 8; ++it) grow[it] = -1;
      auto gather_y = [&](int iu, long long un_) {
        if (un_ < u1 && !bad) {
          const Unit xu = tx_unit(w, p.n_slices, un_);
          if (xu.tile != gtile) {
            gtile = xu.tile;
            const Tile tu = rc_tile(rc, G, xu.tile);
#pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int r = q * 32 + (lane >> 3) + 4 * it;
              const int yr = r < tu.rows ? p.token_rows[tu.row0 + r] : -1;
              grow[it] = (yr >= 0 && yr < p.num_tokens) ? yr : -1;
            }
          }
          const SliceDesc& su = p.sl[xu.j];
          uint8_t* yb = yring + (iu % NYS) * Cfg::Y_BYTES + hf * TM * 128;
          const __nv_bfloat16* yg = static_cast<const __nv_bfloat16*>(su.y);
          const int c = lane & 7;
          const int col = xu.o0 + hf * (XB / XNH) + c * 8;
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int r = q * 32 + (lane >> 3) + 4 * it;
            if (grow[it] >= 0 && col < su.out_dim)
              cp_async16(yb + r * 128 + ((c ^ (r & 7)) << 4), yg + (long long)grow[it] * su.y_row_stride + col);
          }
        }
        cp_async_commit();
      };
      if constexpr (gathered) {
        static_assert(NYS >= 3, "gathered y tiles are copied two units ahead");
        gather_y(0, u0);
        gather_y(1, u0 + 1);
      }
      int i = 0;
      for (long long un = u0; un < u1; ++un, ++i) {
        const Unit x = tx_unit(w, p.n_slices, un);
        if (x.tile != cur_tile || x.j != cur_j) {
          // New segment.  Every MMA of the previous segment has completed
          // (its TMEM results were all consumed), so the u buffer it read is
          // free: fill this segment's buffer if it was not prefetched, then
          // prefetch the next segment's into the freed one.
          if (x.tile != cur_tile) {
            t = rc_tile(rc, G, x.tile);
            if constexpr (gathered) {  // every warp checks the whole tile: the same outcome everywhere
              int badrow = 0;
              for (int r = lane; r < t.rows; r += 32) {
                const int v = p.token_rows[t.row0 + r];
                if (v < 0 || v >= p.num_tokens) badrow = 1;
              }
              tile_skip = __any_sync(0xffffffffu, badrow) != 0;
              if (tile_skip && lane == 0) atomicOr(p.status, LORA_DEV_BAD_ROW);
              yrow = (!tile_skip && row < t.rows) ? p.token_rows[t.row0 + row] : 0;
            }
          }
          cur_tile = x.tile;
          cur_j = x.j;
          ++seg;
          kmax = slot_kmax(p, t.slot);
          if (!PACKED) {
            if (NUB == 1 || seg == 0) stage_u(seg, t, x.j);
            bool staged_next = false;
            if (NUB == 2) {  // the next segment's u loads while this one is multiplied
              const long long next = x.j + 1 < p.n_slices ? (long long)x.tile * w.nbt + w.blk_begin[x.j + 1]
                                                          : (long long)(x.tile + 1) * w.nbt;
              if (next < u1) {
                const Unit nx = tx_unit(w, p.n_slices, next);
                stage_u(seg + 1, nx.tile == x.tile ? t : rc_tile(rc, G, nx.tile), nx.j);
                staged_next = true;
              }
            }
            if (staged_next) cp_async_wait<1>();
            else cp_async_wait<0>();
            finish_u(seg, t, x.j);
          }
        }
        const SliceDesc& sl = p.sl[x.j];
        const bool live = row < t.rows;
        const int yslot = i % NYS, buf = i & 1;
        if constexpr (gathered) {  // this unit's y block has landed; unit i + 2's copies start
          gather_y(i + 2, un + 2);
          cp_async_wait<2>();
          __syncwarp();  // the block was copied by the warp's other lanes
        }
        if (!bad && (!mbar_wait(&tfull[buf], (uint32_t)((i >> 1) & 1)) ||
                     !mbar_wait(&yfull[yslot], (uint32_t)((i / NYS) & 1)))) {
          atomicOr(&s_fail, 1);
          bad = true;
        }
        bad = __any_sync(0xffffffffu, bad);  // tcgen05.ld below needs the whole warp
        tc_fence_after_sync();
        uint8_t* ys = yring + yslot * Cfg::Y_BYTES;
        const int o0 = x.o0;
        const int ovalid = min(XB, sl.out_dim - o0);
        // 32 columns per TMEM load: two 16-column groups.
        const bool work = !bad && !tile_skip;
#pragma unroll 1
        for (int cc = 0; cc < XB / (32 * XNH); ++cc) {
          if (!work) break;
          const int c32 = hf * (XB / (32 * XNH)) + cc;
          float dd[32];
          if (kmax > 0) {
            tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * XB + c32 * 32), dd);
          } else {  // rank 0: no MMA was issued for this unit, the delta is zero
#pragma unroll
            for (int e = 0; e < 32; ++e) dd[e] = 0.f;
          }
#pragma unroll
          for (int g16 = 0; g16 < 2; ++g16) {
            const int c16 = c32 * 2 + g16;
            float* d = dd + 16 * g16;
            if (sl.bias && c16 * 16 < ovalid) {  // bias joins the delta before the one rounding
              const uint4* bp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(sl.bias) +
                                                               (long long)t.slot * sl.bias_slot_stride + o0 + c16 * 16);
              const uint4 b0 = __ldg(bp);
              const uint4 b1 = (c16 * 16 + 8 < ovalid) ? __ldg(bp + 1) : make_uint4(0, 0, 0, 0);
              const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                d[2 * e] += __uint_as_float(bw[e] << 16);
                d[2 * e + 1] += __uint_as_float(bw[e] & 0xFFFF0000u);
              }
            }
            if (live && c16 * 16 < ovalid) {
              // y + delta, rounded once, written back over y in the slot.
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int cch = c16 * 2 + h;  // 16-byte chunk of the 128-column block
                uint4* py = reinterpret_cast<uint4*>(ys + (cch >> 3) * TM * 128 + row * 128 + (((cch & 7) ^ (row & 7)) << 4));
                const uint4 yv = *py;
                const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w};
                uint32_t out[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 yy = make_float2(__uint_as_float(yw[e] << 16), __uint_as_float(yw[e] & 0xFFFF0000u));
                  const float2 r = add_f32x2(yy, make_float2(d[h * 8 + 2 * e], d[h * 8 + 2 * e + 1]));
                  out[e] = round_pack_bf16x2(r.x, r.y);
                }
                *py = make_uint4(out[0], out[1], out[2], out[3]);
              }
            }
          }
        }
        __syncwarp();
        // This warp's 32 rows x XB / XNH columns to y: eight lanes per row,
        // so each store instruction writes whole 128-byte row segments.
        if (work) {
          constexpr int CPR = XB / XNH / 8;   // 16-byte chunks per row
          constexpr int RPI = 32 / CPR;       // rows per store instruction
          const int cch = hf * CPR + lane % CPR;  // this lane's chunk of the 128-column block
          const int r0 = q * 32 + lane / CPR;     // this lane's first tile row
          const uint8_t* sbase = ys + (cch >> 3) * TM * 128;
          if constexpr (gathered) {
            __nv_bfloat16* ybase = static_cast<__nv_bfloat16*>(sl.y) + o0 + cch * 8;
#pragma unroll
            for (int it = 0; it < CPR; ++it) {
              const int tr = r0 + it * RPI;
              const int yr = __shfl_sync(0xffffffffu, yrow, tr - q * 32);  // held by lane tr - 32 q
              if (tr < t.rows && cch * 8 < ovalid)
                st_global_v4_hint(reinterpret_cast<uint4*>(ybase + (long long)yr * sl.y_row_stride),
                                  *reinterpret_cast<const uint4*>(sbase + tr * 128 + (((cch & 7) ^ (tr & 7)) << 4)),
                                  pol_stream);
            }
          } else {
            uint4* gp = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(sl.y) +
                                                 (long long)(t.row0 + r0) * sl.y_row_stride + o0 + cch * 8);
            const long long gstep = (long long)RPI * sl.y_row_stride / 8;  // uint4 per RPI rows
            if (cch * 8 < ovalid) {
#pragma unroll
              for (int it = 0; it < CPR; ++it, gp += gstep) {
                const int tr = r0 + it * RPI;
                if (tr < t.rows)
                  st_global_v4_hint(gp, *reinterpret_cast<const uint4*>(sbase + tr * 128 + (((cch & 7) ^ (tr & 7)) << 4)),
                                    pol_stream);
              }
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&tempty[buf]);
          mbar_arrive(&yempty[yslot]);
        }
      }
    }
  }
  pdl_launch_dependents();  // the next kernel may launch; it waits for this grid to finish
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    if (s_fail) {
      for (int i = 0; i < 2; ++i) (void)mbar_wait(&tfull[i], 0);
      if (lane == 0) atomicOr(p.status, LORA_DEV_TIMEOUT);
    }
    tc_fence_after_sync();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

namespace {

bool encode_tx_maps(const ProblemDesc& p, TxMaps* m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  for (int j = 0; j < p.n_slices; ++j) {
    const SliceDesc& sl = p.sl[j];
    {
      // Ends at row `end` (zero-filled past it): base rows are never read.
      const cuuint64_t dims[2] = {(cuuint64_t)sl.out_dim, (cuuint64_t)p.end};
      const cuuint64_t strides[1] = {(cuuint64_t)sl.y_row_stride * 2};
      const cuuint32_t box[2] = {64, (cuuint32_t)TM};
      if (enc(&m->y[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, sl.y, dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    }
    {
      const cuuint64_t dims[3] = {(cuuint64_t)p.R, (cuuint64_t)sl.out_dim, (cuuint64_t)p.S};
      const cuuint64_t strides[2] = {(cuuint64_t)p.R * 2, (cuuint64_t)sl.B_slot_stride * 2};
      const cuuint32_t box[3] = {64, (cuuint32_t)XB, 1};
      if (enc(&m->b[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(sl.B), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    }
  }
  return true;
}

template <int R, bool PACKED, bool GATHER>
cudaError_t launch_tx_g(const ProblemDesc& p, const TxMaps& maps, const TxWork& w, const float* u,
                        const uint8_t* upk, cudaStream_t s, bool pdl) {
  auto kernel = sgmv_tc_expand_kernel<R, PACKED, GATHER>;
  static unsigned long long done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(g_tc_mu);
    if (!(done & (1ull << (dev & 63)))) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TxCfg<R>::SMEM);
      if (e != cudaSuccess) return e;
      done |= 1ull << (dev & 63);
    }
  }
  // Persistent: one CTA per SM, or fewer when there are fewer units.
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long units_max = ((long long)p.G + p.end / TM) * w.nbt;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max(1LL, std::min<long long>(sms, units_max)));
  cfg.blockDim = dim3(XTHREADS);
  cfg.dynamicSmemBytes = TxCfg<R>::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return noted(cudaLaunchKernelEx(&cfg, kernel, p, maps, w, u, upk), LORA_PATH_TC_EXPAND);
}

template <int R, bool PACKED>
cudaError_t launch_tx_t(const ProblemDesc& p, const TxMaps& maps, const TxWork& w, const float* u,
                        const uint8_t* upk, cudaStream_t s, bool pdl) {
  return p.token_rows ? launch_tx_g<R, PACKED, true>(p, maps, w, u, upk, s, pdl)
                      : launch_tx_g<R, PACKED, false>(p, maps, w, u, upk, s, pdl);
}

TxWork make_tx_work(const ProblemDesc& p, int nsplit) {
  TxWork w{};
  int acc = 0;
  for (int j = 0; j < p.n_slices; ++j) {
    w.blk_begin[j] = acc;
    acc += (p.sl[j].out_dim + XB - 1) / XB;
  }
  w.blk_begin[p.n_slices] = acc;
  w.nbt = acc;
  w.nsplit = nsplit;
  w.plane_stride = (long long)p.end * p.n_slices * p.R;
  return w;
}

bool nr_supported(int n) {
  switch (n) {
    case 16: case 32: case 48: case 64: case 96: case 128: case 192: case 256: case 384: return true;
  }
  return false;
}

}  // namespace

bool tc_expand_shapes_ok(const ProblemDesc& p) {
  return (p.R == 64 || p.R == 128) && p.G <= RC_MAX_G && tc_shapes_ok(p);
}

bool tc_expand_ok(const ProblemDesc& p) { return tc_expand_shapes_ok(p) && tc_shrink_ok(p); }

cudaError_t launch_tc_expand(const ProblemDesc& p, const float* u, cudaStream_t s, bool pdl, int nsplit) {
  TxMaps maps;
  if (!encode_tx_maps(p, &maps)) return cudaErrorNotSupported;
  const TxWork w = make_tx_work(p, nsplit);
  if (p.R == 64) return launch_tx_t<64, false>(p, maps, w, u, nullptr, s, pdl);
  return launch_tx_t<128, false>(p, maps, w, u, nullptr, s, pdl);
}

size_t tc_packed_bytes(int S, int end, int n_slices, int R) {
  if (R != 64 && R != 128) return 0;
  const long long tiles = (long long)S + (end > 0 ? end : 0) / TM;
  return (size_t)tiles * n_slices * 4 * R * TM;
}

int tc_pack_splits(const ProblemDesc& p) {
  // Column parts of the packed shrink: split the n*R columns (whole 16-column
  // groups, a supported tile width) while a lower bound on the tiles times
  // the parts stays within one CTA per SM of this device.
  const int nR = p.n_slices * p.R;
  const long long tiles = (p.end + TM - 1) / TM;
  const int sms = device_sm_count();
  int n = 1;
  while (n < 4 && tiles * n * 2 <= sms && nR % (32 * n) == 0 && nr_supported(nR / (2 * n))) n *= 2;
  return n;
}

// Ring of a K-split CTA: the full-depth ring (one CTA per SM), or a shallow
// one that two CTAs per SM hold (~112 KB each).
template <int NR>
constexpr int shallow_stages() {
  return (112 * 1024 - 1024) / TcCfg<NR>::STAGE;
}

template <int NR, int CL, int NST>
cudaError_t launch_ksplit_t(const ProblemDesc& p, const TcMaps& maps, uint8_t* upk, cudaStream_t s, int nsn) {
  auto kernel = sgmv_tc_shrink_ksplit_kernel<NR, CL, NST>;
  constexpr int SMEM = NST * TcCfg<NR>::STAGE + 1024;
  static unsigned long long done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(g_tc_mu);
    if (!(done & (1ull << (dev & 63)))) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
      if (e != cudaSuccess) return e;
      done |= 1ull << (dev & 63);
    }
  }
  const long long tiles = (long long)p.G + p.end / TM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * CL * nsn));
  cfg.blockDim = dim3(TTHREADS);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return noted(cudaLaunchKernelEx(&cfg, kernel, p, maps, upk, nsn), LORA_PATH_TC_SHRINK);
}

template <int NR, int CL>
cudaError_t launch_ksplit_nr(const ProblemDesc& p, const TcMaps& maps, uint8_t* upk, cudaStream_t s, int nsn,
                             bool shallow) {
  if constexpr (shallow_stages<NR>() >= 2 && (CL - 1) * TM * (NR / CL) * 4 <= shallow_stages<NR>() * TcCfg<NR>::STAGE) {
    if (shallow) return launch_ksplit_t<NR, CL, shallow_stages<NR>()>(p, maps, upk, s, nsn);
  }
  if (shallow) return cudaErrorNotSupported;
  return launch_ksplit_t<NR, CL, TcCfg<NR>::NSTAGE>(p, maps, upk, s, nsn);
}

// The packed shrink with K split over a cluster of `cl` CTAs per tile and
// the n*R columns in `nsn` parts (NR = n*R / nsn per CTA); `shallow` picks
// the two-CTAs-per-SM ring.  cudaErrorNotSupported for other shapes.
cudaError_t launch_ksplit(const ProblemDesc& p, const TcMaps& maps, uint8_t* upk, cudaStream_t s, int cl, int nsn,
                          bool shallow) {
  const int nR = p.n_slices * p.R / nsn;
  if (p.in_dim % (cl * TK) != 0 || (p.n_slices * p.R) % nsn != 0) return cudaErrorNotSupported;
  if (cl == 2) {
    switch (nR) {
      case 64: return launch_ksplit_nr<64, 2>(p, maps, upk, s, nsn, shallow);
      case 128: return launch_ksplit_nr<128, 2>(p, maps, upk, s, nsn, shallow);
      case 192: return launch_ksplit_nr<192, 2>(p, maps, upk, s, nsn, shallow);
      case 256: return launch_ksplit_nr<256, 2>(p, maps, upk, s, nsn, shallow);
      case 384: return launch_ksplit_nr<384, 2>(p, maps, upk, s, nsn, shallow);
    }
  } else if (cl == 4) {
    switch (nR) {
      case 64: return launch_ksplit_nr<64, 4>(p, maps, upk, s, nsn, shallow);
      case 128: return launch_ksplit_nr<128, 4>(p, maps, upk, s, nsn, shallow);
      case 192: return launch_ksplit_nr<192, 4>(p, maps, upk, s, nsn, shallow);
      case 256: return launch_ksplit_nr<256, 4>(p, maps, upk, s, nsn, shallow);
      case 384: return launch_ksplit_nr<384, 4>(p, maps, upk, s, nsn, shallow);
    }
  }
  return cudaErrorNotSupported;
}

cudaError_t launch_tc_apply_packed(const ProblemDesc& p, void* workspace, cudaStream_t s) {
  TcMaps smaps;
  TxMaps xmaps;
  if (!encode_maps(p, &smaps) || !encode_tx_maps(p, &xmaps)) return cudaErrorNotSupported;
  // Fill the SMs.  Few tiles: split K over a cluster of CTAs per tile (x read
  // once) rather than the tile's columns (x read once per column part), one
  // CTA per SM.  Up to two tiles per SM: K split over CTA pairs with shallow
  // rings, two CTAs per SM.  Otherwise one CTA per tile.
  const int nsn = tc_pack_splits(p);
  uint8_t* upk = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaErrorNotSupported;
  {
    const long long tiles_lb = (p.end + TM - 1) / TM;
    if (nsn > 1) e = launch_ksplit(p, smaps, upk, s, nsn, 1, false);
    else if (tiles_lb * 2 <= 2LL * device_sm_count()) e = launch_ksplit(p, smaps, upk, s, 2, 1, true);
  }
  if (e == cudaErrorNotSupported) e = launch_tc_shrink_maps(p, smaps, nullptr, s, 1, nsn, upk);
  if (e != cudaSuccess) return e;
  const TxWork w = make_tx_work(p, 1);
  if (p.R == 64) return launch_tx_t<64, true>(p, xmaps, w, nullptr, upk, s, true);
  return launch_tx_t<128, true>(p, xmaps, w, nullptr, upk, s, true);
}

}  // namespace lora
