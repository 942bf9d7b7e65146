// sgmv_decode.cu -- SGMV for short groups (decode-sized batches) with the
// shrink's operands brought in by the tensor memory accelerator, and the
// one-launch apply.
//
//   shrink  u_c[t, j*R+k] = sum_{i in K split c} A_j[s, k, i] x[t, i]
//   expand  y_j[t, o]     = rn(y_j[t, o] + sum_k B_j[s, o, k] sum_c u_c[t, j*R+k])
// for the routed rows t of a group with slot s ("vLLM LoRA 实现深度解析"
// sections 1 and 6; routing triple of the "max.pipelines.lora.LoRAManagerV3"
// page, get_lora_graph_inputs).
//
// Shrink work item: (64-row tile of a group, K split c), all n*R <= 96
// intermediate columns.  One thread issues, per 64-wide K stage, one TMA box
// of 16 x rows per 16 routed rows of the tile (rows past the group belong to
// the next group, rows at or past `end` are zero-filled by the tensor map:
// neither is stored) and one box of the slot's R A rows per slice, all with
// the 128-byte swizzle; every stage of the split is in flight at once when
// the ring holds them.  The tensor memory accelerator keeps tens of
// kilobytes per CTA in flight without occupying the load/store unit, which
// is what bounds a decode shrink (a few kilobytes per row, a few rows per
// group).  Four warps multiply their 16 rows on the tensor cores (mma.sync
// m16n8k16, fp32 accumulate) from the swizzled stages (ldmatrix), and the
// partial tile is stored as plane c of the intermediate.
//
// sgmv_shrink_tma_kernel: one shrink item per CTA; the mma.sync expand
// kernel, launched after it, sums the planes.
//
// sgmv_decode_apply_kernel: shrink and expand in one cooperative launch (all
// CTAs resident).  CTA b takes shrink items b, b + grid, ... and then expand
// items b, b + grid, ... (expand item: 64-row tile, 256 output columns of one
// slice).  Before its shrink work a CTA starts the 16-byte asynchronous
// copies of its first expand item's y block and B block.  A tile's K splits
// hand their planes to its expand items through one 32-bit counter per tile
// in the workspace: each split, after storing its plane, adds 1 (release);
// each expand item waits (acquire, bounded) until the low half counts every
// split, sums the planes, and adds 1 << 16.  The participant whose addition
// completes the count (splits + expand items << 16) stores zero, so the
// counters are zero again when the launch ends, even if a wait ran out (the
// waiter still adds its count; the late split completes it).  Every CTA does
// its shrink items before it waits, and all CTAs are resident, so every wait
// ends.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tiles.cuh"

namespace lora {

namespace {

constexpr int DT = 64;           // token rows per tile
constexpr int DK = 64;           // K per stage (one 128-byte swizzle row)
constexpr int XBOX = 16;         // rows per x box
constexpr int MAX_STAGES = 8;
constexpr int EOB = 256;         // output columns per expand item
constexpr int ETHREADS = 256;    // one-launch apply: 8 warps

template <int NR>
struct DecCfg {
  static constexpr int X_BYTES = DT * DK * 2;             // 8 KB: up to 4 boxes of 16 rows
  static constexpr int A_BYTES = NR * DK * 2;             // all slices' rank rows
  static constexpr int STAGE = X_BYTES + ((A_BYTES + 1023) / 1024) * 1024;
  static constexpr int PPITCH = NR + 4;                   // floats per staged partial row
  static constexpr int P_BYTES = DT * PPITCH * 4;         // the partial tile, staged over the ring
};

// Expand item buffers of the one-launch apply (rank R, 64 rows x 256 columns).
template <int R>
struct DexCfg {
  static constexpr int YPITCH = EOB * 2 + 16;             // bytes per staged y row
  // Rank 16: 32-byte B rows, the two 16-byte chunks swapped when bit 2 of the
  // row is set (the 8 rows of an ldmatrix phase then hit 8 bank groups);
  // rank 32: 64-byte rows padded by 16 bytes.
  static constexpr bool BSWZ = R == 16;
  static constexpr int BPITCH = BSWZ ? 32 : R * 2 + 16;
  __device__ static constexpr int b_off(int o, int ch) {
    return o * BPITCH + (BSWZ ? (ch ^ ((o >> 2) & 1)) : ch) * 16;
  }
  static constexpr int UPITCH = 4 * R + 16;               // bytes per hi|lo row (2R bf16)
  static constexpr int Y_BYTES = DT * YPITCH;
  static constexpr int B_BYTES = EOB * BPITCH;
  static constexpr int H_BYTES = DT * UPITCH;
  static constexpr int BYTES = Y_BYTES + B_BYTES + H_BYTES;
};

// Byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled block
// (what a TMA box of 64 bf16 columns with the 128-byte swizzle writes, the
// block starting on a 1024-byte boundary).
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Polls of a tile counter before a wait gives up: the first 256 back to
// back, then 128 ns apart (each poll itself an L2 round trip): about one
// second in all.
constexpr uint32_t kCounterPolls = 1u << 21;

}  // namespace

struct DecMaps {
  CUtensorMap x;                   // [end rows, in] bf16, box 64 x 16
  CUtensorMap a[LORA_MAX_SLICES];  // per slice [S, R, in] bf16, box 64 x R x 1
};

// ------------------------------------------------------ tile counter handoff

// One K split of tile `tile` has stored its plane (every thread of the CTA
// passed a barrier after its stores).  Called by one thread.
__device__ __forceinline__ void tile_arrive_split(unsigned* ctrl, long long tile, unsigned total) {
  __threadfence();
  const unsigned old = atomicAdd(ctrl + tile, 1u);
  if (old + 1u == total) ctrl[tile] = 0u;  // last participant: leave the counter zero
}

// One expand item of the tile has read the planes (or given up).  One thread.
__device__ __forceinline__ void tile_arrive_reader(unsigned* ctrl, long long tile, unsigned total) {
  const unsigned old = atomicAdd(ctrl + tile, 1u << 16);
  if (old + (1u << 16) == total) ctrl[tile] = 0u;
}

// Wait until all `splits` K splits of the tile have arrived.  One thread;
// false if the poll budget ran out.
__device__ __forceinline__ bool tile_wait_splits(const unsigned* ctrl, long long tile, unsigned splits,
                                                 uint32_t polls) {
  for (uint32_t i = 0; i < polls; ++i) {
    if ((ld_acquire_gpu(ctrl + tile) & 0xFFFFu) >= splits) return true;
    if (i >= 256) __nanosleep(128);
  }
  return false;
}

// ------------------------------------------------------------ shrink item

// One shrink item: K split c of tile t into plane c.  Thread 0 issues the
// copies; warps 0-3 multiply; all NTH threads store.  `full` holds nstage
// barriers initialised (fresh) for this item.  Returns false on every thread
// if a stage never arrived (nothing is stored then).
template <int NR, int NTH>
__device__ __forceinline__ bool dec_shrink_tile(const ProblemDesc& p, const DecMaps& maps, uint8_t* smem,
                                                uint64_t* full, const Tile& t, int c, int Kc, int nstage,
                                                float* __restrict__ u, long long plane_stride) {
  using Cfg = DecCfg<NR>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.R;
  const int k0 = c * Kc;
  const int nst = Kc / DK;
  const int nxb = (t.rows + XBOX - 1) / XBOX;  // x boxes per stage
  const uint32_t stage_tx = (uint32_t)(nxb * XBOX * DK * 2 + p.n_slices * R * DK * 2);

  auto issue = [&](int s) {
    const int slot = s % nstage;
    uint8_t* xs = smem + slot * Cfg::STAGE;
    uint8_t* as = xs + Cfg::X_BYTES;
    const int kk = k0 + s * DK;
    const uint64_t pol_x = policy_evict_first(), pol_a = policy_evict_last();
    mbar_arrive_expect_tx(&full[slot], stage_tx);
    for (int b = 0; b < nxb; ++b)
      tma_load_2d_hint(xs + b * XBOX * 128, &maps.x, kk, t.row0 + b * XBOX, &full[slot], pol_x);
    for (int j = 0; j < p.n_slices; ++j)
      tma_load_3d_hint(as + j * R * 128, &maps.a[j], kk, 0, t.slot, &full[slot], pol_a);
  };

  if (threadIdx.x == 0)
    for (int s = 0; s < nstage && s < nst; ++s) issue(s);

  float acc[NR / 8][4];
#pragma unroll
  for (int i = 0; i < NR / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const bool active = warp < 4 && warp * 16 < t.rows;  // warp-uniform
  int fail = 0;
  for (int s = 0; s < nst; ++s) {
    const int slot = s % nstage;
    if (warp < 4 && !fail && !mbar_wait(&full[slot], (uint32_t)((s / nstage) & 1))) fail = 1;
    if (active && !fail) {
      const uint32_t xs = smem_addr(smem + slot * Cfg::STAGE);
      const uint32_t as = xs + Cfg::X_BYTES;
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) {
        uint32_t a[4];
        const int ar = warp * 16 + (lane & 15);
        ldsm_x4(xs + swz(ar, ks * 2 + (lane >> 4)), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int np = 0; np < NR / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          const int nrow = np * 16 + (lane & 7) + ((lane >> 4) << 3);
          ldsm_x4(as + swz(nrow, ks * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
          mma_bf16_16816(acc[2 * np], a, b0, b1);
          mma_bf16_16816(acc[2 * np + 1], a, b2, b3);
        }
      }
    }
    if (s + nstage < nst) {  // ring smaller than the split: refill this slot
      __syncthreads();
      if (threadIdx.x == 0 && !fail) issue(s + nstage);
    }
  }
  if (__syncthreads_or(fail)) {
    // A copy never arrived: give the ones in flight a bounded chance to land
    // before the shared memory is reused, flag the launch, store nothing.
    if (threadIdx.x == 0) {
      for (int i = 0; i < nstage && i < nst; ++i) {
        const int last = i + ((nst - 1 - i) / nstage) * nstage;  // last stage using slot i
        (void)mbar_wait_limit(&full[i], (uint32_t)((last / nstage) & 1), 1u << 12);
      }
      atomicOr(p.status, LORA_DEV_TIMEOUT);
    }
    return false;
  }

  // Partial tile -> shared memory (over the ring: every stage has been read).
  float* P = reinterpret_cast<float*>(smem);
  if (active) {
    const int g = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NR / 8; ++nt) {
      const int row = warp * 16 + g, col = nt * 8 + 2 * tq;
      *reinterpret_cast<float2*>(&P[row * Cfg::PPITCH + col]) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(&P[(row + 8) * Cfg::PPITCH + col]) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  __syncthreads();
  float* up = u + c * plane_stride;
  constexpr int Q4 = NR / 4;
  for (int e = threadIdx.x; e < t.rows * Q4; e += NTH) {
    const int r = e / Q4, cc = (e % Q4) * 4;
    *reinterpret_cast<float4*>(&up[(long long)(t.row0 + r) * NR + cc]) =
        *reinterpret_cast<const float4*>(&P[r * Cfg::PPITCH + cc]);
  }
  return true;
}

// grid.x = tiles_max * C.  CTA (tile, c): K range [c*Kc, (c+1)*Kc) in Kc/64
// stages through a ring of nstage slots; partial tile -> plane c.
template <int NR>
__global__ void __launch_bounds__(128) sgmv_shrink_tma_kernel(const __grid_constant__ ProblemDesc p,
                                                              const __grid_constant__ DecMaps maps,
                                                              float* __restrict__ u, int C, int Kc, int nstage,
                                                              long long plane_stride) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[MAX_STAGES];
  __shared__ Tile s_tile;
  __shared__ int s_ok;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  // Programmatic dependent of the preceding kernel: no global memory is
  // touched before it has completed.
  pdl_wait();
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = (int)(blockIdx.x % (unsigned)C);
  const long long tile = blockIdx.x / (unsigned)C;
  if (warp == 0) {
    Tile t{};
    const bool ok = warp_locate_tile(p, DT, tile, t);
    if (lane == 0) {
      s_tile = t;
      s_ok = ok;
      for (int i = 0; i < nstage; ++i) mbar_init(&full[i], 1);
      fence_mbar_init();
    }
  }
  __syncthreads();
  if (!s_ok) return;
  (void)dec_shrink_tile<NR, 128>(p, maps, smem, full, s_tile, c, Kc, nstage, u, plane_stride);
}

// ------------------------------------------------------ one-launch apply

struct DexWork {
  int C, Kc, nstage;
  long long plane_stride;
  int n_shrink, n_expand;             // items (upper bounds from G + end/64 tiles)
  int n_ob_total;                     // expand items per tile, all slices
  int ob_begin[LORA_MAX_SLICES + 1];  // first expand item of each slice within a tile
  int ring_bytes;                     // dynamic shared memory of the shrink ring (1024-aligned)
};

template <int NR, int R>
__global__ void __launch_bounds__(ETHREADS, 2) sgmv_decode_apply_kernel(const __grid_constant__ ProblemDesc p,
                                                                     const __grid_constant__ DecMaps maps,
                                                                     const __grid_constant__ DexWork w,
                                                                     float* __restrict__ u, unsigned* ctrl) {
  using X = DexCfg<R>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[MAX_STAGES];
  __shared__ Tile s_tile[2];
  __shared__ int s_ok[2];
  __shared__ int s_go;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Ys = ring + w.ring_bytes;
  uint8_t* Bs = Ys + X::Y_BYTES;
  uint8_t* Hs = Bs + X::B_BYTES;

  pdl_wait();  // the preceding kernel has completed: its writes are visible

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned total = (unsigned)w.C + ((unsigned)w.n_ob_total << 16);
  const long long first_e = blockIdx.x;

  // Locate this CTA's first shrink tile (warp 0) and first expand tile (warp 1).
  if (warp < 2) {
    const long long item = first_e;
    const bool has = warp == 0 ? item < w.n_shrink : item < w.n_expand;
    const long long tile = warp == 0 ? item / w.C : item / w.n_ob_total;
    Tile t{};
    const bool ok = has && warp_locate_tile(p, DT, tile, t);
    if (lane == 0) {
      s_tile[warp] = t;
      s_ok[warp] = ok;
    }
  }
  __syncthreads();

  // Expand item -> (tile, slice, first column).
  auto e_decode = [&](long long item, int& j, int& o0) {
    const int obg = (int)(item % w.n_ob_total);
    j = 0;
    while (j + 1 < p.n_slices && obg >= w.ob_begin[j + 1]) ++j;
    o0 = (obg - w.ob_begin[j]) * EOB;
  };
  // Start the asynchronous copies of an expand item's y block (routed rows
  // only) and the slot's B block.
  auto e_prefetch = [&](const Tile& t, int j, int o0) {
    const SliceDesc& sl = p.sl[j];
    const int ovalid = min(EOB, sl.out_dim - o0);
    const __nv_bfloat16* yg = static_cast<const __nv_bfloat16*>(sl.y);
    const __nv_bfloat16* bg =
        static_cast<const __nv_bfloat16*>(sl.B) + (long long)t.slot * sl.B_slot_stride + (long long)o0 * R;
    constexpr int YW = EOB / 8, BW = R / 8;
    const int ych = ovalid / 8;
    for (int cidx = threadIdx.x; cidx < t.rows * YW; cidx += ETHREADS) {
      const int r = cidx / YW, ch = cidx % YW;
      if (ch < ych)
        cp_async16(Ys + r * X::YPITCH + ch * 16, yg + (long long)(t.row0 + r) * sl.y_row_stride + o0 + ch * 8);
    }
    for (int cidx = threadIdx.x; cidx < ovalid * BW; cidx += ETHREADS) {
      const int o = cidx / BW, ch = cidx % BW;
      cp_async16(Bs + X::b_off(o, ch), bg + (long long)o * R + ch * 8);
    }
    cp_async_commit();
  };

  int ej = 0, eo0 = 0;
  if (s_ok[1]) {
    e_decode(first_e, ej, eo0);
    e_prefetch(s_tile[1], ej, eo0);
  }

  // ---- shrink items
  for (long long item = first_e; item < w.n_shrink; item += gridDim.x) {
    Tile t{};
    bool ok;
    if (item == first_e) {
      t = s_tile[0];
      ok = s_ok[0] != 0;
    } else {
      __syncthreads();
      if (warp == 0) {
        Tile tt{};
        const bool okk = warp_locate_tile(p, DT, item / w.C, tt);
        if (lane == 0) {
          s_tile[0] = tt;
          s_ok[0] = okk;
        }
      }
      __syncthreads();
      t = s_tile[0];
      ok = s_ok[0] != 0;
    }
    if (!ok) continue;  // uniform across the CTA
    if (threadIdx.x == 0) {
      for (int i = 0; i < w.nstage; ++i) mbar_init(&full[i], 1);
      fence_mbar_init();
    }
    __syncthreads();
    const int c = (int)(item % w.C);
    const bool stored = dec_shrink_tile<NR, ETHREADS>(p, maps, ring, full, t, c, w.Kc, w.nstage, u, w.plane_stride);
    __syncthreads();  // every thread's plane stores are done (or none were made)
    (void)stored;     // a failed split still counts itself: its readers must not wait forever
    if (threadIdx.x == 0) tile_arrive_split(ctrl, item / w.C, total);
  }

  // ---- expand items
  for (long long item = first_e; item < w.n_expand; item += gridDim.x) {
    Tile t{};
    bool ok;
    if (item == first_e) {
      t = s_tile[1];
      ok = s_ok[1] != 0;
    } else {
      __syncthreads();
      if (warp == 1) {
        Tile tt{};
        const bool okk = warp_locate_tile(p, DT, item / w.n_ob_total, tt);
        if (lane == 0) {
          s_tile[1] = tt;
          s_ok[1] = okk;
        }
      }
      __syncthreads();
      t = s_tile[1];
      ok = s_ok[1] != 0;
      if (ok) {
        e_decode(item, ej, eo0);
        e_prefetch(t, ej, eo0);
      }
    }
    if (!ok) continue;
    const long long tile = item / w.n_ob_total;
    if (threadIdx.x == 0) {
      const bool got = tile_wait_splits(ctrl, tile, (unsigned)w.C, kCounterPolls);
      if (!got) atomicOr(p.status, LORA_DEV_TIMEOUT);
      s_go = got;
    }
    __syncthreads();
    const bool go = s_go != 0;
    const int j = ej, o0 = eo0;
    const SliceDesc& sl = p.sl[j];
    const int ovalid = min(EOB, sl.out_dim - o0);
    const int nR = p.n_slices * R;

    // u (sum of the C planes, plane order) -> hi + lo bf16 in Hs.  64 rows x
    // R/4 float4 items; up to 8 plane loads in flight per thread.
    if (go) {
      constexpr int R4 = R / 4;
      constexpr int ITEMS = DT * R4;  // 256 (R = 16) or 512 (R = 32)
      constexpr int IPT = ITEMS / ETHREADS;
      constexpr int PB = 8 / IPT;     // planes per round
      const float* ub = u + (long long)t.row0 * nR + (long long)j * R;
      float4 v[IPT];
      bool live[IPT];
#pragma unroll
      for (int i = 0; i < IPT; ++i) {
        const int e = threadIdx.x + i * ETHREADS, r = e / R4;
        live[i] = r < t.rows;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int q0 = 0; q0 < w.C; q0 += PB) {
        float4 part[IPT][PB];
#pragma unroll
        for (int q = 0; q < PB; ++q)
#pragma unroll
          for (int i = 0; i < IPT; ++i) {
            const int e = threadIdx.x + i * ETHREADS, r = e / R4, k = (e % R4) * 4;
            if (live[i] && q0 + q < w.C)
              part[i][q] = __ldcg(reinterpret_cast<const float4*>(ub + (long long)r * nR + k +
                                                                   (q0 + q) * w.plane_stride));
          }
#pragma unroll
        for (int q = 0; q < PB; ++q)
#pragma unroll
          for (int i = 0; i < IPT; ++i)
            if (live[i] && q0 + q < w.C) {
              v[i].x += part[i][q].x;
              v[i].y += part[i][q].y;
              v[i].z += part[i][q].z;
              v[i].w += part[i][q].w;
            }
      }
#pragma unroll
      for (int i = 0; i < IPT; ++i) {
        if (!live[i]) continue;
        const int e = threadIdx.x + i * ETHREADS, r = e / R4, k = (e % R4) * 4;
        __nv_bfloat16* hrow = reinterpret_cast<__nv_bfloat16*>(Hs + r * X::UPITCH);
        uint32_t hi[2], lo[2];
        split_hi_lo_bf16x2(v[i].x, v[i].y, hi[0], lo[0]);
        split_hi_lo_bf16x2(v[i].z, v[i].w, hi[1], lo[1]);
        *reinterpret_cast<uint2*>(hrow + k) = make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2*>(hrow + R + k) = make_uint2(lo[0], lo[1]);
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // planes read, y / B / hi|lo staged
    if (threadIdx.x == 0) tile_arrive_reader(ctrl, tile, total);

    if (go) {
      // 8 warps: 4 row blocks of 16 x 2 column groups of 64, in two passes
      // over the block's 256 columns (64 accumulators per thread).
      const int m = warp & 3, nh = warp >> 2;
      constexpr int CW = 64, NT = CW / 8;
      const int g = lane >> 2, tq = lane & 3;
      if (m * 16 < t.rows) {
        const uint32_t hs = smem_addr(Hs), bs = smem_addr(Bs);
        uint32_t afr[(2 * R) / 16][4];  // this warp's 16 rows of hi|lo, all K steps
#pragma unroll
        for (int kk = 0; kk < (2 * R) / 16; ++kk)
          ldsm_x4(hs + (m * 16 + (lane & 15)) * X::UPITCH + (kk * 16 + (lane >> 4) * 8) * 2, afr[kk][0],
                  afr[kk][1], afr[kk][2], afr[kk][3]);
#pragma unroll 1
        for (int pass = 0; pass < EOB / (2 * CW); ++pass) {
          const int cbase = pass * 2 * CW + nh * CW;
          float acc[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int col = cbase + nt * 8 + 2 * tq;
            const __nv_bfloat162 v0 =
                *reinterpret_cast<const __nv_bfloat162*>(Ys + (m * 16 + g) * X::YPITCH + col * 2);
            const __nv_bfloat162 v1 =
                *reinterpret_cast<const __nv_bfloat162*>(Ys + (m * 16 + g + 8) * X::YPITCH + col * 2);
            acc[nt][0] = __low2float(v0);
            acc[nt][1] = __high2float(v0);
            acc[nt][2] = __low2float(v1);
            acc[nt][3] = __high2float(v1);
          }
#pragma unroll
          for (int kk = 0; kk < (2 * R) / 16; ++kk) {
            const int kb = (kk * 16) % R;  // the lo half reuses B's K columns
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
              uint32_t b0, b1, b2, b3;
              const int nrow = cbase + np * 16 + (lane & 7) + ((lane >> 4) << 3);
              const int kcol = kb + ((lane >> 3) & 1) * 8;
              ldsm_x4(bs + X::b_off(nrow, kcol / 8), b0, b1, b2, b3);
              mma_bf16_16816(acc[2 * np], afr[kk], b0, b1);
              mma_bf16_16816(acc[2 * np + 1], afr[kk], b2, b3);
            }
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int col = cbase + nt * 8 + 2 * tq;
            *reinterpret_cast<__nv_bfloat162*>(Ys + (m * 16 + g) * X::YPITCH + col * 2) =
                __floats2bfloat162_rn(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<__nv_bfloat162*>(Ys + (m * 16 + g + 8) * X::YPITCH + col * 2) =
                __floats2bfloat162_rn(acc[nt][2], acc[nt][3]);
          }
        }
      }
      __syncthreads();
      // Routed rows of the block back to y, 16 bytes per thread per step.
      constexpr int YW = EOB / 8;
      const int ych = ovalid / 8;
      __nv_bfloat16* yg = static_cast<__nv_bfloat16*>(sl.y);
      for (int cidx = threadIdx.x; cidx < t.rows * YW; cidx += ETHREADS) {
        const int r = cidx / YW, ch = cidx % YW;
        if (ch < ych)
          *reinterpret_cast<uint4*>(yg + (long long)(t.row0 + r) * sl.y_row_stride + o0 + ch * 8) =
              *reinterpret_cast<const uint4*>(Ys + r * X::YPITCH + ch * 16);
      }
    }
  }
  pdl_launch_dependents();  // the next kernel may launch; it waits for this grid to finish
}

// Failure-path self test of the counter handoff: CTA 0 is the one reader of
// tile 0 and gives up after `polls` polls; CTA 1 is its one split and
// arrives only after `delay_ns`.  The reader flags LORA_DEV_TIMEOUT and still
// counts itself; the late split completes the count and leaves the counter
// zero.  Launched cooperatively (both CTAs resident).
__global__ void selftest_handoff_kernel(unsigned* ctrl, unsigned* status, uint32_t polls, uint64_t delay_ns) {
  if (threadIdx.x != 0) return;
  const unsigned total = 1u + (1u << 16);
  if (blockIdx.x == 0) {
    if (!tile_wait_splits(ctrl, 0, 1u, polls)) atomicOr(status, LORA_DEV_TIMEOUT);
    tile_arrive_reader(ctrl, 0, total);
  } else {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < delay_ns) __nanosleep(1000);
    tile_arrive_split(ctrl, 0, total);
  }
}

// ------------------------------------------------------------------ host

namespace {

std::mutex g_dec_mu;

PFN_cuTensorMapEncodeTiled_v12000 dec_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lk(g_dec_mu);
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

bool encode_dec_maps(const ProblemDesc& p, DecMaps* m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = dec_encode_fn();
  if (!enc) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  {
    // Ends at row `end`: rows at or past it are zero-filled, never read.
    const cuuint64_t dims[2] = {(cuuint64_t)p.in_dim, (cuuint64_t)p.end};
    const cuuint64_t strides[1] = {(cuuint64_t)p.x_row_stride * 2};
    const cuuint32_t box[2] = {(cuuint32_t)DK, (cuuint32_t)XBOX};
    if (enc(&m->x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  for (int j = 0; j < p.n_slices; ++j) {
    const cuuint64_t dims[3] = {(cuuint64_t)p.in_dim, (cuuint64_t)p.R, (cuuint64_t)p.S};
    const cuuint64_t strides[2] = {(cuuint64_t)p.in_dim * 2, (cuuint64_t)p.sl[j].A_slot_stride * 2};
    const cuuint32_t box[3] = {(cuuint32_t)DK, (cuuint32_t)p.R, 1};
    if (enc(&m->a[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.sl[j].A), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// Ring depth: every stage of the split when ~`budget` bytes hold them.
template <int NR>
int ring_stages(int nst, int budget) {
  int n = nst < MAX_STAGES ? nst : MAX_STAGES;
  while (n > 2 && n * DecCfg<NR>::STAGE > budget) --n;
  return n;
}

template <int NR>
int ring_bytes(int nstage) {
  const int b = nstage * DecCfg<NR>::STAGE;
  const int need = b > DecCfg<NR>::P_BYTES ? b : DecCfg<NR>::P_BYTES;
  return (need + 1023) & ~1023;
}

// Raise a kernel's dynamic shared memory limit once per device.
template <typename K>
cudaError_t dec_ensure_smem(K kernel, int bytes, unsigned long long* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_dec_mu);
  if (*done & (1ull << (dev & 63))) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) *done |= 1ull << (dev & 63);
  return e;
}

template <int NR>
cudaError_t launch_dec_t(const ProblemDesc& p, const DecMaps& maps, float* u, cudaStream_t s, int C) {
  auto kernel = sgmv_shrink_tma_kernel<NR>;
  const int Kc = p.in_dim / C;
  const int nstage = ring_stages<NR>(Kc / DK, 100 * 1024);
  const int smem = ring_bytes<NR>(nstage) + 1024;  // + alignment slack
  static unsigned long long done = 0;
  cudaError_t e = dec_ensure_smem(kernel, ring_bytes<NR>(MAX_STAGES) + 1024, &done);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)p.G + p.end / DT;
  const long long plane_stride = (long long)p.end * p.n_slices * p.R;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * C));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];  // overlap the launch with the previous kernel's tail
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return noted(cudaLaunchKernelEx(&cfg, kernel, p, maps, u, C, Kc, nstage, plane_stride), LORA_PATH_MMA_SHRINK);
}

template <int NR, int R>
cudaError_t launch_dex_t(const ProblemDesc& p, const DecMaps& maps, float* u, unsigned* ctrl, cudaStream_t s,
                         int C) {
  auto kernel = sgmv_decode_apply_kernel<NR, R>;
  DexWork w{};
  w.C = C;
  w.Kc = p.in_dim / C;
  w.nstage = ring_stages<NR>(w.Kc / DK, 64 * 1024);
  w.ring_bytes = ring_bytes<NR>(w.nstage);
  w.plane_stride = (long long)p.end * p.n_slices * p.R;
  const long long tiles = (long long)p.G + p.end / DT;
  int acc = 0;
  for (int j = 0; j < p.n_slices; ++j) {
    w.ob_begin[j] = acc;
    acc += (p.sl[j].out_dim + EOB - 1) / EOB;
  }
  w.ob_begin[p.n_slices] = acc;
  w.n_ob_total = acc;
  w.n_shrink = (int)(tiles * C);
  w.n_expand = (int)(tiles * acc);
  const int smem = w.ring_bytes + DexCfg<R>::BYTES + 1024;
  static unsigned long long done = 0;
  cudaError_t e = dec_ensure_smem(kernel, ring_bytes<NR>(MAX_STAGES) + DexCfg<R>::BYTES + 1024, &done);
  if (e != cudaSuccess) return e;
  // Every CTA must be resident: the grid is at most what the device holds.
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, ETHREADS, smem);
  if (e != cudaSuccess) return e;
  const long long cap = (long long)per_sm * device_sm_count();
  const long long want = w.n_shrink > w.n_expand ? w.n_shrink : w.n_expand;
  // More than two items per CTA: the items after the first are not prefetched
  // during the shrink, and the two-kernel path is faster.
  if (cap < 1 || want > 2 * cap) return cudaErrorNotSupported;
  const long long grid = want < cap ? want : cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(ETHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kernel, p, maps, w, u, ctrl);
  if (e != cudaSuccess) {  // cooperative + programmatic not accepted together: cooperative alone
    (void)cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, p, maps, w, u, ctrl);
  }
  return noted(e, LORA_PATH_DECODE_FUSED);
}

}  // namespace

bool dec_shrink_ok(const ProblemDesc& p) {
  const int nR = p.n_slices * p.R;
  if (p.token_rows || p.slot_ranks) return false;  // plain batches only
  if (p.R != 16 && p.R != 32) return false;
  return nR <= 96 && p.in_dim % DK == 0;
}

cudaError_t launch_dec_shrink(const ProblemDesc& p, float* u, cudaStream_t s, int C) {
  if (C < 1 || p.in_dim % (C * DK) != 0) return cudaErrorNotSupported;
  DecMaps maps;
  if (!encode_dec_maps(p, &maps)) return cudaErrorNotSupported;
  switch (p.n_slices * p.R) {
    case 16: return launch_dec_t<16>(p, maps, u, s, C);
    case 32: return launch_dec_t<32>(p, maps, u, s, C);
    case 48: return launch_dec_t<48>(p, maps, u, s, C);
    case 64: return launch_dec_t<64>(p, maps, u, s, C);
    case 96: return launch_dec_t<96>(p, maps, u, s, C);
  }
  return cudaErrorNotSupported;
}

bool dec_apply_ok(const ProblemDesc& p) {
  if (!dec_shrink_ok(p)) return false;
  for (int j = 0; j < p.n_slices; ++j)
    if (p.sl[j].bias) return false;  // plain batches only
  // Short groups (at most 64 routed rows per group on average) and a tile
  // count the workspace's counters cover.
  const long long tiles = (long long)p.G + p.end / DT;
  return p.G > 0 && p.end <= 64LL * p.G && tiles <= kWorkspaceCtrlWords;
}

cudaError_t launch_dec_apply(const ProblemDesc& p, float* u, unsigned* ctrl, cudaStream_t s, int C) {
  if (C < 1 || p.in_dim % (C * DK) != 0 || C > 0xFFFF) return cudaErrorNotSupported;
  DecMaps maps;
  if (!encode_dec_maps(p, &maps)) return cudaErrorNotSupported;
  switch (p.n_slices * p.R) {
    case 16: return launch_dex_t<16, 16>(p, maps, u, ctrl, s, C);
    case 32: return p.R == 16 ? launch_dex_t<32, 16>(p, maps, u, ctrl, s, C) : launch_dex_t<32, 32>(p, maps, u, ctrl, s, C);
    case 48: return launch_dex_t<48, 16>(p, maps, u, ctrl, s, C);
    case 64: return launch_dex_t<64, 32>(p, maps, u, ctrl, s, C);
    case 96: return launch_dex_t<96, 32>(p, maps, u, ctrl, s, C);
  }
  return cudaErrorNotSupported;
}

cudaError_t launch_selftest_handoff(unsigned* ctrl, unsigned* status, uint32_t polls, uint64_t delay_ns,
                                    cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return noted(cudaLaunchKernelEx(&cfg, selftest_handoff_kernel, ctrl, status, polls, delay_ns), 0);
}

}  // namespace lora
