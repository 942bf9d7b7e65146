// sgmv_bf16.cu -- bf16 SGMV shrink and boundary-aware expand for sm_103a.
//
// Shrink  u[t, j*R+k] = sum_i A_j[s, k, i] x[t, i]       (rank-R intermediate)
// Expand  y_j[t, o]   = rn(y_j[t, o] + sum_k B_j[s, o, k] u[t, j*R+k])
// for every routed row t < end of group g with slot s = lora_ids[g]
// ("vLLM LoRA 实现深度解析" sections 1 and 6; routing triple of the
// "max.pipelines.lora.LoRAManagerV3" page, get_lora_graph_inputs).
//
// Work decomposition.  The routed rows are cut into 64-row tiles per group
// (tiles.cuh).  The shrink gives each (tile, rank-column block, K split) to
// one CTA; every CTA streams its K range of the tile's x rows and of the
// slot's A rows into shared memory through a ring of 16-byte asynchronous
// copies issued by all threads (exactly the group's own rows: nothing outside
// the group is fetched), and multiplies on the tensor cores (mma.sync
// m16n8k16, fp32 accumulate).  In the apply each K split writes its partial
// tile into its own plane of u and the expand sums the planes in plane order;
// for lora_shrink the K splits form a thread-block cluster (up to 16 CTAs)
// and sum through distributed shared memory in rank order (both
// deterministic).  The expand gives each (tile of 64 or 32 rows, slice,
// output block of 64..512 columns) to one CTA: it starts the loads of the y
// block and of the slot's B block, waits (programmatic dependent launch) for
// the shrink grid, sums the u planes, splits u into hi + lo bf16 terms,
// multiplies with the y block as the initial accumulator, rounds once and
// writes exactly the routed rows back with 16-byte stores.  Rows at or past
// `end` are never read or written.  Rank-16 B blocks are staged unpadded with
// swizzled 16-byte chunks; the plain 32 x 512 rank-16 tile has its own
// kernel held to four CTAs per SM.
//
// Row gathers use per-thread 16-byte copies rather than one bulk (TMA)
// request per row: a tile is tens of short row segments, and per-request
// bulk-copy issue cost dominated (measured: 30 us for a 4.8 MB shrink).
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tiles.cuh"

namespace lora {

namespace {

constexpr int MT = kTileRows;        // token rows per tile
constexpr int KS = 64;               // input elements per shrink stage
constexpr int XPITCH = KS * 2 + 16;  // bytes per staged row (padding: conflict-free ldmatrix)

// NSO: ring depth override (0: by NB).  A K split of at most 4 stages
// (64-wide) uses the 4-stage ring: a third of the shared memory, so three
// CTAs fit on an SM.
template <int NB, int NSO = 0>
struct ShrinkCfg {
  static constexpr int NSTAGE = NSO ? NSO : (NB <= 48 ? 8 : (NB <= 64 ? 6 : 4));
  static constexpr int STAGE_BYTES = (MT + NB) * XPITCH;
  static constexpr int PPITCH = NB + 4;  // floats per partial row (16-byte aligned rows)
  static constexpr int SMEM = NSTAGE * STAGE_BYTES;
  static_assert(MT * PPITCH * 4 <= SMEM, "partial tile must fit in the stage ring");
};

}  // namespace

// grid.x = C * nblk * n_tiles_max.  plane_stride == 0: cluster (C,1,1), the
// C partials are reduced through distributed shared memory into u.
// plane_stride > 0: no cluster; K-split rank c stores its partial tile into
// plane c (u + c * plane_stride) and the expand sums the planes.
// GEN: the problem uses token_rows, slot ranks or a bias.  The plain
// instantiation compiles none of that bookkeeping (it costs registers and a
// barrier ahead of the first loads, which decode-sized launches feel).
template <int NB, bool GEN, int NSO>
__global__ void __launch_bounds__(128) sgmv_shrink_bf16_kernel(const __grid_constant__ ProblemDesc p,
                                                               float* __restrict__ u, int C,
                                                               int nblk, int Kc, long long plane_stride,
                                                               const __grid_constant__ HostTiles ht) {
  using Cfg = ShrinkCfg<NB, NSO>;
  constexpr int NSTAGE = Cfg::NSTAGE;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Tile s_tile;
  __shared__ int s_ok;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = (int)(blockIdx.x % (unsigned)C);
  const int rest = (int)(blockIdx.x / (unsigned)C);
  const int nb = rest % nblk;
  const long long tile = rest / nblk;

  Tile t{};
  if (ht.n > 0) {
    // Tiles made on the host: every thread reads its CTA's entry from the
    // launch parameters, so the first global reads after the wait below are
    // the x / A stages.
    if (tile >= ht.n) return;
    const int2 e = ht.t[tile];
    t.row0 = e.x;
    t.slot = e.y >> 8;
    t.rows = e.y & 0xff;
  }

  // Launched as a programmatic dependent of whatever kernel precedes it: no
  // global memory is touched before that kernel has completed.
  pdl_wait();
  pdl_launch_dependents();

  if (ht.n == 0) {
    if (warp == 0) {
      Tile w{};
      const bool ok = warp_locate_tile(p, MT, tile, w);
      if (lane == 0) {
        s_tile = w;
        s_ok = ok;
      }
    }
    __syncthreads();
    if (!s_ok) return;  // the whole cluster sees the same tile and the same outcome
    t = s_tile;
  }

  const int R = p.R;
  const int nR = p.n_slices * R;
  const int n0 = nb * NB;
  const int nvalid = min(NB, nR - n0);
  const int k0 = crank * Kc;
  const int nst = Kc / KS;
  const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(p.x);
  // Staged rows: the tile's x rows, then the slot's nvalid A rows.  Thread
  // `tid` always copies 16-byte column `tid % 8` of rows tid/8, tid/8 + 16,
  // ... so its source pointers and destinations are fixed for every stage
  // and only advance by the stage's K offset: computed once, here.
  constexpr int MAXR = (MT + NB + 15) / 16;  // rows per thread
  const int nrows_total = t.rows + nvalid;
  const int ch = threadIdx.x & 7;
  const int kmax = GEN ? slot_kmax(p, t.slot) : R;  // rank columns past this are zero: not read
  const __nv_bfloat16* srcs[MAXR];
  uint32_t dsts[MAXR];
  int bad_row = 0;
#pragma unroll
  for (int i = 0; i < MAXR; ++i) {
    const int row = (threadIdx.x >> 3) + 16 * i;
    srcs[i] = nullptr;
    dsts[i] = 0;
    if (row < t.rows) {
      // Row of x holding this token (gathered batches map through token_rows).
      const int xr = (GEN && p.token_rows) ? p.token_rows[t.row0 + row] : t.row0 + row;
      if (GEN && (xr < 0 || xr >= p.num_tokens)) {
        bad_row = 1;
        continue;
      }
      srcs[i] = xg + (long long)xr * p.x_row_stride + k0 + ch * 8;
      dsts[i] = row * XPITCH + ch * 16;
    } else if (row < nrows_total) {
      const int col = n0 + row - t.rows;
      const int j = col / R, k = col - j * R;
      if (!GEN || k < kmax) {
        srcs[i] = static_cast<const __nv_bfloat16*>(p.sl[j].A) + (long long)t.slot * p.sl[j].A_slot_stride +
                  (long long)k * p.in_dim + k0 + ch * 8;
        dsts[i] = (MT + row - t.rows) * XPITCH + ch * 16;
      }
    }
  }
  (void)warp;

  // Every CTA of the tile (and of its cluster) checks all of the tile's rows
  // and reaches the same outcome.
  if (GEN && __syncthreads_or(bad_row)) {
    if (threadIdx.x == 0) atomicOr(p.status, LORA_DEV_BAD_ROW);
    return;
  }

  auto issue = [&](int s) {
    uint8_t* xs = smem + (s % NSTAGE) * Cfg::STAGE_BYTES;
    const int kk = s * KS;
#pragma unroll
    for (int i = 0; i < MAXR; ++i)
      if (srcs[i]) cp_async16(xs + dsts[i], srcs[i] + kk);
  };

#pragma unroll 1
  for (int s = 0; s < NSTAGE - 1; ++s) {
    if (s < nst) issue(s);
    cp_async_commit();
  }

  float acc[NB / 8][4];
#pragma unroll
  for (int i = 0; i < NB / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  const bool active = warp * 16 < t.rows;  // warp-uniform: this warp's 16 rows hold data
#pragma unroll 1
  for (int s = 0; s < nst; ++s) {
    // Refill the slot consumed in the previous iteration (all threads passed
    // the barrier that ended it), then wait for stage s.
    if (s + NSTAGE - 1 < nst) issue(s + NSTAGE - 1);
    cp_async_commit();
    cp_async_wait<NSTAGE - 1>();
    __syncthreads();
    if (active) {
      const uint32_t xs = smem_addr(smem + (s % NSTAGE) * Cfg::STAGE_BYTES);
      const uint32_t as = xs + MT * XPITCH;
#pragma unroll
      for (int ks = 0; ks < KS / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(xs + (warp * 16 + (lane & 15)) * XPITCH + (ks * 16 + (lane >> 4) * 8) * 2, a[0], a[1],
                a[2], a[3]);
#pragma unroll
        for (int np = 0; np < NB / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          const int nrow = np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int kcol = ks * 16 + ((lane >> 3) & 1) * 8;
          ldsm_x4(as + nrow * XPITCH + kcol * 2, b0, b1, b2, b3);
          mma_bf16_16816(acc[2 * np], a, b0, b1);
          mma_bf16_16816(acc[2 * np + 1], a, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();

  // Partial tile -> shared memory (reuses the stage ring: every copy landed).
  float* P = reinterpret_cast<float*>(smem);
  if (active) {
    const int g = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NB / 8; ++nt) {
      const int row = warp * 16 + g, col = nt * 8 + 2 * tq;
      // Columns past the slot's rank read no A rows (stale shared memory): 0.
      const bool keep = !GEN || ((n0 + col) % R) < kmax;
      *reinterpret_cast<float2*>(&P[row * Cfg::PPITCH + col]) =
          keep ? make_float2(acc[nt][0], acc[nt][1]) : make_float2(0.f, 0.f);
      *reinterpret_cast<float2*>(&P[(row + 8) * Cfg::PPITCH + col]) =
          keep ? make_float2(acc[nt][2], acc[nt][3]) : make_float2(0.f, 0.f);
    }
  }
  const int q4 = nvalid / 4;
  if (plane_stride > 0) {
    __syncthreads();
    float* up = u + crank * plane_stride;
    for (int e = threadIdx.x; e < t.rows * q4; e += blockDim.x) {
      const int r = e / q4, c = (e % q4) * 4;
      *reinterpret_cast<float4*>(&up[(long long)(t.row0 + r) * nR + n0 + c]) =
          *reinterpret_cast<const float4*>(&P[r * Cfg::PPITCH + c]);
    }
    return;
  }
  if (C > 1)
    cluster_sync();
  else
    __syncthreads();

  // Each CTA of the cluster sums its share of rows over all C partials, in
  // rank order, and writes them to u, four columns per step (nvalid is a
  // multiple of 16).  The C remote loads of a step are issued back to back.
  const int rpc = MT / C;
  const int r_lo = crank * rpc;
  const int r_hi = min(r_lo + rpc, t.rows);
  const int cnt = (r_hi - r_lo) * q4;
  for (int e = threadIdx.x; e < cnt; e += blockDim.x) {
    const int r = r_lo + e / q4, c = (e % q4) * 4;
    float4 v;
    if (C == 1) {
      v = *reinterpret_cast<const float4*>(&P[r * Cfg::PPITCH + c]);
    } else {
      const uint32_t la = smem_addr(&P[r * Cfg::PPITCH + c]);
      float4 part[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (q < C) part[q] = ld_shared_cluster_f32x4(map_shared_rank(la, (uint32_t)q));
      v = part[0];
#pragma unroll
      for (int q = 1; q < 16; ++q)
        if (q < C) {
          v.x += part[q].x;
          v.y += part[q].y;
          v.z += part[q].z;
          v.w += part[q].w;
        }
    }
    *reinterpret_cast<float4*>(&u[(long long)(t.row0 + r) * nR + n0 + c]) = v;
  }
  if (C > 1) cluster_sync();  // keep this CTA's partial alive for its peers
}

// ------------------------------------------------------------------ expand

// An expand tile is MR routed rows (64, or 32 for short groups) by OB output
// columns; the 8 warps are MR/16 row blocks times 8/(MR/16) column groups.
template <int R, int OB, int MR>
struct ExpandCfg {
  static constexpr int YPITCH = OB * 2 + 16;  // bytes per staged y row
  // Bytes per staged B row.  Rank 16: 32 bytes, unpadded, with the two
  // 16-byte chunks of a row swapped when bit 2 of the row is set (rows r and
  // r + 4 would share banks otherwise); the 8 rows of an ldmatrix phase then
  // hit 8 different bank groups.  Higher ranks: padded by 16 bytes.
  static constexpr bool BSWZ = R == 16;
  static constexpr int BPITCH = BSWZ ? 32 : R * 2 + 16;
  __device__ static constexpr int b_off(int o, int ch) {
    return o * BPITCH + (BSWZ ? (ch ^ ((o >> 2) & 1)) : ch) * 16;
  }
  static constexpr int UPITCH = 4 * R + 16;   // bytes per hi|lo row (2R bf16)
  static constexpr int Y_OFF = 0;
  static constexpr int B_OFF = MR * YPITCH;
  static constexpr int H_OFF = B_OFF + OB * BPITCH;
  static constexpr int SMEM = H_OFF + MR * UPITCH;
  static constexpr int MB = MR / 16;          // row blocks
  static constexpr int NW = 8 / MB;           // column groups
  static constexpr int CW = OB / NW;          // columns per warp
  static_assert(CW % 16 == 0, "column group");
};

struct ExpandMap {
  int n_ob_total;                     // output blocks per tile, all slices
  int ob_begin[LORA_MAX_SLICES + 1];  // first output block of each slice
  int nsplit;                         // partial planes of u to sum (1..16)
  long long plane_stride;             // elements between planes
};

// GEN as for the shrink: token_rows, slot ranks or a bias in use.
template <int R, int OB, int MR, bool GEN>
__device__ __forceinline__ void expand_bf16_body(const ProblemDesc& p, const float* __restrict__ u,
                                                 const ExpandMap& map, const HostRouting& hr) {
  using Cfg = ExpandCfg<R, OB, MR>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Tile s_tile;
  __shared__ int s_ok;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long tile = blockIdx.x / (unsigned)map.n_ob_total;
  const int obg = (int)(blockIdx.x % (unsigned)map.n_ob_total);
  int j = 0;
  while (j + 1 < p.n_slices && obg >= map.ob_begin[j + 1]) ++j;
  const int o0 = (obg - map.ob_begin[j]) * OB;
  const SliceDesc& sl = p.sl[j];
  const int ovalid = min(OB, sl.out_dim - o0);
  const int nR = p.n_slices * R;

  if (warp == 0) {
    Tile t{};
    const bool ok = warp_locate_tile(p, MR, tile, t, &hr);  // also checks the host copy, if any
    if (lane == 0) {
      s_tile = t;
      s_ok = ok;
    }
  }
  __syncthreads();
  if (!s_ok) return;
  const Tile t = s_tile;

  // Row of y holding each token of the tile (gathered batches map through
  // token_rows); an out-of-range entry skips the tile.
  __shared__ int s_rows[MR];
  if constexpr (GEN) {
    int bad_row = 0;
    for (int r = threadIdx.x; r < t.rows; r += blockDim.x) {
      const int yr = p.token_rows ? p.token_rows[t.row0 + r] : t.row0 + r;
      if (yr < 0 || yr >= p.num_tokens) bad_row = 1;
      s_rows[r] = yr;
    }
    if (__syncthreads_or(bad_row)) {
      if (threadIdx.x == 0) atomicOr(p.status, LORA_DEV_BAD_ROW);
      return;
    }
  }
  auto y_row = [&](int r) -> long long { return GEN ? s_rows[r] : t.row0 + r; };

  uint8_t* Ys = smem + Cfg::Y_OFF;
  uint8_t* Bs = smem + Cfg::B_OFF;
  uint8_t* Hs = smem + Cfg::H_OFF;
  __nv_bfloat16* yg = static_cast<__nv_bfloat16*>(sl.y);
  const __nv_bfloat16* bg = static_cast<const __nv_bfloat16*>(sl.B) + (long long)t.slot * sl.B_slot_stride +
                            (long long)o0 * R;

  // y block and B block do not depend on the shrink: fetch them first.  All
  // chunk loops run over compile-time row widths (OB/8 chunks per y row, R/8
  // per B row) so the row/column split is a shift; chunks past a partial
  // block's width are skipped.
  constexpr int YW = OB / 8;  // 16-byte chunks per full y row
  constexpr int BW = R / 8;   // chunks per B row
  const int ych = ovalid / 8;
  for (int c = threadIdx.x; c < t.rows * YW; c += blockDim.x) {
    const int r = c / YW, ch = c % YW;
    if (ch < ych)
      cp_async16(Ys + r * Cfg::YPITCH + ch * 16, yg + y_row(r) * sl.y_row_stride + o0 + ch * 8);
  }
  const int kmax = GEN ? slot_kmax(p, t.slot) : R;  // B columns past this are not read
  for (int c = threadIdx.x; c < ovalid * BW; c += blockDim.x) {
    const int o = c / BW, ch = c % BW;
    if (!GEN || ch * 8 < kmax) cp_async16(Bs + Cfg::b_off(o, ch), bg + (long long)o * R + ch * 8);
  }
  cp_async_commit();

  pdl_wait();  // the shrink grid (if any) has finished and its u is visible

  // u (sum of the nsplit planes) -> hi + lo bf16: u = hi + lo to 16
  // significant bits; the subtraction is exact.  Read through L2 only.  The
  // planes are dependent L2 round trips, so a thread keeps up to 8 float4
  // loads in flight across its items (plane-major, each item summed in plane
  // order).  Where a tile has fewer float4 items than threads (R = 16 with
  // 32-row tiles), two threads share an item: one sums the first half of the
  // planes, the other the second, and the halves meet in shared memory.
  {
    constexpr int R4 = R / 4;
    constexpr int ITEMS = MR * R4;                     // float4 items of a full tile's u
    constexpr int TPI = ITEMS < 256 ? 256 / ITEMS : 1;  // threads sharing an item
    constexpr int IPT = ITEMS > 256 ? ITEMS / 256 : 1;  // items per thread
    constexpr int PB = IPT < 8 ? 8 / IPT : 1;          // planes per round
    static_assert(TPI <= 2, "plane halves");
    __shared__ float4 s_uhalf[TPI > 1 ? ITEMS : 1];
    const float* ub = u + (long long)t.row0 * nR + (long long)j * R;
    const int sub = TPI > 1 ? (int)threadIdx.x / ITEMS : 0;
    const int e0 = TPI > 1 ? (int)threadIdx.x % ITEMS : (int)threadIdx.x;
    const int share = (map.nsplit + TPI - 1) / TPI;
    const int q_lo = sub * share, q_hi = min(map.nsplit, q_lo + share);
    float4 v[IPT];
    const float* src[IPT];
    bool live[IPT];
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
      const int e = e0 + i * 256, r = e / R4, k = (e % R4) * 4;
      live[i] = r < t.rows;
      src[i] = ub + (long long)r * nR + k;
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int q0 = q_lo; q0 < q_hi; q0 += PB) {
      float4 part[IPT][PB];
#pragma unroll
      for (int q = 0; q < PB; ++q)
#pragma unroll
        for (int i = 0; i < IPT; ++i)
          if (live[i] && q0 + q < q_hi)
            part[i][q] = __ldcg(reinterpret_cast<const float4*>(src[i] + (q0 + q) * map.plane_stride));
#pragma unroll
      for (int q = 0; q < PB; ++q)
#pragma unroll
        for (int i = 0; i < IPT; ++i)
          if (live[i] && q0 + q < q_hi) {
            v[i].x += part[i][q].x;
            v[i].y += part[i][q].y;
            v[i].z += part[i][q].z;
            v[i].w += part[i][q].w;
          }
    }
    if constexpr (TPI > 1) {
      if (sub == 1) s_uhalf[e0] = v[0];
      __syncthreads();
      if (sub == 0) {
        const float4 w = s_uhalf[e0];
        v[0].x += w.x;
        v[0].y += w.y;
        v[0].z += w.z;
        v[0].w += w.w;
      }
    }
    if (sub == 0) {
#pragma unroll
      for (int i = 0; i < IPT; ++i) {
        if (!live[i]) continue;
        const int e = e0 + i * 256, r = e / R4, k = (e % R4) * 4;
        __nv_bfloat16* hrow = reinterpret_cast<__nv_bfloat16*>(Hs + r * Cfg::UPITCH);
        uint32_t hi[2], lo[2];
        split_hi_lo_bf16x2(v[i].x, v[i].y, hi[0], lo[0]);
        split_hi_lo_bf16x2(v[i].z, v[i].w, hi[1], lo[1]);
        *reinterpret_cast<uint2*>(hrow + k) = make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2*>(hrow + R + k) = make_uint2(lo[0], lo[1]);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  const int m = warp % Cfg::MB, nh = warp / Cfg::MB;
  constexpr int NT = Cfg::CW / 8;  // n8 tiles per warp
  const int g = lane >> 2, tq = lane & 3;
  if (m * 16 < t.rows) {
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = nh * Cfg::CW + nt * 8 + 2 * tq;
      const __nv_bfloat162 v0 =
          *reinterpret_cast<const __nv_bfloat162*>(Ys + (m * 16 + g) * Cfg::YPITCH + col * 2);
      const __nv_bfloat162 v1 =
          *reinterpret_cast<const __nv_bfloat162*>(Ys + (m * 16 + g + 8) * Cfg::YPITCH + col * 2);
      acc[nt][0] = __low2float(v0);
      acc[nt][1] = __high2float(v0);
      acc[nt][2] = __low2float(v1);
      acc[nt][3] = __high2float(v1);
      if (GEN && sl.bias && o0 + col < sl.out_dim) {  // bias joins y before the one rounding
        const __nv_bfloat162 bv = *reinterpret_cast<const __nv_bfloat162*>(
            static_cast<const __nv_bfloat16*>(sl.bias) + (long long)t.slot * sl.bias_slot_stride + o0 + col);
        acc[nt][0] += __low2float(bv);
        acc[nt][1] += __high2float(bv);
        acc[nt][2] += __low2float(bv);
        acc[nt][3] += __high2float(bv);
      }
    }
    const uint32_t hs = smem_addr(Hs), bs = smem_addr(Bs);
#pragma unroll
    for (int kk = 0; kk < (2 * R) / 16; ++kk) {
      const int kb = (kk * 16) % R;
      if (GEN && kb >= kmax) continue;  // past the slot's rank (hi and lo halves alike)
      uint32_t a[4];
      ldsm_x4(hs + (m * 16 + (lane & 15)) * Cfg::UPITCH + (kk * 16 + (lane >> 4) * 8) * 2, a[0], a[1],
              a[2], a[3]);
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        uint32_t b0, b1, b2, b3;
        const int nrow = nh * Cfg::CW + np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int kcol = kb + ((lane >> 3) & 1) * 8;
        ldsm_x4(bs + Cfg::b_off(nrow, kcol / 8), b0, b1, b2, b3);
        mma_bf16_16816(acc[2 * np], a, b0, b1);
        mma_bf16_16816(acc[2 * np + 1], a, b2, b3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = nh * Cfg::CW + nt * 8 + 2 * tq;
      *reinterpret_cast<__nv_bfloat162*>(Ys + (m * 16 + g) * Cfg::YPITCH + col * 2) =
          __floats2bfloat162_rn(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<__nv_bfloat162*>(Ys + (m * 16 + g + 8) * Cfg::YPITCH + col * 2) =
          __floats2bfloat162_rn(acc[nt][2], acc[nt][3]);
    }
  }
  __syncthreads();
  // Routed rows of the block back to y, 16 bytes per thread per step.
  for (int c = threadIdx.x; c < t.rows * YW; c += blockDim.x) {
    const int r = c / YW, ch = c % YW;
    if (ch < ych)
      *reinterpret_cast<uint4*>(yg + y_row(r) * sl.y_row_stride + o0 + ch * 8) =
          *reinterpret_cast<const uint4*>(Ys + r * Cfg::YPITCH + ch * 16);
  }
  pdl_launch_dependents();  // the next kernel may launch; it waits for this grid to finish
}

template <int R, int OB, int MR, bool GEN>
__global__ void __launch_bounds__(256) sgmv_expand_bf16_kernel(const __grid_constant__ ProblemDesc p,
                                                               const float* __restrict__ u,
                                                               const __grid_constant__ ExpandMap map,
                                                               const __grid_constant__ HostRouting hr) {
  expand_bf16_body<R, OB, MR, GEN>(p, u, map, hr);
}

// The plain 32 x 512 rank-16 tile (short groups over wide outputs, grids of
// several waves) held to 64 registers, so four CTAs share an SM.
__global__ void __launch_bounds__(256, 4) sgmv_expand_bf16_w4_kernel(const __grid_constant__ ProblemDesc p,
                                                                     const float* __restrict__ u,
                                                                     const __grid_constant__ ExpandMap map,
                                                                     const __grid_constant__ HostRouting hr) {
  expand_bf16_body<16, 512, 32, false>(p, u, map, hr);
}

// ------------------------------------------------------------------ host

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int pick_nb(int nR, int* nblk) {
  static const int choices[] = {16, 32, 48, 64, 96, 128};
  const int nb_count = (nR + 127) / 128;
  const int need = (nR + nb_count - 1) / nb_count;
  for (int c : choices)
    if (c >= need) {
      *nblk = (nR + c - 1) / c;
      return c;
    }
  *nblk = nb_count;
  return 128;
}

std::mutex g_attr_mu;

// Raise a kernel's dynamic shared-memory limit once per device.  `done` is
// the caller's per-instantiation bitmask of devices already configured.
template <typename K>
cudaError_t ensure_smem(K kernel, int bytes, unsigned long long* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (*done & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) *done |= bit;
  return e;
}

int num_sms() { return device_sm_count(); }

// lora_shrink's cluster size: the input dimension is split over up to 16
// CTAs while the grid stays within two CTAs per SM (decode-sized launches
// have few tiles, and shorter K ranges per CTA put more loads in flight).
static int cluster_splits(const ProblemDesc& p, int nblk) {
  const long long tiles = (long long)p.G + p.end / MT;
  const int ksteps = p.in_dim / KS;
  const long long target = 2LL * num_sms();
  int C = 1;
  while (C < 16 && tiles * nblk * C * 2 <= target && ksteps % (C * 2) == 0) C *= 2;
  return C;
}

template <int NB, bool GEN, int NSO>
cudaError_t launch_shrink_ns(const ProblemDesc& p, float* u, cudaStream_t s, int nblk, bool partial,
                             const HostTiles& ht);

template <int NB, bool GEN>
cudaError_t launch_shrink_nb(const ProblemDesc& p, float* u, cudaStream_t s, int nblk, bool partial,
                             const HostTiles& ht) {
  bool short_ring = false;
  if (partial)
    (void)apply_splits_for(p, &short_ring, ht.n > 0 ? ht.n : -1);
  else
    short_ring = cluster_splits(p, nblk) == 16;  // smaller CTAs: a 16-CTA cluster packs into a GPC
  if (short_ring) return launch_shrink_ns<NB, GEN, 4>(p, u, s, nblk, partial, ht);
  return launch_shrink_ns<NB, GEN, 0>(p, u, s, nblk, partial, ht);
}

template <int NB, bool GEN, int NSO>
cudaError_t launch_shrink_ns(const ProblemDesc& p, float* u, cudaStream_t s, int nblk, bool partial,
                             const HostTiles& ht) {
  auto kernel = sgmv_shrink_bf16_kernel<NB, GEN, NSO>;
  const int smem = ShrinkCfg<NB, NSO>::SMEM;
  static unsigned long long done = 0;
  cudaError_t e = ensure_smem(kernel, smem, &done);
  if (e != cudaSuccess) return e;
  // A tile table gives the exact count; else an upper bound (CTAs past the
  // last tile return).
  const long long tiles = ht.n > 0 ? ht.n : (long long)p.G + p.end / MT;
  int C = 1;
  long long plane_stride = 0;
  if (partial) {
    C = apply_splits_for(p, nullptr, ht.n > 0 ? ht.n : -1);
    if (C > 1) plane_stride = (long long)p.end * p.n_slices * p.R;
  } else {
    C = cluster_splits(p, nblk);
    if (C == 16) {
      // 16 CTAs per cluster is beyond the portable 8: opt in, and fall back
      // to 8 if a cluster of this kernel cannot be placed.
      static unsigned long long big_ok = 0, big_no = 0;
      int dev = 0;
      e = cudaGetDevice(&dev);
      if (e != cudaSuccess) return e;
      const unsigned long long bit = 1ull << (dev & 63);
      std::lock_guard<std::mutex> lk(g_attr_mu);
      if (!((big_ok | big_no) & bit)) {
        int clusters = 0;
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(16);
        q.blockDim = dim3(128);
        q.dynamicSmemBytes = smem;
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = 16;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        q.attrs = a;
        q.numAttrs = 1;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
            cudaOccupancyMaxActiveClusters(&clusters, kernel, &q) == cudaSuccess && clusters > 0)
          big_ok |= bit;
        else
          big_no |= bit;
        (void)cudaGetLastError();  // a refused query leaves no sticky error
      }
      if (big_no & bit) C = 8;
    }
  }
  const int Kc = p.in_dim / C;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * nblk * C));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (C > 1 && !partial) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  } else if (partial) {  // the apply's shrink overlaps its launch with the previous kernel's tail
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return noted(cudaLaunchKernelEx(&cfg, kernel, p, u, C, nblk, Kc, plane_stride, ht), LORA_PATH_MMA_SHRINK);
}

// The kernel of an expand tile shape (only the one that runs is instantiated).
template <int R, int OB, int MR, bool GEN>
constexpr auto expand_kernel() {
  if constexpr (R == 16 && OB == 512 && MR == 32 && !GEN)
    return &sgmv_expand_bf16_w4_kernel;
  else
    return &sgmv_expand_bf16_kernel<R, OB, MR, GEN>;
}

template <int R, int OB, int MR, bool GEN>
cudaError_t launch_expand_r(const ProblemDesc& p, const float* u, cudaStream_t s, bool pdl, int nsplit,
                            const HostRouting& hr) {
  auto kernel = expand_kernel<R, OB, MR, GEN>();
  const int smem = ExpandCfg<R, OB, MR>::SMEM;
  static unsigned long long done = 0;
  cudaError_t e = ensure_smem(kernel, smem, &done);
  if (e != cudaSuccess) return e;
  ExpandMap map{};
  int acc = 0;
  for (int j = 0; j < p.n_slices; ++j) {
    map.ob_begin[j] = acc;
    acc += (p.sl[j].out_dim + OB - 1) / OB;
  }
  map.ob_begin[p.n_slices] = acc;
  map.n_ob_total = acc;
  map.nsplit = nsplit;
  map.plane_stride = (long long)p.end * p.n_slices * R;
  const long long tiles = (long long)p.G + p.end / MR;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * acc));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return noted(cudaLaunchKernelEx(&cfg, kernel, p, u, map, hr), LORA_PATH_MMA_EXPAND);
}

}  // namespace

bool fast_path_ok(const ProblemDesc& p, const void* u) {
  if (p.dtype != LORA_DTYPE_BF16) return false;
  if (p.R != 16 && p.R != 32 && p.R != 64 && p.R != 128) return false;
  if (p.in_dim % KS != 0) return false;
  if (!aligned16(p.x) || p.x_row_stride % 8 != 0) return false;
  if (u && !aligned16(u)) return false;
  for (int j = 0; j < p.n_slices; ++j) {
    const SliceDesc& sl = p.sl[j];
    if (!aligned16(sl.A) || !aligned16(sl.B) || !aligned16(sl.y)) return false;
    if (sl.A_slot_stride % 8 != 0 || sl.B_slot_stride % 8 != 0) return false;
    if (sl.out_dim % 8 != 0 || sl.y_row_stride % 8 != 0) return false;
    if (sl.bias && (!aligned16(sl.bias) || sl.bias_slot_stride % 8 != 0)) return false;
  }
  return true;
}

int apply_splits_for(const ProblemDesc& p, bool* short_ring, long long exact_tiles) {
  // At launch the group count is known: size the split on the tiles (their
  // count when a host-made table gives it, else the upper bound G + end/64)
  // and on how many of these CTAs share an SM, to
  // about two waves, never above the shape-only bound the workspace holds.
  // With the 4-stage ring three times as many CTAs share an SM: it is taken
  // when that allows more splits, or when a split is at most 4 stages long.
  const int cap = apply_splits(p.end, p.in_dim, p.n_slices * p.R);
  int nblk = 1;
  const int nb = pick_nb(p.n_slices * p.R, &nblk);
  int smem = ShrinkCfg<128>::SMEM, smem4 = ShrinkCfg<128, 4>::SMEM;
  switch (nb) {
    case 16: smem = ShrinkCfg<16>::SMEM; smem4 = ShrinkCfg<16, 4>::SMEM; break;
    case 32: smem = ShrinkCfg<32>::SMEM; smem4 = ShrinkCfg<32, 4>::SMEM; break;
    case 48: smem = ShrinkCfg<48>::SMEM; smem4 = ShrinkCfg<48, 4>::SMEM; break;
    case 64: smem = ShrinkCfg<64>::SMEM; smem4 = ShrinkCfg<64, 4>::SMEM; break;
    case 96: smem = ShrinkCfg<96>::SMEM; smem4 = ShrinkCfg<96, 4>::SMEM; break;
  }
  const long long tiles = exact_tiles >= 0 ? exact_tiles : (long long)p.G + p.end / MT;
  const int ksteps = p.in_dim / KS;
  auto pick = [&](int sm_bytes) {
    const long long per_sm = std::max(1, (228 * 1024) / (sm_bytes + 1024));
    int C = 1;
    while (C < cap && tiles * nblk * C * 2 <= 2LL * num_sms() * per_sm && ksteps % (C * 2) == 0) C *= 2;
    return C;
  };
  int c8 = pick(smem), c4 = pick(smem4);
  // A single rank-16 block over an input below 8192 goes past 8 splits only
  // while 8 would leave SMs without a CTA (decode-sized batches: o_proj apply
  // 7.07 -> 6.69 us); with more tiles the extra planes cost the expand more
  // than the shorter K ranges save (many64's o_proj 17.6 -> 17.9 us).
  if (nb == 16 && p.in_dim < 8192 && tiles * nblk * 8 >= num_sms()) {
    c8 = std::min(c8, 8);
    c4 = std::min(c4, 8);
  }
  const int C = c4 > c8 ? c4 : c8;
  if (short_ring) *short_ring = c4 > c8 || ksteps / C <= 4;
  return C;
}

int apply_splits(int end, int in_dim, int nR) {
  // Largest power of two <= 8 dividing the input stages such that the
  // partial-plane shrink grid (a lower bound on its tiles: ceil(end / 64))
  // stays within 256 CTAs; up to 16 for inputs of 8192 and more (long K
  // ranges), for rank blocks of 48 columns or more (long stage loops) and for
  // a single 16-column block (decode-sized o_proj grids).
  // Depends on shapes only, so the workspace bound can be computed without a
  // device.
  if (end <= 0 || in_dim % KS != 0) return 1;
  int nblk = 1;
  const int nb = pick_nb(nR, &nblk);
  const long long tiles = (end + MT - 1) / MT;
  const int ksteps = in_dim / KS;
  int C = 1;
  const int cmax = (in_dim >= 8192 || nb >= 48 || nb == 16) ? 16 : 8;
  while (C < cmax && tiles * nblk * C * 2 <= 256 && ksteps % (C * 2) == 0) C *= 2;
  return C;
}

// Any of token_rows, slot ranks or a bias selects the general kernels.
static bool needs_general(const ProblemDesc& p) {
  if (p.token_rows || p.slot_ranks) return true;
  for (int j = 0; j < p.n_slices; ++j)
    if (p.sl[j].bias) return true;
  return false;
}

template <bool GEN>
static cudaError_t dispatch_shrink_g(const ProblemDesc& p, float* u, cudaStream_t s, bool partial,
                                     const HostTiles& ht) {
  int nblk = 1;
  const int nb = pick_nb(p.n_slices * p.R, &nblk);
  switch (nb) {
    case 16: return launch_shrink_nb<16, GEN>(p, u, s, nblk, partial, ht);
    case 32: return launch_shrink_nb<32, GEN>(p, u, s, nblk, partial, ht);
    case 48: return launch_shrink_nb<48, GEN>(p, u, s, nblk, partial, ht);
    case 64: return launch_shrink_nb<64, GEN>(p, u, s, nblk, partial, ht);
    case 96: return launch_shrink_nb<96, GEN>(p, u, s, nblk, partial, ht);
    default: return launch_shrink_nb<128, GEN>(p, u, s, nblk, partial, ht);
  }
}

static cudaError_t dispatch_shrink(const ProblemDesc& p, float* u, cudaStream_t s, bool partial,
                                   const HostTiles& ht) {
  return needs_general(p) ? dispatch_shrink_g<true>(p, u, s, partial, ht)
                          : dispatch_shrink_g<false>(p, u, s, partial, ht);
}

template <bool GEN>
static cudaError_t dispatch_expand_g(const ProblemDesc& p, const float* u, cudaStream_t s, bool pdl, int nsplit,
                                     const HostRouting& hr) {
  // Short groups (at most 32 routed rows each on average): 32-row tiles twice
  // as wide, so a tile's fixed costs (routing lookup, u, B block) cover twice
  // the outputs and the grid has half the CTAs -- unless that leaves fewer
  // than two CTAs per SM (decode-sized batches: o_proj's 4096 columns, fused
  // qkv's 6144), where 256-wide blocks give twice the CTAs, each with half the
  // y and B to load, and more loads in flight per SM.
  const bool short_groups = (long long)p.end <= 32LL * p.G;
  switch (p.R) {
    case 16:
      if (short_groups) {
        long long blocks = 0;
        for (int j = 0; j < p.n_slices; ++j) blocks += (p.sl[j].out_dim + 511) / 512;
        const long long tiles = (long long)p.G + p.end / 32;
        return tiles * blocks < 2LL * num_sms() ? launch_expand_r<16, 256, 32, GEN>(p, u, s, pdl, nsplit, hr)
                                                : launch_expand_r<16, 512, 32, GEN>(p, u, s, pdl, nsplit, hr);
      }
      return launch_expand_r<16, 256, 64, GEN>(p, u, s, pdl, nsplit, hr);
    case 32: return launch_expand_r<32, 256, 64, GEN>(p, u, s, pdl, nsplit, hr);
    case 64: return launch_expand_r<64, 128, 64, GEN>(p, u, s, pdl, nsplit, hr);
    default: return launch_expand_r<128, 64, 64, GEN>(p, u, s, pdl, nsplit, hr);
  }
}

// The shrink's MT-row tiles of the groups the launch works on (lengths in
// [seg_lo, seg_hi)), numbered as warp_locate_tile numbers them, from the
// routing's (validated) host copies.  n = 0 when there are none or the tiles
// do not fit the table.
static HostTiles make_host_tiles(const ProblemDesc& p, const lora_routing_t* r) {
  HostTiles ht{};
  if (!r || !r->host_grouped_offsets || !r->host_lora_ids || r->num_groups <= 0 || p.S > (1 << 22)) return ht;
  const int32_t* offs = r->host_grouped_offsets;
  int n = 0;
  for (int g = 0; g < r->num_groups; ++g) {
    const int o0 = offs[g], o1 = offs[g + 1];
    const int len = o1 - o0;
    if (len <= 0 || len < p.seg_lo || len >= p.seg_hi) continue;
    for (int row = o0; row < o1; row += MT) {
      if (n == kHostTilesMax) return HostTiles{};
      ht.t[n++] = make_int2(row, (r->host_lora_ids[g] << 8) | std::min(MT, o1 - row));
    }
  }
  ht.n = n;
  return ht;
}

cudaError_t launch_shrink_bf16(const ProblemDesc& p, float* u, cudaStream_t s) {
  return dispatch_shrink(p, u, s, false, HostTiles{});
}

cudaError_t launch_shrink_partial_bf16(const ProblemDesc& p, float* u, cudaStream_t s, const lora_routing_t* r,
                                       int* splits) {
  const HostTiles ht = make_host_tiles(p, r);
  if (splits) *splits = apply_splits_for(p, nullptr, ht.n > 0 ? ht.n : -1);  // what the launch below takes
  return dispatch_shrink(p, u, s, true, ht);
}

cudaError_t launch_expand_bf16(const ProblemDesc& p, const float* u, cudaStream_t s, bool pdl, int nsplit,
                               const HostRouting* hr) {
  const HostRouting h = hr ? *hr : HostRouting{};
  return needs_general(p) ? dispatch_expand_g<true>(p, u, s, pdl, nsplit, h)
                          : dispatch_expand_g<false>(p, u, s, pdl, nsplit, h);
}

}  // namespace lora
