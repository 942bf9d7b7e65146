// sgmv_decode.cu -- the apply's shrink for short groups (decode-sized
// batches) with its operands brought in by the tensor memory accelerator.
//
//   u_c[t, j*R+k] = sum_{i in K split c} A_j[s, k, i] x[t, i]
// for the routed rows t of a group with slot s ("vLLM LoRA 实现深度解析"
// sections 1 and 6; routing triple of the "max.pipelines.lora.LoRAManagerV3"
// page, get_lora_graph_inputs).  Each K split c writes its partial tile into
// plane c of the workspace; the expand sums the planes in plane order.
//
// One CTA per (64-row tile of a group, K split), all n*R <= 128 intermediate
// columns.  Thread 0 issues, per 64-wide K stage, one TMA box of 16 x rows
// per 16 routed rows of the tile (rows past the group belong to the next
// group, rows at or past `end` are zero-filled by the tensor map: neither is
// stored) and one box of the slot's R A rows per slice, all with the 128-byte
// swizzle; every stage of the split is in flight at once when the ring holds
// them.  The tensor memory accelerator keeps tens of kilobytes per CTA in
// flight without occupying the load/store unit, which is what a decode shrink
// (a few kilobytes per row, a few rows per group) is bound by.  Four warps
// multiply their 16 rows on the tensor cores (mma.sync m16n8k16, fp32
// accumulate), reading the swizzled stages with ldmatrix.
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
constexpr int DTHREADS = 128;    // 4 warps x 16 rows
constexpr int MAX_STAGES = 8;

template <int NR>
struct DecCfg {
  static constexpr int X_BYTES = DT * DK * 2;             // 8 KB: up to 4 boxes of 16 rows
  static constexpr int A_BYTES = NR * DK * 2;             // all slices' rank rows
  static constexpr int STAGE = X_BYTES + ((A_BYTES + 1023) / 1024) * 1024;
  static constexpr int PPITCH = NR + 4;                   // floats per staged partial row
  static constexpr int P_BYTES = DT * PPITCH * 4;         // the partial tile, staged over the ring
};

// Byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled block
// (what a TMA box of 64 bf16 columns with the 128-byte swizzle writes, the
// block starting on a 1024-byte boundary).
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

}  // namespace

struct DecMaps {
  CUtensorMap x;                   // [end rows, in] bf16, box 64 x 16
  CUtensorMap a[LORA_MAX_SLICES];  // per slice [S, R, in] bf16, box 64 x R x 1
};

// grid.x = tiles_max * C.  CTA (tile, c): K range [c*Kc, (c+1)*Kc) in nst
// stages through a ring of nstage slots; partial tile -> plane c.
template <int NR>
__global__ void __launch_bounds__(DTHREADS) sgmv_shrink_tma_kernel(const __grid_constant__ ProblemDesc p,
                                                                   const __grid_constant__ DecMaps maps,
                                                                   float* __restrict__ u, int C, int Kc,
                                                                   int nstage, long long plane_stride) {
  using Cfg = DecCfg<NR>;
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
  const Tile t = s_tile;
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
  const bool active = warp * 16 < t.rows;  // warp-uniform
  int fail = 0;
  for (int s = 0; s < nst; ++s) {
    const int slot = s % nstage;
    if (!fail && !mbar_wait(&full[slot], (uint32_t)((s / nstage) & 1))) fail = 1;
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
      if (threadIdx.x == 0) issue(s + nstage);
    }
  }
  if (__syncthreads_or(fail)) {
    // A copy never arrived: give the ones in flight a bounded chance to land
    // before the shared memory is released, flag the launch and store nothing.
    if (threadIdx.x == 0) {
      for (int i = 0; i < nstage; ++i) (void)mbar_wait_limit(&full[i], (uint32_t)(((nst - 1 - i) / nstage) & 1), 1u << 12);
      atomicOr(p.status, LORA_DEV_TIMEOUT);
    }
    return;
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
  for (int e = threadIdx.x; e < t.rows * Q4; e += DTHREADS) {
    const int r = e / Q4, cc = (e % Q4) * 4;
    *reinterpret_cast<float4*>(&up[(long long)(t.row0 + r) * NR + cc]) =
        *reinterpret_cast<const float4*>(&P[r * Cfg::PPITCH + cc]);
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

template <int NR>
cudaError_t launch_dec_t(const ProblemDesc& p, const DecMaps& maps, float* u, cudaStream_t s, int C) {
  auto kernel = sgmv_shrink_tma_kernel<NR>;
  const int Kc = p.in_dim / C;
  const int nst = Kc / DK;
  // Ring: every stage of the split when ~100 KB hold them, else as many.
  int nstage = nst < MAX_STAGES ? nst : MAX_STAGES;
  while (nstage > 2 && nstage * DecCfg<NR>::STAGE > 100 * 1024) --nstage;
  int smem = nstage * DecCfg<NR>::STAGE;
  if (smem < DecCfg<NR>::P_BYTES) smem = DecCfg<NR>::P_BYTES;
  smem += 1024;  // alignment slack
  static unsigned long long done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(g_dec_mu);
    if (!(done & (1ull << (dev & 63)))) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               MAX_STAGES * DecCfg<NR>::STAGE + 1024);  // >= P_BYTES + 1024
      if (e != cudaSuccess) return e;
      done |= 1ull << (dev & 63);
    }
  }
  const long long tiles = (long long)p.G + p.end / DT;
  const long long plane_stride = (long long)p.end * p.n_slices * p.R;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * C));
  cfg.blockDim = dim3(DTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];  // overlap the launch with the previous kernel's tail
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return noted(cudaLaunchKernelEx(&cfg, kernel, p, maps, u, C, Kc, nstage, plane_stride), LORA_PATH_MMA_SHRINK);
}

}  // namespace

bool dec_shrink_ok(const ProblemDesc& p) {
  const int nR = p.n_slices * p.R;
  if (p.token_rows || p.slot_ranks) return false;  // plain batches only
  if (p.R != 16 && p.R != 32) return false;
  return nR <= 128 && p.in_dim % DK == 0;
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

}  // namespace lora
