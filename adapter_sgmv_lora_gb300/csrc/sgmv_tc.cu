// sgmv_tc.cu -- SGMV shrink on the 5th-generation tensor cores (tcgen05) for
// long groups (prefill), bf16, sm_103a.
//
//   u[t, j*R+k] = sum_i A_j[s, k, i] x[t, i]      for the routed rows t of a group
// ("vLLM LoRA 实现深度解析" sections 1 and 6; routing triple of the
// "max.pipelines.lora.LoRAManagerV3" page, get_lora_graph_inputs).
//
// One CTA per (128-row tile of a group, K split).  Warp-specialised:
//   warp 0  TMA producer: per 64-wide K stage, one box of the tile's x rows
//           (128 x 64) and one box per slice of the slot's A rows (R x 64),
//           both with the 128-byte swizzle, into a ring of stages;
//   warp 1  TMEM owner and MMA issuer: tcgen05.mma M=128, N=n*R (two MMAs of
//           N/2 when n*R > 256), K=16 per instruction, accumulating in TMEM;
//           a tcgen05.commit per stage hands the slot back to the producer;
//   warps 2-5  epilogue: tcgen05.ld of their 32 TMEM lanes (= rows) and
//           16-byte stores of the routed rows of u (partial plane per split).
// Rows of the 128-row box past the group (other groups, base rows, or past
// the tensor: zero-filled) are read but their u rows are never stored.
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
  static constexpr int NSTAGE = (200 * 1024) / STAGE >= 4 ? 4 : (200 * 1024) / STAGE;
  static constexpr int SMEM = NSTAGE * STAGE + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = NR <= 32 ? 32 : NR <= 64 ? 64 : NR <= 128 ? 128 : NR <= 256 ? 256 : 512;
};

}  // namespace

struct TcMaps {
  CUtensorMap x;                    // [T rows, in] bf16, box 64 x 128
  CUtensorMap a[LORA_MAX_SLICES];   // per slice [S, R, in] bf16, box 64 x R x 1
};

template <int NR>
__global__ void __launch_bounds__(TTHREADS, 1) sgmv_tc_shrink_kernel(const __grid_constant__ ProblemDesc p,
                                                                    const __grid_constant__ TcMaps maps,
                                                                    float* __restrict__ u, int nsplit,
                                                                    long long plane_stride) {
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

  pdl_launch_dependents();
  // 1024-byte aligned ring (the 128-byte swizzle repeats every 1024 bytes).
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = (int)(blockIdx.x % (unsigned)nsplit);
  const long long tile = blockIdx.x / (unsigned)nsplit;
  if (warp == 0) {
    Tile t{};
    const bool ok = warp_locate_tile(p, TM, tile, t);
    if (lane == 0) {
      s_tile = t;
      s_ok = ok;
      s_fail = 0;
      for (int i = 0; i < NSTAGE; ++i) {
        mbar_init(&full[i], 1);
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
  const uint32_t tmem = s_tmem;
  const Tile t = s_tile;
  const bool ok = s_ok != 0;
  const int R = p.R;
  const int kc = p.in_dim / nsplit;
  const int k0 = split * kc;
  const int nst = kc / TK;

  if (ok && warp == 0 && lane == 0) {
    // ---- producer
    for (int s = 0; s < nst; ++s) {
      const int slot = s % NSTAGE;
      if (s >= NSTAGE && !mbar_wait(&empty[slot], (uint32_t)(((s / NSTAGE) - 1) & 1))) {
        atomicOr(&s_fail, 1);
        break;
      }
      uint8_t* xs = smem + slot * Cfg::STAGE;
      uint8_t* as = xs + Cfg::X_BYTES;
      mbar_arrive_expect_tx(&full[slot], (uint32_t)(Cfg::X_BYTES + p.n_slices * R * TK * 2));
      const int kk = k0 + s * TK;
      tma_load_2d(xs, &maps.x, kk, t.row0, &full[slot]);
      for (int j = 0; j < p.n_slices; ++j) tma_load_3d(as + j * R * TK * 2, &maps.a[j], kk, 0, t.slot, &full[slot]);
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
    // ---- epilogue: warp w reads TMEM lanes 32*(w % 4) .. +31 (= tile rows)
    const bool got = mbar_wait(&done, 0);
    tc_fence_after_sync();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int nR = p.n_slices * R;
    float* up = u + split * plane_stride + (long long)(t.row0 + row) * nR;
    if (!got) {
      atomicOr(&s_fail, 1);
    } else {
      for (int c = 0; c < nR; c += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
        if (row < t.rows) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(up + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
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
    const cuuint64_t dims[2] = {(cuuint64_t)p.in_dim, (cuuint64_t)p.num_tokens};
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
    if (enc(&m->a[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.sl[j].A), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

template <int NR>
cudaError_t launch_tc_t(const ProblemDesc& p, const TcMaps& maps, float* u, cudaStream_t s, int nsplit) {
  auto kernel = sgmv_tc_shrink_kernel<NR>;
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
  cfg.gridDim = dim3((unsigned)(tiles * nsplit));
  cfg.blockDim = dim3(TTHREADS);
  cfg.dynamicSmemBytes = TcCfg<NR>::SMEM;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kernel, p, maps, u, nsplit, plane_stride);
}

}  // namespace

int tc_shrink_splits(int end, int in_dim) {
  // Shape-only: split K (1, 2 or 4 planes) while a lower bound on the tiles
  // times the split stays within 152 CTAs and each split is whole stages.
  if (end <= 0 || in_dim % TK != 0) return 1;
  const long long tiles = (end + TM - 1) / TM;
  int n = 1;
  while (n < 4 && tiles * n * 2 <= 152 && (in_dim / TK) % (n * 2) == 0) n *= 2;
  return n;
}

bool tc_shrink_ok(const ProblemDesc& p) {
  const int nR = p.n_slices * p.R;
  switch (nR) {
    case 16: case 32: case 48: case 64: case 96: case 128: case 192: case 256: case 384: break;
    default: return false;
  }
  if (p.R % 8 != 0 || p.in_dim % TK != 0) return false;
  // Long groups only: on average at least 96 routed rows per group.
  return p.G > 0 && p.end >= 96LL * p.G;
}

cudaError_t launch_tc_shrink(const ProblemDesc& p, float* u, cudaStream_t s, int nsplit) {
  TcMaps maps;
  if (!encode_maps(p, &maps)) return cudaErrorNotSupported;
  switch (p.n_slices * p.R) {
    case 16: return launch_tc_t<16>(p, maps, u, s, nsplit);
    case 32: return launch_tc_t<32>(p, maps, u, s, nsplit);
    case 48: return launch_tc_t<48>(p, maps, u, s, nsplit);
    case 64: return launch_tc_t<64>(p, maps, u, s, nsplit);
    case 96: return launch_tc_t<96>(p, maps, u, s, nsplit);
    case 128: return launch_tc_t<128>(p, maps, u, s, nsplit);
    case 192: return launch_tc_t<192>(p, maps, u, s, nsplit);
    case 256: return launch_tc_t<256>(p, maps, u, s, nsplit);
    case 384: return launch_tc_t<384>(p, maps, u, s, nsplit);
  }
  return cudaErrorNotSupported;
}

}  // namespace lora
