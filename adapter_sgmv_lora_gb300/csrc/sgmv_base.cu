// sgmv_base.cu -- the LoRA delta fused into the base projection:
//
//   y_j[t, o] = rn( sum_i W0_j[o, i] x[t, i]
//                   + [t < end] (bias_j[s, o] + sum_k B_j[s, o, k] u[t, j*R + k]) )
//
// for every row t of the batch, with s the slot of t's group ("vLLM LoRA
// 实现深度解析" section 1: h = W0 x + (alpha/r) B A x, the scale folded into B;
// the routing triple of the "max.pipelines.lora.LoRAManagerV3" page,
// get_lora_graph_inputs).  y is written, not read: the delta joins the base
// product in the accumulator, so the expand's read-modify-write of y
// disappears.  u (the shrink's fp32 partial planes, summed here) comes from
// the library's shrink kernels, launched first on the same stream.
//
// Tensor cores (tcgen05), one CTA per (128-row tile of the batch, 128- or
// 256-column block of one slice's outputs), 6 warps:
//   warp 0   TMA producer: per 64-wide K stage one box of the tile's x rows
//            (128 x 64) and one of the block's W0 rows (N x 64), 128-byte
//            swizzle, through a ring of stages;
//   warp 1   TMEM owner and MMA issuer: M=128 N=128 or 256, K=16 per instruction,
//            then the LoRA K tail: for every group overlapping the tile, K = 2R
//            more steps with the masked u image (u's hi part, then its lo part:
//            u = hi + lo, both bf16, exact split) against the slot's B block;
//   warps 2-5  first build the K-tail operands (one tile row / one output row
//            per thread): u rows of the group (other rows zero) summed over
//            the planes and split into hi | lo, and the slot's B rows, in the
//            same 128-byte-swizzled K-major layout the TMA boxes have; then the
//            epilogue: TMEM -> registers, + bias, one rounding, stores.
// The K tail reuses one operand buffer per group (built while the previous
// group's MMAs drain).  Every mbarrier wait is bounded; on expiry the CTA
// raises LORA_DEV_TIMEOUT, stores nothing and still releases its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tiles.cuh"

namespace lora {

namespace {

constexpr int BM = 128;        // rows per tile (MMA M)
constexpr int BK = 64;         // K per stage
constexpr int BTHREADS = 192;  // 6 warps
constexpr int MAX_STAGES_B = 4;
constexpr int MAX_TILE_GROUPS = BM;  // a 128-row tile overlaps at most 128 non-empty groups

// BN: output columns per tile (MMA N): 128, or 256 for batches of many
// rows (twice the MMA work per byte staged).
template <int R, int BN_>
struct BaseCfg {
  static constexpr int BN = BN_;
  static constexpr int X_BYTES = BM * BK * 2;                // 16 KB
  static constexpr int W_BYTES = BN * BK * 2;                // 16 or 32 KB
  static constexpr int STAGE = X_BYTES + W_BYTES;
  static constexpr int UB = (2 * R + 63) / 64;               // 64-wide K blocks of u's hi | lo
  static constexpr int BB = (R + 63) / 64;                   // 64-wide K blocks of B
  static constexpr int U_BYTES = UB * BM * 128;
  static constexpr int B_BYTES = BB * BN * 128;
  // Ring depth: as many stages as ~224 KB hold next to the K-tail operands.
  static constexpr int BSTAGES_RAW = (224 * 1024 - U_BYTES - B_BYTES - 1024) / STAGE;
  static constexpr int BSTAGES = BSTAGES_RAW > 4 ? 4 : BSTAGES_RAW;
  static_assert(BSTAGES >= 2, "ring too shallow");
  static constexpr int SMEM = BSTAGES * STAGE + U_BYTES + B_BYTES + 1024;
};

template <typename T>
__device__ __forceinline__ float to_float(T v);
template <>
__device__ __forceinline__ float to_float<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T>
__device__ __forceinline__ T from_float(float v);
template <>
__device__ __forceinline__ float from_float<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Byte offset of bf16 element (row r, k) in a K-major operand of [rows x 64]
// blocks with the 128-byte swizzle (16-byte chunk c of row r at c ^ (r % 8)).
__device__ __forceinline__ uint32_t bsw(int r, int k, int rows) {
  const int kb = k >> 6, kk = k & 63;
  return (uint32_t)(kb * rows * 128 + r * 128 + ((((kk >> 3) ^ (r & 7))) << 4) + ((kk & 7) << 1));
}

}  // namespace

struct BaseMaps {
  CUtensorMap x;                    // [T rows, in] bf16, box 64 x 128
  CUtensorMap w[LORA_MAX_SLICES];   // per slice W0 [out_j rows, in] bf16, box 64 x BN
};

struct BaseWork {
  int nbt;                             // column blocks, all slices
  int blk_begin[LORA_MAX_SLICES + 1];  // first block of each slice
  int nsplit;                          // partial planes of u
  long long plane_stride;              // floats between planes
  int wait_first;                      // 1: no shrink precedes; every role waits for the previous kernel
};

template <int R, int BN>
__global__ void __launch_bounds__(BTHREADS, 1) sgmv_base_gemm_kernel(const __grid_constant__ ProblemDesc p,
                                                                     const __grid_constant__ BaseMaps maps,
                                                                     const __grid_constant__ BaseWork w,
                                                                     const float* __restrict__ u) {
  using Cfg = BaseCfg<R, BN>;
  constexpr int BSTAGES = Cfg::BSTAGES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[MAX_STAGES_B], empty[MAX_STAGES_B], uready, ufree, done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_ok, s_fail, s_ng;
  __shared__ int s_glo[MAX_TILE_GROUPS], s_ghi[MAX_TILE_GROUPS], s_gslot[MAX_TILE_GROUPS];
  __shared__ int s_rowslot[BM];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Us = smem + BSTAGES * Cfg::STAGE;
  uint8_t* Bs = Us + Cfg::U_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x;   // column block over all slices
  const int row0 = blockIdx.y * BM;
  int j = 0;
  while (j + 1 < p.n_slices && b >= w.blk_begin[j + 1]) ++j;
  const int o0 = (b - w.blk_begin[j]) * BN;
  const SliceDesc& sl = p.sl[j];

  if (w.wait_first) pdl_wait();  // x may come from the previous kernel
  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < BSTAGES; ++i) {
        mbar_init(&full[i], 1);
        mbar_init(&empty[i], 1);
      }
      mbar_init(&uready, 4 * 32);
      mbar_init(&ufree, 1);
      mbar_init(&done, 1);
      s_fail = 0;
      fence_mbar_init();
    }
  } else if (warp == 1) {
    tmem_alloc(&s_tmem, BN);
    tmem_relinquish();
  } else if (warp == 2) {
    // The routing (validated) and the groups overlapping this tile's rows.
    bool valid = true;
    if (p.G > 0) valid = warp_check_routing(p);
    const int lo_t = row0, hi_t = min(row0 + BM, p.end);
    int n = 0;
    for (int c = 0; valid && c < p.G; c += 32) {
      const int g = c + lane;
      bool hit = false;
      int lo = 0, hi = 0, slot = 0;
      if (g < p.G) {
        lo = max(p.offs[g], lo_t);
        hi = min(p.offs[g + 1], hi_t);
        slot = p.lora_ids[g];
        hit = hi > lo;
      }
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      const int pos = n + __popc(m & ((1u << lane) - 1u));
      if (hit && pos < MAX_TILE_GROUPS) {
        s_glo[pos] = lo;
        s_ghi[pos] = hi;
        s_gslot[pos] = slot;
      }
      n += __popc(m);
    }
    if (lane == 0) {
      s_ok = valid;
      s_ng = n < MAX_TILE_GROUPS ? n : MAX_TILE_GROUPS;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;
  const bool ok = s_ok != 0;
  const int ng = s_ng;
  const int nst = p.in_dim / BK;

  if (ok && warp >= 2) {  // slot of each tile row (bias), -1 for rows without a group
    for (int r = threadIdx.x - 64; r < BM; r += 128) s_rowslot[r] = -1;
  }
  __syncthreads();
  if (ok && warp >= 2) {
    for (int g = 0; g < ng; ++g)
      for (int r = s_glo[g] + (int)threadIdx.x - 64; r < s_ghi[g]; r += 128) s_rowslot[r - row0] = s_gslot[g];
  }

  if (ok && warp == 0 && lane == 0) {
    // ---- producer: x rows of the tile and W0 rows of the block
    const uint64_t pol_x = policy_evict_last(), pol_w = policy_evict_first();
    for (int s = 0; s < nst; ++s) {
      const int slot = s % BSTAGES;
      if (s >= BSTAGES && !mbar_wait(&empty[slot], (uint32_t)(((s / BSTAGES) - 1) & 1))) {
        atomicOr(&s_fail, 1);
        break;
      }
      uint8_t* xs = smem + slot * Cfg::STAGE;
      mbar_arrive_expect_tx(&full[slot], (uint32_t)Cfg::STAGE);
      tma_load_2d_hint(xs, &maps.x, s * BK, row0, &full[slot], pol_x);
      tma_load_2d_hint(xs + Cfg::X_BYTES, &maps.w[j], s * BK, o0, &full[slot], pol_w);
    }
  } else if (ok && warp == 1 && lane == 0) {
    // ---- MMA issuer: base product, then one K tail per group
    constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
    bool bad = false;
    for (int s = 0; s < nst && !bad; ++s) {
      const int slot = s % BSTAGES;
      if (!mbar_wait(&full[slot], (uint32_t)((s / BSTAGES) & 1))) {
        bad = true;
        break;
      }
      tc_fence_after_sync();
      const uint32_t xs = smem_addr(smem + slot * Cfg::STAGE);
      const uint32_t ws = xs + Cfg::X_BYTES;
#pragma unroll
      for (int ks = 0; ks < BK / 16; ++ks)
        tc_mma_bf16(tmem, sw128_desc(xs + ks * 32), sw128_desc(ws + ks * 32), idesc, (s > 0 || ks > 0) ? 1u : 0u);
      tc_commit(&empty[slot]);
    }
    for (int g = 0; g < ng && !bad; ++g) {
      if (!mbar_wait(&uready, (uint32_t)(g & 1))) {
        bad = true;
        break;
      }
      tc_fence_after_sync();
      const int kmax = slot_kmax(p, s_gslot[g]);
      const uint32_t ua = smem_addr(Us), ba = smem_addr(Bs);
#pragma unroll
      for (int ks = 0; ks < 2 * R / 16; ++ks) {
        const int kb = (ks * 16) % R;  // the lo half reuses B's K columns
        if (kb >= kmax) continue;      // past the slot's rank
        tc_mma_bf16(tmem, sw128_desc(ua + (ks >> 2) * BM * 128 + (ks & 3) * 32),
                    sw128_desc(ba + (kb >> 6) * BN * 128 + ((kb & 63) >> 4) * 32), idesc, 1u);
      }
      tc_commit(&ufree);  // the operand buffer is free once these MMAs finish
    }
    if (bad) atomicOr(&s_fail, 1);
    tc_commit(&done);  // accumulator complete (every MMA issued so far)
  } else if (ok && warp >= 2) {
    // ---- K-tail operands, then the epilogue.  Thread = tile row / block row.
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int nR = p.n_slices * R;
    if (!w.wait_first) pdl_wait();  // the planes of u come from the shrink grid
    bool bad = false;
    for (int g = 0; g < ng; ++g) {
      if (g > 0 && !bad && !mbar_wait(&ufree, (uint32_t)((g - 1) & 1))) bad = true;
      bad = __any_sync(0xffffffffu, bad);
      if (!bad) {
        // B rows: outputs o0 + r (+ 128, ...) of the slot, K columns [0, min(R, kmax)).
        const int slot = s_gslot[g];
        const int kmax = slot_kmax(p, slot);
        for (int br = r; br < BN; br += BM) {
          if (o0 + br < sl.out_dim) {
            const __nv_bfloat16* brow = static_cast<const __nv_bfloat16*>(sl.B) +
                                        (long long)slot * sl.B_slot_stride + (long long)(o0 + br) * R;
            for (int c = 0; c * 8 < kmax; ++c) cp_async16(Bs + bsw(br, 8 * c, BN), brow + 8 * c);
          }
        }
        cp_async_commit();
        // u rows of the group (sum of the planes, plane order), hi | lo; zero elsewhere.
        const int t = row0 + r;
        const bool mine = t >= s_glo[g] && t < s_ghi[g];
        const float* ur = u + (long long)(mine ? t : 0) * nR + (long long)j * R;
        for (int k = 0; k < R; k += 8) {
          float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (mine && k < kmax) {
            for (int sp = 0; sp < w.nsplit; ++sp) {
              const float4 a = __ldcg(reinterpret_cast<const float4*>(ur + sp * w.plane_stride + k));
              const float4 c4 = __ldcg(reinterpret_cast<const float4*>(ur + sp * w.plane_stride + k + 4));
              v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
              v[4] += c4.x; v[5] += c4.y; v[6] += c4.z; v[7] += c4.w;
            }
          }
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_hi_lo_bf16x2(v[2 * e], v[2 * e + 1], hi[e], lo[e]);
          *reinterpret_cast<uint4*>(Us + bsw(r, k, BM)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(Us + bsw(r, R + k, BM)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        cp_async_wait<0>();
      }
      fence_proxy_async_smem();  // generic and async-copy writes -> visible to the tensor cores
      mbar_arrive(&uready);
    }
    // ---- epilogue
    if (!bad && !mbar_wait(&done, 0)) bad = true;
    bad = __any_sync(0xffffffffu, bad);  // tcgen05.ld below needs the whole warp
    tc_fence_after_sync();
    if (bad) {
      if (lane == 0) atomicOr(&s_fail, 1);
    } else {
      const int t = row0 + r;
      const int rs = s_rowslot[r];
      const int ovalid = min(BN, sl.out_dim - o0);
      __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(sl.y) + (long long)t * sl.y_row_stride + o0;
      const __nv_bfloat16* brow =
          (sl.bias && rs >= 0) ? static_cast<const __nv_bfloat16*>(sl.bias) + (long long)rs * sl.bias_slot_stride + o0
                               : nullptr;
      for (int c32 = 0; c32 < BN / 32; ++c32) {
        float d[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c32 * 32), d);
        if (t < p.num_tokens) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int c = c32 * 32 + h * 8;
            if (c >= ovalid) continue;
            float e[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) e[i] = d[h * 8 + i];
            if (brow) {  // the bias joins the sum before the one rounding
              const uint4 bv = __ldg(reinterpret_cast<const uint4*>(brow + c));
              const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                e[2 * i] += __uint_as_float(bw[i] << 16);
                e[2 * i + 1] += __uint_as_float(bw[i] & 0xFFFF0000u);
              }
            }
            uint4 o;
            o.x = round_pack_bf16x2(e[0], e[1]);
            o.y = round_pack_bf16x2(e[2], e[3]);
            o.z = round_pack_bf16x2(e[4], e[5]);
            o.w = round_pack_bf16x2(e[6], e[7]);
            *reinterpret_cast<uint4*>(yrow + c) = o;
          }
        }
      }
    }
  }
  pdl_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    if (s_fail) {
      (void)mbar_wait(&done, 0);  // MMAs in flight finish before the columns are released
      if (lane == 0) atomicOr(p.status, LORA_DEV_TIMEOUT);
    }
    tc_fence_after_sync();
    tmem_dealloc(tmem, BN);
  }
}

// Any shape and storage type: one thread per output element, fp32 sums.
// u is the generic shrink's single plane [end, n*R].
template <typename T>
__global__ void __launch_bounds__(256) base_gemm_simple_kernel(const __grid_constant__ ProblemDesc p,
                                                               const __grid_constant__ BaseWeights wts,
                                                               const float* __restrict__ u, int wait_first) {
  __shared__ int s_ok;
  (void)wait_first;
  pdl_wait();  // x from the kernel before, u from the shrink
  if ((threadIdx.x >> 5) == 0) {
    const bool ok = p.G == 0 || warp_check_routing(p);
    if ((threadIdx.x & 31) == 0) s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;
  int O = 0;
  for (int jj = 0; jj < p.n_slices; ++jj) O += p.sl[jj].out_dim;
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)p.num_tokens * O) return;
  const int t = (int)(e / O);
  int col = (int)(e % O);
  int j = 0;
  while (col >= p.sl[j].out_dim) col -= p.sl[j++].out_dim;
  const SliceDesc& sl = p.sl[j];
  const T* x = static_cast<const T*>(p.x) + (long long)t * p.x_row_stride;
  const T* w0 = static_cast<const T*>(wts.W0[j]) + (long long)col * wts.row_stride[j];
  float acc = 0.f;
  for (int i = 0; i < p.in_dim; ++i) acc += to_float(w0[i]) * to_float(x[i]);
  if (t < p.end) {
    const int slot = p.lora_ids[group_of_row(p, t)];
    const int kmax = slot_kmax(p, slot);
    const T* brow = static_cast<const T*>(sl.B) + (long long)slot * sl.B_slot_stride + (long long)col * p.R;
    const float* ur = u + (long long)t * p.n_slices * p.R + (long long)j * p.R;
    for (int k = 0; k < kmax; ++k) acc += to_float(brow[k]) * ur[k];
    if (sl.bias) acc += to_float(static_cast<const T*>(sl.bias)[(long long)slot * sl.bias_slot_stride + col]);
  }
  static_cast<T*>(sl.y)[(long long)t * sl.y_row_stride + col] = from_float<T>(acc);
}

// ------------------------------------------------------------------ host

namespace {

std::mutex g_base_mu;

PFN_cuTensorMapEncodeTiled_v12000 base_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lk(g_base_mu);
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

// Tile width: 256 output columns for batches of at least this many rows
// (long K loops at full MMA rate need twice the work per staged byte), 128
// otherwise (more CTAs for small batches).  Ranks above 64 keep 128 (the
// K-tail operands would leave too shallow a ring).
constexpr int kWideTileRows = 1024;
int base_bn(const ProblemDesc& p) { return (p.num_tokens >= kWideTileRows && p.R <= 64) ? 256 : 128; }

bool encode_base_maps(const ProblemDesc& p, const BaseWeights& wts, BaseMaps* m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = base_encode_fn();
  if (!enc) return false;
  const cuuint32_t es[2] = {1, 1};
  const cuuint32_t box[2] = {(cuuint32_t)BK, 128};
  const cuuint32_t wbox[2] = {(cuuint32_t)BK, (cuuint32_t)base_bn(p)};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.in_dim, (cuuint64_t)p.num_tokens};
    const cuuint64_t strides[1] = {(cuuint64_t)p.x_row_stride * 2};
    if (enc(&m->x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  for (int j = 0; j < p.n_slices; ++j) {
    const cuuint64_t dims[2] = {(cuuint64_t)p.in_dim, (cuuint64_t)p.sl[j].out_dim};
    const cuuint64_t strides[1] = {(cuuint64_t)wts.row_stride[j] * 2};
    if (enc(&m->w[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(wts.W0[j]), dims, strides, wbox, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

template <int R, int BN>
cudaError_t launch_base_t(const ProblemDesc& p, const BaseMaps& maps, const BaseWork& w, const float* u,
                          cudaStream_t s) {
  auto kernel = sgmv_base_gemm_kernel<R, BN>;
  static unsigned long long done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(g_base_mu);
    if (!(done & (1ull << (dev & 63)))) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BaseCfg<R, BN>::SMEM);
      if (e != cudaSuccess) return e;
      done |= 1ull << (dev & 63);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)w.nbt, (unsigned)((p.num_tokens + BM - 1) / BM));
  cfg.blockDim = dim3(BTHREADS);
  cfg.dynamicSmemBytes = BaseCfg<R, BN>::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return noted(cudaLaunchKernelEx(&cfg, kernel, p, maps, w, u), LORA_PATH_BASE_GEMM);
}

}  // namespace

bool base_tc_ok(const ProblemDesc& p, const BaseWeights& wts) {
  if (!fast_path_ok(p, nullptr) || p.token_rows) return false;
  if (p.in_dim % BK != 0 || p.num_tokens < 1) return false;
  for (int j = 0; j < p.n_slices; ++j) {
    if ((reinterpret_cast<uintptr_t>(wts.W0[j]) & 15u) != 0 || wts.row_stride[j] % 8 != 0) return false;
    if (p.sl[j].bias && (reinterpret_cast<uintptr_t>(p.sl[j].bias) & 15u) != 0) return false;
  }
  return true;
}

bool base_maps_ok(const ProblemDesc& p, const BaseWeights& wts) {
  BaseMaps maps;
  return encode_base_maps(p, wts, &maps);
}

cudaError_t launch_base_gemm(const ProblemDesc& p, const BaseWeights& wts, const float* u, int nsplit, bool after_shrink,
                             cudaStream_t s) {
  BaseMaps maps;
  if (!encode_base_maps(p, wts, &maps)) return cudaErrorNotSupported;
  BaseWork w{};
  const int BN = base_bn(p);
  int acc = 0;
  for (int j = 0; j < p.n_slices; ++j) {
    w.blk_begin[j] = acc;
    acc += (p.sl[j].out_dim + BN - 1) / BN;
  }
  w.blk_begin[p.n_slices] = acc;
  w.nbt = acc;
  w.nsplit = nsplit;
  w.plane_stride = (long long)p.end * p.n_slices * p.R;
  w.wait_first = after_shrink ? 0 : 1;
  if (BN == 256) {
    switch (p.R) {
      case 16: return launch_base_t<16, 256>(p, maps, w, u, s);
      case 32: return launch_base_t<32, 256>(p, maps, w, u, s);
      case 64: return launch_base_t<64, 256>(p, maps, w, u, s);
    }
    return cudaErrorNotSupported;
  }
  switch (p.R) {
    case 16: return launch_base_t<16, 128>(p, maps, w, u, s);
    case 32: return launch_base_t<32, 128>(p, maps, w, u, s);
    case 64: return launch_base_t<64, 128>(p, maps, w, u, s);
    case 128: return launch_base_t<128, 128>(p, maps, w, u, s);
  }
  return cudaErrorNotSupported;
}

cudaError_t launch_base_gemm_simple(const ProblemDesc& p, const BaseWeights& wts, const float* u, bool after_shrink,
                                    cudaStream_t s) {
  int O = 0;
  for (int j = 0; j < p.n_slices; ++j) O += p.sl[j].out_dim;
  const long long elems = (long long)p.num_tokens * O;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((elems + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int wf = after_shrink ? 0 : 1;
  if (p.dtype == LORA_DTYPE_BF16)
    return noted(cudaLaunchKernelEx(&cfg, base_gemm_simple_kernel<__nv_bfloat16>, p, wts, u, wf), LORA_PATH_BASE_GEMM);
  return noted(cudaLaunchKernelEx(&cfg, base_gemm_simple_kernel<float>, p, wts, u, wf), LORA_PATH_BASE_GEMM);
}

}  // namespace lora
