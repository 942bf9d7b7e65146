// simple_kernels.cu -- the generic SGMV kernels (any storage type, any
// alignment, any rank) and the load-time slot preparation kernel.
//
// These serve fp32 problems and bf16 problems whose shapes or alignments the
// tensor-core path does not take.  One warp computes one element of the
// rank-R intermediate (lanes split the input dimension, shuffle reduction);
// one thread computes one output element of the expand.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "tiles.cuh"

namespace lora {

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// u[t, j*R + k] = sum_i A_j[slot, k, i] * x[t, i]; one warp per (t, j*R+k).
template <typename T>
__global__ void __launch_bounds__(256) shrink_simple_kernel(const __grid_constant__ ProblemDesc p,
                                                            float* __restrict__ u) {
  __shared__ int s_ok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    const bool ok = warp_check_routing(p);
    if (lane == 0) s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;
  const int nR = p.n_slices * p.R;
  const long long task = (long long)blockIdx.x * 8 + warp;
  if (task >= (long long)p.end * nR) return;
  const int t = (int)(task / nR);
  const int col = (int)(task % nR);
  const int j = col / p.R, k = col % p.R;
  const int slot = p.lora_ids[group_of_row(p, t)];
  if (k >= slot_kmax(p, slot)) {  // past the slot's rank: zero, A not read
    if (lane == 0) u[(long long)t * nR + col] = 0.f;
    return;
  }
  const T* a = static_cast<const T*>(p.sl[j].A) + (long long)slot * p.sl[j].A_slot_stride +
               (long long)k * p.in_dim;
  const int xr = p.token_rows ? p.token_rows[t] : t;  // row of x holding token t
  if (xr < 0 || xr >= p.num_tokens) {
    if (lane == 0) atomicOr(p.status, LORA_DEV_BAD_ROW);
    return;
  }
  const T* x = static_cast<const T*>(p.x) + (long long)xr * p.x_row_stride;
  float acc = 0.f;
  for (int i = lane; i < p.in_dim; i += 32) acc = fmaf(to_f32(a[i]), to_f32(x[i]), acc);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
  if (lane == 0) u[(long long)t * nR + col] = acc;
}

// y_j[t, o] = rn(y_j[t, o] + sum_k B_j[slot, o, k] * u[t, j*R + k]); one
// thread per (t, output column across all slices).
template <typename T>
__global__ void __launch_bounds__(256) expand_simple_kernel(const __grid_constant__ ProblemDesc p,
                                                            const float* __restrict__ u) {
  __shared__ int s_ok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    const bool ok = warp_check_routing(p);
    if (lane == 0) s_ok = ok;
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!s_ok) return;
  int O = 0;
  for (int j = 0; j < p.n_slices; ++j) O += p.sl[j].out_dim;
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)p.end * O) return;
  const int t = (int)(e / O);
  int o = (int)(e % O);
  int j = 0;
  while (o >= p.sl[j].out_dim) o -= p.sl[j++].out_dim;
  const int slot = p.lora_ids[group_of_row(p, t)];
  const int nR = p.n_slices * p.R;
  const T* b = static_cast<const T*>(p.sl[j].B) + (long long)slot * p.sl[j].B_slot_stride +
               (long long)o * p.R;
  const float* ut = u + (long long)t * nR + (long long)j * p.R;
  const int yr = p.token_rows ? p.token_rows[t] : t;  // row of y holding token t
  if (yr < 0 || yr >= p.num_tokens) {
    atomicOr(p.status, LORA_DEV_BAD_ROW);
    return;
  }
  T* y = static_cast<T*>(p.sl[j].y) + (long long)yr * p.sl[j].y_row_stride + o;
  float acc = 0.f;
  const int kmax = slot_kmax(p, slot);
  for (int k = 0; k < kmax; ++k) acc = fmaf(to_f32(b[k]), ut[k], acc);
  if (p.sl[j].bias)
    acc += to_f32(static_cast<const T*>(p.sl[j].bias)[(long long)slot * p.sl[j].bias_slot_stride + o]);
  *y = from_f32<T>(to_f32(*y) + acc);
}

// Slot preparation: A rows k < r copied (cast to the storage type), rows >= r
// zero; B columns k < r get rn(fp32(B_raw) * scale), columns >= r zero.
template <typename T, typename RawT>
__global__ void set_slot_kernel(const __grid_constant__ ProblemDesc p, int slice, int slot, int r,
                                float scale, const RawT* __restrict__ A_raw,
                                const RawT* __restrict__ B_raw) {
  const SliceDesc& sl = p.sl[slice];
  const long long na = (long long)p.R * p.in_dim;
  const long long nb = (long long)sl.out_dim * p.R;
  T* A = static_cast<T*>(const_cast<void*>(sl.A)) + (long long)slot * sl.A_slot_stride;
  T* B = static_cast<T*>(const_cast<void*>(sl.B)) + (long long)slot * sl.B_slot_stride;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < na + nb;
       e += (long long)gridDim.x * blockDim.x) {
    if (e < na) {
      const int k = (int)(e / p.in_dim);
      const int i = (int)(e % p.in_dim);
      A[e] = k < r ? from_f32<T>(to_f32(A_raw[(long long)k * p.in_dim + i])) : from_f32<T>(0.f);
    } else {
      const long long f = e - na;
      const int o = (int)(f / p.R);
      const int k = (int)(f % p.R);
      float v = 0.f;
      if (k < r) v = __fmul_rn(to_f32(B_raw[(long long)o * r + k]), scale);
      B[f] = from_f32<T>(v);
    }
  }
}

// Bias preparation: bias[slot, o] = cast(bias_raw[o]), or zero when bias_raw is null.
template <typename T, typename RawT>
__global__ void set_bias_kernel(const __grid_constant__ ProblemDesc p, int slice, int slot,
                                const RawT* __restrict__ bias_raw) {
  const SliceDesc& sl = p.sl[slice];
  T* b = static_cast<T*>(const_cast<void*>(sl.bias)) + (long long)slot * sl.bias_slot_stride;
  for (int o = blockIdx.x * blockDim.x + threadIdx.x; o < sl.out_dim; o += gridDim.x * blockDim.x)
    b[o] = bias_raw ? from_f32<T>(to_f32(bias_raw[o])) : from_f32<T>(0.f);
}

cudaError_t launch_set_bias(const ProblemDesc& p, int slice, int slot, const void* bias_raw, int raw_dtype,
                            cudaStream_t s) {
  const unsigned g = (unsigned)((p.sl[slice].out_dim + 255) / 256);
  if (p.dtype == LORA_DTYPE_BF16) {
    if (raw_dtype == LORA_DTYPE_BF16)
      set_bias_kernel<__nv_bfloat16, __nv_bfloat16><<<g, 256, 0, s>>>(p, slice, slot, (const __nv_bfloat16*)bias_raw);
    else
      set_bias_kernel<__nv_bfloat16, float><<<g, 256, 0, s>>>(p, slice, slot, (const float*)bias_raw);
  } else {
    if (raw_dtype == LORA_DTYPE_BF16)
      set_bias_kernel<float, __nv_bfloat16><<<g, 256, 0, s>>>(p, slice, slot, (const __nv_bfloat16*)bias_raw);
    else
      set_bias_kernel<float, float><<<g, 256, 0, s>>>(p, slice, slot, (const float*)bias_raw);
  }
  return noted(cudaGetLastError(), LORA_PATH_PREP);
}

cudaError_t launch_shrink_simple(const ProblemDesc& p, float* u, cudaStream_t s) {
  const long long tasks = (long long)p.end * p.n_slices * p.R;
  const long long blocks = (tasks + 7) / 8;
  if (p.dtype == LORA_DTYPE_BF16)
    shrink_simple_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(p, u);
  else
    shrink_simple_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(p, u);
  return noted(cudaGetLastError(), LORA_PATH_GENERIC_SHRINK);
}

cudaError_t launch_expand_simple(const ProblemDesc& p, const float* u, cudaStream_t s, bool pdl) {
  int O = 0;
  for (int j = 0; j < p.n_slices; ++j) O += p.sl[j].out_dim;
  const long long elems = (long long)p.end * O;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((elems + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (p.dtype == LORA_DTYPE_BF16)
    return noted(cudaLaunchKernelEx(&cfg, expand_simple_kernel<__nv_bfloat16>, p, u), LORA_PATH_GENERIC_EXPAND);
  return noted(cudaLaunchKernelEx(&cfg, expand_simple_kernel<float>, p, u), LORA_PATH_GENERIC_EXPAND);
}

cudaError_t launch_set_slot(const ProblemDesc& p, int slice, int slot, int r, float scale,
                            const void* A_raw, const void* B_raw, int raw_dtype, cudaStream_t s) {
  const long long total = (long long)p.R * p.in_dim + (long long)p.sl[slice].out_dim * p.R;
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  const unsigned g = (unsigned)blocks;
  if (p.dtype == LORA_DTYPE_BF16) {
    if (raw_dtype == LORA_DTYPE_BF16)
      set_slot_kernel<__nv_bfloat16, __nv_bfloat16><<<g, 256, 0, s>>>(
          p, slice, slot, r, scale, (const __nv_bfloat16*)A_raw, (const __nv_bfloat16*)B_raw);
    else
      set_slot_kernel<__nv_bfloat16, float><<<g, 256, 0, s>>>(p, slice, slot, r, scale,
                                                               (const float*)A_raw,
                                                               (const float*)B_raw);
  } else {
    if (raw_dtype == LORA_DTYPE_BF16)
      set_slot_kernel<float, __nv_bfloat16><<<g, 256, 0, s>>>(
          p, slice, slot, r, scale, (const __nv_bfloat16*)A_raw, (const __nv_bfloat16*)B_raw);
    else
      set_slot_kernel<float, float><<<g, 256, 0, s>>>(p, slice, slot, r, scale,
                                                       (const float*)A_raw, (const float*)B_raw);
  }
  return noted(cudaGetLastError(), LORA_PATH_PREP);
}

// Failure-path self test: one thread waits on a fresh barrier that nothing
// ever completes, gives up after `limit` polls and records the timeout in the
// status word, exactly as the pipelined kernels do when a wait expires.
__global__ void selftest_timeout_kernel(unsigned* status, uint32_t limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_limit(&bar, 0, limit)) atomicOr(status, LORA_DEV_TIMEOUT);
  }
}

cudaError_t launch_selftest_timeout(unsigned* status, uint32_t limit, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 32, 0, s>>>(status, limit);
  return noted(cudaGetLastError(), 0);
}

}  // namespace lora
