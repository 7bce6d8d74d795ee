// Row-wise RMSNorm (nnterp "input_layernorm" / "post_attention_layernorm";
// "LlamaForCausalLM-32L-4096d" sheet: rmsnorm(x, ..., eps=1e-05)):
//   y[r, :] = x[r, :] * rsqrt(mean(x[r, :]^2) + eps) * g
// Statistics in fp32. HBM-bound: one read and one write of the row with
// 128-bit accesses, the row held in registers between the two passes. x may be
// fp32 while g and y are bf16 (the bf16 path keeps its residual stream in fp32).
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&f)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&f)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = unpack_bf16x2(w[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

template <typename T>
__device__ __forceinline__ void store8(T* p, const float (&f)[8]);
template <>
__device__ __forceinline__ void store8<float>(float* p, const float (&f)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float (&f)[8]) {
  *reinterpret_cast<uint4*>(p) =
      make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}
template <>
__device__ __forceinline__ void store8<__half>(__half* p, const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// NC = chunks of 8 elements per thread, NT threads; TX: x, TY: the gain, TO: y
template <typename TX, typename TY, typename TO, int NC, int NT>
__global__ void __launch_bounds__(NT) rmsnorm_kernel(const TX* __restrict__ x, const TY* __restrict__ g, int rows,
                                                     int n, float eps, TO* __restrict__ y, int* zero_word) {
  constexpr int kThreads = NT;
  pdl_launch_dependents();
  pdl_wait();
  if (zero_word && blockIdx.x == 0 && threadIdx.x == 0) *zero_word = 0;
  __shared__ float red[kThreads / 32];
  const int nchunk = n / 8;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const TX* xr = x + (size_t)r * n;
    float buf[NC][8];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = threadIdx.x + j * kThreads;
      if (c < nchunk) {
        load8<TX>(xr + c * 8, buf[j]);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += buf[j][i] * buf[j][i];
      }
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) tot += red[w];
    __syncthreads();  // red is reused by the next row
    const float inv = rsqrtf(tot / (float)n + eps);
    TO* yr = y + (size_t)r * n;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = threadIdx.x + j * kThreads;
      if (c < nchunk) {
        float gg[8], o[8];
        load8<TY>(g + c * 8, gg);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = buf[j][i] * inv * gg[i];
        store8<TO>(yr + c * 8, o);
      }
    }
  }
}

// Rows of up to 8192 elements take 128 threads (up to 8 chunks of 8 each), so that
// 16 CTAs fit on an SM and every row of a prefill normalises at once; longer rows 256.
template <typename TX, typename TY, typename TO = TY>
cudaError_t launch_t(const void* x, const void* g, int rows, int n, float eps, void* y, cudaStream_t s,
                     int* zero_word) {
  const int nt = n / 8 <= 128 * 8 ? 128 : 256;
  const int nc = (n / 8 + nt - 1) / nt;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int per_sm = nt == 128 ? 16 : 8;
  const int grid = rows < sms * per_sm ? rows : sms * per_sm;
  auto X = static_cast<const TX*>(x);
  auto G = static_cast<const TY*>(g);
  auto Y = static_cast<TO*>(y);
#define BLK_RMS(NC, NT) launch_pdl(rmsnorm_kernel<TX, TY, TO, NC, NT>, grid, NT, 0, s, X, G, rows, n, eps, Y, zero_word)
  if (nt == 128) {
    switch (nc) {
      case 1: BLK_RMS(1, 128); break;
      case 2: BLK_RMS(2, 128); break;
      case 3: BLK_RMS(3, 128); break;
      case 4: BLK_RMS(4, 128); break;
      case 5: BLK_RMS(5, 128); break;
      case 6: BLK_RMS(6, 128); break;
      case 7: BLK_RMS(7, 128); break;
      case 8: BLK_RMS(8, 128); break;
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (nc) {
      case 5: BLK_RMS(5, 256); break;
      case 6: BLK_RMS(6, 256); break;
      case 7: BLK_RMS(7, 256); break;
      case 8: BLK_RMS(8, 256); break;
      default: return cudaErrorInvalidValue;
    }
  }
#undef BLK_RMS
  return cudaGetLastError();
}

template <int NC>
__global__ void __launch_bounds__(kThreads) norm_prep_kernel(const __nv_bfloat16* __restrict__ x,
                                                             const __nv_bfloat16* __restrict__ g, int rows, int n,
                                                             float eps, __nv_bfloat16* __restrict__ xg,
                                                             float* __restrict__ row_scale,
                                                             float* __restrict__ zero_rows) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float red[kThreads / 32];
  const int nchunk = n / 8;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const __nv_bfloat16* xr = x + (size_t)r * n;
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = threadIdx.x + j * kThreads;
      if (c < nchunk) {
        float f[8], gg[8];
        load8<__nv_bfloat16>(xr + c * 8, f);
        load8<__nv_bfloat16>(g + c * 8, gg);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ss += f[i] * f[i];
          f[i] *= gg[i];
        }
        store8<__nv_bfloat16>(xg + (size_t)r * n + c * 8, f);
      }
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) tot += red[w];
      row_scale[r] = rsqrtf(tot / (float)n + eps);
      if (zero_rows) zero_rows[r] = 0.f;
    }
    __syncthreads();
  }
}

__global__ void cast_f16_bf16_kernel(const __half* __restrict__ src, __nv_bfloat16* __restrict__ dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = __float2bfloat16_rn(__half2float(src[i]));
}

__global__ void cast_bf16_f16_kernel(const __nv_bfloat16* __restrict__ src, __half* __restrict__ dst, size_t n,
                                     int* __restrict__ overflow) {
  bool bad = false;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float f = __bfloat162float(src[i]);
    bad |= !(fabsf(f) <= 65504.f);
    dst[i] = __float2half_rn(f);
  }
  if (bad) atomicExch(overflow, 1);
}

}  // namespace

cudaError_t launch_cast_bf16_f16(const void* src, void* dst, size_t n, int* overflow, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  size_t grid = (n + 255) / 256;
  if (grid > 8192) grid = 8192;
  cast_bf16_f16_kernel<<<(int)grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src), static_cast<__half*>(dst), n,
                                                 overflow);
  return cudaGetLastError();
}

cudaError_t launch_norm_prep(const void* x, const void* g, int rows, int n, float eps, void* xg, float* row_scale,
                             float* zero_rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (n % 8) return cudaErrorInvalidValue;
  const int nc = (n / 8 + kThreads - 1) / kThreads;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = rows < sms * 8 ? rows : sms * 8;
  auto X = static_cast<const __nv_bfloat16*>(x);
  auto G = static_cast<const __nv_bfloat16*>(g);
  auto XG = static_cast<__nv_bfloat16*>(xg);
  switch (nc) {
    case 1: launch_pdl(norm_prep_kernel<1>, grid, kThreads, 0, s, X, G, rows, n, eps, XG, row_scale, zero_rows); break;
    case 2: launch_pdl(norm_prep_kernel<2>, grid, kThreads, 0, s, X, G, rows, n, eps, XG, row_scale, zero_rows); break;
    case 3: launch_pdl(norm_prep_kernel<3>, grid, kThreads, 0, s, X, G, rows, n, eps, XG, row_scale, zero_rows); break;
    case 4: launch_pdl(norm_prep_kernel<4>, grid, kThreads, 0, s, X, G, rows, n, eps, XG, row_scale, zero_rows); break;
    case 5: launch_pdl(norm_prep_kernel<5>, grid, kThreads, 0, s, X, G, rows, n, eps, XG, row_scale, zero_rows); break;
    case 6: launch_pdl(norm_prep_kernel<6>, grid, kThreads, 0, s, X, G, rows, n, eps, XG, row_scale, zero_rows); break;
    case 7: launch_pdl(norm_prep_kernel<7>, grid, kThreads, 0, s, X, G, rows, n, eps, XG, row_scale, zero_rows); break;
    case 8: launch_pdl(norm_prep_kernel<8>, grid, kThreads, 0, s, X, G, rows, n, eps, XG, row_scale, zero_rows); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_cast_f16_bf16(const void* src, void* dst, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  size_t grid = (n + 255) / 256;
  if (grid > 4096) grid = 4096;
  cast_f16_bf16_kernel<<<(int)grid, 256, 0, s>>>(static_cast<const __half*>(src), static_cast<__nv_bfloat16*>(dst), n);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const void* x, const void* g, int rows, int n, float eps, void* y, bool bf16,
                           cudaStream_t s, bool x_f32, bool y_f16, int* zero_word) {
  if (rows <= 0) return cudaSuccess;
  if (n % 8) return cudaErrorInvalidValue;
  if (!bf16) return launch_t<float, float>(x, g, rows, n, eps, y, s, zero_word);
  if (y_f16) {  // the fp16 A operand of a GEMM with prepared (fp16) weights: normalized first, so in range
    if (x_f32) return launch_t<float, __nv_bfloat16, __half>(x, g, rows, n, eps, y, s, zero_word);
    return launch_t<__nv_bfloat16, __nv_bfloat16, __half>(x, g, rows, n, eps, y, s, zero_word);
  }
  if (x_f32) return launch_t<float, __nv_bfloat16>(x, g, rows, n, eps, y, s, zero_word);
  return launch_t<__nv_bfloat16, __nv_bfloat16>(x, g, rows, n, eps, y, s, zero_word);
}

}  // namespace blk
