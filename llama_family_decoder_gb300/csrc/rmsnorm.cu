// Row-wise RMSNorm (nnterp "input_layernorm" / "post_attention_layernorm";
// "LlamaForCausalLM-32L-4096d" sheet: rmsnorm(x, ..., eps=1e-05)):
//   y[r, :] = x[r, :] * rsqrt(mean(x[r, :]^2) + eps) * g
// Statistics in fp32. HBM-bound: one read and one write of the row, 128-bit
// loads/stores, the row held in registers between the two passes.
#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

constexpr int kThreads = 256;

template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = unpack_bf16x2(w[i]);
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
  }
};

template <typename T, int NV>
__global__ void __launch_bounds__(kThreads) rmsnorm_kernel(const T* __restrict__ x, const T* __restrict__ g, int rows,
                                                           int n, float eps, T* __restrict__ y) {
  constexpr int E = Vec<T>::N;
  __shared__ float red[kThreads / 32];
  const int nvec = n / E;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)r * n);
    uint4 buf[NV];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int v = threadIdx.x + j * kThreads;
      if (v < nvec) {
        buf[j] = xr[v];
        float f[E];
        Vec<T>::unpack(buf[j], f);
#pragma unroll
        for (int i = 0; i < E; ++i) ss += f[i] * f[i];
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
    uint4* yr = reinterpret_cast<uint4*>(y + (size_t)r * n);
    const uint4* gv = reinterpret_cast<const uint4*>(g);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int v = threadIdx.x + j * kThreads;
      if (v < nvec) {
        float f[E], gg[E];
        Vec<T>::unpack(buf[j], f);
        Vec<T>::unpack(gv[v], gg);
#pragma unroll
        for (int i = 0; i < E; ++i) f[i] = f[i] * inv * gg[i];
        yr[v] = Vec<T>::pack(f);
      }
    }
  }
}

template <typename T>
cudaError_t launch_t(const void* x, const void* g, int rows, int n, float eps, void* y, cudaStream_t s) {
  const int nvec = n / Vec<T>::N;
  const int nv = (nvec + kThreads - 1) / kThreads;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = rows < sms * 8 ? rows : sms * 8;
  auto X = static_cast<const T*>(x);
  auto G = static_cast<const T*>(g);
  auto Y = static_cast<T*>(y);
  switch (nv) {
    case 1: rmsnorm_kernel<T, 1><<<grid, kThreads, 0, s>>>(X, G, rows, n, eps, Y); break;
    case 2: rmsnorm_kernel<T, 2><<<grid, kThreads, 0, s>>>(X, G, rows, n, eps, Y); break;
    case 3: rmsnorm_kernel<T, 3><<<grid, kThreads, 0, s>>>(X, G, rows, n, eps, Y); break;
    case 4: rmsnorm_kernel<T, 4><<<grid, kThreads, 0, s>>>(X, G, rows, n, eps, Y); break;
    case 5: rmsnorm_kernel<T, 5><<<grid, kThreads, 0, s>>>(X, G, rows, n, eps, Y); break;
    case 6: rmsnorm_kernel<T, 6><<<grid, kThreads, 0, s>>>(X, G, rows, n, eps, Y); break;
    case 7: rmsnorm_kernel<T, 7><<<grid, kThreads, 0, s>>>(X, G, rows, n, eps, Y); break;
    case 8: rmsnorm_kernel<T, 8><<<grid, kThreads, 0, s>>>(X, G, rows, n, eps, Y); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm(const void* x, const void* g, int rows, int n, float eps, void* y, bool bf16,
                           cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  return bf16 ? launch_t<__nv_bfloat16>(x, g, rows, n, eps, y, s) : launch_t<float>(x, g, rows, n, eps, y, s);
}

}  // namespace blk
