// fp32 SIMT GEMM for the fp32 path: C[m, n] = sum_k A[m, k] * B[n, k]
// (A [M, K], B [N, K] row-major, i.e. h @ W^T with PyTorch Linear weights).
// fp32 FMA only: tensor-core TF32 rounds inputs to 10 mantissa bits, which the
// fp32 parity bound (1e-4 of RMS) does not leave room for.
#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

constexpr int kTile = 64;
constexpr int kBK = 16;

__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, const float* __restrict__ B,
                                                       float* __restrict__ C, int ldc, int M, int N, int K) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float As[kBK][kTile + 4];
  __shared__ float Bs[kBK][kTile + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * kTile, n0 = blockIdx.x * kTile;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kBK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = threadIdx.x + i * 256;
      const int r = idx >> 4, c = idx & 15;
      As[c][r] = (m0 + r < M && k0 + c < K) ? A[(size_t)(m0 + r) * K + k0 + c] : 0.f;
      Bs[c][r] = (n0 + r < N && k0 + c < K) ? B[(size_t)(n0 + r) * K + k0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) C[(size_t)m * ldc + n] = acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_gemm_f32(const float* A, const float* B, float* C, int ldc, int M, int N, int K, cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + kTile - 1) / kTile, (M + kTile - 1) / kTile);
  launch_pdl(gemm_f32_kernel, grid, 256, 0, s, A, B, C, ldc, M, N, K);
  return cudaGetLastError();
}

}  // namespace blk
