// Post-GEMM kernels over fp32 (split-K) partial sums. They finish the
// projections of the fp32 path and of the weight-streaming decode path:
//  * post_qkv: q/k/v heads, optional per-head q/k RMSNorm ("apertus", "Queries
//    and keys are normed per head, before the rotary"), RoPE (rotate-half
//    pairing, angle = position * theta^(-2i/d)), scatter to head-major q and
//    to the K/V buffers or cache slots;
//  * post_resid: residual add after o_proj / down_proj ("arcee", "The block, in
//    order"), summed in fp32 (the residual stream stays fp32 inside the block),
//    with the next RMSNorm fused;
//  * post_act: SiLU-gated, squared-ReLU and xIELU activations.
#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

__device__ __forceinline__ float split_sum(const float* C, int splits, size_t split_stride, size_t idx) {
  float v = 0.f;
  for (int s = 0; s < splits; ++s) v += C[s * split_stride + idx];
  return v;
}

constexpr int kMaxPairsPerLane = 4;  // head_dim <= 256

template <typename T>
__global__ void post_qkv_kernel(const float* __restrict__ C, int splits, int rows, int ldc, int seq,
                                const int* __restrict__ pos0, const int* __restrict__ decode_lens, int H, int Hkv,
                                int d, int qk_norm, const T* __restrict__ q_gain, const T* __restrict__ k_gain,
                                float eps, const float2* __restrict__ rope, int rope_max_pos, T* __restrict__ q,
                                T* __restrict__ k,
                                T* __restrict__ v, int kv_stride) {
  const int r = blockIdx.x;
  if (r >= rows) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int b = r / seq, t = r - b * seq;
  const int pos = decode_lens ? decode_lens[b] : (pos0 ? pos0[b] : 0) + t;
  const int slot = decode_lens ? pos : t;
  const int rpos = min(max(pos, 0), rope_max_pos - 1);  // the host checks positions; never read past the table
  const size_t sstride = (size_t)rows * ldc;
  const int half = d / 2;
  for (int hid = warp; hid < H + 2 * Hkv; hid += nwarps) {
    const int seg = hid < H ? 0 : (hid < H + Hkv ? 1 : 2);
    const int head = seg == 0 ? hid : (seg == 1 ? hid - H : hid - H - Hkv);
    const size_t base = (size_t)r * ldc + (size_t)hid * d;
    float x1[kMaxPairsPerLane], x2[kMaxPairsPerLane];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxPairsPerLane; ++j) {
      const int i = lane + 32 * j;
      x1[j] = x2[j] = 0.f;
      if (i < half) {
        x1[j] = split_sum(C, splits, sstride, base + i);
        x2[j] = split_sum(C, splits, sstride, base + half + i);
        ss += x1[j] * x1[j] + x2[j] * x2[j];
      }
    }
    if (seg != 0 && (slot < 0 || slot >= kv_stride)) continue;  // a full cache: never write past it
    T* dst;
    if (seg == 0)
      dst = q + (((size_t)b * H + head) * seq + t) * d;
    else
      dst = (seg == 1 ? k : v) + (((size_t)b * Hkv + head) * kv_stride + slot) * d;
    if (seg == 2) {
#pragma unroll
      for (int j = 0; j < kMaxPairsPerLane; ++j) {
        const int i = lane + 32 * j;
        if (i < half) {
          dst[i] = from_f32<T>(x1[j]);
          dst[half + i] = from_f32<T>(x2[j]);
        }
      }
      continue;
    }
    float rr = 1.f;
    const T* gain = seg == 0 ? q_gain : k_gain;
    if (qk_norm) rr = rsqrtf(warp_sum(ss) / (float)d + eps);
#pragma unroll
    for (int j = 0; j < kMaxPairsPerLane; ++j) {
      const int i = lane + 32 * j;
      if (i < half) {
        float a = x1[j], c = x2[j];
        if (qk_norm) {
          a = a * rr * to_f32<T>(gain[i]);
          c = c * rr * to_f32<T>(gain[half + i]);
        }
        const float2 sc = rope[(size_t)rpos * half + i];
        dst[i] = from_f32<T>(a * sc.x - c * sc.y);
        dst[half + i] = from_f32<T>(c * sc.x + a * sc.y);
      }
    }
  }
}

// TR: residual type, TO: output type, TY: storage type (gain, y, out2, tap).
template <typename TR, typename TO, typename TY>
__global__ void post_resid_kernel(const float* __restrict__ C, int splits, int rows, int n, int ldc,
                                  const TR* __restrict__ resid, TO* __restrict__ out, TY* __restrict__ out2,
                                  TY* __restrict__ tap, const TY* __restrict__ g, float eps, TY* __restrict__ y,
                                  int* __restrict__ bump_lens) {
  __shared__ float red[32];
  const int r = blockIdx.x;
  if (r >= rows) return;
  const size_t sstride = (size_t)rows * ldc;
  float ss = 0.f;
  for (int c = threadIdx.x; c < n; c += blockDim.x) {
    const float contrib = split_sum(C, splits, sstride, (size_t)r * ldc + c);
    const float o = to_f32<TR>(resid[(size_t)r * n + c]) + contrib;  // the residual stream, summed in fp32
    const TO os = from_f32<TO>(o);
    out[(size_t)r * n + c] = os;
    if (out2) out2[(size_t)r * n + c] = from_f32<TY>(o);
    if (tap) tap[(size_t)r * n + c] = from_f32<TY>(contrib);
    const float of = to_f32<TO>(os);
    ss += of * of;
  }
  if (g == nullptr) {
    if (bump_lens && threadIdx.x == 0) bump_lens[r] += 1;
    return;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
  const float inv = rsqrtf(tot / (float)n + eps);
  for (int c = threadIdx.x; c < n; c += blockDim.x)
    y[(size_t)r * n + c] = from_f32<TY>(to_f32<TO>(out[(size_t)r * n + c]) * inv * to_f32<TY>(g[c]));
  if (bump_lens && threadIdx.x == 0) bump_lens[r] += 1;
}

template <typename T>
__global__ void post_act_kernel(const float* __restrict__ C, int splits, int rows, int F, int ldc, int act,
                                float alpha_p, float alpha_n, float beta, float xeps, T* __restrict__ out) {
  const size_t total = (size_t)rows * F;
  const size_t sstride = (size_t)rows * ldc;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx / F), f = (int)(idx - (size_t)r * F);
    const size_t base = (size_t)r * ldc;
    float n;
    if (act == 0) {  // SwiGLU: silu(gate) * up
      const float gt = split_sum(C, splits, sstride, base + f);
      const float up = split_sum(C, splits, sstride, base + F + f);
      n = gt / (1.0f + expf(-gt)) * up;
    } else {
      const float u = split_sum(C, splits, sstride, base + f);
      if (act == 1) {
        const float rl = fmaxf(u, 0.f);
        n = rl * rl;
      } else {
        n = u > 0.f ? alpha_p * u * u + beta * u : alpha_n * (expm1f(fminf(u, xeps)) - u) + beta * u;
      }
    }
    out[idx] = from_f32<T>(n);
  }
}

}  // namespace

cudaError_t launch_post_qkv(const float* C, int splits, int rows, int ldc, int seq, const int* pos0,
                            const int* decode_lens, int H, int Hkv, int d, int qk_norm, const void* q_gain,
                            const void* k_gain, float eps, const float2* rope, int rope_max_pos, void* q, void* k,
                            void* v, int kv_stride, bool bf16, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (d > 2 * 32 * kMaxPairsPerLane || d % 2) return cudaErrorInvalidValue;
  if (bf16) {
    using T = __nv_bfloat16;
    post_qkv_kernel<T><<<rows, 256, 0, s>>>(C, splits, rows, ldc, seq, pos0, decode_lens, H, Hkv, d, qk_norm,
                                           static_cast<const T*>(q_gain), static_cast<const T*>(k_gain), eps, rope, rope_max_pos,
                                           static_cast<T*>(q), static_cast<T*>(k), static_cast<T*>(v), kv_stride);
  } else {
    using T = float;
    post_qkv_kernel<T><<<rows, 256, 0, s>>>(C, splits, rows, ldc, seq, pos0, decode_lens, H, Hkv, d, qk_norm,
                                           static_cast<const T*>(q_gain), static_cast<const T*>(k_gain), eps, rope, rope_max_pos,
                                           static_cast<T*>(q), static_cast<T*>(k), static_cast<T*>(v), kv_stride);
  }
  return cudaGetLastError();
}

cudaError_t launch_post_resid(const float* C, int splits, int rows, int n, int ldc, const void* resid, bool resid_f32,
                              void* out, bool out_f32, void* out2, void* tap, const void* g, float eps, void* y,
                              int* bump_lens, bool bf16, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  using B = __nv_bfloat16;
#define BLK_POST_RESID(TR, TO, TY)                                                                              \
  post_resid_kernel<TR, TO, TY><<<rows, 256, 0, s>>>(C, splits, rows, n, ldc, static_cast<const TR*>(resid),   \
                                                     static_cast<TO*>(out), static_cast<TY*>(out2),             \
                                                     static_cast<TY*>(tap), static_cast<const TY*>(g), eps,     \
                                                     static_cast<TY*>(y), bump_lens)
  if (!bf16) {
    BLK_POST_RESID(float, float, float);
  } else if (resid_f32 && out_f32) {
    BLK_POST_RESID(float, float, B);
  } else if (resid_f32) {
    BLK_POST_RESID(float, B, B);
  } else if (out_f32) {
    BLK_POST_RESID(B, float, B);
  } else {
    BLK_POST_RESID(B, B, B);
  }
#undef BLK_POST_RESID
  return cudaGetLastError();
}

cudaError_t launch_post_act(const float* C, int splits, int rows, int F, int ldc, int act, float alpha_p,
                            float alpha_n, float beta, float xeps, void* out, bool bf16, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const size_t total = (size_t)rows * F;
  int grid = (int)((total + 255) / 256);
  if (grid > 4096) grid = 4096;
  if (bf16)
    post_act_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(C, splits, rows, F, ldc, act, alpha_p, alpha_n, beta, xeps,
                                                        static_cast<__nv_bfloat16*>(out));
  else
    post_act_kernel<float><<<grid, 256, 0, s>>>(C, splits, rows, F, ldc, act, alpha_p, alpha_n, beta, xeps,
                                                static_cast<float*>(out));
  return cudaGetLastError();
}

}  // namespace blk
