// Post-GEMM kernels over fp32 (split-K) partial sums. They finish the
// projections of the fp32 path and of the weight-streaming decode path:
//  * post_qkv: q/k/v heads, optional per-head q/k RMSNorm ("apertus", "Queries
//    and keys are normed per head, before the rotary"), RoPE (rotate-half
//    pairing, angle = position * theta^(-2i/d)), scatter to head-major q and
//    to the K/V buffers or cache slots;
//  * post_resid: residual add after o_proj / down_proj ("arcee", "The block, in
//    order"), summed in fp32 (the residual stream stays fp32 inside the block),
//    with the next RMSNorm fused and, for the sandwich block ("afmoe", "The
//    block, in order"), the post-norm of the sublayer's output before the add;
//  * post_act: SiLU-gated, squared-ReLU and xIELU activations.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

__device__ __forceinline__ float split_sum(const float* C, int splits, size_t split_stride, size_t idx) {
  float v = 0.f;
#pragma unroll 4
  for (int s = 0; s < splits; ++s) v += C[s * split_stride + idx];
  return v;
}

constexpr int kMaxPairsPerLane = 4;  // head_dim <= 256
constexpr int kQkvWarps = 4;

// The attention gate's storage: fp16 beside bf16 tensors, fp32 on the fp32 path.
template <typename T>
__device__ __forceinline__ void store_gate(void* g, size_t i, float v) {
  if constexpr (sizeof(T) == 4)
    static_cast<float*>(g)[i] = v;
  else
    static_cast<__half*>(g)[i] = __float2half_rn(v);
}

template <typename T>
__global__ void post_qkv_kernel(const float* __restrict__ C, int splits, int rows, int ldc, int seq,
                                const int* __restrict__ pos0, const int* __restrict__ decode_lens, int H, int Hkv,
                                int d, int qk_norm, const T* __restrict__ q_gain, const T* __restrict__ k_gain,
                                float eps, const float2* __restrict__ rope, int rope_max_pos, T* __restrict__ q,
                                T* __restrict__ k,
                                T* __restrict__ v, int kv_stride, void* __restrict__ gate) {
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.x;
  if (r >= rows) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = r / seq, t = r - b * seq;
  const int pos = decode_lens ? decode_lens[b] : (pos0 ? pos0[b] : 0) + t;
  const int slot = decode_lens ? pos : t;
  const int rpos = min(max(pos, 0), rope_max_pos - 1);  // the host checks positions; never read past the table
  const size_t sstride = (size_t)rows * ldc;
  const int half = d / 2;
  {
    const int hid = blockIdx.y * kQkvWarps + warp;  // one warp per (row, head)
    if (hid >= H + 2 * Hkv + (gate ? H : 0)) return;
    const size_t base = (size_t)r * ldc + (size_t)hid * d;
    if (hid >= H + 2 * Hkv) {
      // the attention gate of query head hid - H - 2 Hkv ("afmoe"): sigmoid, in o's layout
      const size_t g0 = ((size_t)r * H + (hid - H - 2 * Hkv)) * d;
      for (int i = lane; i < d; i += 32) store_gate<T>(gate, g0 + i, sigmoid_f(split_sum(C, splits, sstride, base + i)));
      return;
    }
    const int seg = hid < H ? 0 : (hid < H + Hkv ? 1 : 2);
    const int head = seg == 0 ? hid : (seg == 1 ? hid - H : hid - H - Hkv);
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
    if (seg != 0 && (slot < 0 || slot >= kv_stride)) return;  // a full cache: never write past it
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
      return;
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

template <typename T>
__device__ __forceinline__ float4 ld4(const T* p);
template <>
__device__ __forceinline__ float4 ld4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y);
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename T>
__device__ __forceinline__ void st4(T* p, float4 v);
template <>
__device__ __forceinline__ void st4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void st4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

template <typename T>
__device__ __forceinline__ float4 round4(float4 v) {
  return make_float4(round_to<T>(v.x), round_to<T>(v.y), round_to<T>(v.z), round_to<T>(v.w));
}

__device__ __forceinline__ float4 split_sum4(const float* C, int splits, size_t split_stride, size_t idx) {
  float4 acc = *reinterpret_cast<const float4*>(C + idx);
#pragma unroll 4
  for (int s = 1; s < splits; ++s) {
    const float4 t = *reinterpret_cast<const float4*>(C + s * split_stride + idx);
    acc.x += t.x;
    acc.y += t.y;
    acc.z += t.z;
    acc.w += t.w;
  }
  return acc;
}

constexpr int kResidThreads = 256;

// One CTA per row; each thread owns VPT groups of 4 columns, issues all their
// loads up front and keeps the sums in registers for the fused RMSNorm.
// TR: residual type, TO: output type, TY: storage type (gain, y, out2, tap).
// Sum of v over the CTA (every thread gets it); red holds one float per warp.
__device__ __forceinline__ float cta_sum(float v, float* red) {
  v = warp_sum(v);
  __syncthreads();  // red may still be read from an earlier call
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kResidThreads / 32; ++w) tot += red[w];
  return tot;
}

template <typename TR, typename TO, typename TY, int VPT>
__global__ void __launch_bounds__(kResidThreads) post_resid_kernel(
    const float* __restrict__ C, int splits, int rows, int n, int ldc, const TR* __restrict__ resid,
    TO* __restrict__ out, TY* __restrict__ out2, TY* __restrict__ tap, const TY* __restrict__ g, float eps,
    TY* __restrict__ y, int* __restrict__ bump_lens, const TY* __restrict__ g_post, int y_f16) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float red[kResidThreads / 32];
  const int r = blockIdx.x;
  if (r >= rows) return;
  const size_t sstride = (size_t)rows * ldc;
  const int nv = n / 4;
  float4 o[VPT], a[VPT], rr[VPT];
  float ss = 0.f, ssa = 0.f;
  // the residual is loaded with the sublayer's output: it does not wait for the post-norm
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = threadIdx.x + j * kResidThreads;
    a[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    rr[j] = a[j];
    if (v < nv) {
      rr[j] = ld4<TR>(resid + (size_t)r * n + 4 * v);
      a[j] = split_sum4(C, splits, sstride, (size_t)r * ldc + 4 * v);
      ssa += a[j].x * a[j].x + a[j].y * a[j].y + a[j].z * a[j].z + a[j].w * a[j].w;
    }
  }
  if (g_post != nullptr) {
    // the sandwich post-norm of the sublayer's output ("afmoe", "The block, in order")
    const float inv = rsqrtf(cta_sum(ssa, red) / (float)n + eps);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = threadIdx.x + j * kResidThreads;
      if (v < nv) {
        const float4 gg = ld4<TY>(g_post + 4 * v);
        a[j] = make_float4(a[j].x * inv * gg.x, a[j].y * inv * gg.y, a[j].z * inv * gg.z, a[j].w * inv * gg.w);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = threadIdx.x + j * kResidThreads;
    if (v < nv) {
      const float4 contrib = a[j];
      // the residual stream, summed in fp32
      const float4 oo =
          make_float4(rr[j].x + contrib.x, rr[j].y + contrib.y, rr[j].z + contrib.z, rr[j].w + contrib.w);
      st4<TO>(out + (size_t)r * n + 4 * v, oo);
      if (out2) st4<TY>(out2 + (size_t)r * n + 4 * v, oo);
      if (tap) st4<TY>(tap + (size_t)r * n + 4 * v, contrib);
      o[j] = round4<TO>(oo);
      ss += o[j].x * o[j].x + o[j].y * o[j].y + o[j].z * o[j].z + o[j].w * o[j].w;
    }
  }
  if (g != nullptr) {
    const float inv = rsqrtf(cta_sum(ss, red) / (float)n + eps);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = threadIdx.x + j * kResidThreads;
      if (v < nv) {
        const float4 gg = ld4<TY>(g + 4 * v);
        const float4 yy =
            make_float4(o[j].x * inv * gg.x, o[j].y * inv * gg.y, o[j].z * inv * gg.z, o[j].w * inv * gg.w);
        if (y_f16) {  // the fp16 operand of a GEMM with prepared (fp16) weights
          const __half2 h01 = __floats2half2_rn(yy.x, yy.y), h23 = __floats2half2_rn(yy.z, yy.w);
          *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(y) + (size_t)r * n + 4 * v) =
              make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
        } else {
          st4<TY>(y + (size_t)r * n + 4 * v, yy);
        }
      }
    }
  }
  if (bump_lens && threadIdx.x == 0) bump_lens[r] += 1;
}

__device__ __forceinline__ float act_one(int act, float gt, float u, float alpha_p, float alpha_n, float beta,
                                         float xeps) {
  if (act == 0) return gt / (1.0f + expf(-gt)) * u;  // SwiGLU: silu(gate) * up
  if (act == 1) {
    const float rl = fmaxf(u, 0.f);
    return rl * rl;
  }
  return u > 0.f ? alpha_p * u * u + beta * u : alpha_n * (expm1f(fminf(u, xeps)) - u) + beta * u;
}

// 1/rms of row r from its partial sums of squares (summed in order), or 1 without them.
__device__ __forceinline__ float row_rms_factor(const float* row_ss, int ss_parts, int ss_n, float ss_eps, int r) {
  if (!row_ss) return 1.0f;
  float t = 0.f;
  for (int i = 0; i < ss_parts; ++i) t += row_ss[(size_t)r * ss_parts + i];
  return rsqrtf(t / (float)ss_n + ss_eps);
}

// Four consecutive neurons per thread (F % 4 == 0).
template <typename T>
__global__ void post_act4_kernel(const float* __restrict__ C, int splits, int rows, int F, int ldc, int act,
                                 float alpha_p, float alpha_n, float beta, float xeps, T* __restrict__ out,
                                 const float* __restrict__ row_ss, int ss_parts, int ss_n, float ss_eps) {
  pdl_launch_dependents();
  pdl_wait();
  const int F4 = F / 4;
  const int total = rows * F4;
  const size_t sstride = (size_t)rows * ldc;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int r = i / F4, f = (i - r * F4) * 4;
    const size_t base = (size_t)r * ldc;
    const float rs = row_rms_factor(row_ss, ss_parts, ss_n, ss_eps, r);
    float4 u = act == 0 ? split_sum4(C, splits, sstride, base + F + f) : split_sum4(C, splits, sstride, base + f);
    float4 gt = act == 0 ? split_sum4(C, splits, sstride, base + f) : u;
    u = make_float4(u.x * rs, u.y * rs, u.z * rs, u.w * rs);
    gt = make_float4(gt.x * rs, gt.y * rs, gt.z * rs, gt.w * rs);
    const float4 n = make_float4(act_one(act, gt.x, u.x, alpha_p, alpha_n, beta, xeps),
                                 act_one(act, gt.y, u.y, alpha_p, alpha_n, beta, xeps),
                                 act_one(act, gt.z, u.z, alpha_p, alpha_n, beta, xeps),
                                 act_one(act, gt.w, u.w, alpha_p, alpha_n, beta, xeps));
    st4<T>(out + (size_t)r * F + f, n);
  }
}

template <typename T>
__global__ void post_act_kernel(const float* __restrict__ C, int splits, int rows, int F, int ldc, int act,
                                float alpha_p, float alpha_n, float beta, float xeps, T* __restrict__ out,
                                const float* __restrict__ row_ss, int ss_parts, int ss_n, float ss_eps) {
  pdl_launch_dependents();
  pdl_wait();
  const size_t total = (size_t)rows * F;
  const size_t sstride = (size_t)rows * ldc;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx / F), f = (int)(idx - (size_t)r * F);
    const size_t base = (size_t)r * ldc;
    const float rs = row_rms_factor(row_ss, ss_parts, ss_n, ss_eps, r);
    const float u = split_sum(C, splits, sstride, base + (act == 0 ? F + f : f)) * rs;
    const float gt = act == 0 ? split_sum(C, splits, sstride, base + f) * rs : u;
    out[idx] = from_f32<T>(act_one(act, gt, u, alpha_p, alpha_n, beta, xeps));
  }
}

}  // namespace

cudaError_t launch_post_qkv(const float* C, int splits, int rows, int ldc, int seq, const int* pos0,
                            const int* decode_lens, int H, int Hkv, int d, int qk_norm, const void* q_gain,
                            const void* k_gain, float eps, const float2* rope, int rope_max_pos, void* q, void* k,
                            void* v, int kv_stride, bool bf16, cudaStream_t s, void* gate) {
  if (rows <= 0) return cudaSuccess;
  if (d > 2 * 32 * kMaxPairsPerLane || d % 2) return cudaErrorInvalidValue;
  const int heads = H + 2 * Hkv + (gate ? H : 0);
  if (bf16) {
    using T = __nv_bfloat16;
    launch_pdl(post_qkv_kernel<T>, dim3(rows, (heads + kQkvWarps - 1) / kQkvWarps), 32 * kQkvWarps, 0, s, C, splits, rows, ldc, seq, pos0, decode_lens, H, Hkv, d, qk_norm,
                                           static_cast<const T*>(q_gain), static_cast<const T*>(k_gain), eps, rope, rope_max_pos,
                                           static_cast<T*>(q), static_cast<T*>(k), static_cast<T*>(v), kv_stride, gate);
  } else {
    using T = float;
    launch_pdl(post_qkv_kernel<T>, dim3(rows, (heads + kQkvWarps - 1) / kQkvWarps), 32 * kQkvWarps, 0, s, C, splits, rows, ldc, seq, pos0, decode_lens, H, Hkv, d, qk_norm,
                                           static_cast<const T*>(q_gain), static_cast<const T*>(k_gain), eps, rope, rope_max_pos,
                                           static_cast<T*>(q), static_cast<T*>(k), static_cast<T*>(v), kv_stride, gate);
  }
  return cudaGetLastError();
}

cudaError_t launch_post_resid(const float* C, int splits, int rows, int n, int ldc, const void* resid, bool resid_f32,
                              void* out, bool out_f32, void* out2, void* tap, const void* g, float eps, void* y,
                              int* bump_lens, bool bf16, cudaStream_t s, const void* g_post, bool y_f16) {
  if (rows <= 0) return cudaSuccess;
  if (n % 4 || ldc % 4) return cudaErrorInvalidValue;
  const int nv = n / 4;
  const int vpt = (nv + kResidThreads - 1) / kResidThreads;
  using B = __nv_bfloat16;
#define BLK_POST_RESID_V(TR, TO, TY, V)                                                                        \
  launch_pdl(post_resid_kernel<TR, TO, TY, V>, rows, kResidThreads, 0, s,                                            \
      C, splits, rows, n, ldc, static_cast<const TR*>(resid), static_cast<TO*>(out), static_cast<TY*>(out2),  \
      static_cast<TY*>(tap), static_cast<const TY*>(g), eps, static_cast<TY*>(y), bump_lens,              \
      static_cast<const TY*>(g_post), (bf16 && y_f16) ? 1 : 0)
#define BLK_POST_RESID(TR, TO, TY)                  \
  do {                                              \
    if (vpt <= 1)                                   \
      BLK_POST_RESID_V(TR, TO, TY, 1);              \
    else if (vpt <= 2)                              \
      BLK_POST_RESID_V(TR, TO, TY, 2);              \
    else if (vpt <= 4)                              \
      BLK_POST_RESID_V(TR, TO, TY, 4);              \
    else if (vpt <= 8)                              \
      BLK_POST_RESID_V(TR, TO, TY, 8);              \
    else if (vpt <= 16)                             \
      BLK_POST_RESID_V(TR, TO, TY, 16);             \
    else                                            \
      return cudaErrorInvalidValue;                 \
  } while (0)
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
#undef BLK_POST_RESID_V
  return cudaGetLastError();
}

cudaError_t launch_post_act(const float* C, int splits, int rows, int F, int ldc, int act, float alpha_p,
                            float alpha_n, float beta, float xeps, void* out, bool bf16, cudaStream_t s,
                            const float* row_ss, int ss_parts, int ss_n, float ss_eps) {
  if (rows <= 0) return cudaSuccess;
  const bool vec = F % 4 == 0 && ldc % 4 == 0;
  const size_t total = (size_t)rows * F / (vec ? 4 : 1);
  int grid = (int)((total + 255) / 256);
  if (grid > 8192) grid = 8192;
  if (vec) {
    if (bf16)
      launch_pdl(post_act4_kernel<__nv_bfloat16>, grid, 256, 0, s, C, splits, rows, F, ldc, act, alpha_p, alpha_n, beta,
                                                           xeps, static_cast<__nv_bfloat16*>(out), row_ss, ss_parts, ss_n, ss_eps);
    else
      launch_pdl(post_act4_kernel<float>, grid, 256, 0, s, C, splits, rows, F, ldc, act, alpha_p, alpha_n, beta, xeps,
                                                   static_cast<float*>(out), row_ss, ss_parts, ss_n, ss_eps);
  } else {
    if (bf16)
      launch_pdl(post_act_kernel<__nv_bfloat16>, grid, 256, 0, s, C, splits, rows, F, ldc, act, alpha_p, alpha_n, beta, xeps,
                                                          static_cast<__nv_bfloat16*>(out), row_ss, ss_parts, ss_n, ss_eps);
    else
      launch_pdl(post_act_kernel<float>, grid, 256, 0, s, C, splits, rows, F, ldc, act, alpha_p, alpha_n, beta, xeps,
                                                  static_cast<float*>(out), row_ss, ss_parts, ss_n, ss_eps);
  }
  return cudaGetLastError();
}

}  // namespace blk
