// fp32 causal grouped-query attention for the fp32 path (small shapes):
// o[b, i, h, :] = sum_j softmax_j(q[b,h,i] . k[b,kv,j] / sqrt(d)) v[b,kv,j, :],
// kv = h / (H / Hkv), keys j visible iff position(j) <= position(i)
// ("LlamaForCausalLM-32L-4096d": softmax(q @ k.T / sqrt(128), mask=causal) @ v;
// "arcee", "Grouped-query attention, 128-wide heads").
// Options of the "afmoe" block: a window over the last W positions and a
// per-channel sigmoid gate on the output (the gate values come in already
// passed through the sigmoid).
// One warp per (b, h, query); scores held in shared memory.
#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

__global__ void attn_f32_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                                float* __restrict__ o, int H, int Hkv, int Tq, int d, int kv_stride,
                                const int* __restrict__ kv_lens, int len_add, int window,
                                const float* __restrict__ gate, float* __restrict__ ungated,
                                const int2* __restrict__ key_range) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sc[];
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x;
  const int kv_len = kv_lens ? min(kv_lens[b] + len_add, kv_stride) : Tq;  // never read past the cache
  const int2 kr = key_range ? key_range[b] : make_int2(0, kv_len);  // visible (non-padding) keys
  const int qend = min(kv_len - Tq + i, kr.y - 1);  // keys j0 .. qend are visible: causal, not padding,
  const int j0 = max(kr.x, window > 0 ? kv_len - Tq + i - window + 1 : 0);  // ... and within the window
  const int kvh = h / (H / Hkv);
  const float* qr = q + (((size_t)b * H + h) * Tq + i) * d;
  const float* kb = k + ((size_t)b * Hkv + kvh) * kv_stride * d;
  const float* vb = v + ((size_t)b * Hkv + kvh) * kv_stride * d;
  const float scale = 1.0f / sqrtf((float)d);
  float m = -INFINITY;
  for (int j = j0 + lane; j <= qend; j += 32) {
    float s = 0.f;
    for (int c = 0; c < d; ++c) s = fmaf(qr[c], kb[(size_t)j * d + c], s);
    s *= scale;
    sc[j] = s;
    m = fmaxf(m, s);
  }
  m = warp_max(m);
  float l = 0.f;
  for (int j = j0 + lane; j <= qend; j += 32) {
    const float p = expf(sc[j] - m);
    sc[j] = p;
    l += p;
  }
  l = warp_sum(l);
  __syncwarp();
  const size_t orow = (((size_t)b * Tq + i) * H + h) * d;
  for (int c = lane; c < d; c += 32) {
    float acc = 0.f;
    for (int j = j0; j <= qend; ++j) acc = fmaf(sc[j], vb[(size_t)j * d + c], acc);
    const float r = l > 0.f ? acc / l : 0.f;  // a padding query that sees no key: 0
    if (ungated) ungated[orow + c] = r;
    o[orow + c] = gate ? r * gate[orow + c] : r;
  }
}

}  // namespace

cudaError_t launch_attn_f32(const float* q, const float* k, const float* v, float* o, int B, int H, int Hkv, int Tq,
                            int d, int kv_stride, const int* kv_lens, int len_add, cudaStream_t s,
                            const AttnOpts& opt) {
  if (B <= 0 || Tq <= 0) return cudaSuccess;
  const size_t smem = (size_t)kv_stride * sizeof(float);
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(Tq, H, B);
  launch_pdl(attn_f32_kernel, grid, 32, smem, s, q, k, v, o, H, Hkv, Tq, d, kv_stride, kv_lens, len_add,
             opt.window > 0 ? opt.window : 0, static_cast<const float*>(opt.gate), static_cast<float*>(opt.ungated),
             opt.key_range);
  return cudaGetLastError();
}

}  // namespace blk
