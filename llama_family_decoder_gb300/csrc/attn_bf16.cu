// bf16 decode attention over a KV cache ("LlamaForCausalLM-32L-4096d" sheet:
// softmax(q @ k.T / sqrt(128)) @ v, per head; "arcee", "Grouped-query
// attention, 128-wide heads": query head h reads KV head h / (H / Hkv)).
// HBM-bound: K/V tiles of 64 keys stream through a double-buffered,
// XOR-swizzled shared-memory ring (cp.async, zero-filled past the valid keys);
// the small products run on bf16 mma.sync with fp32 accumulation and an
// online softmax (running max and sum in the log2 domain).
//
// One query per sequence; a CTA takes one (sequence, KV head, key
// split), puts the G = H/Hkv query heads of the group on the MMA's rows, and
// its four warps each own 16 keys of every 64-key tile (their partial softmax
// states merge at the end). Splits are merged by a second small kernel.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

constexpr int kD = 128;
constexpr int kRowBytes = kD * 2;
constexpr int kTileKeys = 64;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Loads rows [0, rows) of a [*, 128] bf16 matrix into a swizzled smem tile;
// rows >= valid are zero-filled (the source address is clamped in bounds).
template <int ROWS, int THREADS>
__device__ __forceinline__ void load_tile(uint32_t s_base, const __nv_bfloat16* g, int valid) {
  constexpr int kChunks = ROWS * 16;
#pragma unroll
  for (int i = 0; i < (kChunks + THREADS - 1) / THREADS; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (kChunks % THREADS == 0 || idx < kChunks) {
      const int r = idx >> 4, ch = idx & 15;
      const bool ok = r < valid;
      const __nv_bfloat16* src = g + (size_t)(ok ? r : 0) * kD + ch * 8;
      cp_async16(s_base + swz(r, ch), src, ok);
    }
  }
}

// ------------------------------------------------------------------ decode

constexpr int kDWarps = 4;
constexpr int kDThreads = kDWarps * 32;
constexpr int kDSmem = 16 * kRowBytes + 4 * kTileKeys * kRowBytes;  // Q (16 rows) + 2x(K,V)

__global__ void __launch_bounds__(kDThreads) attn_decode_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    float* __restrict__ ws_ml, float* __restrict__ ws_o, int H, int Hkv, int kv_stride, const int* __restrict__ kv_lens,
    int len_add, int chunk, int splits) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + 16 * kRowBytes;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = H / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int kv_len = min(kv_lens[b] + len_add, kv_stride);  // never read past the cache
  const int k_begin = split * chunk;
  const int k_end = min(kv_len, k_begin + chunk);
  const int n_keys = max(0, k_end - k_begin);
  const int n_tiles = (n_keys + kTileKeys - 1) / kTileKeys;

  const __nv_bfloat16* qg = q + ((size_t)b * H + (size_t)kvh * G) * kD;
  const __nv_bfloat16* kg = k + (((size_t)b * Hkv + kvh) * kv_stride + k_begin) * kD;
  const __nv_bfloat16* vg = v + (((size_t)b * Hkv + kvh) * kv_stride + k_begin) * kD;
  auto kbuf = [&](int i) { return sK0 + (uint32_t)((i & 1) * 2 * kTileKeys * kRowBytes); };
  auto vbuf = [&](int i) { return kbuf(i) + (uint32_t)(kTileKeys * kRowBytes); };

  load_tile<16, kDThreads>(sQ, qg, G);
  if (n_tiles > 0) {
    load_tile<kTileKeys, kDThreads>(kbuf(0), kg, n_keys);
    load_tile<kTileKeys, kDThreads>(vbuf(0), vg, n_keys);
  }
  cp_async_commit();

  uint32_t qf[8][4];
  float acc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const float sl2 = kLog2e * rsqrtf((float)kD);

  for (int it = 0; it < n_tiles; ++it) {
    if (it + 1 < n_tiles) {
      const int n1 = (it + 1) * kTileKeys;
      load_tile<kTileKeys, kDThreads>(kbuf(it + 1), kg + (size_t)n1 * kD, n_keys - n1);
      load_tile<kTileKeys, kDThreads>(vbuf(it + 1), vg + (size_t)n1 * kD, n_keys - n1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (it == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int mi = lane >> 3, rr = lane & 7;
        ldsm_x4(sQ + swz(rr + 8 * (mi & 1), kk * 2 + (mi >> 1)), qf[kk]);
      }
    }
    const int n0 = it * kTileKeys + warp * 16;  // this warp's 16 keys (relative to k_begin)
    const uint32_t sK = kbuf(it), sV = vbuf(it);
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int mi = lane >> 3, rr = lane & 7;
      uint32_t bb[4];
      ldsm_x4(sK + swz(warp * 16 + rr + 8 * (mi >> 1), kk * 2 + (mi & 1)), bb);
      mma_bf16(s[0], qf[kk], bb[0], bb[1]);
      mma_bf16(s[1], qf[kk], bb[2], bb[3]);
    }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[j][e] * sl2;
        const int key = n0 + j * 8 + 2 * tq + (e & 1);
        if (key >= n_keys) x = -INFINITY;
        s[j][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    float alpha[2], mu[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mnew = fmaxf(mrow[r], mx[r]);
      mu[r] = mnew == -INFINITY ? 0.f : mnew;
      alpha[r] = exp2f(mrow[r] - mu[r]);
      mrow[r] = mnew;
      lrow[r] *= alpha[r];
    }
    uint32_t a[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float p0 = exp2f(s[j][0] - mu[0]), p1 = exp2f(s[j][1] - mu[0]);
      const float p2 = exp2f(s[j][2] - mu[1]), p3 = exp2f(s[j][3] - mu[1]);
      lrow[0] += p0 + p1;
      lrow[1] += p2 + p3;
      a[j * 2 + 0] = pack_bf16x2(p0, p1);
      a[j * 2 + 1] = pack_bf16x2(p2, p3);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      acc[i][0] *= alpha[0];
      acc[i][1] *= alpha[0];
      acc[i][2] *= alpha[1];
      acc[i][3] *= alpha[1];
    }
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      const int mi = lane >> 3, rr = lane & 7;
      uint32_t bb[4];
      ldsm_x4_t(sV + swz(warp * 16 + rr + 8 * (mi & 1), dp * 2 + (mi >> 1)), bb);
      mma_bf16(acc[2 * dp], a, bb[0], bb[1]);
      mma_bf16(acc[2 * dp + 1], a, bb[2], bb[3]);
    }
    __syncthreads();
  }
  cp_async_wait<0>();  // the Q copy is still in flight when the split is empty
  // merge the four warps' states (rows < G) through shared memory
  float* sm = reinterpret_cast<float*>(smem + 16 * kRowBytes);  // reuse the K/V ring
  float* sm_m = sm;                    // [4][16]
  float* sm_l = sm + 64;               // [4][16]
  float* sm_o = sm + 128;              // [4][16][128]
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
  }
  __syncthreads();
  if (tq == 0) {
    sm_m[warp * 16 + g] = mrow[0];
    sm_m[warp * 16 + g + 8] = mrow[1];
    sm_l[warp * 16 + g] = lrow[0];
    sm_l[warp * 16 + g + 8] = lrow[1];
  }
#pragma unroll
  for (int dt = 0; dt < 16; ++dt) {
    const int c = dt * 8 + 2 * tq;
    sm_o[(warp * 16 + g) * kD + c] = acc[dt][0];
    sm_o[(warp * 16 + g) * kD + c + 1] = acc[dt][1];
    sm_o[(warp * 16 + g + 8) * kD + c] = acc[dt][2];
    sm_o[(warp * 16 + g + 8) * kD + c + 1] = acc[dt][3];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * kD; idx += kDThreads) {
    const int r = idx / kD, c = idx - r * kD;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) m = fmaxf(m, sm_m[w * 16 + r]);
    const float mu = m == -INFINITY ? 0.f : m;
    float l = 0.f, oo = 0.f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) {
      const float f = exp2f(sm_m[w * 16 + r] - mu);
      l += sm_l[w * 16 + r] * f;
      oo += sm_o[(w * 16 + r) * kD + c] * f;
    }
    const size_t hs = ((size_t)b * H + (size_t)kvh * G + r) * splits + split;
    ws_o[hs * kD + c] = oo;
    if (c == 0) {
      ws_ml[hs * 2 + 0] = m;
      ws_ml[hs * 2 + 1] = l;
    }
  }
}

__global__ void attn_decode_combine_kernel(const float* __restrict__ ws_ml, const float* __restrict__ ws_o,
                                           __nv_bfloat16* __restrict__ o, int H, int splits) {
  const int h = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const size_t base = ((size_t)b * H + h) * splits;
  float m = -INFINITY;
  for (int s = 0; s < splits; ++s) m = fmaxf(m, ws_ml[(base + s) * 2]);
  const float mu = m == -INFINITY ? 0.f : m;
  float l = 0.f, acc = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float f = exp2f(ws_ml[(base + s) * 2] - mu);
    l += ws_ml[(base + s) * 2 + 1] * f;
    acc += ws_o[(base + s) * kD + c] * f;
  }
  o[((size_t)b * H + h) * kD + c] = __float2bfloat16_rn(acc / l);
}

}  // namespace

int attn_decode_splits(int B, int Hkv, int max_len, int num_sms) {
  const int units = B * Hkv;
  int splits = (3 * num_sms + units - 1) / units;  // about three resident CTAs per SM
  const int max_by_len = (max_len + kTileKeys - 1) / kTileKeys;
  if (splits > max_by_len) splits = max_by_len;
  if (splits < 1) splits = 1;
  if (splits > 64) splits = 64;
  return splits;
}

size_t attn_decode_ws_bytes(int B, int H, int d, int max_splits) {
  return (size_t)B * H * max_splits * (2 + d) * sizeof(float);
}

cudaError_t launch_attn_decode_bf16(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv,
                                    int d, int kv_stride, const int* kv_lens, int len_add, int max_len, void* ws,
                                    int num_sms, cudaStream_t s, const char** why) {
  if (d != kD) {
    *why = "bf16 attention: head_dim must be 128";
    return cudaErrorInvalidValue;
  }
  if (H / Hkv > 16) {
    *why = "bf16 decode attention: at most 16 query heads per KV head";
    return cudaErrorInvalidValue;
  }
  if (B <= 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  // max_len: upper bound of the keys per sequence this step (lens + len_add)
  const int splits = attn_decode_splits(B, Hkv, max_len, num_sms);
  int chunk = (max_len + splits - 1) / splits;
  chunk = (chunk + kTileKeys - 1) / kTileKeys * kTileKeys;
  float* ws_ml = static_cast<float*>(ws);
  float* ws_o = ws_ml + (size_t)B * H * splits * 2;
  dim3 grid(splits, Hkv, B);
  attn_decode_kernel<<<grid, kDThreads, kDSmem, s>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), ws_ml, ws_o, H, Hkv, kv_stride, kv_lens, len_add, chunk, splits);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_decode_combine_kernel<<<dim3(H, B), kD, 0, s>>>(ws_ml, ws_o, static_cast<__nv_bfloat16*>(o), H, splits);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ allocation-free decode variant

// Fixed device scratch for the allocation-free decode attention entry point:
// the per-split softmax partials (max, sum, unnormalised output) that the
// workspace-taking path keeps in caller memory. Every device that loads the
// library holds it until exit; every call shares it.
static __device__ __align__(256) float g_decode_scratch[kDecodeStaticScratchBytes / sizeof(float)];

namespace {
std::mutex g_scratch_mu;
constexpr int kMaxDevices = 64;
float* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, looked up once
// per device (host code cannot use the symbol itself as a device pointer).
cudaError_t scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    float* p = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_attn_decode_bf16_static(const void* q, const void* k, const void* v, void* o, int B, int H,
                                           int Hkv, int d, int kv_stride, const int* kv_lens, int num_sms,
                                           cudaStream_t s, const char** why) {
  if (d != kD) {
    *why = "bf16 attention: head_dim must be 128";
    return cudaErrorInvalidValue;
  }
  if (H / Hkv > 16) {
    *why = "bf16 decode attention: at most 16 query heads per KV head";
    return cudaErrorInvalidValue;
  }
  if (B <= 0) return cudaSuccess;
  const size_t per_split = (size_t)B * H * (2 + d) * sizeof(float);
  if (per_split > kDecodeStaticScratchBytes) {
    *why = "allocation-free decode attention: batch * n_heads * (head_dim + 2) * 4 bytes exceeds the 16 MiB scratch";
    return cudaErrorInvalidValue;
  }
  float* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    *why = "cudaGetSymbolAddress of the decode scratch failed";
    return e;
  }
  static bool configured = false;
  if (!configured) {
    e = cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  int splits = attn_decode_splits(B, Hkv, kv_stride, num_sms);
  const int fit = (int)(kDecodeStaticScratchBytes / per_split);
  if (splits > fit) splits = fit;
  int chunk = (kv_stride + splits - 1) / splits;
  chunk = (chunk + kTileKeys - 1) / kTileKeys * kTileKeys;
  // every partial the combine step reads is written by this call first: nothing to clear
  float* ws_ml = scratch;
  float* ws_o = ws_ml + (size_t)B * H * splits * 2;
  dim3 grid(splits, Hkv, B);
  attn_decode_kernel<<<grid, kDThreads, kDSmem, s>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), ws_ml, ws_o, H, Hkv, kv_stride, kv_lens, 0, chunk, splits);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_decode_combine_kernel<<<dim3(H, B), kD, 0, s>>>(ws_ml, ws_o, static_cast<__nv_bfloat16*>(o), H, splits);
  return cudaGetLastError();
}

}  // namespace blk
