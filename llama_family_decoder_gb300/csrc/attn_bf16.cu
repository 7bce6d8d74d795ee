// bf16 decode attention over a KV cache ("LlamaForCausalLM-32L-4096d" sheet:
// softmax(q @ k.T / sqrt(128)) @ v, per head; "arcee", "Grouped-query
// attention, 128-wide heads": query head h reads KV head h / (H / Hkv)).
// HBM-bound: a persistent kernel whose producer warp streams K/V tiles of 64
// keys through a 6-stage TMA ring (128-byte swizzle); the small products run
// on bf16 mma.sync with fp32 accumulation and an online softmax (running max
// and sum in the log2 domain).
//
// One query per sequence; a work unit is (sequence, KV head, key split of
// about 512 keys): the G = H/Hkv query heads of the group sit on the MMA's
// rows, and the four compute warps each own 16 keys of every tile (their
// partial softmax states merge at the end of the unit). Splits are merged by
// a second small kernel, which also applies the "afmoe" head gate. With a
// sliding window the splits cover only the last `window` keys.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

constexpr int kD = 128;
constexpr int kTileKeys = 64;
constexpr float kLog2e = 1.4426950408889634f;

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

// ------------------------------------------------------------------ decode

constexpr int kStages = 6;                       // TMA ring depth (tiles of 64 keys)
constexpr int kHalfBytes = kTileKeys * 128;      // one 64-column half of a 64-key tile (8 KB)
constexpr int kStageBytes = 4 * kHalfBytes;      // K and V, two halves each (32 KB)
constexpr int kCompute = 4;                      // compute warps; warp 4 is the TMA producer
constexpr int kThreads = (kCompute + 1) * 32;
constexpr int kMergeFloats = 2 * 64 + kCompute * 16 * kD;
constexpr int kUq = 4;  // units handed from the producer to the compute warps, in flight
constexpr int kSmem = 1024 + kStages * kStageBytes + kMergeFloats * 4 + 256;
constexpr unsigned long long kDrainNs = 2000000000ULL;

struct DecodeParams {
  CUtensorMap tk, tv;  // [B * Hkv * kv_stride, 128] bf16, boxes of 64 x 64, 128-byte swizzle
  const __nv_bfloat16* q;
  float* ws_ml;
  float* ws_o;
  const int* kv_lens;
  int* work;  // units taken so far beyond the first round (zero at launch), or null: round robin
  int len_add, B, H, Hkv, kv_stride, chunk, splits, units;
  int window;  // > 0: only the last `window` keys of each sequence
  DevStatus* status;
  unsigned long long wait_ns;
};

// Byte offset of (row, 16-byte chunk C of 16) in a tile written by TMA with the
// 128-byte swizzle: two 64-column halves, rows of 128 bytes, chunks XOR (row & 7).
__device__ __forceinline__ uint32_t tsw(int row, int C) {
  return (uint32_t)((C >> 3) * kHalfBytes + row * 128 + (((C & 7) ^ (row & 7)) << 4));
}

struct DecodeUnit {
  int b, kvh, split, k0, n_keys, n_tiles;
};

__device__ __forceinline__ DecodeUnit decode_unit(const DecodeParams& p, int u) {
  DecodeUnit r;
  // the splits of one (sequence, KV head) are consecutive units: the CTAs working
  // at the same time stream neighbouring stretches of the cache
  r.split = u % p.splits;
  r.kvh = (u / p.splits) % p.Hkv;
  r.b = u / (p.splits * p.Hkv);
  const int kv_len = min(p.kv_lens[r.b] + p.len_add, p.kv_stride);  // never read past the cache
  const int first = p.window > 0 ? max(0, kv_len - p.window) : 0;    // the oldest key in the window
  r.k0 = first + r.split * p.chunk;
  // the last split takes every key left (up to a chunk more): no unit of a handful of keys
  const int end = r.split == p.splits - 1 ? kv_len : min(kv_len, r.k0 + p.chunk);
  r.n_keys = max(0, end - r.k0);
  r.n_tiles = (r.n_keys + kTileKeys - 1) / kTileKeys;
  return r;
}

// Persistent split-KV decode attention: each CTA starts on unit blockIdx.x (a
// sequence, a KV head, a key split) and takes its next ones from a shared
// counter, so that CTAs the memory system serves faster take more; its producer
// lane streams every unit's K/V tiles through a 6-stage TMA ring without pausing
// between units and hands the unit indices to the 4 compute warps (a queue of
// kUq, mbarriers both ways), which each own 16 keys of every tile.
__global__ void __launch_bounds__(kThreads, 1) attn_decode_kernel(const __grid_constant__ DecodeParams p) {
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  float* merge = reinterpret_cast<float*>(ring + kStages * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(merge + kMergeFloats);
  // full[kStages], empty[kStages], csync, (abort flag), uq_full[kUq], uq_empty[kUq], unit ids[kUq]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages + 1);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kStages + s]); };
  const uint32_t csync = smem_u32(&bars[2 * kStages]);
  auto uq_full = [&](int s) { return smem_u32(&bars[2 * kStages + 2 + s]); };
  auto uq_empty = [&](int s) { return smem_u32(&bars[2 * kStages + 2 + kUq + s]); };
  volatile int* unit_q = reinterpret_cast<volatile int*>(bars + 2 * kStages + 2 + 2 * kUq);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.H / p.Hkv;
  const unsigned long long budget = p.wait_ns;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), kCompute);
    }
    mbar_init(csync, kCompute * 32);
    for (int i = 0; i < kUq; ++i) {
      mbar_init(uq_full(i), 1);
      mbar_init(uq_empty(i), kCompute);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // the new key/value rows and q come from the previous kernel
  // the ring stages the producer issued (with the parity of their last phase): an abort
  // drains them after the CTA's final barrier
  uint32_t issued = 0, parity = 0;

  if (warp == kCompute) {
    if (lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(&p.tk);
      tma_prefetch_desc(&p.tv);
      int stage = 0;
      uint32_t ph = 0;
      bool failed = false;
      const uint64_t stream_once = l2_policy_evict_first();  // the cache is read once per step
      int u = blockIdx.x;
      for (int k = 0; !failed; ++k) {
        // hand unit u (p.units or more: none left) to the compute warps
        const int slot = k % kUq;
        if (!mbar_wait(uq_empty(slot), ((k / kUq) & 1) ^ 1, budget, abort_flag)) {
          failed = true;
          break;
        }
        unit_q[slot] = u;
        mbar_arrive(uq_full(slot));
        if (u >= p.units) break;
        // the next unit, asked for now: the answer is needed only after this unit's tiles
        const int next = p.work ? atomicAdd(p.work, 1) + (int)gridDim.x : u + (int)gridDim.x;
        const DecodeUnit un = decode_unit(p, u);
        const int row0 = (un.b * p.Hkv + un.kvh) * p.kv_stride + un.k0;
        for (int t = 0; t < un.n_tiles; ++t) {
          if (!mbar_wait(empty(stage), ph ^ 1, budget, abort_flag)) {
            failed = true;
            break;
          }
          const uint32_t dst = smem_u32(ring + stage * kStageBytes);
          mbar_arrive_expect_tx(full(stage), kStageBytes);
          const int row = row0 + t * kTileKeys;
          tma_load_2d_hint(dst, &p.tk, 0, row, full(stage), stream_once);
          tma_load_2d_hint(dst + kHalfBytes, &p.tk, 64, row, full(stage), stream_once);
          tma_load_2d_hint(dst + 2 * kHalfBytes, &p.tv, 0, row, full(stage), stream_once);
          tma_load_2d_hint(dst + 3 * kHalfBytes, &p.tv, 64, row, full(stage), stream_once);
          issued |= 1u << stage;
          parity = (parity & ~(1u << stage)) | (ph << stage);
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1;
          }
        }
        u = next;
      }
      if (failed) {
        *abort_flag = 1;
        report_timeout(p.status, 0x30);
      }
    }
  } else {
    // ---------------- compute warps 0..3
    const int g = lane >> 2, tq = lane & 3;
    const float sl2 = kLog2e * rsqrtf((float)kD);
    int stage = 0, n_sync = 0;
    uint32_t ph = 0;
    bool failed = false;
    auto csync_all = [&]() {  // the 128 compute threads meet (bounded)
      mbar_arrive(csync);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(csync, n_sync & 1, budget, abort_flag));
      ++n_sync;
      return ok;
    };
    for (int k = 0; !failed; ++k) {
      const int slot = k % kUq;
      if (!__all_sync(0xffffffffu, mbar_wait(uq_full(slot), (k / kUq) & 1, budget, abort_flag))) {
        failed = true;
        break;
      }
      const int u = unit_q[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(uq_empty(slot));
      if (u >= p.units) break;
      const DecodeUnit un = decode_unit(p, u);
      // Q fragments straight from global memory: rows = the group's heads (zero past G)
      const __nv_bfloat16* qg = p.q + ((size_t)un.b * p.H + (size_t)un.kvh * G) * kD;
      uint32_t qf[8][4];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int c = kk * 16 + 2 * tq;
        qf[kk][0] = g < G ? *reinterpret_cast<const uint32_t*>(qg + (size_t)g * kD + c) : 0u;
        qf[kk][1] = g + 8 < G ? *reinterpret_cast<const uint32_t*>(qg + (size_t)(g + 8) * kD + c) : 0u;
        qf[kk][2] = g < G ? *reinterpret_cast<const uint32_t*>(qg + (size_t)g * kD + c + 8) : 0u;
        qf[kk][3] = g + 8 < G ? *reinterpret_cast<const uint32_t*>(qg + (size_t)(g + 8) * kD + c + 8) : 0u;
      }
      float acc[16][4];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
      float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
      for (int t = 0; t < un.n_tiles; ++t) {
        if (!__all_sync(0xffffffffu, mbar_wait(full(stage), ph, budget, abort_flag))) {
          failed = true;
          break;
        }
        const uint32_t sK = smem_u32(ring + stage * kStageBytes), sV = sK + 2 * kHalfBytes;
        const int n0 = t * kTileKeys + warp * 16;  // this warp's 16 keys (within the unit)
        const int valid = un.n_keys - n0;           // < 16: the rest of this warp's V rows are stale
        if (valid < 16) {
          // cache slots past the valid keys may hold anything: zero this warp's stale V rows
          uint8_t* vb = ring + stage * kStageBytes + 2 * kHalfBytes;
          for (int i = lane; i < 16 * 16; i += 32) {
            const int rr = i >> 4, C = i & 15;
            if (rr >= valid) *reinterpret_cast<uint4*>(vb + tsw(warp * 16 + rr, C)) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int mi = lane >> 3, rr = lane & 7;
          uint32_t bb[4];
          ldsm_x4(sK + tsw(warp * 16 + rr + 8 * (mi >> 1), kk * 2 + (mi & 1)), bb);
          mma_bf16(sc[0], qf[kk], bb[0], bb[1]);
          mma_bf16(sc[1], qf[kk], bb[2], bb[3]);
        }
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x = sc[j][e] * sl2;
            if (j * 8 + 2 * tq + (e & 1) >= valid) x = -INFINITY;
            sc[j][e] = x;
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
          const float p0 = exp2f(sc[j][0] - mu[0]), p1 = exp2f(sc[j][1] - mu[0]);
          const float p2 = exp2f(sc[j][2] - mu[1]), p3 = exp2f(sc[j][3] - mu[1]);
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
          ldsm_x4_t(sV + tsw(warp * 16 + rr + 8 * (mi & 1), dp * 2 + (mi >> 1)), bb);
          mma_bf16(acc[2 * dp], a, bb[0], bb[1]);
          mma_bf16(acc[2 * dp + 1], a, bb[2], bb[3]);
        }
        if (valid < 16) fence_proxy_async_smem();  // generic writes before the next TMA into this stage
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(stage));
        if (++stage == kStages) {
          stage = 0;
          ph ^= 1;
        }
      }
      if (failed) break;
      // merge the four warps' softmax states (rows < G) and write this split's partial
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
        lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
      }
      float* sm_m = merge;
      float* sm_l = merge + 64;
      float* sm_o = merge + 128;
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
      if (!csync_all()) {
        failed = true;
        break;
      }
      for (int idx = threadIdx.x; idx < G * kD; idx += kCompute * 32) {
        const int r = idx / kD, c = idx - r * kD;
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCompute; ++w) m = fmaxf(m, sm_m[w * 16 + r]);
        const float mu = m == -INFINITY ? 0.f : m;
        float l = 0.f, oo = 0.f;
#pragma unroll
        for (int w = 0; w < kCompute; ++w) {
          const float f = exp2f(sm_m[w * 16 + r] - mu);
          l += sm_l[w * 16 + r] * f;
          oo += sm_o[(w * 16 + r) * kD + c] * f;
        }
        const size_t hs = ((size_t)un.b * p.H + (size_t)un.kvh * G + r) * p.splits + un.split;
        p.ws_o[hs * kD + c] = oo;
        if (c == 0) {
          p.ws_ml[hs * 2 + 0] = m;
          p.ws_ml[hs * 2 + 1] = l;
        }
      }
      if (!csync_all()) {  // the merge buffer is reused by the next unit
        failed = true;
        break;
      }
    }
    if (failed) {
      *abort_flag = 1;
      if (lane == 0) report_timeout(p.status, 0x31);
    }
  }
  __syncthreads();
  // Every role has stopped. After an abort, tiles that no compute warp waited for may
  // still be landing: they complete before the CTA exits (every thread reads the same flag).
  if (*abort_flag && warp == kCompute && lane == 0) {
    volatile int never = 0;
    for (int st = 0; st < kStages; ++st)
      if (issued & (1u << st)) mbar_wait(full(st), (parity >> st) & 1, kDrainNs, &never);
  }
}

// Merge of the KV splits. One warp per (sequence, head), four channels a lane;
// one 256-thread block per SM with at most 128 registers a thread, so that the
// o_proj GEMM's CTA fits beside it and streams its first weight stages while
// the merge runs. gate (fp16, o's layout) multiplies the result; ungated (bf16)
// receives it before the gate; o is fp16 when o_f16 (the operand of an o_proj
// on prepared fp16 weights), else bf16.
constexpr int kCombineThreads = 256;
constexpr int kCombineBatch = 8;  // splits whose loads are issued together

__global__ void __launch_bounds__(kCombineThreads, 2)
    attn_decode_combine_kernel(const float* __restrict__ ws_ml, const float* __restrict__ ws_o, void* __restrict__ o,
                               int pairs, int splits, const __half* __restrict__ gate,
                               __nv_bfloat16* __restrict__ ungated, int o_f16, const DevStatus* poison) {
  pdl_launch_dependents();
  pdl_wait();
  // a split that gave up a wait wrote no partial: every output becomes NaN, so that a
  // caller without a status word to read cannot take stale partials for a result
  const bool bad = poison != nullptr && *reinterpret_cast<const volatile int*>(&poison->code) != 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kCombineThreads / 32;
  for (int pr = blockIdx.x * kWarps + warp; pr < pairs; pr += gridDim.x * kWarps) {
    const size_t base = (size_t)pr * splits;  // pr = b * H + h
    // groups of kCombineBatch splits whose loads are all in flight together; a
    // later group with a larger maximum rescales what the earlier ones summed
    float m = -INFINITY, l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < splits; s0 += kCombineBatch) {
      float2 ml[kCombineBatch];
      float4 ov[kCombineBatch];
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) {
        const bool in = s0 + j < splits;
        ml[j] = in ? *reinterpret_cast<const float2*>(ws_ml + (base + s0 + j) * 2) : make_float2(-INFINITY, 0.f);
        ov[j] = in ? *reinterpret_cast<const float4*>(ws_o + (base + s0 + j) * kD + 4 * lane)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float gm = m;
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) gm = fmaxf(gm, ml[j].x);
      const float mu = gm == -INFINITY ? 0.f : gm;
      const float sc = exp2f(m - mu);  // 0 for the first group
      l *= sc;
      acc = make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc);
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) {
        const float f = exp2f(ml[j].x - mu);
        l += ml[j].y * f;
        acc = make_float4(acc.x + ov[j].x * f, acc.y + ov[j].y * f, acc.z + ov[j].z * f, acc.w + ov[j].w * f);
      }
      m = gm;
    }
    const size_t i = (size_t)pr * kD + 4 * lane;
    float r[4] = {acc.x / l, acc.y / l, acc.z / l, acc.w / l};
    if (bad) r[0] = r[1] = r[2] = r[3] = __int_as_float(0x7fc00000);
    if (ungated) {
      const __nv_bfloat162 a = __floats2bfloat162_rn(r[0], r[1]), b = __floats2bfloat162_rn(r[2], r[3]);
      *reinterpret_cast<uint2*>(ungated + i) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    }
    if (gate) {
      const uint2 gw = *reinterpret_cast<const uint2*>(gate + i);
      const float2 g01 = __half22float2(*reinterpret_cast<const __half2*>(&gw.x));
      const float2 g23 = __half22float2(*reinterpret_cast<const __half2*>(&gw.y));
      r[0] *= g01.x;
      r[1] *= g01.y;
      r[2] *= g23.x;
      r[3] *= g23.y;
    }
    uint2 ow;
    if (o_f16) {
      const __half2 a = __floats2half2_rn(r[0], r[1]), b = __floats2half2_rn(r[2], r[3]);
      ow = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
      *reinterpret_cast<uint2*>(static_cast<__half*>(o) + i) = ow;
    } else {
      const __nv_bfloat162 a = __floats2bfloat162_rn(r[0], r[1]), b = __floats2bfloat162_rn(r[2], r[3]);
      ow = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o) + i) = ow;
    }
  }
}

}  // namespace

// Splits of about 2048 keys (32 tiles), the last one up to twice that: units that the
// persistent CTAs take in turn from a shared counter. Each unit pays a fixed cost (its q
// fragments, the merge of the compute warps' softmax states, the partial writes and the
// combine's reads of them), so long units win once the (sequence, KV head) pairs alone
// give the SMs enough of them; with too few pairs to keep ~80% of the SMs busy the splits
// shrink, down to 256 keys. (64 sequences x 8 KV heads x 4097 keys: splits of 512 keys
// take 252 us a step, of 1024 to 2048 keys 244.5 us.)
int attn_decode_splits(int B, int Hkv, int max_len, int num_sms) {
  const int groups = std::max(1, B * Hkv);
  int s = std::max(1, max_len / 2048);
  const int fill = (num_sms * 4 / 5 + groups - 1) / groups;
  if (s < fill) s = std::min(fill, std::max(1, max_len / 256));
  return std::min(s, 64);
}

int attn_decode_split_cap(int max_len) { return std::min(64, std::max(1, max_len / 512)); }

size_t attn_decode_ws_bytes(int B, int H, int d, int max_splits) {
  return kAttnCounterBytes + (size_t)B * H * max_splits * (2 + d) * sizeof(float);
}

namespace {

cudaError_t decode_core(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv, int kv_stride,
                        const int* kv_lens, int len_add, int splits, int max_len, float* ws, int num_sms,
                        DevStatus* st, unsigned long long wait_ns, cudaStream_t s, const char** why,
                        const AttnOpts& opt) {
  static std::atomic<unsigned long long> configured{0};  // one bit per device
  {
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(attn_decode_kernel), kSmem, configured);
    if (e != cudaSuccess) return e;
  }
  DecodeParams p;
  memset(static_cast<void*>(&p), 0, sizeof(p));
  if (!make_tma_2d_16b(&p.tk, k, B * Hkv * kv_stride, kD, kTileKeys, false) ||
      !make_tma_2d_16b(&p.tv, v, B * Hkv * kv_stride, kD, kTileKeys, false)) {
    *why = "cuTensorMapEncodeTiled failed for the KV cache";
    return cudaErrorInvalidValue;
  }
  // max_len: the most keys a sequence attends to (at most the window)
  if (opt.window > 0 && opt.window < max_len) max_len = opt.window;
  // whole 64-key tiles per split; the last split also takes the remainder
  const int chunk = std::max(kTileKeys, max_len / splits / kTileKeys * kTileKeys);
  p.q = static_cast<const __nv_bfloat16*>(q);
  // the unit counter, then the partials
  p.work = reinterpret_cast<int*>(ws);
  if (!opt.counter_zeroed) {
    cudaError_t e = cudaMemsetAsync(p.work, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
  }
  p.ws_ml = ws + kAttnCounterBytes / sizeof(float);
  p.ws_o = p.ws_ml + (size_t)B * H * splits * 2;
  p.kv_lens = kv_lens;
  p.len_add = len_add;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.kv_stride = kv_stride;
  p.chunk = chunk;
  p.splits = splits;
  p.units = B * Hkv * splits;
  p.window = opt.window > 0 ? opt.window : 0;
  p.status = st;
  p.wait_ns = wait_ns;
  const int grid = p.units < num_sms ? p.units : num_sms;
  launch_pdl(attn_decode_kernel, grid, kThreads, kSmem, s, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int pairs = B * H;
  const int cwarps = kCombineThreads / 32;
  const int cgrid = std::min(num_sms, (pairs + cwarps - 1) / cwarps);
  launch_pdl(attn_decode_combine_kernel, cgrid, kCombineThreads, 0, s, p.ws_ml, p.ws_o, o, pairs, splits,
             static_cast<const __half*>(opt.gate), static_cast<__nv_bfloat16*>(opt.ungated), opt.o_f16 ? 1 : 0,
             opt.poison_on_timeout);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_decode_bf16(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv,
                                    int d, int kv_stride, const int* kv_lens, int len_add, int max_len,
                                    int split_cap, void* ws, int num_sms, DevStatus* st, unsigned long long wait_ns,
                                    cudaStream_t s, const char** why, const AttnOpts& opt) {
  if (d != kD) {
    *why = "bf16 attention: head_dim must be 128";
    return cudaErrorInvalidValue;
  }
  if (H / Hkv > 16) {
    *why = "bf16 decode attention: at most 16 query heads per KV head";
    return cudaErrorInvalidValue;
  }
  if (B <= 0) return cudaSuccess;
  // max_len: upper bound of the keys per sequence this step (lens + len_add); a window caps it
  const int span = opt.window > 0 && opt.window < max_len ? opt.window : max_len;
  int splits = attn_decode_splits(B, Hkv, span, num_sms);
  if (splits > split_cap) splits = split_cap;  // the workspace holds split_cap splits: chunks grow instead
  return decode_core(q, k, v, o, B, H, Hkv, kv_stride, kv_lens, len_add, splits, max_len, static_cast<float*>(ws),
                     num_sms, st, wait_ns, s, why, opt);
}

// ------------------------------------------------------------------ allocation-free decode variant

// Fixed device scratch for the allocation-free decode attention entry point:
// the per-split softmax partials (max, sum, unnormalised output) that the
// workspace-taking path keeps in caller memory. Every device that loads the
// library holds it until exit; every call shares it.
static __device__ __align__(256) float g_decode_scratch[kDecodeStaticScratchBytes / sizeof(float)];

namespace {
std::mutex g_scratch_mu;
constexpr size_t kStaticStatusOffset = 64;  // the status word's byte offset in the counter region
static_assert(kStaticStatusOffset + sizeof(DevStatus) <= kAttnCounterBytes, "counter region");
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
                                           unsigned long long wait_ns, cudaStream_t s, const char** why) {
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
  if (per_split > kDecodeStaticScratchBytes - kAttnCounterBytes) {
    *why = "allocation-free decode attention: batch * n_heads * (head_dim + 2) * 4 bytes exceeds the 16 MiB scratch";
    return cudaErrorInvalidValue;
  }
  float* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    *why = "cudaGetSymbolAddress of the decode scratch failed";
    return e;
  }
  int splits = attn_decode_split_cap(kv_stride);  // splits of 512 keys, at most 64
  const int fit = (int)((kDecodeStaticScratchBytes - kAttnCounterBytes) / per_split);
  if (splits > fit) splits = fit;
  // The scratch's first kAttnCounterBytes hold the unit counter (byte 0) and this
  // call's status word (byte kStaticStatusOffset); both are zeroed before the launch.
  // Every partial the combine step reads is written by this call first, unless a wait
  // gave up: the status word then records it and the combine step writes NaN to o.
  cudaError_t e2 = cudaMemsetAsync(scratch, 0, kStaticStatusOffset + sizeof(DevStatus), s);
  if (e2 != cudaSuccess) return e2;
  DevStatus* st = reinterpret_cast<DevStatus*>(reinterpret_cast<uint8_t*>(scratch) + kStaticStatusOffset);
  AttnOpts opt;
  opt.counter_zeroed = true;
  opt.poison_on_timeout = st;
  return decode_core(q, k, v, o, B, H, Hkv, kv_stride, kv_lens, 0, splits, kv_stride, scratch, num_sms, st, wait_ns,
                     s, why, opt);
}

}  // namespace blk
