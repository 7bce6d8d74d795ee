// tcgen05 / TMEM GEMM for sm_103a: C = A * B^T with A [M, K] and B [N, K] both
// K-major bf16, fp32 accumulation in tensor memory, operands staged by TMA.
//
// One persistent CTA per SM (192 threads):
//   warp 0      TMA producer: fills a ring of shared-memory stages (A tile
//               128 x 64, B tile BN x 64, 128-byte swizzled) on mbarriers.
//   warp 1      allocates 2*BN TMEM columns; lane 0 issues tcgen05.mma
//               (128 x BN x 16 per instruction, 4 per stage) into one of two
//               accumulators and commits stage releases / accumulator-ready.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one row per thread),
//               fused post-processing, stores to global memory.
// The two accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
// A CTA pair (cluster of 2, tcgen05 cta_group::2) computes a 256 x BN tile: each
// CTA loads its 128 A rows and half of the B tile, the even CTA issues the MMAs for
// both. The prefill GEMMs walk their tiles in bands of M tiles (all N tiles of a band
// before the next), so that a band's A rows stay in L2 while the B panels stream.
// The decode GEMMs put the weights on the MMA's M side, split K over the CTAs of a
// cluster and finish each tile inside the cluster (distributed shared memory).
//
// Fused epilogues cover the projections of the decoder block ("LlamaForCausalLM-
// 32L-4096d" sheet, "Implementing it"): per-head q/k RMSNorm + RoPE + scatter
// to head-major q/k/v ("apertus", "Queries and keys are normed per head, before
// the rotary"), the residual adds after o_proj and down_proj, SiLU-gated,
// squared-ReLU ("arcee") and xIELU ("apertus") activations, and transposed
// split-K partials for the weight-streaming decode GEMMs (tokens on the MMA's
// N dimension).
//
// Every wait is bounded in wall time; on expiry the CTA records a timeout in
// the status word, drains its own copies and MMAs in flight, frees its TMEM
// and returns.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kThreadsEpi = 128;  // epilogue warps 2..5
// Drains after an abort wait for copies/MMAs already issued; they use their
// own limit so that a tiny debug timeout cannot cut them short.
constexpr unsigned long long kDrainNs = 2000000000ULL;
// After an abort, how long the odd CTA of a pair stays resident past its last
// load issue (it cannot observe its loads complete; a load takes microseconds).
constexpr unsigned long long kSettleNs = 2000000ULL;

constexpr int kMaxSmem = 232448;  // 227 KB of dynamic shared memory per CTA

constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p *= 2;
  return p;
}

// SwiGLU tiles 256 wide (a 128-column bf16 output) store through shared memory and TMA:
// their ring keeps its depth with the 8 KB of staging, narrower ones would lose a stage
template <int BN, int EPI>
__host__ __device__ constexpr bool swiglu_tma() {
  return EPI == (int)Epi::kSwiglu && BN == 256;
}

template <int BN, int EPI = -1, bool PAIR = false>
struct TcCfg {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = (PAIR ? BN / 2 : BN) * kBK * 2;  // a pair: each CTA holds half of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarBytes = 256;
  // kDecAct: two partial-tile buffers [BN tokens][128 rows] fp32 and the 1/rms of up to BN tokens
  static constexpr int kPartBytes = BN * kBM * 4;
  // kResidTma: two 4 KB staging buffers (32 rows x 32 fp32 columns) per epilogue warp
  static constexpr int kStoreBytes = 4 * 2 * 4096;
  // 256-wide SwiGLU: one staging box of 32 rows x 32 bf16 columns (2 KB) per epilogue warp
  static constexpr int kExtraBytes = EPI == (int)Epi::kDecAct
                                         ? 2 * kPartBytes + 4 * BN
                                         : (EPI == (int)Epi::kResidTma ? kStoreBytes
                                                                        : (swiglu_tma<BN, EPI>() ? 4 * 2048 : 0));
  static constexpr int kFit = (kMaxSmem - 1024 - kBarBytes - kExtraBytes) / kStageBytes;
  static constexpr int kStages = kFit > 8 ? 8 : kFit;  // as deep a TMA ring as fits
  static constexpr int kTmemCols = pow2_at_least(2 * BN);  // two accumulators
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kExtraBytes + kBarBytes;
  static_assert(BN % 16 == 0 && BN >= 64 && BN <= 256, "UMMA N for M = 128");
  static_assert(kSmemBytes <= kMaxSmem, "shared memory");
};

// the residual epilogues: kResid, and kResidTma (its fp32 output through TMA stores)
template <int EPI>
__host__ __device__ constexpr bool is_resid() {
  return EPI == (int)Epi::kResid || EPI == (int)Epi::kResidTma;
}

template <int EPI>
__host__ __device__ constexpr bool is_dec_epi() {
  return EPI == (int)Epi::kDecQkv || EPI == (int)Epi::kDecResid;
}

// Launched as thread-block clusters of the K splits.
template <int EPI>
__host__ __device__ constexpr bool is_cluster_epi() {
  return is_dec_epi<EPI>() || EPI == (int)Epi::kDecAct;
}

// Tile widths built per epilogue (a GEMM picks its width on the host).
template <int BN, int EPI>
__host__ __device__ constexpr bool tc_supported() {
  if (is_dec_epi<EPI>()) return BN == 64 || BN == 128 || BN == 256;
  if (EPI == (int)Epi::kDecAct) return BN == 64;
  if (EPI == (int)Epi::kQkv) return BN == 128 || BN == 256;  // whole heads
  if (EPI == (int)Epi::kPartialT) return BN == 64 || BN == 128 || BN == 256;
  if (EPI == (int)Epi::kStore) return true;
  if (EPI == (int)Epi::kSwiglu) return BN == 128 || BN == 192 || BN == 256 || BN == 224;
  return BN == 128 || BN == 192 || BN == 224 || BN == 256;
}

struct TcParams {
  CUtensorMap ta[kMaxSegs];
  CUtensorMap tb[kMaxSegs];
  CUtensorMap tout;  // kResidTma: the fp32 output [rows, ldo], boxes of 32 x 32, 128-byte swizzle
  int a_tiles[kMaxSegs + 1];  // prefix sums of m-tiles per A segment
  int a_rows[kMaxSegs];
  int a_out[kMaxSegs];
  int b_tiles[kMaxSegs + 1];  // prefix sums of n-tiles per B segment
  int b_rows[kMaxSegs];
  int b_out[kMaxSegs];
  int na, nb;
  int b_paired;
  int a_paired;  // A tile = 64 rows of ta[0] over 64 rows of ta[1] (kDecAct: gate over up)
  int f16;  // fp16 operands (else bf16)
  int const_op;  // 1: A, 2: B is constant over the stream (may be loaded before pdl_wait)
  int a_once;    // every A tile is read by one unit only (a weight stream): L2 evict-first
  int num_kb;
  int k_splits;
  int m_tiles, n_tiles;
  int num_units;
  int group_m;  // > 1: tiles walk bands of group_m M tiles, N within a band (L2 reuse of A and B)
  TcEpiArgs e;
  DevStatus* status;
  unsigned long long wait_ns;
};

struct Unit {
  int a_seg, a_row0;  // A segment and first row of the tile inside it
  int b_seg, b_row0;
  int m_tile;
  int ks, kb_begin, kb_end;
};

// (M tile, N tile) of tile index t. The CTAs working at one time hold consecutive
// indices; walking bands of group_m M tiles with N varying across the band makes
// that set a near-square patch of tiles, whose A row blocks and B column blocks are
// each read by several of them while in L2 (M fastest over all M tiles would make
// every round of the grid stream the whole of A again).
template <bool kGrouped>
__device__ __forceinline__ void tile_mn(const TcParams& p, int t, int& m_tile, int& n_tile) {
  if (!kGrouped || p.group_m <= 1) {
    m_tile = t % p.m_tiles;
    n_tile = t / p.m_tiles;
    return;
  }
  const int per_band = p.group_m * p.n_tiles;
  const int band = t / per_band;
  const int idx = t - band * per_band;
  const int m0 = band * p.group_m;
  const int gm = min(p.group_m, p.m_tiles - m0);  // the last band may be narrower
  m_tile = m0 + idx % gm;
  n_tile = idx / gm;
}

// kGrouped: the prefill GEMMs' banded order (the decode GEMMs keep M fastest)
template <bool kGrouped = false>
__device__ __forceinline__ Unit decode_unit(const TcParams& p, int u, int bn_rows) {
  Unit r;
  const int tile = u / p.k_splits;
  r.ks = u - tile * p.k_splits;
  int m_tile, n_tile;
  tile_mn<kGrouped>(p, tile, m_tile, n_tile);
  r.m_tile = m_tile;
  int s = 0;
  while (s + 1 < p.na && m_tile >= p.a_tiles[s + 1]) ++s;
  r.a_seg = s;
  r.a_row0 = (m_tile - p.a_tiles[s]) * (p.a_paired ? kBM / 2 : kBM);
  s = 0;
  while (s + 1 < p.nb && n_tile >= p.b_tiles[s + 1]) ++s;
  r.b_seg = p.b_paired ? 0 : s;
  r.b_row0 = (n_tile - p.b_tiles[r.b_seg]) * bn_rows;
  r.kb_begin = (int)(((long long)r.ks * p.num_kb) / p.k_splits);
  r.kb_end = (int)(((long long)(r.ks + 1) * p.num_kb) / p.k_splits);
  return r;
}

// Work unit of a CTA pair (M = 256 tiles, no K split): m_tiles counts 256-row
// tiles; this CTA's A rows and epilogue rows are the pair tile's half prank.
__device__ __forceinline__ Unit pair_unit(const TcParams& p, int u, int bn_rows, int prank) {
  Unit r;
  int m_pair, n_tile;
  tile_mn<true>(p, u, m_pair, n_tile);
  r.ks = 0;
  r.kb_begin = 0;
  r.kb_end = p.num_kb;
  r.m_tile = 2 * m_pair + prank;
  r.a_seg = 0;
  r.a_row0 = r.m_tile * kBM;
  int s = 0;
  while (s + 1 < p.nb && n_tile >= p.b_tiles[s + 1]) ++s;
  r.b_seg = p.b_paired ? 0 : s;
  r.b_row0 = (n_tile - p.b_tiles[r.b_seg]) * bn_rows;
  return r;
}

// ------------------------------------------------------------------ epilogues

template <typename F>
__device__ __forceinline__ void store_bf16_row(__nv_bfloat16* dst, const float* v, int n_valid, F&& f) {
  // writes up to 16 values (f applied) to dst[0..16) with the tail predicated
  if (n_valid >= 16) {
    uint4 a, b;
    a.x = pack_bf16x2(f(v[0], 0), f(v[1], 1));
    a.y = pack_bf16x2(f(v[2], 2), f(v[3], 3));
    a.z = pack_bf16x2(f(v[4], 4), f(v[5], 5));
    a.w = pack_bf16x2(f(v[6], 6), f(v[7], 7));
    b.x = pack_bf16x2(f(v[8], 8), f(v[9], 9));
    b.y = pack_bf16x2(f(v[10], 10), f(v[11], 11));
    b.z = pack_bf16x2(f(v[12], 12), f(v[13], 13));
    b.w = pack_bf16x2(f(v[14], 14), f(v[15], 15));
    reinterpret_cast<uint4*>(dst)[0] = a;
    reinterpret_cast<uint4*>(dst)[1] = b;
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)  // compile-time indices keep v in registers
      if (i < n_valid) dst[i] = __float2bfloat16_rn(f(v[i], i));
  }
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 16 values to 16 consecutive 2-byte elements: fp16 when f16, else bf16.
__device__ __forceinline__ void store16_2b(void* dst, const float* v, bool f16) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = f16 ? pack_f16x2(v[2 * i], v[2 * i + 1]) : pack_bf16x2(v[2 * i], v[2 * i + 1]);
  reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// g / (1 + e^-g) with the fast division, as sigmoid_f
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// e^x - 1 for x <= 0 to well within bf16 output precision: the Taylor series
// x + x^2/2! + ... + x^5/5! near 0 (truncation below 1e-9 relative for |x| < 1/16),
// 2^(x log2 e) - 1 on the MUFU unit elsewhere (|e^x - 1| >= 0.06 there).
__device__ __forceinline__ float expm1_nonpos(float x) {
  const float taylor = x * fmaf(x, fmaf(x, fmaf(x, fmaf(x, 1.0f / 120.0f, 1.0f / 24.0f), 1.0f / 6.0f), 0.5f), 1.0f);
  float e2;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e2) : "f"(x * 1.4426950408889634f));
  return x > -0.0625f ? taylor : e2 - 1.0f;
}

// 32 values of a residual row from the element at off (fp32 or bf16 stream), zero where
// n_valid (the row's valid columns from off) runs out or there is no residual.
__device__ __forceinline__ void load_resid32(const TcEpiArgs& e, size_t off, int n_valid, float (&rr)[32]) {
  if (!e.resid || n_valid <= 0) {
#pragma unroll
    for (int j = 0; j < 32; ++j) rr[j] = 0.f;
  } else if (e.resid_f32) {
    const float* rf = reinterpret_cast<const float*>(e.resid) + off;
    if (n_valid >= 32) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 f4 = reinterpret_cast<const float4*>(rf)[j];
        rr[4 * j] = f4.x;
        rr[4 * j + 1] = f4.y;
        rr[4 * j + 2] = f4.z;
        rr[4 * j + 3] = f4.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) rr[j] = j < n_valid ? rf[j] : 0.f;
    }
  } else {
    const __nv_bfloat16* rb = reinterpret_cast<const __nv_bfloat16*>(e.resid) + off;
    if (n_valid >= 32) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 u = reinterpret_cast<const uint4*>(rb)[j];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f2 = unpack_bf16x2(w[i]);
          rr[8 * j + 2 * i] = f2.x;
          rr[8 * j + 2 * i + 1] = f2.y;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) rr[j] = j < n_valid ? __bfloat162float(rb[j]) : 0.f;
    }
  }
}

// Pulls a residual row segment [off, off + n) into L2 ahead of the epilogue that reads it.
__device__ __forceinline__ void prefetch_resid_l2(const TcEpiArgs& e, size_t off, int n) {
  if (!e.resid || n <= 0) return;
  const int es = e.resid_f32 ? 4 : 2;
  const char* base = reinterpret_cast<const char*>(e.resid) + off * es;
  const char* end = base + (size_t)n * es;
  for (const char* a = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(base) & ~uintptr_t(127)); a < end;
       a += 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// Per-row RMSNorm factor rsqrt(mean(row^2) + eps) from an accumulated sum of squares.
// The partial sums of a row (one per producer tile) are added in a fixed order: deterministic.
__device__ __forceinline__ float row_norm_factor(const TcEpiArgs& e, int row, bool row_ok) {
  if (!e.row_ss || !row_ok) return 1.0f;
  const float* ps = e.row_ss + (size_t)row * e.ss_parts;
  float t = 0.f;
  for (int i = 0; i < e.ss_parts; ++i) t += ps[i];
  return rsqrtf(t / (float)e.ss_n + e.ss_eps);
}

// kResid, after a row of a tile is stored: its sum of squares for the next RMSNorm, and a
// prefill chunk's length bump (once per sequence).
template <int BN>
__device__ __forceinline__ void resid_row_done(const TcParams& p, const Unit& un, int row, bool row_ok,
                                               float ss_part) {
  const TcEpiArgs& e = p.e;
  if (e.norm_ss && row_ok) e.norm_ss[(size_t)row * e.norm_parts + un.b_row0 / BN] = ss_part;
  // a prefill chunk appended to a KV cache: its sequence's length grows by seq, once
  if (e.bump_lens && row_ok && un.b_row0 == 0 && un.b_seg == 0 && row % e.seq == e.seq - 1)
    atomicAdd(e.bump_lens + row / e.seq, e.seq);
}

// stage: the decode finishers' partial tile, or (kResidTma) this warp's staging buffers;
// store_chunks (kResidTma): the warp's count of chunks stored so far (its buffer parity).
template <int BN, int EPI>
__device__ __forceinline__ void run_epilogue(const TcParams& p, const Unit& un, uint32_t taddr, int r_in_tile,
                                             float* stage, int* store_chunks = nullptr) {
  const TcEpiArgs& e = p.e;
  if constexpr (is_cluster_epi<EPI>()) {
    // decode finishers: this split's partial tile [token in tile][128 tile rows] in shared memory
    // (the idle operand ring, or a kDecAct partial buffer), read by the cluster's CTAs
    float* blk = stage + r_in_tile;
    const int ntok = min(BN, e.n_tok - un.b_row0);
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      if (c0 >= ntok) break;  // uniform across the warp
      float v0[16], v1[16];
      tmem_ld16(taddr + c0, v0);
      tmem_ld16(taddr + c0 + 16, v1);
      tc_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + j < ntok) blk[(c0 + j) * kBM] = v0[j];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + 16 + j < ntok) blk[(c0 + 16 + j) * kBM] = v1[j];
    }
    return;
  } else if constexpr (EPI == (int)Epi::kPartialT) {
    // rows of the tile are output features, columns are tokens
    const int f_local = un.a_row0 + r_in_tile;
    const bool ok = f_local < p.a_rows[un.a_seg];
    const int f = p.a_out[un.a_seg] + f_local;
    float* part = reinterpret_cast<float*>(e.out) + (size_t)un.ks * e.n_tok * e.part_ld;
    const int tok0 = un.b_row0;  // tokens are the B rows
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      if (tok0 + c0 >= e.n_tok) break;  // uniform across the warp
      float v0[16], v1[16];
      tmem_ld16(taddr + c0, v0);
      tmem_ld16(taddr + c0 + 16, v1);
      tc_wait_ld();
      if (ok) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (tok0 + c0 + j < e.n_tok) part[(size_t)(tok0 + c0 + j) * e.part_ld + f] = v0[j];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (tok0 + c0 + 16 + j < e.n_tok) part[(size_t)(tok0 + c0 + 16 + j) * e.part_ld + f] = v1[j];
      }
    }
    return;
  } else {
    const int row = un.m_tile * kBM + r_in_tile;  // activations are a single A segment
    const bool row_ok = row < p.a_rows[0];
    if constexpr (EPI == (int)Epi::kQkv) {
      const int d = e.head_dim;  // 128
      const int seg = un.b_seg;
      const int b = row_ok ? row / e.seq : 0;
      const int t = row_ok ? row - b * e.seq : 0;
      const int pos = (e.pos0 ? e.pos0[b] : 0) + t;
      // (a padding row of a left-padded batch sits at a negative position: never read before the table)
      const float2* cs = e.rope + (size_t)min(max(pos, 0), e.rope_max_pos - 1) * (d / 2);
      // the input RMSNorm's 1/rms, applied here instead of to the GEMM's A rows
      const float rs = (e.row_scale && row_ok) ? e.row_scale[row] : 1.0f;
      const bool f16 = e.qkv_f16 != 0;
      int qk_heads = 0;  // the tile's q/k heads (bit hh), handled after the loop
      uint16_t* qk_dst[BN / 128];
      bool qk_ok = false;
#pragma unroll
      for (int hh = 0; hh < BN / 128; ++hh) {
        const int head = (un.b_row0 >> 7) + hh;
        const uint32_t tcol = taddr + hh * 128;
        if (seg == 3) {
          // the attention gate ("afmoe": one value per channel of every head): sigmoid, fp16,
          // in the attention output's layout [row][head][d]
          uint16_t* gd = reinterpret_cast<uint16_t*>(e.gate) + ((size_t)row * e.n_heads + head) * d;
#pragma unroll 1
          for (int c0 = 0; c0 < 128; c0 += 32) {
            float v0[16], v1[16];
            tmem_ld16(tcol + c0, v0);
            tmem_ld16(tcol + c0 + 16, v1);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              v0[j] = sigmoid_f(v0[j] * rs);
              v1[j] = sigmoid_f(v1[j] * rs);
            }
            if (row_ok) {
              store16_2b(gd + c0, v0, true);
              store16_2b(gd + c0 + 16, v1, true);
            }
          }
          continue;
        }
        uint16_t* dst;  // 2-byte elements (bf16 or fp16)
        if (seg == 0)
          dst = reinterpret_cast<uint16_t*>(e.q) + (((size_t)b * e.n_heads + head) * e.seq + t) * d;
        else
          dst = reinterpret_cast<uint16_t*>(seg == 1 ? e.k : e.v) +
                (((size_t)b * e.n_kv_heads + head) * e.kv_stride + (e.kv_at_pos ? pos : t)) * d;
        // a cache slot past the capacity is never written (the host refuses such calls first)
        const bool store_ok = row_ok && (seg == 0 || !e.kv_at_pos || (pos >= 0 && pos < e.kv_stride));
        if (seg == 2) {
#pragma unroll 1
          for (int c0 = 0; c0 < 128; c0 += 32) {
            float v0[16], v1[16];
            tmem_ld16(tcol + c0, v0);
            tmem_ld16(tcol + c0 + 16, v1);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              v0[j] *= rs;
              v1[j] *= rs;
            }
            if (store_ok) {
              store16_2b(dst + c0, v0, f16);
              store16_2b(dst + c0 + 16, v1, f16);
            }
          }
          continue;
        }
        qk_heads |= 1 << hh;  // q or k: normed and rotated below, both heads of the tile at once
        qk_dst[hh] = dst;
        qk_ok = store_ok;
      }
      if (qk_heads) {
        // q/k heads: the optional RMSNorm per head, then the rotary with the row's (cos, sin)
        // read once for the tile's heads (16-byte loads, a 16-pair chunk at a time)
        const int nh = BN / 128;
        const __nv_bfloat16* gain =
            e.qk_norm ? reinterpret_cast<const __nv_bfloat16*>(seg == 0 ? e.q_gain : e.k_gain) : nullptr;
        float rn[BN / 128];
#pragma unroll
        for (int hh = 0; hh < nh; ++hh) {
          rn[hh] = 1.0f;
          if (gain) {
            float ss = 0.f;
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
              float v0[16], v1[16];
              tmem_ld16(taddr + hh * 128 + c0, v0);
              tmem_ld16(taddr + hh * 128 + c0 + 16, v1);
              tc_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) ss += v0[j] * v0[j] + v1[j] * v1[j];
            }
            rn[hh] = rsqrtf(ss * rs * rs / 128.0f + e.eps);
          }
        }
#pragma unroll 1
        for (int i0 = 0; i0 < 64; i0 += 16) {
          float2 sc[16];
          const float4* cs4 = reinterpret_cast<const float4*>(cs + i0);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 f = cs4[j];
            sc[2 * j] = make_float2(f.x, f.y);
            sc[2 * j + 1] = make_float2(f.z, f.w);
          }
          float g1[16], g2[16];
          if (gain) {
            const uint4* ga = reinterpret_cast<const uint4*>(gain + i0);
            const uint4* gb = reinterpret_cast<const uint4*>(gain + 64 + i0);
            const uint4 a0 = ga[0], a1 = ga[1], b0 = gb[0], b1 = gb[1];
            const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float2 fa = unpack_bf16x2(wa[j]), fb = unpack_bf16x2(wb[j]);
              g1[2 * j] = fa.x;
              g1[2 * j + 1] = fa.y;
              g2[2 * j] = fb.x;
              g2[2 * j + 1] = fb.y;
            }
          }
#pragma unroll
          for (int hh = 0; hh < nh; ++hh) {
            if (!((qk_heads >> hh) & 1)) continue;
            float x1[16], x2[16];
            tmem_ld16(taddr + hh * 128 + i0, x1);
            tmem_ld16(taddr + hh * 128 + 64 + i0, x2);
            tc_wait_ld();
            float y1[16], y2[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float a = x1[j] * rs, c = x2[j] * rs;
              if (gain) {
                a = a * rn[hh] * g1[j];
                c = c * rn[hh] * g2[j];
              }
              y1[j] = a * sc[j].x - c * sc[j].y;
              y2[j] = c * sc[j].x + a * sc[j].y;
            }
            if (qk_ok) {
              store16_2b(qk_dst[hh] + i0, y1, f16);
              store16_2b(qk_dst[hh] + 64 + i0, y2, f16);
            }
          }
        }
      }
      return;
    } else if constexpr (EPI == (int)Epi::kSwiglu) {
      // B halves: gate rows at TMEM columns [0, BN/2), up rows at [BN/2, BN)
      const int col0 = un.b_row0;
      const int n_valid = p.b_rows[0] - col0;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(e.out) + (size_t)row * e.ldo + col0;
      const float r2 = row_norm_factor(e, row, row_ok);  // the post-attention RMSNorm's 1/rms
      if constexpr (swiglu_tma<BN, EPI>()) {
        // the 128 output columns leave through shared memory: each 32-column chunk of the
        // warp's 32 rows goes into its 2 KB staging box in the output map's 64-byte swizzle
        // (16-byte chunk q of row r at q ^ ((r / 2) % 4)) and one lane stores the box with a
        // bulk tensor copy; rows past the output and columns past its width are clipped
        const int lane = r_in_tile & 31;
        const int row0 = un.m_tile * kBM + (r_in_tile & ~31);  // the warp's first row
        const uint32_t buf = smem_u32(stage);
#pragma unroll 1
        for (int c0 = 0; c0 < BN / 2; c0 += 32) {
          float g[32], u[32];
          tmem_ld16(taddr + c0, *reinterpret_cast<float(*)[16]>(&g[0]));
          tmem_ld16(taddr + c0 + 16, *reinterpret_cast<float(*)[16]>(&g[16]));
          tmem_ld16(taddr + BN / 2 + c0, *reinterpret_cast<float(*)[16]>(&u[0]));
          tmem_ld16(taddr + BN / 2 + c0 + 16, *reinterpret_cast<float(*)[16]>(&u[16]));
          tc_wait_ld();
          if (c0 >= n_valid) continue;  // uniform across the warp
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(silu_f(g[2 * i] * r2) * (u[2 * i] * r2), silu_f(g[2 * i + 1] * r2) * (u[2 * i + 1] * r2));
          if (lane == 0) bulk_wait_group_read<0>();  // the previous box has left the buffer
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_shared_u4(buf + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4), w[4 * q], w[4 * q + 1], w[4 * q + 2],
                         w[4 * q + 3]);
          fence_proxy_async_smem();  // the generic-proxy writes, before the bulk copy reads them
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.tout, buf, col0 + c0, row0);
            bulk_commit_group();
          }
        }
        return;
      }
#pragma unroll 1
      for (int c0 = 0; c0 < BN / 2; c0 += 16) {
        float g[16], u[16];
        tmem_ld16(taddr + c0, g);
        tmem_ld16(taddr + BN / 2 + c0, u);
        tc_wait_ld();
        if (row_ok && c0 < n_valid) {
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = silu_f(g[j] * r2) * (u[j] * r2);
          auto id = [](float x, int) { return x; };
          store_bf16_row(out + c0, v, min(16, n_valid - c0), id);
        }
      }
      return;
    } else if constexpr (EPI == (int)Epi::kResidTma) {
      // kResid whose fp32 output goes through shared memory: each 32-column chunk of the
      // warp's 32 rows is written into one of the warp's two 4 KB staging buffers (the
      // 128-byte swizzle the output's tensor map uses: 16-byte chunk q of row r at q ^ (r % 8)),
      // and one lane stores the 32 x 32 box with a bulk tensor copy, so the residual stream
      // leaves the SM as whole lines. Rows past the output and columns past its width are
      // clipped by the tensor map. The fp16 normed rows, the taps and the row's sum of
      // squares are stored as in kResid.
      const int lane = r_in_tile & 31;
      const int row0 = un.m_tile * kBM + (r_in_tile & ~31);  // the warp's first row
      const int col0 = p.b_out[un.b_seg] + un.b_row0;
      const int n_valid = p.b_rows[un.b_seg] - un.b_row0;
      __nv_bfloat16* tap = (e.tap && row_ok) ? reinterpret_cast<__nv_bfloat16*>(e.tap) + (size_t)row * e.ldo + col0
                                             : nullptr;
      const uint32_t sbase = smem_u32(stage);
      auto id = [](float x, int) { return x; };
      float ss_part = 0.f;
      const size_t roff = (size_t)row * e.ldo + col0;
      float rnext[32];
      load_resid32(e, roff, row_ok ? n_valid : 0, rnext);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float v[32];
        tmem_ld16(taddr + c0, *reinterpret_cast<float(*)[16]>(&v[0]));
        tmem_ld16(taddr + c0 + 16, *reinterpret_cast<float(*)[16]>(&v[16]));
        float rcur[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) rcur[j] = rnext[j];
        if (c0 + 32 < BN) load_resid32(e, roff + c0 + 32, row_ok ? n_valid - c0 - 32 : 0, rnext);
        tc_wait_ld();
        if (c0 >= n_valid) continue;  // uniform across the warp
        float o[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = rcur[j] + v[j];
        // this chunk's buffer is free once the store issued two chunks back has read it
        const uint32_t buf = sbase + (static_cast<uint32_t>(*store_chunks & 1) << 12);
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          st_shared_f4(buf + lane * 128 + ((q ^ (lane & 7)) << 4), o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        fence_proxy_async_smem();  // the generic-proxy writes, before the bulk copy reads them
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&p.tout, buf, col0 + c0, row0);
          bulk_commit_group();
        }
        ++*store_chunks;
        if (!row_ok) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int cc = c0 + 16 * h;
          if (cc >= n_valid) break;
          const int nv = min(16, n_valid - cc);
          const float* oo = &o[16 * h];
          if (tap) store_bf16_row(tap + cc, &v[16 * h], nv, id);
          if (e.out2)
            store_bf16_row(reinterpret_cast<__nv_bfloat16*>(e.out2) + (size_t)row * e.ldo + col0 + cc, oo, nv, id);
          if (e.norm_out) {
            // next RMSNorm, split: its gain here (the next GEMM's A), its 1/rms from the
            // row's sum of squares, applied in that GEMM's epilogue
            const __nv_bfloat16* gn = reinterpret_cast<const __nv_bfloat16*>(e.norm_gain) + col0 + cc;
            uint16_t* nd = reinterpret_cast<uint16_t*>(e.norm_out) + (size_t)row * e.ldo + col0 + cc;
            float og[16];
            if (nv == 16) {
              uint4 g2[2];
              g2[0] = reinterpret_cast<const uint4*>(gn)[0];
              g2[1] = reinterpret_cast<const uint4*>(gn)[1];
              const uint32_t* gw = reinterpret_cast<const uint32_t*>(g2);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float2 gf = unpack_bf16x2(gw[j]);
                ss_part += oo[2 * j] * oo[2 * j] + oo[2 * j + 1] * oo[2 * j + 1];
                og[2 * j] = oo[2 * j] * gf.x;
                og[2 * j + 1] = oo[2 * j + 1] * gf.y;
              }
              store16_2b(nd, og, e.norm_f16 != 0);
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if (j < nv) {
                  ss_part += oo[j] * oo[j];
                  const float g = oo[j] * __bfloat162float(gn[j]);
                  if (e.norm_f16) {
                    const __half hv = __float2half_rn(g);
                    nd[j] = *reinterpret_cast<const uint16_t*>(&hv);
                  } else {
                    const __nv_bfloat16 bv = __float2bfloat16_rn(g);
                    nd[j] = *reinterpret_cast<const uint16_t*>(&bv);
                  }
                }
              }
            }
          }
        }
      }
      resid_row_done<BN>(p, un, row, row_ok, ss_part);
      return;
    } else {
      const int col0 = p.b_out[un.b_seg] + un.b_row0;
      const int n_valid = p.b_rows[un.b_seg] - un.b_row0;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(e.out) + (size_t)row * e.ldo + col0;
      __nv_bfloat16* tap = nullptr;
      float r2 = 1.0f, ss_part = 0.f;
      if constexpr (EPI == (int)Epi::kResid) {
        if (e.tap) tap = reinterpret_cast<__nv_bfloat16*>(e.tap) + (size_t)row * e.ldo + col0;
      } else if constexpr (EPI == (int)Epi::kRelu2 || EPI == (int)Epi::kXielu) {
        r2 = row_norm_factor(e, row, row_ok);  // the post-attention RMSNorm's 1/rms
      }
      // kResid: the residual of the next 32 columns is loaded while this chunk is stored
      const size_t roff = (size_t)row * e.ldo + col0;
      float rnext[32];
      if constexpr (EPI == (int)Epi::kResid) load_resid32(e, roff, row_ok ? n_valid : 0, rnext);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float v[32];
        tmem_ld16(taddr + c0, *reinterpret_cast<float(*)[16]>(&v[0]));
        tmem_ld16(taddr + c0 + 16, *reinterpret_cast<float(*)[16]>(&v[16]));
        float rcur[32];
        if constexpr (EPI == (int)Epi::kResid) {
#pragma unroll
          for (int j = 0; j < 32; ++j) rcur[j] = rnext[j];
          if (c0 + 32 < BN) load_resid32(e, roff + c0 + 32, row_ok ? n_valid - c0 - 32 : 0, rnext);
        }
        tc_wait_ld();
        if (!row_ok || c0 >= n_valid) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int cc = c0 + 16 * h;
          if (cc >= n_valid) break;
          const int nv = min(16, n_valid - cc);
          float* vv = &v[16 * h];
          if constexpr (EPI == (int)Epi::kStore) {
            store_bf16_row(out + cc, vv, nv, [](float x, int) { return x; });
          } else if constexpr (EPI == (int)Epi::kRelu2) {
            store_bf16_row(out + cc, vv, nv, [=](float x, int) {
              const float r = fmaxf(x * r2, 0.0f);
              return r * r;
            });
          } else if constexpr (EPI == (int)Epi::kXielu) {
            const float ap = e.alpha_p, an = e.alpha_n, be = e.beta, xe = e.xeps;
            store_bf16_row(out + cc, vv, nv, [=](float x, int) {
              x *= r2;
              return x > 0.0f ? ap * x * x + be * x : an * (expm1_nonpos(fminf(x, xe)) - x) + be * x;
            });
          } else if constexpr (EPI == (int)Epi::kResid) {
            // residual stream carried in fp32: out = resid + acc, rounded once
            const float* rr = &rcur[16 * h];
            float o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = rr[j] + vv[j];
            auto id = [](float x, int) { return x; };
            if (tap) store_bf16_row(tap + cc, vv, nv, id);
            if (e.out_f32) {
              float* of = reinterpret_cast<float*>(e.out) + (size_t)row * e.ldo + col0 + cc;
              if (nv == 16) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  reinterpret_cast<float4*>(of)[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (j < nv) of[j] = o[j];
              }
            } else {
              store_bf16_row(out + cc, o, nv, id);
            }
            if (e.out2)
              store_bf16_row(reinterpret_cast<__nv_bfloat16*>(e.out2) + (size_t)row * e.ldo + col0 + cc, o, nv, id);
            if (e.norm_out) {
              // next RMSNorm, split: its gain here (out * g in bf16, the next GEMM's A), its
              // 1/rms from the row's sum of squares, applied in that GEMM's epilogue
              const __nv_bfloat16* gn = reinterpret_cast<const __nv_bfloat16*>(e.norm_gain) + col0 + cc;
              float og[16];
              uint16_t* nd = reinterpret_cast<uint16_t*>(e.norm_out) + (size_t)row * e.ldo + col0 + cc;
              if (nv == 16) {
                uint4 g2[2];
                g2[0] = reinterpret_cast<const uint4*>(gn)[0];
                g2[1] = reinterpret_cast<const uint4*>(gn)[1];
                const uint32_t* gw = reinterpret_cast<const uint32_t*>(g2);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float2 gf = unpack_bf16x2(gw[j]);
                  ss_part += o[2 * j] * o[2 * j] + o[2 * j + 1] * o[2 * j + 1];
                  og[2 * j] = o[2 * j] * gf.x;
                  og[2 * j + 1] = o[2 * j + 1] * gf.y;
                }
                store16_2b(nd, og, e.norm_f16 != 0);
              } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  if (j < nv) {
                    ss_part += o[j] * o[j];
                    const float v = o[j] * __bfloat162float(gn[j]);
                    if (e.norm_f16) {
                      const __half hv = __float2half_rn(v);
                      nd[j] = *reinterpret_cast<const uint16_t*>(&hv);
                    } else {
                      const __nv_bfloat16 bv = __float2bfloat16_rn(v);
                      nd[j] = *reinterpret_cast<const uint16_t*>(&bv);
                    }
                  }
                }
              }
            }
          }
        }
      }
      if constexpr (EPI == (int)Epi::kResid) {
        if (e.norm_ss && row_ok) e.norm_ss[(size_t)row * e.norm_parts + un.b_row0 / BN] = ss_part;
        // a prefill chunk appended to a KV cache: its sequence's length grows by seq, once
        if (e.bump_lens && row_ok && un.b_row0 == 0 && un.b_seg == 0 && row % e.seq == e.seq - 1)
          atomicAdd(e.bump_lens + row / e.seq, e.seq);
      }
    }
  }
}

// ------------------------------------------------------------------ decode finishers
//
// The decode GEMMs put the weights on the MMA's M side and the few tokens on N,
// and split K over CTAs so that the weight stream covers every SM. Each split
// stores its fp32 partial tile; the split that arrives last at the tile's
// counter sums the partials in split order (the result does not depend on which
// split that is) and applies the projection's post-op. Warp w of the epilogue
// finishes tokens 4w..4w+3, 16+4w.., and lane l holds the tile's features
// 4l..4l+3, so every per-token reduction or pairing is a warp shuffle.

__device__ __forceinline__ void st_bf16x4(__nv_bfloat16* dst, float a, float b, float c, float d) {
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
}

__device__ __forceinline__ float4 ld_bf16x4(const __nv_bfloat16* src) {
  const uint2 u = *reinterpret_cast<const uint2*>(src);
  const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y);
  return make_float4(a.x, a.y, b.x, b.y);
}

// Decode finisher, run by the four epilogue warps of every CTA of a tile's
// cluster (one CTA per K split, all resident together) after a cluster barrier:
// CTA r takes tokens [r * ceil(ntok / S), ...) of the tile; for each token it
// sums the S partials (distributed shared memory, in split order, so every
// token's result is the same whichever CTA finishes it) and applies the
// post-op. Warp w takes tokens lo + w + 4k (k = 0, 1, ...) of the slice, four
// per step; lane l holds the tile's features 4l .. 4l + 3, so per-token
// reductions and the RoPE pairing are warp shuffles.
//
// The per-token inputs of the first kDecPre tokens of each warp (positions and
// RoPE rows, or residual rows) and the gains are loaded into registers by
// dec_load_side while the MMA main loop still runs; the rest, if any, are loaded
// in the finish itself.
constexpr int kDecPre = 8;

struct DecSide {
  float4 a[kDecPre], b[kDecPre];  // kDecQkv: (cos, sin) of features 4l .. 4l + 3 (mod 64); kDecResid: residual (a)
  int pos[kDecPre];               // kDecQkv: lens of the token
  float4 gain;
};

struct DecSlice {
  int lo, hi, tok0;
};

__device__ __forceinline__ DecSlice dec_slice(const TcParams& p, const Unit& un, int bn) {
  const int S = p.k_splits;
  const int ntok = min(bn, p.e.n_tok - un.b_row0);
  const int per = (ntok + S - 1) / S;
  DecSlice sl;
  sl.lo = (int)cluster_ctarank() * per;
  sl.hi = min(ntok, sl.lo + per);
  sl.tok0 = un.b_row0;
  return sl;
}

// Inputs of token row tl (tl < ntok) for one lane: RoPE rows and position, or the residual row.
template <int EPI>
__device__ __forceinline__ void dec_token_inputs(const TcParams& p, const Unit& un, int tok0, int tl, int lane,
                                                 float4& a, float4& b, int& pos) {
  const TcEpiArgs& e = p.e;
  if constexpr (EPI == (int)Epi::kDecQkv) {
    pos = e.lens[tok0 + tl];
    if (un.a_seg < 2) {  // q and k take the rotary; v and the attention gate do not
      const int rpos = min(max(pos, 0), e.rope_max_pos - 1);
      const float4* cs4 = reinterpret_cast<const float4*>(e.rope + (size_t)rpos * 64 + 4 * (lane & 15));
      a = cs4[0];
      b = cs4[1];
    }
  } else {
    const int f = un.m_tile * kBM + 4 * lane;
    a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (f < e.ldo) {
      const size_t i = (size_t)(tok0 + tl) * e.ldo + f;
      if (e.resid_f32) {
        a = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(e.resid) + i);
      } else {
        const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(e.resid) + i);
        const float2 x = unpack_bf16x2(u.x), y = unpack_bf16x2(u.y);
        a = make_float4(x.x, x.y, y.x, y.y);
      }
    }
  }
}

template <int BN, int EPI>
__device__ __forceinline__ void dec_load_side(const TcParams& p, const Unit& un, int ew, int lane, DecSide& sd) {
  const TcEpiArgs& e = p.e;
  const DecSlice sl = dec_slice(p, un, BN);
  sd.gain = make_float4(1.f, 1.f, 1.f, 1.f);
  if constexpr (EPI == (int)Epi::kDecQkv) {
    if (un.a_seg < 2 && e.qk_norm)
      sd.gain = ld_bf16x4(reinterpret_cast<const __nv_bfloat16*>(un.a_seg == 0 ? e.q_gain : e.k_gain) + 4 * lane);
  } else {
    const int f = un.m_tile * kBM + 4 * lane;
    if (e.norm_out && f < e.ldo) sd.gain = ld_bf16x4(reinterpret_cast<const __nv_bfloat16*>(e.norm_gain) + f);
  }
  if (sl.hi <= sl.lo) return;
#pragma unroll
  for (int k = 0; k < kDecPre; ++k)  // rows clamped into the slice: every address is valid
    dec_token_inputs<EPI>(p, un, sl.tok0, min(sl.lo + ew + 4 * k, sl.hi - 1), lane, sd.a[k], sd.b[k], sd.pos[k]);
}

template <int BN, int EPI>
__device__ __forceinline__ void dec_finish(const TcParams& p, const Unit& un, int ew, int lane, const float* stage,
                                           const DecSide& sd) {
  const TcEpiArgs& e = p.e;
  constexpr bool qkv = EPI == (int)Epi::kDecQkv;
  const int S = p.k_splits;
  const DecSlice sl = dec_slice(p, un, BN);
  const int lo = sl.lo, hi = sl.hi, tok0 = sl.tok0;
  const bool rope = qkv && un.a_seg < 2;
  const int f0 = un.m_tile * kBM;                     // kDecResid: first feature of the tile
  const bool fok = qkv || f0 + 4 * lane < e.ldo;      // kDecResid: this lane's features exist
  const uint32_t stage_s = smem_u32(stage) + 16 * lane;
  const float4 gain = sd.gain;
  // one step: the warp's tokens k0 .. k0 + 3 (rows lo + ew + 4k below hi; tl clamped so every address is valid)
  auto step = [&](int k0, const int (&tl)[4], const float4 (&side0)[4], const float4 (&side1)[4],
                  const int (&pos)[4]) {
    // the splits' partials, in split order
    float v[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k][0] = v[k][1] = v[k][2] = v[k][3] = 0.f;
    for (int sp0 = 0; sp0 < S; sp0 += 4) {
      // up to four splits' loads in flight together (ranks clamped: a valid CTA), then added in order
      float4 a[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t base = map_shared_rank(stage_s, (uint32_t)min(sp0 + j, S - 1));
#pragma unroll
        for (int k = 0; k < 4; ++k) a[j][k] = ld_dsmem_f4(base + (uint32_t)tl[k] * (kBM * 4));
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (sp0 + j >= S) break;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[k][0] += a[j][k].x;
          v[k][1] += a[j][k].y;
          v[k][2] += a[j][k].z;
          v[k][3] += a[j][k].w;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (lo + ew + 4 * (k0 + k) >= hi) break;  // warp-uniform
      const int t = tok0 + tl[k];
      float* vv = v[k];
      if constexpr (qkv) {
        // one head (head_dim 128) per tile; token t is sequence t, at position lens[t]
        const int seg = un.a_seg;  // 0: q, 1: k, 2: v, 3: the attention gate
        const int head = un.a_row0 >> 7;
        if (seg == 3) {
          const float g0 = sigmoid_f(vv[0]), g1 = sigmoid_f(vv[1]), g2 = sigmoid_f(vv[2]), g3 = sigmoid_f(vv[3]);
          const __half2 h01 = __floats2half2_rn(g0, g1), h23 = __floats2half2_rn(g2, g3);
          *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(e.gate) + ((size_t)t * e.n_heads + head) * 128 +
                                    4 * lane) =
              make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
          continue;
        }
        const bool write = seg == 0 || (pos[k] >= 0 && pos[k] < e.kv_stride);  // never past a full cache
        if (rope) {
          if (e.qk_norm) {
            const float ss = warp_sum(vv[0] * vv[0] + vv[1] * vv[1] + vv[2] * vv[2] + vv[3] * vv[3]);
            const float r = rsqrtf(ss * (1.0f / 128.0f) + e.eps);
            vv[0] *= r * gain.x;
            vv[1] *= r * gain.y;
            vv[2] *= r * gain.z;
            vv[3] *= r * gain.w;
          }
          // RoPE, rotate-half pairing: feature i (lane l < 16) with i + 64 (lane l + 16)
          const float cs[4][2] = {{side0[k].x, side0[k].y}, {side0[k].z, side0[k].w},
                                  {side1[k].x, side1[k].y}, {side1[k].z, side1[k].w}};
          float pr[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) pr[c] = __shfl_xor_sync(0xffffffffu, vv[c], 16);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            vv[c] = lane < 16 ? vv[c] * cs[c][0] - pr[c] * cs[c][1] : vv[c] * cs[c][0] + pr[c] * cs[c][1];
        }
        if (write) {
          __nv_bfloat16* dst = seg == 0 ? reinterpret_cast<__nv_bfloat16*>(e.q) + ((size_t)t * e.n_heads + head) * 128
                                        : reinterpret_cast<__nv_bfloat16*>(seg == 1 ? e.k : e.v) +
                                              (((size_t)t * e.n_kv_heads + head) * e.kv_stride + pos[k]) * 128;
          st_bf16x4(dst + 4 * lane, vv[0], vv[1], vv[2], vv[3]);
        }
      } else {
        // the residual stream, summed in fp32 and rounded once
        const float4 r = side0[k];
        const float o0 = r.x + vv[0], o1 = r.y + vv[1], o2 = r.z + vv[2], o3 = r.w + vv[3];
        const size_t i = (size_t)t * e.ldo + f0 + 4 * lane;
        if (fok) {
          if (e.out_f32)
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out) + i) = make_float4(o0, o1, o2, o3);
          else
            st_bf16x4(reinterpret_cast<__nv_bfloat16*>(e.out) + i, o0, o1, o2, o3);
          if (e.out2) st_bf16x4(reinterpret_cast<__nv_bfloat16*>(e.out2) + i, o0, o1, o2, o3);
          if (e.tap) st_bf16x4(reinterpret_cast<__nv_bfloat16*>(e.tap) + i, vv[0], vv[1], vv[2], vv[3]);
          // next RMSNorm, split: out * g here (the MLP GEMM's B), 1/rms from the tiles' sums of squares later
          if (e.norm_out) {
            if (e.norm_f16) {  // the operand of an MLP GEMM on prepared fp16 weights
              const __half2 h01 = __floats2half2_rn(o0 * gain.x, o1 * gain.y);
              const __half2 h23 = __floats2half2_rn(o2 * gain.z, o3 * gain.w);
              *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(e.norm_out) + i) =
                  make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
            } else {
              st_bf16x4(reinterpret_cast<__nv_bfloat16*>(e.norm_out) + i, o0 * gain.x, o1 * gain.y, o2 * gain.z,
                        o3 * gain.w);
            }
          }
        }
        if (e.norm_ss) {
          const float ss = warp_sum(fok ? o0 * o0 + o1 * o1 + o2 * o2 + o3 * o3 : 0.f);
          if (lane == 0) e.norm_ss[(size_t)t * e.norm_parts + un.m_tile] = ss;
        }
        if (e.bump_lens && un.m_tile == 0 && lane == 0) atomicAdd(e.bump_lens + t, 1);  // no round trip
      }
    }
  };
  // tokens whose inputs were loaded during the main loop: compile-time indices, registers only
#pragma unroll
  for (int kb = 0; kb < kDecPre / 4; ++kb) {
    const int k0 = 4 * kb;
    if (lo + ew + 4 * k0 >= hi) break;  // warp-uniform
    int tl[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) tl[k] = min(lo + ew + 4 * (k0 + k), hi - 1);
    const float4 s0[4] = {sd.a[k0], sd.a[k0 + 1], sd.a[k0 + 2], sd.a[k0 + 3]};
    const float4 s1[4] = {sd.b[k0], sd.b[k0 + 1], sd.b[k0 + 2], sd.b[k0 + 3]};
    const int ps[4] = {sd.pos[k0], sd.pos[k0 + 1], sd.pos[k0 + 2], sd.pos[k0 + 3]};
    step(k0, tl, s0, s1, ps);
  }
  // the rest (tiles of more than 32 tokens per CTA), inputs loaded here
#pragma unroll 1
  for (int k0 = kDecPre; lo + ew + 4 * k0 < hi; k0 += 4) {
    int tl[4], ps[4];
    float4 s0[4], s1[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      tl[k] = min(lo + ew + 4 * (k0 + k), hi - 1);
      dec_token_inputs<EPI>(p, un, tok0, tl[k], lane, s0[k], s1[k], ps[k]);
    }
    step(k0, tl, s0, s1, ps);
  }
}

// kDecAct: CTA r of the cluster sums its token slice [lo, hi) of the tile over the
// splits' partial buffers (distributed shared memory, split order), multiplies by the
// tokens' 1/rms and applies the activation; 128 threads, four features a thread.
template <int BN>
__device__ __forceinline__ void dec_act_reduce(const TcParams& p, const Unit& un, uint32_t part_s, int tid,
                                               const float* rs_s, int lo, int hi) {
  const TcEpiArgs& e = p.e;
  const int S = p.k_splits;
  const bool paired = p.a_paired != 0;
  const int nf = paired ? kBM / 2 : kBM;  // output features of the tile
  const int tpt = nf / 4;                 // threads per token
  const int f_local = 4 * (tid % tpt);
  const int feat = un.m_tile * nf + f_local;
  const bool fok = feat < e.ldo;          // ldo = features (a multiple of 4)
  const uint32_t u_off = (uint32_t)(paired ? kBM / 2 + f_local : f_local) * 4, g_off = (uint32_t)f_local * 4;
  for (int t0 = lo; t0 < hi; t0 += kThreadsEpi / tpt) {
    const int tl = t0 + tid / tpt;
    const int tc = tl < hi ? tl : lo;  // clamped: every address is valid
    float4 ag[8], au[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < S) {
        const uint32_t base = map_shared_rank(part_s, (uint32_t)j) + (uint32_t)tc * (kBM * 4);
        au[j] = ld_dsmem_f4(base + u_off);
        ag[j] = paired ? ld_dsmem_f4(base + g_off) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < S) {
        u = make_float4(u.x + au[j].x, u.y + au[j].y, u.z + au[j].z, u.w + au[j].w);
        g = make_float4(g.x + ag[j].x, g.y + ag[j].y, g.z + ag[j].z, g.w + ag[j].w);
      }
    }
    if (tl >= hi || !fok) continue;
    const float rs = rs_s[tl - lo];
    float v[4] = {u.x * rs, u.y * rs, u.z * rs, u.w * rs};
    if (e.act == 0) {
      const float gg[4] = {g.x * rs, g.y * rs, g.z * rs, g.w * rs};
#pragma unroll
      for (int c = 0; c < 4; ++c) v[c] = silu_f(gg[c]) * v[c];
    } else if (e.act == 1) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float r = fmaxf(v[c], 0.0f);
        v[c] = r * r;
      }
    } else {
      const float ap = e.alpha_p, an = e.alpha_n, be = e.beta, xe = e.xeps;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float x = v[c];
        v[c] = x > 0.0f ? ap * x * x + be * x : an * (expm1_nonpos(fminf(x, xe)) - x) + be * x;
      }
    }
    st_bf16x4(reinterpret_cast<__nv_bfloat16*>(e.out) + (size_t)(un.b_row0 + tl) * e.ldo + feat, v[0], v[1], v[2],
              v[3]);
  }
}

// ------------------------------------------------------------------ the kernel

template <int BN, int EPI, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<BN, EPI, PAIR>;
  constexpr int S = C::kStages;
  // the prefill epilogues walk the banded tile order; the decode ones keep M fastest
  constexpr bool kGrp = !is_cluster_epi<EPI>() && EPI != (int)Epi::kPartialT;
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * C::kABytes;
  float* pb = reinterpret_cast<float*>(sB + S * C::kBBytes);  // kDecAct: partial buffers, then 1/rms
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S * C::kBBytes + C::kExtraBytes);
  // bars: full[S], empty[S], tfull[2], tempty[2], drain, pbfull[2], pbfree[2] (kDecAct)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * S + 9);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[S + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * S + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * S + 2 + a]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * S + 4]);
  auto pbfull_bar = [&](int b) { return smem_u32(&bars[2 * S + 5 + b]); };
  auto pbfree_bar = [&](int b) { return smem_u32(&bars[2 * S + 7 + b]); };
  // A CTA pair (cluster of 2): the even CTA issues the MMAs and owns the full and
  // tempty barriers both CTAs' copies and epilogues count on.
  const int prank = PAIR ? (int)(cluster_ctarank() & 1u) : 0;
  const bool mma_cta = prank == 0;
  const uint32_t lead_rank = PAIR ? (cluster_ctarank() & ~1u) : 0u;
  constexpr uint16_t kPairMask = 3;  // both CTAs of the (only) pair of the cluster
  const int u0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ustep = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), PAIR ? 8 : 128);  // a pair: one lane of each epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    if constexpr (EPI == (int)Epi::kDecAct)
      for (int b = 0; b < 2; ++b) {
        mbar_init(pbfull_bar(b), p.k_splits);  // one arrival from each split's CTA
        mbar_init(pbfree_bar(b), p.k_splits);
      }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.na; ++i) tma_prefetch_desc(&p.ta[i]);
    for (int i = 0; i < p.nb; ++i) tma_prefetch_desc(&p.tb[i]);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_holder), C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (EPI == (int)Epi::kDecAct || PAIR)
    cluster_sync_all();  // every CTA's barriers are initialised before any peer arrives on them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int bn_rows = p.b_paired ? BN / 2 : BN;
  const unsigned long long budget = p.wait_ns;
  DecSide dec_side;  // decode finishers only (epilogue warps)
  // What the producer and MMA lanes have in flight, for the drain after an abort:
  // the stages whose loads were issued (with the parity of their last phase), and
  // whether any MMA was issued.
  uint32_t issued_mask = 0, parity_mask = 0;
  unsigned long long last_issue_ns = 0;
  bool mma_issued = false;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t ph = 0;
      bool failed = false;
      // A streamed once (decode weights) must not push the activations that the
      // next kernels read out of L2
      const uint64_t a_policy = l2_policy_evict_first();
      // a pair: both CTAs' copies complete on the even CTA's full barrier
      auto full_tx = [&](int st) { return PAIR ? map_shared_rank(full_bar(st), lead_rank) : full_bar(st); };
      auto load_a = [&](int st, const Unit& un, int kb) {
        if constexpr (PAIR) {
          tma_load_2d_pair(smem_u32(sA + st * C::kABytes), &p.ta[0], kb * kBK, un.a_row0, full_tx(st));
          return;
        }
        if constexpr (EPI == (int)Epi::kPartialT || is_cluster_epi<EPI>()) {  // the decode GEMMs
          if (p.a_paired) {  // gate rows over up rows: two 64-row boxes make one 128-row swizzled tile
            const uint32_t dst = smem_u32(sA + st * C::kABytes);
            tma_load_2d_hint(dst, &p.ta[0], kb * kBK, un.a_row0, full_bar(st), a_policy);
            tma_load_2d_hint(dst + (kBM / 2) * kBK * 2, &p.ta[1], kb * kBK, un.a_row0, full_bar(st), a_policy);
            return;
          }
          if (p.a_once) {
            tma_load_2d_hint(smem_u32(sA + st * C::kABytes), &p.ta[un.a_seg], kb * kBK, un.a_row0, full_bar(st),
                             a_policy);
            return;
          }
        }
        tma_load_2d(smem_u32(sA + st * C::kABytes), &p.ta[un.a_seg], kb * kBK, un.a_row0, full_bar(st));
      };
      auto load_b = [&](int st, const Unit& un, int kb) {
        const uint32_t b_dst = smem_u32(sB + st * C::kBBytes);
        if constexpr (PAIR) {
          // the even CTA holds B's first N/2 rows, the odd one the rest: paired B
          // (gate | up) splits into its halves, a plain B tile into two row ranges
          if (p.b_paired)
            tma_load_2d_pair(b_dst, &p.tb[prank], kb * kBK, un.b_row0, full_tx(st));
          else
            tma_load_2d_pair(b_dst, &p.tb[un.b_seg], kb * kBK, un.b_row0 + prank * (BN / 2), full_tx(st));
          return;
        }
        if (p.b_paired) {
          tma_load_2d(b_dst, &p.tb[0], kb * kBK, un.b_row0, full_bar(st));
          tma_load_2d(b_dst + (BN / 2) * kBK * 2, &p.tb[1], kb * kBK, un.b_row0, full_bar(st));
        } else {
          tma_load_2d(b_dst, &p.tb[un.b_seg], kb * kBK, un.b_row0, full_bar(st));
        }
      };
      // The weights of the first unit's first stages are fetched while the
      // previous kernel finishes; the activations only after pdl_wait().
      // (a pair: the even CTA expects both CTAs' bytes)
      constexpr uint32_t kTxBytes = (PAIR ? 2 : 1) * C::kStageBytes;
      auto unit_of = [&](int u) { return PAIR ? pair_unit(p, u, bn_rows, prank) : decode_unit<kGrp>(p, u, bn_rows); };
      int pre = 0;
      if (p.const_op != 0 && u0 < p.num_units) {
        const Unit un = unit_of(u0);
        pre = min(S, un.kb_end - un.kb_begin);
        for (int i = 0; i < pre; ++i) {  // fresh ring: every stage is free
          if (mma_cta) mbar_arrive_expect_tx(full_bar(i), kTxBytes);
          if (p.const_op == 1)
            load_a(i, un, un.kb_begin + i);
          else
            load_b(i, un, un.kb_begin + i);
          issued_mask |= 1u << i;
          if constexpr (PAIR) last_issue_ns = globaltimer_ns();
        }
      }
      pdl_wait();
      int g = 0;  // k-blocks issued by this CTA
      for (int u = u0; u < p.num_units && !failed; u += ustep) {
        const Unit un = unit_of(u);
        for (int kb = un.kb_begin; kb < un.kb_end; ++kb, ++g) {
          if (g < pre) {  // the stage's constant half is already in flight
            if (p.const_op == 1)
              load_b(stage, un, kb);
            else
              load_a(stage, un, kb);
          } else {
            if (!mbar_wait(empty_bar(stage), ph ^ 1, budget, abort_flag)) {
              failed = true;
              break;
            }
            if (mma_cta) mbar_arrive_expect_tx(full_bar(stage), kTxBytes);
            load_a(stage, un, kb);
            load_b(stage, un, kb);
          }
          issued_mask |= 1u << stage;
          parity_mask = (parity_mask & ~(1u << stage)) | (ph << stage);
          if constexpr (PAIR) last_issue_ns = globaltimer_ns();
          if (++stage == S) {
            stage = 0;
            ph ^= 1;
          }
        }
      }
      if (failed) {  // the loads in flight are drained after the CTA's final barrier
        *abort_flag = 1;
        report_timeout(p.status, 0x10 + 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && mma_cta) {
      // ---------------- MMA issuer (a pair: the even CTA's, for both)
      // kind::f16 operand formats: bf16 (1) or fp16 (0) for A and B
      constexpr int kM = PAIR ? 2 * kBM : kBM;
      const uint32_t idesc = p.f16 ? (idesc_bf16_f32(kM, BN) & ~((7u << 7) | (7u << 10))) : idesc_bf16_f32(kM, BN);
      int stage = 0;
      uint32_t ph = 0;
      int it = 0;
      bool failed = false;
      for (int u = u0; u < p.num_units && !failed; u += ustep, ++it) {
        const Unit un = PAIR ? pair_unit(p, u, bn_rows, prank) : decode_unit<kGrp>(p, u, bn_rows);
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait(tempty_bar(acc), aph ^ 1, budget, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = un.kb_begin; kb < un.kb_end; ++kb) {
          if (!mbar_wait(full_bar(stage), ph, budget, abort_flag)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(smem_u32(sA + stage * C::kABytes));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + stage * C::kBBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // advance 16 elements (32 bytes) along K inside the swizzle atom
            if constexpr (PAIR)
              tc_mma_bf16_pair(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc,
                               (kb > un.kb_begin || kk > 0) ? 1u : 0u);
            else
              tc_mma_bf16(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc,
                          (kb > un.kb_begin || kk > 0) ? 1u : 0u);
          }
          mma_issued = true;
          if constexpr (PAIR)
            tc_commit_pair(empty_bar(stage), kPairMask);  // the stage is free in both CTAs
          else
            tc_commit(empty_bar(stage));
          if (++stage == S) {
            stage = 0;
            ph ^= 1;
          }
        }
        if (failed) break;
        if constexpr (PAIR)
          tc_commit_pair(tfull_bar(acc), kPairMask);  // both CTAs' halves of D are ready
        else
          tc_commit(tfull_bar(acc));
      }
      if (failed) {  // the MMAs in flight are drained after the CTA's final barrier
        *abort_flag = 1;
        report_timeout(p.status, 0x10 + 1);
      }
    }
  } else {
    // ---------------- epilogue warps 2..5: TMEM lane quarter = warp % 4
    pdl_wait();  // the epilogue reads and writes activations of earlier kernels
    if constexpr (is_dec_epi<EPI>())  // the finisher's per-token inputs, while the main loop runs
      dec_load_side<BN, EPI>(p, decode_unit(p, blockIdx.x, bn_rows), warp - 2, lane, dec_side);
    const int quarter = warp & 3;
    const int tid = threadIdx.x - 64;  // 0..127
    // kDecAct: this CTA's token slice and its tokens' 1/rms (the MLP input's RMSNorm, applied after the product)
    DecSlice act_sl{0, 0, 0};
    float* rs_s = pb + 2 * (C::kPartBytes / 4);
    if constexpr (EPI == (int)Epi::kDecAct) {
      act_sl = dec_slice(p, decode_unit(p, blockIdx.x, bn_rows), BN);
      const TcEpiArgs& e = p.e;
      for (int t = act_sl.lo + (warp - 2); t < act_sl.hi; t += 4) {
        float ss = 0.f;
        if (e.row_ss)
          for (int i = lane; i < e.ss_parts; i += 32) ss += e.row_ss[(size_t)(act_sl.tok0 + t) * e.ss_parts + i];
        ss = warp_sum(ss);
        if (lane == 0) rs_s[t - act_sl.lo] = e.row_ss ? rsqrtf(ss / (float)e.ss_n + e.ss_eps) : 1.0f;
      }
      named_bar_sync(1, kThreadsEpi);
    }
    int it = 0;
    bool failed = false;
    int store_chunks = 0;  // kResidTma: bulk stores issued by this warp
    for (int u = u0; u < p.num_units; u += ustep, ++it) {
      const Unit un = PAIR ? pair_unit(p, u, bn_rows, prank) : decode_unit<kGrp>(p, u, bn_rows);
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      if constexpr (EPI == (int)Epi::kDecAct) {
        // The four epilogue warps decide together (barrier-OR) whether to go on, so
        // that none is left alone at a named barrier after another gave up.
        float* part = pb + acc * (C::kPartBytes / 4);
        bool ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), aph, budget, abort_flag));
        // partial buffer acc is free once every split's CTA has read this CTA's tile it - 2 from it
        if (ok && it >= 2)
          ok = __all_sync(0xffffffffu,
                          mbar_wait_cluster(pbfree_bar(acc), ((it >> 1) - 1) & 1, budget, abort_flag));
        if (ok) {
          __syncwarp();
          tc_fence_after();
          run_epilogue<BN, EPI>(p, un, taddr, quarter * 32 + lane, part);
          tc_fence_before();
          mbar_arrive(tempty_bar(acc));
        }
        if (named_bar_or(1, kThreadsEpi, !ok)) {
          failed = true;
          break;
        }
        // hand the partial to the cluster: every split's CTA arrives on every CTA's pbfull
        // (lane r of the first epilogue warp on CTA r's: the arrivals travel in parallel)
        if (tid < p.k_splits) mbar_arrive_cluster(map_shared_rank(pbfull_bar(acc), (uint32_t)tid));
        ok = __all_sync(0xffffffffu, mbar_wait_cluster(pbfull_bar(acc), (it >> 1) & 1, budget, abort_flag));
        if (ok) dec_act_reduce<BN>(p, un, smem_u32(part), tid, rs_s, act_sl.lo, act_sl.hi);
        if (named_bar_or(1, kThreadsEpi, !ok)) {
          failed = true;
          break;
        }
        // this CTA has read every split's buffer acc: release them for tile it + 2
        if (tid < p.k_splits) mbar_arrive_cluster(map_shared_rank(pbfree_bar(acc), (uint32_t)tid));
      } else {
        if constexpr (is_resid<EPI>()) {  // this row's residual into L2 while the MMAs run
          const int row = un.m_tile * kBM + quarter * 32 + lane;
          if (row < p.a_rows[0])
            prefetch_resid_l2(p.e, (size_t)row * p.e.ldo + p.b_out[un.b_seg] + un.b_row0,
                              min(BN, p.b_rows[un.b_seg] - un.b_row0));
        }
        // warp-uniform: every lane waits, the warp gives up together
        if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), aph, budget, abort_flag))) {
          failed = true;
          break;
        }
        __syncwarp();
        tc_fence_after();
        if constexpr (EPI == (int)Epi::kResidTma)
          run_epilogue<BN, EPI>(p, un, taddr, quarter * 32 + lane, pb + (warp - 2) * 2048, &store_chunks);
        else if constexpr (swiglu_tma<BN, EPI>())
          run_epilogue<BN, EPI>(p, un, taddr, quarter * 32 + lane, pb + (warp - 2) * 512);
        else
          run_epilogue<BN, EPI>(p, un, taddr, quarter * 32 + lane, reinterpret_cast<float*>(smem));
        tc_fence_before();
        if constexpr (PAIR) {  // one lane a warp, on the even CTA's barrier
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(map_shared_rank(tempty_bar(acc), lead_rank));
        } else {
          mbar_arrive(tempty_bar(acc));
        }
      }
    }
    if (failed) {
      *abort_flag = 1;
      if (lane == 0) report_timeout(p.status, 0x10 + 2);
    }
    if constexpr (EPI == (int)Epi::kResidTma || swiglu_tma<BN, EPI>()) {
      // every bulk store of the warp complete (its shared-memory reads and its global writes)
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  }

  if constexpr (EPI == (int)Epi::kDecAct) {
    // no CTA leaves while another CTA of its cluster may still read its partial
    // buffers (every thread gets here: all earlier waits are bounded)
    __syncwarp();
    cluster_sync_all();
  }
  if constexpr (is_dec_epi<EPI>()) {
    // Every thread of every CTA of the cluster reaches both barriers, whatever
    // happened above (all earlier waits are bounded): the split partials are in
    // shared memory before the first, and no CTA exits while others may still
    // read its shared memory before the second.
    __syncwarp();
    cluster_sync_all();
    if (warp >= 2) dec_finish<BN, EPI>(p, decode_unit(p, blockIdx.x, bn_rows), warp - 2, lane,
                                       reinterpret_cast<const float*>(smem), dec_side);
    __syncwarp();
    cluster_sync_all();
  }
  tc_fence_before();
  if constexpr (PAIR) {
    // neither CTA of a pair leaves (or frees TMEM, a collective step) while the
    // other's copies or the pair's MMAs may still use its memory
    __syncwarp();
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  // Every role has stopped issuing. After an abort (a wait that ran out anywhere in
  // the CTA, or in either CTA of a pair) loads and MMAs that no role waited for may
  // still be in flight: they must complete before TMEM is freed and the CTA exits.
  // The decision is uniform: every thread reads the same flags after the barrier.
  bool aborted = *abort_flag != 0;
  if constexpr (PAIR)
    aborted = aborted || ld_dsmem_u32(map_shared_rank(smem_u32((const void*)abort_flag), cluster_ctarank() ^ 1u)) != 0;
  if (aborted) {
    volatile int never = 0;
    if (warp == 0 && lane == 0) {
      if (mma_cta) {
        // both CTAs' bytes of a pair complete on the even CTA's full barriers
        for (int s = 0; s < S; ++s)
          if (issued_mask & (1u << s)) mbar_wait(full_bar(s), (parity_mask >> s) & 1, kDrainNs, &never);
      } else if constexpr (PAIR) {
        // the odd CTA of a pair cannot watch its loads land (they count on the even
        // CTA's barriers, which cannot complete a phase the even CTA never armed): it
        // stays resident for kSettleNs after its last issue, far beyond a load's latency
        if (issued_mask != 0)
          while (globaltimer_ns() - last_issue_ns < kSettleNs) {
          }
      }
    }
    if (warp == 1 && lane == 0 && mma_cta && mma_issued) {
      if constexpr (PAIR)
        tc_commit_pair(drain_bar, (uint16_t)(1u << lead_rank));
      else
        tc_commit(drain_bar);
      mbar_wait(drain_bar, 0, kDrainNs, &never);
    }
    tc_fence_before();
    if constexpr (PAIR) {
      __syncwarp();
      cluster_sync_all();  // the pair's MMAs are done before either CTA frees its TMEM
    } else {
      __syncthreads();
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* ptr, int rows, int K, int box_rows, bool f16 = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

bool make_tma_2d_16b(CUtensorMap* m, const void* ptr, int rows, int cols, int box_rows, bool f16) {
  return make_map(m, ptr, rows, cols, box_rows, f16);
}

namespace {

template <int BN, int EPI, bool PAIR = false>
cudaError_t configure() {
  static std::atomic<unsigned long long> done{0};  // once per instantiation and device
  return set_smem_limit_once(reinterpret_cast<const void*>(tc_gemm_kernel<BN, EPI, PAIR>),
                             TcCfg<BN, EPI, PAIR>::kSmemBytes, done);
}

// Launch configuration of a clustered GEMM: clusters of `csize` CTAs along x
// (a decode GEMM's K splits, or a CTA pair).
template <int BN, int EPI, bool PAIR = false>
void cluster_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int grid, int csize, cudaStream_t s) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3(grid);
  cfg->blockDim = dim3(kThreads);
  cfg->dynamicSmemBytes = TcCfg<BN, EPI, PAIR>::kSmemBytes;
  cfg->stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 2;
}

template <int BN, int EPI, bool PAIR>
cudaError_t launch_one(const TcParams& p, int grid, cudaStream_t s) {
  cudaError_t e = configure<BN, EPI, PAIR>();
  if (e != cudaSuccess) return e;
  if constexpr (is_cluster_epi<EPI>() || PAIR) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    cluster_config<BN, EPI, PAIR>(&cfg, attr, grid, PAIR ? 2 : p.k_splits, s);
    e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<BN, EPI, PAIR>, p);
    if (e != cudaSuccess) return e;
  } else {
    launch_pdl(tc_gemm_kernel<BN, EPI, PAIR>, grid, kThreads, TcCfg<BN, EPI, PAIR>::kSmemBytes, s, p);
  }
  return cudaGetLastError();
}

template <int BN, int EPI>
int max_clusters(int splits) {
  if (configure<BN, EPI>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cluster_config<BN, EPI>(&cfg, attr, splits, splits, nullptr);
  cfg.numAttrs = 1;  // the cluster shape alone
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<BN, EPI, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// CTA-pair (M = 256) instantiations: the prefill epilogues, B halves of 96-128 rows.
template <int BN, int EPI>
constexpr bool tc_pair_supported() {
  if (EPI == (int)Epi::kQkv) return BN == 256;  // whole heads
  if (is_resid<EPI>() || EPI == (int)Epi::kSwiglu || EPI == (int)Epi::kRelu2 || EPI == (int)Epi::kXielu ||
      EPI == (int)Epi::kStore)
    return BN == 192 || BN == 224 || BN == 256;
  return false;
}

template <int BN, int EPI>
cudaError_t launch_if(const TcParams& p, bool pair, int grid, cudaStream_t s) {
  if (pair) {
    if constexpr (tc_pair_supported<BN, EPI>())
      return launch_one<BN, EPI, true>(p, grid, s);
    else
      return cudaErrorInvalidValue;
  }
  if constexpr (tc_supported<BN, EPI>())
    return launch_one<BN, EPI, false>(p, grid, s);
  else
    return cudaErrorInvalidValue;
}

template <int BN>
cudaError_t dispatch_epi(const TcParams& p, Epi epi, bool pair, int grid, cudaStream_t s) {
  switch (epi) {
    case Epi::kStore: return launch_if<BN, (int)Epi::kStore>(p, pair, grid, s);
    case Epi::kResid: return launch_if<BN, (int)Epi::kResid>(p, pair, grid, s);
    case Epi::kResidTma: return launch_if<BN, (int)Epi::kResidTma>(p, pair, grid, s);
    case Epi::kQkv: return launch_if<BN, (int)Epi::kQkv>(p, pair, grid, s);
    case Epi::kSwiglu: return launch_if<BN, (int)Epi::kSwiglu>(p, pair, grid, s);
    case Epi::kRelu2: return launch_if<BN, (int)Epi::kRelu2>(p, pair, grid, s);
    case Epi::kXielu: return launch_if<BN, (int)Epi::kXielu>(p, pair, grid, s);
    case Epi::kPartialT: return launch_if<BN, (int)Epi::kPartialT>(p, pair, grid, s);
    case Epi::kDecQkv: return launch_if<BN, (int)Epi::kDecQkv>(p, pair, grid, s);
    case Epi::kDecResid: return launch_if<BN, (int)Epi::kDecResid>(p, pair, grid, s);
    case Epi::kDecAct: return launch_if<BN, (int)Epi::kDecAct>(p, pair, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int tc_dec_max_clusters(int bn, Epi epi, int splits) {
  if (splits < 1 || splits > 8) return 0;
  static std::mutex mu;
  static int cache[5][3][9] = {};  // bn index, epilogue, splits (0: not queried yet)
  const int bi = bn == 64 ? 0 : bn == 128 ? 1 : bn == 256 ? 2 : -1;
  const int ei = epi == Epi::kDecQkv ? 0 : epi == Epi::kDecResid ? 1 : epi == Epi::kDecAct ? 2 : -1;
  if (bi < 0 || ei < 0 || (ei == 2 && bn != 64)) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[bi][ei][splits];
  if (c == 0) {
    int n = 0;
    if (ei == 2)
      n = max_clusters<64, (int)Epi::kDecAct>(splits);
    else if (bn == 64)
      n = ei == 0 ? max_clusters<64, (int)Epi::kDecQkv>(splits) : max_clusters<64, (int)Epi::kDecResid>(splits);
    if (bn == 128)
      n = ei == 0 ? max_clusters<128, (int)Epi::kDecQkv>(splits) : max_clusters<128, (int)Epi::kDecResid>(splits);
    if (bn == 256)
      n = ei == 0 ? max_clusters<256, (int)Epi::kDecQkv>(splits) : max_clusters<256, (int)Epi::kDecResid>(splits);
    c = n > 0 ? n : -1;
  }
  return c > 0 ? c : 0;
}

namespace {
bool is_dec(Epi e) { return e == Epi::kDecQkv || e == Epi::kDecResid || e == Epi::kDecAct; }
}  // namespace

cudaError_t launch_tc_gemm(const TcGemmDesc& d, int max_ctas, DevStatus* st, unsigned long long wait_ns,
                           cudaStream_t s, const char** why) {
  TcParams p;
  memset(static_cast<void*>(&p), 0, sizeof(p));
  const int bn_rows = d.b_paired ? d.bn / 2 : d.bn;
  if (d.bn != 64 && d.bn != 128 && d.bn != 192 && d.bn != 224 && d.bn != 256) {
    *why = "tcgen05 GEMM: BN must be 64, 128, 192, 224 or 256";
    return cudaErrorInvalidValue;
  }
  if (d.K <= 0 || d.K % 8 != 0) {
    *why = "tcgen05 GEMM: K must be a positive multiple of 8 (16-byte rows)";
    return cudaErrorInvalidValue;
  }
  if (d.na < 1 || d.na > kMaxSegs || d.nb < 1 || d.nb > kMaxSegs || (d.b_paired && d.nb != 2)) {
    *why = "tcgen05 GEMM: bad segment count";
    return cudaErrorInvalidValue;
  }
  p.na = d.na;
  p.nb = d.nb;
  if (d.a_paired && (d.epi != Epi::kDecAct || d.na != 2 || d.a[0].rows != d.a[1].rows)) {
    *why = "tcgen05 GEMM: paired A operands are two equal segments of a decode activation GEMM";
    return cudaErrorInvalidValue;
  }
  const int a_box = d.a_paired ? kBM / 2 : kBM;
  p.a_tiles[0] = 0;
  for (int i = 0; i < d.na; ++i) {
    if (!make_map(&p.ta[i], d.a[i].ptr, d.a[i].rows, d.K, a_box, d.f16)) {
      *why = "cuTensorMapEncodeTiled failed for an A operand";
      return cudaErrorInvalidValue;
    }
    p.a_rows[i] = d.a[i].rows;
    p.a_out[i] = d.a[i].out_offset;
    // paired: one tile sequence over both segments (rows of a[0] and a[1] side by side)
    p.a_tiles[i + 1] = d.a_paired ? (d.a[0].rows + a_box - 1) / a_box : p.a_tiles[i] + (d.a[i].rows + kBM - 1) / kBM;
  }
  p.a_paired = d.a_paired ? 1 : 0;
  if (d.pair && (is_dec(d.epi) || d.epi == Epi::kPartialT || d.k_splits > 1 || d.na != 1 || d.a_paired ||
                 max_ctas < 2)) {
    *why = "tcgen05 GEMM: a CTA pair runs a prefill GEMM (one A segment, no K split)";
    return cudaErrorInvalidValue;
  }
  // a pair's CTA loads half of the B tile: BN / 2 rows (a paired B's half is one segment's tile)
  const int b_box = d.pair ? d.bn / 2 : bn_rows;
  p.b_tiles[0] = 0;
  for (int i = 0; i < d.nb; ++i) {
    if (!make_map(&p.tb[i], d.b[i].ptr, d.b[i].rows, d.K, b_box, d.f16)) {
      *why = "cuTensorMapEncodeTiled failed for a B operand";
      return cudaErrorInvalidValue;
    }
    p.b_rows[i] = d.b[i].rows;
    p.b_out[i] = d.b[i].out_offset;
    p.b_tiles[i + 1] = p.b_tiles[i] + (d.b[i].rows + bn_rows - 1) / bn_rows;
  }
  p.b_paired = d.b_paired ? 1 : 0;
  p.f16 = d.f16 ? 1 : 0;
  p.const_op = d.const_op;
  p.m_tiles = d.pair ? (d.a[0].rows + 2 * kBM - 1) / (2 * kBM) : p.a_tiles[d.na];  // a pair: 256-row tiles
  p.n_tiles = d.b_paired ? (d.b[0].rows + bn_rows - 1) / bn_rows : p.b_tiles[d.nb];
  p.num_kb = (d.K + kBK - 1) / kBK;
  p.k_splits = d.k_splits < 1 ? 1 : (d.k_splits > p.num_kb ? p.num_kb : d.k_splits);
  p.num_units = p.m_tiles * p.n_tiles * p.k_splits;
  p.a_once = d.const_op == 1 && p.n_tiles == 1;
  if (d.epi == Epi::kDecAct) {
    // persistent clusters of the K splits: the grid (max_ctas) is whole clusters; one N tile
    if (d.nb != 1 || d.b_paired || d.e.n_tok != d.b[0].rows || p.n_tiles != 1 || p.k_splits > 8 ||
        d.k_splits != p.k_splits || max_ctas < p.k_splits || max_ctas % p.k_splits != 0 || d.e.ldo % 4 != 0 ||
        d.e.ldo != d.a[0].rows || d.na != (d.a_paired ? 2 : 1)) {
      *why = "tcgen05 GEMM: a decode activation GEMM needs one N tile, whole clusters of at most 8 K splits";
      return cudaErrorInvalidValue;
    }
  }
  if (d.epi == Epi::kDecQkv || d.epi == Epi::kDecResid) {
    // one unit per CTA, the K splits of a tile forming one cluster (at most 8), all resident at once
    if (d.nb != 1 || d.b_paired || d.e.n_tok != d.b[0].rows || p.k_splits > 8 || p.num_units > max_ctas ||
        tc_dec_max_clusters(d.bn, d.epi, p.k_splits) < p.m_tiles * p.n_tiles) {
      *why = "tcgen05 GEMM: a decode finisher needs one unit per CTA and every cluster of K splits resident";
      return cudaErrorInvalidValue;
    }
  }
  if (d.epi == Epi::kResidTma) {
    // the fp32 output [rows, ldo] as a tensor of 32 x 32 boxes: one B segment covering its columns
    auto fn = encode_fn();
    if (d.nb != 1 || d.b_paired || d.na != 1 || !d.e.out_f32 || !d.e.out || d.b[0].out_offset != 0 ||
        d.b[0].rows != d.e.ldo || d.e.ldo % 4 != 0 || (reinterpret_cast<uintptr_t>(d.e.out) & 15) || !fn) {
      *why = "tcgen05 GEMM: a TMA-stored residual output is fp32, one B segment as wide as the output";
      return cudaErrorInvalidValue;
    }
    cuuint64_t dims[2] = {(cuuint64_t)d.e.ldo, (cuuint64_t)d.a[0].rows};
    cuuint64_t strides[1] = {(cuuint64_t)d.e.ldo * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&p.tout, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, d.e.out, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "cuTensorMapEncodeTiled failed for the residual output";
      return cudaErrorInvalidValue;
    }
  }
  if (d.epi == Epi::kSwiglu && d.bn == 256) {
    // the 256-wide SwiGLU's bf16 output [rows, ldo] as a tensor of 32 x 32 boxes
    auto fn = encode_fn();
    if (!d.b_paired || d.nb != 2 || d.na != 1 || !d.e.out || d.b[0].rows != d.e.ldo || d.e.ldo % 8 != 0 ||
        (reinterpret_cast<uintptr_t>(d.e.out) & 15) || !fn) {
      *why = "tcgen05 GEMM: a SwiGLU output is paired gate/up segments as wide as the output";
      return cudaErrorInvalidValue;
    }
    cuuint64_t dims[2] = {(cuuint64_t)d.e.ldo, (cuuint64_t)d.a[0].rows};
    cuuint64_t strides[1] = {(cuuint64_t)d.e.ldo * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&p.tout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d.e.out, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "cuTensorMapEncodeTiled failed for the SwiGLU output";
      return cudaErrorInvalidValue;
    }
  }
  p.e = d.e;
  p.status = st;
  p.wait_ns = wait_ns;
  if (p.num_units == 0) return cudaSuccess;
  // a pair: two CTAs per unit, whole pairs
  const int grid = d.pair ? 2 * std::min(p.num_units, max_ctas / 2) : std::min(p.num_units, max_ctas);
  // Prefill GEMMs (one unit per tile) walk bands of group_m M tiles: the units in flight
  // at once (one per CTA or pair) then form a patch of about sqrt(units * BN / tile rows)
  // M tiles by the rest in N, so that the A and B blocks a round reads are about equal in
  // bytes. Decode GEMMs keep M fastest (their clusters and splits assume it).
  p.group_m = 1;
  if (p.k_splits == 1 && d.epi != Epi::kPartialT && d.epi != Epi::kDecQkv && d.epi != Epi::kDecResid &&
      d.epi != Epi::kDecAct) {
    const int in_flight = d.pair ? grid / 2 : grid;
    const double rows = d.pair ? 2.0 * kBM : (double)kBM;
    const int gm = (int)std::lround(std::sqrt(in_flight * (double)d.bn / rows));
    p.group_m = std::max(1, std::min(gm, p.m_tiles));
  }
  cudaError_t e;
  switch (d.bn) {
    case 64: e = dispatch_epi<64>(p, d.epi, d.pair, grid, s); break;
    case 128: e = dispatch_epi<128>(p, d.epi, d.pair, grid, s); break;
    case 192: e = dispatch_epi<192>(p, d.epi, d.pair, grid, s); break;
    case 224: e = dispatch_epi<224>(p, d.epi, d.pair, grid, s); break;
    default: e = dispatch_epi<256>(p, d.epi, d.pair, grid, s); break;
  }
  if (e == cudaErrorInvalidValue && !*why) *why = "tcgen05 GEMM: tile width not built for this epilogue";
  return e;
}

}  // namespace blk
