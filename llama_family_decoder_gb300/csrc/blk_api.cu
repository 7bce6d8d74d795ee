// Host library behind the C ABI in include/blk.h: descriptor validation,
// caller-owned workspace layout, and the launch sequence of the decoder block
// ("LlamaForCausalLM-32L-4096d" sheet, "Implementing it"; nnterp "arcee" and
// "apertus", "The block, in order").
//
// bf16 prefill:  rmsnorm -> tcgen05 QKV GEMM (+q/k norm, RoPE, head scatter)
//                -> flash attention -> tcgen05 o_proj (+residual) -> rmsnorm
//                -> tcgen05 up/gate GEMM (+activation) -> tcgen05 down (+residual)
// bf16 decode:   rmsnorm -> weight-streaming tcgen05 GEMMs (tokens on N,
//                split-K partials) with post kernels (q/k norm + RoPE + cache
//                append; residual + next rmsnorm; activation) and split-KV
//                attention.
// fp32 path:     the same sequence on SIMT fp32 GEMMs and fp32 attention.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/blk.h"
#include "common.cuh"
#include "kernels.h"

using namespace blk;

// Per-stage event timing of blk_forward (blk_profile_*).
struct StageProfile {
  static constexpr int kMax = 24;
  bool on = false;
  bool pending = false;
  int n = 0;
  const char* names[kMax] = {};
  int launches[kMax] = {};
  cudaEvent_t ev[kMax + 1] = {};
  double total_ms[kMax] = {};
  long long total_launches[kMax] = {};
};

struct blk_handle {
  blk_desc d;
  int device;
  int num_sms;
  float2* rope;        // [max_seq][head_dim/2] (cos, sin) as fp32, from double
  DevStatus* status;   // device
  int* dev_flag;       // device int: weight-range check of blk_prepare_weights
  StageProfile prof;
};

// Status word of the debug GEMM entry point (it runs without a handle).
static __device__ DevStatus g_debug_status;

namespace {

thread_local std::string g_err;
std::atomic<long long> g_wait_ns{2000000000LL};

// Device address of g_debug_status on the current device (host code cannot use
// the symbol itself as a device pointer).
cudaError_t debug_status_address(DevStatus** out) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_debug_status);
}

blk_status fail(blk_status s, const std::string& msg) {
  g_err = msg;
  return s;
}

blk_status cuda_fail(cudaError_t e, const char* where, const char* why = nullptr) {
  std::string m = std::string(where) + ": " + cudaGetErrorString(e);
  if (why) m += std::string(" (") + why + ")";
  return fail(BLK_ERR_CUDA, m);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t esize(const blk_desc& d) { return d.dtype == BLK_BF16 ? 2 : 4; }

// Bump allocator over the caller's workspace (or a size counter when base is null).
struct Carve {
  uint8_t* base;
  size_t off = 0;
  explicit Carve(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    off = (off + 255) & ~size_t(255);
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

// fp16 copies of the weights the prefill's fp16 GEMMs read (blk_prepare_weights).
struct Prepared {
  const void *wo, *wg, *wu;
  const void *wq, *wk, *wv, *wag;  // the Q/K/V projection and the attention gate
};

size_t prepared_layout(const blk_desc& d, const void* base, Prepared* out) {
  Carve c(const_cast<void*>(base));
  Prepared p{};
  const size_t Hd = (size_t)d.n_heads * d.head_dim, KVd = (size_t)d.n_kv_heads * d.head_dim;
  p.wo = c.take((size_t)d.hidden * Hd * 2);
  if (d.act == BLK_ACT_SWIGLU) p.wg = c.take((size_t)d.ffn * d.hidden * 2);
  p.wu = c.take((size_t)d.ffn * d.hidden * 2);
  p.wq = c.take(Hd * d.hidden * 2);
  p.wk = c.take(KVd * d.hidden * 2);
  p.wv = c.take(KVd * d.hidden * 2);
  if (d.attn_gate) p.wag = c.take(Hd * d.hidden * 2);
  if (out) *out = p;
  return c.off;
}

// Columns of the fused Q/K/V (and attention gate) projection.
int qkv_cols(const blk_desc& d) { return (d.n_heads * (d.attn_gate ? 2 : 1) + 2 * d.n_kv_heads) * d.head_dim; }
int mlp_cols(const blk_desc& d) { return d.act == BLK_ACT_SWIGLU ? 2 * d.ffn : d.ffn; }
int max_cols(const blk_desc& d) {
  int n = qkv_cols(d);
  if (d.hidden > n) n = d.hidden;
  if (mlp_cols(d) > n) n = mlp_cols(d);
  return n;
}

constexpr int kMaxDecodeSplits = 16;

// Decode GEMMs: weight tiles of 128 rows, token tiles of 64, 128 or 256.
int dec_bn(int B) { return B <= 64 ? 64 : (B <= 128 ? 128 : 256); }
int dec_tiles_qkv(const blk_desc& d) {
  return (d.attn_gate ? 2 : 1) * ((d.n_heads * d.head_dim + 127) / 128) + 2 * ((d.n_kv_heads * d.head_dim + 127) / 128);
}

// Tile of a prefill GEMM: one CTA per 128-row tile, or (pair) a CTA pair per
// 256-row tile, each CTA loading half of the B tile (a third less operand traffic
// per MMA than one CTA with the same width, which the measured per-SM TMA feed
// rate caps). The fewest waves of tiles, weighted by each form's per-tile rate.
struct TileChoice {
  int bn;
  bool pair;
};
constexpr double kPairRate = 1.12;  // a pair tile's MMA rate over a single CTA's at BN >= 192
// Pairs pay off when a tile's main loop is long against its epilogue and the
// accumulator hand-off across the pair: K >= 2048 (measured: Llama-7B, Arcee and
// Apertus shapes 6-8% faster per block; at K = 1024 slower). The SwiGLU MLP-up
// GEMM already runs at the sustained MMA rate with one CTA per tile.
constexpr int kPairMinK = 2048;

TileChoice choose_tile(int m_rows, int n_cols, bool paired, const int* cands, int ncand, int num_sms,
                       bool allow_pair) {
  TileChoice best{cands[0], false};
  double best_cost = 1e30;
  for (int pr = 0; pr < (allow_pair && num_sms >= 2 ? 2 : 1); ++pr)
    for (int i = 0; i < ncand; ++i) {
      const int bn = cands[i];
      if (pr && bn < 192) continue;
      const int cols = paired ? bn / 2 : bn;
      const int rows = pr ? 256 : 128;
      const int slots = pr ? num_sms / 2 : num_sms;
      const long long tiles = (long long)((m_rows + rows - 1) / rows) * ((n_cols + cols - 1) / cols);
      const long long waves = (tiles + slots - 1) / slots;
      const double eff = (bn >= 256 ? 1.0 : bn >= 224 ? 0.99 : bn >= 192 ? 0.90 : 0.88) * (pr ? kPairRate : 1.0);
      const double cost = (double)waves * cols / eff;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = {bn, pr != 0};
      }
    }
  return best;
}

// N-tile width for a GEMM with m_rows rows and n_cols output columns (per half
// when paired): the fewest waves of tiles over the SMs, weighted by each width's
// per-tile efficiency (narrower tiles re-read A more often).
int choose_bn(int m_rows, int n_cols, bool paired, const int* cands, int ncand, int num_sms) {
  return choose_tile(m_rows, n_cols, paired, cands, ncand, num_sms, false).bn;
}

// Tile of the residual GEMMs (o_proj, down) for `rows` rows of hidden outputs.
TileChoice resid_tile(const blk_handle* h, int rows, int n, int K) {
  static const int c[] = {256, 224, 192, 128};
  return choose_tile(rows, n, false, c, 4, h->num_sms, K >= kPairMinK);
}
int resid_bn(const blk_handle* h, int rows, int n, int K) { return resid_tile(h, rows, n, K).bn; }

// Partial sums of squares per row that the o_proj epilogue leaves for the MLP's
// norm: one per o_proj N-tile (at most hidden / 128 of them).
int norm_parts(int hidden, int bn) { return (hidden + bn - 1) / bn; }

// Workspace regions of a forward call.
struct Ws {
  void *y, *q, *k, *v, *o, *mid, *neur, *C, *attn;
  float *rs1, *ss2;  // bf16: input-norm 1/rms per row (prefill); post-attention partial sums of squares
  void* gate;        // attn_gate: sigmoid of the gate projection, o's layout (fp16; fp32 on the fp32 path)
  int2* ranges;      // prefill with an attention_mask: each sequence's run of real tokens [lo, hi)
  int* pos0;         // ... and its rotary offset -lo
};

Ws carve_forward(const blk_handle* h, void* base, int B, int T, bool decode, size_t* total) {
  const blk_desc& d = h->d;
  const size_t es = esize(d);
  const size_t M = (size_t)B * T;
  Carve c(base);
  Ws w{};
  w.y = c.take(M * d.hidden * es);
  w.q = c.take(M * d.n_heads * d.head_dim * es);
  if (!decode) {
    w.k = c.take(M * d.n_kv_heads * d.head_dim * es);
    w.v = c.take(M * d.n_kv_heads * d.head_dim * es);
  }
  w.o = c.take(M * d.n_heads * d.head_dim * es);
  w.mid = c.take(M * d.hidden * sizeof(float));  // the residual stream after attention, kept in fp32
  w.neur = c.take(M * d.ffn * es);
  if (decode) {
    if (d.dtype == BLK_BF16) {
      w.C = c.take((size_t)kMaxDecodeSplits * M * max_cols(d) * sizeof(float));
      const int s = attn_decode_split_cap(d.max_seq);
      w.attn = c.take(attn_decode_ws_bytes(B, d.n_heads, d.head_dim, s));
      w.ss2 = static_cast<float*>(c.take(M * norm_parts(d.hidden, 128) * sizeof(float)));
    } else {
      w.C = c.take(M * max_cols(d) * sizeof(float));
    }
  } else if (d.dtype == BLK_F32) {
    w.C = c.take(M * max_cols(d) * sizeof(float));
  } else {
    w.rs1 = static_cast<float*>(c.take(M * sizeof(float)));
    w.ss2 = static_cast<float*>(c.take(M * norm_parts(d.hidden, 128) * sizeof(float)));
    if (d.sandwich_norm) w.C = c.take(M * d.hidden * sizeof(float));  // a sublayer's output before its post-norm
  }
  if (d.attn_gate) w.gate = c.take(M * d.n_heads * d.head_dim * (d.dtype == BLK_BF16 ? 2 : 4));
  if (!decode) {
    w.ranges = static_cast<int2*>(c.take((size_t)B * sizeof(int2)));
    w.pos0 = static_cast<int*>(c.take((size_t)B * sizeof(int)));
  }
  *total = c.off;
  return w;
}

// Split count for a weight-streaming GEMM: balance the work units over the SMs
// (units = tiles x splits), charging each extra split for its partial-sum traffic.
int choose_splits(int tiles, int num_kb, int num_sms) {
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= kMaxDecodeSplits && s <= num_kb / 4 + (s == 1); ++s) {
    const double units = (double)tiles * s;
    const double waves = std::ceil(units / num_sms);
    const double cost = waves * num_sms / units + 0.03 * s;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

TcEpiArgs qkv_epi(const blk_handle* h, const blk_weights* w, int seq, const int* pos0, void* q, void* k, void* v) {
  const blk_desc& d = h->d;
  TcEpiArgs e;
  e.q = q;
  e.k = k;
  e.v = v;
  e.seq = seq;
  e.n_heads = d.n_heads;
  e.n_kv_heads = d.n_kv_heads;
  e.head_dim = d.head_dim;
  e.kv_stride = seq;
  e.q_gain = w->q_norm_g;
  e.k_gain = w->k_norm_g;
  e.eps = d.eps;
  e.rope = h->rope;
  e.rope_max_pos = d.max_seq;
  e.pos0 = pos0;
  e.qk_norm = d.qk_norm;
  return e;
}

// ------------------------------------------------------------------ bf16 prefill pieces

blk_status tc(const blk_handle* h, const TcGemmDesc& g, cudaStream_t s, const char* what) {
  const char* why = nullptr;
  cudaError_t e = launch_tc_gemm(g, h->num_sms, h->status, (unsigned long long)g_wait_ns.load(), s, &why);
  if (e != cudaSuccess) return cuda_fail(e, what, why);
  return BLK_OK;
}

// cache_stride > 0: k and v are a KV cache of cache_stride rows per (sequence, KV head),
// written at rows pos0[b] + t.
// gate != null: the attention gate projection joins as a 4th segment; its sigmoid goes to gate (fp16).
// f16: q/k/v stored as fp16; prep: the GEMM runs on the prepared fp16 weights (y is then fp16).
blk_status bf16_qkv(const blk_handle* h, const void* y, const blk_weights* w, int B, int T, const int* pos0, void* q,
                    void* k, void* v, cudaStream_t s, const float* row_scale = nullptr, bool f16 = false,
                    int cache_stride = 0, void* gate = nullptr, const Prepared* prep = nullptr) {
  const blk_desc& d = h->d;
  TcGemmDesc g;
  g.na = 1;
  g.a[0] = {y, B * T, 0};
  g.nb = 3;
  g.b[0] = {prep ? prep->wq : w->wq, d.n_heads * d.head_dim, 0};
  g.b[1] = {prep ? prep->wk : w->wk, d.n_kv_heads * d.head_dim, d.n_heads * d.head_dim};
  g.b[2] = {prep ? prep->wv : w->wv, d.n_kv_heads * d.head_dim, (d.n_heads + d.n_kv_heads) * d.head_dim};
  if (gate) {
    g.nb = 4;
    g.b[3] = {prep ? prep->wag : w->w_attn_gate, d.n_heads * d.head_dim, (d.n_heads + 2 * d.n_kv_heads) * d.head_dim};
  }
  g.f16 = prep != nullptr;
  g.K = d.hidden;
  const bool whole256 = (d.n_heads * d.head_dim) % 256 == 0 && (d.n_kv_heads * d.head_dim) % 256 == 0;
  static const int qkv_c[] = {256, 128};
  const TileChoice tq = whole256 ? choose_tile(B * T, qkv_cols(d), false, qkv_c, 2, h->num_sms,
                                             d.hidden >= kPairMinK)
                                 : TileChoice{128, false};
  g.bn = tq.bn;
  g.pair = tq.pair;
  g.epi = Epi::kQkv;
  g.const_op = 2;
  g.e = qkv_epi(h, w, T, pos0, q, k, v);
  if (cache_stride > 0) {
    g.e.kv_stride = cache_stride;
    g.e.kv_at_pos = 1;
  }
  g.e.row_scale = row_scale;
  g.e.qkv_f16 = f16 ? 1 : 0;
  g.e.gate = gate;
  return tc(h, g, s, "QKV GEMM");
}

blk_status bf16_linear_resid(const blk_handle* h, const void* a, int rows, int K, const void* W, int N,
                             const void* resid, bool resid_f32, void* out, bool out_f32, void* out2, void* tap,
                             cudaStream_t s, const char* what, void* norm_out = nullptr,
                             const void* norm_gain = nullptr, float* norm_ss = nullptr, bool f16 = false,
                             int* bump_lens = nullptr, int seq = 0) {
  TcGemmDesc g;
  g.na = 1;
  g.a[0] = {a, rows, 0};
  g.nb = 1;
  g.b[0] = {W, N, 0};
  g.K = K;
  const TileChoice tr = resid_tile(h, rows, N, K);
  g.bn = tr.bn;
  g.pair = tr.pair;
  // o_proj (the fp32 residual stream plus the next norm's rows) stores its fp32 output
  // through shared memory with TMA; the others store from registers
  g.epi = out_f32 ? Epi::kResidTma : Epi::kResid;
  g.const_op = 2;
  g.e.out = out;
  g.e.ldo = N;
  g.e.resid = resid;
  g.e.resid_f32 = resid_f32 ? 1 : 0;
  g.e.out_f32 = out_f32 ? 1 : 0;
  g.e.out2 = out2;
  g.e.tap = tap;
  g.e.norm_out = norm_out;
  g.e.norm_gain = norm_gain;
  g.e.norm_ss = norm_ss;
  g.e.norm_parts = norm_parts(N, g.bn);
  g.e.norm_f16 = f16 ? 1 : 0;  // the MLP-up GEMM that reads norm_out has the same operand type
  g.e.bump_lens = bump_lens;    // lens[b] += seq after the block (a prefill chunk appended to a cache)
  g.e.seq = seq;
  g.f16 = f16;
  return tc(h, g, s, what);
}

blk_status bf16_mlp_up(const blk_handle* h, const void* y2, int rows, const blk_weights* w, void* neur,
                       cudaStream_t s, const float* row_ss = nullptr, int ss_parts = 0,
                       const Prepared* prep = nullptr) {
  const blk_desc& d = h->d;
  TcGemmDesc g;
  g.e.row_ss = row_ss;  // set: y2 rows are un-normalised (gain applied); 1/rms from their sum of squares
  g.e.ss_parts = ss_parts;
  g.e.ss_n = d.hidden;
  g.e.ss_eps = d.eps;
  g.na = 1;
  g.a[0] = {y2, rows, 0};
  g.K = d.hidden;
  static const int act_c[] = {256, 224, 192, 128};
  const TileChoice ta = choose_tile(rows, d.ffn, d.act == BLK_ACT_SWIGLU, act_c, 4, h->num_sms,
                                    d.hidden >= kPairMinK && d.act != BLK_ACT_SWIGLU);
  g.bn = ta.bn;
  g.pair = ta.pair;
  g.e.out = neur;
  g.e.ldo = d.ffn;
  if (d.act == BLK_ACT_SWIGLU) {
    g.nb = 2;
    g.b_paired = true;
    g.b[0] = {prep ? prep->wg : w->w_gate, d.ffn, 0};
    g.b[1] = {prep ? prep->wu : w->w_up, d.ffn, 0};
    g.epi = Epi::kSwiglu;
  } else {
    g.nb = 1;
    g.b[0] = {prep ? prep->wu : w->w_up, d.ffn, 0};
    g.epi = d.act == BLK_ACT_RELU2 ? Epi::kRelu2 : Epi::kXielu;
    g.e.alpha_p = d.xielu_alpha_p;
    g.e.alpha_n = d.xielu_alpha_n;
    g.e.beta = d.xielu_beta;
    g.e.xeps = d.xielu_eps;
  }
  g.f16 = prep != nullptr;
  g.const_op = 2;
  return tc(h, g, s, "MLP up GEMM");
}

// ------------------------------------------------------------------ decode pieces (bf16)

// Split count of a fused decode GEMM (the K splits of a tile form one cluster):
// every CTA resident at once (units <= SMs, all clusters resident), at most 8
// splits; 0 when no split count fits.
int dec_fused_splits(const blk_handle* h, int tiles, int num_kb, int B, Epi epi) {
  const int bn = dec_bn(B);
  const int units1 = tiles * ((B + bn - 1) / bn);
  if (units1 > h->num_sms) return 0;
  int sp = std::min({choose_splits(units1, num_kb, h->num_sms), 8, h->num_sms / units1, std::max(num_kb, 1)});
  for (; sp >= 1; --sp)
    if (tc_dec_max_clusters(bn, epi, sp) >= units1) return sp;
  return 0;
}

// Cluster size of the decode MLP-up + activation GEMM (kDecAct): persistent clusters
// of S K-splits walk the tiles (64 gate over 64 up features when paired, else 128 up
// features). A tile's epilogue (the partials' hand-off and the activation, about
// 3.4 us) overlaps the next tile's weight stream, so a CTA takes about
//   t_unit + (rounds - 1) * max(t_unit, t_epi) + t_epi,
// t_unit = its 128 x K/S weight bytes at min(55 GB/s, 7 TB/s / active CTAs).
// 0 when the form does not apply (more than 64 tokens, a width not a multiple of
// 4, no cluster fits).
int dec_act_splits(const blk_handle* h, int B, int* clusters_out) {
  const blk_desc& d = h->d;
  if (dec_bn(B) != 64 || d.ffn % 4 != 0) return 0;
  const bool paired = d.act == BLK_ACT_SWIGLU;
  const int tiles = paired ? (d.ffn + 63) / 64 : (d.ffn + 127) / 128;
  const int num_kb = (d.hidden + 63) / 64;
  constexpr double kCtaBw = 55e9, kHbmBw = 7.0e12, kEpi = 3.4e-6;
  int best = 0, best_nc = 0;
  double best_t = 1e30;
  for (int sp = 1; sp <= 8 && sp <= num_kb; ++sp) {
    const int nc = std::min(tiles, tc_dec_max_clusters(64, Epi::kDecAct, sp));
    if (nc <= 0) continue;
    const int rounds = (tiles + nc - 1) / nc;
    const double bw = std::min(kCtaBw, kHbmBw / (nc * sp));
    const double t_unit = 128.0 * 64.0 * ((num_kb + sp - 1) / sp) * 2.0 / bw;
    const double t = t_unit + (rounds - 1) * std::max(t_unit, kEpi) + kEpi;
    if (t < best_t * 0.99) {
      best_t = t;
      best = sp;
      best_nc = nc;
    }
  }
  *clusters_out = best_nc;
  return best;
}

// The decode MLP up GEMM with its activation (kDecAct): neurons[B, F] (bf16) from the
// MLP input rows y; row_ss: the o_proj epilogue's per-tile sums of squares (1/rms
// applied after the product), or null when y is already normalised.
blk_status dec_act_gemm(const blk_handle* h, const blk_weights* w, const Prepared& prep, bool f16, const void* y,
                        int B, int splits, int clusters, const float* row_ss, int parts, void* neur, cudaStream_t s) {
  const blk_desc& d = h->d;
  TcGemmDesc g;
  g.f16 = f16;
  if (d.act == BLK_ACT_SWIGLU) {
    g.na = 2;
    g.a[0] = {f16 ? prep.wg : w->w_gate, d.ffn, 0};
    g.a[1] = {f16 ? prep.wu : w->w_up, d.ffn, 0};
    g.a_paired = true;
  } else {
    g.na = 1;
    g.a[0] = {f16 ? prep.wu : w->w_up, d.ffn, 0};
  }
  g.nb = 1;
  g.b[0] = {y, B, 0};
  g.K = d.hidden;
  g.bn = 64;
  g.k_splits = splits;
  g.epi = Epi::kDecAct;
  g.const_op = 1;  // A = the weights
  g.e.out = neur;
  g.e.ldo = d.ffn;
  g.e.n_tok = B;
  g.e.act = (int)d.act;
  g.e.alpha_p = d.xielu_alpha_p;
  g.e.alpha_n = d.xielu_alpha_n;
  g.e.beta = d.xielu_beta;
  g.e.xeps = d.xielu_eps;
  g.e.row_ss = row_ss;
  g.e.ss_parts = parts;
  g.e.ss_n = d.hidden;
  g.e.ss_eps = d.eps;
  const char* why = nullptr;
  cudaError_t e = launch_tc_gemm(g, clusters * splits, h->status, (unsigned long long)g_wait_ns.load(), s, &why);
  if (e != cudaSuccess) return cuda_fail(e, "decode MLP-up GEMM with activation", why);
  return BLK_OK;
}

// A fused decode GEMM: the weight segments on the MMA's M side, the B tokens of x
// on N, each tile's K splits one cluster that finishes the tile's post-op.
// f16: fp16 weights (prepared) and x.
blk_status dec_gemm(const blk_handle* h, const TcSeg* segs, int nseg, const void* x, int B, int K, int splits,
                    Epi epi, TcEpiArgs e, cudaStream_t s, const char* what, bool f16 = false) {
  TcGemmDesc g;
  g.f16 = f16;
  g.na = nseg;
  for (int i = 0; i < nseg; ++i) g.a[i] = segs[i];
  g.nb = 1;
  g.b[0] = {x, B, 0};
  g.K = K;
  g.bn = dec_bn(B);
  g.k_splits = splits;
  g.epi = epi;
  g.const_op = 1;  // A = the weights
  e.n_tok = B;
  g.e = e;
  return tc(h, g, s, what);
}

// The unfused form: transposed split-K partials [split][token][column], summed by a post kernel.
blk_status bf16_stream_gemm(const blk_handle* h, const TcSeg* segs, int nseg, const void* x, int B, int K, float* C,
                            int ldc, int* splits_out, cudaStream_t s, const char* what, bool f16 = false) {
  TcGemmDesc g;
  g.f16 = f16;
  g.na = nseg;
  int tiles = 0;
  for (int i = 0; i < nseg; ++i) {
    g.a[i] = segs[i];
    tiles += (segs[i].rows + 127) / 128;
  }
  g.nb = 1;
  g.b[0] = {x, B, 0};
  g.K = K;
  g.bn = dec_bn(B);
  const int n_tiles = (B + g.bn - 1) / g.bn;
  g.k_splits = choose_splits(tiles * n_tiles, (K + 63) / 64, h->num_sms);
  g.epi = Epi::kPartialT;
  g.const_op = 1;  // A = the weight segments
  g.e.out = C;
  g.e.part_ld = ldc;
  g.e.n_tok = B;
  *splits_out = g.k_splits;
  return tc(h, g, s, what);
}

void prof_mark(blk_handle* h, const char* name, int launches, cudaStream_t s) {
  StageProfile& p = h->prof;
  if (!p.on || p.n >= StageProfile::kMax) return;
  // External: under stream capture this becomes an event-record node of the graph
  cudaEventRecordWithFlags(p.ev[p.n], s, cudaEventRecordExternal);
  p.names[p.n] = name;
  p.launches[p.n] = launches;
  ++p.n;
}

void prof_begin(blk_handle* h) {
  if (h->prof.on) h->prof.n = 0;
}

void prof_end(blk_handle* h, cudaStream_t s) {
  StageProfile& p = h->prof;
  if (!p.on || p.n == 0) return;
  cudaEventRecordWithFlags(p.ev[p.n], s, cudaEventRecordExternal);
  p.pending = true;
}

blk_status check_cuda(cudaError_t e, const char* where, const char* why = nullptr) {
  return e == cudaSuccess ? BLK_OK : cuda_fail(e, where, why);
}

#define BLK_TRY(expr)                  \
  do {                                 \
    blk_status st_ = (expr);           \
    if (st_ != BLK_OK) return st_;     \
  } while (0)

template <typename P>
P tap_or(const blk_taps* t, P blk_taps::*m, P dflt) {
  return (t && t->*m) ? t->*m : dflt;
}

// ------------------------------------------------------------------ forward variants

// cache != null: a prefill chunk. The T new tokens of sequence b sit at positions
// lens[b] .. lens[b] + T - 1, append their K/V to the cache and attend to it.
// mask != null (no cache): a padded batch, attention_mask [B, T] (zeros are padding).
blk_status forward_prefill_bf16(blk_handle* h, const void* x, int B, int T, const blk_weights* w, void* out,
                                const Ws& ws, const blk_taps* taps, cudaStream_t s, blk_kv_cache* cache = nullptr,
                                const int* mask = nullptr) {
  // Both RMSNorms are split around the GEMMs they feed: the gain multiplies the
  // GEMM's A rows (x * g1 is x itself when g1 == 1), the per-row 1/rms multiplies
  // the accumulator in the epilogue. q/k/v and P are kept in fp16 (3 more
  // mantissa bits than bf16 at the same tensor-core rate); o and the neurons,
  // which meet bf16 weights, stay bf16. With the sandwich norms, o_proj and down
  // write their fp32 outputs and a row kernel applies the post-norm, the residual
  // add and (after o_proj) the MLP's input norm.
  const blk_desc& d = h->d;
  const int M = B * T;
  const bool gated = d.attn_gate != 0, sandwich = d.sandwich_norm != 0;
  void* head_tap = taps ? taps->attention_head_outputs : nullptr;
  void* o = (head_tap && !gated) ? head_tap : ws.o;
  void* mid_tap = taps ? taps->layer_mid : nullptr;
  void* neur = tap_or(taps, &blk_taps::mlp_neurons, ws.neur);
  // with prepared (fp16) weights the o_proj and MLP-up operands are fp16: 3 more
  // mantissa bits than bf16 at the same tensor-core rate. On a sandwich block, whose
  // post-norms scale each sublayer's relative error up to the size of the residual
  // stream, the Q/K/V operand is fp16 too: the input norm then writes normalized
  // rows (within fp16's range), which waits for each row's reduction; plain blocks
  // keep the split norm (x * g1 in bf16 written in the same pass, 1/rms in the QKV
  // epilogue), a few microseconds faster at the Llama-7B shape.
  Prepared prep{};
  const bool f16 = w->prepared != nullptr;
  if (f16) prepared_layout(d, w->prepared, &prep);
  const bool qkv16 = f16 && sandwich;
  if (mask) {  // each sequence's run of real tokens: hidden padding keys, positions from the run's start
    prof_mark(h, "mask_ranges", 1, s);
    BLK_TRY(check_cuda(launch_mask_ranges(mask, B, T, ws.ranges, ws.pos0, h->status, s), "attention mask"));
  }
  prof_mark(h, "norm1_prep", 1, s);
  if (qkv16)
    BLK_TRY(check_cuda(launch_rmsnorm(x, w->ln1_g, M, d.hidden, d.eps, ws.y, true, s, false, true), "input norm"));
  else
    BLK_TRY(check_cuda(launch_norm_prep(x, w->ln1_g, M, d.hidden, d.eps, ws.y, ws.rs1, nullptr, s), "input norm"));
  const float* rs1 = qkv16 ? nullptr : ws.rs1;
  const Prepared* qprep = qkv16 ? &prep : nullptr;
  prof_mark(h, "qkv_gemm_rope", 1, s);
  void* gate = gated ? ws.gate : nullptr;
  if (cache) {
    // bf16 q (the cache's K/V are bf16, so the attention runs on bf16 operands); K/V into the cache
    BLK_TRY(bf16_qkv(h, ws.y, w, B, T, cache->lens, tap_or(taps, &blk_taps::attention_queries, ws.q), cache->k,
                     cache->v, s, rs1, false, cache->capacity, gate, qprep));
  } else {
    BLK_TRY(bf16_qkv(h, ws.y, w, B, T, mask ? ws.pos0 : nullptr, ws.q, ws.k, ws.v, s, rs1, true, 0, gate, qprep));
  }
  if (taps && !cache) {  // the taps are bf16
    const size_t nq = (size_t)M * d.n_heads * d.head_dim, nkv = (size_t)M * d.n_kv_heads * d.head_dim;
    if (taps->attention_queries)
      BLK_TRY(check_cuda(launch_cast_f16_bf16(ws.q, taps->attention_queries, nq, s), "q tap"));
    if (taps->attention_keys) BLK_TRY(check_cuda(launch_cast_f16_bf16(ws.k, taps->attention_keys, nkv, s), "k tap"));
    if (taps->attention_values)
      BLK_TRY(check_cuda(launch_cast_f16_bf16(ws.v, taps->attention_values, nkv, s), "v tap"));
  }
  void* o_buf = f16 ? ws.o : o;
  AttnOpts opt;
  opt.window = d.sliding_window;
  opt.gate = gate;
  opt.ungated = gated ? head_tap : nullptr;  // the tap reads the heads before the gate
  opt.key_range = mask ? ws.ranges : nullptr;
  prof_mark(h, "attention", 1, s);
  const char* why = nullptr;
  cudaError_t e =
      cache ? launch_attn_prefill_tc(tap_or(taps, &blk_taps::attention_queries, ws.q), cache->k, cache->v, o_buf, B,
                                     d.n_heads, d.n_kv_heads, T, d.head_dim, false, f16, h->status,
                                     (unsigned long long)g_wait_ns.load(), s, &why, cache->lens, cache->capacity, opt)
            : launch_attn_prefill_tc(ws.q, ws.k, ws.v, o_buf, B, d.n_heads, d.n_kv_heads, T, d.head_dim, true, f16,
                                     h->status, (unsigned long long)g_wait_ns.load(), s, &why, nullptr, 0, opt);
  BLK_TRY(check_cuda(e, "attention", why));
  if (f16 && head_tap && !gated)
    BLK_TRY(check_cuda(launch_cast_f16_bf16(o_buf, head_tap, (size_t)M * d.n_heads * d.head_dim, s),
                       "head-output tap"));
  const int Hd = d.n_heads * d.head_dim;
  if (sandwich) {
    prof_mark(h, "o_proj_gemm", 1, s);
    BLK_TRY(bf16_linear_resid(h, o_buf, M, Hd, f16 ? prep.wo : w->wo, d.hidden, nullptr, false, ws.C, true, nullptr,
                              nullptr, s, "o_proj GEMM", nullptr, nullptr, nullptr, f16));
    prof_mark(h, "post_attn_norm_resid_norm2", 1, s);
    BLK_TRY(check_cuda(launch_post_resid(static_cast<float*>(ws.C), 1, M, d.hidden, d.hidden, x, false, ws.mid, true,
                                         mid_tap, taps ? taps->attention_output : nullptr, w->ln2_g, d.eps, ws.y,
                                         nullptr, true, s, w->post_attn_g, f16),
                       "post-attention norm"));
    prof_mark(h, "mlp_up_gemm_act", 1, s);
    BLK_TRY(bf16_mlp_up(h, ws.y, M, w, neur, s, nullptr, 0, f16 ? &prep : nullptr));
    prof_mark(h, "down_gemm", 1, s);
    BLK_TRY(bf16_linear_resid(h, neur, M, d.ffn, w->w_down, d.hidden, nullptr, false, ws.C, true, nullptr, nullptr, s,
                              "down GEMM", nullptr, nullptr, nullptr, false, cache ? cache->lens : nullptr, T));
    prof_mark(h, "post_mlp_norm_resid", 1, s);
    BLK_TRY(check_cuda(launch_post_resid(static_cast<float*>(ws.C), 1, M, d.hidden, d.hidden, ws.mid, true, out,
                                         false, nullptr, taps ? taps->mlp_output : nullptr, nullptr, d.eps, nullptr,
                                         nullptr, true, s, w->post_mlp_g),
                       "post-MLP norm"));
    prof_end(h, s);
    return BLK_OK;
  }
  prof_mark(h, "o_proj_gemm_resid_norm2", 1, s);
  BLK_TRY(bf16_linear_resid(h, o_buf, M, Hd, f16 ? prep.wo : w->wo, d.hidden, x, false, ws.mid, true, mid_tap,
                            taps ? taps->attention_output : nullptr, s, "o_proj GEMM", ws.y, w->ln2_g, ws.ss2, f16));
  prof_mark(h, "mlp_up_gemm_act", 1, s);
  BLK_TRY(bf16_mlp_up(h, ws.y, M, w, neur, s, ws.ss2, norm_parts(d.hidden, resid_bn(h, M, d.hidden, d.n_heads * d.head_dim)),
                      f16 ? &prep : nullptr));
  prof_mark(h, "down_gemm_resid", 1, s);
  BLK_TRY(bf16_linear_resid(h, neur, M, d.ffn, w->w_down, d.hidden, ws.mid, true, out, false, nullptr,
                            taps ? taps->mlp_output : nullptr, s, "down GEMM", nullptr, nullptr, nullptr, false,
                            cache ? cache->lens : nullptr, T));
  prof_end(h, s);
  return BLK_OK;
}

blk_status forward_decode_bf16(blk_handle* h, const void* x, int B, const blk_weights* w, blk_kv_cache* cache,
                               int max_len, void* out, const Ws& ws, const blk_taps* taps, cudaStream_t s) {
  const blk_desc& d = h->d;
  const bool bf = true;
  const int Hd = d.n_heads * d.head_dim, KVd = d.n_kv_heads * d.head_dim;
  const int parts = norm_parts(d.hidden, 128);
  float* C = static_cast<float*>(ws.C);
  const bool gated = d.attn_gate != 0, sandwich = d.sandwich_norm != 0;
  // prepared (fp16) weights: the normed rows, the attention output and the MLP's input are fp16 operands
  Prepared prep{};
  const bool f16 = w->prepared != nullptr;
  if (f16) prepared_layout(d, w->prepared, &prep);
  void* q = tap_or(taps, &blk_taps::attention_queries, ws.q);
  void* head_tap = taps ? taps->attention_head_outputs : nullptr;
  void* o = (head_tap && !gated && !f16) ? head_tap : ws.o;
  void* mid_tap = taps ? taps->layer_mid : nullptr;
  void* neur = tap_or(taps, &blk_taps::mlp_neurons, ws.neur);
  // QKV, o_proj and down finish their tiles inside the GEMM when every unit fits
  // on the SMs at once; otherwise (and for the MLP-up GEMM, whose tiles outnumber
  // the SMs) a post kernel sums the split partials. A sandwich post-norm needs the
  // whole row, so o_proj and down then always take the post kernel.
  const int hid_tiles = (d.hidden + 127) / 128;
  const int s_qkv = dec_fused_splits(h, dec_tiles_qkv(d), (d.hidden + 63) / 64, B, Epi::kDecQkv);
  const int s_o = sandwich ? 0 : dec_fused_splits(h, hid_tiles, (Hd + 63) / 64, B, Epi::kDecResid);
  const int s_down = sandwich ? 0 : dec_fused_splits(h, hid_tiles, (d.ffn + 63) / 64, B, Epi::kDecResid);
  void* gate = gated ? ws.gate : nullptr;
  int sp = 1;
  prof_mark(h, "rmsnorm1", 1, s);
  // (it also zeroes the attention's unit counter, at the start of its workspace)
  BLK_TRY(check_cuda(launch_rmsnorm(x, w->ln1_g, B, d.hidden, d.eps, ws.y, bf, s, false, f16,
                                    static_cast<int*>(ws.attn)),
                     "rmsnorm 1"));
  prof_mark(h, "qkv_gemm_rope_append", s_qkv ? 1 : 2, s);
  {
    const TcSeg segs[4] = {{f16 ? prep.wq : w->wq, Hd, 0},
                           {f16 ? prep.wk : w->wk, KVd, Hd},
                           {f16 ? prep.wv : w->wv, KVd, Hd + KVd},
                           {f16 ? prep.wag : w->w_attn_gate, Hd, Hd + 2 * KVd}};
    const int nseg = gated ? 4 : 3;
    if (s_qkv) {
      TcEpiArgs e;
      e.q = q;
      e.k = cache->k;
      e.v = cache->v;
      e.n_heads = d.n_heads;
      e.n_kv_heads = d.n_kv_heads;
      e.head_dim = d.head_dim;
      e.kv_stride = cache->capacity;
      e.q_gain = w->q_norm_g;
      e.k_gain = w->k_norm_g;
      e.eps = d.eps;
      e.rope = h->rope;
      e.rope_max_pos = d.max_seq;
      e.qk_norm = d.qk_norm;
      e.lens = cache->lens;
      e.gate = gate;
      BLK_TRY(dec_gemm(h, segs, nseg, ws.y, B, d.hidden, s_qkv, Epi::kDecQkv, e, s, "decode QKV GEMM", f16));
    } else {
      BLK_TRY(bf16_stream_gemm(h, segs, nseg, ws.y, B, d.hidden, C, qkv_cols(d), &sp, s, "decode QKV GEMM", f16));
      BLK_TRY(check_cuda(launch_post_qkv(C, sp, B, qkv_cols(d), 1, nullptr, cache->lens, d.n_heads, d.n_kv_heads,
                                         d.head_dim, d.qk_norm, w->q_norm_g, w->k_norm_g, d.eps, h->rope,
                                         d.max_seq, q, cache->k, cache->v, cache->capacity, bf, s, gate),
                         "decode qkv post"));
    }
  }
  prof_mark(h, "attention_splitkv", 2, s);
  const char* why = nullptr;
  AttnOpts opt;
  opt.window = d.sliding_window;
  opt.gate = gate;
  opt.ungated = (gated || f16) ? head_tap : nullptr;  // the tap: bf16, before the gate
  opt.o_f16 = f16;
  opt.counter_zeroed = true;  // by the input norm above
  cudaError_t ce = launch_attn_decode_bf16(q, cache->k, cache->v, o, B, d.n_heads, d.n_kv_heads, d.head_dim,
                                           cache->capacity, cache->lens, 1, max_len,
                                           attn_decode_split_cap(d.max_seq), ws.attn,
                                           h->num_sms, h->status, (unsigned long long)g_wait_ns.load(), s, &why, opt);
  BLK_TRY(check_cuda(ce, "decode attention", why));
  prof_mark(h, "o_proj_gemm_resid_norm2", s_o ? 1 : 2, s);
  {
    const TcSeg segs[1] = {{f16 ? prep.wo : w->wo, d.hidden, 0}};
    if (s_o) {
      // mid = x + o Wo^T (fp32), and the post-attention RMSNorm split: ws.y = mid * g2,
      // ws.ss2 = per-tile sums of squares (the activation kernel applies 1/rms)
      TcEpiArgs e;
      e.out = ws.mid;
      e.out_f32 = 1;
      e.ldo = d.hidden;
      e.resid = x;
      e.out2 = mid_tap;
      e.tap = taps ? taps->attention_output : nullptr;
      e.norm_out = ws.y;
      e.norm_gain = w->ln2_g;
      e.norm_ss = ws.ss2;
      e.norm_parts = parts;
      e.norm_f16 = f16 ? 1 : 0;
      BLK_TRY(dec_gemm(h, segs, 1, o, B, Hd, s_o, Epi::kDecResid, e, s, "decode o_proj GEMM", f16));
    } else {
      BLK_TRY(bf16_stream_gemm(h, segs, 1, o, B, Hd, C, d.hidden, &sp, s, "decode o_proj GEMM", f16));
      BLK_TRY(check_cuda(launch_post_resid(C, sp, B, d.hidden, d.hidden, x, false, ws.mid, true, mid_tap,
                                           taps ? taps->attention_output : nullptr, w->ln2_g, d.eps, ws.y, nullptr,
                                           bf, s, sandwich ? w->post_attn_g : nullptr, f16),
                         "decode o_proj post"));
    }
  }
  int act_clusters = 0;
  const int s_act = dec_act_splits(h, B, &act_clusters);
  if (s_act) {
    // the activation inside the GEMM: the splits of each tile meet in a cluster's shared memory
    prof_mark(h, "mlp_up_gemm_act", 1, s);
    BLK_TRY(dec_act_gemm(h, w, prep, f16, ws.y, B, s_act, act_clusters, s_o ? ws.ss2 : nullptr, parts, neur, s));
  } else {
    prof_mark(h, "mlp_up_gemm", 1, s);
    if (d.act == BLK_ACT_SWIGLU) {
      const TcSeg segs[2] = {{f16 ? prep.wg : w->w_gate, d.ffn, 0}, {f16 ? prep.wu : w->w_up, d.ffn, d.ffn}};
      BLK_TRY(bf16_stream_gemm(h, segs, 2, ws.y, B, d.hidden, C, 2 * d.ffn, &sp, s, "decode gate/up GEMM", f16));
    } else {
      const TcSeg segs[1] = {{f16 ? prep.wu : w->w_up, d.ffn, 0}};
      BLK_TRY(bf16_stream_gemm(h, segs, 1, ws.y, B, d.hidden, C, d.ffn, &sp, s, "decode up GEMM", f16));
    }
    prof_mark(h, "mlp_act", 1, s);
    BLK_TRY(check_cuda(launch_post_act(C, sp, B, d.ffn, mlp_cols(d), (int)d.act, d.xielu_alpha_p, d.xielu_alpha_n,
                                       d.xielu_beta, d.xielu_eps, neur, bf, s, s_o ? ws.ss2 : nullptr, parts,
                                       d.hidden, d.eps),
                       "decode activation"));
  }
  prof_mark(h, "down_gemm_resid", s_down ? 1 : 2, s);
  {
    const TcSeg segs[1] = {{w->w_down, d.hidden, 0}};
    if (s_down) {
      TcEpiArgs e;
      e.out = out;
      e.ldo = d.hidden;
      e.resid = ws.mid;
      e.resid_f32 = 1;
      e.tap = taps ? taps->mlp_output : nullptr;
      e.bump_lens = cache->lens;
      BLK_TRY(dec_gemm(h, segs, 1, neur, B, d.ffn, s_down, Epi::kDecResid, e, s, "decode down GEMM"));
    } else {
      BLK_TRY(bf16_stream_gemm(h, segs, 1, neur, B, d.ffn, C, d.hidden, &sp, s, "decode down GEMM"));
      BLK_TRY(check_cuda(launch_post_resid(C, sp, B, d.hidden, d.hidden, ws.mid, true, out, false, nullptr,
                                           taps ? taps->mlp_output : nullptr, nullptr, d.eps, nullptr, cache->lens,
                                           bf, s, sandwich ? w->post_mlp_g : nullptr),
                         "decode down post"));
    }
  }
  prof_end(h, s);
  return BLK_OK;
}

// fp32 path: prefill (cache == null) or decode (cache != null, T == 1).
blk_status forward_f32(blk_handle* h, const void* x, int B, int T, const blk_weights* w, blk_kv_cache* cache,
                       void* out, const Ws& ws, const blk_taps* taps, cudaStream_t s, const int* mask = nullptr) {
  const blk_desc& d = h->d;
  const bool bf = false;
  const int M = B * T;
  const int Hd = d.n_heads * d.head_dim, KVd = d.n_kv_heads * d.head_dim;
  float* C = static_cast<float*>(ws.C);
  const bool decode = cache != nullptr;
  void* q = tap_or(taps, &blk_taps::attention_queries, ws.q);
  void* k = decode ? cache->k : tap_or(taps, &blk_taps::attention_keys, ws.k);
  void* v = decode ? cache->v : tap_or(taps, &blk_taps::attention_values, ws.v);
  const int kv_stride = decode ? cache->capacity : T;
  const bool gated = d.attn_gate != 0, sandwich = d.sandwich_norm != 0;
  void* head_tap = taps ? taps->attention_head_outputs : nullptr;
  void* o = (head_tap && !gated) ? head_tap : ws.o;
  void* mid = tap_or(taps, &blk_taps::layer_mid, ws.mid);
  void* neur = tap_or(taps, &blk_taps::mlp_neurons, ws.neur);
  const float* y = static_cast<const float*>(ws.y);
  prof_mark(h, "fp32_block", (d.act == BLK_ACT_SWIGLU ? 13 : 12) + (gated ? 1 : 0) + (mask ? 1 : 0), s);
  if (mask) BLK_TRY(check_cuda(launch_mask_ranges(mask, B, T, ws.ranges, ws.pos0, h->status, s), "attention mask"));
  BLK_TRY(check_cuda(launch_rmsnorm(x, w->ln1_g, M, d.hidden, d.eps, ws.y, bf, s), "rmsnorm 1"));
  const int nq = qkv_cols(d);
  BLK_TRY(check_cuda(launch_gemm_f32(y, (const float*)w->wq, C, nq, M, Hd, d.hidden, s), "q GEMM"));
  BLK_TRY(check_cuda(launch_gemm_f32(y, (const float*)w->wk, C + Hd, nq, M, KVd, d.hidden, s), "k GEMM"));
  BLK_TRY(check_cuda(launch_gemm_f32(y, (const float*)w->wv, C + Hd + KVd, nq, M, KVd, d.hidden, s), "v GEMM"));
  if (gated)
    BLK_TRY(check_cuda(launch_gemm_f32(y, (const float*)w->w_attn_gate, C + Hd + 2 * KVd, nq, M, Hd, d.hidden, s),
                       "attention gate GEMM"));
  BLK_TRY(check_cuda(launch_post_qkv(C, 1, M, nq, T, mask ? ws.pos0 : nullptr, decode ? cache->lens : nullptr, d.n_heads,
                                     d.n_kv_heads, d.head_dim, d.qk_norm, w->q_norm_g, w->k_norm_g, d.eps, h->rope,
                                     d.max_seq, q, k, v, kv_stride, bf, s, gated ? ws.gate : nullptr),
                     "qkv post"));
  AttnOpts opt;
  opt.window = d.sliding_window;
  opt.gate = gated ? ws.gate : nullptr;
  opt.ungated = gated ? head_tap : nullptr;
  opt.key_range = mask ? ws.ranges : nullptr;
  BLK_TRY(check_cuda(launch_attn_f32((const float*)q, (const float*)k, (const float*)v, (float*)o, B, d.n_heads,
                                     d.n_kv_heads, T, d.head_dim, kv_stride, decode ? cache->lens : nullptr,
                                     decode ? 1 : 0, s, opt),
                     "attention"));
  BLK_TRY(check_cuda(launch_gemm_f32((const float*)o, (const float*)w->wo, C, d.hidden, M, d.hidden, Hd, s),
                     "o_proj GEMM"));
  BLK_TRY(check_cuda(launch_post_resid(C, 1, M, d.hidden, d.hidden, x, true, mid, true, nullptr,
                                       taps ? taps->attention_output : nullptr, w->ln2_g, d.eps, ws.y, nullptr, bf, s,
                                       sandwich ? w->post_attn_g : nullptr),
                     "o_proj post"));
  const int nm = mlp_cols(d);
  if (d.act == BLK_ACT_SWIGLU) {
    BLK_TRY(check_cuda(launch_gemm_f32(y, (const float*)w->w_gate, C, nm, M, d.ffn, d.hidden, s), "gate GEMM"));
    BLK_TRY(check_cuda(launch_gemm_f32(y, (const float*)w->w_up, C + d.ffn, nm, M, d.ffn, d.hidden, s), "up GEMM"));
  } else {
    BLK_TRY(check_cuda(launch_gemm_f32(y, (const float*)w->w_up, C, nm, M, d.ffn, d.hidden, s), "up GEMM"));
  }
  BLK_TRY(check_cuda(launch_post_act(C, 1, M, d.ffn, nm, (int)d.act, d.xielu_alpha_p, d.xielu_alpha_n, d.xielu_beta,
                                     d.xielu_eps, neur, bf, s),
                     "activation"));
  BLK_TRY(check_cuda(launch_gemm_f32((const float*)neur, (const float*)w->w_down, C, d.hidden, M, d.hidden, d.ffn, s),
                     "down GEMM"));
  BLK_TRY(check_cuda(launch_post_resid(C, 1, M, d.hidden, d.hidden, mid, true, out, true, nullptr,
                                       taps ? taps->mlp_output : nullptr, nullptr, d.eps, nullptr,
                                       decode ? cache->lens : nullptr, bf, s, sandwich ? w->post_mlp_g : nullptr),
                     "down post"));
  prof_end(h, s);
  return BLK_OK;
}

blk_status check_weights(const blk_desc& d, const blk_weights* w) {
  if (!w) return fail(BLK_ERR_INVALID_ARG, "weights is NULL");
  const void* req[] = {w->ln1_g, w->wq, w->wk, w->wv, w->wo, w->ln2_g, w->w_up, w->w_down};
  for (const void* p : req) {
    if (!p) return fail(BLK_ERR_INVALID_ARG, "a required weight pointer is NULL");
    if (!aligned16(p)) return fail(BLK_ERR_ALIGNMENT, "a weight pointer is not 16-byte aligned");
  }
  if (d.act == BLK_ACT_SWIGLU && (!w->w_gate || !aligned16(w->w_gate)))
    return fail(w->w_gate ? BLK_ERR_ALIGNMENT : BLK_ERR_INVALID_ARG, "SWIGLU needs an aligned w_gate");
  if (d.qk_norm && (!w->q_norm_g || !w->k_norm_g || !aligned16(w->q_norm_g) || !aligned16(w->k_norm_g)))
    return fail(BLK_ERR_INVALID_ARG, "qk_norm needs aligned q_norm_g and k_norm_g");
  if (w->prepared && (d.dtype != BLK_BF16 || !aligned16(w->prepared)))
    return fail(BLK_ERR_INVALID_ARG, "prepared weights: bf16 handles only, 16-byte aligned");
  if (d.attn_gate && (!w->w_attn_gate || !aligned16(w->w_attn_gate)))
    return fail(w->w_attn_gate ? BLK_ERR_ALIGNMENT : BLK_ERR_INVALID_ARG, "attn_gate needs an aligned w_attn_gate");
  if (d.sandwich_norm && (!w->post_attn_g || !w->post_mlp_g || !aligned16(w->post_attn_g) || !aligned16(w->post_mlp_g)))
    return fail(BLK_ERR_INVALID_ARG, "sandwich_norm needs aligned post_attn_g and post_mlp_g");
  // A sandwich post-norm rescales its sublayer's output to the size of the residual
  // stream, and with it the relative error of that sublayer's GEMM operands. With bf16
  // operands (the only type that meets bf16 weights) that error reaches the block's
  // output at the size of its whole bf16 tolerance; the prepared fp16 operands keep it
  // at a fraction of it. So the bf16 path runs sandwich blocks on prepared weights only.
  if (d.dtype == BLK_BF16 && d.sandwich_norm && !w->prepared)
    return fail(BLK_ERR_UNSUPPORTED, "sandwich_norm on the bf16 path needs prepared weights (blk_prepare_weights)");
  return BLK_OK;
}

}  // namespace

// ================================================================== C ABI

extern "C" {

const char* blk_version(void) { return "gb300-decoder-block 0.1 (sm_103a)"; }

const char* blk_error_string(blk_status s) {
  switch (s) {
    case BLK_OK: return "BLK_OK";
    case BLK_ERR_INVALID_ARG: return "BLK_ERR_INVALID_ARG";
    case BLK_ERR_UNSUPPORTED: return "BLK_ERR_UNSUPPORTED";
    case BLK_ERR_ALIGNMENT: return "BLK_ERR_ALIGNMENT";
    case BLK_ERR_CACHE_FULL: return "BLK_ERR_CACHE_FULL";
    case BLK_ERR_CUDA: return "BLK_ERR_CUDA";
    case BLK_ERR_TIMEOUT: return "BLK_ERR_TIMEOUT";
    case BLK_ERR_WORKSPACE: return "BLK_ERR_WORKSPACE";
  }
  return "BLK_ERR_UNKNOWN";
}

const char* blk_last_error_message(void) { return g_err.c_str(); }

void blk_debug_set_wait_timeout_ns(long long ns) { g_wait_ns.store(ns > 0 ? ns : 2000000000LL); }

void blk_xielu_effective(float raw_alpha_p, float raw_alpha_n, float beta, float* alpha_p, float* alpha_n) {
  auto softplus = [](double t) { return t > 30.0 ? t : std::log1p(std::exp(t)); };
  if (alpha_p) *alpha_p = (float)softplus(raw_alpha_p);
  if (alpha_n) *alpha_n = (float)(beta + softplus(raw_alpha_n));
}

blk_status blk_create(const blk_desc* desc, blk_handle** out) {
  if (!desc || !out) return fail(BLK_ERR_INVALID_ARG, "desc/out is NULL");
  *out = nullptr;
  const blk_desc& d = *desc;
  if (d.hidden <= 0 || d.n_heads <= 0 || d.n_kv_heads <= 0 || d.head_dim <= 0 || d.ffn <= 0 || d.max_batch <= 0 ||
      d.max_seq <= 0)
    return fail(BLK_ERR_INVALID_ARG, "sizes must be positive");
  if (d.n_heads % d.n_kv_heads) return fail(BLK_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads");
  if (d.head_dim % 2) return fail(BLK_ERR_INVALID_ARG, "head_dim must be even");
  if (!(d.eps > 0.f) || !(d.rope_theta > 0.f)) return fail(BLK_ERR_INVALID_ARG, "eps and rope_theta must be > 0");
  if (d.rope_type != BLK_ROPE_PLAIN) {
    if (d.rope_type != BLK_ROPE_YARN && d.rope_type != BLK_ROPE_LLAMA3)
      return fail(BLK_ERR_INVALID_ARG, "unknown rope_type");
    if (!(d.rope_factor >= 1.f) || d.rope_orig_max_pos <= 0 || !(d.rope_low > 0.f) || !(d.rope_high > d.rope_low))
      return fail(BLK_ERR_INVALID_ARG, "rope scaling needs factor >= 1, original positions > 0, high > low > 0");
  }
  if (d.act != BLK_ACT_SWIGLU && d.act != BLK_ACT_RELU2 && d.act != BLK_ACT_XIELU)
    return fail(BLK_ERR_INVALID_ARG, "unknown activation");
  if (d.sliding_window < 0) return fail(BLK_ERR_INVALID_ARG, "sliding_window must be >= 0");
  if ((d.no_rope | d.attn_gate | d.sandwich_norm) & ~1)
    return fail(BLK_ERR_INVALID_ARG, "no_rope, attn_gate and sandwich_norm are 0 or 1");
  if (d.no_rope && d.rope_type != BLK_ROPE_PLAIN) return fail(BLK_ERR_INVALID_ARG, "no_rope with a rope scaling");
  if (d.dtype != BLK_F32 && d.dtype != BLK_BF16) return fail(BLK_ERR_INVALID_ARG, "unknown dtype");
  if (d.dtype == BLK_BF16) {
    if (d.head_dim != 128) return fail(BLK_ERR_UNSUPPORTED, "bf16 path: head_dim must be 128");
    if (d.hidden % 8 || d.ffn % 8) return fail(BLK_ERR_UNSUPPORTED, "bf16 path: hidden and ffn must be multiples of 8");
    if (d.hidden > 16384 * 4) return fail(BLK_ERR_UNSUPPORTED, "hidden too large");
    if (d.hidden / 8 > 8 * 256) return fail(BLK_ERR_UNSUPPORTED, "bf16 rmsnorm: hidden <= 16384");
    if (d.n_heads / d.n_kv_heads > 16) return fail(BLK_ERR_UNSUPPORTED, "bf16 decode: at most 16 heads per KV head");
  } else {
    if (d.hidden % 8) return fail(BLK_ERR_UNSUPPORTED, "fp32 path: hidden must be a multiple of 8");
    if (d.hidden / 8 > 8 * 256) return fail(BLK_ERR_UNSUPPORTED, "fp32 rmsnorm: hidden <= 16384");
    if (d.head_dim > 256) return fail(BLK_ERR_UNSUPPORTED, "fp32 path: head_dim <= 256");
    if (d.max_seq > 50000) return fail(BLK_ERR_UNSUPPORTED, "fp32 attention: max_seq <= 50000");
  }
  blk_handle* h = new blk_handle();
  h->d = d;
  h->rope = nullptr;
  h->status = nullptr;
  h->dev_flag = nullptr;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "blk_create: device query");
  }
  // RoPE table [max_seq][head_dim / 2] of (cos, sin), in double: inv_freq_i = theta^(-2i/d),
  // stretched by the descriptor's scaling. A frequency f of wavelength lam = 2 pi / f makes
  // r = L / lam turns over the original context L; fast components are kept, slow ones
  // divided by the factor s, and the rest blended. llama3 blends linearly in r:
  // (1 - g) f / s + g f, g = (r - lo) / (hi - lo). YaRN, as its published implementation
  // builds it, blends linearly in the pair index: the index where a component makes R turns
  // is i(R) = d ln(L / (2 pi R)) / (2 ln theta), and between a = floor(i(hi)) and
  // b = ceil(i(lo)) the weight of f / s grows from 0 to 1.
  const int half = d.head_dim / 2;
  std::vector<double> inv_freq(half);
  const double s_f = d.rope_factor, L = d.rope_orig_max_pos, lo = d.rope_low, hi = d.rope_high;
  const double theta = (double)d.rope_theta, dd = (double)d.head_dim;
  auto index_of_turns = [&](double r) { return dd * std::log(L / (2.0 * M_PI * r)) / (2.0 * std::log(theta)); };
  double ya = 0.0, yb = 1.0;
  if (d.rope_type == BLK_ROPE_YARN) {
    ya = std::max(std::floor(index_of_turns(hi)), 0.0);
    yb = std::min(std::ceil(index_of_turns(lo)), dd - 1.0);
    if (yb == ya) yb = ya + 0.001;
  }
  for (int i = 0; i < half; ++i) {
    const double f = std::pow(theta, -2.0 * i / dd);
    double fi = f;
    if (d.rope_type == BLK_ROPE_LLAMA3) {
      const double lam = 2.0 * M_PI / f;
      if (lam > L / lo) {
        fi = f / s_f;
      } else if (lam >= L / hi) {
        const double g = (L / lam - lo) / (hi - lo);
        fi = (1.0 - g) * f / s_f + g * f;
      }
    } else if (d.rope_type == BLK_ROPE_YARN) {
      const double w = std::min(1.0, std::max(0.0, (i - ya) / (yb - ya)));
      fi = (1.0 - w) * f + w * f / s_f;
    }
    inv_freq[i] = d.no_rope ? 0.0 : fi;  // no rotary: every angle 0, the identity rotation
  }
  const double att = d.rope_type == BLK_ROPE_YARN ? 0.1 * std::log(s_f) + 1.0 : 1.0;  // YaRN's sqrt(1/t)
  std::vector<float2> table((size_t)d.max_seq * half);
  for (int p = 0; p < d.max_seq; ++p)
    for (int i = 0; i < half; ++i) {
      const double ang = (double)p * inv_freq[i];
      table[(size_t)p * half + i] = make_float2((float)(att * std::cos(ang)), (float)(att * std::sin(ang)));
    }
  e = cudaMalloc(&h->rope, table.size() * sizeof(float2));
  if (e == cudaSuccess) e = cudaMemcpy(h->rope, table.data(), table.size() * sizeof(float2), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMalloc(&h->status, sizeof(DevStatus));
  if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof(DevStatus));
  if (e == cudaSuccess) e = cudaMalloc(&h->dev_flag, sizeof(int));
  if (e != cudaSuccess) {
    if (h->rope) cudaFree(h->rope);
    if (h->status) cudaFree(h->status);
    if (h->dev_flag) cudaFree(h->dev_flag);
    delete h;
    return cuda_fail(e, "blk_create: allocation");
  }
  *out = h;
  return BLK_OK;
}

blk_status blk_destroy(blk_handle* h) {
  if (!h) return BLK_OK;
  blk_profile_enable(h, 0);
  if (h->rope) cudaFree(h->rope);
  if (h->status) cudaFree(h->status);
  if (h->dev_flag) cudaFree(h->dev_flag);
  delete h;
  return BLK_OK;
}

size_t blk_prepared_bytes(const blk_handle* h) {
  if (!h || h->d.dtype != BLK_BF16) return 0;
  return prepared_layout(h->d, nullptr, nullptr);
}

blk_status blk_prepare_weights(blk_handle* h, const blk_weights* w, void* prepared, size_t bytes, void* stream) {
  if (!h || !w || !prepared) return fail(BLK_ERR_INVALID_ARG, "NULL argument");
  const blk_desc& d = h->d;
  if (d.dtype != BLK_BF16) return fail(BLK_ERR_UNSUPPORTED, "prepared weights exist for the bf16 path only");
  if (!w->wo || !w->w_up || (d.act == BLK_ACT_SWIGLU && !w->w_gate) || !w->wq || !w->wk || !w->wv || !w->ln1_g ||
      !w->ln2_g || (d.attn_gate && !w->w_attn_gate))
    return fail(BLK_ERR_INVALID_ARG, "a weight to prepare is NULL");
  if (!aligned16(prepared)) return fail(BLK_ERR_ALIGNMENT, "prepared buffer not 16-byte aligned");
  if (bytes < blk_prepared_bytes(h)) return fail(BLK_ERR_WORKSPACE, "prepared buffer too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Prepared p{};
  prepared_layout(d, prepared, &p);
  BLK_TRY(check_cuda(cudaMemsetAsync(h->dev_flag, 0, sizeof(int), s), "prepare"));
  const size_t n_o = (size_t)d.hidden * d.n_heads * d.head_dim, n_f = (size_t)d.ffn * d.hidden;
  BLK_TRY(check_cuda(launch_cast_bf16_f16(w->wo, const_cast<void*>(p.wo), n_o, h->dev_flag, s), "prepare wo"));
  if (p.wg)
    BLK_TRY(check_cuda(launch_cast_bf16_f16(w->w_gate, const_cast<void*>(p.wg), n_f, h->dev_flag, s), "prepare w_gate"));
  BLK_TRY(check_cuda(launch_cast_bf16_f16(w->w_up, const_cast<void*>(p.wu), n_f, h->dev_flag, s), "prepare w_up"));
  const size_t n_q = (size_t)d.n_heads * d.head_dim * d.hidden, n_kv = (size_t)d.n_kv_heads * d.head_dim * d.hidden;
  BLK_TRY(check_cuda(launch_cast_bf16_f16(w->wq, const_cast<void*>(p.wq), n_q, h->dev_flag, s), "prepare wq"));
  BLK_TRY(check_cuda(launch_cast_bf16_f16(w->wk, const_cast<void*>(p.wk), n_kv, h->dev_flag, s), "prepare wk"));
  BLK_TRY(check_cuda(launch_cast_bf16_f16(w->wv, const_cast<void*>(p.wv), n_kv, h->dev_flag, s), "prepare wv"));
  if (p.wag)
    BLK_TRY(check_cuda(launch_cast_bf16_f16(w->w_attn_gate, const_cast<void*>(p.wag), n_q, h->dev_flag, s),
                       "prepare w_attn_gate"));
  // A normed row has |x_i| / rms(x) <= sqrt(D), so its fp16 copy (x / rms * g) stays finite when
  // max|g| * sqrt(D) <= 65504: checked for the norms whose fp16 output is normalized first
  // (input_layernorm, and the MLP's input norm of the sandwich block).
  std::vector<uint16_t> gains((size_t)d.hidden);
  const void* checked[2] = {w->ln1_g, d.sandwich_norm ? w->ln2_g : nullptr};
  for (const void* gp : checked) {
    if (!gp) continue;
    BLK_TRY(check_cuda(cudaMemcpyAsync(gains.data(), gp, gains.size() * 2, cudaMemcpyDeviceToHost, s), "prepare"));
    BLK_TRY(check_cuda(cudaStreamSynchronize(s), "prepare"));
    float gmax = 0.f;
    for (uint16_t u : gains) {
      uint32_t bits = (uint32_t)u << 16;
      float f;
      std::memcpy(&f, &bits, 4);
      gmax = std::max(gmax, std::fabs(f));
    }
    if (!(gmax * std::sqrt((float)d.hidden) <= 65504.f))
      return fail(BLK_ERR_UNSUPPORTED, "a norm gain is too large for fp16 normed rows: use the weights unprepared");
  }
  int overflow = 0;
  BLK_TRY(check_cuda(cudaMemcpyAsync(&overflow, h->dev_flag, sizeof(int), cudaMemcpyDeviceToHost, s), "prepare"));
  BLK_TRY(check_cuda(cudaStreamSynchronize(s), "prepare"));
  if (overflow) return fail(BLK_ERR_UNSUPPORTED, "a weight lies outside the fp16 range: use the weights unprepared");
  return BLK_OK;
}

size_t blk_workspace_bytes(const blk_handle* h, int batch, int seq, int decode) {
  if (!h || batch <= 0 || seq <= 0) return 0;
  size_t total = 0;
  carve_forward(h, nullptr, batch, seq, decode != 0 && seq == 1, &total);  // a chunk: the prefill layout
  return total;
}

}  // extern "C"

namespace {

blk_status forward_impl(blk_handle* h, const void* x, int batch, int seq, const blk_weights* w, blk_kv_cache* cache,
                        int host_lens_max, const int* mask, void* out, void* workspace, size_t workspace_bytes,
                        const blk_taps* taps, void* stream) {
  if (!h || !x || !out) return fail(BLK_ERR_INVALID_ARG, "handle, x and out must be non-NULL");
  const blk_desc& d = h->d;
  if (batch <= 0 || seq <= 0) return fail(BLK_ERR_INVALID_ARG, "batch and seq must be positive");
  if (batch > d.max_batch) return fail(BLK_ERR_INVALID_ARG, "batch exceeds max_batch");
  if (!aligned16(x) || !aligned16(out)) return fail(BLK_ERR_ALIGNMENT, "x/out not 16-byte aligned");
  if (x == out) return fail(BLK_ERR_INVALID_ARG, "out must not alias x");
  BLK_TRY(check_weights(d, w));
  if (taps) {
    void* tp[] = {taps->attention_queries, taps->attention_keys, taps->attention_values,
                  taps->attention_head_outputs, taps->attention_output, taps->layer_mid,
                  taps->mlp_neurons, taps->mlp_output};
    for (void* p : tp)
      if (p && !aligned16(p)) return fail(BLK_ERR_ALIGNMENT, "a tap pointer is not 16-byte aligned");
  }
  const bool decode = cache != nullptr && seq == 1;
  const bool chunk = cache != nullptr && seq > 1;  // a prefill chunk appended to the cache
  int max_len = 0;
  if (chunk) {
    if (d.dtype != BLK_BF16) return fail(BLK_ERR_UNSUPPORTED, "a prefill chunk over a KV cache takes the bf16 path");
    if (!cache->k || !cache->v || !cache->lens || cache->capacity <= 0)
      return fail(BLK_ERR_INVALID_ARG, "incomplete KV cache");
    if (!aligned16(cache->k) || !aligned16(cache->v)) return fail(BLK_ERR_ALIGNMENT, "cache not 16-byte aligned");
    if (host_lens_max < 0) return fail(BLK_ERR_INVALID_ARG, "a prefill chunk needs host_lens_max (the largest lens)");
    if (host_lens_max + seq > cache->capacity) return fail(BLK_ERR_CACHE_FULL, "cache capacity exceeded");
    if (host_lens_max + seq > d.max_seq) return fail(BLK_ERR_INVALID_ARG, "position beyond max_seq");
    if (taps && (taps->attention_keys || taps->attention_values))
      return fail(BLK_ERR_UNSUPPORTED, "a prefill chunk writes its keys and values to the cache, not to taps");
  } else if (decode) {
    if (!cache->k || !cache->v || !cache->lens || cache->capacity <= 0)
      return fail(BLK_ERR_INVALID_ARG, "incomplete KV cache");
    if (!aligned16(cache->k) || !aligned16(cache->v)) return fail(BLK_ERR_ALIGNMENT, "cache not 16-byte aligned");
    if (host_lens_max >= 0) {
      if (host_lens_max + 1 > cache->capacity) return fail(BLK_ERR_CACHE_FULL, "cache capacity exceeded");
      if (host_lens_max + 1 > d.max_seq) return fail(BLK_ERR_INVALID_ARG, "position beyond max_seq");
      max_len = host_lens_max + 1;
    } else {
      max_len = cache->capacity < d.max_seq ? cache->capacity : d.max_seq;
    }
  } else if (seq > d.max_seq) {
    return fail(BLK_ERR_INVALID_ARG, "seq exceeds max_seq");
  }
  size_t need = 0;
  Ws ws = carve_forward(h, workspace, batch, seq, decode, &need);
  if (!workspace || workspace_bytes < need) return fail(BLK_ERR_WORKSPACE, "workspace missing or too small");
  if (!aligned16(workspace)) return fail(BLK_ERR_ALIGNMENT, "workspace not 16-byte aligned");
  if (mask && (cache || !aligned16(mask)))
    return fail(cache ? BLK_ERR_UNSUPPORTED : BLK_ERR_ALIGNMENT, "attention_mask: prefill only, 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  prof_begin(h);
  if (d.dtype == BLK_F32) return forward_f32(h, x, batch, seq, w, cache, out, ws, taps, s, mask);
  if (decode) return forward_decode_bf16(h, x, batch, w, cache, max_len, out, ws, taps, s);
  return forward_prefill_bf16(h, x, batch, seq, w, out, ws, taps, s, chunk ? cache : nullptr, mask);
}

}  // namespace

extern "C" {

blk_status blk_forward(blk_handle* h, const void* x, int batch, int seq, const blk_weights* w, blk_kv_cache* cache,
                       int host_lens_max, void* out, void* workspace, size_t workspace_bytes, const blk_taps* taps,
                       void* stream) {
  return forward_impl(h, x, batch, seq, w, cache, host_lens_max, nullptr, out, workspace, workspace_bytes, taps,
                      stream);
}

blk_status blk_forward_masked(blk_handle* h, const void* x, int batch, int seq, const int* attention_mask,
                              const blk_weights* w, void* out, void* workspace, size_t workspace_bytes,
                              const blk_taps* taps, void* stream) {
  if (!attention_mask) return fail(BLK_ERR_INVALID_ARG, "attention_mask is NULL");
  return forward_impl(h, x, batch, seq, w, nullptr, -1, attention_mask, out, workspace, workspace_bytes, taps,
                      stream);
}

// ------------------------------------------------------------------ the model around the block

namespace {
struct ModelWs {
  void *block, *act0, *act1, *ynorm;
  size_t block_bytes, total;
};

ModelWs carve_model(const blk_handle* h, void* base, int batch, int seq, bool decode) {
  const blk_desc& d = h->d;
  ModelWs m{};
  m.block_bytes = blk_workspace_bytes(h, batch, seq, decode ? 1 : 0);
  const size_t act = (size_t)batch * seq * d.hidden * esize(d);
  Carve c(base);
  m.block = c.take(m.block_bytes);
  m.act0 = c.take(act);
  m.act1 = c.take(act);
  m.ynorm = c.take(act);
  m.total = c.off;
  return m;
}
}  // namespace

size_t blk_model_workspace_bytes(const blk_handle* h, int batch, int seq, int decode) {
  if (!h || batch <= 0 || seq <= 0) return 0;
  return carve_model(h, nullptr, batch, seq, decode != 0).total;
}

blk_status blk_model_forward(blk_handle* h, const blk_model* m, const int* tokens, int batch, int seq,
                             blk_kv_cache* caches, int host_lens_max, void* logits, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!h || !m || !tokens || !logits) return fail(BLK_ERR_INVALID_ARG, "handle, model, tokens and logits must be non-NULL");
  const blk_desc& d = h->d;
  if (m->n_layers < 1 || !m->layers || !m->embed || !m->norm_g || !m->lm_head || m->vocab <= 0)
    return fail(BLK_ERR_INVALID_ARG, "model: n_layers >= 1, layers, embed, norm_g, lm_head and vocab > 0");
  if (m->vocab % 8) return fail(BLK_ERR_UNSUPPORTED, "model: vocab must be a multiple of 8 (16-byte logit rows)");
  if (batch <= 0 || seq <= 0) return fail(BLK_ERR_INVALID_ARG, "batch and seq must be positive");
  if (!aligned16(m->embed) || !aligned16(m->lm_head) || !aligned16(logits) || !aligned16(workspace))
    return fail(BLK_ERR_ALIGNMENT, "model: embed, lm_head, logits and workspace must be 16-byte aligned");
  const ModelWs mw = carve_model(h, workspace, batch, seq, caches != nullptr);
  if (!workspace || workspace_bytes < mw.total) return fail(BLK_ERR_WORKSPACE, "model workspace missing or too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int M = batch * seq;
  BLK_TRY(check_cuda(launch_embed(tokens, m->embed, M, (int)(d.hidden * esize(d)), m->vocab, mw.act0, h->status,
                                  h->num_sms, s),
                     "embedding"));
  void* bufs[2] = {mw.act0, mw.act1};
  for (int l = 0; l < m->n_layers; ++l)  // each layer reads one buffer and writes the other
    BLK_TRY(blk_forward(h, bufs[l & 1], batch, seq, &m->layers[l], caches ? &caches[l] : nullptr, host_lens_max,
                        bufs[(l + 1) & 1], mw.block, mw.block_bytes, nullptr, stream));
  const void* last = bufs[m->n_layers & 1];
  const bool bf = d.dtype == BLK_BF16;
  BLK_TRY(check_cuda(launch_rmsnorm(last, m->norm_g, M, d.hidden, d.eps, mw.ynorm, bf, s), "final norm"));
  if (!bf)
    return check_cuda(launch_gemm_f32(static_cast<const float*>(mw.ynorm), static_cast<const float*>(m->lm_head),
                                      static_cast<float*>(logits), m->vocab, M, m->vocab, d.hidden, s),
                      "lm_head GEMM");
  TcGemmDesc g;
  g.na = 1;
  g.a[0] = {mw.ynorm, M, 0};
  g.nb = 1;
  g.b[0] = {m->lm_head, m->vocab, 0};
  g.K = d.hidden;
  static const int cands[] = {256, 224, 192, 128};
  const TileChoice tl = choose_tile(M, m->vocab, false, cands, 4, h->num_sms, d.hidden >= kPairMinK);
  g.bn = tl.bn;
  g.pair = tl.pair;
  g.epi = Epi::kStore;
  g.const_op = 2;
  g.e.out = logits;
  g.e.ldo = m->vocab;
  return tc(h, g, s, "lm_head GEMM");
}

struct blk_graph {
  blk_handle* h;
  cudaGraphExec_t exec;
  bool profiled;
};

blk_status blk_forward_graph_create(blk_handle* h, const void* x, int batch, int seq, const blk_weights* w,
                                    blk_kv_cache* cache, int host_lens_max, void* out, void* workspace,
                                    size_t workspace_bytes, const blk_taps* taps, blk_graph** out_graph) {
  if (!h || !out_graph) return fail(BLK_ERR_INVALID_ARG, "NULL handle or out_graph");
  *out_graph = nullptr;
  cudaStream_t cs = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e, "graph: stream");
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) {
    cudaStreamDestroy(cs);
    return cuda_fail(e, "graph: begin capture");
  }
  blk_status st = blk_forward(h, x, batch, seq, w, cache, host_lens_max, out, workspace, workspace_bytes, taps, cs);
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(cs, &graph);
  h->prof.pending = false;  // nothing ran: the events fire on replays
  cudaStreamDestroy(cs);
  if (st != BLK_OK) {
    if (graph) cudaGraphDestroy(graph);
    return st;
  }
  if (e != cudaSuccess) return cuda_fail(e, "graph: end capture");
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return cuda_fail(e, "graph: instantiate");
  *out_graph = new blk_graph{h, exec, h->prof.on};
  return BLK_OK;
}

blk_status blk_graph_launch(blk_graph* g, void* stream) {
  if (!g) return fail(BLK_ERR_INVALID_ARG, "NULL graph");
  cudaError_t e = cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "graph launch");
  if (g->profiled && g->h->prof.on) g->h->prof.pending = true;
  return BLK_OK;
}

blk_status blk_graph_destroy(blk_graph* g) {
  if (!g) return BLK_OK;
  cudaGraphExecDestroy(g->exec);
  delete g;
  return BLK_OK;
}

blk_status blk_rmsnorm(const void* x, const void* g, int rows, int n, float eps, void* y, blk_dtype dtype,
                       void* stream) {
  if (!x || !g || !y) return fail(BLK_ERR_INVALID_ARG, "x, g and y must be non-NULL");
  if (rows < 0 || n <= 0) return fail(BLK_ERR_INVALID_ARG, "bad sizes");
  if (!aligned16(x) || !aligned16(g) || !aligned16(y)) return fail(BLK_ERR_ALIGNMENT, "pointers not 16-byte aligned");
  if (n % 8) return fail(BLK_ERR_UNSUPPORTED, "n must be a multiple of 8");
  if (n / 8 > 8 * 256) return fail(BLK_ERR_UNSUPPORTED, "n too large (<= 16384)");
  return check_cuda(launch_rmsnorm(x, g, rows, n, eps, y, dtype == BLK_BF16, static_cast<cudaStream_t>(stream)),
                    "rmsnorm");
}

size_t blk_stage_workspace_bytes(const blk_handle* h, int rows) {
  if (!h || rows <= 0) return 0;
  const blk_desc& d = h->d;
  Carve c(nullptr);
  c.take((size_t)rows * d.ffn * esize(d));                              // neurons
  c.take((size_t)rows * max_cols(d) * sizeof(float));                   // fp32 GEMM output
  const int s = attn_decode_split_cap(d.max_seq);
  c.take(attn_decode_ws_bytes(rows, d.n_heads, d.head_dim, s));         // decode attention partials
  return c.off;
}

blk_status blk_qkv_rope(blk_handle* h, const void* y, const blk_weights* w, int batch, int seq, const int* pos0,
                        void* q, void* k, void* v, void* workspace, size_t workspace_bytes, void* stream) {
  if (!h || !y || !w || !q || !k || !v) return fail(BLK_ERR_INVALID_ARG, "NULL argument");
  const blk_desc& d = h->d;
  if (batch <= 0 || seq <= 0) return fail(BLK_ERR_INVALID_ARG, "bad sizes");
  if (!aligned16(y) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return fail(BLK_ERR_ALIGNMENT, "alignment");
  if (!w->wq || !w->wk || !w->wv) return fail(BLK_ERR_INVALID_ARG, "wq/wk/wv NULL");
  if (d.qk_norm && (!w->q_norm_g || !w->k_norm_g)) return fail(BLK_ERR_INVALID_ARG, "q/k norm gains NULL");
  if (d.qk_norm && (!aligned16(w->q_norm_g) || !aligned16(w->k_norm_g)))
    return fail(BLK_ERR_ALIGNMENT, "q/k norm gains not 16-byte aligned");
  if (!pos0 && seq > d.max_seq) return fail(BLK_ERR_INVALID_ARG, "seq exceeds max_seq");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d.dtype == BLK_BF16) return bf16_qkv(h, y, w, batch, seq, pos0, q, k, v, s);
  const int M = batch * seq;
  if (!workspace || workspace_bytes < blk_stage_workspace_bytes(h, M)) return fail(BLK_ERR_WORKSPACE, "workspace");
  Carve c(workspace);
  c.take((size_t)M * d.ffn * esize(d));
  float* C = static_cast<float*>(c.take((size_t)M * max_cols(d) * sizeof(float)));
  const int Hd = d.n_heads * d.head_dim, KVd = d.n_kv_heads * d.head_dim, nq = qkv_cols(d);
  const float* yy = static_cast<const float*>(y);
  BLK_TRY(check_cuda(launch_gemm_f32(yy, (const float*)w->wq, C, nq, M, Hd, d.hidden, s), "q GEMM"));
  BLK_TRY(check_cuda(launch_gemm_f32(yy, (const float*)w->wk, C + Hd, nq, M, KVd, d.hidden, s), "k GEMM"));
  BLK_TRY(check_cuda(launch_gemm_f32(yy, (const float*)w->wv, C + Hd + KVd, nq, M, KVd, d.hidden, s), "v GEMM"));
  return check_cuda(launch_post_qkv(C, 1, M, nq, seq, pos0, nullptr, d.n_heads, d.n_kv_heads, d.head_dim, d.qk_norm,
                                    w->q_norm_g, w->k_norm_g, d.eps, h->rope, d.max_seq, q, k, v, seq, false, s),
                    "qkv post");
}

blk_status blk_attn_gqa(blk_handle* h, const void* q, const void* k, const void* v, int batch, int seq_q,
                        int kv_stride, const int* kv_lens, void* o, void* workspace, size_t workspace_bytes,
                        void* stream) {
  if (!h || !q || !k || !v || !o) return fail(BLK_ERR_INVALID_ARG, "NULL argument");
  const blk_desc& d = h->d;
  if (batch <= 0 || seq_q <= 0 || kv_stride < (kv_lens ? 1 : seq_q)) return fail(BLK_ERR_INVALID_ARG, "bad sizes");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return fail(BLK_ERR_ALIGNMENT, "alignment");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const char* why = nullptr;
  AttnOpts opt;
  opt.window = d.sliding_window;  // the head outputs: before any attention gate
  if (d.dtype == BLK_F32) {
    if ((size_t)kv_stride * 4 > 200 * 1024) return fail(BLK_ERR_UNSUPPORTED, "fp32 attention: kv_stride too large");
    return check_cuda(launch_attn_f32((const float*)q, (const float*)k, (const float*)v, (float*)o, batch, d.n_heads,
                                      d.n_kv_heads, seq_q, d.head_dim, kv_stride, kv_lens, 0, s, opt),
                      "attention");
  }
  if (!kv_lens) {
    if (kv_stride != seq_q) return fail(BLK_ERR_UNSUPPORTED, "bf16 prefill attention: kv_stride must equal seq_q");
    return check_cuda(launch_attn_prefill_tc(q, k, v, o, batch, d.n_heads, d.n_kv_heads, seq_q, d.head_dim,
                                             false, false, h->status, (unsigned long long)g_wait_ns.load(), s, &why,
                                             nullptr, 0, opt),
                      "attention", why);
  }
  if (seq_q != 1) return fail(BLK_ERR_UNSUPPORTED, "bf16 attention over a cache: one query per sequence");
  if (!workspace || workspace_bytes < blk_stage_workspace_bytes(h, batch)) return fail(BLK_ERR_WORKSPACE, "workspace");
  Carve c(workspace);
  c.take((size_t)batch * d.ffn * esize(d));
  c.take((size_t)batch * max_cols(d) * sizeof(float));
  void* aw = c.take(0);
  return check_cuda(launch_attn_decode_bf16(q, k, v, o, batch, d.n_heads, d.n_kv_heads, d.head_dim, kv_stride, kv_lens,
                                            0, kv_stride, attn_decode_split_cap(d.max_seq),
                                            aw, h->num_sms, h->status, (unsigned long long)g_wait_ns.load(), s, &why,
                                            opt),
                    "decode attention", why);
}

blk_status blk_mlp(blk_handle* h, const void* resid, const void* h_normed, const blk_weights* w, int rows, void* out,
                   void* workspace, size_t workspace_bytes, void* stream) {
  if (!h || !resid || !h_normed || !w || !out) return fail(BLK_ERR_INVALID_ARG, "NULL argument");
  const blk_desc& d = h->d;
  if (rows <= 0) return fail(BLK_ERR_INVALID_ARG, "bad sizes");
  if (!aligned16(resid) || !aligned16(h_normed) || !aligned16(out)) return fail(BLK_ERR_ALIGNMENT, "alignment");
  if (!w->w_up || !w->w_down || (d.act == BLK_ACT_SWIGLU && !w->w_gate))
    return fail(BLK_ERR_INVALID_ARG, "MLP weights NULL");
  if (!workspace || workspace_bytes < blk_stage_workspace_bytes(h, rows)) return fail(BLK_ERR_WORKSPACE, "workspace");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Carve c(workspace);
  void* neur = c.take((size_t)rows * d.ffn * esize(d));
  float* C = static_cast<float*>(c.take((size_t)rows * max_cols(d) * sizeof(float)));
  if (d.sandwich_norm && (!w->post_mlp_g || !aligned16(w->post_mlp_g)))
    return fail(BLK_ERR_INVALID_ARG, "sandwich_norm needs an aligned post_mlp_g");
  // the stage's operand h_normed is the caller's bf16: a post-norm would scale its
  // rounding up to the residual's size (the whole block runs it on prepared weights)
  if (d.dtype == BLK_BF16 && d.sandwich_norm)
    return fail(BLK_ERR_UNSUPPORTED, "the MLP stage of a sandwich_norm block takes the fp32 path or blk_forward");
  const void* g_post = d.sandwich_norm ? w->post_mlp_g : nullptr;
  if (d.dtype == BLK_BF16) {
    BLK_TRY(bf16_mlp_up(h, h_normed, rows, w, neur, s));
    if (!g_post)
      return bf16_linear_resid(h, neur, rows, d.ffn, w->w_down, d.hidden, resid, false, out, false, nullptr, nullptr,
                               s, "down GEMM");
    BLK_TRY(bf16_linear_resid(h, neur, rows, d.ffn, w->w_down, d.hidden, nullptr, false, C, true, nullptr, nullptr, s,
                              "down GEMM"));
    return check_cuda(launch_post_resid(C, 1, rows, d.hidden, d.hidden, resid, false, out, false, nullptr, nullptr,
                                        nullptr, d.eps, nullptr, nullptr, true, s, g_post),
                      "post-MLP norm");
  }
  const float* y = static_cast<const float*>(h_normed);
  const int nm = mlp_cols(d);
  if (d.act == BLK_ACT_SWIGLU) {
    BLK_TRY(check_cuda(launch_gemm_f32(y, (const float*)w->w_gate, C, nm, rows, d.ffn, d.hidden, s), "gate GEMM"));
    BLK_TRY(check_cuda(launch_gemm_f32(y, (const float*)w->w_up, C + d.ffn, nm, rows, d.ffn, d.hidden, s), "up GEMM"));
  } else {
    BLK_TRY(check_cuda(launch_gemm_f32(y, (const float*)w->w_up, C, nm, rows, d.ffn, d.hidden, s), "up GEMM"));
  }
  BLK_TRY(check_cuda(launch_post_act(C, 1, rows, d.ffn, nm, (int)d.act, d.xielu_alpha_p, d.xielu_alpha_n,
                                     d.xielu_beta, d.xielu_eps, neur, false, s),
                     "activation"));
  BLK_TRY(check_cuda(launch_gemm_f32((const float*)neur, (const float*)w->w_down, C, d.hidden, rows, d.hidden, d.ffn, s),
                     "down GEMM"));
  return check_cuda(launch_post_resid(C, 1, rows, d.hidden, d.hidden, resid, true, out, true, nullptr, nullptr,
                                      nullptr, d.eps, nullptr, nullptr, false, s, g_post),
                    "down post");
}

blk_status blk_profile_enable(blk_handle* h, int on) {
  if (!h) return fail(BLK_ERR_INVALID_ARG, "NULL handle");
  StageProfile& p = h->prof;
  if (on && !p.on) {
    for (auto& e : p.ev)
      if (cudaEventCreate(&e) != cudaSuccess) return fail(BLK_ERR_CUDA, "cudaEventCreate");
    p.on = true;
    p.n = 0;
    p.pending = false;
  } else if (!on && p.on) {
    for (auto& e : p.ev) {
      cudaEventDestroy(e);
      e = nullptr;
    }
    p.on = false;
    p.pending = false;
  }
  return BLK_OK;
}

int blk_profile_collect(blk_handle* h, double* total_ms, long long* launches, int max_stages) {
  if (!h || !h->prof.on) return -1;
  StageProfile& p = h->prof;
  if (p.pending) {
    if (cudaEventSynchronize(p.ev[p.n]) != cudaSuccess) return -1;
    for (int i = 0; i < p.n; ++i) {
      float ms = 0.f;
      cudaEventElapsedTime(&ms, p.ev[i], p.ev[i + 1]);
      p.total_ms[i] += ms;
      p.total_launches[i] += p.launches[i];
    }
    p.pending = false;
  }
  for (int i = 0; i < p.n && i < max_stages; ++i) {
    if (total_ms) total_ms[i] = p.total_ms[i];
    if (launches) launches[i] = p.total_launches[i];
  }
  return p.n;
}

const char* blk_profile_stage_name(const blk_handle* h, int i) {
  if (!h || i < 0 || i >= h->prof.n || !h->prof.names[i]) return "";
  return h->prof.names[i];
}

void blk_profile_reset(blk_handle* h) {
  if (!h) return;
  for (int i = 0; i < StageProfile::kMax; ++i) {
    h->prof.total_ms[i] = 0.0;
    h->prof.total_launches[i] = 0;
  }
}

blk_status blk_debug_gemm_bf16(const void* a, const void* b, void* c, int M, int N, int K, int bn, int split_k,
                               int pair, void* stream) {
  if (!a || !b || !c) return fail(BLK_ERR_INVALID_ARG, "NULL argument");
  if (M <= 0 || N <= 0 || K <= 0 || K % 8 || (bn != 64 && bn != 128 && bn != 192 && bn != 224 && bn != 256) ||
      split_k < 1)
    return fail(BLK_ERR_INVALID_ARG, "bad sizes");
  if (split_k > 1 && bn != 64) return fail(BLK_ERR_INVALID_ARG, "split_k > 1 needs bn == 64");
  if (pair && (split_k != 1 || bn < 192)) return fail(BLK_ERR_INVALID_ARG, "pair needs split_k == 1, bn >= 192");
  if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return fail(BLK_ERR_ALIGNMENT, "alignment");
  if (split_k == 1 && N % 8) return fail(BLK_ERR_INVALID_ARG, "N % 8 != 0");
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  TcGemmDesc g;
  g.na = 1;
  g.nb = 1;
  g.K = K;
  g.bn = bn;
  g.k_splits = split_k;
  g.pair = pair != 0;
  if (split_k == 1) {
    g.a[0] = {a, M, 0};
    g.b[0] = {b, N, 0};
    g.epi = Epi::kStore;
    g.e.out = c;
    g.e.ldo = N;
  } else {  // swap-AB partials: "weights" b on the MMA rows, tokens a on its columns
    g.a[0] = {b, N, 0};
    g.b[0] = {a, M, 0};
    g.epi = Epi::kPartialT;
    g.e.out = c;
    g.e.part_ld = N;
    g.e.n_tok = M;
  }
  const char* why = nullptr;
  DevStatus* st = nullptr;
  cudaError_t e = debug_status_address(&st);
  if (e != cudaSuccess) return cuda_fail(e, "debug GEMM status word");
  e = launch_tc_gemm(g, sms, st, (unsigned long long)g_wait_ns.load(), static_cast<cudaStream_t>(stream), &why);
  return e == cudaSuccess ? BLK_OK : cuda_fail(e, "debug GEMM", why);
}

blk_status blk_debug_last_status(void) {
  DevStatus* dst = nullptr;
  cudaError_t e = debug_status_address(&dst);
  DevStatus st{0, 0};
  if (e == cudaSuccess) e = cudaMemcpy(&st, dst, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "blk_debug_last_status");
  if (st.code != 0) {
    cudaMemset(dst, 0, sizeof(DevStatus));
    char buf[96];
    snprintf(buf, sizeof(buf), "device wait timed out (site 0x%x)", st.where);
    return fail((blk_status)st.code, buf);
  }
  return BLK_OK;
}

blk_status blk_attn_decode_noalloc(const void* q, const void* k, const void* v, const int* kv_lens, int batch,
                                   int n_heads, int n_kv_heads, int head_dim, int kv_stride, void* o, void* stream) {
  if (!q || !k || !v || !kv_lens || !o) return fail(BLK_ERR_INVALID_ARG, "NULL argument");
  if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0 || kv_stride <= 0 || n_heads % n_kv_heads)
    return fail(BLK_ERR_INVALID_ARG, "bad sizes");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return fail(BLK_ERR_ALIGNMENT, "alignment");
  if (head_dim != 128) return fail(BLK_ERR_UNSUPPORTED, "head_dim must be 128");
  if (n_heads / n_kv_heads > 16) return fail(BLK_ERR_UNSUPPORTED, "at most 16 query heads per KV head");
  if ((size_t)batch * n_heads * (head_dim + 2) * sizeof(float) > kDecodeStaticScratchBytes - kAttnCounterBytes)
    return fail(BLK_ERR_UNSUPPORTED,
                "batch * n_heads * (head_dim + 2) * 4 bytes exceeds the 16 MiB allocation-free scratch");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  const char* why = nullptr;
  e = launch_attn_decode_bf16_static(q, k, v, o, batch, n_heads, n_kv_heads, head_dim, kv_stride, kv_lens, sms,
                                     (unsigned long long)g_wait_ns.load(), static_cast<cudaStream_t>(stream), &why);
  return e == cudaSuccess ? BLK_OK : cuda_fail(e, "allocation-free decode attention", why);
}

blk_status blk_last_status(blk_handle* h) {
  if (!h) return fail(BLK_ERR_INVALID_ARG, "NULL handle");
  DevStatus st{0, 0};
  cudaError_t e = cudaMemcpy(&st, h->status, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "blk_last_status");
  if (st.code != 0) {
    cudaMemset(h->status, 0, sizeof(DevStatus));
    char buf[96];
    snprintf(buf, sizeof(buf), "device wait timed out (site 0x%x)", st.where);
    return fail((blk_status)st.code, buf);
  }
  return BLK_OK;
}

}  // extern "C"
