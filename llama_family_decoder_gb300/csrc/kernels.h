// Internal launch interface between the host library (blk_api.cu) and the
// kernel translation units. Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace blk {

struct DevStatus;

// ---------------------------------------------------------------- RMSNorm
// y[r,:] = x[r,:] * rsqrt(mean(x[r,:]^2) + eps) * g   (fp32 statistics)
// x_f32: x is fp32 while g and y have the storage type (the bf16 path's fp32 residual stream).
// y_f16 (bf16 path): y is fp16, the operand of a GEMM with prepared fp16 weights.
// zero_word (optional): set to 0 once the kernel's predecessors are done (a later
// kernel's counter, e.g. the decode attention's).
cudaError_t launch_rmsnorm(const void* x, const void* g, int rows, int n, float eps, void* y, bool bf16,
                           cudaStream_t s, bool x_f32 = false, bool y_f16 = false, int* zero_word = nullptr);

// The input RMSNorm split for the fused bf16 prefill: row_scale[r] = rsqrt(mean(x[r]^2) + eps),
// xg[r, :] = bf16(x[r, :] * g) (the QKV GEMM's A; x itself when g == 1); zeroes zero_rows[r].
cudaError_t launch_norm_prep(const void* x, const void* g, int rows, int n, float eps, void* xg, float* row_scale,
                             float* zero_rows, cudaStream_t s);

// ---------------------------------------------------------------- embedding
// out[r, :] = table[tokens[r], :] (row_bytes per row, a multiple of 16); ids outside
// [0, vocab) give zero rows and set the status word to INVALID_ARG.
cudaError_t launch_embed(const int* tokens, const void* table, int rows, int row_bytes, int vocab, void* out,
                         DevStatus* st, int num_sms, cudaStream_t s);

// attention_mask [B, T] (int32, zeros are padding) -> ranges[b] = [lo, hi) of row b's ones
// ((T, T) for a row of zeros) and pos0[b] = -lo. A row whose ones are not contiguous records
// INVALID_ARG in the status word and is treated as its hull.
cudaError_t launch_mask_ranges(const int* mask, int B, int T, int2* ranges, int* pos0, DevStatus* st,
                               cudaStream_t s);

// dst[i] = bf16(src[i]) for fp16 src (n elements).
cudaError_t launch_cast_f16_bf16(const void* src, void* dst, size_t n, cudaStream_t s);

// dst[i] = fp16(src[i]) for bf16 src; *overflow = 1 if some |src[i]| > 65504.
cudaError_t launch_cast_bf16_f16(const void* src, void* dst, size_t n, int* overflow, cudaStream_t s);

// ---------------------------------------------------------------- fp32 SIMT GEMM
// C[m, c0 + n] = sum_k A[m, k] * B[n, k] for m < M, n < N  (fp32, row-major, ld = K for A/B).
cudaError_t launch_gemm_f32(const float* A, const float* B, float* C, int ldc, int M, int N, int K, cudaStream_t s);

// ---------------------------------------------------------------- tcgen05 GEMM (bf16 in, fp32 accumulate)

enum class Epi : int {
  kStore = 0,     // out[row, col] = bf16(acc)
  kResid = 1,     // out = resid + acc (fp32 sum, stored fp32 or bf16); optional bf16 copy and tap = bf16(acc)
  kQkv = 2,       // per-head optional RMSNorm, RoPE, scatter to q/k/v head-major layouts;
                  // a 4th B segment (the attention gate) stores sigmoid(acc) as fp16
  kSwiglu = 3,    // paired B halves [gate | up]: out = bf16(silu(gate) * up)
  kRelu2 = 4,     // out = bf16(relu(acc)^2)
  kXielu = 5,     // out = bf16(xielu(acc))
  kPartialT = 6,  // swap-AB split-K: part[split][token][feature] = acc^T (fp32)
  // Decode (swap-AB) with the K splits of a tile launched as one thread-block
  // cluster: each split keeps its fp32 partial in shared memory, and CTA r of
  // the cluster sums slice r of the tile's tokens over all splits (distributed
  // shared memory, split order) and applies the post-op.
  kDecQkv = 7,    // per-head q/k RMSNorm, RoPE at position lens[t], q store, K/V cache append,
                  // a 4th A segment (the attention gate): sigmoid(acc) as fp16
  kDecResid = 8,  // resid + acc (fp32), optional taps, next RMSNorm (gained rows + sum of squares)
  // Decode MLP up + activation: persistent clusters of K splits walk the tiles,
  // the splits' partials of a tile meet in shared memory (two buffers, mbarrier
  // hand-off across the cluster) while the next tile streams; with paired A
  // (64 gate rows over 64 up rows) out = bf16(silu(gate * rs) * (up * rs)), else
  // relu^2 or xIELU of up * rs; rs = the MLP input's 1/rms (row_ss), or 1.
  kDecAct = 9,
  // kResid with an fp32 output written through shared memory by TMA bulk tensor stores
  // (one B segment covering the output's columns): the o_proj of the prefill block
  kResidTma = 10,
};

// How many clusters of `splits` CTAs of the decode GEMM kernel (tile width bn,
// epilogue epi) can be resident at once; 0 if the query fails.
int tc_dec_max_clusters(int bn, Epi epi, int splits);

// One row-segment of an operand: a contiguous [rows, K] bf16 matrix.
struct TcSeg {
  const void* ptr;
  int rows;
  int out_offset;  // where this segment's rows land in the concatenated output
};

struct TcEpiArgs {
  void* out = nullptr;  // kStore/kResid/activations: bf16 [rows, ldo]; kPartialT: float partial base
  int ldo = 0;
  const void* resid = nullptr;  // kResid: [rows, ldo], bf16 or (resid_f32) fp32; null: out = acc
  int resid_f32 = 0;
  int out_f32 = 0;              // kResid: out is fp32 (the block's residual stream)
  void* out2 = nullptr;         // kResid: optional bf16 copy of out
  void* tap = nullptr;          // kResid: optional bf16 contribution [rows, ldo]
  // kQkv
  void* q = nullptr;
  void* k = nullptr;
  void* v = nullptr;
  int seq = 0;          // tokens per sequence (row -> (b, t))
  int n_heads = 0;
  int n_kv_heads = 0;
  int head_dim = 0;
  int kv_stride = 0;    // rows per (b, kv head) in k/v (== seq for prefill)
  const void* q_gain = nullptr;
  const void* k_gain = nullptr;
  float eps = 0.f;
  const float2* rope = nullptr;  // [max_pos][head_dim/2] (cos, sin)
  int rope_max_pos = 0;
  const int* pos0 = nullptr;     // [B] first position of each sequence, or null
  int kv_at_pos = 0;             // kQkv: k/v go to row pos0[b] + t of a cache (kv_stride rows), not row t
  int qk_norm = 0;
  const float* row_scale = nullptr;  // kQkv: per-row factor of the accumulator (the input norm's 1/rms)
  int qkv_f16 = 0;                   // kQkv: store q/k/v as fp16 (else bf16)
  void* gate = nullptr;              // kQkv/kDecQkv: fp16 [rows, n_heads * head_dim], sigmoid of the gate segment
  // activations: per-row RMSNorm of the A rows from a sum of squares, 1/rms = rsqrt(row_ss / ss_n + ss_eps)
  // (row_ss holds ss_parts partial sums per row, summed in order)
  const float* row_ss = nullptr;
  int ss_parts = 0;
  int ss_n = 0;
  float ss_eps = 0.f;
  // kResid: the next RMSNorm split in two: norm_out = bf16(out * norm_gain), and
  // norm_ss[row * norm_parts + n_tile] = sum over the tile's columns of out^2
  void* norm_out = nullptr;
  int norm_f16 = 0;  // norm_out in fp16 (else bf16)
  const void* norm_gain = nullptr;
  float* norm_ss = nullptr;
  int norm_parts = 0;
  // activations
  float alpha_p = 0.f, alpha_n = 0.f, beta = 0.f, xeps = 0.f;
  // kPartialT
  int part_ld = 0;  // features per token row of the partial buffer
  int n_tok = 0;    // valid tokens (B operand rows)
  int act = 0;  // kDecAct: 0 SwiGLU (paired A), 1 relu^2, 2 xIELU
  // decode finishers
  const int* lens = nullptr;  // kDecQkv: positions already in the cache, per sequence
  int* bump_lens = nullptr;   // kDecResid: lens[t] += 1 once per token (the tile of m_tile 0);
                              // kResid: lens[b] += seq once per sequence (its last row, first N tile)
};

constexpr int kMaxSegs = 4;

struct TcGemmDesc {
  TcSeg a[kMaxSegs];
  int na = 1;
  TcSeg b[kMaxSegs];
  int nb = 1;
  bool b_paired = false;  // B tile = halves from b[0] and b[1] at the same rows (gate/up)
  bool a_paired = false;  // A tile = 64 rows of a[0] over 64 rows of a[1] at the same rows (kDecAct)
  // A CTA pair (cluster of 2, tcgen05 cta_group::2) computes each 256 x BN tile: the
  // even CTA issues M = 256 MMAs over both CTAs' shared memory, each CTA loading its
  // 128 A rows and half of B. Prefill epilogues, one A segment, no K split.
  bool pair = false;
  bool f16 = false;       // A and B are fp16 (else bf16)
  int K = 0;              // inner dimension; every segment has row stride K
  int k_splits = 1;
  int bn = 256;           // 64, 128, 192, 224 or 256
  // Operand that no earlier kernel of the stream writes (the weights): 1 = A,
  // 2 = B, 0 = none. Its first ring stages are loaded before the kernel waits
  // for its predecessor (programmatic dependent launch).
  int const_op = 0;
  Epi epi = Epi::kStore;
  TcEpiArgs e;
};

// 2-D TMA map over a row-major bf16 (or fp16) [rows, cols] matrix: boxes of 64
// columns x box_rows rows, 128-byte swizzle, zero fill out of bounds.
bool make_tma_2d_16b(CUtensorMap* m, const void* ptr, int rows, int cols, int box_rows, bool f16);

cudaError_t launch_tc_gemm(const TcGemmDesc& d, int max_ctas, DevStatus* st, unsigned long long wait_ns,
                           cudaStream_t s, const char** why);

// ---------------------------------------------------------------- post-GEMM kernels (fp32 partial sums in)
// C is [splits][rows][ldc] fp32; each reads the split-sum of its elements.

// Q/K/V from C columns [0, H*d) | [H*d, (H+Hkv)*d) | [.., (H+2Hkv)*d):
// optional per-head RMSNorm (q/k), RoPE at pos, write q[b,h,t_q,:] (Tq rows per
// (b,h)) and k/v at slot `pos` of [b, j, kv_stride, d] (prefill: slot t).
// decode_lens != null: decode mode (seq == 1, pos = decode_lens[b]).
// gate != null: columns [(H+2Hkv)*d, (2H+2Hkv)*d) are the attention gate;
// gate[r, :] = sigmoid(them), fp16 on the bf16 path, fp32 on the fp32 path.
cudaError_t launch_post_qkv(const float* C, int splits, int rows, int ldc, int seq, const int* pos0,
                            const int* decode_lens, int H, int Hkv, int d, int qk_norm, const void* q_gain,
                            const void* k_gain, float eps, const float2* rope, int rope_max_pos, void* q, void* k,
                            void* v, int kv_stride, bool bf16, cudaStream_t s, void* gate = nullptr);

// out[r, c] = resid[r, c] + a[r, c] for c < n, a = sum_s C[s, r, c] (fp32
// sum, stored as fp32 when out_f32, else in the storage type); with g_post,
// a = rmsnorm(sum_s C[s, r, :]) * g_post instead (a sandwich post-norm);
// optional storage-type copy out2 and contribution tap (a); optional fused
// RMSNorm of the new row into y (gain g; y in fp16 when y_f16 on the bf16
// path); optional lens bump (lens[r] += 1 for r < rows). resid is fp32 when
// resid_f32, else the storage type.
cudaError_t launch_post_resid(const float* C, int splits, int rows, int n, int ldc, const void* resid, bool resid_f32,
                              void* out, bool out_f32, void* out2, void* tap, const void* g, float eps, void* y,
                              int* bump_lens, bool bf16, cudaStream_t s, const void* g_post = nullptr,
                              bool y_f16 = false);

// neurons[r, f] = act(C * rs[r]) for f < F; SwiGLU reads gate at column f and up at F + f.
// rs[r] = rsqrt(sum of row_ss[r, 0..ss_parts) / ss_n + ss_eps) (the RMSNorm of the GEMM's
// input rows, applied after the product), or 1 when row_ss is null.
cudaError_t launch_post_act(const float* C, int splits, int rows, int F, int ldc, int act, float alpha_p,
                            float alpha_n, float beta, float xeps, void* out, bool bf16, cudaStream_t s,
                            const float* row_ss = nullptr, int ss_parts = 0, int ss_n = 1, float ss_eps = 0.f);

// ---------------------------------------------------------------- attention
// The attention options of every kernel below: window > 0 limits query i to
// the keys at positions i - window + 1 .. i; gate != null (layout of o, fp16
// on the bf16 kernels, fp32 on the fp32 one) multiplies the output, and
// ungated (bf16 / fp32, layout of o), when set, receives it before the gate;
// key_range (prefill) hides padding keys. A query that sees no key gets a
// zero output.
struct AttnOpts {
  int window = 0;
  const void* gate = nullptr;
  void* ungated = nullptr;
  bool o_f16 = false;            // decode: o in fp16 (else bf16)
  bool counter_zeroed = false;   // decode: an earlier kernel of the stream zeroed the workspace's unit counter
  // decode: when this status word records a timeout, the combine step writes NaN to o (for
  // callers that have no handle to read a status from)
  const DevStatus* poison_on_timeout = nullptr;
  const int2* key_range = nullptr;  // prefill: per sequence, only keys lo <= j < hi are visible
};

// Causal GQA attention; q [B,H,Tq,d], k/v [B,Hkv,kv_stride,d], o [B,Tq,H,d].
// kv_lens null: kv_len = Tq.
cudaError_t launch_attn_f32(const float* q, const float* k, const float* v, float* o, int B, int H, int Hkv, int Tq,
                            int d, int kv_stride, const int* kv_lens, int len_add, cudaStream_t s,
                            const AttnOpts& opt = AttnOpts());

// tcgen05/TMEM flash attention (prefill, causal, kv_len == T, head_dim 128).
// f16: q, k, v are fp16 (else bf16); o_f16: o is fp16 (else bf16).
// With q_off (positions already in a KV cache, per sequence) the T queries of sequence b sit at
// q_off[b] .. q_off[b] + T - 1 and attend to cache rows 0 .. q_off[b] + t of k/v, which hold
// kv_stride rows per (sequence, KV head); without it, kv_stride == T.
cudaError_t launch_attn_prefill_tc(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv, int T,
                                   int d, bool f16, bool o_f16, DevStatus* st, unsigned long long wait_ns,
                                   cudaStream_t s, const char** why, const int* q_off = nullptr,
                                   int kv_stride = 0, const AttnOpts& opt = AttnOpts());

// Decode (Tq == 1), split over the keys: partial results in ws, combined into o.
// The decode attention workspace starts with its unit counter (kAttnCounterBytes,
// an int the attention kernel counts up from 0), then the split partials.
constexpr size_t kAttnCounterBytes = 256;
size_t attn_decode_ws_bytes(int B, int H, int d, int max_splits);
// Keys per sequence: kv_lens[b] + len_add (<= max_len, which sizes the splits; at most
// split_cap of them, the number ws holds); with a window, the last `window` of them.
cudaError_t launch_attn_decode_bf16(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv,
                                    int d, int kv_stride, const int* kv_lens, int len_add, int max_len,
                                    int split_cap, void* ws, int num_sms, DevStatus* st, unsigned long long wait_ns,
                                    cudaStream_t s, const char** why, const AttnOpts& opt = AttnOpts());
// Key splits per (sequence, KV head) of a decode step: units of about 2048 keys, shorter
// when B * Hkv pairs are too few to keep the SMs busy.
int attn_decode_splits(int B, int Hkv, int max_len, int num_sms);
// The splits a workspace holds for keys up to max_len (512-key units, at most 64): the
// bound attn_decode_splits is clamped to, and the allocation-free path's split rule.
int attn_decode_split_cap(int max_len);

// Decode attention with its split partials in a fixed file-scope device array
// (no workspace, no allocation); kv_lens[b] keys per sequence, <= kv_stride.
constexpr size_t kDecodeStaticScratchBytes = 16u << 20;
cudaError_t launch_attn_decode_bf16_static(const void* q, const void* k, const void* v, void* o, int B, int H,
                                           int Hkv, int d, int kv_stride, const int* kv_lens, int num_sms,
                                           unsigned long long wait_ns, cudaStream_t s, const char** why);

}  // namespace blk
