// Prefill attention on the 5th-generation tensor core (tcgen05 + TMEM), causal,
// grouped-query, head_dim 128 ("LlamaForCausalLM-32L-4096d" sheet: softmax(q @
// k.T / sqrt(128), mask=causal) @ v per head; "arcee", "Grouped-query attention,
// 128-wide heads": query head h reads KV head h / (H / Hkv)).
//
// Work items of two 128-query slots that share every K/V tile: two query heads of
// one KV group at the same query tile (an even group size), or two consecutive
// query tiles of one head (otherwise). Persistent: one CTA per SM walks the items,
// heaviest first, dealt out in a snake order; barrier phases and ring positions run
// on across items, so that the next item's Q, first K/V tiles and first score
// products overlap the current item's last softmax, PV and output store.
// 352 threads:
//   warp 0      TMA producers: lane 0 both slots' Q tiles once, then K tiles of
//               128 keys through a 2-stage ring; lane 1 the V tiles through their
//               own 2-stage ring (128-byte swizzle, 64-column boxes).
//   warps 1, 10 MMA issuers, lane 0 of warp 1 for slot 0 and of warp 10 for slot 1
//               (warp 1 also allocates TMEM): per key tile j, O_g += P_g V_j (A = P
//               from tensor memory, B = V as an MN-major operand) as soon as the
//               slot's P_j is written, then at once S_g = Q_g K_{j+1}^T (M=128,
//               N=128) into the slot's score buffer.
//   warps 2..9  softmax, four warps per slot, one query row per thread: read S_j
//               from TMEM, mask, exponentiate in the log2 domain against a running
//               reference max, and write P_j (fp16 or bf16 pairs) over the first 64
//               columns of the same TMEM buffer; rescale O in TMEM only when the row
//               max grew by more than 2^8 (exact: softmax does not depend on the
//               reference); finally O / l to the head-major output.
// The slots take turns: while one slot's softmax works on its tile, the tensor
// core runs the other slot's PV and next score product. P never touches shared
// memory, so the tensor core's shared-memory reads are Q, K and V alone. The MMAs
// of one thread run in issue order: S_{j+1} of a slot, issued after that slot's
// PV_j, overwrites P_j only once PV_j has read it, and a commit after S_j also
// covers PV_{j-1} (so O is stable whenever S_j is ready).
// Options of the "afmoe" block ("Rotary runs on the sliding-window blocks only";
// "Attention: per-head q/k norms and a sigmoid gate on every head"): a window
// over the last W positions (key tiles before the first query's oldest key are
// skipped, the rest masked), and a per-channel gate on the output; a padded batch
// hides the keys outside each sequence's run of real tokens.
// Every wait is bounded; on expiry the CTA records a timeout, drains its own
// copies and MMAs, frees its TMEM and returns.
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

constexpr int kD = 128;
constexpr int kBQ = 128;                    // queries per slot (MMA M)
constexpr int kBK = 128;                    // keys per tile
constexpr int kSlots = 2;
constexpr int kThreads = 64 + kSlots * 128 + 32;  // + warp 10: the second slot's MMA issuer
constexpr int kQSub = kBQ * 128;            // one 64-column half of a Q tile (bytes)
constexpr int kQBytes = 2 * kQSub;          // 128 queries x 128 dims
constexpr int kKVSub = kBK * 128;           // one 64-column half of a K or V tile
constexpr int kKVBytes = 2 * kKVSub;        // 128 keys x 128 dims
constexpr int kKStages = 2;                 // K ring
constexpr int kVStages = 2;                 // V ring
constexpr int kSmem = 1024 + kSlots * kQBytes + (kKStages + kVStages) * kKVBytes + 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr unsigned long long kDrainNs = 2000000000ULL;
constexpr float kLog2e = 1.4426950408889634f;
static_assert(kSmem <= 227 * 1024, "shared memory");
static_assert(kQSub == kKVSub && kKStages == 2 && kVStages == 2, "the MMA issuers' descriptor steps and stage selects");

struct AttnParams {
  CUtensorMap tq, tk, tv;
  void* o;
  int o_f16;
  int B, H, Hkv, T, n_qtiles;
  int head_pairs;  // 1: the two slots are heads 2i, 2i+1 at one query tile; 0: query tiles 2k, 2k+1 of one head
  int n_items;
  // K/V rows per (sequence, KV head): T, or a cache's capacity; q_off: positions already
  // in that cache per sequence (the T queries sit at q_off[b] ..), or null for 0
  int kv_stride;
  const int* q_off;
  // "afmoe": window > 0 keeps the keys at positions > query - window; gate (fp16, the
  // output's layout) multiplies the output, ungated (bf16) receives it before the gate
  int window;
  const __half* gate;
  __nv_bfloat16* ungated;
  const int2* key_range;  // per sequence [lo, hi): the visible (non-padding) keys, or null
  float sl2;
  DevStatus* status;
  unsigned long long wait_ns;
};

// 2^x on the MUFU unit (one instruction; -inf gives +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Blackwell's packed fp32 arithmetic: two lanes of fp32 in one 64-bit register pair,
// one instruction for both (each lane rounded as its scalar form would be).
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2_make(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three (one instruction; like fmaxf, a NaN operand is ignored)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool f16) {
  if (f16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  return pack_bf16x2(lo, hi);
}

// D[tmem] (+)= A[tmem] * B[smem desc]: the A operand (M rows on the TMEM lanes, K
// 16-bit elements packed two per 32-bit column) read from tensor memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct Slot {
  int h, qt, m0, valid;
};

// A work item: two slots over one KV head of one sequence, and its key-tile range.
struct Item {
  Slot sl[kSlots];
  int b, kv_row, off, kv_lo, kv_hi, n_keys, t0, n_tiles;
};

// Item id, heaviest first: the far query tiles (more keys) get the small ids. Reads
// the cache positions and key ranges, so it runs after pdl_wait.
__device__ __forceinline__ Item item_of(const AttnParams& p, int id) {
  Item it;
  if (p.head_pairs) {
    const int hp_n = p.H / 2;
    const int qt = p.n_qtiles - 1 - id / (p.B * hp_n);
    const int r = id % (p.B * hp_n);
    const int hp = r % hp_n;
    it.b = r / hp_n;
#pragma unroll
    for (int g = 0; g < kSlots; ++g) it.sl[g] = {2 * hp + g, qt, qt * kBQ, 1};
  } else {
    const int np = (p.n_qtiles + 1) / 2;
    const int k = np - 1 - id / (p.B * p.H);
    const int r = id % (p.B * p.H);
    const int h = r % p.H;
    it.b = r / p.H;
#pragma unroll
    for (int g = 0; g < kSlots; ++g) {
      const int qt = 2 * k + g;
      const int ok = qt < p.n_qtiles;
      it.sl[g] = {h, ok ? qt : 2 * k, (ok ? qt : 2 * k) * kBQ, ok};
    }
  }
  const int kvh = it.sl[0].h / (p.H / p.Hkv);
  it.kv_row = (it.b * p.Hkv + kvh) * p.kv_stride;
  it.off = p.q_off ? p.q_off[it.b] : 0;  // keys 0 .. off - 1 are earlier positions in the cache
  // visible keys: [kv_lo, kv_hi) (an attention_mask's run of real tokens, else all)
  const int2 kr = p.key_range ? p.key_range[it.b] : make_int2(0, it.off + p.T);
  it.kv_lo = kr.x;
  it.kv_hi = kr.y;
  // the key tiles the item needs: the union of both slots' ranges
  int n_keys = 0, first_key = 1 << 30;
#pragma unroll
  for (int g = 0; g < kSlots; ++g) {
    const int kv_end = min(p.T, it.sl[g].m0 + kBQ);
    n_keys = max(n_keys, min(it.off + kv_end, it.kv_hi));
    first_key = min(first_key, max(it.kv_lo, p.window > 0 ? it.off + it.sl[g].m0 - p.window + 1 : 0));
  }
  it.n_keys = n_keys;
  it.t0 = max(0, first_key) / kBK;
  it.n_tiles = max(0, (n_keys + kBK - 1) / kBK - it.t0);  // none when every query is padding
  return it;
}

// Round k of CTA c among G: the heaviest-first ids dealt out in a snake (c, then
// 2G - 1 - c, ...), so that every CTA's rounds sum to about the same work.
__device__ __forceinline__ int item_id(int k, int G, int c) { return k * G + ((k & 1) ? G - 1 - c : c); }

// F16: q, k, v (and so P) are fp16; otherwise bf16. Persistent: CTA c runs items
// item_id(0, G, c), item_id(1, G, c), ... Barrier phases and ring positions run on
// across items, so that the next item's Q, first K/V tiles and first score products
// overlap the current item's last softmax, PV and output store.
template <bool F16>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnParams p) {
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                   // [slot]: two 64-column halves of 16 KB
  uint8_t* sK = sQ + kSlots * kQBytes;                  // [stage]: two halves of 16 KB
  uint8_t* sV = sK + kKStages * kKVBytes;               // [stage]: two halves of 16 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kVStages * kKVBytes);
  // q_full, q_empty, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_ready[2][4],
  // o_done[2], o_free[2], drain[2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 26);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  const uint32_t q_full = smem_u32(&bars[0]);
  const uint32_t q_empty = smem_u32(&bars[1]);
  auto k_full = [&](int s) { return smem_u32(&bars[2 + s]); };
  auto k_empty = [&](int s) { return smem_u32(&bars[4 + s]); };
  auto v_full = [&](int s) { return smem_u32(&bars[6 + s]); };
  auto v_empty = [&](int s) { return smem_u32(&bars[8 + s]); };
  auto s_full = [&](int g) { return smem_u32(&bars[10 + g]); };
  // P is released in quarters of 32 keys, each on its own barrier (one phase per tile):
  // the PV steps of a quarter run while the softmax computes the next quarter
  auto p_ready = [&](int g, int q) { return smem_u32(&bars[12 + 4 * g + q]); };
  auto o_done = [&](int g) { return smem_u32(&bars[20 + g]); };
  auto o_free = [&](int g) { return smem_u32(&bars[22 + g]); };
  auto drain = [&](int g) { return smem_u32(&bars[24 + g]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long budget = p.wait_ns;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, kSlots);  // one commit from each slot's MMA issuer after its item's last S
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), kSlots);  // one commit from each slot's MMA issuer
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), kSlots);
    }
    for (int g = 0; g < kSlots; ++g) {
      mbar_init(s_full(g), 1);
      for (int q = 0; q < 4; ++q) mbar_init(p_ready(g, q), 128);
      mbar_init(o_done(g), 1);
      mbar_init(o_free(g), 128);  // the slot's softmax threads, once they have read O out
      mbar_init(drain(g), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tq);
    tma_prefetch_desc(&p.tk);
    tma_prefetch_desc(&p.tv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // q, k, v (and the cache positions, the key ranges) come from earlier kernels
  const uint32_t tmem = *tmem_holder;  // S[g] (and P[g] over its first 64 columns): cols 128 g; O[g]: 256 + 128 g
  // What the producer lanes and the MMA lanes have in flight, for the drain after an
  // abort: the ring stages issued (with the parity of their last phase), the last Q
  // load's parity, and whether any MMA was issued.
  uint32_t issued = 0, parity = 0, q_parity = 0;
  bool q_issued = false, mma_issued = false;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: each item's Q, then its K tiles through the ring
      bool failed = false;
      int J = 0;  // K tiles issued over all items
      for (int k = 0; !failed; ++k) {
        const int id = item_id(k, G, cta);
        if (id >= p.n_items) break;
        const Item it = item_of(p, id);
        // the Q buffer is free once both slots' score products of the previous item are done
        if (!mbar_wait(q_empty, (k & 1) ^ 1, budget, abort_flag)) {
          failed = true;
          break;
        }
        mbar_arrive_expect_tx(q_full, kSlots * kQBytes);
#pragma unroll
        for (int g = 0; g < kSlots; ++g) {
          const int q_row = (it.b * p.H + it.sl[g].h) * p.T + it.sl[g].m0;
          tma_load_2d(smem_u32(sQ + g * kQBytes), &p.tq, 0, q_row, q_full);
          tma_load_2d(smem_u32(sQ + g * kQBytes + kQSub), &p.tq, 64, q_row, q_full);
        }
        q_issued = true;
        q_parity = k & 1;
        for (int j = 0; j < it.n_tiles; ++j, ++J) {
          const int s = J % kKStages;
          const uint32_t ph = (J / kKStages) & 1;
          if (!mbar_wait(k_empty(s), ph ^ 1, budget, abort_flag)) {
            failed = true;
            break;
          }
          mbar_arrive_expect_tx(k_full(s), kKVBytes);
          const int row = it.kv_row + (it.t0 + j) * kBK;
          tma_load_2d(smem_u32(sK + s * kKVBytes), &p.tk, 0, row, k_full(s));
          tma_load_2d(smem_u32(sK + s * kKVBytes + kKVSub), &p.tk, 64, row, k_full(s));
          issued |= 1u << s;
          parity = (parity & ~(1u << s)) | (ph << s);
        }
      }
      if (failed) {  // the loads in flight are drained after the CTA's final barrier
        *abort_flag = 1;
        report_timeout(p.status, 0x20 + 0);
      }
    } else if (lane == 1) {
      // ---------------- TMA producer: the V ring (its own thread, so that K never waits behind V)
      bool failed = false;
      int J = 0;
      for (int k = 0; !failed; ++k) {
        const int id = item_id(k, G, cta);
        if (id >= p.n_items) break;
        const Item it = item_of(p, id);
        for (int j = 0; j < it.n_tiles; ++j, ++J) {
          const int s = J % kVStages;
          const uint32_t ph = (J / kVStages) & 1;
          if (!mbar_wait(v_empty(s), ph ^ 1, budget, abort_flag)) {
            failed = true;
            break;
          }
          mbar_arrive_expect_tx(v_full(s), kKVBytes);
          const int row = it.kv_row + (it.t0 + j) * kBK;
          tma_load_2d(smem_u32(sV + s * kKVBytes), &p.tv, 0, row, v_full(s));
          tma_load_2d(smem_u32(sV + s * kKVBytes + kKVSub), &p.tv, 64, row, v_full(s));
          issued |= 1u << s;
          parity = (parity & ~(1u << s)) | (ph << s);
        }
      }
      if (failed) {
        *abort_flag = 1;
        report_timeout(p.status, 0x20 + 3);
      }
    }
  } else if (warp == 1 || warp == kThreads / 32 - 1) {
    if (lane == 0) {
      // ---------------- MMA issuer of slot g (warp 1: slot 0, the last warp: slot 1). Each
      // slot has its own issuing thread, so that a slot whose P is ready never waits
      // behind the other slot's waits and commits: its PV queues on the tensor pipe at once.
      const int g = warp == 1 ? 0 : 1;
      // kind::f16 operand formats: bf16 (1) or fp16 (0) for both A and B
      constexpr uint32_t fmt_clear = F16 ? ~((7u << 7) | (7u << 10)) : ~0u;
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBQ, kBK) & fmt_clear;
      constexpr uint32_t idesc_pv = (idesc_bf16_f32(kBQ, kD) & fmt_clear) | (1u << 16);  // B (V) is MN-major
      // Shared-memory descriptors, built once: a descriptor's start-address field counts
      // 16-byte units, so K step kk of a 128-byte-swizzled operand sits (kk / 4) halves of
      // 16 KB and (kk % 4) 32-byte steps further; V's 16-key steps are 2 KB apart.
      const uint64_t dq = smem_desc_sw128(smem_u32(sQ + g * kQBytes));
      uint64_t dk[kKStages], dv[kVStages];
#pragma unroll
      for (int st = 0; st < kKStages; ++st) dk[st] = smem_desc_sw128(smem_u32(sK + st * kKVBytes));
#pragma unroll
      for (int st = 0; st < kVStages; ++st) dv[st] = smem_desc_sw128_mn(smem_u32(sV + st * kKVBytes), kKVSub, 1024);
      auto kstep = [](int kk) { return (uint64_t)((kk >> 2) * (kQSub >> 4) + (kk & 3) * 2); };
      const uint32_t s_tmem = tmem + g * kBK, o_tmem = tmem + 256 + g * kD;
      auto issue_s = [&](int J) {  // S of global tile J (K stage J % 2) into the slot's score buffer
        const int s = J % kKStages;
        const uint64_t dks = s == 0 ? dk[0] : dk[1];
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) tc_mma_bf16(s_tmem, dq + kstep(kk), dks + kstep(kk), idesc_s, kk > 0 ? 1u : 0u);
        tc_commit(s_full(g));
        tc_commit(k_empty(s));  // this slot is done with the K stage once this S is
        mma_issued = true;
      };
      bool failed = false;
      int J = 0;  // tiles over all items
      for (int k = 0; !failed; ++k) {
        const int id = item_id(k, G, cta);
        if (id >= p.n_items) break;
        const Item it = item_of(p, id);
        if (!mbar_wait(q_full, k & 1, budget, abort_flag)) {
          failed = true;
          break;
        }
        if (it.n_tiles > 0) {
          if (!mbar_wait(k_full(J % kKStages), (J / kKStages) & 1, budget, abort_flag)) {
            failed = true;
            break;
          }
          tc_fence_after();
          issue_s(J);
        }
        if (it.n_tiles <= 1) tc_commit(q_empty);  // no further score product of this item reads Q
        for (int j = 0; j < it.n_tiles; ++j, ++J) {
          // PV_j as soon as V_j has landed, O is free (the previous item's output read out)
          // and each quarter of P_j is in tensor memory ...
          const int vs = J % kVStages;
          if (!mbar_wait(v_full(vs), (J / kVStages) & 1, budget, abort_flag) ||
              (j == 0 && k >= 1 && !mbar_wait(o_free(g), (k - 1) & 1, budget, abort_flag))) {
            failed = true;
            break;
          }
          const uint64_t dvs = vs == 0 ? dv[0] : dv[1];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (!mbar_wait(p_ready(g, q), J & 1, budget, abort_flag)) {
              failed = true;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 2 * q; kk < 2 * q + 2; ++kk)
              tc_mma_ts(o_tmem, s_tmem + kk * 8, dvs + (uint64_t)(kk * (16 * 128 >> 4)), idesc_pv,
                        (j > 0 || kk > 0) ? 1u : 0u);
          }
          if (failed) break;
          tc_commit(v_empty(vs));  // this slot is done with the V stage once PV_j is
          // ... then S_{j+1}, which overwrites P_j after PV_j has read it (issue order)
          if (j + 1 < it.n_tiles) {
            if (!mbar_wait(k_full((J + 1) % kKStages), ((J + 1) / kKStages) & 1, budget, abort_flag)) {
              failed = true;
              break;
            }
            tc_fence_after();
            issue_s(J + 1);
            if (j + 2 == it.n_tiles) tc_commit(q_empty);  // that was the item's last score product
          }
        }
        if (failed) break;
        // An item without key tiles has no PV that waited for the previous item's O to be
        // read out: wait here, so that o_done runs at most one phase ahead of its waiter.
        if (it.n_tiles == 0 && k >= 1 && !mbar_wait(o_free(g), (k - 1) & 1, budget, abort_flag)) {
          failed = true;
          break;
        }
        tc_commit(o_done(g));  // every PV of the slot's item is complete
      }
      if (failed) {  // the MMAs in flight are drained after the CTA's final barrier
        *abort_flag = 1;
        report_timeout(p.status, 0x20 + 1);
      }
    }
  } else {
    // ---------------- softmax / correction / epilogue: slot g, one query row per thread
    const int g = (warp - 2) / 4;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_taddr = tmem + lane_off + g * kBK;
    const uint32_t o_taddr = tmem + lane_off + 256 + g * kD;
    bool failed = false;
    int J = 0;  // tiles over all items
    for (int k = 0; !failed; ++k) {
      const int id = item_id(k, G, cta);
      if (id >= p.n_items) break;
      const Item it = item_of(p, id);
      const Slot me = g == 0 ? it.sl[0] : it.sl[1];  // a select, not a run-time index into local memory
      const int m0 = me.m0;
      const int qi = m0 + r;
      const int qc = min(qi, p.T - 1);
      const int off = it.off, kv_lo = it.kv_lo, kv_hi = it.kv_hi, n_keys = it.n_keys;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < it.n_tiles; ++j, ++J) {
        // The slots take turns (slot 0 tile J, slot 1 tile J, slot 0 tile J + 1, ...): each
        // softmax runs alone on the SM's exponential units while the tensor core works on
        // the other slot's PV and next scores. Slot 1 starts tile J once slot 0's P_J is
        // written, slot 0 starts tile J + 1 once slot 1's P_J is.
        if (g == 1 || J >= 1) {
          if (!__all_sync(0xffffffffu, mbar_wait(p_ready(1 - g, 3), (g == 1 ? J : J - 1) & 1, budget, abort_flag))) {
            failed = true;
            break;
          }
        }
        // warp-uniform: every lane waits, the warp gives up together. S_J ready also means
        // that this slot's PV_{J-1} is done: O is stable and the P buffer free
        if (!__all_sync(0xffffffffu, mbar_wait(s_full(g), J & 1, budget, abort_flag))) {
          failed = true;
          break;
        }
        __syncwarp();
        tc_fence_after();
        float x[kBK];
#pragma unroll
        for (int c = 0; c < kBK; c += 16) tmem_ld16(s_taddr + c, *reinterpret_cast<float(*)[16]>(&x[c]));
        tc_wait_ld();
        const int n0 = (it.t0 + j) * kBK;
        // raw scores: masked entries become -inf (tiles on the diagonal, past the last key,
        // before the first visible key, or before the window)
        if ((n0 + kBK - 1 > off + m0) || (n0 + kBK > kv_hi) || n0 < kv_lo ||
            (p.window > 0 && n0 < off + min(m0 + kBQ - 1, p.T - 1) - p.window + 1)) {
          const int causal = off + qc - n0;                    // keys n0 + c with c <= causal are not ahead
          const int lim = min(causal, kv_hi - 1 - n0);         // ... nor padding after the run
          const int first = max(p.window > 0 ? causal - p.window + 1 : -kBK, kv_lo - n0);  // c >= first
#pragma unroll
          for (int c = 0; c < kBK; ++c)
            if (c > lim || c < first) x[c] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = x[i];
#pragma unroll
        for (int c = 8; c < kBK; c += 2) mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], x[c], x[c + 1]);
        const float mraw = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float mt = mraw * p.sl2;  // the scale is positive: the max commutes with it
        const bool need = mt > m_ref + kRescaleLog2;
        const bool any = __any_sync(0xffffffffu, need);
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m_ref - mt);
          m_ref = mt;
        }
        const float neg_mu = m_ref == -INFINITY ? 0.f : -m_ref;
        if (j >= 1 && any) {  // PV_{J-1} is done (see above): rescale this warp's O rows
#pragma unroll 1
          for (int c = 0; c < kD; c += 16) {
            float ov[16];
            tmem_ld16(o_taddr + c, ov);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] *= alpha;
            tmem_st16(o_taddr + c, ov);
          }
        }
        if (n0 + kBK > n_keys) {
          // V rows past the item's last key may hold anything (unused cache slots): zero them,
          // so that P = 0 meets finite values, once the tile has landed. Both slots write the
          // same zeros, each before its own p_ready (the fence below), as either slot's PV
          // may run first
          const int vs = J % kVStages;
          if (!__all_sync(0xffffffffu, mbar_wait(v_full(vs), (J / kVStages) & 1, budget, abort_flag))) {
            failed = true;
            break;
          }
          if (r >= n_keys - n0) {
            uint8_t* vrow = sV + vs * kKVBytes + r * 128;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb)
#pragma unroll
              for (int c16 = 0; c16 < 8; ++c16) *reinterpret_cast<uint4*>(vrow + hb * kKVSub + c16 * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        // P row r into tensor memory over the scores it came from: 64 columns of element
        // pairs (keys 2c, 2c + 1 in column c), a quarter (16 columns) at a time. Keys 2c and
        // 2c + 1 go as one packed pair through the scale and shift and the row sum. A
        // quarter is released to the PV steps once its store has landed, which the warp
        // waits for only after computing the next quarter.
        const f32x2 sl2x2 = f2_make(p.sl2, p.sl2), mu2 = f2_make(neg_mu, neg_mu);
        f32x2 ls2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
        float w[2][16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = q4 * 32 + 2 * i;
            float t0, t1;
            f2_split(f2_fma(f2_make(x[c], x[c + 1]), sl2x2, mu2), t0, t1);
            const float p0 = ex2_approx(t0);
            const float p1 = ex2_approx(t1);
            ls2[i & 1] = f2_add(ls2[i & 1], f2_make(p0, p1));
            w[q4 & 1][i] = __uint_as_float(pack2(p0, p1, F16));
          }
          if (q4 >= 1) {
            tc_wait_st();  // quarter q4 - 1 of P (and a rescaled O) in tensor memory before its PV steps
            tc_fence_before();
            mbar_arrive(p_ready(g, q4 - 1));
          }
          tmem_st16(s_taddr + q4 * 16, w[q4 & 1]);
        }
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(p_ready(g, 3));
        float ls[4];
        f2_split(ls2[0], ls[0], ls[1]);
        f2_split(ls2[1], ls[2], ls[3]);
        l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      }
      if (failed) break;
      // the slot's last PV of this item is complete (every item commits, with tiles or not)
      if (!__all_sync(0xffffffffu, mbar_wait(o_done(g), k & 1, budget, abort_flag))) {
        failed = true;
        break;
      }
      __syncwarp();
      tc_fence_after();
      const bool seen = l > 0.f;  // false: a padding query that sees no key (its output is 0)
      const float inv = seen ? 1.f / l : 0.f;
      const size_t orow_i = (((size_t)it.b * p.T + qi) * p.H + me.h) * kD;
      uint16_t* orow = static_cast<uint16_t*>(p.o) + orow_i;
      const bool of16 = p.o_f16 != 0;
      const bool store = me.valid && qi < p.T;
      auto pack16 = [](const float (&v)[16], bool f16, uint4& w0, uint4& w1) {
        w0 = make_uint4(pack2(v[0], v[1], f16), pack2(v[2], v[3], f16), pack2(v[4], v[5], f16),
                        pack2(v[6], v[7], f16));
        w1 = make_uint4(pack2(v[8], v[9], f16), pack2(v[10], v[11], f16), pack2(v[12], v[13], f16),
                        pack2(v[14], v[15], f16));
      };
#pragma unroll 1
      for (int c = 0; c < kD; c += 16) {
        float ov[16];
        tmem_ld16(o_taddr + c, ov);
        tc_wait_ld();
        if (store) {
#pragma unroll
          for (int i = 0; i < 16; ++i) ov[i] = seen ? ov[i] * inv : 0.f;
          uint4 w0, w1;
          if (p.ungated) {  // the head outputs before the gate (bf16)
            pack16(ov, false, w0, w1);
            reinterpret_cast<uint4*>(p.ungated + orow_i + c)[0] = w0;
            reinterpret_cast<uint4*>(p.ungated + orow_i + c)[1] = w1;
          }
          if (p.gate) {
            const uint4* g4 = reinterpret_cast<const uint4*>(p.gate + orow_i + c);
            const uint4 ga = g4[0], gb = g4[1];
            const uint32_t gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 gf = __half22float2(*reinterpret_cast<const __half2*>(&gw[i]));
              ov[2 * i] *= gf.x;
              ov[2 * i + 1] *= gf.y;
            }
          }
          pack16(ov, of16, w0, w1);
          reinterpret_cast<uint4*>(orow + c)[0] = w0;
          reinterpret_cast<uint4*>(orow + c)[1] = w1;
        }
      }
      tc_fence_before();
      mbar_arrive(o_free(g));  // O is read out: the next item's first PV may overwrite it
    }
    if (failed) {
      *abort_flag = 1;
      if (lane == 0) report_timeout(p.status, 0x20 + 2);
    }
  }

  tc_fence_before();
  __syncthreads();
  // Every role has stopped issuing. After an abort (a wait that ran out anywhere in
  // the CTA), copies and MMAs that no role waited for may still be in flight: they
  // complete before TMEM is freed and the CTA exits. Every thread reads the same flag.
  if (*abort_flag) {
    volatile int never = 0;
    if (warp == 0 && lane == 0) {
      if (q_issued) mbar_wait(q_full, q_parity, kDrainNs, &never);
      for (int s = 0; s < kKStages; ++s)
        if (issued & (1u << s)) mbar_wait(k_full(s), (parity >> s) & 1, kDrainNs, &never);
    } else if (warp == 0 && lane == 1) {
      for (int s = 0; s < kVStages; ++s)
        if (issued & (1u << s)) mbar_wait(v_full(s), (parity >> s) & 1, kDrainNs, &never);
    } else if ((warp == 1 || warp == kThreads / 32 - 1) && lane == 0 && mma_issued) {
      const int g = warp == 1 ? 0 : 1;
      tc_commit(drain(g));
      mbar_wait(drain(g), 0, kDrainNs, &never);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_attn_prefill_tc(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv, int T,
                                   int d, bool f16, bool o_f16, DevStatus* st, unsigned long long wait_ns,
                                   cudaStream_t s, const char** why, const int* q_off, int kv_stride,
                                   const AttnOpts& opt) {
  if (d != kD) {
    *why = "tcgen05 attention: head_dim must be 128";
    return cudaErrorInvalidValue;
  }
  if (B <= 0 || T <= 0) return cudaSuccess;
  if (kv_stride <= 0) kv_stride = T;
  if (!q_off && kv_stride != T) {
    *why = "tcgen05 attention: K/V rows per head differ from T only with cache positions";
    return cudaErrorInvalidValue;
  }
  AttnParams p;
  memset(static_cast<void*>(&p), 0, sizeof(p));
  if (!make_tma_2d_16b(&p.tq, q, B * H * T, kD, kBQ, f16) ||
      !make_tma_2d_16b(&p.tk, k, B * Hkv * kv_stride, kD, kBK, f16) ||
      !make_tma_2d_16b(&p.tv, v, B * Hkv * kv_stride, kD, kBK, f16)) {
    *why = "cuTensorMapEncodeTiled failed for q/k/v";
    return cudaErrorInvalidValue;
  }
  p.o = o;
  p.o_f16 = o_f16 ? 1 : 0;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.T = T;
  p.kv_stride = kv_stride;
  p.q_off = q_off;
  p.window = opt.window > 0 ? opt.window : 0;
  p.key_range = opt.key_range;
  p.gate = static_cast<const __half*>(opt.gate);
  p.ungated = static_cast<__nv_bfloat16*>(opt.ungated);
  p.n_qtiles = (T + kBQ - 1) / kBQ;
  p.head_pairs = (H / Hkv) % 2 == 0 ? 1 : 0;
  p.n_items = p.head_pairs ? B * (H / 2) * p.n_qtiles : B * H * ((p.n_qtiles + 1) / 2);
  p.sl2 = kLog2e / sqrtf((float)kD);
  p.status = st;
  p.wait_ns = wait_ns;
  static std::atomic<unsigned long long> configured[2];  // per instantiation, one bit per device
  cudaError_t ce = f16 ? set_smem_limit_once(reinterpret_cast<const void*>(attn_tc_kernel<true>), kSmem, configured[1])
                       : set_smem_limit_once(reinterpret_cast<const void*>(attn_tc_kernel<false>), kSmem, configured[0]);
  if (ce != cudaSuccess) return ce;
  // persistent: one CTA per SM (at most one per item) walks the items
  int dev = 0, sms = 0;
  ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce != cudaSuccess) return ce;
  const int grid = std::min(p.n_items, sms);
  if (f16)
    launch_pdl(attn_tc_kernel<true>, grid, kThreads, kSmem, s, p);
  else
    launch_pdl(attn_tc_kernel<false>, grid, kThreads, kSmem, s, p);
  return cudaGetLastError();
}

}  // namespace blk
