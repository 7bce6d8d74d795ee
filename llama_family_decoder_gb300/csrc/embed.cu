// Token-level inputs of the block and the model.
//  * Token embedding lookup ("LlamaForCausalLM-32L-4096d" sheet, "Implementing
//    it": embed_tokens): x[r, :] = embed[tokens[r], :]. HBM-bound: each row is
//    copied with 128-bit loads and stores. An id outside [0, vocab) gives a zero
//    row and records INVALID_ARG in the status word.
//  * The padding run of an attention_mask row ("arcee", "The API": zeros are
//    padding): [lo, hi) of its ones, and the rotary offset -lo of the row.
#include "common.cuh"
#include "kernels.h"

namespace blk {

namespace {

constexpr int kStatusInvalidArg = 1;  // == BLK_ERR_INVALID_ARG

__global__ void embed_kernel(const int* __restrict__ tokens, const uint4* __restrict__ table, int rows,
                             int row_vecs, int vocab, uint4* __restrict__ out, DevStatus* st) {
  pdl_launch_dependents();
  pdl_wait();
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const int id = tokens[r];
    const bool ok = id >= 0 && id < vocab;
    if (!ok && threadIdx.x == 0 && st) atomicCAS(&st->code, 0, kStatusInvalidArg);
    const uint4* src = table + (size_t)(ok ? id : 0) * row_vecs;
    uint4* dst = out + (size_t)r * row_vecs;
    for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) dst[i] = ok ? src[i] : make_uint4(0, 0, 0, 0);
  }
}

// One CTA per sequence: the first and last one of mask row b and their count.
__global__ void mask_ranges_kernel(const int* __restrict__ mask, int T, int2* __restrict__ ranges,
                                   int* __restrict__ pos0, DevStatus* st) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int s_lo, s_hi, s_cnt;
  if (threadIdx.x == 0) {
    s_lo = T;
    s_hi = -1;
    s_cnt = 0;
  }
  __syncthreads();
  const int* row = mask + (size_t)blockIdx.x * T;
  int lo = T, hi = -1, cnt = 0;
  for (int t = threadIdx.x; t < T; t += blockDim.x)
    if (row[t] != 0) {
      lo = min(lo, t);
      hi = max(hi, t);
      ++cnt;
    }
  if (cnt) {
    atomicMin(&s_lo, lo);
    atomicMax(&s_hi, hi);
    atomicAdd(&s_cnt, cnt);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int a = s_lo, b = s_hi + 1;
    if (s_cnt == 0) a = b = T;                                  // a row of padding only
    if (s_cnt != b - a && st) atomicCAS(&st->code, 0, kStatusInvalidArg);  // a hole: its hull is used
    ranges[blockIdx.x] = make_int2(a, b);
    pos0[blockIdx.x] = -a;
  }
}

}  // namespace

cudaError_t launch_mask_ranges(const int* mask, int B, int T, int2* ranges, int* pos0, DevStatus* st,
                               cudaStream_t s) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  launch_pdl(mask_ranges_kernel, B, 256, 0, s, mask, T, ranges, pos0, st);
  return cudaGetLastError();
}

cudaError_t launch_embed(const int* tokens, const void* table, int rows, int row_bytes, int vocab, void* out,
                         DevStatus* st, int num_sms, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (row_bytes % 16) return cudaErrorInvalidValue;
  const int grid = rows < num_sms * 8 ? rows : num_sms * 8;
  launch_pdl(embed_kernel, grid, 128, 0, s, tokens, static_cast<const uint4*>(table), rows, row_bytes / 16, vocab,
             static_cast<uint4*>(out), st);
  return cudaGetLastError();
}

}  // namespace blk
