// Token embedding lookup ("LlamaForCausalLM-32L-4096d" sheet, "Implementing it":
// embed_tokens): x[r, :] = embed[tokens[r], :]. HBM-bound: each row is copied
// with 128-bit loads and stores. An id outside [0, vocab) gives a zero row and
// records INVALID_ARG in the status word.
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

}  // namespace

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
