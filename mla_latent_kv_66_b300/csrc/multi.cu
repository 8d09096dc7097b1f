// Several query tokens per sequence (speculative / multi-token decode).
//
// Method (mtrt.cn DeepSeek-Coder-V2 MLA page, forward flow, applied to every
// new token; the hotdry.top MoA page mentions multi-token prediction): the
// T newest tokens of a sequence of n cached tokens are the queries, token i
// at position n - T + i, and attends to cache tokens 0 .. n - T + i (causal
// mask).  That is exactly the one-token decode of a sequence of length
// n - T + 1 + i over the same pages, so the expansion below turns each
// sequence into T such rows; the absorption, decode, combine and
// out-projection then run on B*T rows unchanged (the query RoPE too: it
// rotates row r at its length minus one).
#include "kernels.h"

namespace mla {
namespace {

// One thread per (row, page-table column): row r = b*T + i copies page-table
// row b; column 0 also writes the row's length.
__global__ void multi_token_expand_kernel(const int32_t* __restrict__ page_table, const int32_t* __restrict__ seq_lens,
                                          int B, int T, int maxp, int32_t* __restrict__ table_out,
                                          int32_t* __restrict__ lens_out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long rows = (long long)B * T;
  if (idx >= rows * maxp) return;
  const long long r = idx / maxp;
  const int col = (int)(idx % maxp);
  const int b = (int)(r / T), i = (int)(r % T);
  table_out[idx] = page_table[(size_t)b * maxp + col];
  if (col == 0) lens_out[r] = seq_lens[b] - T + 1 + i;  // < 1 when n < T: rejected by the decode
}

}  // namespace

cudaError_t launch_multi_token_expand(const int32_t* page_table, const int32_t* seq_lens, int B, int T, int maxp,
                                      int32_t* table_out, int32_t* lens_out, cudaStream_t stream) {
  const long long n = (long long)B * T * maxp;
  if (n == 0) return cudaSuccess;
  multi_token_expand_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(page_table, seq_lens, B, T, maxp,
                                                                             table_out, lens_out);
  return cudaGetLastError();
}

}  // namespace mla
