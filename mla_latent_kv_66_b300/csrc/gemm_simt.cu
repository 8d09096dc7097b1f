// Query absorption and value out-projection on the CUDA cores.
//   q_lat[b,h,:] = W_UK[h]^T q_nope[b,h,:]     out[b,h,:] = W_UV[h] o_lat[b,h,:]
// (the key and value halves of kv_b_proj on the mtrt.cn DeepSeek-Coder-V2
// MLA page, moved off the per-token path by absorption).
#include "common.cuh"
#include "kernels.h"

namespace mla {
namespace {

constexpr int kBChunk = 16;

// grid (H, 4): block = 128 latent columns of one head; loops over batch chunks.
__global__ void __launch_bounds__(128) absorb_simt_kernel(const __nv_bfloat16* __restrict__ q_nope,
                                                          const __nv_bfloat16* __restrict__ w_uk,
                                                          __nv_bfloat16* __restrict__ q_lat, int B, int H) {
  __shared__ float qs[kBChunk][kNope];
  const int h = blockIdx.x, k = blockIdx.y * 128 + threadIdx.x;
  const __nv_bfloat16* w = w_uk + (size_t)h * kNope * kLatent + k;
  for (int b0 = 0; b0 < B; b0 += kBChunk) {
    const int nb = min(kBChunk, B - b0);
    __syncthreads();
    for (int i = threadIdx.x; i < nb * kNope; i += 128) {
      int bb = i / kNope, n = i % kNope;
      qs[bb][n] = __bfloat162float(q_nope[((size_t)(b0 + bb) * H + h) * kNope + n]);
    }
    __syncthreads();
    float acc[kBChunk];
#pragma unroll
    for (int i = 0; i < kBChunk; ++i) acc[i] = 0.f;
    for (int n = 0; n < kNope; ++n) {
      const float wv = __bfloat162float(w[(size_t)n * kLatent]);
#pragma unroll
      for (int i = 0; i < kBChunk; ++i) acc[i] = fmaf(wv, qs[i][n], acc[i]);
    }
    for (int i = 0; i < nb; ++i)
      q_lat[((size_t)(b0 + i) * H + h) * kLatent + k] = __float2bfloat16_rn(acc[i]);
  }
}

// grid (H): 8 warps, warp = 16 value rows; lanes split the 512-long dot.
__global__ void __launch_bounds__(256) out_proj_simt_kernel(const __nv_bfloat16* __restrict__ o_lat,
                                                            const __nv_bfloat16* __restrict__ w_uv,
                                                            void* __restrict__ out, bool out_bf16, int B, int H) {
  __shared__ float os[kBChunk][kLatent];
  const int h = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b0 = 0; b0 < B; b0 += kBChunk) {
    const int nb = min(kBChunk, B - b0);
    __syncthreads();
    for (int i = threadIdx.x; i < kBChunk * kLatent; i += 256) {
      int bb = i / kLatent, k = i % kLatent;
      os[bb][k] = bb < nb ? __bfloat162float(o_lat[((size_t)(b0 + bb) * H + h) * kLatent + k]) : 0.f;
    }
    __syncthreads();
    for (int r = warp; r < kV; r += 8) {
      const __nv_bfloat16* wr = w_uv + ((size_t)h * kV + r) * kLatent;
      float wv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) wv[i] = __bfloat162float(wr[i * 32 + lane]);
      for (int bb = 0; bb < nb; ++bb) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) s = fmaf(wv[i], os[bb][i * 32 + lane], s);
#pragma unroll
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) {
          const size_t idx = ((size_t)(b0 + bb) * H + h) * kV + r;
          if (out_bf16) static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(s);
          else static_cast<float*>(out)[idx] = s;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_absorb_simt(const __nv_bfloat16* q_nope, const __nv_bfloat16* w_uk,
                               __nv_bfloat16* q_lat, int B, int H, cudaStream_t stream) {
  absorb_simt_kernel<<<dim3(H, kLatent / 128), 128, 0, stream>>>(q_nope, w_uk, q_lat, B, H);
  return cudaGetLastError();
}

cudaError_t launch_out_proj_simt(const __nv_bfloat16* o_lat, const __nv_bfloat16* w_uv, void* out,
                                 bool out_bf16, int B, int H, cudaStream_t stream) {
  out_proj_simt_kernel<<<H, 256, 0, stream>>>(o_lat, w_uv, out, out_bf16, B, H);
  return cudaGetLastError();
}

}  // namespace mla
