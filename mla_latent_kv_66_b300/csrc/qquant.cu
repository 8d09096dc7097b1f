// E4M3 query of the 8-bit tensor-core decode.
//
// Method (hotdry.top "DeepSeek-V3.2-Exp 中多头潜在注意力的优化", deployment
// paragraph: FP8 quantisation when serving MLA; the format follows the
// cache's own per-token rule): each (b, h) query row of 576 values, q_lat
// (512) then the rotated q_pe (64), becomes E4M3 codes under one fp32 scale
//   scale = max|v| / 448 (1 for an all-zero row),  y = v / scale,
//   hi = E4M3(y),  lo = E4M3(y - value(hi))   (second term optional),
// so that v ~ scale * (value(hi) + value(lo)).  Divisions are IEEE fp32 and
// the E4M3 conversion rounds to nearest even with saturation at 448, so the
// codes are a deterministic function of the bf16 inputs.
//
// Output layout: codes [B, H, 2, 576] (term 0 row, then term 1 row; the
// term-1 row is left untouched for one term), scale [B, H] fp32.
#include <cuda_fp16.h>

#include "kernels.h"
#include "tc.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

__device__ inline uint32_t e4m3x2(float lo, float hi) {  // lo -> byte 0, hi -> byte 1
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ inline float2 e4m3x2_value(uint32_t c) {  // exact: every E4M3 value is an f16
  uint32_t h2;
  const uint16_t c16 = (uint16_t)c;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c16));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// One warp per query row.  Lane l holds latent values [16 l, 16 l + 16) and
// RoPE values [2 l, 2 l + 2).
__global__ void __launch_bounds__(256) quantize_q_kernel(const __nv_bfloat16* __restrict__ q_lat,
                                                         const __nv_bfloat16* __restrict__ q_pe, long long rows,
                                                         int terms, uint8_t* __restrict__ codes,
                                                         float* __restrict__ scale) {
  tc::grid_dep_wait();  // q_lat comes from the preceding kernel on the stream
  tc::grid_dep_trigger();
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(q_lat + row * kLatent) + 2 * lane;
  const uint4 a = src[0], b = src[1];
  const uint32_t pe = reinterpret_cast<const uint32_t*>(q_pe + row * kRope)[lane];
  float v[18];
  const uint32_t w[9] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, pe};
#pragma unroll
  for (int i = 0; i < 9; ++i) {
    v[2 * i] = bf16lo(w[i]);
    v[2 * i + 1] = bf16hi(w[i]);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 18; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  float y[18];
#pragma unroll
  for (int i = 0; i < 18; ++i) y[i] = __fdiv_rn(v[i], s);
  uint32_t hi[9];
#pragma unroll
  for (int i = 0; i < 9; ++i) hi[i] = e4m3x2(y[2 * i], y[2 * i + 1]);
  uint8_t* out = codes + row * (2 * kRow);
  *reinterpret_cast<uint4*>(out + 16 * lane) =
      make_uint4(hi[0] | hi[1] << 16, hi[2] | hi[3] << 16, hi[4] | hi[5] << 16, hi[6] | hi[7] << 16);
  *reinterpret_cast<uint16_t*>(out + kLatent + 2 * lane) = (uint16_t)hi[8];
  if (terms == 2) {
    uint32_t lo[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const float2 h = e4m3x2_value(hi[i]);
      lo[i] = e4m3x2(y[2 * i] - h.x, y[2 * i + 1] - h.y);  // exact differences
    }
    uint8_t* out1 = out + kRow;
    *reinterpret_cast<uint4*>(out1 + 16 * lane) =
        make_uint4(lo[0] | lo[1] << 16, lo[2] | lo[3] << 16, lo[4] | lo[5] << 16, lo[6] | lo[7] << 16);
    *reinterpret_cast<uint16_t*>(out1 + kLatent + 2 * lane) = (uint16_t)lo[8];
  }
  if (lane == 0) scale[row] = s;
}

}  // namespace

cudaError_t launch_quantize_q(const __nv_bfloat16* q_lat, const __nv_bfloat16* q_pe, long long rows, int terms,
                              uint8_t* codes, float* scale, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_dependent(quantize_q_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, q_lat, q_pe, rows, terms,
                          codes, scale);
}

}  // namespace mla
