// Cache write (RMSNorm on the latent, RoPE on k_pe, optional E4M3 with a
// per-token scale) and query RoPE.
//
// Method (mtrt.cn DeepSeek-Coder-V2 MLA page, forward flow): the KV
// down-projection row is split into a 512-d latent and a 64-d k_pe, the
// latent is RMS-normalised, only k_pe is rotated, and both are cached.
#include "common.cuh"
#include "kernels.h"

namespace mla {
namespace {

// Rotation of pair (x_i, x_{i+32}) at position pos: angle pos * 10000^(-i/32),
// in double precision so that long-context positions keep full accuracy.
__device__ inline void rope_pair(float x1, float x2, int i, long long pos, double* y1, double* y2) {
  const double inv_freq = pow(10000.0, -(double)i / 32.0);
  const double ang = (double)pos * inv_freq;
  double s, c;
  sincos(ang, &s, &c);
  *y1 = (double)x1 * c - (double)x2 * s;
  *y2 = (double)x2 * c + (double)x1 * s;
}

// One warp per token row.  Lane l holds latent values 16l..16l+15 and the
// RoPE pair (l, l+32).
__global__ void __launch_bounds__(256) cache_append_kernel(const __nv_bfloat16* __restrict__ rows,
                                                           const int32_t* __restrict__ slots,
                                                           const int32_t* __restrict__ pos, int T,
                                                           int flags, bool fp8, long long num_slots,
                                                           void* ckv, void* kpe, float* scale) {
  const int lane = threadIdx.x & 31;
  const long long t = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const long long slot = slots[t];
  if (slot < 0 || slot >= num_slots) return;
  const __nv_bfloat16* r = rows + t * kRow;
  float x[16];
  {
    const uint4* src = reinterpret_cast<const uint4*>(r + lane * 16);
    uint4 v0 = src[0], v1 = src[1];
    uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) { x[2 * i] = bf16lo(w[i]); x[2 * i + 1] = bf16hi(w[i]); }
  }
  __nv_bfloat16 yc[16];
  if (flags & MLA_APPEND_RMSNORM) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rms = sqrtf(ss / (float)kLatent);
#pragma unroll
    for (int i = 0; i < 16; ++i) yc[i] = __float2bfloat16_rn(x[i] / rms);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) yc[i] = r[lane * 16 + i];
  }
  __nv_bfloat16 k1 = r[kLatent + lane], k2 = r[kLatent + 32 + lane];
  if (flags & MLA_APPEND_ROPE) {
    double y1, y2;
    rope_pair(__bfloat162float(k1), __bfloat162float(k2), lane, pos[t], &y1, &y2);
    k1 = __double2bfloat16(y1);
    k2 = __double2bfloat16(y2);
  }
  const long long page = slot / kPage, off = slot % kPage;
  if (!fp8) {
    __nv_bfloat16* dc = static_cast<__nv_bfloat16*>(ckv) + (page * kPage + off) * kLatent + lane * 16;
    uint4 o0, o1;
    uint32_t* ow = reinterpret_cast<uint32_t*>(yc);
    o0 = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    o1 = make_uint4(ow[4], ow[5], ow[6], ow[7]);
    reinterpret_cast<uint4*>(dc)[0] = o0;
    reinterpret_cast<uint4*>(dc)[1] = o1;
    __nv_bfloat16* dk = static_cast<__nv_bfloat16*>(kpe) + (page * kPage + off) * kRope;
    dk[lane] = k1;
    dk[32 + lane] = k2;
    return;
  }
  // E4M3: one fp32 scale over the token's 576 bf16 values.
  float amax = fmaxf(fabsf(__bfloat162float(k1)), fabsf(__bfloat162float(k2)));
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(__bfloat162float(yc[i])));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = amax == 0.f ? 1.f : amax / 448.f;
  uint8_t q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    q[i] = __nv_cvt_float_to_fp8(__bfloat162float(yc[i]) / sc, __NV_SATFINITE, __NV_E4M3);
  uint8_t* dc = static_cast<uint8_t*>(ckv) + (page * kPage + off) * kLatent + lane * 16;
  *reinterpret_cast<uint4*>(dc) = *reinterpret_cast<const uint4*>(q);
  uint8_t* dk = static_cast<uint8_t*>(kpe) + (page * kPage + off) * kRope;
  dk[lane] = __nv_cvt_float_to_fp8(__bfloat162float(k1) / sc, __NV_SATFINITE, __NV_E4M3);
  dk[32 + lane] = __nv_cvt_float_to_fp8(__bfloat162float(k2) / sc, __NV_SATFINITE, __NV_E4M3);
  if (lane == 0) scale[page * kPage + off] = sc;
}

__global__ void rope_q_kernel(const __nv_bfloat16* __restrict__ q_raw, const int32_t* __restrict__ seq_lens,
                              __nv_bfloat16* __restrict__ q, int B, int H) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)B * H * 32) return;
  const int i = idx % 32;
  const long long row = idx / 32;
  const int b = (int)(row / H);
  const long long p = max(0, seq_lens[b] - 1);
  const __nv_bfloat16* src = q_raw + row * kRope;
  double y1, y2;
  rope_pair(__bfloat162float(src[i]), __bfloat162float(src[i + 32]), i, p, &y1, &y2);
  q[row * kRope + i] = __double2bfloat16(y1);
  q[row * kRope + i + 32] = __double2bfloat16(y2);
}

}  // namespace

cudaError_t launch_cache_append(const __nv_bfloat16* rows, const int32_t* slots, const int32_t* pos,
                                int T, int flags, bool fp8, long long num_slots, void* ckv,
                                void* kpe, float* scale, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  cache_append_kernel<<<(T + 7) / 8, 256, 0, stream>>>(rows, slots, pos, T, flags, fp8, num_slots,
                                                       ckv, kpe, scale);
  return cudaGetLastError();
}

cudaError_t launch_rope_q(const __nv_bfloat16* q_raw, const int32_t* seq_lens, __nv_bfloat16* q,
                          int B, int H, cudaStream_t stream) {
  const long long n = (long long)B * H * 32;
  rope_q_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(q_raw, seq_lens, q, B, H);
  return cudaGetLastError();
}

}  // namespace mla
