// Latent-attention decode on the CUDA cores, one CTA per (KV worker range,
// group of 16 heads), and the split-KV combine kernel.
//
// Method (mtrt.cn DeepSeek-Coder-V2 MLA page, forward flow; absorbed form):
// s_t = scale * (q_lat . c_t + q_pe . k_pe_t), online softmax over the pages
// of a sequence, o_lat = sum_t p_t c_t.
#include "common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr int kHeadsPerCta = 16;
constexpr int kThreads = 256;
constexpr int kBf16TileWords = kRow / 2 + 1;   // 289: odd stride, no bank conflicts
constexpr int kFp8TileWords = kRow / 4 + 1;    // 145

template <bool kFp8>
struct SimtSmem {
  static constexpr int kTileWords = kFp8 ? kFp8TileWords : kBf16TileWords;
  static constexpr size_t q = 0;                                   // [16][576] f32
  static constexpr size_t s = q + kHeadsPerCta * kRow * 4;         // [16][64] f32
  static constexpr size_t alpha = s + kHeadsPerCta * kPage * 4;    // [16]
  static constexpr size_t lsum = alpha + kHeadsPerCta * 4;         // [16]
  static constexpr size_t mrun = lsum + kHeadsPerCta * 4;          // [16]
  static constexpr size_t tscale = mrun + kHeadsPerCta * 4;        // [64]
  static constexpr size_t tile = tscale + kPage * 4;               // [64][words]
  static constexpr size_t total = tile + (size_t)kPage * kTileWords * 4;
};

template <bool kFp8>
__device__ void simt_unit(const DecodeArgs& a, uint8_t* smem, int b, int pb, int pe, int n,
                          bool split, int slot, int h0) {
  using L = SimtSmem<kFp8>;
  float* q_s = reinterpret_cast<float*>(smem + L::q);
  float* s_s = reinterpret_cast<float*>(smem + L::s);
  float* alpha_s = reinterpret_cast<float*>(smem + L::alpha);
  float* l_s = reinterpret_cast<float*>(smem + L::lsum);
  float* m_s = reinterpret_cast<float*>(smem + L::mrun);
  float* ts_s = reinterpret_cast<float*>(smem + L::tscale);
  uint32_t* tile = reinterpret_cast<uint32_t*>(smem + L::tile);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H;

  __syncthreads();  // previous unit finished with shared memory
  for (int i = tid; i < kHeadsPerCta * kRow; i += kThreads) {
    int hh = i / kRow, k = i % kRow;
    size_t row = (size_t)b * H + h0 + hh;
    float v = k < kLatent ? __bfloat162float(a.q_lat[row * kLatent + k])
                          : __bfloat162float(a.q_pe[row * kRope + (k - kLatent)]);
    q_s[i] = v * a.scale_log2;
  }
  // per-head running max / sum live in the softmax warps' registers
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float acc[kHeadsPerCta][2];
#pragma unroll
  for (int h = 0; h < kHeadsPerCta; ++h) acc[h][0] = acc[h][1] = 0.f;

  for (int j = pb; j < pe; ++j) {
    const int page = a.page_table[(size_t)b * a.maxp + j];
    if (page < 0 || page >= a.num_pages) {  // uniform across the CTA
      if (tid == 0) set_error(a.err, MLA_ERR_PAGE_OOB);
      continue;
    }
    const int valid = min(kPage, n - j * kPage);
    __syncthreads();  // previous page's PV is done with the tile
    if (!kFp8) {
      const uint4* src_c = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(a.ckv) + (size_t)page * kPage * kLatent);
      const uint4* src_k = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(a.kpe) + (size_t)page * kPage * kRope);
      for (int i = tid; i < kPage * (kRow / 8); i += kThreads) {
        int r = i / (kRow / 8), c8 = i % (kRow / 8);
        uint4 v = c8 < kLatent / 8 ? src_c[r * (kLatent / 8) + c8] : src_k[r * (kRope / 8) + c8 - kLatent / 8];
        uint32_t* d = tile + r * L::kTileWords + c8 * 4;
        d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
      }
    } else {
      const uint4* src_c = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(a.ckv) + (size_t)page * kPage * kLatent);
      const uint4* src_k = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(a.kpe) + (size_t)page * kPage * kRope);
      for (int i = tid; i < kPage * (kRow / 16); i += kThreads) {
        int r = i / (kRow / 16), c16 = i % (kRow / 16);
        uint4 v = c16 < kLatent / 16 ? src_c[r * (kLatent / 16) + c16]
                                     : src_k[r * (kRope / 16) + c16 - kLatent / 16];
        uint32_t* d = tile + r * L::kTileWords + c16 * 4;
        d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
      }
      if (tid < kPage) ts_s[tid] = a.kv_scale[(size_t)page * kPage + tid];
    }
    __syncthreads();

    // scores: thread = (token, 4 heads)
    {
      const int tok = tid % kPage, hq = tid / kPage;
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      if (tok < valid) {
        const uint32_t* row = tile + tok * L::kTileWords;
        if (!kFp8) {
          for (int k2 = 0; k2 < kRow / 2; ++k2) {
            uint32_t v = row[k2];
            float x0 = bf16lo(v), x1 = bf16hi(v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float* q = q_s + (hq * 4 + i) * kRow + 2 * k2;
              sc[i] = fmaf(q[0], x0, fmaf(q[1], x1, sc[i]));
            }
          }
        } else {
          const uint8_t* rb = reinterpret_cast<const uint8_t*>(row);
          for (int k = 0; k < kRow; ++k) {
            float x = e4m3_to_float(rb[k]);
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[i] = fmaf(q_s[(hq * 4 + i) * kRow + k], x, sc[i]);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) sc[i] *= ts_s[tok];
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) s_s[(hq * 4 + i) * kPage + tok] = tok < valid ? sc[i] : -INFINITY;
    }
    __syncthreads();

    // online softmax: warp = 2 heads, lane = tokens lane, lane+32
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int h = warp * 2 + i;
      float x0 = s_s[h * kPage + lane], x1 = s_s[h * kPage + lane + 32];
      float mx = fmaxf(x0, x1);
#pragma unroll
      for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m_run[i], mx);
      const float p0 = exp2f(x0 - m_new), p1 = exp2f(x1 - m_new);
      float ps = p0 + p1;
#pragma unroll
      for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      const float alpha = exp2f(m_run[i] - m_new);
      l_run[i] = l_run[i] * alpha + ps;
      m_run[i] = m_new;
      float w0 = p0, w1 = p1;
      if (kFp8) { w0 *= ts_s[lane]; w1 *= ts_s[lane + 32]; }
      s_s[h * kPage + lane] = w0;
      s_s[h * kPage + lane + 32] = w1;
      if (lane == 0) alpha_s[h] = alpha;
    }
    __syncthreads();

    // P.V over the latent: thread = latent columns 2*tid, 2*tid+1
#pragma unroll
    for (int h = 0; h < kHeadsPerCta; ++h) {
      const float al = alpha_s[h];
      acc[h][0] *= al;
      acc[h][1] *= al;
    }
    for (int tok = 0; tok < valid; ++tok) {
      float x0, x1;
      if (!kFp8) {
        uint32_t v = tile[tok * L::kTileWords + tid];
        x0 = bf16lo(v); x1 = bf16hi(v);
      } else {
        const uint8_t* rb = reinterpret_cast<const uint8_t*>(tile + tok * L::kTileWords);
        x0 = e4m3_to_float(rb[2 * tid]); x1 = e4m3_to_float(rb[2 * tid + 1]);
      }
#pragma unroll
      for (int h = 0; h < kHeadsPerCta; ++h) {
        const float p = s_s[h * kPage + tok];
        acc[h][0] = fmaf(p, x0, acc[h][0]);
        acc[h][1] = fmaf(p, x1, acc[h][1]);
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) { l_s[warp * 2 + i] = l_run[i]; m_s[warp * 2 + i] = m_run[i]; }
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < kHeadsPerCta; ++h) {
    const float l = l_s[h];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? (m_s[h] + log2f(l)) * kLn2 : -INFINITY;
    const size_t row = (size_t)b * H + h0 + h;
    if (!split) {
      __nv_bfloat162 o = __floats2bfloat162_rn(acc[h][0] * inv, acc[h][1] * inv);
      reinterpret_cast<__nv_bfloat162*>(a.o_lat + row * kLatent)[tid] = o;
      if (tid == 0 && a.lse) a.lse[row] = lse;
    } else {
      const size_t prow = (size_t)slot * H + h0 + h;
      reinterpret_cast<float2*>(a.part_o + prow * kLatent)[tid] = make_float2(acc[h][0] * inv, acc[h][1] * inv);
      if (tid == 0) a.part_lse[prow] = lse;
    }
  }
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int sh_b0;
  __shared__ long long sh_s0, sh_P;
  const int w = blockIdx.x, h0 = blockIdx.y * kHeadsPerCta;
  const bool lead = blockIdx.y == 0;
  if (threadIdx.x < 32) {
    long long P = warp_total_pages(a.seq_lens, a.B, a.maxp, (w == 0 && lead) ? a.err : nullptr,
                                   (w == 0 && lead) ? a.seq_start : nullptr);
    long long lo = range_lo(w, a.G, P), hi = range_lo(w + 1, a.G, P);
    int b0 = a.B;
    long long s0 = 0;
    if (lo < hi) warp_find_seq(a.seq_lens, a.B, a.maxp, lo, &b0, &s0);
    if (threadIdx.x == 0) { sh_b0 = b0; sh_s0 = s0; sh_P = P; }
  }
  __syncthreads();
  const long long P = sh_P, lo = range_lo(w, a.G, P), hi = range_lo(w + 1, a.G, P);
  int b = sh_b0;
  long long sb = sh_s0;
  int4 first = make_int4(-1, 0, 0, 0), last = make_int4(-1, 0, 0, 0);
  while (b < a.B && sb < hi) {
    const int n = a.seq_lens[b];
    const int np = seq_pages(n, a.maxp, nullptr);
    if (np > 0) {
      const long long ub = max(lo, sb), ue = min(hi, sb + np);
      const bool split = sb < lo || sb + np > hi;
      const int slot = ub == lo ? w : a.G + w;
      int4 r = make_int4(b, (int)(ub - sb), (int)(ue - sb), split ? 1 : 0);
      if (ub == lo) first = r;
      else if (ue == hi) last = r;
      simt_unit<kFp8>(a, smem, b, r.y, r.z, n, split, slot, h0);
    }
    sb += np;
    ++b;
  }
  if (lead && threadIdx.x == 0) {
    a.rec[w] = first;
    a.rec[a.G + w] = last;
  }
}

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      const int* __restrict__ seq_start,
                                                      __nv_bfloat16* __restrict__ o_lat,
                                                      float* __restrict__ lse_out, int B, int H, int G) {
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 8 + warp;
  if (h >= H) return;
  const long long P = seq_start[B];
  const long long sb = seq_start[b], se = seq_start[b + 1];
  if (se <= sb) return;
  const int wf = worker_of(sb, G, P), wl = worker_of(se - 1, G, P);
  if (wf == wl) return;  // finished by the decode kernel
  float mx = -INFINITY;
  for (int w = wf; w <= wl; ++w) {
    if (range_lo(w + 1, G, P) == range_lo(w, G, P)) continue;  // empty range: no partial
    const int slot = sb <= range_lo(w, G, P) ? w : G + w;
    mx = fmaxf(mx, part_lse[(size_t)slot * H + h]);
  }
  float4 acc[4] = {};
  float sum = 0.f;
  for (int w = wf; w <= wl; ++w) {
    if (range_lo(w + 1, G, P) == range_lo(w, G, P)) continue;
    const int slot = sb <= range_lo(w, G, P) ? w : G + w;
    const float l = part_lse[(size_t)slot * H + h];
    const float wt = l == -INFINITY ? 0.f : __expf(l - mx);
    sum += wt;
    const float4* src = reinterpret_cast<const float4*>(part_o + ((size_t)slot * H + h) * kLatent);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float4 v = src[k * 32 + lane];
      acc[k].x = fmaf(wt, v.x, acc[k].x);
      acc[k].y = fmaf(wt, v.y, acc[k].y);
      acc[k].z = fmaf(wt, v.z, acc[k].z);
      acc[k].w = fmaf(wt, v.w, acc[k].w);
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat16* dst = o_lat + ((size_t)b * H + h) * kLatent;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c = (k * 32 + lane) * 4;
    reinterpret_cast<__nv_bfloat162*>(dst + c)[0] = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
    reinterpret_cast<__nv_bfloat162*>(dst + c)[1] = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
  }
  if (lane == 0 && lse_out) lse_out[(size_t)b * H + h] = mx + logf(sum);
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream) {
  const bool fp8 = a.kv_scale != nullptr;
  const size_t smem = fp8 ? SimtSmem<true>::total : SimtSmem<false>::total;
  dim3 grid(a.G, a.H / kHeadsPerCta);
  if (fp8) {
    cudaFuncSetAttribute(decode_simt_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    decode_simt_kernel<true><<<grid, kThreads, smem, stream>>>(a);
  } else {
    cudaFuncSetAttribute(decode_simt_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    decode_simt_kernel<false><<<grid, kThreads, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* part_o, const float* part_lse, const int* seq_start,
                           __nv_bfloat16* o_lat, float* lse, int B, int H, int G, cudaStream_t stream) {
  dim3 grid(B, (H + 7) / 8);
  combine_kernel<<<grid, 256, 0, stream>>>(part_o, part_lse, seq_start, o_lat, lse, B, H, G);
  return cudaGetLastError();
}

}  // namespace mla
