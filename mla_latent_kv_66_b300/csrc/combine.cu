// Split-KV combine: merge the partial results of sequences whose cache pages
// were divided between several decode workers.
//
// Method (flash-decoding style log-sum-exp merge of attention over disjoint
// token ranges; the page "DeepSeek-Coder-V2 的 MLA ... 512维潜空间" motivates
// splitting with its 128K contexts): for the partials s of one (sequence,
// head), o = sum_s exp(lse_s - L) O_s with L = log sum_s exp(lse_s), each O_s
// normalised over its own range.
#include <atomic>

#include "combine.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace tc;

// Per-head form: one CTA per (sequence, head) of a split sequence; thread t
// owns latent columns [4t, 4t+4).  The partials of the sequence are the records of the
// workers whose page ranges it overlaps, in page order.  Their slots and
// weights are worked out once per CTA (128 at a time) into shared memory.
__global__ void __launch_bounds__(128) combine_head_kernel(const __nv_bfloat16* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      const int* __restrict__ seq_start,
                                                      __nv_bfloat16* __restrict__ o_lat,
                                                      float* __restrict__ lse_out, int B, int H, int G) {
  __shared__ int s_slot[128];
  __shared__ float s_val[128];
  __shared__ float s_red[4];
  grid_dep_wait();  // the decode kernel's partials
  grid_dep_trigger();
  const int b = blockIdx.x, h = blockIdx.y, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  __shared__ int s_wf, s_n;
  __shared__ long long s_sb;
  if (t == 0) {  // the workers holding this sequence's pages (one thread: 64-bit divisions)
    const long long P = seq_start[B];
    const long long sb = seq_start[b], se = seq_start[b + 1];
    int wf = 0, n = 0;
    if (se > sb) {
      wf = worker_of(sb, G, P);
      n = worker_of(se - 1, G, P) - wf + 1;
    }
    s_wf = wf;
    s_n = n;
    s_sb = sb;
  }
  __syncthreads();
  const int wf = s_wf, n = s_n;
  const long long sb = s_sb;
  if (n <= 1) return;  // empty, or finished by the decode kernel
  const long long P = seq_start[B];
  // slot of partial i, or -1 for an empty worker range (no partial written)
  auto slot_of = [&](int i) {
    const int w = wf + i;
    const long long lo = range_lo(w, G, P), hi = range_lo(w + 1, G, P);
    return lo == hi ? -1 : (sb <= lo ? w : G + w);
  };
  // pass 1: the largest partial log-sum-exp (slots kept when they all fit)
  float mx = -INFINITY;
  for (int i = t; i < n; i += 128) {
    const int sl = slot_of(i);
    const float l = sl >= 0 ? part_lse[(size_t)sl * H + h] : -INFINITY;
    mx = fmaxf(mx, l);
    if (n <= 128) {
      s_slot[i] = sl;
      s_val[i] = l;
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) s_red[warp] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3]));
  // pass 2: weighted sum, 128 partials at a time
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float sum = 0.f;
  for (int c0 = 0; c0 < n; c0 += 128) {
    const int m = min(128, n - c0);
    __syncthreads();  // the previous chunk's entries are no longer read
    if (t < m) {
      int sl;
      float l;
      if (n <= 128) {
        sl = s_slot[t];
        l = s_val[t];
      } else {
        sl = slot_of(c0 + t);
        l = sl >= 0 ? part_lse[(size_t)sl * H + h] : -INFINITY;
      }
      s_slot[t] = sl;
      s_val[t] = l == -INFINITY ? 0.f : __expf(l - mx);
    }
    __syncthreads();
#pragma unroll 4
    for (int i = 0; i < m; ++i) {
      const int sl = s_slot[i];
      if (sl < 0) continue;
      const float wt = s_val[i];
      sum += wt;
      const uint2 v = reinterpret_cast<const uint2*>(part_o + ((size_t)sl * H + h) * kLatent)[t];
      acc.x = fmaf(wt, bf16lo(v.x), acc.x);
      acc.y = fmaf(wt, bf16hi(v.x), acc.y);
      acc.z = fmaf(wt, bf16lo(v.y), acc.z);
      acc.w = fmaf(wt, bf16hi(v.y), acc.w);
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(o_lat + ((size_t)b * H + h) * kLatent + 4 * t);
  dst[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  dst[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  if (t == 0 && lse_out) lse_out[(size_t)b * H + h] = mx + logf(sum);
}

// Grouped form: one CTA per (sequence, group of kHeads heads) of a split
// sequence; warp j merges head kHeads * blockIdx.y + j (warp_merge_partials).
constexpr int kHeads = 8;

__global__ void __launch_bounds__(32 * kHeads) combine_group_kernel(const __nv_bfloat16* __restrict__ part_o,
                                                              const float* __restrict__ part_lse,
                                                              const int* __restrict__ seq_start,
                                                              __nv_bfloat16* __restrict__ o_lat,
                                                              float* __restrict__ lse_out, int B, int H, int G) {
  __shared__ SeqWorkers s_sw;
  grid_dep_wait();  // the decode kernel's partials
  grid_dep_trigger();
  const int b = blockIdx.x, t = threadIdx.x, lane = t & 31;
  const int h = blockIdx.y * kHeads + (t >> 5);
  if (t == 0) s_sw = seq_workers(seq_start, B, G, b);
  __syncthreads();
  const SeqWorkers sw = s_sw;
  if (sw.n <= 1 || h >= H) return;  // empty, or finished by the decode kernel
  float acc[16];
  const float lse = warp_merge_partials(part_o, part_lse, sw, G, H, h, acc);
  uint32_t o8[8];
  pack_row16(acc, o8);
  uint4* dst = reinterpret_cast<uint4*>(o_lat + ((size_t)b * H + h) * kLatent) + 2 * lane;
  dst[0] = make_uint4(o8[0], o8[1], o8[2], o8[3]);
  dst[1] = make_uint4(o8[4], o8[5], o8[6], o8[7]);
  if (lane == 0 && lse_out) lse_out[(size_t)b * H + h] = lse;
}

// SM count of the current device, cached per device (it only picks the
// faster of two equivalent kernels, so a failed query falls back to 148).
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];

int device_sm_count() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return 148;
  int n = g_sms[d].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 148;
    g_sms[d].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace

cudaError_t launch_combine(const __nv_bfloat16* part_o, const float* part_lse, const int* seq_start,
                           __nv_bfloat16* o_lat, float* lse, int B, int H, int G, cudaStream_t stream) {
  // The grouped form needs fewer CTAs and global round trips; with fewer
  // than two of its CTAs per SM (few sequences, e.g. one long context whose
  // every worker holds a partial) the per-head form spreads the partials over
  // more SMs.
  const int sms = device_sm_count();
  const int groups = (H + kHeads - 1) / kHeads;
  if ((long long)B * groups >= 2LL * sms)
    return launch_dependent(combine_group_kernel, dim3(B, groups), dim3(32 * kHeads), 0, stream, part_o, part_lse,
                            seq_start, o_lat, lse, B, H, G);
  return launch_dependent(combine_head_kernel, dim3(B, H), dim3(128), 0, stream, part_o, part_lse, seq_start, o_lat,
                          lse, B, H, G);
}

}  // namespace mla
