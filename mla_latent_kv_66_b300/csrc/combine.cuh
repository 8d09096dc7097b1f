// One warp's log-sum-exp merge of the partial results of one (sequence,
// head): shared by the grouped split-KV combine and the combine fused into
// the out-projection, so that both produce the same bits.
//
// Method (flash-decoding style merge of attention over disjoint token
// ranges): o = sum_s exp(lse_s - L) O_s / sum_s exp(lse_s - L), L the largest
// lse_s, each O_s normalised over its own range.
#pragma once

#include "common.cuh"

namespace mla {

// The decode workers whose page ranges overlap sequence b (seq_start: the
// batch's page offsets, B+1 entries): the first one and their number (0 for
// an empty sequence).  One thread.
struct SeqWorkers {
  int wf, n;
  long long sb, P;
};
__device__ inline SeqWorkers seq_workers(const int* seq_start, int B, int G, int b) {
  SeqWorkers s;
  s.P = seq_start[B];
  s.sb = seq_start[b];
  const long long se = seq_start[b + 1];
  s.wf = 0;
  s.n = 0;
  if (se > s.sb) {
    s.wf = worker_of(s.sb, G, s.P);
    s.n = worker_of(se - 1, G, s.P) - s.wf + 1;
  }
  return s;
}

// Slot of partial i of a split sequence: the worker's first-unit record if
// its range starts in the sequence, else its last-unit record; -1 for an
// empty worker range (it wrote none).
__device__ inline int partial_slot(const SeqWorkers& sw, int G, int i) {
  const int w = sw.wf + i;
  const long long lo = range_lo(w, G, sw.P), hi = range_lo(w + 1, G, sw.P);
  return lo == hi ? -1 : (sw.sb <= lo ? w : G + w);
}

// Run by one full warp, reading only the sequence lengths (the page counts
// of the decode's schedule, seq_pages): the batch's total page count, and
// for sequences [b0, b0 + nrows) their first flattened page (sb) and page
// count (np), in shared or global memory.
__device__ inline long long warp_page_offsets(const int32_t* __restrict__ seq_lens, int B, int maxp, int b0,
                                              int nrows, long long* sb, int* np_out) {
  const int lane = threadIdx.x & 31;
  long long run = 0;
  for (int base = 0; base < B; base += 32) {
    const int b = base + lane;
    const int np = b < B ? seq_pages(__ldg(seq_lens + b), maxp, nullptr) : 0;
    const int incl = warp_incl_scan(np);
    if (b >= b0 && b < b0 + nrows && b < B) {
      sb[b - b0] = run + incl - np;
      np_out[b - b0] = np;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  return run;
}

// Lane l of the calling warp gets latent columns [16 l, 16 l + 16) of the
// merged, normalised o (acc) and every lane the merged log-sum-exp.  The
// partials are taken 32 at a time (slot and lse one per lane) with a running
// maximum, so each is read once; four partials' loads are kept in flight.
__device__ inline float warp_merge_partials(const __nv_bfloat16* __restrict__ part_o,
                                            const float* __restrict__ part_lse, const SeqWorkers& sw, int G, int H,
                                            int h, float (&acc)[16]) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY, sum = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  for (int c0 = 0; c0 < sw.n; c0 += 32) {
    const int i = c0 + lane;
    const int sl = i < sw.n ? partial_slot(sw, G, i) : -1;
    const float l = sl >= 0 ? part_lse[(size_t)sl * H + h] : -INFINITY;
    float cm = l;
#pragma unroll
    for (int o = 16; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
    const float nm = fmaxf(m, cm);
    if (nm > m && m != -INFINITY) {  // rescale what the earlier chunks added
      const float r = __expf(m - nm);
      sum *= r;
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] *= r;
    }
    m = nm;
    const float wt = l == -INFINITY ? 0.f : __expf(l - m);
    float ws = wt;
#pragma unroll
    for (int o = 16; o; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    sum += ws;
    const int cn = min(32, sw.n - c0);
    for (int k0 = 0; k0 < cn; k0 += 4) {
      uint4 v[4][2];
      float wk[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = k0 + u;
        const int slk = __shfl_sync(0xffffffffu, sl, k & 31);
        wk[u] = __shfl_sync(0xffffffffu, wt, k & 31);
        if (k < cn && slk >= 0) {
          const uint4* src = reinterpret_cast<const uint4*>(part_o + ((size_t)slk * H + h) * kLatent) + 2 * lane;
          v[u][0] = src[0];
          v[u][1] = src[1];
        } else {
          v[u][0] = v[u][1] = make_uint4(0, 0, 0, 0);
          wk[u] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t w8[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w,
                                v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc[2 * e] = fmaf(wk[u], bf16lo(w8[e]), acc[2 * e]);
          acc[2 * e + 1] = fmaf(wk[u], bf16hi(w8[e]), acc[2 * e + 1]);
        }
      }
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] *= inv;
  return sum > 0.f ? m + logf(sum) : -INFINITY;
}

// Two rows at once, each with 2..4 partials (the common case of a batch
// split across a few workers): the same operations as warp_merge_partials
// row by row, in the same order (so the same bits).  sl[i]: lane u < n[i]
// holds the slot of partial u of row i (partial_slot), the other lanes -1.
// Every load of both rows (log-sum-exps and partial rows) is issued before
// any of them is used: one memory round trip.
__device__ inline void warp_merge_two_small(const __nv_bfloat16* __restrict__ part_o,
                                            const float* __restrict__ part_lse, const int (&sl)[2],
                                            const int (&n)[2], int H, int h, float (&acc)[2][16],
                                            float (&lse)[2]) {
  const int lane = threadIdx.x & 31;
  float l[2];
  uint4 v[2][4][2];
  bool on[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l[i] = sl[i] >= 0 ? part_lse[(size_t)sl[i] * H + h] : -INFINITY;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int slk = __shfl_sync(0xffffffffu, sl[i], u);
      on[i][u] = u < n[i] && slk >= 0;
      if (on[i][u]) {
        const uint4* src = reinterpret_cast<const uint4*>(part_o + ((size_t)slk * H + h) * kLatent) + 2 * lane;
        v[i][u][0] = src[0];
        v[i][u][1] = src[1];
      } else {
        v[i][u][0] = v[i][u][1] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  float m[2], wt[2], sum[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float cm = l[i];
#pragma unroll
    for (int o = 16; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
    m[i] = cm;  // the first chunk: nothing to rescale
    wt[i] = l[i] == -INFINITY ? 0.f : __expf(l[i] - m[i]);
    float ws = wt[i];
#pragma unroll
    for (int o = 16; o; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    sum[i] = 0.f + ws;
  }
  float wk[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      wk[i][u] = __shfl_sync(0xffffffffu, wt[i], u);
      if (!on[i][u]) wk[i][u] = 0.f;
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[i][k] = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t w8[8] = {v[i][u][0].x, v[i][u][0].y, v[i][u][0].z, v[i][u][0].w,
                              v[i][u][1].x, v[i][u][1].y, v[i][u][1].z, v[i][u][1].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc[i][2 * e] = fmaf(wk[i][u], bf16lo(w8[e]), acc[i][2 * e]);
        acc[i][2 * e + 1] = fmaf(wk[i][u], bf16hi(w8[e]), acc[i][2 * e + 1]);
      }
    }
    const float inv = sum[i] > 0.f ? 1.f / sum[i] : 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[i][k] *= inv;
    lse[i] = sum[i] > 0.f ? m[i] + logf(sum[i]) : -INFINITY;
  }
}

// acc (16 fp32, lane l's columns) as 8 bf16 pairs.
__device__ inline void pack_row16(const float (&acc)[16], uint32_t (&o8)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    __nv_bfloat162 q = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
    o8[e] = *reinterpret_cast<uint32_t*>(&q);
  }
}

}  // namespace mla
