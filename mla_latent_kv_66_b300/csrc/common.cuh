// Device helpers shared by the libmla kernels: dimensions, the workspace
// layout, the KV-partition schedule and number-format conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

constexpr int kLatent = 512;   // kv_lora_rank
constexpr int kRope = 64;      // qk_rope_head_dim
constexpr int kRow = kLatent + kRope;
constexpr int kNope = 128;
constexpr int kV = 128;
constexpr int kPage = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ----------------------------------------------------------------------------
// Workspace layout (see mla_decode_workspace_size in the header).
// ----------------------------------------------------------------------------
struct WsLayout {
  size_t err, rec, seq_start, part_lse, part_o, q8, q8_scale, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// q8: the 8-bit tensor-core decode also keeps the E4M3 query there (codes
// [B,H,2,576], scales [B,H] fp32); otherwise those two offsets are 0.
__host__ __device__ inline WsLayout ws_layout(int B, int H, int G, bool q8 = false) {
  WsLayout l;
  l.err = 0;
  l.rec = 256;
  l.seq_start = align_up(l.rec + (size_t)2 * G * 16, 256);
  l.part_lse = align_up(l.seq_start + (size_t)(B + 1) * 4, 256);
  l.part_o = align_up(l.part_lse + (size_t)2 * G * H * 4, 256);
  l.total = align_up(l.part_o + (size_t)2 * G * H * kLatent * 2, 256);
  l.q8 = l.q8_scale = 0;
  if (q8) {
    l.q8 = l.total;
    l.q8_scale = align_up(l.q8 + (size_t)B * H * 2 * kRow, 256);
    l.total = align_up(l.q8_scale + (size_t)B * H * 4, 256);
  }
  return l;
}

struct DecodeArgs {
  const __nv_bfloat16* q_lat;  // [B,H,512]
  const __nv_bfloat16* q_pe;   // [B,H,64]
  const void* ckv;             // [pages,64,512]
  const void* kpe;             // [pages,64,64]
  const float* kv_scale;       // [pages,64] or null
  const int32_t* page_table;   // [B,maxp]
  const int32_t* seq_lens;     // [B]
  __nv_bfloat16* o_lat;        // [B,H,512]
  float* lse;                  // [B,H] or null
  int* err;                    // workspace error word
  int4* rec;                   // [2G]
  int* seq_start;              // [B+1]
  float* part_lse;             // [2G,H]
  __nv_bfloat16* part_o;       // [2G,H,512], normalised
  const uint8_t* q8;           // 8-bit tensor-core decode: E4M3 query [B,H,2,576]
  const float* q8_scale;       // [B,H]
  int q_terms, p_terms;        // E4M3 terms of the query and of the probabilities (1 or 2)
  int B, H, G, maxp, num_pages;
  float scale_log2;            // softmax_scale * log2(e)
};

__device__ inline void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);  // first error wins
}

// Pages of a sequence of length n; 0 (and an error) for an invalid length.
__device__ inline int seq_pages(int n, int maxp, int* err) {
  if (n < 1 || (long long)n > (long long)maxp * kPage) {
    set_error(err, MLA_ERR_SEQ_LEN);
    return 0;
  }
  return (n + kPage - 1) / kPage;
}

__device__ inline int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// Worker range [lo, hi) of flattened pages for worker w of G over P pages.
// A 64-bit division is a long dependent instruction sequence on the GPU, so
// the common case (the product fits in 32 bits) divides in 32 bits; both
// give the same integer (non-negative operands).
__host__ __device__ inline long long range_lo(int w, int G, long long P) {
  const unsigned long long prod = (unsigned long long)w * (unsigned long long)P;
  if (w >= 0 && P >= 0 && prod <= 0xFFFFFFFFull) return (long long)((unsigned)prod / (unsigned)G);
  return (long long)w * P / G;
}

// Index of the worker whose range holds flattened page x (0 <= x < P).
__host__ __device__ inline int worker_of(long long x, int G, long long P) {
  const long long num = (x + 1) * (long long)G - 1;
  if (num >= 0 && num <= 0xFFFFFFFFll && P > 0 && P <= 0xFFFFFFFFll) return (int)((unsigned)num / (unsigned)P);
  return (int)(num / P);
}

// Run by one full warp.  Returns the total page count P and, for flattened
// page `lo`, the sequence b0 holding it and that sequence's first page s0
// (b0 = B when lo >= P).  If seq_start != null the warp also writes the
// page offset of every sequence (B+1 entries).
struct SeqPos {
  long long P;
  int b0;
  long long s0;
};

__device__ inline long long warp_total_pages(const int32_t* seq_lens, int B, int maxp, int* err,
                                             int* seq_start) {
  const int lane = threadIdx.x & 31;
  long long run = 0;
  for (int base = 0; base < B; base += 32) {
    int b = base + lane;
    int n = b < B ? seq_pages(seq_lens[b], maxp, err) : 0;
    int incl = warp_incl_scan(n);
    if (seq_start && b < B) seq_start[b] = (int)(run + incl - n);
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (seq_start && lane == 0) seq_start[B] = (int)run;
  return run;
}

__device__ inline void warp_find_seq(const int32_t* seq_lens, int B, int maxp, long long lo,
                                     int* b_out, long long* s_out) {
  const int lane = threadIdx.x & 31;
  long long run = 0;
  int found_b = B;
  long long found_s = 0;
  for (int base = 0; base < B; base += 32) {
    int b = base + lane;
    int n = b < B ? seq_pages(seq_lens[b], maxp, nullptr) : 0;
    int incl = warp_incl_scan(n);
    long long start = run + incl - n;
    bool hit = (b < B) && n > 0 && start <= lo && lo < start + n;
    unsigned m = __ballot_sync(0xffffffffu, hit);
    if (m) {
      int src = __ffs(m) - 1;
      found_b = base + src;
      found_s = __shfl_sync(0xffffffffu, start, src);
      break;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  *b_out = found_b;
  *s_out = found_s;
}

// ----------------------------------------------------------------------------
// Number formats
// ----------------------------------------------------------------------------
__device__ inline float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ inline float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ inline float e4m3_to_float(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

}  // namespace mla
