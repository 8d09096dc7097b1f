// Host side of the libmla C ABI: argument checks, workspace layout, the
// choice of KV partition count, and kernel launches.
#include <math.h>
#include <atomic>
#include <string.h>

#include "common.cuh"
#include "kernels.h"

using namespace mla;

namespace {

constexpr int kMaxDevices = 64;
// cached device property, 0 = not queried yet.  Threads that race on the
// first query compute the same value, so relaxed atomics suffice.
std::atomic<int> g_workers[kMaxDevices];

// Decode workers that run at once: co-resident clusters of the decode kernel
// (one per pair of SMs where the GPCs allow it).
int device_workers() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = g_workers[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    n = decode_tc_max_clusters();
    if (n <= 0) {
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
      n = sms / 2;
    }
    g_workers[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

mla_status check_params(const mla_params* p) {
  if (!p) return MLA_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || p->max_pages_per_seq < 1 || p->num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if (!(p->softmax_scale > 0.f) || !isfinite(p->softmax_scale)) return MLA_ERR_INVALID_ARG;
  if (p->kv_dtype != MLA_KV_BF16 && p->kv_dtype != MLA_KV_E4M3 && p->kv_dtype != MLA_KV_E4M3_MMA &&
      p->kv_dtype != MLA_KV_E4M3_MMA1)
    return MLA_ERR_INVALID_ARG;
  if (p->out_dtype != MLA_OUT_F32 && p->out_dtype != MLA_OUT_BF16) return MLA_ERR_INVALID_ARG;
  if (p->kv_lora_rank != kLatent || p->rope_dim != kRope || p->nope_dim != kNope ||
      p->v_dim != kV || p->page_size != kPage)
    return MLA_ERR_UNSUPPORTED;
  if (p->H % 16 != 0 || p->H > 128) return MLA_ERR_UNSUPPORTED;
  if ((long long)p->num_pages * kPage > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  if ((long long)p->B * p->max_pages_per_seq > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

// 0 = automatic: one worker per co-resident decode cluster, but never more workers than the
// batch can have pages (B * max_pages_per_seq).
int resolve_splits(const mla_params* p, int num_splits) {
  if (num_splits < 0) return -1;
  if (num_splits > 0) return num_splits <= 65536 ? num_splits : -1;
  const int nw = device_workers();
  long long g = nw > 0 ? nw : 1;
  const long long cap = (long long)p->B * p->max_pages_per_seq;
  return (int)(g < cap ? g : cap);
}

mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

// The decode and combine kernels move 16 bytes at a time.
bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

bool is_e4m3(const mla_params* p) { return p->kv_dtype != MLA_KV_BF16; }
bool is_mma8(const mla_params* p) { return p->kv_dtype == MLA_KV_E4M3_MMA || p->kv_dtype == MLA_KV_E4M3_MMA1; }
WsLayout layout_of(const mla_params* p, int G) { return ws_layout(p->B, p->H, G, is_mma8(p)); }

}  // namespace

extern "C" {

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_PAGE_OOB: return "page id out of range";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_SEQ_LEN: return "sequence length out of range";
    case MLA_ERR_TIMEOUT: return "kernel wait timed out";
  }
  return "unknown status";
}

int mla_version(void) { return 200; }

int mla_decode_num_splits(const mla_params* p, int num_splits) {
  if (check_params(p) != MLA_OK) return -1;
  return resolve_splits(p, num_splits);
}

void mla_workspace_offsets(const mla_params* p, int num_splits, size_t offsets[5]) {
  const int G = mla_decode_num_splits(p, num_splits);
  if (G < 1 || !offsets) {
    if (offsets) memset(offsets, 0, 5 * sizeof(size_t));
    return;
  }
  WsLayout l = layout_of(p, G);
  offsets[0] = l.err;
  offsets[1] = l.rec;
  offsets[2] = l.seq_start;
  offsets[3] = l.part_lse;
  offsets[4] = l.part_o;
}

void mla_workspace_query_offsets(const mla_params* p, int num_splits, size_t offsets[2]) {
  if (!offsets) return;
  const int G = mla_decode_num_splits(p, num_splits);
  if (G < 1) {
    offsets[0] = offsets[1] = 0;
    return;
  }
  const WsLayout l = layout_of(p, G);
  offsets[0] = l.q8;
  offsets[1] = l.q8_scale;
}

size_t mla_decode_workspace_size(const mla_params* p, int num_splits) {
  const int G = mla_decode_num_splits(p, num_splits);
  if (G < 1) return 0;
  return layout_of(p, G).total;
}

mla_status mla_absorb_q(const mla_params* p, const void* q_nope, const void* w_uk, void* q_lat,
                        mla_stream_t stream) {
  mla_status s = check_params(p);
  if (s != MLA_OK) return s;
  if (!q_nope || !w_uk || !q_lat) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(q_lat)) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_absorb_tc(static_cast<const __nv_bfloat16*>(q_nope),
                                        static_cast<const __nv_bfloat16*>(w_uk),
                                        static_cast<__nv_bfloat16*>(q_lat), p->B, p->H,
                                        (cudaStream_t)stream));
}

mla_status mla_decode(const mla_params* p, const void* q_lat, const void* q_pe,
                      const void* ckv_cache, const void* kpe_cache, const float* kv_scale,
                      const int32_t* page_table, const int32_t* seq_lens, int num_splits,
                      void* workspace, size_t ws_bytes, void* o_lat, float* lse,
                      mla_stream_t stream) {
  mla_status s = check_params(p);
  if (s != MLA_OK) return s;
  if (!q_lat || !q_pe || !ckv_cache || !kpe_cache || !page_table || !seq_lens || !o_lat)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_lat) || !aligned16(q_pe) || !aligned16(o_lat) || !aligned16(ckv_cache) || !aligned16(kpe_cache) ||
      !aligned16(kv_scale) || !aligned16(workspace))
    return MLA_ERR_INVALID_ARG;
  if (is_e4m3(p) != (kv_scale != nullptr)) return MLA_ERR_INVALID_ARG;
  const int G = resolve_splits(p, num_splits);
  if (G < 1) return MLA_ERR_INVALID_ARG;
  const WsLayout l = layout_of(p, G);
  if (!workspace || ws_bytes < l.total) return MLA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeArgs a;
  a.q_lat = static_cast<const __nv_bfloat16*>(q_lat);
  a.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
  a.ckv = ckv_cache;
  a.kpe = kpe_cache;
  a.kv_scale = kv_scale;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.o_lat = static_cast<__nv_bfloat16*>(o_lat);
  a.lse = lse;
  a.err = reinterpret_cast<int*>(ws + l.err);
  a.rec = reinterpret_cast<int4*>(ws + l.rec);
  a.seq_start = reinterpret_cast<int*>(ws + l.seq_start);
  a.part_lse = reinterpret_cast<float*>(ws + l.part_lse);
  a.part_o = reinterpret_cast<__nv_bfloat16*>(ws + l.part_o);
  a.q8 = nullptr;
  a.q8_scale = nullptr;
  a.q_terms = a.p_terms = 0;
  a.B = p->B;
  a.H = p->H;
  a.G = G;
  a.maxp = p->max_pages_per_seq;
  a.num_pages = p->num_pages;
  a.scale_log2 = p->softmax_scale * kLog2e;
  if (is_mma8(p)) {
    const int terms = p->kv_dtype == MLA_KV_E4M3_MMA ? 2 : 1;
    a.q8 = ws + l.q8;
    a.q8_scale = reinterpret_cast<const float*>(ws + l.q8_scale);
    a.q_terms = a.p_terms = terms;
    const cudaError_t e = launch_quantize_q(a.q_lat, a.q_pe, (long long)p->B * p->H, terms, ws + l.q8,
                                            reinterpret_cast<float*>(ws + l.q8_scale), (cudaStream_t)stream);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
  }
  return cuda_status(launch_decode_tc(a, (cudaStream_t)stream));
}

mla_status mla_split_kv_combine(const mla_params* p, const void* workspace, size_t ws_bytes,
                                int num_splits, void* o_lat, float* lse, mla_stream_t stream) {
  mla_status s = check_params(p);
  if (s != MLA_OK) return s;
  if (!o_lat || !aligned16(o_lat) || !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  const int G = resolve_splits(p, num_splits);
  if (G < 1) return MLA_ERR_INVALID_ARG;
  const WsLayout l = layout_of(p, G);
  if (!workspace || ws_bytes < l.total) return MLA_ERR_WORKSPACE;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  return cuda_status(launch_combine(reinterpret_cast<const __nv_bfloat16*>(ws + l.part_o),
                                    reinterpret_cast<const float*>(ws + l.part_lse),
                                    reinterpret_cast<const int*>(ws + l.seq_start),
                                    static_cast<__nv_bfloat16*>(o_lat), lse, p->B, p->H, G,
                                    (cudaStream_t)stream));
}

mla_status mla_combine_out_proj(const mla_params* p, const void* workspace, size_t ws_bytes, int num_splits,
                                const int32_t* seq_lens, void* o_lat, float* lse, const void* w_uv, void* out,
                                mla_stream_t stream) {
  mla_status s = check_params(p);
  if (s != MLA_OK) return s;
  if (!seq_lens || !o_lat || !w_uv || !out || !aligned16(o_lat) || !aligned16(workspace) || !aligned16(w_uv))
    return MLA_ERR_INVALID_ARG;
  const int G = resolve_splits(p, num_splits);
  if (G < 1) return MLA_ERR_INVALID_ARG;
  const WsLayout l = layout_of(p, G);
  if (!workspace || ws_bytes < l.total) return MLA_ERR_WORKSPACE;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  return cuda_status(launch_outproj_combine(reinterpret_cast<const __nv_bfloat16*>(ws + l.part_o),
                                            reinterpret_cast<const float*>(ws + l.part_lse), seq_lens,
                                            p->max_pages_per_seq, static_cast<__nv_bfloat16*>(o_lat), lse,
                                            static_cast<const __nv_bfloat16*>(w_uv), out,
                                            p->out_dtype == MLA_OUT_BF16, p->B, p->H, G, (cudaStream_t)stream));
}

mla_status mla_out_proj(const mla_params* p, const void* o_lat, const void* w_uv, void* out,
                        mla_stream_t stream) {
  mla_status s = check_params(p);
  if (s != MLA_OK) return s;
  if (!o_lat || !w_uv || !out) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_out_proj_tc(static_cast<const __nv_bfloat16*>(o_lat),
                                          static_cast<const __nv_bfloat16*>(w_uv), out,
                                          p->out_dtype == MLA_OUT_BF16, p->B, p->H,
                                          (cudaStream_t)stream));
}

mla_status mla_cache_append(const mla_params* p, const void* kv_rows, const int32_t* slots,
                            const int32_t* positions, int T, int flags, void* ckv_cache,
                            void* kpe_cache, float* kv_scale, mla_stream_t stream) {
  mla_status s = check_params(p);
  if (s != MLA_OK) return s;
  if (T < 0 || (flags & ~(MLA_APPEND_RMSNORM | MLA_APPEND_ROPE))) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!kv_rows || !slots || !ckv_cache || !kpe_cache) return MLA_ERR_INVALID_ARG;
  if ((flags & MLA_APPEND_ROPE) && !positions) return MLA_ERR_INVALID_ARG;
  const bool fp8 = is_e4m3(p);
  if (fp8 && !kv_scale) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_cache_append(static_cast<const __nv_bfloat16*>(kv_rows), slots,
                                         positions, T, flags, fp8,
                                         (long long)p->num_pages * kPage, ckv_cache, kpe_cache,
                                         kv_scale, (cudaStream_t)stream));
}

mla_status mla_rope_q(const mla_params* p, const void* q_pe_raw, const int32_t* seq_lens,
                      void* q_pe, mla_stream_t stream) {
  mla_status s = check_params(p);
  if (s != MLA_OK) return s;
  if (!q_pe_raw || !seq_lens || !q_pe) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_rope_q(static_cast<const __nv_bfloat16*>(q_pe_raw), seq_lens,
                                   static_cast<__nv_bfloat16*>(q_pe), p->B, p->H,
                                   (cudaStream_t)stream));
}

mla_status mla_multi_token_expand(const mla_params* p, int q_len, const int32_t* page_table,
                                  const int32_t* seq_lens, int32_t* page_table_out, int32_t* seq_lens_out,
                                  mla_stream_t stream) {
  mla_status s = check_params(p);
  if (s != MLA_OK) return s;
  if (q_len < 1 || !page_table || !seq_lens || !page_table_out || !seq_lens_out) return MLA_ERR_INVALID_ARG;
  if ((long long)p->B * q_len > 0x7fffffffLL || (long long)p->B * q_len * p->max_pages_per_seq > 0x7fffffffLL)
    return MLA_ERR_UNSUPPORTED;
  return cuda_status(launch_multi_token_expand(page_table, seq_lens, p->B, q_len, p->max_pages_per_seq,
                                               page_table_out, seq_lens_out, (cudaStream_t)stream));
}

mla_status mla_workspace_status(void* workspace, int clear, mla_stream_t stream) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  int v = 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  if (clear && v != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return (mla_status)v;
}

}  // extern "C"
