// Launch functions of the libmla kernels (internal to the library).
#pragma once
#include "common.cuh"

namespace mla {

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t stream);
int decode_tc_max_clusters();
cudaError_t launch_combine(const __nv_bfloat16* part_o, const float* part_lse, const int* seq_start,
                           __nv_bfloat16* o_lat, float* lse, int B, int H, int G, cudaStream_t stream);
cudaError_t launch_absorb_tc(const __nv_bfloat16* q_nope, const __nv_bfloat16* w_uk,
                             __nv_bfloat16* q_lat, int B, int H, cudaStream_t stream);
cudaError_t launch_out_proj_tc(const __nv_bfloat16* o_lat, const __nv_bfloat16* w_uv, void* out,
                               bool out_bf16, int B, int H, cudaStream_t stream);
cudaError_t launch_outproj_combine(const __nv_bfloat16* part_o, const float* part_lse, const int32_t* seq_lens,
                                   int maxp, __nv_bfloat16* o_lat, float* lse, const __nv_bfloat16* w_uv,
                                   void* out, bool out_bf16, int B, int H, int G, cudaStream_t stream);
cudaError_t launch_cache_append(const __nv_bfloat16* rows, const int32_t* slots, const int32_t* pos,
                                int T, int flags, bool fp8, long long num_slots, void* ckv,
                                void* kpe, float* scale, cudaStream_t stream);
cudaError_t launch_multi_token_expand(const int32_t* page_table, const int32_t* seq_lens, int B, int T, int maxp,
                                      int32_t* table_out, int32_t* lens_out, cudaStream_t stream);
cudaError_t launch_quantize_q(const __nv_bfloat16* q_lat, const __nv_bfloat16* q_pe, long long rows, int terms,
                              uint8_t* codes, float* scale, cudaStream_t stream);
cudaError_t launch_rope_q(const __nv_bfloat16* q_raw, const int32_t* seq_lens, __nv_bfloat16* q,
                          int B, int H, cudaStream_t stream);

}  // namespace mla
