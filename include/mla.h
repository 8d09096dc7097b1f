/*
 * mla.h - C ABI of libmla: Multi-head Latent Attention (MLA) decode over a
 * paged, compressed latent KV cache, for one B300 GPU (sm_103a).
 *
 * The method (page "DeepSeek-Coder-V2 的 MLA 多头潜在注意力深度解析：512维
 * 潜空间压缩 KV 缓存", mtrt.cn, sections on the two MLA components, the
 * forward flow and the cache-size table; and the aiboss88.com wiki page
 * "什么是多头潜在注意力", section "工作机制"): every cached token of a layer
 * holds only a 512-d latent c (kv_lora_rank) and a 64-d rotated key part
 * k_pe shared by all heads, 576 values.  Per head h the key is
 * [W_UK,h c ; k_pe] (192-d) and the value W_UV,h c (128-d).  Because the
 * up-projection is linear, decode runs in the weight-absorbed form:
 *
 *   q_lat[b,h] = W_UK,h^T q_nope[b,h]                       (mla_absorb_q)
 *   s[b,h,t]   = scale * (q_lat[b,h].c_t + q_pe[b,h].k_pe_t) (mla_decode)
 *   o_lat[b,h] = sum_t softmax_t(s) c_t                      (mla_decode,
 *                                                  mla_split_kv_combine)
 *   out[b,h]   = W_UV,h o_lat[b,h]                           (mla_out_proj)
 *
 * Conventions for every call:
 *  - All tensors are dense, row-major, contiguous, in device memory unless
 *    a comment says "host".  The caller owns every buffer and the stream.
 *    mla_absorb_q, mla_decode, mla_split_kv_combine and mla_combine_out_proj
 *    want every tensor and the workspace 16-byte aligned
 *    (MLA_ERR_INVALID_ARG otherwise).
 *  - No call allocates memory or synchronises, except mla_workspace_status
 *    and mla_decode_static_status, which read one word back.  Calls only
 *    enqueue work on `stream`.
 *  - Arguments are checked on the host; a bad argument returns
 *    MLA_ERR_INVALID_ARG (or MLA_ERR_UNSUPPORTED for a shape this build does
 *    not implement) and enqueues nothing.  A failed launch returns
 *    MLA_ERR_CUDA.  Values that live on the device (sequence lengths, page
 *    ids) are checked by the kernels, which skip the offending work and set
 *    a sticky error word in the workspace (see mla_workspace_status).
 *  - bf16 is IEEE binary32 truncated to its upper 16 bits; E4M3 is the OCP
 *    FP8 E4M3 format (bias 7, max 448, no infinities).
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mla_stream_t; /* same object as cudaStream_t */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,  /* null pointer, bad size or bad dimension */
  MLA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement */
  MLA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  MLA_ERR_PAGE_OOB = 4,     /* a page id outside [0, num_pages) was seen */
  MLA_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required */
  MLA_ERR_SEQ_LEN = 6,      /* a sequence length outside [1, max_pages*64] */
  MLA_ERR_TIMEOUT = 7       /* a kernel gave up a bounded wait (internal fault) */
} mla_status;

/* Storage of the latent cache and the arithmetic of mla_decode.
 *  MLA_KV_BF16       bf16 cache, bf16 tensor-core products.
 *  MLA_KV_E4M3       E4M3 cache + fp32 scale per token; the codes are
 *                    expanded exactly to bf16 and multiplied in bf16.
 *  MLA_KV_E4M3_MMA   the same E4M3 cache multiplied as codes on the 8-bit
 *                    tensor cores (tcgen05 kind::f8f6f4): mla_decode turns
 *                    the query into two E4M3 terms under one fp32 scale per
 *                    head row (see mla_workspace_query_offsets) and the
 *                    probabilities into two E4M3 terms per P . V product, so
 *                    each product carries about 8 significant bits more
 *                    than one E4M3 value.  The cache is never expanded.
 *  MLA_KV_E4M3_MMA1  as MLA_KV_E4M3_MMA with one E4M3 term for the query
 *                    and for the probabilities (fewer products, the query's
 *                    and the probabilities' own E4M3 rounding in the
 *                    result).
 * The three E4M3 values share one cache layout (mla_cache_append writes it
 * for any of them). */
typedef enum {
  MLA_KV_BF16 = 0,
  MLA_KV_E4M3 = 1,
  MLA_KV_E4M3_MMA = 2,
  MLA_KV_E4M3_MMA1 = 3
} mla_kv_dtype;
typedef enum { MLA_OUT_F32 = 0, MLA_OUT_BF16 = 1 } mla_out_dtype;

/* Problem description shared by every call.  The head dimensions are those of
 * the page's model config (kv_lora_rank 512, qk_rope_head_dim 64, 128-d
 * k_nope and 128-d value per head); this build implements exactly those and
 * returns MLA_ERR_UNSUPPORTED for others.  H may be any multiple of 16 up to
 * 128 (the page's model has 128). */
typedef struct {
  int B;                  /* sequences in the batch (one query token each) */
  int H;                  /* attention heads */
  int kv_lora_rank;       /* 512 */
  int rope_dim;           /* 64  */
  int nope_dim;           /* 128 */
  int v_dim;              /* 128 */
  int page_size;          /* 64 tokens per cache page */
  int max_pages_per_seq;  /* columns of page_table */
  int num_pages;          /* pages in the cache pool */
  float softmax_scale;    /* 1/sqrt(nope_dim + rope_dim) = 1/sqrt(192) */
  mla_kv_dtype kv_dtype;  /* storage of the latent cache */
  mla_out_dtype out_dtype;/* dtype of mla_out_proj's output */
} mla_params;

/* Human-readable name of a status code (static storage, never NULL). */
const char* mla_status_string(mla_status s);

/* Library version, major*10000 + minor*100 + patch. */
int mla_version(void);

/* ---------------------------------------------------------------------
 * mla_absorb_q: carry the no-position query into latent space.
 *   q_lat[b,h,:] = W_UK[h]^T q_nope[b,h,:]      (fp32 accumulate)
 * This is the key half of kv_b_proj (the up-projection of the 512-d latent
 * into per-head keys and values; page section "源码里的压缩全流程")
 * moved onto the query: q_nope.(W_UK,h c) = (W_UK,h^T q_nope).c for every
 * cached latent c.
 *   q_nope : [B,H,128] bf16
 *   w_uk   : [H,128,512] bf16, (head, k_nope row, latent column)
 *   q_lat  : [B,H,512] bf16 output (round to nearest even)
 * Runs on the tensor cores (tcgen05, fp32 accumulation in tensor memory).
 */
mla_status mla_absorb_q(const mla_params* p, const void* q_nope, const void* w_uk,
                        void* q_lat, mla_stream_t stream);

/* ---------------------------------------------------------------------
 * KV partitioning.  The cache pages of the whole batch, taken in order
 * (sequence 0's pages, then sequence 1's, ...), are cut into `num_splits`
 * contiguous ranges of equal size (range w holds flattened pages
 * [floor(w*P/G), floor((w+1)*P/G)), P the total, G = num_splits); each
 * range is one persistent worker of the decode kernel.  A sequence that lies
 * inside one range is finished by mla_decode; a sequence cut by a range
 * boundary is split, and its partial results are merged by
 * mla_split_kv_combine.  num_splits == 0 picks the number of worker slots of
 * the device (one per two SMs).  This is the split-KV ("flash-decoding") step
 * for long and ragged contexts: the pages motivate it with 128K contexts.
 */
int mla_decode_num_splits(const mla_params* p, int num_splits);

/* Bytes of workspace mla_decode needs for `num_splits` (0 = automatic).
 * Layout (offsets from mla_workspace_offsets):
 *   [0]  int32 error word (sticky; zero the workspace once before first use)
 *   [1]  split records, 2*G x int32[4] = {seq, page_begin, page_end, split}
 *        record w: the unit holding range w's first page; record G+w: the
 *        unit holding its last page when that is another unit (else seq=-1)
 *   [2]  int32 page offset of each sequence, B+1 entries
 *   [3]  partial LSE, fp32 [2*G, H]
 *   [4]  partial O, bf16 [2*G, H, 512], normalised
 */
size_t mla_decode_workspace_size(const mla_params* p, int num_splits);
void mla_workspace_offsets(const mla_params* p, int num_splits, size_t offsets[5]);

/* MLA_KV_E4M3_MMA / _MMA1 only: where mla_decode keeps the E4M3 query in the
 * workspace (offsets[0], offsets[1]; both 0 for the other kv_dtypes):
 *   codes [B,H,2,576] uint8 at offsets[0]: per (b,h) row, term 0 then term 1
 *         (term 1 unused by _MMA1), each 512 latent codes then 64 RoPE codes
 *   scale [B,H] fp32 at offsets[1]
 * Row v = [q_lat[b,h] ; q_pe[b,h]] (576 bf16 values): scale = max|v| / 448
 * (1 for an all-zero row), y = v / scale, term0 = E4M3(y),
 * term1 = E4M3(y - value(term0)); fp32 divisions, round to nearest even,
 * saturating.  The page (hotdry.top, "DeepSeek-V3.2-Exp 中多头潜在注意力
 * 的优化", deployment paragraph) asks for FP8 when serving MLA and names no
 * format; this mirrors the cache's per-token rule. */
void mla_workspace_query_offsets(const mla_params* p, int num_splits, size_t offsets[2]);

/* ---------------------------------------------------------------------
 * mla_decode: latent attention of one query token per sequence over its
 * paged cache.  For each (b,h), with n = seq_lens[b] and cached token t in
 * slot (page_table[b][t/64], t%64):
 *   s_t = softmax_scale * (q_lat[b,h].c_t + q_pe[b,h].k_pe_t)
 *   o_lat[b,h] = sum_t exp(s_t - lse) c_t,  lse[b,h] = log sum_t exp(s_t)
 * The 576-d score and the 512-d value sum read each cached byte once; all H
 * heads of a sequence share the cache tile (the page's FAQ: one k_pe serves
 * all 128 heads instead of 128 stored copies).  Every cached token is visible to the query
 * (decode of the newest token, whose own row is already in the cache).
 *   q_lat      : [B,H,512] bf16 (from mla_absorb_q)
 *   q_pe       : [B,H,64] bf16, already rotated at position n-1
 *   ckv_cache  : [num_pages,64,512] bf16, or E4M3 bytes (the MLA_KV_E4M3*
 *                kv_dtypes)
 *   kpe_cache  : [num_pages,64,64]  bf16, or E4M3 bytes, rotated keys
 *   kv_scale   : [num_pages,64] fp32 per-token dequantisation scale for
 *                E4M3 (value = code * scale); NULL for bf16
 *   page_table : [B,max_pages_per_seq] int32 physical page ids; entries at
 *                or past ceil(n/64) are never read
 *   seq_lens   : [B] int32, 1 <= n <= max_pages_per_seq*64
 *   workspace  : ws_bytes >= mla_decode_workspace_size(p, num_splits)
 *   o_lat      : [B,H,512] bf16, written for sequences not split
 *   lse        : [B,H] fp32 natural-log LSE, written for sequences not split
 *                (may be NULL)
 * Slots past n in a sequence's last page are ignored and may hold anything.
 * MLA_KV_E4M3_MMA / _MMA1 launch two kernels: the query quantisation into
 * the workspace, then the decode.
 * Device-side faults of the inputs: a page id outside [0,num_pages) sets
 * MLA_ERR_PAGE_OOB and that page's tokens are left out; a length outside
 * [1, max_pages*64] sets MLA_ERR_SEQ_LEN and the sequence is skipped.
 * The kernel never traps and never waits without a bound.
 */
mla_status mla_decode(const mla_params* p, const void* q_lat, const void* q_pe,
                      const void* ckv_cache, const void* kpe_cache, const float* kv_scale,
                      const int32_t* page_table, const int32_t* seq_lens, int num_splits,
                      void* workspace, size_t ws_bytes, void* o_lat, float* lse,
                      mla_stream_t stream);

/* ---------------------------------------------------------------------
 * mla_split_kv_combine: merge the partial results of split sequences.
 *   o_lat[b,h] = sum_s exp(lse_s - L) O_s,  L = log sum_s exp(lse_s)
 * over the splits s of sequence b, in page order; lse[b,h] = L.  Sequences
 * that were not split are left untouched.  Must follow mla_decode on the
 * same stream with the same params, num_splits and workspace.
 *   o_lat : [B,H,512] bf16;  lse : [B,H] fp32 or NULL
 */
mla_status mla_split_kv_combine(const mla_params* p, const void* workspace, size_t ws_bytes,
                                int num_splits, void* o_lat, float* lse, mla_stream_t stream);

/* ---------------------------------------------------------------------
 * mla_out_proj: value up-projection after attention.
 *   out[b,h,:] = W_UV[h] o_lat[b,h,:]            (fp32 accumulate)
 * The value half of kv_b_proj (the latent restored to a 128-d key part and a
 * 128-d value per head; page section "源码里的压缩全流程"), applied
 * once to the attention-weighted latent instead of to every cached token.
 *   o_lat : [B,H,512] bf16;  w_uv : [H,128,512] bf16 (head, value row, latent)
 *   out   : [B,H,128] fp32 (MLA_OUT_F32) or bf16 (MLA_OUT_BF16)
 * Runs on the tensor cores (tcgen05, fp32 accumulation in tensor memory).
 */
mla_status mla_out_proj(const mla_params* p, const void* o_lat, const void* w_uv,
                        void* out, mla_stream_t stream);

/* ---------------------------------------------------------------------
 * mla_combine_out_proj: mla_split_kv_combine and mla_out_proj in one launch
 * (decompression and attention as one layer, page section
 * "源码里的压缩全流程").  For every (b, h) the kernel for head h builds
 * o_lat[b,h] in shared memory -- read from o_lat where mla_decode finished
 * the sequence, merged from the workspace's partials where it was split --
 * and multiplies it by W_UV[h] there, so a merged latent is not read back
 * from memory before its product.  Results equal mla_split_kv_combine
 * followed by mla_out_proj whenever mla_split_kv_combine takes its grouped
 * form (B * ceil(H/8) >= 2 x the SM count), and agree to rounding otherwise.
 * Must follow mla_decode on the same stream with the same params,
 * num_splits, workspace and seq_lens.
 *   seq_lens : [B] int32 device, the array mla_decode was given, unchanged
 *           since: the decode's KV partition is a function of the lengths
 *           alone, so the kernel works out which partials to merge from them
 *           while the decode is still running (it reads them before waiting
 *           for the decode to finish)
 *   o_lat : [B,H,512] bf16, read (finished sequences) and written (split
 *           sequences);  lse : [B,H] fp32 or NULL, written for split sequences
 *   w_uv, out : as mla_out_proj
 * Errors: MLA_ERR_INVALID_ARG for a null seq_lens, o_lat, w_uv or out or a
 * misaligned pointer; MLA_ERR_WORKSPACE as mla_split_kv_combine.
 */
mla_status mla_combine_out_proj(const mla_params* p, const void* workspace, size_t ws_bytes, int num_splits,
                                const int32_t* seq_lens, void* o_lat, float* lse, const void* w_uv, void* out,
                                mla_stream_t stream);

/* ---------------------------------------------------------------------
 * mla_cache_append: write T new tokens into the paged cache (the step before
 * decode, page section "源码里的压缩全流程": the down-projection row is split into the
 * 512-d latent and the 64-d k_pe, the latent is RMS-normalised, RoPE is
 * applied to k_pe only, and both are written to the cache).
 *   kv_rows   : [T,576] bf16 down-projection rows (512 latent, 64 raw k_pe)
 *   slots     : [T] int32 physical slot, page*64 + offset
 *   positions : [T] int32 token positions for RoPE
 *   flags     : MLA_APPEND_RMSNORM | MLA_APPEND_ROPE (0 stores rows as given)
 * Latent: x / sqrt(mean(x^2)) (gain 1, eps 0), rounded to bf16.
 * k_pe: half-split RoPE (pair i with i+32, angle pos*10000^(-i/32)),
 * computed in fp64, rounded to bf16.  For the E4M3 kv_dtypes the bf16 row is then
 * quantised with one fp32 scale per token, scale = max|v| / 448 (1 for a
 * zero row), code = E4M3(v / scale) with fp32 division, round to nearest
 * even, saturating; kv_scale[slot] receives the scale.
 * A slot outside [0, num_pages*64) is skipped (no error word: no workspace).
 */
#define MLA_APPEND_RMSNORM 1
#define MLA_APPEND_ROPE 2
mla_status mla_cache_append(const mla_params* p, const void* kv_rows, const int32_t* slots,
                            const int32_t* positions, int T, int flags, void* ckv_cache,
                            void* kpe_cache, float* kv_scale, mla_stream_t stream);

/* mla_rope_q: rotate the query key-part of each sequence at its decode
 * position seq_lens[b]-1 (same rotation as mla_cache_append).
 *   q_pe_raw : [B,H,64] bf16;  seq_lens : [B] int32;  q_pe : [B,H,64] bf16
 */
mla_status mla_rope_q(const mla_params* p, const void* q_pe_raw, const int32_t* seq_lens,
                      void* q_pe, mla_stream_t stream);

/* ---------------------------------------------------------------------
 * mla_multi_token_expand: several query tokens per sequence (speculative or
 * multi-token decode, with a causal mask).  The page's forward flow applies
 * to every new token; with T new tokens the T newest cache positions of a
 * sequence of n cached tokens are the queries (their rows already in the
 * cache), token i at position n - T + i, and token i attends to cache
 * tokens 0 .. n - T + i.  That is the one-token decode of a sequence of
 * length n - T + 1 + i over the same pages, so this call writes, for the
 * B sequences of p, B*T rows r = b*T + i:
 *   page_table_out[r][:] = page_table[b][:]    [B*T, max_pages_per_seq] int32
 *   seq_lens_out[r]      = seq_lens[b] - T + 1 + i            [B*T] int32
 * and the caller runs mla_rope_q, mla_absorb_q, mla_decode,
 * mla_split_kv_combine and mla_out_proj with B*T in place of B, on queries
 * laid out [B,T,H,...] (= [B*T,H,...]) and these two arrays; the output is
 * [B,T,H,128].  Requires seq_lens[b] >= T on the device (a shorter sequence
 * yields a row of length < 1, which mla_decode reports as MLA_ERR_SEQ_LEN).
 *   q_len : T >= 1;  page_table, seq_lens : as for mla_decode (B rows)
 *   page_table_out, seq_lens_out : caller-allocated device buffers
 */
mla_status mla_multi_token_expand(const mla_params* p, int q_len, const int32_t* page_table,
                                  const int32_t* seq_lens, int32_t* page_table_out, int32_t* seq_lens_out,
                                  mla_stream_t stream);

/* ---------------------------------------------------------------------
 * mla_decode_static: mla_decode followed by mla_split_kv_combine, for
 * callers that cannot allocate device memory.  The pages have no counterpart:
 * this is a calling convention, not a step of the method.
 * Some callers are handed their input and output buffers but may not create
 * any of their own: a plugin inside a host application or serving runtime
 * that has reserved all device memory in its own pool, or a latency-critical
 * path where cudaMalloc (which can synchronise the device) is not allowed.
 * This entry point needs no workspace argument: its scratch is a fixed
 * 32 MiB array inside the library's device image, which every GPU that
 * loads the library keeps until the process exits.  It allocates nothing
 * and calls no allocating routine.
 *   Arguments: as mla_decode, without num_splits and the workspace; the KV
 *   partition count is the automatic one, lowered until the scratch fits.
 *   Returns MLA_ERR_WORKSPACE when even one partition does not fit (very
 *   large B*H); other host-side errors as mla_decode.
 *   Device-side faults are handled as in mla_decode (a bad page id or
 *   length skips that work; a bounded wait that runs out, an internal
 *   fault, stops the kernel with MLA_ERR_TIMEOUT and leaves the outputs
 *   partial).  They are recorded in the array's error word, which every
 *   call clears when it starts: read it with mla_decode_static_status.
 * The first call on a device looks up the array's device address for that
 * device (once, with the device current) and keeps it for the life of the
 * process; make that first call before any stream capture.  A device reset
 * (cudaDeviceReset) reloads the library's device image and invalidates the
 * kept address: do not call this entry point after one.  All calls share
 * the one array, and each call keeps the previous call's contents until it
 * overwrites them: calls that overlap on the GPU (other streams, other
 * threads) race and must be serialised by the caller. */
mla_status mla_decode_static(const mla_params* p, const void* q_lat, const void* q_pe,
                             const void* ckv_cache, const void* kpe_cache, const float* kv_scale,
                             const int32_t* page_table, const int32_t* seq_lens, void* o_lat,
                             float* lse, mla_stream_t stream);

/* mla_decode_static_status: the error word of mla_decode_static's fixed
 * scratch, as a status (MLA_OK, MLA_ERR_PAGE_OOB, MLA_ERR_SEQ_LEN or
 * MLA_ERR_TIMEOUT), for the most recent mla_decode_static call enqueued on
 * `stream` (each call clears the word when it starts).  Copies the word to
 * the host and synchronises `stream`; clears it when `clear` is non-zero.
 * Allocates nothing. */
mla_status mla_decode_static_status(int clear, mla_stream_t stream);

/* mla_workspace_status: copy the workspace's sticky error word to the host
 * (synchronises `stream`) and return it as a status; clear it when `clear`
 * is non-zero. */
mla_status mla_workspace_status(void* workspace, int clear, mla_stream_t stream);

/* ---------------------------------------------------------------------
 * mla_selftest_bounded_wait: diagnostic of the kernels' bounded waits (not a
 * step of the method).  Every mbarrier wait in the library's kernels gives up
 * after 2 s of global time, records MLA_ERR_TIMEOUT in the workspace's error
 * word and lets the kernel return.  This call launches one block that waits
 * on an mbarrier nothing completes; after the limit the error word of
 * `workspace` (4 bytes at offset 0, zeroed by the caller) holds
 * MLA_ERR_TIMEOUT (read it with mla_workspace_status) and the stream goes
 * on.  The kernel takes about 2 s.
 */
mla_status mla_selftest_bounded_wait(void* workspace, mla_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
