// Query absorption and value out-projection on the tcgen05 tensor cores.
//
//   absorb:   q_lat[b,h,m] = sum_n W_UK[h,n,m] q_nope[b,h,n]   M=latent (4 tiles of 128), K=128
//   out_proj: out[b,h,v]   = sum_k W_UV[h,v,k] o_lat[b,h,k]    M=v (128), K=512
//
// Both are the key and value halves of kv_b_proj (mtrt.cn DeepSeek-Coder-V2
// MLA page, section "源码里的压缩全流程", KV decompression) applied on the
// query and output side.  The batch (rounded up to 16) is the MMA's N
// dimension, the weights stream once by TMA into 128-byte-swizzled shared
// memory and the accumulators live in tensor memory.  The absorption takes
// one CTA per head (its four 128-row M tiles of W_UK, read with the latent
// axis as M, i.e. as an MN-major A operand); the out-projection one CTA per
// head's [128 x N] tile (W_UV K-major).
#include <algorithm>

#include "combine.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr uint32_t kABytes = 16384;  // A bytes per 64-wide K block

struct GemmTcArgs {
  int B, H, N;
  int S;                        // out-projection: pipeline stages (K blocks in flight), at most kMaxS
  const __nv_bfloat16* weight;  // [H,128,512]: prefetched into L2 before the dependency wait
  void* out;
  int out_kind;  // absorption: q_lat bf16 [B,H,512] (unused); out-projection: 1 fp32, 2 bf16 [B,H,128]
};

constexpr int kMaxS = 8;

__global__ void __launch_bounds__(128, 1)
    outproj_tc_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                      GemmTcArgs g) {
  constexpr int KB = 8;  // K blocks of 64
  const int S = g.S;                      // pipeline stages
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxS + 1];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t b_bytes = (uint32_t)g.N * 128u;
  const uint32_t stage = kABytes + b_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, nt = blockIdx.z;
  const uint32_t full = smem_u32(&bars[0]), empty = smem_u32(&bars[kMaxS]), done = smem_u32(&bars[2 * kMaxS]);
  const uint32_t ncols = g.N <= 32 ? 32 : g.N <= 64 ? 64 : g.N <= 128 ? 128 : 256;

  // the out-projection follows the combine: its weight slice (independent of
  // the combine) is pulled into L2 while the combine runs
  if (threadIdx.x == 32 && nt == 0) prefetch_l2(g.weight + (size_t)h * kV * kLatent, kV * kLatent * 2);
  grid_dep_wait();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(full + 8 * i, 1);
      mbar_init(empty + 8 * i, 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    prefetch_tmap(&tA);
    prefetch_tmap(&tB);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0 && lane == 0) {
    // TMA producer
    int issued = 0;
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % S;
      if (kb >= S && !mbar_wait(empty + 8 * s, ((kb / S) - 1) & 1, &abort_flag, nullptr)) break;
      const uint32_t a_s = base + s * stage, b_s = a_s + kABytes;
      mbar_expect_tx(full + 8 * s, stage);
      tma_load_2d(a_s, &tA, full + 8 * s, kb * 64, h * 128);
      tma_load_3d(b_s, &tB, full + 8 * s, kb * 64, h, nt * g.N);
      ++issued;
    }
    if (abort_flag) {  // let copies in flight land before the CTA exits
      for (int kb = issued - 1; kb >= 0 && kb >= issued - S; --kb) {
        volatile int no_abort = 0;
        mbar_wait(full + 8 * (kb % S), (kb / S) & 1, &no_abort, nullptr);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    const uint32_t idesc = idesc_bf16(128, g.N, false, false);
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % S;
      if (!mbar_wait(full + 8 * s, (kb / S) & 1, &abort_flag, nullptr)) break;
      tc_fence_after();
      const uint32_t a_s = base + s * stage, b_s = a_s + kABytes;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // K-major operands advance 32 B per 16-wide K step
        const uint64_t ad = sdesc_sw128(a_s + k * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(b_s + k * 32, 16, 1024);
        mma_bf16_ss(tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
      }
      mma_commit(empty + 8 * s);
    }
    mma_commit(done);
  }
  __syncwarp();

  // epilogue: thread = accumulator row (TMEM lane), columns = batch
  const bool ok = mbar_wait(done, 0, &abort_flag, nullptr) && !abort_flag;
  tc_fence_after();
  const int row = warp * 32 + lane;
  for (int c0 = 0; c0 < g.N; c0 += 16) {
    uint32_t r[16];
    tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, r);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int b = nt * g.N + c0 + j;
      if (b >= g.B) break;
      const float v = ok ? __uint_as_float(r[j]) : __int_as_float(0x7fc00000);
      const size_t bh = (size_t)b * g.H + h;
      if (g.out_kind == 1)
        static_cast<float*>(g.out)[bh * kV + row] = v;
      else
        static_cast<__nv_bfloat16*>(g.out)[bh * kV + row] = __float2bfloat16_rn(v);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ---------------------------------------------------------------- q absorption
// One CTA of 128 x kAbsorbTiles threads per (head, group of kAbsorbTiles
// 128-row M tiles of W_UK^T, batch tile): the group's W_UK slice (32 KB per
// tile) goes out by TMA at once, one barrier per tile, followed by the
// q_nope rows; each tile accumulates in its own tensor-memory accumulator,
// and warp w writes tile w / 4 from the lanes of its sub-partition.  With
// all four tiles in one CTA, q_nope is read once per head and a quarter as
// many CTAs are launched as with one tile per CTA.
constexpr int kAbsorbTiles = 4;
constexpr int kAbsorbMaxN = 128;  // four accumulators of N columns fill the 512

template <int kTiles>
__global__ void __launch_bounds__(128 * kTiles, 1)
    absorb_tc_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                     GemmTcArgs g) {
  static_assert(kTiles == 1 || kTiles == 2 || kTiles == 4, "tiles per CTA");
  constexpr int kQ = kTiles;          // barrier: q_nope landed
  constexpr int kDone = kTiles + 1;   // barriers: tile lt done
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kTiles + 1];  // [0, kTiles) W_UK tile lt landed
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t b_blk = (uint32_t)g.N * 128u;               // one 64-wide K block of q_nope
  const uint32_t bbase = base + 2u * kTiles * kABytes;       // A: kTiles tiles x 2 K blocks
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, mt0 = blockIdx.y * kTiles, nt = blockIdx.z;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t acols = g.N <= 32 ? 32 : g.N <= 64 ? 64 : 128;

  // q absorption opens a decode step: the decode kernel may launch at once
  grid_dep_trigger();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < 2 * kTiles + 1; ++i) mbar_init(bar(i), 1);
    fence_mbar_init();
    prefetch_tmap(&tA);
    prefetch_tmap(&tB);
    // W_UK does not depend on the preceding kernel: all of it goes out now
    for (int lt = 0; lt < kTiles; ++lt) {
      const int mt = mt0 + lt;
      mbar_expect_tx(bar(lt), 2 * kABytes);
      for (int kb = 0; kb < 2; ++kb) {
        const uint32_t a_s = base + (uint32_t)(lt * 2 + kb) * kABytes;
        tma_load_2d(a_s, &tA, bar(lt), mt * 128, h * 128 + kb * 64);
        tma_load_2d(a_s + 8192, &tA, bar(lt), mt * 128 + 64, h * 128 + kb * 64);
      }
    }
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_slot), kTiles * acols);
    tmem_relinquish();
  }
  grid_dep_wait();  // q_nope may be written by the preceding kernel
  if (threadIdx.x == 0) {
    mbar_expect_tx(bar(kQ), 2 * b_blk);
    for (int kb = 0; kb < 2; ++kb) tma_load_3d(bbase + kb * b_blk, &tB, bar(kQ), kb * 64, h, nt * g.N);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 1 && lane == 0) {
    // MMA issuer: each tile as soon as its W_UK slice has landed; A is the
    // MN-major weight (16 K-rows = 2 KB per MMA), B the K-major q_nope rows
    const uint32_t idesc = idesc_bf16(128, g.N, true, false);
    bool ok = mbar_wait(bar(kQ), 0, &abort_flag, nullptr);
    for (int lt = 0; ok && lt < kTiles; ++lt) {
      if (!mbar_wait(bar(lt), 0, &abort_flag, nullptr)) break;
      tc_fence_after();
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        const uint32_t a_s = base + (uint32_t)(lt * 2 + kb) * kABytes, b_s = bbase + kb * b_blk;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16_ss(tmem + lt * acols, sdesc_sw128(a_s + k * 2048, 8192, 1024),
                      sdesc_sw128(b_s + k * 32, 16, 1024), idesc, (kb | k) != 0 ? 1u : 0u);
      }
      mma_commit(bar(kDone + lt));
    }
  }
  __syncwarp();

  // epilogue: warp w writes tile lt = w / 4 (latent columns [128 mt, 128 mt
  // + 128)); thread = latent column, columns of the accumulator = batch.  The
  // warp's [N x 32] bf16 block is staged in the tile's own W_UK buffer (its
  // MMAs are done) and leaves in 16-byte stores along the latent axis.
  const int lt = warp >> 2, q = warp & 3;
  const bool ok = mbar_wait(bar(kDone + lt), 0, &abort_flag, nullptr) && !abort_flag;
  tc_fence_after();
  const uint32_t stg = base + (uint32_t)lt * 2u * kABytes + (uint32_t)q * 8192u;  // N x 64 B <= 8 KB
  for (int c0 = 0; c0 < g.N; c0 += 16) {
    uint32_t r[16];
    tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(lt * acols + c0), r);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float v = ok ? __uint_as_float(r[j]) : __int_as_float(0x7fc00000);
      const __nv_bfloat16 hv = __float2bfloat16_rn(v);
      asm volatile("st.shared.b16 [%0], %1;" ::"r"(stg + (uint32_t)((c0 + j) * 32 + lane) * 2u),
                   "h"(*reinterpret_cast<const uint16_t*>(&hv))
                   : "memory");
    }
  }
  __syncwarp();
  const int col0 = (mt0 + lt) * 128 + q * 32;
  for (int k = lane; k < g.N * 4; k += 32) {  // 16-byte chunk p of batch row bl
    const int bl = k >> 2, p = k & 3, b = nt * g.N + bl;
    if (b >= g.B) break;
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(stg + (uint32_t)(bl * 64 + p * 16))
                 : "memory");
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g.out) + ((size_t)b * g.H + h) * kLatent + col0 + p * 8) = v;
  }
  if (abort_flag && threadIdx.x == 0) {  // copies in flight land before the CTA exits
    for (int i = 0; i <= kQ; ++i) {
      volatile int no_abort = 0;
      mbar_wait(bar(i), 0, &no_abort, nullptr);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTiles * acols);
  }
}

// ---------------------------------------------------------------- combine + out-projection
// The split-KV combine fused into the out-projection: CTA (head h, batch
// tile) builds its B operand, o_lat[b, h, :] for the tile's sequences, in
// shared memory -- read from o_lat for a sequence the decode finished, merged
// from the partials (warp_merge_partials, the grouped combine's arithmetic)
// for a split one, which is also written to o_lat / lse -- while W_UV[h]
// streams in by TMA; then the same MMAs as the out-projection.  The merged
// latent never leaves the SM before its product.
struct FusedArgs {
  int B, H, N, S, G;
  const __nv_bfloat16* weight;  // W_UV, prefetched into L2 before the dependency wait
  const __nv_bfloat16* part_o;
  const float* part_lse;
  const int32_t* seq_lens;  // the lengths mla_decode was given (its schedule is a function of them)
  int maxp;
  __nv_bfloat16* o_lat;
  float* lse;
  void* out;
  int out_bf16;
};

constexpr int kFusedThreads = 512;  // 16 warps: two B-operand rows per warp at N = 32
constexpr int kFusedMaxN = 128;

__global__ void __launch_bounds__(kFusedThreads, 1)
    outproj_combine_kernel(const __grid_constant__ CUtensorMap tA, FusedArgs g) {
  constexpr int KB = 8;  // K blocks of 64 latent columns
  const int S = g.S;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxS + 1];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ SeqWorkers s_sw[kFusedMaxN];  // the decode workers of each row's sequence
  __shared__ int s_slot[kFusedMaxN][4];    // and the partial slots of its first four
  __shared__ long long s_sb[kFusedMaxN];   // first flattened page of each row's sequence
  __shared__ int s_np[kFusedMaxN];         // and its page count
  __shared__ long long s_P;                // the batch's page count

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bblk = (uint32_t)g.N * 128u;                 // one K block of the B operand
  const uint32_t bbase = base + (uint32_t)S * kABytes;         // B operand: KB blocks of [N x 128 B]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, nt = blockIdx.z;
  const uint32_t full = smem_u32(&bars[0]), empty = smem_u32(&bars[kMaxS]), done = smem_u32(&bars[2 * kMaxS]);
  const uint32_t ncols = g.N <= 32 ? 32 : g.N <= 64 ? 64 : 128;

  // W_UV and the decode's schedule (a function of the lengths alone) do not
  // depend on the decode: the set-up, the weight's first S K blocks and each
  // row's workers and partial slots are done before the dependency wait,
  // while the decode's last clusters finish
  const int b0 = nt * g.N, nrows = min(g.N, g.B - b0);
  if (threadIdx.x == 32) prefetch_l2(g.weight + (size_t)h * kV * kLatent, kV * kLatent * 2);
  if (warp == 3) {
    const long long P = warp_page_offsets(g.seq_lens, g.B, g.maxp, b0, nrows, s_sb, s_np);
    if (lane == 0) s_P = P;
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(full + 8 * i, 1);
      mbar_init(empty + 8 * i, 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    prefetch_tmap(&tA);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  int issued = 0;  // (producer thread)
  auto issue = [&](int kb) {
    const int s = kb % S;
    const uint32_t a_s = base + s * kABytes;
    mbar_expect_tx(full + 8 * s, kABytes);
    tma_load_2d(a_s, &tA, full + 8 * s, kb * 64, h * 128);
    ++issued;
  };
  if (warp == 0 && lane == 0)
    for (int kb = 0; kb < S && kb < KB; ++kb) issue(kb);
  if (threadIdx.x >= 64 && (int)threadIdx.x - 64 < nrows) {
    const int r = threadIdx.x - 64;
    SeqWorkers sw;
    sw.P = s_P;
    sw.sb = s_sb[r];
    const long long se = sw.sb + s_np[r];
    sw.wf = 0;
    sw.n = 0;
    if (se > sw.sb) {
      sw.wf = worker_of(sw.sb, g.G, sw.P);
      sw.n = worker_of(se - 1, g.G, sw.P) - sw.wf + 1;
    }
    s_sw[r] = sw;
#pragma unroll
    for (int u = 0; u < 4; ++u) s_slot[r][u] = u < sw.n ? partial_slot(sw, g.G, u) : -1;
  }
  __syncthreads();
  grid_dep_wait();  // the decode's o_lat and partials

  // B operand rows: warp w takes rows w + 32 k and w + 32 k + 16; lane l
  // holds latent columns [16 l, 16 l + 16), i.e. 16-byte chunks 2(l%4),
  // 2(l%4)+1 of K block l/4.  Two rows split over 2..4 workers are merged
  // together (their loads in flight at once), any other row on its own.
  auto small_split = [&](int r) { return r < nrows && s_sw[r].n >= 2 && s_sw[r].n <= 4; };
  auto write_merged = [&](int r, const float (&acc)[16], float l, uint32_t (&o8)[8]) {
    const int b = nt * g.N + r;
    pack_row16(acc, o8);
    uint4* row = reinterpret_cast<uint4*>(g.o_lat + ((size_t)b * g.H + h) * kLatent) + 2 * lane;
    row[0] = make_uint4(o8[0], o8[1], o8[2], o8[3]);
    row[1] = make_uint4(o8[4], o8[5], o8[6], o8[7]);
    if (lane == 0 && g.lse) g.lse[(size_t)b * g.H + h] = l;
  };
  auto one_row = [&](int r, uint32_t (&o8)[8]) {
    const int b = nt * g.N + r;
#pragma unroll
    for (int e = 0; e < 8; ++e) o8[e] = 0;
    if (b >= g.B) return;
    const SeqWorkers sw = s_sw[r];
    if (sw.n <= 1) {  // finished by the decode (or empty)
      const uint4* row = reinterpret_cast<const uint4*>(g.o_lat + ((size_t)b * g.H + h) * kLatent) + 2 * lane;
      const uint4 v0 = row[0], v1 = row[1];
      o8[0] = v0.x; o8[1] = v0.y; o8[2] = v0.z; o8[3] = v0.w;
      o8[4] = v1.x; o8[5] = v1.y; o8[6] = v1.z; o8[7] = v1.w;
    } else {
      float acc[16];
      const float l = warp_merge_partials(g.part_o, g.part_lse, sw, g.G, g.H, h, acc);
      write_merged(r, acc, l, o8);
    }
  };
  auto store_row = [&](int r, const uint32_t (&o8)[8]) {
    const uint32_t blk = bbase + (uint32_t)(lane >> 2) * bblk + (uint32_t)r * 128u;
    const uint32_t c0 = 2u * (lane & 3);
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(blk + ((c0 ^ (r & 7)) << 4)), "r"(o8[0]), "r"(o8[1]),
                 "r"(o8[2]), "r"(o8[3])
                 : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(blk + (((c0 + 1) ^ (r & 7)) << 4)), "r"(o8[4]),
                 "r"(o8[5]), "r"(o8[6]), "r"(o8[7])
                 : "memory");
  };
  for (int r0 = warp; r0 < g.N; r0 += 2 * (kFusedThreads / 32)) {
    const int r1 = r0 + kFusedThreads / 32;
    uint32_t o8[2][8];
    if (small_split(r0) && small_split(r1)) {
      const int sl2[2] = {lane < 4 ? s_slot[r0][lane] : -1, lane < 4 ? s_slot[r1][lane] : -1};
      const int n2[2] = {s_sw[r0].n, s_sw[r1].n};
      float acc[2][16], l[2];
      warp_merge_two_small(g.part_o, g.part_lse, sl2, n2, g.H, h, acc, l);
      write_merged(r0, acc[0], l[0], o8[0]);
      write_merged(r1, acc[1], l[1], o8[1]);
    } else {
      one_row(r0, o8[0]);
      if (r1 < g.N) one_row(r1, o8[1]);
    }
    store_row(r0, o8[0]);
    if (r1 < g.N) store_row(r1, o8[1]);
  }
  fence_proxy_async_smem();  // the B operand, for the tensor cores
  __syncthreads();

  if (warp == 0 && lane == 0) {
    // the rest of the weight's K blocks
    for (int kb = S; kb < KB; ++kb) {
      const int s = kb % S;
      if (!mbar_wait(empty + 8 * s, ((kb / S) - 1) & 1, &abort_flag, nullptr)) break;
      issue(kb);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16(128, g.N, false, false);
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % S;
      if (!mbar_wait(full + 8 * s, (kb / S) & 1, &abort_flag, nullptr)) break;
      tc_fence_after();
      const uint32_t a_s = base + s * kABytes, b_s = bbase + kb * bblk;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_bf16_ss(tmem, sdesc_sw128(a_s + k * 32, 16, 1024), sdesc_sw128(b_s + k * 32, 16, 1024), idesc,
                    (kb | k) != 0 ? 1u : 0u);
      mma_commit(empty + 8 * s);
    }
    mma_commit(done);
  }
  __syncwarp();

  // epilogue: warp w reads the tensor-memory lanes of its sub-partition
  // (w % 4: 32 v rows, thread = v row) and batch columns [8 (w / 4), +8) of
  // every 32, so all 16 warps share the stores
  {
    const bool ok = mbar_wait(done, 0, &abort_flag, nullptr) && !abort_flag;
    tc_fence_after();
    const int q = warp & 3, row = q * 32 + lane;
    for (int c0 = (warp >> 2) * 8; c0 < g.N; c0 += 32) {
      uint32_t r[8];
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                   : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                   : "r"(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0)
                   : "memory");
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int b = nt * g.N + c0 + j;
        if (b >= g.B) break;
        const float v = ok ? __uint_as_float(r[j]) : __int_as_float(0x7fc00000);
        const size_t bh = (size_t)b * g.H + h;
        if (g.out_bf16)
          static_cast<__nv_bfloat16*>(g.out)[bh * kV + row] = __float2bfloat16_rn(v);
        else
          static_cast<float*>(g.out)[bh * kV + row] = v;
      }
    }
  }
  if (abort_flag && warp == 0 && lane == 0) {  // copies in flight land before the CTA exits
    for (int kb = issued - 1; kb >= 0 && kb >= issued - S; --kb) {
      volatile int no_abort = 0;
      mbar_wait(full + 8 * (kb % S), (kb / S) & 1, &no_abort, nullptr);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

int batch_tile(int B) {
  const int n = (B + 15) / 16 * 16;
  return n < 256 ? n : 256;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_absorb_tc(const __nv_bfloat16* q_nope, const __nv_bfloat16* w_uk,
                             __nv_bfloat16* q_lat, int B, int H, cudaStream_t stream) {
  if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(q_lat)) return cudaErrorInvalidValue;
  const int N = std::min(batch_tile(B), kAbsorbMaxN);
  CUtensorMap tA, tB;
  const cuuint64_t ad[2] = {kLatent, (cuuint64_t)H * kNope}, as[1] = {kLatent * 2};
  const cuuint32_t abox[2] = {64, 64};
  const cuuint64_t bd[3] = {kNope, (cuuint64_t)H, (cuuint64_t)B},
                   bs[2] = {kNope * 2, (cuuint64_t)H * kNope * 2};
  const cuuint32_t bbox[3] = {64, 1, (cuuint32_t)N};
  if (!make_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_uk, ad, as, abox) ||
      !make_tmap(&tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q_nope, bd, bs, bbox))
    return cudaErrorInvalidValue;
  GemmTcArgs g{B, H, N, 0, w_uk, q_lat, 0};
  const size_t smem = 2 * kAbsorbTiles * kABytes + 2 * (size_t)N * 128 + 1024;
  auto kernel = absorb_tc_kernel<kAbsorbTiles>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(H, 4 / kAbsorbTiles, (B + N - 1) / N);
  kernel<<<grid, 128 * kAbsorbTiles, smem, stream>>>(tA, tB, g);
  return cudaGetLastError();
}

cudaError_t launch_out_proj_tc(const __nv_bfloat16* o_lat, const __nv_bfloat16* w_uv, void* out,
                               bool out_bf16, int B, int H, cudaStream_t stream) {
  if (!aligned16(o_lat) || !aligned16(w_uv)) return cudaErrorInvalidValue;
  const int N = batch_tile(B);
  CUtensorMap tA, tB;
  const cuuint64_t ad[2] = {kLatent, (cuuint64_t)H * kV}, as[1] = {kLatent * 2};
  const cuuint32_t abox[2] = {64, 128};
  const cuuint64_t bd[3] = {kLatent, (cuuint64_t)H, (cuuint64_t)B},
                   bs[2] = {kLatent * 2, (cuuint64_t)H * kLatent * 2};
  const cuuint32_t bbox[3] = {64, 1, (cuuint32_t)N};
  if (!make_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_uv, ad, as, abox) ||
      !make_tmap(&tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o_lat, bd, bs, bbox))
    return cudaErrorInvalidValue;
  // as many of the 8 K blocks in flight as shared memory holds (all 8 for
  // batches up to 112): the weight slice streams in one go
  const size_t stage = kABytes + (size_t)N * 128;
  const int S = (int)std::min<size_t>(kMaxS, (200u << 10) / stage);
  GemmTcArgs g{B, H, N, S, w_uv, out, out_bf16 ? 2 : 1};
  const size_t smem = S * stage + 1024;
  cudaError_t e = cudaFuncSetAttribute(outproj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(H, 1, (B + N - 1) / N);
  return launch_dependent(outproj_tc_kernel, grid, dim3(128), smem, stream, tA, tB, g);
}

cudaError_t launch_outproj_combine(const __nv_bfloat16* part_o, const float* part_lse, const int32_t* seq_lens,
                                   int maxp, __nv_bfloat16* o_lat, float* lse, const __nv_bfloat16* w_uv,
                                   void* out, bool out_bf16, int B, int H, int G, cudaStream_t stream) {
  if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(part_o)) return cudaErrorInvalidValue;
  const int N = std::min(batch_tile(B), kFusedMaxN);
  CUtensorMap tA;
  const cuuint64_t ad[2] = {kLatent, (cuuint64_t)H * kV}, as[1] = {kLatent * 2};
  const cuuint32_t abox[2] = {64, 128};
  if (!make_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_uv, ad, as, abox)) return cudaErrorInvalidValue;
  // the B operand (N KB) stays; as many weight K blocks in flight as fit
  const size_t bbytes = (size_t)N * 128 * 8;
  const int S = (int)std::min<size_t>(kMaxS, ((200u << 10) - bbytes) / kABytes);
  FusedArgs g{B, H, N, S, G, w_uv, part_o, part_lse, seq_lens, maxp, o_lat, lse, out, out_bf16 ? 1 : 0};
  const size_t smem = S * kABytes + bbytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(outproj_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(H, 1, (B + N - 1) / N);
  return launch_dependent(outproj_combine_kernel, grid, dim3(kFusedThreads), smem, stream, tA, g);
}

}  // namespace mla
