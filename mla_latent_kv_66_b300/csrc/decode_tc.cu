// Latent-attention decode on the tcgen05 tensor cores.
//
// Method (mtrt.cn DeepSeek-Coder-V2 MLA page, forward flow; absorbed form):
//   s_t = scale * (q_lat . c_t + q_pe . k_pe_t),  o_lat = sum_t softmax(s)_t c_t
// for all H <= 128 heads of one sequence at once: the heads are the M = 128
// rows of every MMA, so each 64-token cache page is read from HBM once and
// shared by all heads.  Three cache modes (template parameter kMode):
//   0  bf16 cache, kind::f16 MMAs;
//   1  E4M3 cache + fp32 scale per token, the codes expanded exactly to bf16
//      in shared memory by the exchange warps, kind::f16 MMAs;
//   2  the same E4M3 cache multiplied as codes by kind::f8f6f4 MMAs, with the
//      query and the probabilities as E4M3 terms (hotdry.top DeepSeek-V3.2-Exp
//      MLA page, deployment paragraph: FP8 when serving).
//
// The fp32 latent accumulator O[128 heads x 512] alone needs all 512 tensor
// memory columns of an SM, so a cluster of two CTAs splits the latent axis
// and the shared RoPE key evenly:
//   rank 0: latent columns [0,256), k_pe [0,32);
//   rank 1: latent columns [256,512), k_pe [32,64).
// Each CTA TMA-loads only its part of every page and computes the partial
// score over its 288 of the 576 dimensions.  The two fp32 partial score tiles
// (log2 domain) are swapped through distributed shared memory by the async
// copy engine; each CTA adds its own partial to the peer's, so both add the
// same two numbers exactly and take the same softmax decisions.  Each CTA
// then accumulates P . c over its own 256 latent columns.
//
// Warp roles (512 threads):
//   warp 0       KV-partition schedule and the first page ids, then the TMA
//                producer (cache pages, stage ring; bf16 pages evict-first
//                in the L2); one stage load is issued before the CTA-wide
//                start-up barrier, the rest of the ring once the first
//                unit's query is in
//   warp 1       MMA issuer for S = Q K^T (A = query in tensor memory)
//   warp 2       tensor-memory allocation
//   warp 3       split records; then MMA issuer for O += P V (a separate
//                issuer lets S = Q K^T run ahead)
//   warps 4..7   exchange: copy each partial score tile out of tensor memory
//                as soon as its S = Q K^T completes (S has one buffer), stage
//                it in shared memory and send each warp's 32 rows to the peer
//                CTA with one bulk copy (one tile each way, each row quarter
//                on its own: warp q hands quarter q back to the peer as soon
//                as its two softmax warps have read it); load each unit's
//                query into tensor memory as soon as the previous unit's last
//                S = Q K^T is done; mode 1: expand the codes; mode 2: load the
//                first unit's query too, publish each page's token-scale
//                logarithms and reciprocals
//   warps 8..15  two softmax warpgroups (mode 0 and 1: the first unit's
//                query into tensor memory first, mode 0 by TMA through two
//                ring stages that are still free); warpgroup j owns tokens
//                [32j, 32j+32) of every page, thread = head row: own staged
//                partial + the peer's, row maximum agreed with the other
//                warpgroup, online softmax with lazy rescaling, its half of P
//                into tensor memory (two P buffers), its half of O rescaled
//                when needed and written at the end of a unit.
// Tensor memory: O [0,256), S [256,320), P double buffer [320,384) (bf16
// pairs, or E4M3 terms), query [384,512).
#include <cuda_fp16.h>

#include "kernels.h"
#include "tc.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr uint32_t kBox = 8192;            // [64 rows x 64 bf16], 128-byte swizzle
constexpr uint32_t kKpeBox = 4096;         // [64 rows x 32 bf16], 64-byte swizzle
constexpr uint32_t kStageBf = 4 * kBox + kKpeBox;  // bf16 stage: 4 latent boxes + this CTA's k_pe half
// Partial-score tile: [128 head rows x 64 tokens] fp32, as four slabs of 32
// rows (one per exchange warp, 8 KB each).
constexpr uint32_t kSlab = 32 * 256;
constexpr uint32_t kXBytes = 4 * kSlab;
// E4M3 cache: a raw page holds this CTA's 256 latent codes of 64 tokens as two
// [64 x 128 B] boxes, its 32 rope codes ([64 x 32 B]) and the page's 64 fp32
// scales; after expansion the bf16 stage also carries the scales.
constexpr uint32_t kRawKpe = 2 * 8192, kRawScale = kRawKpe + 2048, kRawBytes = kRawScale + 256;
// E4M3 cache on the 8-bit tensor cores: a stage holds the codes as the MMAs
// read them, two [64 x 128 B] latent boxes (128-byte swizzle), the
// [64 x 32 B] RoPE box (32-byte swizzle) and the page's 64 scales.
constexpr uint32_t kStage8Kpe = 2 * 8192, kStage8Scale = kStage8Kpe + 2048, kStage8Bytes = 19 * 1024;
static_assert(kStage8Kpe == kRawKpe && kStage8Scale == kRawScale, "one copy schedule for both E4M3 layouts");
constexpr int kMaxStages = 7;

// kMode: 0 bf16 cache; 1 E4M3 cache expanded exactly to bf16; 2 E4M3 cache on
// the 8-bit tensor cores (E4M3 query and probabilities).
template <int kMode>
struct Layout {
  static constexpr bool kExp = kMode == 1, kMma8 = kMode == 2;
  static constexpr int kStages = kMma8 ? 7 : kExp ? 3 : 4;   // stages the MMAs read
  static constexpr int kRaw = kExp ? 2 : 0;                  // raw E4M3 pages (expanded path)
  static constexpr uint32_t kStageBytes = kMma8 ? kStage8Bytes : kExp ? kStageBf + 1024 : kStageBf;
  static constexpr uint32_t kStageScale = kMma8 ? kStage8Scale : kStageBf;  // token scales in a stage
  static constexpr uint32_t kOffRaw = kStages * kStageBytes;
  // query RoPE part (A operand of the RoPE MMAs): bf16 [128 x 32], 64-byte
  // swizzle; 8-bit: two E4M3 terms of [128 x 32 B], 32-byte swizzle, 4 KB apart
  static constexpr uint32_t kOffQpe = kOffRaw + kRaw * kRawBytes;
  static constexpr uint32_t kOffX = kOffQpe + 8192;                // the peer's partial score tile
  static constexpr uint32_t kOffXs = kOffX + kXBytes;              // own partial, outgoing
  static constexpr uint32_t kSmemBytes = kOffXs + kXBytes + 1024;
  static constexpr uint32_t kStaticSmem = kMma8 ? 8 * 1024 : 4 * 1024;  // static shared memory, rounded up
  static_assert(kStageBytes % 1024 == 0 && kRawBytes % 128 == 0 && kOffQpe % 512 == 0,
                "swizzled tiles need 1024-byte (128 B swizzle) / 512-byte (64 B, 32 B) alignment");
  static_assert(kStages <= kMaxStages, "stage barriers");
  static_assert(kSmemBytes + kStaticSmem <= 232448, "shared memory per CTA");
};
constexpr uint32_t kTmO = 0, kTmS = 256, kTmP = 320, kTmQ = 384;
// 8-bit mode: P buffer pb holds term t of tokens [32 j, 32 j + 32) (4 codes
// per column) at kTmP + 32 pb + 16 j + 8 t; the query's latent codes, term t,
// at kTmQ + 64 t.
constexpr int kThreads = 512;
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold: P stays <= 2^8
// 8-bit mode: P = 2^(x - m + kPShift8) with the lazy threshold kRescaleLog2_8,
// so P <= 2^8 < 448 (the largest E4M3 value) and E4M3's normal range covers
// the 14 octaves below the running maximum.
constexpr float kRescaleLog2_8 = 2.f, kPShift8 = 6.f;
constexpr int kIdRing = 16;          // page ids read ahead by the producer
constexpr int kPreIssue = 1;         // stage loads issued before the start-up barrier

enum {
  B_FULL = 0,                       // bf16 stage ready (TMA landed, or E4M3 expanded)
  B_EMPTY = B_FULL + kMaxStages,    // bf16 stage consumed by P . V
  B_RFULL = B_EMPTY + kMaxStages,   // raw E4M3 page landed
  B_RFREE = B_RFULL + 2,            // raw E4M3 page expanded
  B_SFULL = B_RFREE + 2,            // S = Q K^T done
  B_SFREE,                          // the exchange warps have read S
  B_XSTG,                           // [4 row quarters] own slab staged (32 arrivals)
  B_XFULL = B_XSTG + 4,             // [4] the peer's slab landed (local arm + its bulk copy)
  B_XREAD = B_XFULL + 4,            // [4] the quarter's two softmax warps have read both slabs
  B_XFREE = B_XREAD + 4,            // [4] the peer's softmax warps have read our slab
  B_MX = B_XFREE + 4,               // [4] row-value swap between the quarter's two softmax warps
  B_PFULL = B_MX + 4,               // [2] P buffer i written (tensor memory)
  B_PVD = B_PFULL + 2,              // the P . V that read P buffer i is done
  B_ODONE = B_PVD + 2,
  B_OFREE,
  B_QFULL,
  B_IDLE,
  B_QTMA,                           // bf16: the first unit's query landed (TMA)
  B_COUNT
};

struct Unit {
  int b, pb, pe, n, slot;
  bool split, at_lo, at_hi;
};

// Walks the units of one worker range [lo, hi) of flattened pages.  The
// lengths of sequences [sl_b0, sl_b0 + 32) come from a copy in shared memory.
struct Walker {
  int b;
  long long sb, lo, hi;
  int w, G;
  const int* sl;
  int sl_b0;
  __device__ bool next(const DecodeArgs& a, Unit& u) {
    while (b < a.B && sb < hi) {
      const int n = (unsigned)(b - sl_b0) < 32u ? sl[b - sl_b0] : a.seq_lens[b];
      const int np = seq_pages(n, a.maxp, nullptr);
      const int bb = b;
      const long long s0 = sb;
      ++b;
      sb += np;
      if (np > 0) {
        const long long ub = max(lo, s0), ue = min(hi, s0 + np);
        u.b = bb;
        u.n = n;
        u.pb = (int)(ub - s0);
        u.pe = (int)(ue - s0);
        u.split = s0 < lo || s0 + np > hi;
        u.at_lo = ub == lo;
        u.at_hi = ue == hi;
        u.slot = u.at_lo ? w : G + w;
        return true;
      }
    }
    return false;
  }
};

// The pages of one worker range, in order: (unit, page of the sequence).
struct PageIter {
  Walker wk;
  Unit u;
  bool have;
  int j;
  __device__ void start(const DecodeArgs& a, const Walker& w0) {
    wk = w0;
    have = wk.next(a, u);
    j = have ? u.pb : 0;
  }
  __device__ void advance(const DecodeArgs& a) {
    if (++j >= u.pe) {
      have = wk.next(a, u);
      j = have ? u.pb : 0;
    }
  }
  // address of the current page's id in the page table
  __device__ const int32_t* id_ptr(const DecodeArgs& a) const {
    return a.page_table + (size_t)u.b * a.maxp + j;
  }
};

// Run by one full warp, reading only the sequence lengths: the batch's total
// page count P and, for worker w's first flattened page lo, the sequence b0
// holding it and that sequence's first flattened page s0 (b0 = B for an empty
// range).  Lane l stores the length of sequence b0 + l in sl[l] (0 past the
// batch).  Invalid lengths count as 0 pages; they are reported later.
__device__ inline void warp_schedule(const DecodeArgs& a, int w, long long* P_out, int* b0_out, long long* s0_out,
                                     int* sl) {
  const int lane = threadIdx.x & 31;
  const int first = lane < a.B ? __ldg(a.seq_lens + lane) : 0;  // the first 32 lengths stay in registers
  long long P = 0;
  for (int base = 0; base < a.B; base += 32) {
    const int n = base == 0 ? first : (base + lane < a.B ? __ldg(a.seq_lens + base + lane) : 0);
    const int np = base + lane < a.B ? seq_pages(n, a.maxp, nullptr) : 0;
    P += __shfl_sync(0xffffffffu, warp_incl_scan(np), 31);
  }
  const long long lo = range_lo(w, a.G, P), hi = range_lo(w + 1, a.G, P);
  int b0 = a.B;
  long long s0 = 0;
  if (lo < hi) {
    long long run = 0;
    for (int base = 0; base < a.B; base += 32) {
      const int b = base + lane;
      const int n = base == 0 ? first : (b < a.B ? __ldg(a.seq_lens + b) : 0);
      const int np = b < a.B ? seq_pages(n, a.maxp, nullptr) : 0;
      const int incl = warp_incl_scan(np);
      const long long st = run + incl - np;
      const unsigned m = __ballot_sync(0xffffffffu, b < a.B && np > 0 && st <= lo && lo < st + np);
      if (m) {
        const int src = __ffs(m) - 1;
        b0 = base + src;
        s0 = __shfl_sync(0xffffffffu, st, src);
        break;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  const int bl = b0 + lane;
  const int from_regs = __shfl_sync(0xffffffffu, first, bl & 31);  // every lane takes part
  sl[lane] = bl < a.B ? (bl < 32 ? from_regs : __ldg(a.seq_lens + bl)) : 0;
  *P_out = P;
  *b0_out = b0;
  *s0_out = s0;
}

__device__ inline uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ inline void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ inline uint4 ld_shared_v4u(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Two E4M3 codes (low 16 bits of v) as a bf16 pair, exactly: E4M3 -> f16
// (hardware conversion) -> f32 -> bf16 loses nothing, every E4M3 value
// having at most 4 significant bits and an exponent inside both ranges.
__device__ inline uint32_t e4m3x2_to_bf16x2(uint32_t v) {
  uint32_t h2;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n" : "=r"(h2) : "r"(v));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  return pack_bf16(f.x, f.y);
}
// Two fp32 values as an E4M3 pair (nearest even, saturating): lo in the low byte.
__device__ inline uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ inline float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// TMA tile load with an L2 cache policy.  bf16 cache pages are read once per
// step, so they are loaded evict-first and leave the L2 to what is read
// again (the partials the combine merges, the query, the weights).  (The
// E4M3 paths measured slower with the hint, 609 against 595 us, and load
// without it.)
__device__ inline uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ inline void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                        uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(pol)
      : "memory");
}

__device__ inline float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte chunk c (0..15, four fp32 scores) of score row h in
// a partial-score tile.  Within each half-row the chunk order is rotated by
// the row, so that 8 consecutive rows touch 8 different bank groups.
__device__ inline uint32_t x_off(int h, int c) {
  return (uint32_t)((h >> 5) * kSlab + (h & 31) * 256 + (((c & 8) | ((c & 7) ^ (h & 7))) * 16));
}

// Row h of this CTA's half of sequence b's query: latent columns
// [128 hlo, 128 hhi) of the half (each 128 values fill 64 tensor-memory
// columns, two bf16 per column) and, with_pe, the 32 RoPE values into shared
// memory (64-byte swizzle, the A operand of the RoPE MMAs).  Rows h >= H are
// zero.  The caller waits for the tensor-memory stores and publishes them.
__device__ inline void load_q_rows(const DecodeArgs& a, uint32_t tq, uint32_t qpe, int b, int h, uint32_t rank,
                                   int hlo, int hhi, bool with_pe) {
  const bool on = h < a.H;
  const uint4* src = reinterpret_cast<const uint4*>(a.q_lat + ((size_t)b * a.H + h) * kLatent + rank * 256);
  const uint4* sp = reinterpret_cast<const uint4*>(a.q_pe + ((size_t)b * a.H + h) * kRope + rank * 32);
  uint4 xp[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) xp[v] = with_pe && on ? sp[v] : make_uint4(0, 0, 0, 0);
  for (int half = hlo; half < hhi; ++half) {
    uint4 xq[16];
#pragma unroll
    for (int v = 0; v < 16; ++v) xq[v] = on ? src[half * 16 + v] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t r[32];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        r[4 * v] = xq[cc * 8 + v].x;
        r[4 * v + 1] = xq[cc * 8 + v].y;
        r[4 * v + 2] = xq[cc * 8 + v].z;
        r[4 * v + 3] = xq[cc * 8 + v].w;
      }
      tc::tmem_st32(tq + half * 64 + cc * 32, r);
    }
  }
  if (with_pe) {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
      st_shared_v4(qpe + h * 64 + ((cc ^ ((h >> 1) & 3)) * 16), xp[cc].x, xp[cc].y, xp[cc].z, xp[cc].w);
  }
}

// Row h of this CTA's half of sequence b's E4M3 query, every term t <
// a.q_terms: its 256 latent codes into 64 tensor-memory columns at tq + 64 t
// (four codes per column) and its 32 RoPE codes into shared memory at
// qpe + 4096 t (32-byte swizzle: 16-byte chunk c of row h at
// h * 32 + ((c ^ ((h >> 2) & 1)) * 16), the A operand of the RoPE MMAs).
// Rows h >= H are zero.  Returns the row's scale.  The caller waits for the
// tensor-memory stores and publishes them.
__device__ inline float load_q8_rows(const DecodeArgs& a, uint32_t tq, uint32_t qpe, int b, int h, uint32_t rank) {
  const bool on = h < a.H;
  const uint8_t* row = a.q8 + ((size_t)b * a.H + (on ? h : 0)) * (2 * kRow);
  for (int t = 0; t < a.q_terms; ++t) {
    const uint4* src = reinterpret_cast<const uint4*>(row + t * kRow + rank * 256);
    const uint4* sp = reinterpret_cast<const uint4*>(row + t * kRow + kLatent + rank * 32);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 xp = on ? sp[c] : make_uint4(0, 0, 0, 0);
      st_shared_v4(qpe + t * 4096 + h * 32 + ((c ^ ((h >> 2) & 1)) << 4), xp.x, xp.y, xp.z, xp.w);
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t r[32];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint4 x = on ? src[cc * 8 + v] : make_uint4(0, 0, 0, 0);
        r[4 * v] = x.x;
        r[4 * v + 1] = x.y;
        r[4 * v + 2] = x.z;
        r[4 * v + 3] = x.w;
      }
      tc::tmem_st32(tq + t * 64 + cc * 32, r);
    }
  }
  return on ? a.q8_scale[(size_t)b * a.H + h] : 0.f;
}

template <int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_kpe,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qpe,
                     DecodeArgs a) {
  using L = Layout<kMode>;
  constexpr bool kFp8 = kMode == 1;  // E4M3 cache expanded to bf16 in shared memory
  constexpr bool kF8 = kMode == 2;   // E4M3 cache on the 8-bit tensor cores
  constexpr int kStages = L::kStages;
  constexpr uint32_t kStageBytes = L::kStageBytes, kStageScale = L::kStageScale;
  constexpr uint32_t kOffQpe = L::kOffQpe, kOffX = L::kOffX, kOffXs = L::kOffXs;
  // bf16 and 8-bit: pages go straight into the stage ring.  Expanded E4M3:
  // pages go into the raw ring (codes and scales) and the exchange warps
  // expand them.
  constexpr int kRing = kFp8 ? L::kRaw : kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[B_COUNT];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ long long sh_P, sh_s0;
  __shared__ int sh_b0;
  __shared__ float mx_swap[2][2][128];     // row maxima between the two softmax warpgroups
  __shared__ uint32_t lsum_swap[2 * 128];  // row sums between them at the end of a unit
  __shared__ int page_ids[kIdRing];        // producer-private
  __shared__ int sl_cache[32];             // lengths of the range's first sequences
  // 8-bit mode: log2 of a page's token scales and their reciprocals, for the
  // softmax (by page parity and row quarter; 0 past the sequence end)
  __shared__ __align__(16) float tok_lg[kF8 ? 2 * 4 * 64 : 1];
  __shared__ __align__(16) float tok_inv[kF8 ? 2 * 4 * 64 : 1];

  const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
  const int w = blockIdx.x >> 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const smem_base = smem_raw + (base - smem_u32(smem_raw));  // the same aligned address, as a pointer
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(B_FULL + i), kFp8 ? 128 : 1);  // E4M3: the 128 expanding threads
      mbar_init(bar(B_EMPTY + i), 1);
    }
    for (int i = 0; i < L::kRaw; ++i) {
      mbar_init(bar(B_RFULL + i), 1);
      mbar_init(bar(B_RFREE + i), 128);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SFREE), 128);  // the exchange warps have read S
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(B_XSTG + i), 32);   // the 32 lanes of one exchange warp
      mbar_init(bar(B_XFULL + i), 1);   // local arm + one slab of the peer's bulk copy
      mbar_init(bar(B_XREAD + i), 64);  // the quarter's two softmax warps
      mbar_init(bar(B_XFREE + i), 1);   // the peer's exchange warp of this quarter
      mbar_init(bar(B_MX + i), 64);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_PFULL + i), 256);
      mbar_init(bar(B_PVD + i), 1);
    }
    mbar_init(bar(B_ODONE), 1);
    mbar_init(bar(B_OFREE), 256);
    mbar_init(bar(B_QFULL), 256);  // the softmax threads (first unit) or the exchange threads twice
    mbar_init(bar(B_IDLE), 2);
    mbar_init(bar(B_QTMA), 1);
    for (int i = 0; i < 4; ++i) mbar_expect_tx(bar(B_XFULL + i), kSlab);
    fence_mbar_init();
    prefetch_tmap(&tm_ckv);
    prefetch_tmap(&tm_kpe);
    if (kMode == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_qpe);
    }
  }

  // ---------------------------------------------------------------- producer state
  // Warp 0 works out the schedule and issues the first loads of the stage
  // ring before the start-up barrier: they read only the lengths, the page
  // table and the cache, none of which the preceding kernel on the stream
  // (the query absorption) writes, so they may overlap it.
  PageIter pit{};
  uint32_t g_prod = 0, id_count = 0;
  int id_pend = -1;
  bool id_pend_ok = false;
  PageIter ic{};  // id read-ahead cursor (kIdRing pages ahead of pit)
  auto page_at = [&](uint32_t k) {
    const int pg = page_ids[k % kIdRing];
    return pg >= 0 && pg < a.num_pages ? pg : -1;
  };
  auto id_fetch = [&]() {  // stores the id loaded one page ago, loads the next one
    if (id_pend_ok) page_ids[(id_count - 1) % kIdRing] = id_pend;
    id_pend_ok = true;
    id_pend = ic.have ? __ldg(ic.id_ptr(a)) : -1;
    if (ic.have) ic.advance(a);
    ++id_count;
  };
  auto issue = [&](uint32_t g) {
    const uint32_t s = g % kRing;
    int page = page_at(g);
    if (page < 0) page = 0;  // a bad page id: masked by the softmax warps
    if (kFp8 || kF8) {
      // E4M3: this CTA's 256 latent codes (two 128-byte boxes), 32 RoPE codes
      // and the page's 64 scales; straight into a stage (8-bit) or the raw ring
      const uint32_t fb = bar(kF8 ? B_FULL + s : B_RFULL + s);
      const uint32_t dst = kF8 ? base + s * kStageBytes : base + L::kOffRaw + s * kRawBytes;
      mbar_expect_tx(fb, 2 * 8192 + 2048 + kPage * 4);
      tma_load_2d(dst, &tm_ckv, fb, (int)rank * 256, page * kPage);
      tma_load_2d(dst + 8192, &tm_ckv, fb, (int)rank * 256 + 128, page * kPage);
      tma_load_2d(dst + kRawKpe, &tm_kpe, fb, (int)rank * 32, page * kPage);
      bulk_copy_g2s(dst + kRawScale, a.kv_scale + (size_t)page * kPage, kPage * 4, fb);
    } else {
      const uint32_t fb = bar(B_FULL + s);
      const uint32_t st = base + s * kStageBytes;
      const uint64_t l2_once = l2_evict_first_policy();
      mbar_expect_tx(fb, 4 * kBox + kKpeBox);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        tma_load_2d_hint(st + i * kBox, &tm_ckv, fb, (int)rank * 256 + i * 64, page * kPage, l2_once);
      tma_load_2d_hint(st + 4 * kBox, &tm_kpe, fb, (int)rank * 32, page * kPage, l2_once);
    }
  };
  if (warp == 0) {
    long long P;
    int b0;
    long long s0;
    warp_schedule(a, w, &P, &b0, &s0, sl_cache);
    __syncwarp();
    if (lane == 0) {
      sh_P = P;
      sh_b0 = b0;
      sh_s0 = s0;
      const Walker w0{b0, s0, range_lo(w, a.G, P), range_lo(w + 1, a.G, P), w, a.G, sl_cache, b0};
      pit.start(a, w0);
      ic.start(a, w0);
      // the range's first kIdRing page ids, loaded together
      const int32_t* ptr[kIdRing];
#pragma unroll
      for (int i = 0; i < kIdRing; ++i) {
        ptr[i] = ic.have ? ic.id_ptr(a) : nullptr;
        if (ic.have) ic.advance(a);
      }
      int v[kIdRing];
#pragma unroll
      for (int i = 0; i < kIdRing; ++i) v[i] = ptr[i] ? __ldg(ptr[i]) : -1;
#pragma unroll
      for (int i = 0; i < kIdRing; ++i) page_ids[i] = v[i];
      id_count = kIdRing;
      // the first page needs no free slot and its id is loaded; the read-ahead
      // of further ids starts after the start-up barrier
      for (; pit.have && g_prod < (uint32_t)min(kPreIssue, kRing); ++g_prod) {
        issue(g_prod);
        pit.advance(a);
      }
    }
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // barrier inits visible to the peer before any remote arrive (a release
  // arrive would also wait for the stage loads already in flight)
  cluster_sync_relaxed();
  tc_fence_after();
  // launched as a dependent of the previous kernel on the stream: the query
  // and everything written below come after that kernel has finished
  grid_dep_wait();
  grid_dep_trigger();
  const uint32_t tmem = tmem_slot;
  const long long P = sh_P;
  const Walker walker0{sh_b0, sh_s0, range_lo(w, a.G, P), range_lo(w + 1, a.G, P), w, a.G, sl_cache, sh_b0};
  const long long range_n = range_lo(w + 1, a.G, P) - range_lo(w, a.G, P);
  const uint32_t npages = range_n > 0 ? (uint32_t)range_n : 0u;

  // every lane waits, then the warp agrees, so warp-collective operations never
  // run with some lanes gone after an aborted wait
  auto wwait = [&](int i, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, &abort_flag, a.err));
  };
  auto wwait_c = [&](int i, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait<true>(bar(i), parity, &abort_flag, a.err));
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const int free_bar = kFp8 ? B_RFREE : B_EMPTY, full_bar = kFp8 ? B_RFULL : B_FULL;
      bool ok = true;
      // the rest of the ring waits for the first unit's query: its loads
      // would otherwise queue behind every CTA's stage loads
      if (pit.have && !mbar_wait(bar(B_QFULL), 0, &abort_flag, a.err)) ok = false;
      for (; ok && pit.have; ++g_prod) {
        const uint32_t s = g_prod % kRing;
        if (g_prod >= (uint32_t)kRing &&
            !mbar_wait(bar(free_bar + s), ((g_prod / kRing) - 1) & 1, &abort_flag, a.err)) {
          ok = false;
          break;
        }
        issue(g_prod);
        id_fetch();  // keeps the page ids ahead of the ring (kIdRing - kRing pages at least)
        pit.advance(a);
      }
      // copies still in flight must land before the CTA can exit
      for (uint32_t k = g_prod > (uint32_t)kRing ? g_prod - kRing : 0; k < g_prod; ++k) {
        volatile int no_abort = 0;
        mbar_wait(bar(full_bar + k % kRing), (k / kRing) & 1, &no_abort, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S = Q K^T issuer
    if (lane == 0) {
      Walker wk = walker0;
      Unit u;
      uint32_t g = 0, uc = 0;
      bool ok = true;
      const uint32_t idesc_qk = idesc_bf16(128, 64, false, false);
      const uint32_t idesc_qk8 = idesc_e4m3(128, 64, false, false);
      while (ok && wk.next(a, u)) {
        const int np = u.pe - u.pb;
        if (!mbar_wait(bar(B_QFULL), uc & 1, &abort_flag, a.err)) break;
        tc_fence_after();
        for (int i = 0; i < np; ++i) {
          const uint32_t gi = g + i, s = gi % kStages;
          // S has one buffer: the exchange warps copy it out as soon as it is done
          if (!mbar_wait(bar(B_FULL + s), (gi / kStages) & 1, &abort_flag, a.err) ||
              (gi >= 1 && !mbar_wait(bar(B_SFREE), (gi - 1) & 1, &abort_flag, a.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = base + s * kStageBytes, d = tmem + kTmS;
          // one descriptor per operand and page; K-step kk is a constant offset
          // (16-byte units) into it, so the MMAs issue back to back
          const uint64_t kdesc = sdesc_sw128(st, 16, 1024);
          if constexpr (kF8) {
            // 32 codes per K step: 8 steps over the two latent boxes per query
            // term, then one step per term for the 32 RoPE codes
            for (int t = 0; t < a.q_terms; ++t) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_e4m3_ts(d, tmem + kTmQ + t * 64 + kk * 8,
                            kdesc + (uint64_t)(((kk >> 2) * kBox + (kk & 3) * 32) >> 4), idesc_qk8,
                            (t > 0 || kk > 0) ? 1u : 0u);
            }
            const uint64_t rdesc = sdesc_sw32(st + kStage8Kpe, 16, 256);
            for (int t = 0; t < a.q_terms; ++t)
              mma_e4m3_ss(d, sdesc_sw32(base + kOffQpe + t * 4096, 16, 256), rdesc, idesc_qk8, 1u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma_bf16_ts(d, tmem + kTmQ + kk * 8, kdesc + (uint64_t)(((kk >> 2) * kBox + (kk & 3) * 32) >> 4),
                          idesc_qk, kk > 0 ? 1u : 0u);
            // this CTA's 32 dimensions of the RoPE key: A = q_pe half (shared memory)
            const uint64_t qdesc = sdesc_sw64(base + kOffQpe, 16, 512);
            const uint64_t rdesc = sdesc_sw64(st + 4 * kBox, 16, 512);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) mma_bf16_ss(d, qdesc + kk * 2, rdesc + kk * 2, idesc_qk, 1u);
          }
          // completes once every MMA issued so far is done, including all of this
          // unit's reads of the query when i is its last page
          mma_commit(bar(B_SFULL));
        }
        g += np;
        ++uc;
      }
      mma_commit(bar(B_IDLE));  // every issued MMA has finished once this fires
      volatile int no_abort = 0;
      mbar_wait(bar(B_IDLE), 0, &no_abort, nullptr);
    }
  } else if (warp == 2) {
    // tensor-memory allocation only (done at start-up)
  } else if (warp == 3) {
    // the batch's page offsets and the length check (written once, by the
    // first CTA), then the split records of this worker
    if (w == 0 && rank == 0) warp_total_pages(a.seq_lens, a.B, a.maxp, a.err, a.seq_start);
    if (lane == 0) {
      // ---------------------------------------------------------- split records
      if (rank == 0) {
        Walker wk = walker0;
        Unit u;
        int4 first = make_int4(-1, 0, 0, 0), last = make_int4(-1, 0, 0, 0);
        while (wk.next(a, u)) {
          const int4 r = make_int4(u.b, u.pb, u.pe, u.split ? 1 : 0);
          if (u.at_lo) first = r;
          else if (u.at_hi) last = r;
        }
        a.rec[w] = first;
        a.rec[a.G + w] = last;
      }
      // ---------------------------------------------------------- O += P V issuer
      Walker wk = walker0;
      Unit u;
      uint32_t g = 0, uc = 0;
      bool ok = true;
      const uint32_t idesc_pv = idesc_bf16(128, 256, false, true);
      const uint32_t idesc_pv8 = idesc_e4m3(128, 256, false, true);
      while (ok && wk.next(a, u)) {
        const int np = u.pe - u.pb;
        for (int i = 0; i < np; ++i) {
          const uint32_t gp = g + i, s = gp % kStages, pb = gp & 1;
          if (!mbar_wait(bar(B_PFULL + pb), (gp >> 1) & 1, &abort_flag, a.err) ||
              (i == 0 && uc >= 1 && !mbar_wait(bar(B_OFREE), (uc - 1) & 1, &abort_flag, a.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // A = P from tensor memory, B = the stage's latent (MN-major)
          const uint64_t cdesc = sdesc_sw128(base + s * kStageBytes, kBox, 1024);
          if constexpr (kF8) {
            // four codes per column, 32 tokens (4096 bytes of codes) per K
            // step; tokens [32 kk, 32 kk + 32) of term t at 16 kk + 8 t
            for (int t = 0; t < a.p_terms; ++t) {
#pragma unroll
              for (int kk = 0; kk < 2; ++kk)
                mma_e4m3_ts(tmem + kTmO, tmem + kTmP + pb * 32 + kk * 16 + t * 8, cdesc + kk * 256, idesc_pv8,
                            (i > 0 || t > 0 || kk > 0) ? 1u : 0u);
            }
          } else {
            // two bf16 per column, 16 tokens per K step
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ts(tmem + kTmO, tmem + kTmP + pb * 32 + kk * 8, cdesc + kk * 128, idesc_pv,
                          (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(B_PVD + pb));
          mma_commit(bar(B_EMPTY + s));
          if (i == np - 1) mma_commit(bar(B_ODONE));
        }
        g += np;
        ++uc;
      }
      mma_commit(bar(B_IDLE));
      volatile int no_abort = 0;
      mbar_wait(bar(B_IDLE), 0, &no_abort, nullptr);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ exchange warps
    // Copy each page's partial score (log2 domain, fp32) out of tensor
    // memory as soon as its S = Q K^T completes, stage it in shared memory,
    // and hand each warp's slab of 32 rows to the async copy engine, which
    // writes it into the peer CTA and completes the peer's receive barrier
    // for that slab.  (Per-thread remote loads or stores would queue behind
    // the SM-to-SM network.)
    const int q4 = warp & 3;
    const int h = threadIdx.x - 128;
    const int H = a.H;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t xfull_peer = mapa(bar(B_XFULL), peer);
    const uint32_t xfree_peer = mapa(bar(B_XFREE), peer);
    const uint32_t x_peer = mapa(base + kOffX, peer);
    const float c = a.scale_log2;

    // this CTA's half of a later unit's query: 256 latent values -> tensor
    // memory, 32 RoPE values -> shared memory
    float qs_cur = 0.f, qs_nxt = 0.f;  // 8-bit mode: query row scale of this / the next unit
    auto load_q = [&](const Unit& q) {
      if constexpr (kF8)
        qs_nxt = load_q8_rows(a, tmem + lane_base + kTmQ, base + kOffQpe, q.b, h, rank);
      else
        load_q_rows(a, tmem + lane_base + kTmQ, base + kOffQpe, q.b, h, rank, 0, 2, true);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_cnt(bar(B_QFULL), 2);
    };
    // a later unit's query rows into L2 while this unit runs
    auto prefetch_q = [&](int b) {
      if (h != 0) return;
      const uint32_t qb = (uint32_t)H * kLatent * 2;
      const char* ql = reinterpret_cast<const char*>(a.q_lat + (size_t)b * H * kLatent);
      for (uint32_t off = 0; off < qb; off += 16384) prefetch_l2(ql + off, min(16384u, qb - off));
      prefetch_l2(a.q_pe + (size_t)b * H * kRope, (uint32_t)H * kRope * 2);
    };

    // E4M3 only: expand raw page gc into bf16 stage gc % kStages (exact
    // conversion, same 128-byte-swizzled layout TMA gives the bf16 cache) and
    // copy its scales.  Thread h converts 16 codes per step.
    constexpr uint32_t kRawN = L::kRaw > 0 ? L::kRaw : 1;
    auto expand = [&](uint32_t gc) -> bool {
      const uint32_t r = gc % kRawN, s = gc % kStages;
      if (!wwait(B_RFULL + r, (gc / kRawN) & 1)) return false;
      if (gc >= (uint32_t)kStages && !wwait(B_EMPTY + s, ((gc / kStages) - 1) & 1)) return false;
      const uint32_t raw = base + L::kOffRaw + r * kRawBytes, st = base + s * kStageBytes;
#pragma unroll 2
      for (int i = 0; i < 8; ++i) {  // latent: 2 boxes x 64 rows x 8 chunks of 16 codes
        const int q = h + 128 * i, box = q >> 9, row = (q >> 3) & 63, cc = q & 7;
        const uint4 v = ld_shared_v4u(raw + box * 8192 + row * 128 + cc * 16);
        const int col = box * 128 + cc * 16, kb = col >> 6, cb = (col & 63) >> 3;
        const uint32_t rowa = st + kb * kBox + row * 128;
        // Each 8-lane quarter of the warp expands one row: 4 lanes into box kb
        // = 2 box, 4 into box 2 box + 1, chunks (cb, cb + 1) each.  The lanes
        // of the odd box store their second chunk first, so that each store
        // instruction's quarter touches all 8 bank groups of the row (the
        // swizzle is the same in both boxes).
        const uint32_t lo_first = kb & 1;
        const uint32_t c0 = rowa + (((cb + lo_first) ^ (row & 7)) << 4), c1 = rowa + (((cb + 1 - lo_first) ^ (row & 7)) << 4);
        const uint32_t e0 = e4m3x2_to_bf16x2(v.x), e1 = e4m3x2_to_bf16x2(v.x >> 16), e2 = e4m3x2_to_bf16x2(v.y),
                       e3 = e4m3x2_to_bf16x2(v.y >> 16), e4 = e4m3x2_to_bf16x2(v.z), e5 = e4m3x2_to_bf16x2(v.z >> 16),
                       e6 = e4m3x2_to_bf16x2(v.w), e7 = e4m3x2_to_bf16x2(v.w >> 16);
        if (lo_first) {
          st_shared_v4(c0, e4, e5, e6, e7);
          st_shared_v4(c1, e0, e1, e2, e3);
        } else {
          st_shared_v4(c0, e0, e1, e2, e3);
          st_shared_v4(c1, e4, e5, e6, e7);
        }
      }
      {  // this CTA's 32 rope codes per token: 64 rows x 2 chunks of 16, into the
         // 64-byte-swizzled k_pe box (16-byte chunk c of row r at c ^ ((r >> 1) & 3))
        const int row = h >> 1, cc = h & 1, sw = (row >> 1) & 3;
        const uint4 v = ld_shared_v4u(raw + kRawKpe + row * 32 + cc * 16);
        const uint32_t rowa = st + 4 * kBox + row * 64;
        st_shared_v4(rowa + (((2 * cc) ^ sw) << 4), e4m3x2_to_bf16x2(v.x), e4m3x2_to_bf16x2(v.x >> 16),
                     e4m3x2_to_bf16x2(v.y), e4m3x2_to_bf16x2(v.y >> 16));
        st_shared_v4(rowa + (((2 * cc + 1) ^ sw) << 4), e4m3x2_to_bf16x2(v.z), e4m3x2_to_bf16x2(v.z >> 16),
                     e4m3x2_to_bf16x2(v.w), e4m3x2_to_bf16x2(v.w >> 16));
      }
      if (h < kPage / 4) {
        const uint4 v = ld_shared_v4u(raw + kRawScale + h * 16);
        st_shared_v4(st + kStageScale + h * 16, v.x, v.y, v.z, v.w);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(B_FULL + s));
      mbar_arrive(bar(B_RFREE + r));
      return true;
    };

    Walker wk = walker0;
    Unit u;
    uint32_t g = 0;
    bool ok = true;
    bool have = wk.next(a, u);
    if (have) {  // the first unit's query is loaded by the softmax warps (8-bit mode: here)
      if constexpr (kF8) {
        load_q(u);
        qs_cur = qs_nxt;
      }
      Walker pk = wk;
      Unit nu;
      if (pk.next(a, nu)) prefetch_q(nu.b);
    }
    if (kFp8 && npages > 0) ok = expand(0);
    while (ok && have) {
      Walker pk = wk;  // the next unit, if any
      Unit nu;
      const bool have_next = pk.next(a, nu);
      if (g > 0 && have_next) prefetch_q(nu.b);
      for (int jp = u.pb; jp < u.pe; ++jp, ++g) {
        if (!wwait(B_SFULL, g & 1)) { ok = false; break; }
        tc_fence_after();
        const float* tsc = reinterpret_cast<const float*>(smem_base + (g % kStages) * kStageBytes + kStageScale);
        // 8-bit mode: the score of the codes times the query row's scale; the
        // softmax multiplies the sum of both partials by the token scale
        const float cq = kF8 ? c * qs_cur : c;
        float v[64];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t s32[32];
          tmem_ld32(tmem + lane_base + kTmS + half * 32, s32);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) v[half * 32 + k] = __uint_as_float(s32[k]) * cq;
        }
        tc_fence_before();
        mbar_arrive(bar(B_SFREE));
        float inv_a = 0.f, inv_b = 0.f, lg_a = 0.f, lg_b = 0.f;
        if constexpr (kF8) {
          // for the softmax: log2(scale_t), which carries the token scale into
          // the probabilities (P . V multiplies codes), and 1 / scale_t for
          // the row sums (0 past the sequence end)
          const int nv = min(kPage, u.n - jp * kPage);
          inv_a = lane < nv ? __frcp_rn(tsc[lane]) : 0.f;
          inv_b = lane + 32 < nv ? __frcp_rn(tsc[lane + 32]) : 0.f;
          lg_a = lane < nv ? __log2f(tsc[lane]) : 0.f;
          lg_b = lane + 32 < nv ? __log2f(tsc[lane + 32]) : 0.f;
        }
        if constexpr (kFp8) {
          // E4M3: the score of token t is scale_t times the score of its codes
          // (scales copied next to the expanded stage)
#pragma unroll
          for (int k = 0; k < 64; ++k) v[k] *= tsc[k];
        }
        if (g >= 1) {
          // our receive slab of this quarter is free once our softmax warps have
          // read page g-1 from it: arm it for page g and tell the peer
          if (!wwait(B_XREAD + q4, (g - 1) & 1)) { ok = false; break; }
          if (lane == 0) {
            mbar_expect_tx(bar(B_XFULL + q4), kSlab);
            mbar_arrive_remote(xfree_peer + q4 * 8);
          }
          // our outgoing slab (and the peer's receive slab) is free once the
          // peer's softmax warps have read page g-1
          if (!wwait_c(B_XFREE + q4, (g - 1) & 1)) { ok = false; break; }
        }
        if constexpr (kF8) {
          // 1 / scale_t for this quarter's softmax warps (0 past the sequence
          // end); they finished page g-2, which used this slot, before
          // reading page g-1 (waited for above)
          float* inv = tok_inv + ((g & 1) * 4 + q4) * 64;
          inv[lane] = inv_a;
          inv[lane + 32] = inv_b;
          float* lg = tok_lg + ((g & 1) * 4 + q4) * 64;
          lg[lane] = lg_a;
          lg[lane + 32] = lg_b;
        }
        uint8_t* xt = smem_base + kOffXs;
#pragma unroll
        for (int cc = 0; cc < 16; ++cc)
          *reinterpret_cast<float4*>(xt + x_off(h, cc)) = make_float4(v[4 * cc], v[4 * cc + 1], v[4 * cc + 2], v[4 * cc + 3]);
        fence_proxy_async_smem();
        mbar_arrive(bar(B_XSTG + q4));  // for our own softmax warps
        __syncwarp();
        // each warp sends its own slab as soon as it is staged
        if (lane == 0) {
          const uint32_t off = (uint32_t)q4 * kSlab;
          bulk_copy_to_peer(x_peer + off, base + kOffXs + off, kSlab, xfull_peer + q4 * 8);
        }
        // the next unit's query goes in once this unit's last S = Q K^T is done
        if (jp == u.pe - 1 && have_next) load_q(nu);
        if (jp == u.pe - 1) qs_cur = qs_nxt;
        // the next page's expansion waits for the P . V that frees its stage,
        // so it comes after this page's exchange
        if (kFp8 && g + 1 < npages && !expand(g + 1)) { ok = false; break; }
      }
      if (!ok) break;
      u = nu;
      have = have_next;
      wk = pk;
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    // Warpgroup j (warps 8+4j .. 11+4j) owns score columns [32j, 32j+32) of
    // every page (its 32 tokens) for all 128 head rows; thread = head row =
    // tensor-memory lane.  It adds its own CTA's partial score to the peer's
    // and agrees on the row maximum with the other warpgroup.
    const int j = (warp - 8) >> 2;
    const int q4 = warp & 3;
    const int h = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int H = a.H;
    uint32_t xk = 0;  // phases of the warpgroup-exchange barrier consumed
    constexpr float kShift = kF8 ? kPShift8 : 0.f;  // P = 2^(x - m + kShift)

    // Swap one value per row with the other warpgroup's warp of the same row
    // quarter (bounded wait).  Row maxima alternate between two slots, so that
    // a fast warp cannot overwrite a value the other has not read yet.
    auto swap_max = [&](float mine, float& other) -> bool {
      const uint32_t slot = xk & 1;
      mx_swap[slot][j][h] = mine;
      mbar_arrive(bar(B_MX + q4));
      const bool okw = wwait(B_MX + q4, xk & 1);
      ++xk;
      other = mx_swap[slot][j ^ 1][h];
      return okw;
    };
    auto swap_sum = [&](uint32_t mine, uint32_t& other) -> bool {
      lsum_swap[j * 128 + h] = mine;
      mbar_arrive(bar(B_MX + q4));
      const bool okw = wwait(B_MX + q4, xk & 1);
      ++xk;
      other = lsum_swap[(j ^ 1) * 128 + h];
      return okw;
    };

    Walker wk = walker0;
    Unit u;
    uint32_t g = 0, uc = 0;
    bool ok = true;
    bool have = wk.next(a, u);
    if (have && kMode == 0) {
      // the first unit's query: this CTA's latent half by TMA into stages 1-2
      // (free until the rest of the ring goes out, after B_QFULL; four
      // [128 rows x 64] boxes, 128-byte swizzle) and its RoPE half straight
      // into the operand's place (64-byte swizzle); warpgroup j then moves
      // latent half j into tensor memory.  Rows h >= H hold other rows of
      // q_lat or TMA zeros and are zeroed here.
      const uint32_t qs = base + kStageBytes;
      if (h == 0 && j == 0) {
        mbar_expect_tx(bar(B_QTMA), 4 * 16384 + 8192);
        for (int k = 0; k < 4; ++k)
          tma_load_2d(qs + k * 16384, &tm_q, bar(B_QTMA), (int)rank * 256 + k * 64, u.b * H);
        tma_load_2d(base + kOffQpe, &tm_qpe, bar(B_QTMA), (int)rank * 32, u.b * H);
      }
      ok = wwait(B_QTMA, 0);
      if (!ok && h == 0 && j == 0) {  // the copies land before the CTA can exit
        volatile int no_abort = 0;
        mbar_wait(bar(B_QTMA), 0, &no_abort, nullptr);
      }
      const bool on = h < H;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const uint32_t row = qs + (uint32_t)(2 * j + cc) * 16384u + (uint32_t)h * 128u;
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = on ? ld_shared_v4u(row + ((uint32_t)(c ^ (h & 7)) << 4)) : make_uint4(0, 0, 0, 0);
          r[4 * c] = v.x;
          r[4 * c + 1] = v.y;
          r[4 * c + 2] = v.z;
          r[4 * c + 3] = v.w;
        }
        tmem_st32(tmem + lane_base + kTmQ + j * 64 + cc * 32, r);
      }
      if (j == 0 && !on) {
#pragma unroll
        for (int c = 0; c < 4; ++c) st_shared_v4(base + kOffQpe + h * 64 + c * 16, 0, 0, 0, 0);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_QFULL));
    } else if (have && kFp8) {  // the first unit's query: warpgroup j loads half j of the latent part
      load_q_rows(a, tmem + lane_base + kTmQ, base + kOffQpe, u.b, h, rank, j, j + 1, j == 0);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_QFULL));
    }
    while (ok && have) {
      const int np = u.pe - u.pb;
      float m = -INFINITY, l = 0.f;
      const int32_t* ptab = a.page_table + (size_t)u.b * a.maxp;
      int page_nx = ptab[u.pb];
      for (int i = 0; i < np; ++i) {
        const uint32_t gi = g + i, s = gi % kStages;
        const int jp = u.pb + i;
        // page ids are read one page ahead: a global load's latency stays off
        // the softmax's critical path
        const int page = page_nx;
        if (i + 1 < np) page_nx = ptab[jp + 1];
        const bool page_ok = page >= 0 && page < a.num_pages;
        const int valid = page_ok ? min(kPage, u.n - jp * kPage) : 0;
        if (!page_ok && h == 0 && j == 0 && rank == 0) set_error(a.err, MLA_ERR_PAGE_OOB);

        // score in the log2 domain: own fp32 partial (staged by the exchange
        // warps) plus the peer's; both CTAs add the same two numbers
        if (!wwait(B_XSTG + q4, gi & 1) || !wwait_c(B_XFULL + q4, gi & 1)) {
          ok = false;
          break;
        }
        float x[32];
        {
          const uint8_t* xb = smem_base + kOffX;
          const uint8_t* ob = smem_base + kOffXs;
          float4 pv[8], ov[8];
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            pv[cc] = *reinterpret_cast<const float4*>(xb + x_off(h, 8 * j + cc));
            ov[cc] = *reinterpret_cast<const float4*>(ob + x_off(h, 8 * j + cc));
          }
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            x[4 * cc] = ov[cc].x + pv[cc].x;
            x[4 * cc + 1] = ov[cc].y + pv[cc].y;
            x[4 * cc + 2] = ov[cc].z + pv[cc].z;
            x[4 * cc + 3] = ov[cc].w + pv[cc].w;
          }
        }
        mbar_arrive(bar(B_XREAD + q4));  // the exchange warp of this quarter tells the peer
        const uint32_t sca = base + s * kStageBytes + kStageScale + j * 128;  // E4M3 token scales
        if constexpr (kF8) {
          // the token scale: on the score, and as log2(scale_t) into P
          const float4* ts4 = reinterpret_cast<const float4*>(smem_base + s * kStageBytes + kStageScale) + 8 * j;
          const float4* lg4 = reinterpret_cast<const float4*>(tok_lg + ((gi & 1) * 4 + q4) * 64 + 32 * j);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 f = ts4[c4], o = lg4[c4];
            x[4 * c4] = fmaf(x[4 * c4], f.x, o.x);
            x[4 * c4 + 1] = fmaf(x[4 * c4 + 1], f.y, o.y);
            x[4 * c4 + 2] = fmaf(x[4 * c4 + 2], f.z, o.z);
            x[4 * c4 + 3] = fmaf(x[4 * c4 + 3], f.w, o.w);
          }
        }
        if constexpr (kFp8) {
          if (!wwait(B_FULL + s, (gi / kStages) & 1)) { ok = false; break; }  // scales visible
        }
        if (valid < kPage) {  // tokens past the sequence end (or a bad page)
#pragma unroll
          for (int k = 0; k < 32; ++k) x[k] = 32 * j + k < valid ? x[k] : -INFINITY;
        }
        float t8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) t8[k] = fmaxf(fmaxf(x[k], x[k + 8]), fmaxf(x[k + 16], x[k + 24]));
#pragma unroll
        for (int k = 0; k < 4; ++k) t8[k] = fmaxf(t8[k], t8[k + 4]);
        const float mine = fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3]));
        float other;
        if (!swap_max(mine, other)) { ok = false; break; }
        const float mx = fmaxf(mine, other);

        // online softmax with lazy rescaling: both warpgroups hold the same m
        // and take the same decisions
        float alpha = 1.f;
        bool resc = false;
        if (mx > m + (kF8 ? kRescaleLog2_8 : kRescaleLog2)) {
          alpha = ex2(m - mx);
          resc = i > 0;
          m = mx;
        }
        const float mm = (m == -INFINITY ? 0.f : m) - kShift;
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[16];
        if constexpr (kF8) {
          // x carries log2(scale_t) (added above), so P = 2^(x - mm) is
          // the probability times the token scale, as P . V on the codes needs
          // it; the row sum takes P / scale_t.  P becomes E4M3 terms: hi is P
          // rounded to 4 significant bits (half up; exact in E4M3's normal
          // range, P >= 0), lo = P - hi exactly (|lo| <= 2^-4 P), rounded to
          // E4M3; each pair of codes is one conversion (the lo codes go
          // unused with one term).
          const float* inv = tok_inv + ((gi & 1) * 4 + q4) * 64 + 32 * j;
#pragma unroll
          for (int kq = 0; kq < 8; ++kq) {
            float hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int k = 4 * kq + e;
              const float pe = ex2(x[k] - mm);
              hi[e] = __uint_as_float((__float_as_uint(pe) + 0x80000u) & 0xFFF00000u);
              lo[e] = __fsub_rn(pe, hi[e]);
              ps[e] = fmaf(pe, inv[k], ps[e]);  // inv is 0 past the sequence end
            }
            pk[kq] = f32x2_to_e4m3x2(hi[0], hi[1]) | (f32x2_to_e4m3x2(hi[2], hi[3]) << 16);
            pk[8 + kq] = f32x2_to_e4m3x2(lo[0], lo[1]) | (f32x2_to_e4m3x2(lo[2], lo[3]) << 16);
          }
          // a bad page: every P is 0, but the scales read in its place may be
          // anything (0 * inf)
          if (!page_ok) ps[0] = ps[1] = ps[2] = ps[3] = 0.f;
        } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float p0 = ex2(x[2 * k] - mm), p1 = ex2(x[2 * k + 1] - mm);
          ps[k & 3] += p0 + p1;
          if constexpr (kFp8) {
            // P . V multiplies codes: fold each token's scale into its
            // probability (0 past the end, where the scale may be garbage)
            float s0 = 0.f, s1 = 0.f;
            if (32 * j + 2 * k < valid) s0 = ld_shared_f32(sca + 8 * k);
            if (32 * j + 2 * k + 1 < valid) s1 = ld_shared_f32(sca + 8 * k + 4);
            pk[k] = pack_bf16(p0 * s0, p1 * s1);
          } else {
            pk[k] = pack_bf16(p0, p1);
          }
        }
        }
        l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));

        // zero cache rows past the sequence end (garbage could be NaN)
        if (valid < kPage) {
          const uint32_t st = base + s * kStageBytes;
          const int rows = kPage - valid, per_box = rows * 8;
          constexpr int kBoxes = kF8 ? 2 : 4;  // latent boxes of a stage (128-byte rows)
          for (int idx = h + 128 * j; idx < kBoxes * per_box; idx += 256) {
            const int box = idx / per_box, rem = idx % per_box;
            st_shared_v4(st + box * kBox + (valid + rem / 8) * 128 + (rem % 8) * 16, 0, 0, 0, 0);
          }
        }

        // P buffer gi&1 (tensor memory) is free once the P . V of page gi-2 has
        // finished; O may be rescaled only after the P . V of page gi-1
        const uint32_t pb = gi & 1;
        if (gi >= 2 && !wwait(B_PVD + pb, ((gi >> 1) - 1) & 1)) { ok = false; break; }
        const bool any_resc = __any_sync(0xffffffffu, resc);
        if (any_resc && !wwait(B_PVD + (pb ^ 1), ((gi - 1) >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (any_resc) {  // this warpgroup's 128 O columns
          const float f = resc ? alpha : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t r[32];
            const uint32_t col = tmem + lane_base + kTmO + j * 128 + cc * 32;
            tmem_ld32(col, r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * f);
            tmem_st32(col, r);
          }
          tmem_wait_st();
        }
        // this warpgroup's 32 tokens of P in 16 tensor-memory columns: bf16
        // pairs, or (8-bit) the hi term's codes in 8 columns, then the lo term's
        tmem_st16(tmem + lane_base + kTmP + pb * 32 + j * 16, pk);
        tmem_wait_st();
        fence_proxy_async_smem();  // the zeroed stage rows above
        tc_fence_before();
        mbar_arrive(bar(B_PFULL + pb));
      }
      if (!ok) break;

      Unit nu;
      const bool have_next = wk.next(a, nu);

      // epilogue: the row sum is the two warpgroups' partial sums; each
      // normalises its 128 of this CTA's 256 latent columns
      if (!wwait(B_ODONE, uc & 1)) break;
      tc_fence_after();
      uint32_t l_other;
      if (!swap_sum(__float_as_uint(l), l_other)) break;
      const float lt = l + __uint_as_float(l_other);
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const size_t row = (size_t)u.b * H + h;
      const size_t prow = (size_t)u.slot * H + h;
      const int col0 = rank * 256 + j * 128;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kTmO + j * 128 + cc * 32, r);
        tmem_wait_ld();
        if (h < H) {
          // a whole sequence goes to o_lat, a split one to its partial slot
          __nv_bfloat16* dst_row = u.split ? a.part_o + prow * kLatent : a.o_lat + row * kLatent;
          uint4* dst = reinterpret_cast<uint4*>(dst_row + col0 + cc * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pack_bf16(__uint_as_float(r[8 * v]) * inv, __uint_as_float(r[8 * v + 1]) * inv),
                                pack_bf16(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv),
                                pack_bf16(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv),
                                pack_bf16(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv));
        }
      }
      if (rank == 0 && j == 0 && h < H) {
        const float lse = lt > 0.f ? (m - kShift + log2f(lt)) * kLn2 : -INFINITY;
        if (!u.split) {
          if (a.lse) a.lse[row] = lse;
        } else {
          a.part_lse[prow] = lse;
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_OFREE));
      g += np;
      ++uc;
      u = nu;
      have = have_next;
    }
  }
  tc_fence_before();
  __syncthreads();
  // the peer no longer touches this CTA's shared memory: every copy and
  // remote arrive it sent here has been waited for by this CTA, so the
  // barrier need not wait for this CTA's output stores to drain
  cluster_sync_relaxed();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// Clusters of the decode kernel that fit on the device at once (0 on error).
int decode_tc_max_clusters() {
  constexpr uint32_t smem = Layout<0>::kSmemBytes;
  if (cudaFuncSetAttribute(decode_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<0>, &cfg) != cudaSuccess) return 0;
  return n;
}

// bf16 cache: tiles TMA-loaded straight into the 128-byte-swizzled stages.
// E4M3 cache (kv_scale != null): raw tiles without swizzle, expanded in the
// kernel; or, with the E4M3 query (q8 != null), tiles in the layouts the
// 8-bit MMAs read (128-byte swizzle for the latent, 32-byte for k_pe).
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t stream) {
  const bool fp8 = a.kv_scale != nullptr, mma8 = fp8 && a.q8 != nullptr;
  if ((reinterpret_cast<uintptr_t>(a.ckv) & 15) || (reinterpret_cast<uintptr_t>(a.kpe) & 15) ||
      (reinterpret_cast<uintptr_t>(a.kv_scale) & 15))
    return cudaErrorInvalidValue;
  if (mma8 && (a.q_terms < 1 || a.q_terms > 2 || a.p_terms < 1 || a.p_terms > 2 || !a.q8_scale ||
               (reinterpret_cast<uintptr_t>(a.q8) & 15)))
    return cudaErrorInvalidValue;
  CUtensorMap tc_map, tk_map;
  const cuuint64_t rows = (cuuint64_t)a.num_pages * kPage;
  const cuuint64_t es = fp8 ? 1 : 2;
  const cuuint64_t cd[2] = {kLatent, rows}, cs[1] = {kLatent * es};
  const cuuint64_t kd[2] = {kRope, rows}, ks[1] = {kRope * es};
  if (fp8) {
    const cuuint32_t cbox[2] = {128, 64}, kbox[2] = {32, 64};
    if (!make_tmap(&tc_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.ckv, cd, cs, cbox,
                   mma8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap(&tk_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.kpe, kd, ks, kbox,
                   mma8 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    const cuuint32_t box[2] = {64, 64}, kbox[2] = {32, 64};
    if (!make_tmap(&tc_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.ckv, cd, cs, box) ||
        !make_tmap(&tk_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.kpe, kd, ks, kbox,
                   CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  // the first unit's query (bf16 cache): [B*H rows x 512] latent, [B*H x 64] RoPE
  CUtensorMap tq_map, tqp_map;
  const cuuint64_t rows_q = (cuuint64_t)a.B * a.H;
  const cuuint64_t qd[2] = {kLatent, rows_q}, qst[1] = {kLatent * 2}, pd[2] = {kRope, rows_q}, pst[1] = {kRope * 2};
  const cuuint32_t qbox[2] = {64, 128}, pbox[2] = {32, 128};
  if ((reinterpret_cast<uintptr_t>(a.q_lat) & 15) || (reinterpret_cast<uintptr_t>(a.q_pe) & 15) ||
      !make_tmap(&tq_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q_lat, qd, qst, qbox) ||
      !make_tmap(&tqp_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q_pe, pd, pst, pbox, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  auto kernel = mma8 ? decode_tc_kernel<2> : fp8 ? decode_tc_kernel<1> : decode_tc_kernel<0>;
  const uint32_t smem = mma8 ? Layout<2>::kSmemBytes : fp8 ? Layout<1>::kSmemBytes : Layout<0>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(kernel, dim3(2 * a.G), dim3(kThreads), smem, stream, tc_map, tk_map, tq_map, tqp_map, a);
}

}  // namespace mla
