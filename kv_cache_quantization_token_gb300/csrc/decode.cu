// decode.cu -- KVarN decode attention over the compressed cache on sm_103a.
//
// Split-tile design (SharpInference issue #433, item 2: a fixed worst-case
// grid over (head, tile range) with early exit, followed by an LSE combine;
// the deferred inverse WHT is applied after combining the rotated partials):
//
//   split kernel   grid (item, KV head, sequence), 4 or 8 warps per CTA.
//                  Items 0..tile_items-1 own 2 or 4 consecutive packed tiles,
//                  staged in shared memory by TMA, one per warp pair; each warp takes 64
//                  tokens of its tile: the score and value contractions run
//                  as mma.sync m16n8k16 with A fragments built straight from
//                  the packed codes, and the warp keeps its own streaming-
//                  softmax state, merged with the others' once per item. The
//                  remaining items own chunks of FP32 window rows (raw rows,
//                  unrotated query), one chunk per warp.
//   combine kernel grid (query head, sequence): LSE merge of the items, one
//                  inverse rotation of the merged tile accumulator, plus the
//                  (unrotated) window accumulator, divided by the softmax sum.
//
// Scores use the scales folded at read time (SharpInference issue #180,
// "Algorithm (per 128-token tile)" step 4): with q' = scale * H q,
//   z_t = r_t * sum_c q'_c s_c (delta_c code_tc + lo_c)
//       = r_t * (sum_c wd_c code_tc + bias),   wd_c = q'_c s_c delta_c,
// and the value aggregate stays in the rotated space:
//   acc_c = s_c * (sum_t p_t r_t delta_tg code_tc + sum_t p_t r_t lo_tg).
// Every query head of a KV head's GQA group is served from one pass over the
// packed codes. Every wait on a copy is bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "kvarn_common.cuh"

// Built six times: for records with fp32 or binary16 scale fields
// (KVARN_BUILD_SCALE_BYTES 4 or 2) and 2-, 3- or 4-bit value codes
// (KVARN_BUILD_V_BITS). The fp32 / 2-bit unit also holds the plan, the
// combine kernel and the dispatch.
#ifndef KVARN_BUILD_SCALE_BYTES
#define KVARN_BUILD_SCALE_BYTES 4
#endif
#ifndef KVARN_BUILD_V_BITS
#define KVARN_BUILD_V_BITS 2
#endif
#define KVARN_PRIMARY_UNIT (KVARN_BUILD_SCALE_BYTES == 4 && KVARN_BUILD_V_BITS == 2)

namespace kvarn {
namespace {

constexpr int kSB = KVARN_BUILD_SCALE_BYTES;
constexpr int kVB = KVARN_BUILD_V_BITS;
// Width of the value codes the value contraction reads: 3-bit records are
// repacked into 4-bit codes in shared memory first (see repack_v3_to_v4).
constexpr int kVF = kVB == 3 ? 4 : kVB;

constexpr float kNegInf = -INFINITY;
constexpr float kLog2eD = 1.4426950408889634f;
constexpr float kLn2D = 0.6931471805599453f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Bounded wait for a copy: gives up after a fixed time (reporting
// KVARN_DEVERR_WAIT) instead of spinning forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err) {
  return mbar_wait_timed(bar, parity, err, KVARN_DEVERR_WAIT);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
// Sums v[j] over the 32 lanes for every j < N (N a power of two <= 32) with
// halving exchanges; returns the total of row win_row_of_lane<N>(lane).
template <int N>
__device__ __forceinline__ int win_row_of_lane(int lane) {
  int r = 0;
#pragma unroll
  for (int s = 0; (1 << s) < N; ++s) r |= ((lane >> s) & 1) * (N >> (s + 1));
  return r;
}
template <int N>
__device__ __forceinline__ float warp_reduce_rows(float (&v)[N], int lane) {
#pragma unroll
  for (int s = 0; (1 << s) < N; ++s) {
    const int n = N >> s, m = 1 << s;
    const bool up = lane & m;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float send = up ? v[j] : v[j + n / 2];
      const float keep = up ? v[j + n / 2] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  float r = v[0];
#pragma unroll
  for (int m = N; m < 32; m <<= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
  return r;
}

// One warp rotates one query head: x = scale/sqrt(D) * H q, written to
// qs[c * GP + h]. Heads h >= G (padding of the GQA group) are zero.
template <int D, int GP>
__device__ __forceinline__ void rotate_head_to_smem(const float* qh, bool valid, float scale,
                                                    float* qs, int h, int lane) {
  constexpr int E = D / 32;
  float x[E];
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = valid ? qh[lane * E + e] : 0.f;
#pragma unroll
  for (int s = 1; s < E; s <<= 1)
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (!(e & s)) {
        const float a = x[e], b = x[e | s];
        x[e] = a + b;
        x[e | s] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool up = lane & m;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = up ? (o - x[e]) : (x[e] + o);
    }
  }
  const float f = scale / sqrtf((float)D);
#pragma unroll
  for (int e = 0; e < E; ++e) qs[(lane * E + e) * GP + h] = x[e] * f;
}

// ---------------------------------------------------------------------------
// Tensor-core (mma.sync m16n8k16, fp16 x fp16 -> fp32) formulation of the two
// contractions of a packed tile, with fragments built straight from the codes:
//  scores  S[t][n] = sum_c A[t][c] B[c][n]   A = code 2^-20 (an fp16 subnormal,
//                                            exact), B = the folded query,
//                                            split hi+lo
//          sum_c wd_c code_tc = 2^20 S
//  values  O[c][n] = sum_t A[c][t] B[t][n]   A = code 2^-18 (2-bit codes) or
//                                            code 2^-20 (4-bit), B = p r delta
//                                            hi+lo
//          sum_t pd_t code_tc = 2^18 O or 2^20 O
// A code moved to the top of the mantissa bits of its 16-bit half (bits 4..7
// for a nibble, 6..7 for a 2-bit field) and masked is a subnormal, so a
// fragment register is at most one shift and one AND of the loaded codes. The
// tensor core sums subnormal products in a window placed as if each were as
// large as the smallest normal, so codes sit near the top of the subnormal
// range: low in the mantissa they would lose up to 12 bits of the sum.
// Columns n are (query head, hi/lo part) pairs, 8 per n-tile. Each B operand is
// scaled by a power of two per head (exact) so the fp16 parts stay in range.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// fp16 pair {c_lo 2^-20, c_hi 2^-20} (subnormals) from nibble n (0..3) of the
// low and of the high 16-bit half of x: the nibble moved to bits 4..7.
__device__ __forceinline__ uint32_t k_frag(uint32_t x, int n) {
  const uint32_t y = n == 0 ? x << 4 : n == 1 ? x : x >> (4 * n - 4);
  return y & 0x00F000F0u;
}
// fp16 pair {c_lo 2^-18, c_hi 2^-18} (subnormals) from 2-bit field f (0..7) of
// each 16-bit half of x: the field moved to bits 6..7.
__device__ __forceinline__ uint32_t v_frag(uint32_t x, int f) {
  const uint32_t y = f < 3 ? x << (6 - 2 * f) : f == 3 ? x : x >> (2 * f - 6);
  return y & 0x00C000C0u;
}
// 2^20 and 2^18: the inverse scale of a fragment's codes
constexpr float kKCodeInv = 1048576.0f;
constexpr float kVCodeInv = kVF == 2 ? 262144.0f : 1048576.0f;
// Physical offset of logical byte o of a 1024-byte aligned region written by a
// TMA copy with 128-byte swizzling (16-byte chunk index XOR 128-byte line index).
__device__ __forceinline__ uint32_t swz128(uint32_t o) { return o ^ (((o >> 7) & 7u) << 4); }
// Four 8x8 matrices of 16-bit elements, transposed: lanes 8i..8i+7 give the
// row addresses of matrix i, whose fragment lands in r[i].
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
// 2D tensor copy (box of the tensor map) into shared memory, completing on bar.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// 2^e for the power-of-two scale that brings max |x| = m into [2^10, 2^11)
// (1 when m is zero or not finite), and its inverse times `k`.
__device__ __forceinline__ void pow2_scale(float m, float k, float& scale, float& inv_k) {
  const int ex = (__float_as_int(m) >> 23) & 0xFF;  // biased exponent of m (m >= 0)
  int e = (m > 0.f && ex < 255) ? 137 - ex : 0;     // m * 2^e in [2^10, 2^11)
  e = max(-120, min(120, e));
  scale = __int_as_float((127 + e) << 23);
  inv_k = k * __int_as_float((127 - e) << 23);
}

// Transposes an 8x8 matrix of 16-bit pairs held one row pair per lane (lane
// 4g + q holds row g, columns 2q and 2q+1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
// {fp16(x), fp16(x - fp16(x))} packed low/high: x to about 22 bits.
__device__ __forceinline__ uint32_t hilo_one(float x) {
  const float hf = __half2float(__float2half_rn(x));
  const __half2 r = __floats2half2_rn(x, x - hf);
  return *reinterpret_cast<const uint32_t*>(&r);
}
// 2^x on the special-function unit (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One warp rotates one query head for the tile path: x = f / sqrt(D) * H q,
// stored as channel pairs interleaved by head (qs[((c/2) * GP + h) * 2 + c % 2])
// so that the lanes of a fragment read their pairs without bank conflicts,
// plus max_c |x_c| in qmax[h].
template <int D, int GP>
__device__ __forceinline__ void rotate_head_pairs(const float* qh, bool valid, float f_scale,
                                                  float* qs, float* qmax, int h, int lane) {
  constexpr int E = D / 32;
  float x[E];
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = valid ? qh[lane * E + e] : 0.f;
#pragma unroll
  for (int s = 1; s < E; s <<= 1)
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (!(e & s)) {
        const float a = x[e], b = x[e | s];
        x[e] = a + b;
        x[e | s] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool up = lane & m;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = up ? (o - x[e]) : (x[e] + o);
    }
  }
  const float f = f_scale / sqrtf((float)D);
  float mx = 0.f;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const int c = lane * E + e;
    const float2 v = make_float2(x[e] * f, x[e + 1] * f);
    *reinterpret_cast<float2*>(qs + ((c >> 1) * GP + h) * 2) = v;
    mx = fmaxf(mx, fmaxf(fabsf(v.x), fabsf(v.y)));
  }
  mx = warp_max(mx);
  if (lane == 0) qmax[h] = mx;
}

// Eight 3-bit fields of x (bits 3i..3i+2) to eight 4-bit ones (bits 4i..).
__device__ __forceinline__ uint32_t spread3to4(uint32_t x) {
  uint32_t y = (x & 0xFFFu) | ((x & 0xFFF000u) << 4);     // fields 4-7 to the high half-word
  y = (y & 0x003F003Fu) | ((y & 0x0FC00FC0u) << 2);        // fields 2, 3 (6, 7) to the next byte
  return (y & 0x07070707u) | ((y & 0x38383838u) << 1);     // the odd field of each byte up a bit
}

// 3-bit value codes of a landed record (token rows of 3 D / 8 bytes at 64 D,
// a little-endian bit stream per row) rewritten as 4-bit rows of D / 2 bytes
// at offset 0, over the K codes; both regions carry the record box's 128-byte
// swizzle (64 D is a multiple of 1024, so offsets map alike). Thread `id` of
// `nth` converts 32-channel blocks: 12 bytes in, 16 bytes out.
template <int D>
__device__ __forceinline__ void repack_v3_to_v4(unsigned char* slot, int id, int nth) {
  constexpr int CB = D / 32;  // 32-channel blocks per token
  for (int u = id; u < 128 * CB; u += nth) {
    const int t = u / CB, cb = u % CB;
    const uint32_t src = (uint32_t)(64 * D + t * (3 * D / 8) + 12 * cb);
    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(slot + swz128(src));
    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(slot + swz128(src + 4));
    const uint32_t w2 = *reinterpret_cast<const uint32_t*>(slot + swz128(src + 8));
    uint4 o;
    o.x = spread3to4(w0 & 0xFFFFFFu);
    o.y = spread3to4((w0 >> 24) | ((w1 & 0xFFFFu) << 8));
    o.z = spread3to4((w1 >> 16) | ((w2 & 0xFFu) << 16));
    o.w = spread3to4(w2 >> 8);
    *reinterpret_cast<uint4*>(slot + swz128((uint32_t)(t * (D / 2) + 16 * cb))) = o;
  }
}

template <int D, int GP, int NW_, int WPT_, bool MR_ = false>
struct DC {
  static constexpr int NW = NW_;                                // warps per CTA (2, 4 or 8)
  static constexpr int NTHR = 32 * NW;
  static constexpr int WPT = WPT_;                              // warps per tile (2 or 4)
  static constexpr int TPS = NW / WPT;                          // tiles per round
  static constexpr int CH = 4 / WPT;                            // 32-token chunks per warp
  static constexpr int RB = Rec<D, kSB, kVB>::kBytes;           // record bytes
  static constexpr int SLOT = Rec<D, kSB, kVB>::kSlot;          // record slot stride in shared memory
  static constexpr int GV = Rec<D, kSB, kVB>::kGv;
  static constexpr int K_BYTES = 64 * D;                        // K codes: D rows of 64 bytes
  static constexpr int CODE_BYTES = (64 + 16 * kVB) * D;        // K + V codes, one TMA box
  static constexpr int CODE_LINES = CODE_BYTES / 128;           // 128-byte lines of that box
  static constexpr int NT = GP > 4 ? 2 : 1;                     // n8-tiles of (head, part) columns
  static constexpr int NCB = D / 16;                            // 16-channel blocks
  static constexpr int HB = NCB / WPT;                          // blocks whose B fragments a warp builds
  // value contraction: slices of VSL channels of a V row, MU m-blocks of 16
  // channels each; lane group g8 owns channels VSL sl + CPL g8 + 2 mu + {0, 1}
  static constexpr int VSL = kVF == 2 ? 64 : 32;
  static constexpr int NS = D / VSL;
  static constexpr int MU = kVF == 2 ? 4 : 2;
  static constexpr int CPL = kVF == 2 ? 8 : 4;
  // where the value contraction finds its codes in a record slot, and the
  // bytes per token row there: 3-bit codes are repacked into 4-bit rows over
  // the K codes (dead once the scores are formed; the same 64 D bytes)
  static constexpr int V_OFF = kVB == 3 ? 0 : K_BYTES;
  static constexpr int V_ROW = kVF * D / 8;
  // window rows staged per warp, sized by the record region of the fp32
  // layout (two slots per group with multi-round items), whatever the scale width
  static constexpr int WCH0 = ((MR_ ? 2 : 1) * TPS * Rec<D, 4>::kBytes) / (NW * 2 * D * 4);
  static constexpr int WCH = WCH0 >= 16 ? 16 : WCH0 >= 8 ? 8 : WCH0 >= 4 ? 4 : 2;
  static constexpr int DP = D + 8;                              // padded channel stride of the merge
  static constexpr int MRG = NW * GP * DP * 4;                  // merge region [NW][GP][DP], over records
  // Small regions first, then the record slots (1024-byte aligned for the
  // swizzled boxes): TPS slots, or 2 TPS when the warp groups take several
  // tiles in turn.
  static constexpr int OFF_QS = 0;                              // f32 query [D/2][GP][2] (window: [D][GP])
  static constexpr int OFF_QMAX = OFF_QS + D * GP * 4;          // f32 [8] max |q'| per head
  // tile items: B fragments [TPS][NCB][NT][32] x u32x2; window items: their
  // probabilities [NW WCH][GP] and reduction slots [NW][32] in the same bytes
  static constexpr int BX_BYTES = TPS * NCB * NT * 32 * 8;
  static constexpr int SCW_BYTES = (NW * WCH * GP * 4 + 15) / 16 * 16;
  static constexpr int WIN_BYTES = SCW_BYTES + NW * 32 * 4;
  static constexpr int OFF_BX = OFF_QMAX + 32;
  static constexpr int OFF_SCW = OFF_BX;
  static constexpr int OFF_WRED = OFF_BX + SCW_BYTES;
  static constexpr int OFF_PT = OFF_BX + (BX_BYTES > WIN_BYTES ? BX_BYTES : WIN_BYTES);  // bias [TPS][WPT][GP]
  static constexpr int OFF_FLG = OFF_PT + TPS * WPT * GP * 4;   // int [2 TPS]: slot copy issued / parity pending
  static constexpr int NBAR = 2 * TPS > NW ? 2 * TPS : NW;       // one per record slot, or per window chunk
  static constexpr int OFF_BAR = (OFF_FLG + 2 * TPS * 4 + 7) / 8 * 8;
  static constexpr int OFF_REC = (OFF_BAR + NBAR * 8 + 1023) / 1024 * 1024;
  static constexpr int WSTAGE = 2 * WCH * D * 4 * NW;           // window rows of one item
  static constexpr int REC_MIN0 = TPS * SLOT > MRG + NW * 128 ? TPS * SLOT : MRG + NW * 128;
  static constexpr int REC_MIN = REC_MIN0 > WSTAGE ? REC_MIN0 : WSTAGE;
  static constexpr int OFF_TRED = MRG;                          // tile items' reduction slots (record-relative)
  // dynamic shared memory for `slots` record slots (without the alignment slack)
  static constexpr int smem_bytes(int slots) {
    return OFF_REC + (slots * SLOT > REC_MIN ? slots * SLOT : REC_MIN);
  }
  static_assert(D == 64 || D == 128 || D == 256, "head_dim");
  static_assert(SLOT % 1024 == 0 && K_BYTES % 1024 == 0, "slots and V codes on swizzle atoms");
  static_assert(CODE_LINES <= 256 && CODE_BYTES == Rec<D, kSB, kVB>::kKDelta, "code box");
  static_assert(HB >= 1 && WPT * HB == NCB && (WPT == 2 || WPT == 4), "channel blocks per warp");
  static_assert(NW * GP * D * 4 <= REC_MIN, "window partials fit the record region");
};

// Sum over the CTA (NW warps) of per-thread vectors v[N]; every thread gets the totals.
template <int N, int NW>
__device__ __forceinline__ void cta_sum(float (&v)[N], float* red, int tid) {
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = warp_sum(v[i]);
  __syncthreads();  // red may still be read from the previous use
  if ((tid & 31) == 0)
#pragma unroll
    for (int i = 0; i < N; ++i) red[(tid >> 5) * 32 + i] = v[i];
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += red[w * 32 + i];
    v[i] = s;
  }
}
template <int N, int NW>
__device__ __forceinline__ void cta_max(float (&v)[N], float* red, int tid) {
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = warp_max(v[i]);
  __syncthreads();
  if ((tid & 31) == 0)
#pragma unroll
    for (int i = 0; i < N; ++i) red[(tid >> 5) * 32 + i] = v[i];
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float s = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) s = fmaxf(s, red[w * 32 + i]);
    v[i] = s;
  }
}

// MR: multi-round items (each warp group takes several tiles in turn, records
// double-buffered); without it every group takes at most one tile.
template <int D, int GP, int NW_, int WPT_, bool MR>
__global__ void __launch_bounds__(32 * NW_, GP <= 4 ? (MR || NW_ == 8 ? 3 : 6) : 1)
decode_split_kernel(const float* __restrict__ q, const uint8_t* __restrict__ tiles,
                    const int64_t* __restrict__ tile_table, const int32_t* __restrict__ n_tiles,
                    const float* __restrict__ win_k, const float* __restrict__ win_v,
                    const int32_t* __restrict__ win_start, const int32_t* __restrict__ win_len,
                    int cap, int Hq, int Hkv, int G, int max_tiles, int items, int tile_items,
                    int rounds_arg, float scale, float* __restrict__ ws_ml, float* __restrict__ ws_acc,
                    int prefetch, int64_t tiles_bytes, unsigned* err,
                    const __grid_constant__ CUtensorMap tmap) {
  using C = DC<D, GP, NW_, WPT_, MR>;
  using R = Rec<D, kSB, kVB>;
  constexpr int NW = C::NW, NT = C::NT, GV = C::GV, NCB = C::NCB, NS = C::NS, TPS = C::TPS;
  constexpr int HB = C::HB, WPT = C::WPT, CH = C::CH;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzled TMA boxes need 1024-byte aligned slots (the launch adds the slack)
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* rec = smem + C::OFF_REC;
  const int item = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = lane >> 2, q4 = lane & 3;  // mma fragment coordinates
  const bool is_win = item >= tile_items;
  const int64_t part = ((int64_t)b * Hq + (int64_t)kvh * G) * items + item;
  const int rounds = MR ? rounds_arg : 1;
  const int span = TPS * rounds;  // packed tiles of a tile item
  // Under programmatic dependent launch, wait for the previous kernel on the
  // stream before touching memory; with prefetch, tile items first read
  // n_tiles, the tile table and their records (which, by the caller's
  // guarantee, no earlier kernel still running writes) and wait afterwards.
  const bool early = prefetch && !is_win;
  if (!early) pdl_wait();

  // work of this item: packed tiles, or window chunks of WCH rows (one per warp)
  int nslot, wlen = 0, wstart = 0, wj0 = 0;
  if (!is_win) {
    const int nt = min(max(n_tiles[b], 0), max_tiles);
    nslot = min(max(nt - item * span, 0), span);
  } else {
    wlen = min(max(win_len[b], 0), cap);
    wstart = ((win_start[b] % cap) + cap) % cap;
    wj0 = C::WCH * NW * (item - tile_items);
    nslot = min(max((wlen - wj0 + C::WCH - 1) / C::WCH, 0), NW);
  }
  if (nslot == 0) {
    if (early) pdl_wait();
    pdl_trigger();
    if (tid < G) {
      ws_ml[(part + (int64_t)tid * items) * 2 + 0] = kNegInf;
      ws_ml[(part + (int64_t)tid * items) * 2 + 1] = 0.f;
    }
    return;
  }
  float* sc = reinterpret_cast<float*>(smem + C::OFF_SCW);
  float* qs = reinterpret_cast<float*>(smem + C::OFF_QS);
  float* red = reinterpret_cast<float*>(is_win ? smem + C::OFF_WRED : rec + C::OFF_TRED);
  int* okf = reinterpret_cast<int*>(smem + C::OFF_FLG);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

  if (is_win) {
    // ===================== window chunk: raw rows, SIMT =====================
    pdl_trigger();
    const int64_t head_base = ((int64_t)b * Hkv + kvh) * cap;
    if (tid == 0) {
      for (int kk = 0; kk < nslot; ++kk) mbar_init(&bar[kk], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (lane == 0 && warp < nslot) {
      // this warp's chunk: n consecutive ring slots from s0, in at most two pieces
      const int kk = warp;
      const int n = min(C::WCH, wlen - (wj0 + C::WCH * kk));
      const int s0 = (wstart + wj0 + C::WCH * kk) % cap;
      const int n1 = min(n, cap - s0);
      mbar_expect_tx(&bar[kk], (uint32_t)(n * D * 4 * 2));
      unsigned char* dst = rec + kk * (2 * C::WCH * D * 4);
      bulk_g2s(dst, win_k + (head_base + s0) * D, n1 * D * 4, &bar[kk]);
      bulk_g2s(dst + C::WCH * D * 4, win_v + (head_base + s0) * D, n1 * D * 4, &bar[kk]);
      if (n1 < n) {
        bulk_g2s(dst + n1 * D * 4, win_k + head_base * D, (n - n1) * D * 4, &bar[kk]);
        bulk_g2s(dst + (C::WCH + n1) * D * 4, win_v + head_base * D, (n - n1) * D * 4, &bar[kk]);
      }
    }
    for (int idx = tid; idx < D * GP; idx += C::NTHR) {
      const int c = idx / GP, h = idx % GP;
      qs[idx] = h < G ? scale * q[((int64_t)b * Hq + (int64_t)kvh * G + h) * D + c] : 0.f;
    }
    __syncthreads();
    const int k = warp;
    const bool have = k < nslot;
    bool ok = have && mbar_wait(&bar[k], 0, err);
    const float* Kw = reinterpret_cast<const float*>(rec + k * (2 * C::WCH * D * 4));
    const float* Vw = Kw + C::WCH * D;
    const int wn = min(C::WCH, wlen - (wj0 + C::WCH * k));
    constexpr int E = D / 32;
    const int wtok = win_row_of_lane<C::WCH>(lane);
    float zw[GP], mx[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) { zw[h] = kNegInf; mx[h] = kNegInf; }
    if (ok) {
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        float qv[E];
#pragma unroll
        for (int e = 0; e < E; ++e) qv[e] = qs[(lane * E + e) * GP + h];
        float part_[C::WCH];
#pragma unroll
        for (int j = 0; j < C::WCH; ++j) {
          float a = 0.f;
          if (j < wn) {
#pragma unroll
            for (int e = 0; e < E; ++e) a = fmaf(qv[e], Kw[j * D + lane * E + e], a);
          }
          part_[j] = a;
        }
        zw[h] = warp_reduce_rows<C::WCH>(part_, lane);
        if (wtok < wn) mx[h] = zw[h];
      }
    }
    cta_max<GP, NW>(mx, red, tid);
    float l[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) l[h] = 0.f;
    if (ok && lane < C::WCH) {
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float p = wtok < wn ? expf(zw[h] - mx[h]) : 0.f;
        l[h] = p;
        sc[(k * C::WCH + wtok) * GP + h] = p;
      }
    }
    __syncwarp();
    float acc[E][GP];
#pragma unroll
    for (int e = 0; e < E; ++e)
#pragma unroll
      for (int h = 0; h < GP; ++h) acc[e][h] = 0.f;
    if (ok) {
#pragma unroll
      for (int j = 0; j < C::WCH; ++j) {
        if (j < wn) {
          float pv[GP];
#pragma unroll
          for (int h = 0; h < GP; ++h) pv[h] = sc[(k * C::WCH + j) * GP + h];
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float x = Vw[j * D + lane * E + e];
#pragma unroll
            for (int h = 0; h < GP; ++h) acc[e][h] = fmaf(pv[h], x, acc[e][h]);
          }
        }
      }
    }
    bool bad = have && !ok;
    bad = __syncthreads_or(bad);
    cta_sum<GP, NW>(l, red, tid);
    // the partial acc of the warps is summed through the (now free) staging region
    float* vred = reinterpret_cast<float*>(rec);
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e)
#pragma unroll
      for (int h = 0; h < GP; ++h) vred[(warp * GP + h) * D + lane * E + e] = acc[e][h];
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += C::NTHR) {
      const int h = idx / D, c = idx % D;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) s += vred[(w * GP + h) * D + c];
      ws_acc[(part + (int64_t)h * items) * D + c] = bad ? NAN : s;
    }
    if (tid < G) {
      float Mh = mx[0], lh = l[0];
#pragma unroll
      for (int h = 1; h < GP; ++h)
        if (h == tid) { Mh = mx[h]; lh = l[h]; }
      ws_ml[(part + (int64_t)tid * items) * 2 + 0] = bad ? NAN : Mh;
      ws_ml[(part + (int64_t)tid * items) * 2 + 1] = bad ? NAN : lh;
    }
    return;
  }

  // ========================= packed tiles, tensor cores ======================
  // Warp group p = warp / WPT owns tile p of the item; warp w of the group
  // takes the tile's tokens 32 CH (w % WPT) .. +32 CH - 1 (CH = 4 / WPT
  // chunks of 32). The group shares the folded query (each warp builds 1/WPT
  // of its channel blocks; one group barrier per tile), each warp contracts
  // scores and values of its tokens on mma.sync and keeps its own
  // streaming-softmax state (m, l, acc) per query head; the NW warps' states
  // are merged at the end of the item.
  //
  // Each record slot holds the K and V codes as one 128B-swizzled TMA box
  // (K: channel rows of 64 bytes, V: token rows of D/4 bytes) followed by the
  // scales. ldmatrix.trans reads 8 rows x 16 bytes of codes and leaves in lane
  // (g8, q4) rows 2q4 and 2q4+1 at byte pair g8: two channels x four tokens
  // (K) or two tokens x eight channels (V), a fragment's worth of codes.
  const int64_t* trow = tile_table + ((int64_t)b * Hkv + kvh) * max_tiles + (int64_t)item * span;
  const int pair = warp / WPT, half = warp % WPT;  // warp group, warp within the group
  const bool dbuf = MR && rounds > 1;              // two record slots per group
  float* qmax = reinterpret_cast<float*>(smem + C::OFF_QMAX);
  uint2* bx = reinterpret_cast<uint2*>(smem + C::OFF_BX);     // [TPS][NCB][NT][32]
  float* pt = reinterpret_cast<float*>(smem + C::OFF_PT);     // [TPS][WPT][GP]
  const bool issuer = lane == 0 && half == 0;                 // the group's copy issuer
  // Copies a packed tile into a record slot (one TMA box of codes plus one bulk
  // copy of the scales, completing on the slot's barrier); okf[slot] tells
  // the group whether a copy was issued (record offsets must be multiples of
  // 128 bytes and the record must lie inside the pool; others poison the
  // result and are reported).
  auto issue = [&](int li, int slot) {
    const int64_t off = trow[li];
    const bool aligned = (off & 127) == 0 && off >= 0 && off <= tiles_bytes - C::RB &&
                         (off >> 7) < 0x7FFFFFFFLL;
    if (!aligned) report(err, KVARN_DEVERR_RECORD);
    okf[slot] = aligned;
    if (aligned) {
      mbar_expect_tx(&bar[slot], C::RB);
      tma_load_2d(rec + slot * C::SLOT, &tmap, 0, (int)(off >> 7), &bar[slot]);
      bulk_g2s(rec + slot * C::SLOT + C::CODE_BYTES, tiles + off + C::CODE_BYTES,
               C::RB - C::CODE_BYTES, &bar[slot]);
    }
    return aligned;
  };
  if (tid == 0) {
    for (int kk = 0; kk < (dbuf ? 2 * TPS : TPS); ++kk) mbar_init(&bar[kk], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // copies in flight that this issuer has not seen land: parity + 1, per slot of its group
  int pend0 = 0, pend1 = 0;
  if (issuer) {
    if (pair < nslot && issue(pair, pair)) pend0 = 1;
    if (dbuf && pair + TPS < nslot && issue(pair + TPS, pair + TPS)) pend1 = 1;
  }
  if (early) pdl_wait();
  pdl_trigger();
  // scores are kept in base-2 units (scale * log2 e folded into the query); the
  // item's (max, sum) pair is converted back to natural-log units when stored
  for (int h = warp; h < GP; h += NW)
    rotate_head_pairs<D, GP>(q + ((int64_t)b * Hq + (int64_t)kvh * G + h) * D, h < G,
                             scale * kLog2eD, qs, qmax, h, lane);
  __syncthreads();
  int bad = 0;

  // B view (fragment column g8): head 4nt + hb, hi part when is_hi.
  // Accumulator view (columns 2q4, 2q4+1): head 4nt + q4, hi + lo parts.
  const int hb = g8 >> 1;
  const bool is_hi = !(g8 & 1);
  float m_run[NT], l_run[NT];
  constexpr int MU = C::MU;
  float out_acc[NS][MU][2][NT];  // channel VSL sl + CPL g8 + 2 mu + rr, head 4nt + q4
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) { m_run[nt] = kNegInf; l_run[nt] = 0.f; }
#pragma unroll
  for (int sl = 0; sl < NS; ++sl)
#pragma unroll
    for (int mu = 0; mu < MU; ++mu)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) out_acc[sl][mu][rr][nt] = 0.f;

  // group `pair` takes the item's tiles pair, pair + TPS, ... in turn
  for (int k = 0; k < rounds && pair + TPS * k < nslot; ++k) {  // uniform over the group
    const int kk = pair;
    const int slot = pair + (dbuf ? TPS * (k & 1) : 0);
    const uint32_t par = dbuf ? (uint32_t)((k >> 1) & 1) : 0u;
    const unsigned char* Rk = rec + slot * C::SLOT;
    const uint32_t rk = smem_u32(Rk);
    const bool landed = okf[slot] && mbar_wait(&bar[slot], par, err);
    if (!landed) bad = 1;  // computed on, result poisoned
    if (issuer && landed) {
      if (k & 1) pend1 = 0; else pend0 = 0;
    }
    const unsigned char* kS = Rk + R::kKS;  // scale fields (fp32 or binary16)
    const unsigned char* kD = Rk + R::kKDelta;
    const unsigned char* kL = Rk + R::kKLo;
    const unsigned char* kR = Rk + R::kKR;

    // ---- folded query wd_c = q'_c s_c delta_c, one power-of-two scale per head
    // from the bound max|q'| * max_c s_c delta_c (the same in both warps)
    float mf = 0.f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i)
      mf = fmaxf(mf, fabsf(sc_ld<kSB>(kS, lane + 32 * i) * sc_ld<kSB>(kD, lane + 32 * i)));
    mf = warp_max(mf);
    float scB[NT], invA[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float s_, i_;
      const float qb = 4 * nt + hb < GP ? qmax[4 * nt + hb] : 0.f;
      const float qa = 4 * nt + q4 < GP ? qmax[4 * nt + q4] : 0.f;
      pow2_scale(qb * mf, 1.0f, scB[nt], i_);
      pow2_scale(qa * mf, 1.0f, s_, invA[nt]);
    }
    // this warp's share of the channel blocks: B fragments to shared memory, and
    // per-head partial sums of the bias q' s lo. In block cb,
    // lane (g8, q4) forms both fp16 parts of wd for head 4nt + hb on the channel
    // pair 16 cb + 2 q4 + 8 (g8 & 1) and swaps one part with lane ^ 4, which
    // took the other pair of the same head: the hi lane keeps both hi parts,
    // the lo lane both lo parts.
    const int hl = g8 & 1;
    float2 bsum[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) bsum[nt] = make_float2(0.f, 0.f);
#pragma unroll
    for (int u = 0; u < HB; ++u) {
      const int cb = HB * half + u;
      const int c = 16 * cb + 2 * q4 + 8 * hl;
      const float2 s = sc_ld2<kSB>(kS, c);
      const float2 dd = sc_ld2<kSB>(kD, c);
      const float2 lo = sc_ld2<kSB>(kL, c);
      const float2 sd = __fmul2_rn(s, dd), sl = __fmul2_rn(s, lo);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h = 4 * nt + hb;
        const float2 qv = h < GP ? *reinterpret_cast<const float2*>(qs + ((c >> 1) * GP + h) * 2)
                                 : make_float2(0.f, 0.f);
        const float2 x = __fmul2_rn(qv, sd);
        bsum[nt] = __ffma2_rn(qv, sl, bsum[nt]);
        const float2 xs = __fmul2_rn(x, make_float2(scB[nt], scB[nt]));
        const __half2 hi = __floats2half2_rn(xs.x, xs.y);
        const float2 hf = __half22float2(hi);
        const __half2 lo16 = __floats2half2_rn(xs.x - hf.x, xs.y - hf.y);
        const uint32_t hu = *reinterpret_cast<const uint32_t*>(&hi);
        const uint32_t lu = *reinterpret_cast<const uint32_t*>(&lo16);
        const uint32_t got = __shfl_xor_sync(0xffffffffu, hl ? hu : lu, 4);
        bx[((kk * NCB + cb) * NT + nt) * 32 + lane] = hl ? make_uint2(got, lu) : make_uint2(hu, got);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float bs = bsum[nt].x + bsum[nt].y;
#pragma unroll
      for (int m = 1; m <= 4; m <<= 1)  // over q4 and the hi/lo lane: all channels of this warp's share
        bs += __shfl_xor_sync(0xffffffffu, bs, m);
      if (q4 == 0 && is_hi && 4 * nt + hb < GP) pt[(kk * WPT + half) * GP + 4 * nt + hb] = bs;
    }
    asm volatile("bar.sync %0, %1;" ::"r"(1 + pair), "n"(32 * WPT) : "memory");  // the group's barrier

    // the bias sum_c q'_c s_c lo_c per head of the accumulator view (head 4nt + q4)
    float cstA[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float bs = 0.f;
      if (4 * nt + q4 < GP) {
#pragma unroll
        for (int w = 0; w < WPT; ++w) bs += pt[(kk * WPT + w) * GP + 4 * nt + q4];
      }
      cstA[nt] = bs;
    }

    // ---- phase A: scores of this warp's 32 CH tokens. Chunk w4 = tokens 32 w4 ..
    // +31 (w4 = CH half + w2); M-block j: row g8 <-> token 32 w4 + 4 g8 + 2j,
    // row g8 + 8 <-> that token + 1.
    const int mi = lane >> 3, ri = lane & 7;
    const uint32_t kaddr0 =
        (uint32_t)((16 * (mi >> 1) + 8 * (mi & 1) + ri) * 64 + 16 * (CH * half));
    float acc[CH][2][NT][4];
#pragma unroll
    for (int w2 = 0; w2 < CH; ++w2)
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[w2][j][nt][e] = 0.f;
#pragma unroll
    for (int cp = 0; cp < NCB; cp += 2) {
      uint2 bf[2][NT];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) bf[u][nt] = bx[((kk * NCB + cp + u) * NT + nt) * 32 + lane];
#pragma unroll
      for (int w2 = 0; w2 < CH; ++w2) {
        uint32_t x[4];  // channel blocks cp, cp+1; channels +0..7 and +8..15 of each
        ldsm_x4_t(rk + swz128(kaddr0 + (uint32_t)(cp * 16 * 64 + 16 * w2)), x[0], x[1], x[2], x[3]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t xl = x[2 * u], xh = x[2 * u + 1];
          const uint32_t a00 = k_frag(xl, 0), a01 = k_frag(xl, 1), a02 = k_frag(xh, 0), a03 = k_frag(xh, 1);
          const uint32_t a10 = k_frag(xl, 2), a11 = k_frag(xl, 3), a12 = k_frag(xh, 2), a13 = k_frag(xh, 3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(acc[w2][0][nt], a00, a01, a02, a03, bf[u][nt].x, bf[u][nt].y);
            mma16816(acc[w2][1][nt], a10, a11, a12, a13, bf[u][nt].x, bf[u][nt].y);
          }
        }
      }
    }

    // ---- scores z = r_t (sum_c wd_c code_tc + bias) and the warp's softmax
    float z[CH][2][2][NT];
#pragma unroll
    for (int w2 = 0; w2 < CH; ++w2) {
      const float4 r4 = sc_ld4<kSB>(kR, 32 * (CH * half + w2) + 4 * g8);
      const float rt[2][2] = {{r4.x, r4.y}, {r4.z, r4.w}};
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            z[w2][j][rr][nt] =
                rt[j][rr] * fmaf((acc[w2][j][nt][2 * rr] + acc[w2][j][nt][2 * rr + 1]) * kKCodeInv,
                                 invA[nt], cstA[nt]);
    }
    // streaming state of the warp: the running maximum moves to mn, earlier
    // sums are rescaled by alpha (0 on the group's first tile)
    float alpha[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float mx = kNegInf;
#pragma unroll
      for (int w2 = 0; w2 < CH; ++w2)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) mx = fmaxf(mx, z[w2][j][rr][nt]);
#pragma unroll
      for (int m = 4; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
      const float mn = fmaxf(m_run[nt], mx);
      alpha[nt] = ex2_approx(m_run[nt] - mn);
      m_run[nt] = mn;
      float ls = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < CH; ++w2)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            z[w2][j][rr][nt] = ex2_approx(z[w2][j][rr][nt] - mn);  // now p
            ls += z[w2][j][rr][nt];
          }
      l_run[nt] = k == 0 ? ls : fmaf(l_run[nt], alpha[nt], ls);
    }

    // ---- value side: pd_t = p_t r_t delta_tg as fp16 hi + lo, transposed into
    // B fragments with movmatrix. K-block (w2, j) of phase B holds tokens
    // 32 w4 + 8 q4 + 2j + {0, 4} (b0) and + {1, 5} (b1).
    const unsigned char* vR = Rk + R::kVR;
    const unsigned char* vD = Rk + R::kVDelta;
    const unsigned char* vL = Rk + R::kVLo;
    const unsigned char* vS = Rk + R::kVS;
    uint32_t bB[GV][CH][2][NT][2];
    float invP[GV][NT], cstP[GV][NT];
#pragma unroll
    for (int gv = 0; gv < GV; ++gv) {
      float pd[CH][2][2][NT], pm[NT], lt[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) { pm[nt] = 0.f; lt[nt] = 0.f; }
#pragma unroll
      for (int w2 = 0; w2 < CH; ++w2) {
        const int t0 = 32 * (CH * half + w2) + 4 * g8;
        const float4 vr4 = sc_ld4<kSB>(vR, t0);
        const float vrt[4] = {vr4.x, vr4.y, vr4.z, vr4.w};
        float dv[4], lv[4];
        if constexpr (GV == 1) {
          const float4 d4 = sc_ld4<kSB>(vD, t0);
          const float4 l4 = sc_ld4<kSB>(vL, t0);
          dv[0] = d4.x; dv[1] = d4.y; dv[2] = d4.z; dv[3] = d4.w;
          lv[0] = l4.x; lv[1] = l4.y; lv[2] = l4.z; lv[3] = l4.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dv[e] = sc_ld<kSB>(vD, (t0 + e) * GV + gv);
            lv[e] = sc_ld<kSB>(vL, (t0 + e) * GV + gv);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float d = dv[e], lo = lv[e];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float pv = z[w2][e >> 1][e & 1][nt] * vrt[e];
            pd[w2][e >> 1][e & 1][nt] = pv * d;
            pm[nt] = fmaxf(pm[nt], fabsf(pv * d));
            lt[nt] = fmaf(pv, lo, lt[nt]);
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int m = 4; m < 32; m <<= 1) pm[nt] = fmaxf(pm[nt], __shfl_xor_sync(0xffffffffu, pm[nt], m));
        float sc2, inv2;
        pow2_scale(pm[nt], 1.0f, sc2, inv2);
#pragma unroll
        for (int w2 = 0; w2 < CH; ++w2)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float xa = pd[w2][j][0][nt] * sc2, xb = pd[w2][j][1][nt] * sc2;
            const uint32_t xl = hilo_one(xa);  // row g8: token 4 g8 + 2j
            const uint32_t xh = hilo_one(xb);  // token 4 g8 + 2j + 1
            bB[gv][w2][j][nt][0] = movmatrix_t(xl);
            bB[gv][w2][j][nt][1] = movmatrix_t(xh);
          }
        float l2 = lt[nt];
#pragma unroll
        for (int m = 4; m < 32; m <<= 1) l2 += __shfl_xor_sync(0xffffffffu, l2, m);
        invP[gv][nt] = inv2;
        cstP[gv][nt] = l2;
      }
    }

    if constexpr (kVB == 3) {
      // every warp of the group is past its reads of the K codes: the value
      // codes go over them as 4-bit rows, then the group reads those
      asm volatile("bar.sync %0, %1;" ::"r"(1 + pair), "n"(32 * WPT) : "memory");
      repack_v3_to_v4<D>(const_cast<unsigned char*>(Rk), 32 * half + lane, 32 * WPT);
      asm volatile("bar.sync %0, %1;" ::"r"(1 + pair), "n"(32 * WPT) : "memory");
    }

    // ---- phase B: this warp's 32 CH tokens against all channels, one slice of
    // VSL channels of the V rows at a time. 2-bit codes: m-block mu of slice sl
    // row g8 <-> channel 64 sl + 8 g8 + 2 mu, row g8 + 8 <-> that channel + 1;
    // 4-bit codes: row g8 <-> channel 32 sl + 4 g8 + 2 mu, row g8 + 8 <-> + 1.
    const uint32_t vaddr0 =
        (uint32_t)(C::V_OFF + (32 * CH * half + 4 * ri + 2 * (mi >> 1) + (mi & 1)) * C::V_ROW);
#pragma unroll
    for (int sl = 0; sl < NS; ++sl) {
      const int gv = (C::VSL * sl) / R::kVGroup;
      float o[MU][NT][4];
#pragma unroll
      for (int mu = 0; mu < MU; ++mu)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[mu][nt][e] = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < CH; ++w2) {
        uint32_t y[4];  // (K-block j, b0/b1 tokens) = (0,0), (0,1), (1,0), (1,1)
        ldsm_x4_t(rk + swz128(vaddr0 + (uint32_t)(32 * w2 * C::V_ROW + 16 * sl)), y[0], y[1], y[2],
                  y[3]);
#pragma unroll
        for (int mu = 0; mu < MU; ++mu)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint32_t a0, a1, a2, a3;
            if constexpr (kVF == 2) {  // fields 2 mu and 2 mu + 1
              a0 = v_frag(y[2 * j], 2 * mu); a1 = v_frag(y[2 * j], 2 * mu + 1);
              a2 = v_frag(y[2 * j + 1], 2 * mu); a3 = v_frag(y[2 * j + 1], 2 * mu + 1);
            } else {  // nibbles 2 mu and 2 mu + 1
              a0 = k_frag(y[2 * j], 2 * mu); a1 = k_frag(y[2 * j], 2 * mu + 1);
              a2 = k_frag(y[2 * j + 1], 2 * mu); a3 = k_frag(y[2 * j + 1], 2 * mu + 1);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816(o[mu][nt], a0, a1, a2, a3, bB[gv][w2][j][nt][0], bB[gv][w2][j][nt][1]);
          }
      }
      // acc_c = alpha acc_c + s_c (2^-e 2^18 O + sum p r lo) (2^20 for 4-bit codes)
      float sv[MU][2];
#pragma unroll
      for (int h4 = 0; h4 < MU / 2; ++h4) {
        const float4 s4 = sc_ld4<kSB>(vS, C::VSL * sl + C::CPL * g8 + 4 * h4);
        sv[2 * h4][0] = s4.x; sv[2 * h4][1] = s4.y;
        sv[2 * h4 + 1][0] = s4.z; sv[2 * h4 + 1][1] = s4.w;
      }
      if (k == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int mu = 0; mu < MU; ++mu)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const float O = (o[mu][nt][2 * rr] + o[mu][nt][2 * rr + 1]) * kVCodeInv;
              out_acc[sl][mu][rr][nt] = sv[mu][rr] * fmaf(O, invP[gv][nt], cstP[gv][nt]);
            }
      } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int mu = 0; mu < MU; ++mu)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const float O = (o[mu][nt][2 * rr] + o[mu][nt][2 * rr + 1]) * kVCodeInv;
              out_acc[sl][mu][rr][nt] = fmaf(out_acc[sl][mu][rr][nt], alpha[nt],
                                             sv[mu][rr] * fmaf(O, invP[gv][nt], cstP[gv][nt]));
            }
      }
    }
    if (dbuf) {
      // the group is done with this slot (and with its fragments): refill it
      // with the group's tile two turns ahead, unless its copy never landed
      asm volatile("bar.sync %0, %1;" ::"r"(1 + pair), "n"(32 * WPT) : "memory");
      const int nxt = pair + TPS * (k + 2);
      if (issuer && k + 2 < rounds && nxt < nslot && landed && issue(nxt, slot)) {
        const int pv = (int)(((k + 2) >> 1) & 1) + 1;
        if (k & 1) pend1 = pv; else pend0 = pv;
      }
      if (issuer && k + 2 < rounds && nxt < nslot && !landed) okf[slot] = 0;
    }
  }
  bad = __syncthreads_or(bad);
  if (bad && issuer)  // let every copy that was issued land before the CTA exits (bounded)
  {
    if (pend0) mbar_wait(&bar[pair], (uint32_t)(pend0 - 1), err);
    if (pend1) mbar_wait(&bar[pair + TPS], (uint32_t)(pend1 - 1), err);
  }

  // ---------------- merge the warps' (m, l, acc) ---------------------------
  // Every warp stores its own (m, l) per head and its unscaled accumulator
  // (over the dead records); each output then takes the maximum over the
  // warps and sums their accumulators rescaled to it.
  float* vred = reinterpret_cast<float*>(rec);  // [NW][GP][DP], over the dead records
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int m = 4; m < 32; m <<= 1) l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], m);
    const int h = 4 * nt + q4;
    if (h < GP) {
      if (g8 == 0) {
        red[warp * 32 + h] = m_run[nt];
        red[warp * 32 + 8 + h] = l_run[nt];
      }
#pragma unroll
      for (int sl = 0; sl < NS; ++sl)
#pragma unroll
        for (int mu = 0; mu < MU; ++mu)
          *reinterpret_cast<float2*>(vred + (warp * GP + h) * C::DP + C::VSL * sl + C::CPL * g8 + 2 * mu) =
              make_float2(out_acc[sl][mu][0][nt], out_acc[sl][mu][1][nt]);
    }
  }
  __syncthreads();
  {
    // each thread takes channels of one head, so that the head's maximum and
    // the warps' weights are formed once per thread, not once per channel
    constexpr int TPH = C::NTHR / GP;  // threads per head slot
    const int h = tid / TPH;
    if (h < G) {
      float M = kNegInf;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, red[w * 32 + h]);
      float f[NW];
      unsigned has = 0u;  // warps with a tile (m = -inf: none)
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float mw = red[w * 32 + h];
        f[w] = ex2_approx(mw - M);
        if (mw != kNegInf) has |= 1u << w;
      }
      for (int c = tid % TPH; c < D; c += TPH) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w)
          if (has & (1u << w)) s = fmaf(vred[(w * GP + h) * C::DP + c], f[w], s);
        ws_acc[(part + (int64_t)h * items) * D + c] = bad ? NAN : s;
      }
    }
  }
  if (tid < G) {
    float M = kNegInf, L = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red[w * 32 + tid]);
#pragma unroll
    for (int w = 0; w < NW; ++w)
      if (red[w * 32 + tid] != kNegInf) L += red[w * 32 + 8 + tid] * ex2_approx(red[w * 32 + tid] - M);
    ws_ml[(part + (int64_t)tid * items) * 2 + 0] = bad ? NAN : M * kLn2D;
    ws_ml[(part + (int64_t)tid * items) * 2 + 1] = bad ? NAN : L;
  }
}

#if KVARN_PRIMARY_UNIT
// LSE combine: one CTA of 512 threads per (query head, sequence). Each group
// of D/4 threads reads whole item rows (float4 per thread, coalesced) of
// every (512/(D/4))-th item in one pass, keeping its own running maximum; the
// groups are merged in shared memory, the tile part is rotated back with one
// FWHT, the window part added, and the result divided by the softmax sum.
template <int D>
__global__ void __launch_bounds__(512)
decode_combine_kernel(const float* __restrict__ ws_ml, const float* __restrict__ ws_acc, int Hq,
                      int items, int tile_items, float* __restrict__ out) {
  constexpr int NTH = 512, TPR = D / 4, NG = NTH / TPR;
  __shared__ float4 grp[2][NG][TPR];
  __shared__ float gm[NG], gl[NG];
  __shared__ float x[D];
  const int hq = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int64_t base = ((int64_t)b * Hq + hq) * items;
  pdl_trigger();
  pdl_wait();
  const int gi = tid / TPR, c4 = tid % TPR;
  float m = kNegInf, L = 0.f;
  float4 ar = make_float4(0.f, 0.f, 0.f, 0.f), aw = ar;
  int poison = 0;
  constexpr int U = 8;  // items per thread whose loads are issued together
  for (int j0 = gi; j0 < items; j0 += U * NG) {
    float2 mlv[U];
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u * NG;
      mlv[u] = make_float2(kNegInf, 0.f);
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < items) {
        mlv[u] = reinterpret_cast<const float2*>(ws_ml)[base + j];
        v[u] = reinterpret_cast<const float4*>(ws_acc + (base + j) * D)[c4];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u * NG;
      const float mj = mlv[u].x, lj = mlv[u].y;
      if (j < items && !(lj >= 0.f)) poison = 1;  // NaN partial (a failed split item)
      if (lj > 0.f) {  // empty items (never written) are skipped before any arithmetic
        const float mn = fmaxf(m, mj);
        const float a = expf(m - mn), w = expf(mj - mn);  // a = 0 while m = -inf
        const bool tile = j < tile_items;
        const float wt = tile ? w : 0.f, ww = tile ? 0.f : w;
        ar = make_float4(fmaf(ar.x, a, wt * v[u].x), fmaf(ar.y, a, wt * v[u].y),
                         fmaf(ar.z, a, wt * v[u].z), fmaf(ar.w, a, wt * v[u].w));
        aw = make_float4(fmaf(aw.x, a, ww * v[u].x), fmaf(aw.y, a, ww * v[u].y),
                         fmaf(aw.z, a, ww * v[u].z), fmaf(aw.w, a, ww * v[u].w));
        L = fmaf(L, a, w * lj);
        m = mn;
      }
    }
  }
  grp[0][gi][c4] = ar;
  grp[1][gi][c4] = aw;
  if (c4 == 0) {
    gm[gi] = m;
    gl[gi] = L;
  }
  poison = __syncthreads_or(poison);
  float xr = 0.f, xw = 0.f, Lt = 0.f;
  if (tid < D) {
    float M = kNegInf;
#pragma unroll
    for (int g = 0; g < NG; ++g) M = fmaxf(M, gm[g]);
    const float* g0 = reinterpret_cast<const float*>(grp[0]);
    const float* g1 = reinterpret_cast<const float*>(grp[1]);
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const float f = gm[g] == kNegInf ? 0.f : expf(gm[g] - M);
      xr = fmaf(f, g0[g * D + tid], xr);
      xw = fmaf(f, g1[g * D + tid], xw);
      Lt = fmaf(f, gl[g], Lt);
    }
    // FWHT: butterflies within the warp by shuffles, across warps through x[]
#pragma unroll
    for (int h = 1; h < 32 && h < D; h <<= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, xr, h);
      xr = (tid & h) ? (o - xr) : (xr + o);
    }
  }
  for (int h = 32; h < D; h <<= 1) {
    if (tid < D) x[tid] = xr;
    __syncthreads();
    if (tid < D) {
      const float o = x[tid ^ h];
      xr = (tid & h) ? (o - xr) : (xr + o);
    }
    __syncthreads();
  }
  if (tid < D) {
    float r = 0.f;
    if (Lt > 0.f) r = (xr * (1.0f / sqrtf((float)D)) + xw) / Lt;
    if (poison) r = NAN;
    out[((int64_t)b * Hq + hq) * D + tid] = r;
  }
}

#endif  // KVARN_PRIMARY_UNIT

// cuTensorMapEncodeTiled, fetched once from the driver (the library links the
// static CUDA runtime only).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// Tensor map over the record pool seen as rows of 128 bytes: a box of
// code_lines rows starting at row offset/128 is the K and V codes of the
// record at that offset, copied with 128-byte swizzling. The row count is the
// pool's, so no box reaches past it (rows beyond are zero-filled; the kernel
// also refuses offsets whose record would not fit).
cudaError_t code_map(CUtensorMap* m, const void* tiles, int64_t tiles_bytes, int code_lines) {
  memset(m, 0, sizeof(*m));
  if (!tiles || tiles_bytes < 128) return cudaSuccess;  // no record can be read: the map is never used
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return cudaErrorNotSupported;
  const int64_t rows = tiles_bytes / 128 < 0x7FFFFFFF ? tiles_bytes / 128 : 0x7FFFFFFF;
  const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, (cuuint32_t)code_lines};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(tiles), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int GP, int NW, int WPT, bool MR>
cudaError_t launch_split_t(const DecodePlan& p, const DecodeArgs& a, float* ws_ml, float* ws_acc,
                           cudaStream_t st) {
  using C = DC<D, GP, NW, WPT, MR>;
  constexpr int kMaxSmem = C::smem_bytes(MR ? 2 * C::TPS : C::TPS) + 1024;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(decode_split_kernel<D, GP, NW, WPT, MR>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  CUtensorMap tmap;
  e = code_map(&tmap, p.tile_items > 0 ? a.tiles : nullptr, a.tiles_bytes, C::CODE_LINES);
  if (e != cudaSuccess) return e;
  const unsigned fl = a.flags;
  const int prefetch = (fl & KVARN_LAUNCH_PDL) && (fl & KVARN_LAUNCH_PREFETCH);
  const int slots = MR && p.rounds > 1 ? 2 * C::TPS : C::TPS;
  LaunchCfg L(dim3(p.items, a.Hkv, a.B), dim3(C::NTHR), C::smem_bytes(slots) + 1024, st, fl);
  return cudaLaunchKernelEx(&L.cfg, decode_split_kernel<D, GP, NW, WPT, MR>, a.q, a.tiles, a.tile_table,
                            a.n_tiles, a.win_k, a.win_v, a.win_start, a.win_len, a.win_capacity,
                            a.Hq, a.Hkv, a.Hq / a.Hkv, a.max_tiles, p.items, p.tile_items, p.rounds,
                            a.scale, ws_ml, ws_acc, prefetch, a.tiles_bytes, a.err, tmap);
}

template <int D, int GP>
cudaError_t launch_split_g(const DecodePlan& p, const DecodeArgs& a, float* ws_ml, float* ws_acc,
                           cudaStream_t st) {
  // The plans decode_plan() makes: head_dim <= 128 takes a warp pair per
  // tile, 4 tiles per round (one round) or 2 (one or more rounds); head_dim
  // 256 four warps per tile, one tile per round.
  if constexpr (D <= 128) {
    if (p.warps_per_tile != 2) return cudaErrorInvalidValue;
    if (p.tiles_per_round == 4 && p.rounds == 1)
      return launch_split_t<D, GP, 8, 2, false>(p, a, ws_ml, ws_acc, st);
    if (p.tiles_per_round == 2)
      return p.rounds > 1 ? launch_split_t<D, GP, 4, 2, true>(p, a, ws_ml, ws_acc, st)
                          : launch_split_t<D, GP, 4, 2, false>(p, a, ws_ml, ws_acc, st);
  } else {
    if (p.warps_per_tile == 4 && p.tiles_per_round == 1)
      return p.rounds > 1 ? launch_split_t<D, GP, 4, 4, true>(p, a, ws_ml, ws_acc, st)
                          : launch_split_t<D, GP, 4, 4, false>(p, a, ws_ml, ws_acc, st);
  }
  return cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_split_d(const DecodePlan& p, const DecodeArgs& a, float* ws_ml, float* ws_acc,
                           cudaStream_t st) {
  switch (p.g_pad) {
    case 1: return launch_split_g<D, 1>(p, a, ws_ml, ws_acc, st);
    case 2: return launch_split_g<D, 2>(p, a, ws_ml, ws_acc, st);
    case 4: return launch_split_g<D, 4>(p, a, ws_ml, ws_acc, st);
    case 8: return launch_split_g<D, 8>(p, a, ws_ml, ws_acc, st);
    default: return cudaErrorInvalidValue;
  }
}

void ws_split(const DecodePlan& p, int B, int Hq, void* ws, float** ml, float** acc) {
  const size_t parts = (size_t)B * Hq * p.items;
  const size_t mlb = (parts * 2 * sizeof(float) + 255) / 256 * 256;
  *ml = reinterpret_cast<float*>(ws);
  *acc = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + mlb);
}

}  // namespace

#if KVARN_PRIMARY_UNIT
int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

int decode_plan(int B, int Hq, int Hkv, int D, int max_tiles, int win_capacity, DecodePlan* p) {
  const int G = Hq / Hkv;
  p->g_pad = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8;
  // head_dim <= 128: a warp pair per tile, 2 tiles per CTA at a time, or 4
  // (eight warps) once the grid has at least 4 tiles per SM, which halves the
  // partials the combine reads and the per-CTA set-up. head_dim 256: four
  // warps per tile (32 tokens each) and one tile per CTA at a time, whose
  // record is twice as large; the extra warps per SM hide more of each warp's
  // mma.sync / shuffle chain. When there are many more tiles than the SMs hold
  // at once, each warp group takes several tiles in turn (rounds), its next
  // record streaming into a second slot while it works on the current one:
  // the query rotation, the merge of the warps and the partial written for
  // the combine are then paid once per item instead of once per tile.
  const int64_t total = (int64_t)B * Hkv * max_tiles;
  const int64_t per_sm = total / sm_count();
  const int wpt = D <= 128 ? 2 : 4;
  const bool multi = D <= 128 ? per_sm > 8 : per_sm >= 12;
  const int tps = D <= 128 ? (multi ? 2 : total >= 4LL * sm_count() ? 4 : 2) : 1;
  const int nw = wpt * tps;
  // window rows per warp and per item, as DC<D, GP, NW, WPT, MR>::WCH and its NW warps
  const int rb = 112 * D + 1024 + 1024 * (D > 128 ? D / 128 : 1);
  const int w0 = ((multi ? 2 : 1) * tps * rb) / (nw * 2 * D * 4);
  const int wch = w0 >= 16 ? 16 : w0 >= 8 ? 8 : w0 >= 4 ? 4 : 2;
  p->win_items = win_capacity > 0 ? (win_capacity + nw * wch - 1) / (nw * wch) : 0;
  // rounds: the fewest (2..8) whose grid fits one wave of the multi-round
  // kernel's resident CTAs (3 per SM, by shared memory), so that no second,
  // partial wave runs after the first; 8 when even that does not fit (many
  // waves: the last one matters little).
  int rounds = 1;
  if (multi) {
    const int64_t groups = (int64_t)B * Hkv, slots = 3LL * sm_count();
    for (rounds = 2; rounds < 8; ++rounds) {
      const int64_t ctas = groups * ((max_tiles + tps * rounds - 1) / (tps * rounds) + p->win_items);
      if (ctas <= slots) break;
    }
  }
  p->tiles_per_round = tps;
  p->rounds = rounds;
  p->tiles_per_item = tps * rounds;
  p->warps_per_tile = wpt;
  p->tile_items = max_tiles > 0 ? (max_tiles + p->tiles_per_item - 1) / p->tiles_per_item : 0;
  p->items = p->tile_items + p->win_items;
  const size_t parts = (size_t)B * Hq * p->items;
  const size_t ml = (parts * 2 * sizeof(float) + 255) / 256 * 256;
  p->ws_bytes = ml + parts * (size_t)D * sizeof(float);
  return 0;
}

cudaError_t launch_decode_split(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                cudaStream_t st) {
  const int key = 10 * a.scale_bytes + a.v_bits;
  switch (key) {
    case 42: return launch_decode_split_sb4_v2(p, a, ws, st);
    case 22: return launch_decode_split_sb2_v2(p, a, ws, st);
    case 44: return launch_decode_split_sb4_v4(p, a, ws, st);
    case 24: return launch_decode_split_sb2_v4(p, a, ws, st);
    case 43: return launch_decode_split_sb4_v3(p, a, ws, st);
    case 23: return launch_decode_split_sb2_v3(p, a, ws, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_combine(const DecodePlan& p, int B, int Hq, int D, const void* ws,
                                  float* out, unsigned flags, cudaStream_t st) {
  float *ml, *acc;
  ws_split(p, B, Hq, const_cast<void*>(ws), &ml, &acc);
  LaunchCfg L(dim3(Hq, B), dim3(512), 0, st, flags);
  const float* cml = ml;
  const float* cacc = acc;
  switch (D) {
    case 64: return cudaLaunchKernelEx(&L.cfg, decode_combine_kernel<64>, cml, cacc, Hq, p.items, p.tile_items, out);
    case 128: return cudaLaunchKernelEx(&L.cfg, decode_combine_kernel<128>, cml, cacc, Hq, p.items, p.tile_items, out);
    case 256: return cudaLaunchKernelEx(&L.cfg, decode_combine_kernel<256>, cml, cacc, Hq, p.items, p.tile_items, out);
    default: return cudaErrorInvalidValue;
  }
}

#endif  // KVARN_PRIMARY_UNIT

#if KVARN_BUILD_SCALE_BYTES == 4 && KVARN_BUILD_V_BITS == 2
cudaError_t launch_decode_split_sb4_v2(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st) {
#elif KVARN_BUILD_SCALE_BYTES == 2 && KVARN_BUILD_V_BITS == 2
cudaError_t launch_decode_split_sb2_v2(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st) {
#elif KVARN_BUILD_SCALE_BYTES == 4 && KVARN_BUILD_V_BITS == 4
cudaError_t launch_decode_split_sb4_v4(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st) {
#elif KVARN_BUILD_SCALE_BYTES == 2 && KVARN_BUILD_V_BITS == 4
cudaError_t launch_decode_split_sb2_v4(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st) {
#elif KVARN_BUILD_SCALE_BYTES == 4 && KVARN_BUILD_V_BITS == 3
cudaError_t launch_decode_split_sb4_v3(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st) {
#else
cudaError_t launch_decode_split_sb2_v3(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st) {
#endif
  if (p.items == 0) return cudaSuccess;
  float *ml, *acc;
  ws_split(p, a.B, a.Hq, ws, &ml, &acc);
  switch (a.D) {
    case 64: return launch_split_d<64>(p, a, ml, acc, st);
    case 128: return launch_split_d<128>(p, a, ml, acc, st);
    case 256: return launch_split_d<256>(p, a, ml, acc, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvarn
