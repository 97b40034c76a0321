// compress.cu -- KVarN tile compression on sm_103a.
//
// Per (128-token tile, KV head) unit and per tensor (K or V), as the method
// states it (SharpInference issue #180, "Algorithm (per 128-token tile)",
// steps 1-3; SharpInference PR #434, commit 82efc4f):
//   1. Walsh-Hadamard rotation of each token row along head_dim,
//   2. n rounds of dual-axis std normalisation, channel step first,
//   3. asymmetric RTN: K 4-bit per channel over the tile's tokens, V 2-bit (3 or 4 in the variants) per
//      token over 128-channel groups; codes packed into the record.
//
// GPU formulation (same result up to rounding as the log-space statement):
//  - The rotation is computed unnormalised (entries +-1); the 1/sqrt(D) factor
//    is carried by the channel factor s' = sqrt(D) s, which the normalisation
//    is invariant to.
//  - Log-space accumulation telescopes: after a channel step,
//    alpha_c = ln std_t(Y_tc e^{-beta_t}), and after a token step
//    beta_t = ln std_c(Y_tc e^{-alpha_c}). So the kernel keeps s' and r
//    directly and never evaluates log or exp; a skipped step (std not larger
//    than 2^-20 times the group's RMS) keeps the previous factor, which is
//    what ln(sigma) := 0 does in log space.
//  - Each std is a two-pass (mean, M2) per thread followed by Chan pairwise
//    merges across threads, so large group means do not cancel.
//
// Work decomposition: one CTA of 2*D threads per (unit, tensor); every thread
// holds an 8-token x 8-channel block of the tile in registers (64 floats, as
// channel pairs: the per-element arithmetic uses packed fp32x2 instructions).
//   phase 1: each thread loads 16-byte chunks of 512/D tokens straight from
//            global memory (fully coalesced) and runs the butterflies of the
//            channel bits it holds (bits 0,1 and 5..log2D-1);
//   phase 2: a swizzled shared-memory transpose gives the block layout, whose
//            in-thread channel bits 2..4 take the remaining butterflies.
// In the block layout token reductions run across lanes with shuffles only,
// channel reductions across lanes and then across warps through shared memory.
#include "kvarn_common.cuh"

namespace kvarn {
namespace {

template <int D>
struct CC {
  static constexpr int L = (D == 64) ? 6 : (D == 128) ? 7 : 8;
  static constexpr int NT = 2 * D;          // threads per CTA
  static constexpr int NCG = D / 8;         // channel groups (lanes sharing a token group)
  static constexpr int CG_BITS = L - 3;     // lane bits that index the channel group
  static constexpr int WARPS = NT / 32;
  static constexpr int TGW = 5 - CG_BITS;   // token-group bits inside a warp
  static constexpr int P1_TOK = 512 / D;    // tokens per thread in phase 1
  static constexpr int P1_K = D / 32;       // 16-byte chunks per token per thread in phase 1
  static constexpr int TOK_PER_WARP = 8 << TGW;
  // dynamic shared memory: tile, channel-reduction partials, two channel arrays
  static constexpr int OFF_RED = 128 * D * 4;
  static constexpr int OFF_CH = OFF_RED + WARPS * D * 8;
  static constexpr int SMEM = OFF_CH + 2 * D * 4;
  static_assert(D == 64 || D == 128 || D == 256, "head_dim");
};

// 16-byte chunk swizzle of the tile in shared memory: chunk J of token t is
// stored at J ^ sigma(t, J). It keeps the phase-1 128-byte row segments intact
// and makes the phase-2 scalar reads hit 32 distinct banks.
template <int L>
__device__ __forceinline__ int swz(int t, int J) {
  return J ^ (((J >> 3) | ((t >> 3) << (L - 5))) & 7);
}

__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }

// Packed fp32x2 arithmetic (one instruction for two IEEE round-to-nearest
// results): the per-element work below runs on channel pairs.
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// In-register butterflies over the two low bits of a float4.
__device__ __forceinline__ void fwht4(float4& v) {
  const float a = v.x + v.y, b = v.x - v.y, c = v.z + v.w, d = v.z - v.w;
  v.x = a + c; v.y = b + d; v.z = a - c; v.w = b - d;
}
__device__ __forceinline__ void bfly(float4& a, float4& b) {
  const float4 s = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
  b = make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w);
  a = s;
}

// Equal-count merge of (mean, M2) summaries; symmetric in its two arguments,
// so both lanes of a full exchange get bit-identical results.
__device__ __forceinline__ void merge_eq(float& mean, float& m2, float mb, float m2b, float cnt) {
  const float d = mb - mean;
  mean = (mean + mb) * 0.5f;
  m2 = (m2 + m2b) + d * d * (cnt * 0.5f);
}

// Halving stage over one lane bit for N (mean, M2) pairs: the lane keeps the
// lower half of its pairs when its lane bit is 0, the upper half otherwise,
// and merges in the partner's copy of the half it keeps.
template <int N>
__device__ __forceinline__ void halve_mv(float (&mn)[8], float (&m2)[8], int mask, bool upper,
                                         float cnt) {
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    const float sm = upper ? mn[j] : mn[j + N / 2];
    const float sq = upper ? m2[j] : m2[j + N / 2];
    const float km = upper ? mn[j + N / 2] : mn[j];
    const float kq = upper ? m2[j + N / 2] : m2[j];
    const float rm = shfl_xor(sm, mask), rq = shfl_xor(sq, mask);
    mn[j] = km; m2[j] = kq;
    merge_eq(mn[j], m2[j], rm, rq, cnt);
  }
}
template <int N>
__device__ __forceinline__ void halve_mm(float (&lo)[8], float (&hi)[8], int mask, bool upper) {
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    const float sl = upper ? lo[j] : lo[j + N / 2];
    const float sh = upper ? hi[j] : hi[j + N / 2];
    const float kl = upper ? lo[j + N / 2] : lo[j];
    const float kh = upper ? hi[j + N / 2] : hi[j];
    lo[j] = fminf(kl, shfl_xor(sl, mask));
    hi[j] = fmaxf(kh, shfl_xor(sh, mask));
  }
}

// Three-input minimum / maximum (a NaN operand is ignored, as in fminf).
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// floor(u) for 0 <= u < 2^23, in the low bits of the result: u + 2^23
// rounded toward -inf is 2^23 + floor(u) exactly (the spacing of floats in
// [2^23, 2^24) is 1). The RTN value u = (y - lo) / delta + 1/2 lies in
// [1/2, 2^b - 1/2] up to rounding, so its floor is the code itself.
__device__ __forceinline__ uint32_t floor_bits(float u) {
  return __float_as_uint(__fadd_rd(u, 8388608.0f));
}
// base with its bits pos .. pos + len - 1 replaced by the low len bits of
// field (one bit-field insert)
__device__ __forceinline__ uint32_t bfi(uint32_t field, uint32_t base, uint32_t pos, uint32_t len) {
  uint32_t r;
  asm("bfi.b32 %0, %1, %2, %3, %4;" : "=r"(r) : "r"(field), "r"(base), "r"(pos), "r"(len));
  return r;
}
// 1 / delta, or 0 when delta is 0 or subnormal (every code of the group is
// then 0 and the group reconstructs to lo)
__device__ __forceinline__ float rtn_inv(float delta) {
  return delta >= 1.17549435e-38f ? 1.0f / delta : 0.f;
}

// Usable std: larger than 2^-20 times the RMS of the same group, compared in
// squares, var > 2^-40 (var + mean^2) (false for NaN).
__device__ __forceinline__ bool usable(float var, float mean) {
  return var > 0x1p-40f * fmaf(mean, mean, var);
}

template <int D, int SB, int VB>
__global__ void __launch_bounds__(CC<D>::NT, (D == 256) ? 1 : 2)
compress_kernel(const float* __restrict__ k_raw, const float* __restrict__ v_raw,
                int64_t row_stride, int64_t n_rows, const int64_t* __restrict__ src_row0,
                uint8_t* __restrict__ tiles, int64_t tiles_bytes,
                const int64_t* __restrict__ dst_record, int iters, unsigned* err) {
  using C = CC<D>;
  using R = Rec<D, SB, VB>;
  extern __shared__ __align__(16) unsigned char smem[];
  float* xs = reinterpret_cast<float*>(smem);
  float2* red = reinterpret_cast<float2*>(smem + C::OFF_RED);
  float* ch_a = reinterpret_cast<float*>(smem + C::OFF_CH);
  float* ch_b = ch_a + D;
  unsigned char* stage = smem;  // output staging aliases the tile (used after it is consumed)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t unit = blockIdx.x >> 1;
  const bool is_v = blockIdx.x & 1;
  // a unit whose rows or record lie outside the buffers is skipped (and reported)
  const int64_t row0 = src_row0[unit], dst = dst_record[unit];
  if (row0 < 0 || row0 > n_rows - 128 || dst < 0 || (dst & 15) || dst > tiles_bytes - R::kBytes) {
    if (tid == 0 && !is_v) report(err, KVARN_DEVERR_RECORD);
    return;
  }
  const float* src = (is_v ? v_raw : k_raw) + row0 * row_stride;

  // ---------------- phase 1: coalesced loads + butterflies of bits 0,1,5.. --
  {
    const int j0 = tid & 7, trow = tid >> 3;
    float4 x[C::P1_TOK][C::P1_K];
#pragma unroll
    for (int i = 0; i < C::P1_TOK; ++i) {
      const float4* row = reinterpret_cast<const float4*>(src + (int64_t)(trow + (D / 4) * i) * row_stride);
#pragma unroll
      for (int k = 0; k < C::P1_K; ++k) x[i][k] = ld_stream(row + j0 + 8 * k);
    }
#pragma unroll
    for (int i = 0; i < C::P1_TOK; ++i) {
#pragma unroll
      for (int k = 0; k < C::P1_K; ++k) fwht4(x[i][k]);
#pragma unroll
      for (int h = 1; h < C::P1_K; h <<= 1)
#pragma unroll
        for (int k = 0; k < C::P1_K; ++k)
          if (!(k & h)) bfly(x[i][k], x[i][k | h]);
      const int t = trow + (D / 4) * i;
#pragma unroll
      for (int k = 0; k < C::P1_K; ++k)
        *reinterpret_cast<float4*>(xs + t * D + 4 * swz<C::L>(t, j0 + 8 * k)) = x[i][k];
    }
  }
  __syncthreads();

  // ---------------- phase 2: block layout + butterflies of bits 2..4 --------
  const int cg = tid % C::NCG, tg = tid / C::NCG;
  // y2[i][k] = (channel slot 2k, 2k+1) of token 8 tg + i
  float2 y2[8][4];
  const float2 neg1 = f2(-1.f, -1.f);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = 8 * tg + i;
    float v[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int J = ((cg >> 2) << 3) + m;
      v[m] = xs[t * D + 4 * swz<C::L>(t, J) + (cg & 3)];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) y2[i][k] = f2(v[2 * k] + v[2 * k + 1], v[2 * k] - v[2 * k + 1]);
#pragma unroll
    for (int h = 1; h < 4; h <<= 1)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (!(k & h)) {
          const float2 a = y2[i][k], b = y2[i][k | h];
          y2[i][k] = add2(a, b);
          y2[i][k | h] = fma2(b, neg1, a);  // a - b, exactly
        }
  }

  // Sinkhorn state. sinv[m] = 1/s'_c for the thread's channels, rinv[i] = 1/r_t
  // for its tokens; s_own is owned by the thread pair (2p, 2p+1) of permuted
  // channel p, r_own by the lanes whose channel-group bits 0..2 encode token i.
  const float sqrt_d = sqrtf((float)D);
  float2 sinv2[4], rinv2[8];  // (1/s') of channel pairs; (1/r, 1/r) per token
#pragma unroll
  for (int k = 0; k < 4; ++k) sinv2[k] = f2(1.0f / sqrt_d, 1.0f / sqrt_d);
#pragma unroll
  for (int i = 0; i < 8; ++i) rinv2[i] = f2(1.0f, 1.0f);
  float s_own = sqrt_d, r_own = 1.0f;             // the factors (stored in the record)
  float si_own = 1.0f / sqrt_d, ri_own = 1.0f;    // their reciprocals (applied to the tile)
  const int p_own = tid >> 1, h_own = tid & 1;
  // token held by this lane after the row halving: bits (cg&1, cg>>1&1, cg>>2&1) -> 4,2,1
  const int tau = ((cg & 1) << 2) | (((cg >> 1) & 1) << 1) | ((cg >> 2) & 1);
  auto src_lane = [&](int i) {  // a lane of this token group that owns token i
    return (lane & ~7) | ((i >> 2) & 1) | (((i >> 1) & 1) << 1) | ((i & 1) << 2);
  };
  // channel index of permuted slot p = m * NCG + cg
  auto chan_of = [&](int p) {
    const int g = p % C::NCG, m = p / C::NCG;
    return (g & 3) | (m << 2) | ((g >> 2) << 5);
  };
  // which channels m a lane keeps after the in-warp token-group halving
  const int m_keep0 = (C::TGW == 0) ? 0
                    : (C::TGW == 1) ? 4 * ((lane >> 4) & 1)
                                    : 4 * ((lane >> 3) & 1) + 2 * ((lane >> 4) & 1);
  constexpr int KEEP = 8 >> C::TGW;

  for (int it = 0; it < iters; ++it) {
    // ---- channel step: std over the 128 tokens of Y' / r ----
    float cm[8], cq[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 s2 = f2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 8; ++i) s2 = fma2(y2[i][k], rinv2[i], s2);
      const float2 nmean = mul2(s2, f2(-0.125f, -0.125f));
      float2 q2 = f2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 d = fma2(y2[i][k], rinv2[i], nmean);
        q2 = fma2(d, d, q2);
      }
      cm[2 * k] = -nmean.x; cm[2 * k + 1] = -nmean.y;
      cq[2 * k] = q2.x; cq[2 * k + 1] = q2.y;
    }
    if (C::TGW >= 1) halve_mv<8>(cm, cq, 1 << C::CG_BITS, (lane >> C::CG_BITS) & 1, 8.f);
    if (C::TGW >= 2) halve_mv<4>(cm, cq, 1 << (C::CG_BITS + 1), (lane >> (C::CG_BITS + 1)) & 1, 16.f);
#pragma unroll
    for (int j = 0; j < KEEP; ++j)
      red[warp * D + (m_keep0 + j) * C::NCG + cg] = make_float2(cm[j], cq[j]);
    __syncthreads();
    {
      constexpr int HW = C::WARPS / 2;
      const float n1 = (float)C::TOK_PER_WARP;
      float2 a = red[(h_own * HW) * D + p_own];
      float mean = a.x, m2 = a.y, n = n1;
#pragma unroll
      for (int w = 1; w < HW; ++w) {
        const float2 b = red[(h_own * HW + w) * D + p_own];
        chan_merge(mean, m2, n, b.x, b.y, n1);
        n += n1;
      }
      merge_eq(mean, m2, shfl_xor(mean, 1), shfl_xor(m2, 1), 64.f);
      const float var = m2 * (1.0f / 128.0f);
      if (usable(var, mean)) {  // the std and its reciprocal from one rsqrt
        si_own = rsqrtf(var);
        s_own = var * si_own;
      }
      if (h_own == 0) ch_a[p_own] = si_own;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; ++k) sinv2[k] = f2(ch_a[(2 * k) * C::NCG + cg], ch_a[(2 * k + 1) * C::NCG + cg]);

    // ---- token step: std over the D channels of Y' / s' ----
    float rm[8], rq[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 s2 = f2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 4; ++k) s2 = fma2(y2[i][k], sinv2[k], s2);
      const float mean = (s2.x + s2.y) * 0.125f;
      const float2 nmean = f2(-mean, -mean);
      float2 q2 = f2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 d = fma2(y2[i][k], sinv2[k], nmean);
        q2 = fma2(d, d, q2);
      }
      rm[i] = mean; rq[i] = q2.x + q2.y;
    }
    halve_mv<8>(rm, rq, 1, lane & 1, 8.f);
    halve_mv<4>(rm, rq, 2, (lane >> 1) & 1, 16.f);
    halve_mv<2>(rm, rq, 4, (lane >> 2) & 1, 32.f);
    if (C::CG_BITS >= 4) merge_eq(rm[0], rq[0], shfl_xor(rm[0], 8), shfl_xor(rq[0], 8), 64.f);
    if (C::CG_BITS >= 5) merge_eq(rm[0], rq[0], shfl_xor(rm[0], 16), shfl_xor(rq[0], 16), 128.f);
    {
      const float var = rq[0] * (1.0f / (float)D);
      if (usable(var, rm[0])) {
        ri_own = rsqrtf(var);
        r_own = var * ri_own;
      }
      const float ri = ri_own;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float r = __shfl_sync(0xffffffffu, ri, src_lane(i));
        rinv2[i] = f2(r, r);
      }
    }
  }

  // ---------------- normalised values -------------------------------------
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) y2[i][k] = mul2(mul2(y2[i][k], sinv2[k]), rinv2[i]);
  // scalar view of the normalised block: y(i, m)
  auto y = [&](int i, int m) -> float { return (m & 1) ? y2[i][m >> 1].y : y2[i][m >> 1].x; };

  const int t_own = 8 * tg + tau;
  const bool tok_writer = (C::CG_BITS == 3) || ((cg >> 3) & 1) == 0;

  if (!is_v) {
    // ---------------- K: 4-bit RTN per channel over the 128 tokens ----------
    float lo[8], hi[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      lo[m] = fminf(min3f(min3f(min3f(y(0, m), y(1, m), y(2, m)), y(3, m), y(4, m)), y(5, m), y(6, m)), y(7, m));
      hi[m] = fmaxf(max3f(max3f(max3f(y(0, m), y(1, m), y(2, m)), y(3, m), y(4, m)), y(5, m), y(6, m)), y(7, m));
    }
    if (C::TGW >= 1) halve_mm<8>(lo, hi, 1 << C::CG_BITS, (lane >> C::CG_BITS) & 1);
    if (C::TGW >= 2) halve_mm<4>(lo, hi, 1 << (C::CG_BITS + 1), (lane >> (C::CG_BITS + 1)) & 1);
#pragma unroll
    for (int j = 0; j < KEEP; ++j) red[warp * D + (m_keep0 + j) * C::NCG + cg] = make_float2(lo[j], hi[j]);
    __syncthreads();  // also: every thread is past its last read of the tile
    {
      constexpr int HW = C::WARPS / 2;
      float2 a = red[(h_own * HW) * D + p_own];
      float l = a.x, h = a.y;
#pragma unroll
      for (int w = 1; w < HW; ++w) {
        const float2 b = red[(h_own * HW + w) * D + p_own];
        l = fminf(l, b.x); h = fmaxf(h, b.y);
      }
      l = fminf(l, shfl_xor(l, 1));
      h = fmaxf(h, shfl_xor(h, 1));
      const float delta = (h - l) / 15.0f;
      const float inv = rtn_inv(delta);
      if (h_own == 0) {
        ch_a[p_own] = l;
        ch_b[p_own] = inv;
        const int c = chan_of(p_own);
        sc_st<SB>(stage + R::kKDelta, c, delta);
        sc_st<SB>(stage + R::kKLo, c, l);
        sc_st<SB>(stage + R::kKS, c, s_own / sqrt_d);
      }
    }
    if (tok_writer) sc_st<SB>(stage + R::kKR, t_own, r_own);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // code = floor((y - lo) / delta + 1/2) for channel slots 2k, 2k+1
      const float2 nl = f2(-ch_a[(2 * k) * C::NCG + cg], -ch_a[(2 * k + 1) * C::NCG + cg]);
      const float2 inv = f2(ch_b[(2 * k) * C::NCG + cg], ch_b[(2 * k + 1) * C::NCG + cg]);
      uint32_t w0 = 0, w1 = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 u = fma2(add2(y2[i][k], nl), inv, f2(0.5f, 0.5f));
        w0 = bfi(floor_bits(u.x), w0, 4 * i, 4);
        w1 = bfi(floor_bits(u.y), w1, 4 * i, 4);
      }
      const int ca = (cg & 3) | ((2 * k) << 2) | ((cg >> 2) << 5);
      const int cb = (cg & 3) | ((2 * k + 1) << 2) | ((cg >> 2) << 5);
      *reinterpret_cast<uint32_t*>(stage + R::kKCodes + ca * (kTile / 2) + 4 * tg) = w0;
      *reinterpret_cast<uint32_t*>(stage + R::kKCodes + cb * (kTile / 2) + 4 * tg) = w1;
    }
  } else {
    // ---------------- V: VB-bit RTN per token over 128-channel groups --------
    constexpr int kVMax = (1 << VB) - 1;  // largest value code
    float lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lo[i] = fminf(min3f(min3f(min3f(y(i, 0), y(i, 1), y(i, 2)), y(i, 3), y(i, 4)), y(i, 5), y(i, 6)), y(i, 7));
      hi[i] = fmaxf(max3f(max3f(max3f(y(i, 0), y(i, 1), y(i, 2)), y(i, 3), y(i, 4)), y(i, 5), y(i, 6)), y(i, 7));
    }
    halve_mm<8>(lo, hi, 1, lane & 1);
    halve_mm<4>(lo, hi, 2, (lane >> 1) & 1);
    halve_mm<2>(lo, hi, 4, (lane >> 2) & 1);
    if (C::CG_BITS >= 4) {  // channel bit 5 (lane bit 3) stays inside one 128-channel group
      lo[0] = fminf(lo[0], shfl_xor(lo[0], 8));
      hi[0] = fmaxf(hi[0], shfl_xor(hi[0], 8));
    }
    const float delta = (hi[0] - lo[0]) / (float)kVMax;
    const float inv = rtn_inv(delta);
    const int g = (D == 256) ? ((cg >> 4) & 1) : 0;
    __syncthreads();  // every thread is past its last read of the tile
    if (tok_writer) {
      sc_st<SB>(stage + R::kVDelta, t_own * R::kGv + g, delta);
      sc_st<SB>(stage + R::kVLo, t_own * R::kGv + g, lo[0]);
      if (g == 0) sc_st<SB>(stage + R::kVR, t_own, r_own);
    }
    if (h_own == 0) sc_st<SB>(stage + R::kVS, chan_of(p_own), s_own / sqrt_d);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float l = __shfl_sync(0xffffffffu, lo[0], src_lane(i));
      const float iv = __shfl_sync(0xffffffffu, inv, src_lane(i));
      const float2 nl = f2(-l, -l), iv2 = f2(iv, iv);
      const int t = 8 * tg + i;
      if constexpr (VB == 2) {
        // channel 32 (cg >> 2) + 4 m + (cg & 3) of slot m: byte 8 (cg >> 2) + m
        // of the token row, bits 2 (cg & 3); the four lanes of a channel
        // quadruple fill eight bytes together
        uint32_t wl = 0, wh = 0;  // slot m's code in bits 8 (m % 4) of word m / 4
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 u = fma2(add2(y2[i][k], nl), iv2, f2(0.5f, 0.5f));
          if (k < 2) {
            wl = bfi(floor_bits(u.x), wl, 16 * k, 2);
            wl = bfi(floor_bits(u.y), wl, 16 * k + 8, 2);
          } else {
            wh = bfi(floor_bits(u.x), wh, 16 * (k - 2), 2);
            wh = bfi(floor_bits(u.y), wh, 16 * (k - 2) + 8, 2);
          }
        }
        unsigned long long w = (((unsigned long long)wh << 32) | wl) << (2 * (cg & 3));
        w |= __shfl_xor_sync(0xffffffffu, w, 1);
        w |= __shfl_xor_sync(0xffffffffu, w, 2);
        if ((i & 3) == (cg & 3))
          *reinterpret_cast<unsigned long long*>(stage + R::kVCodes + t * R::kVRow + 8 * (cg >> 2)) = w;
      } else if constexpr (VB == 3) {
        // 3-bit codes: the token row is a bit stream, channel c at bits 3 c.
        // Channel 32 (cg >> 2) + 4 m + q (q = cg & 3) of slot m sits at bit
        // 12 m + 3 q of the 96-bit run of its 32-channel block, which starts
        // at byte 12 (cg >> 2) of the row; the four lanes of a channel
        // quadruple assemble the run together (bits 0..63 and 64..95).
        const int q = cg & 3;
        unsigned long long lo64 = 0ull;
        uint32_t hi32 = 0u;
        auto place = [&](uint32_t c, int m) {
          const int b = 12 * m + 3 * q;
          if (b < 64) {
            lo64 |= (unsigned long long)c << b;
            if (b > 61) hi32 |= c >> (64 - b);  // the code straddles bit 64
          } else {
            hi32 |= c << (b - 64);
          }
        };
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 u = fma2(add2(y2[i][k], nl), iv2, f2(0.5f, 0.5f));
          place(floor_bits(u.x) & 7u, 2 * k);
          place(floor_bits(u.y) & 7u, 2 * k + 1);
        }
        lo64 |= __shfl_xor_sync(0xffffffffu, lo64, 1);
        hi32 |= __shfl_xor_sync(0xffffffffu, hi32, 1);
        lo64 |= __shfl_xor_sync(0xffffffffu, lo64, 2);
        hi32 |= __shfl_xor_sync(0xffffffffu, hi32, 2);
        if ((i & 3) == q) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(stage + R::kVCodes + t * R::kVRow + 12 * (cg >> 2));
          dst[0] = (uint32_t)lo64;
          dst[1] = (uint32_t)(lo64 >> 32);
          dst[2] = hi32;
        }
      } else {
        // 4-bit codes: channel 32 (cg >> 2) + 4 m + (cg & 3) sits in byte
        // 16 (cg >> 2) + 2 m + ((cg & 3) >> 1), nibble (cg & 3) & 1; the four
        // lanes of a channel quadruple fill sixteen bytes together
        const int sh = 8 * ((cg & 3) >> 1) + 4 * (cg & 1);
        uint32_t h4[4];  // slots 2q, 2q+1 in bits 0 and 16 of word q
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 u = fma2(add2(y2[i][k], nl), iv2, f2(0.5f, 0.5f));
          h4[k] = bfi(floor_bits(u.y), floor_bits(u.x) & 15u, 16, 4);
        }
        // bytes 0..7 (slots 0..3), 8..15 (slots 4..7)
        unsigned long long w0 = (((unsigned long long)h4[1] << 32) | h4[0]) << sh;
        unsigned long long w1 = (((unsigned long long)h4[3] << 32) | h4[2]) << sh;
        w0 |= __shfl_xor_sync(0xffffffffu, w0, 1);
        w1 |= __shfl_xor_sync(0xffffffffu, w1, 1);
        w0 |= __shfl_xor_sync(0xffffffffu, w0, 2);
        w1 |= __shfl_xor_sync(0xffffffffu, w1, 2);
        if ((i & 3) == (cg & 3)) {
          unsigned long long* dst =
              reinterpret_cast<unsigned long long*>(stage + R::kVCodes + t * R::kVRow + 16 * (cg >> 2));
          dst[0] = w0;
          dst[1] = w1;
        }
      }
    }
  }
  __syncthreads();

  // ---------------- copy the staged halves of the record out --------------
  uint8_t* rec = tiles + dst;
  const int a0 = is_v ? R::kVCodes : R::kKCodes;
  const int a1 = is_v ? R::kKDelta : R::kVCodes;
  const int b0 = is_v ? R::kVDelta : R::kKDelta;
  const int b1 = is_v ? R::kBytes : R::kVDelta;
  for (int o = a0 + 16 * tid; o < a1; o += 16 * C::NT)
    __stcs(reinterpret_cast<uint4*>(rec + o), *reinterpret_cast<const uint4*>(stage + o));
  for (int o = b0 + 16 * tid; o < b1; o += 16 * C::NT)
    __stcs(reinterpret_cast<uint4*>(rec + o), *reinterpret_cast<const uint4*>(stage + o));
}

template <int D, int SB, int VB>
cudaError_t launch_compress_d(int iters, const float* k_raw, const float* v_raw, int64_t row_stride,
                              int64_t n_rows, const int64_t* src_row0, uint8_t* tiles,
                              int64_t tiles_bytes, const int64_t* dst_record, int64_t n_units,
                              unsigned* err, cudaStream_t st) {
  using C = CC<D>;
  static bool configured[64] = {};  // the smem opt-in is set once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(compress_kernel<D, SB, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const int64_t blocks = 2 * n_units;
  compress_kernel<D, SB, VB><<<(unsigned)blocks, C::NT, C::SMEM, st>>>(
      k_raw, v_raw, row_stride, n_rows, src_row0, tiles, tiles_bytes, dst_record, iters, err);
  return cudaGetLastError();
}

template <int SB, int VB>
cudaError_t launch_compress_sb(int D, int iters, const float* k_raw, const float* v_raw,
                               int64_t row_stride, int64_t n_rows, const int64_t* src_row0,
                               uint8_t* tiles, int64_t tiles_bytes, const int64_t* dst_record,
                               int64_t n_units, unsigned* err, cudaStream_t st) {
  switch (D) {
    case 64: return launch_compress_d<64, SB, VB>(iters, k_raw, v_raw, row_stride, n_rows, src_row0, tiles, tiles_bytes, dst_record, n_units, err, st);
    case 128: return launch_compress_d<128, SB, VB>(iters, k_raw, v_raw, row_stride, n_rows, src_row0, tiles, tiles_bytes, dst_record, n_units, err, st);
    case 256: return launch_compress_d<256, SB, VB>(iters, k_raw, v_raw, row_stride, n_rows, src_row0, tiles, tiles_bytes, dst_record, n_units, err, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_compress(int D, int iters, int scale_bytes, int v_bits, const float* k_raw,
                            const float* v_raw, int64_t row_stride, int64_t n_rows,
                            const int64_t* src_row0, uint8_t* tiles, int64_t tiles_bytes,
                            const int64_t* dst_record, int64_t n_units, unsigned* err,
                            cudaStream_t st) {
  const int key = 10 * scale_bytes + v_bits;
  switch (key) {
    case 42: return launch_compress_sb<4, 2>(D, iters, k_raw, v_raw, row_stride, n_rows, src_row0, tiles, tiles_bytes, dst_record, n_units, err, st);
    case 22: return launch_compress_sb<2, 2>(D, iters, k_raw, v_raw, row_stride, n_rows, src_row0, tiles, tiles_bytes, dst_record, n_units, err, st);
    case 44: return launch_compress_sb<4, 4>(D, iters, k_raw, v_raw, row_stride, n_rows, src_row0, tiles, tiles_bytes, dst_record, n_units, err, st);
    case 24: return launch_compress_sb<2, 4>(D, iters, k_raw, v_raw, row_stride, n_rows, src_row0, tiles, tiles_bytes, dst_record, n_units, err, st);
    case 43: return launch_compress_sb<4, 3>(D, iters, k_raw, v_raw, row_stride, n_rows, src_row0, tiles, tiles_bytes, dst_record, n_units, err, st);
    case 23: return launch_compress_sb<2, 3>(D, iters, k_raw, v_raw, row_stride, n_rows, src_row0, tiles, tiles_bytes, dst_record, n_units, err, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvarn
