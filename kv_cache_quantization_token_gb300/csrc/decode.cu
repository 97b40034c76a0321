// decode.cu -- KVarN decode attention over the compressed cache on sm_103a.
//
// Split-tile design (SharpInference issue #433, item 2: a fixed worst-case
// grid over (head, tile range) with early exit, followed by an LSE combine;
// the deferred inverse WHT is applied after combining the rotated partials):
//
//   split kernel   grid (item, KV head, sequence), 4 warps per CTA. Items
//                  0..tile_items-1 own TPS consecutive packed tiles: the four
//                  warps share each tile, the scores and the value aggregate
//                  run as mma.sync m16n8k16 contractions whose A fragments
//                  are built straight from the packed codes. The remaining
//                  items own 4 chunks of FP32 window rows (raw rows,
//                  unrotated query), one per warp, staged by bulk copies.
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
// packed codes. Records are staged in shared memory with bulk async copies
// (cp.async.bulk, mbarrier completion); every wait is bounded.
#include <cuda_fp16.h>
#include <math.h>

#include "kvarn_common.cuh"

namespace kvarn {
namespace {

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
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up (returns false) instead of spinning forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (int i = 0; i < (1 << 22); ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
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

// exact small-integer to float: the code sits in the mantissa of 2^23
__device__ __forceinline__ float code_f(uint32_t c) {
  return __int_as_float((int)(c | 0x4B000000u)) - 8388608.0f;
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
//  scores  S[t][n] = sum_c A[t][c] B[c][n]   A = 1 + code/16 (exact in fp16),
//                                            B = the folded query, split hi+lo
//          sum_c wd_c code_tc = 16 (S - sum_c wd_c)
//  values  O[c][n] = sum_t A[c][t] B[t][n]   A = 1 + code/4, B = p r delta hi+lo
//          sum_t pd_t code_tc = 4 (O - sum_t pd_t)
// Columns n are (query head, hi/lo part) pairs, 8 per n-tile. Each B operand is
// scaled by a power of two per head (exact) so the fp16 parts stay in range.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// {fp16(1 + n_a/16), fp16(1 + n_b/16)} from byte `byte` of words wa, wb; the
// nibble is the low one when sh == 6 and the high one when sh == 2.
__device__ __forceinline__ uint32_t nib_pair(uint32_t wa, uint32_t wb, uint32_t sel, int sh) {
  return ((prmt(wa, wb, sel) << sh) & 0x03C003C0u) | 0x3C003C00u;
}
// {fp16(1 + c_a/4), fp16(1 + c_b/4)}: 2-bit fields at bit `2*f` of the selected bytes.
__device__ __forceinline__ uint32_t crumb_pair(uint32_t wa, uint32_t wb, uint32_t sel, int sh) {
  return ((prmt(wa, wb, sel) << sh) & 0x03000300u) | 0x3C003C00u;
}
// Packed fp16 pair of the hi (odd == false) or lo parts of (x0, x1): x = hi + lo
// to about 22 bits.
__device__ __forceinline__ uint32_t hilo_pair(float x0, float x1, bool lo_part) {
  const __half2 hi = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(hi);
  const __half2 r = lo_part ? __floats2half2_rn(x0 - hf.x, x1 - hf.y) : hi;
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ float pair_sum(uint32_t v) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
  return f.x + f.y;
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

template <int D, int GP, int TPS>
struct DC {
  static constexpr int NW = 4;                                  // warps per CTA
  static constexpr int RB = Rec<D>::kBytes;
  static constexpr int GV = Rec<D>::kGv;
  static constexpr int NT = GP > 4 ? 2 : 1;                     // n8-tiles of (head, part) columns
  static constexpr int NCB = D / 16;                            // 16-channel blocks
  static constexpr int CBA = NCB / NW;                          // channel blocks per warp (phase A)
  // window rows staged per warp (K and V rows of one chunk fit the record region)
  static constexpr int WCH0 = (TPS * RB) / (NW * 2 * D * 4);
  static constexpr int WCH = WCH0 >= 16 ? 16 : WCH0 >= 8 ? 8 : WCH0 >= 4 ? 4 : 2;
  static constexpr int OFF_SC = TPS * RB;                       // f32 [TPS][128][GP]
  static constexpr int OFF_QS = OFF_SC + TPS * 128 * GP * 4;    // f32 [D][GP] query
  // score shares [TPS][NW][128][GP]; reused for the value partials [NW][GP][D]
  static constexpr int PART = (TPS * NW * 128 * GP > NW * GP * D ? TPS * NW * 128 * GP : NW * GP * D) * 4;
  static constexpr int OFF_PART = OFF_QS + D * GP * 4;
  static constexpr int OFF_RED = OFF_PART + PART;               // f32 reduction scratch [NW][32]
  static constexpr int OFF_FLG = OFF_RED + NW * 32 * 4;         // int [TPS]
  static constexpr int OFF_BAR = (OFF_FLG + TPS * 4 + 7) / 8 * 8;
  static constexpr int SMEM = (OFF_BAR + TPS * 8 + 15) / 16 * 16;
  static_assert(D == 64 || D == 128 || D == 256, "head_dim");
  static_assert(CBA >= 1, "channel blocks per warp");
  static_assert(2 * WCH * D * 4 * NW <= TPS * RB, "window chunks must fit the record region");
  static_assert(NW * GP * D * 4 <= OFF_QS, "window partials fit below the query (over dead scores)");
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

template <int D, int GP, int TPS>
__global__ void __launch_bounds__(128)
decode_split_kernel(const float* __restrict__ q, const uint8_t* __restrict__ tiles,
                    const int64_t* __restrict__ tile_table, const int32_t* __restrict__ n_tiles,
                    const float* __restrict__ win_k, const float* __restrict__ win_v,
                    const int32_t* __restrict__ win_start, const int32_t* __restrict__ win_len,
                    int cap, int Hq, int Hkv, int G, int max_tiles, int items, int tile_items,
                    float scale, float* __restrict__ ws_ml, float* __restrict__ ws_acc) {
  using C = DC<D, GP, TPS>;
  using R = Rec<D>;
  constexpr int NW = C::NW, NT = C::NT, GV = C::GV;
  extern __shared__ __align__(16) unsigned char smem[];
  const int item = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = lane >> 2, q4 = lane & 3;  // mma fragment coordinates
  const bool is_win = item >= tile_items;
  const int64_t part = ((int64_t)b * Hq + (int64_t)kvh * G) * items + item;

  // slots of this item: packed tiles, or window chunks of WCH rows (one per warp)
  int nslot, wlen = 0, wstart = 0, wj0 = 0;
  if (!is_win) {
    const int nt = min(max(n_tiles[b], 0), max_tiles);
    nslot = min(max(nt - item * TPS, 0), TPS);
  } else {
    wlen = min(max(win_len[b], 0), cap);
    wstart = ((win_start[b] % cap) + cap) % cap;
    wj0 = C::WCH * NW * (item - tile_items);
    nslot = min(max((wlen - wj0 + C::WCH - 1) / C::WCH, 0), NW);
  }
  if (nslot == 0) {
    if (tid < G) {
      ws_ml[(part + (int64_t)tid * items) * 2 + 0] = kNegInf;
      ws_ml[(part + (int64_t)tid * items) * 2 + 1] = 0.f;
    }
    return;
  }
  float* sc = reinterpret_cast<float*>(smem + C::OFF_SC);
  float* qs = reinterpret_cast<float*>(smem + C::OFF_QS);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  int* okf = reinterpret_cast<int*>(smem + C::OFF_FLG);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

  if (is_win) {
    // ===================== window chunk: raw rows, SIMT =====================
    const int64_t head_base = ((int64_t)b * Hkv + kvh) * cap;
    if (tid == 0) {
      for (int kk = 0; kk < nslot; ++kk) mbar_init(&bar[kk], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      for (int kk = 0; kk < nslot; ++kk) {
        const int n = min(C::WCH, wlen - (wj0 + C::WCH * kk));
        mbar_expect_tx(&bar[kk], (uint32_t)(n * D * 4 * 2));
        unsigned char* dst = smem + kk * (2 * C::WCH * D * 4);
        for (int j = 0; j < n; ++j) {
          const int slot = (wstart + wj0 + C::WCH * kk + j) % cap;
          bulk_g2s(dst + j * D * 4, win_k + (head_base + slot) * D, D * 4, &bar[kk]);
          bulk_g2s(dst + (C::WCH + j) * D * 4, win_v + (head_base + slot) * D, D * 4, &bar[kk]);
        }
      }
    }
    for (int idx = tid; idx < D * GP; idx += 128) {
      const int c = idx / GP, h = idx % GP;
      qs[idx] = h < G ? scale * q[((int64_t)b * Hq + (int64_t)kvh * G + h) * D + c] : 0.f;
    }
    __syncthreads();
    const int k = warp;
    const bool have = k < nslot;
    bool ok = have && mbar_wait(&bar[k], 0);
    const float* Kw = reinterpret_cast<const float*>(smem + k * (2 * C::WCH * D * 4));
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
    float* vred = reinterpret_cast<float*>(smem);
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e)
#pragma unroll
      for (int h = 0; h < GP; ++h) vred[(warp * GP + h) * D + lane * E + e] = acc[e][h];
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += 128) {
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
  const int64_t* trow = tile_table + ((int64_t)b * Hkv + kvh) * max_tiles + item * TPS;
  if (tid == 0) {
    for (int kk = 0; kk < nslot; ++kk) mbar_init(&bar[kk], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int kk = 0; kk < nslot; ++kk) {
      const int64_t off = trow[kk];
      const bool aligned = (off & 15) == 0 && off >= 0;
      okf[kk] = aligned;
      if (aligned) {
        mbar_expect_tx(&bar[kk], C::RB);
        bulk_g2s(smem + kk * C::RB, tiles + off, C::RB, &bar[kk]);
      }
    }
  }
  // scores are kept in base-2 units (scale * log2 e folded into the query); the
  // item's (max, sum) pair is converted back to natural-log units when stored
  for (int h = warp; h < GP; h += NW)
    rotate_head_to_smem<D, GP>(q + ((int64_t)b * Hq + (int64_t)kvh * G + h) * D, h < G,
                               scale * kLog2eD, qs, h, lane);
  __syncthreads();
  int bad = 0;
  for (int kk = 0; kk < nslot; ++kk) bad |= !okf[kk];
  // the 8 lanes of one query head in a fragment: g8 in {2h', 2h'+1} (hi, lo), any q4
  const int hcol = g8 >> 1;      // head within an n-tile
  const bool is_hi = !(g8 & 1);  // this lane's B column holds the hi part

  // ---------------- phase A: warp w contracts channel blocks CBA*w.. ------
  // share[k][w][t][h]: this warp's share of the score of token t, head h
  float* share = reinterpret_cast<float*>(smem + C::OFF_PART);
  for (int k = 0; k < nslot; ++k) {
    const unsigned char* Rk = smem + k * C::RB;
    if (!bad && !mbar_wait(&bar[k], 0)) bad = 1;
    if (__any_sync(0xffffffffu, bad)) { bad = 1; continue; }
    const float* kS = reinterpret_cast<const float*>(Rk + R::kKS);
    const float* kD = reinterpret_cast<const float*>(Rk + R::kKDelta);
    const float* kL = reinterpret_cast<const float*>(Rk + R::kKLo);
    // B fragments of this warp's channels, in registers: channels 16cb + 2q4 + {0,1,8,9}
    float wdv[C::CBA][4][NT];
    float amax[NT], bsum[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) { amax[nt] = 0.f; bsum[nt] = 0.f; }
#pragma unroll
    for (int u = 0; u < C::CBA; ++u) {
      const int cbase = 16 * (C::CBA * warp + u) + 2 * q4;
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int c = cbase + 8 * hlf;
        const float2 s = *reinterpret_cast<const float2*>(kS + c);
        const float2 dd = *reinterpret_cast<const float2*>(kD + c);
        const float2 lo = *reinterpret_cast<const float2*>(kL + c);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float w0 = qs[c * GP + 4 * nt + hcol] * s.x;
          const float w1 = qs[(c + 1) * GP + 4 * nt + hcol] * s.y;
          wdv[u][2 * hlf][nt] = w0 * dd.x;
          wdv[u][2 * hlf + 1][nt] = w1 * dd.y;
          amax[nt] = fmaxf(amax[nt], fmaxf(fabsf(w0 * dd.x), fabsf(w1 * dd.y)));
          if (is_hi) bsum[nt] = fmaf(w1, lo.y, fmaf(w0, lo.x, bsum[nt]));
        }
      }
    }
    uint32_t bfr[C::CBA][NT][2];
    float sumwd[NT], inv[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int m = 1; m <= 4; m <<= 1) amax[nt] = fmaxf(amax[nt], __shfl_xor_sync(0xffffffffu, amax[nt], m));
      float sc2;
      pow2_scale(amax[nt], 16.0f, sc2, inv[nt]);
      float ssum = 0.f;
#pragma unroll
      for (int u = 0; u < C::CBA; ++u) {
        bfr[u][nt][0] = hilo_pair(wdv[u][0][nt] * sc2, wdv[u][1][nt] * sc2, !is_hi);
        bfr[u][nt][1] = hilo_pair(wdv[u][2][nt] * sc2, wdv[u][3][nt] * sc2, !is_hi);
        ssum += pair_sum(bfr[u][nt][0]) + pair_sum(bfr[u][nt][1]);
      }
#pragma unroll
      for (int m = 1; m <= 4; m <<= 1) {
        ssum += __shfl_xor_sync(0xffffffffu, ssum, m);
        bsum[nt] += __shfl_xor_sync(0xffffffffu, bsum[nt], m);
      }
      sumwd[nt] = ssum;
    }
    float acc[8][NT][4];
#pragma unroll
    for (int tb = 0; tb < 8; ++tb)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[tb][nt][e] = 0.f;
    const uint32_t sel = (uint32_t)(g8 >> 1) | ((uint32_t)((g8 >> 1) + 4) << 8);
    const int sh = (g8 & 1) ? 2 : 6;
#pragma unroll
    for (int u = 0; u < C::CBA; ++u) {
      const int r0 = 16 * (C::CBA * warp + u) + 2 * q4;
      const uint4* row0 = reinterpret_cast<const uint4*>(Rk + R::kKCodes + (r0 + 0) * 64);
      const uint4* row1 = reinterpret_cast<const uint4*>(Rk + R::kKCodes + (r0 + 1) * 64);
      const uint4* row8 = reinterpret_cast<const uint4*>(Rk + R::kKCodes + (r0 + 8) * 64);
      const uint4* row9 = reinterpret_cast<const uint4*>(Rk + R::kKCodes + (r0 + 9) * 64);
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {  // 16-byte quarter of the rows: token blocks 2qd, 2qd+1
        const uint4 w0 = row0[qd], w1 = row1[qd], w8 = row8[qd], w9 = row9[qd];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma16816(acc[2 * qd][nt], nib_pair(w0.x, w1.x, sel, sh), nib_pair(w0.y, w1.y, sel, sh),
                   nib_pair(w8.x, w9.x, sel, sh), nib_pair(w8.y, w9.y, sel, sh), bfr[u][nt][0],
                   bfr[u][nt][1]);
          mma16816(acc[2 * qd + 1][nt], nib_pair(w0.z, w1.z, sel, sh), nib_pair(w0.w, w1.w, sel, sh),
                   nib_pair(w8.z, w9.z, sel, sh), nib_pair(w8.w, w9.w, sel, sh), bfr[u][nt][0],
                   bfr[u][nt][1]);
        }
      }
    }
    // this warp's share: sum_c (wd code + w lo) over its channels = 16 (S - sum wd) 2^-e + bias
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = 4 * nt + q4;
      // lanes hold heads q4 of the accumulator columns; sum wd / bias of head h live in
      // the lanes whose fragment column is head h: fetch them from lane 8*(h%4)
      const float swd = __shfl_sync(0xffffffffu, sumwd[nt], 8 * q4);
      const float bia = __shfl_sync(0xffffffffu, bsum[nt], 8 * q4);
      const float iv = __shfl_sync(0xffffffffu, inv[nt], 8 * q4);
      if (h < GP) {
#pragma unroll
        for (int tb = 0; tb < 8; ++tb)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int t = 16 * tb + g8 + 8 * rr;
            const float S = acc[tb][nt][2 * rr] + acc[tb][nt][2 * rr + 1];
            share[((k * NW + warp) * 128 + t) * GP + h] = fmaf(S - swd, iv, bia);
          }
      }
    }
  }
  bad = __syncthreads_or(bad);

  // ---------------- scores and the item's softmax maximum ------------------
  float M[GP];
#pragma unroll
  for (int h = 0; h < GP; ++h) M[h] = kNegInf;
  if (!bad) {
    const int t = tid;
    for (int k = 0; k < nslot; ++k) {
      const float r = reinterpret_cast<const float*>(smem + k * C::RB + R::kKR)[t];
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        float z = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) z += share[((k * NW + w) * 128 + t) * GP + h];
        z *= r;
        sc[(k * 128 + t) * GP + h] = z;
        M[h] = fmaxf(M[h], z);
      }
    }
  }
  cta_max<GP, NW>(M, red, tid);  // its barriers also publish sc

  // ---------------- phase B: warp w aggregates tokens 32w .. 32w+31 --------
  // out_acc: this warp's share of acc_rot for channels 16cb + g8 (+8), head q4 (+4 nt)
  float out_acc[C::NCB][2][NT];
#pragma unroll
  for (int cb = 0; cb < C::NCB; ++cb)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) out_acc[cb][rr][nt] = 0.f;
  float lsum[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) lsum[nt] = 0.f;
  const uint32_t sel0 = (uint32_t)(g8 >> 2) | ((uint32_t)((g8 >> 2) + 4) << 8);
  const uint32_t sel1 = sel0 + 0x0202u;  // channel g8 + 8
  const int shc = 8 - 2 * (g8 & 3);
  for (int k = 0; k < nslot && !bad; ++k) {
    const unsigned char* Rk = smem + k * C::RB;
    const float* vR = reinterpret_cast<const float*>(Rk + R::kVR);
    const float* vD = reinterpret_cast<const float*>(Rk + R::kVDelta);
    const float* vL = reinterpret_cast<const float*>(Rk + R::kVLo);
    const float* vS = reinterpret_cast<const float*>(Rk + R::kVS);
    // B fragments: tokens 16tb + 2q4 + {0,1,8,9} of tb = 2w, 2w+1, column g8
    uint32_t bfr[GV][2][NT][2];
    float sumpd[GV][NT], Lw[GV][NT], invp[GV][NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = 4 * nt + hcol;
      const bool hv_ok = h < GP;
      const float Mh = M[hv_ok ? h : 0];
      float pdv[GV][2][4], pm[GV], ls[GV];
#pragma unroll
      for (int g = 0; g < GV; ++g) { pm[g] = 0.f; ls[g] = 0.f; }
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
          const int t = 16 * (2 * warp + j) + 2 * q4 + 8 * hlf;
          const float2 r = *reinterpret_cast<const float2*>(vR + t);
          const float p0 = hv_ok ? exp2f(sc[(k * 128 + t) * GP + h] - Mh) : 0.f;
          const float p1 = hv_ok ? exp2f(sc[(k * 128 + t + 1) * GP + h] - Mh) : 0.f;
          const float pv0 = p0 * r.x, pv1 = p1 * r.y;
          if (is_hi) lsum[nt] += p0 + p1;
#pragma unroll
          for (int g = 0; g < GV; ++g) {
            const float d0 = vD[t * GV + g], d1 = vD[(t + 1) * GV + g];
            pdv[g][j][2 * hlf] = pv0 * d0;
            pdv[g][j][2 * hlf + 1] = pv1 * d1;
            pm[g] = fmaxf(pm[g], fmaxf(fabsf(pv0 * d0), fabsf(pv1 * d1)));
            if (is_hi) ls[g] = fmaf(pv1, vL[(t + 1) * GV + g], fmaf(pv0, vL[t * GV + g], ls[g]));
          }
        }
#pragma unroll
      for (int g = 0; g < GV; ++g) {
#pragma unroll
        for (int m = 1; m <= 4; m <<= 1) pm[g] = fmaxf(pm[g], __shfl_xor_sync(0xffffffffu, pm[g], m));
        float sc2;
        pow2_scale(pm[g], 4.0f, sc2, invp[g][nt]);
        float ssum = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          bfr[g][j][nt][0] = hilo_pair(pdv[g][j][0] * sc2, pdv[g][j][1] * sc2, !is_hi);
          bfr[g][j][nt][1] = hilo_pair(pdv[g][j][2] * sc2, pdv[g][j][3] * sc2, !is_hi);
          ssum += pair_sum(bfr[g][j][nt][0]) + pair_sum(bfr[g][j][nt][1]);
        }
#pragma unroll
        for (int m = 1; m <= 4; m <<= 1) {
          ssum += __shfl_xor_sync(0xffffffffu, ssum, m);
          ls[g] += __shfl_xor_sync(0xffffffffu, ls[g], m);
        }
        sumpd[g][nt] = ssum;
        Lw[g][nt] = ls[g];
      }
    }
    // the accumulator column of lane (g8, q4) is head q4: fetch its scalars from lane 8*q4
    float swd_o[GV][NT], lw_o[GV][NT], iv_o[GV][NT];
#pragma unroll
    for (int g = 0; g < GV; ++g)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        swd_o[g][nt] = __shfl_sync(0xffffffffu, sumpd[g][nt], 8 * q4);
        lw_o[g][nt] = __shfl_sync(0xffffffffu, Lw[g][nt], 8 * q4);
        iv_o[g][nt] = __shfl_sync(0xffffffffu, invp[g][nt], 8 * q4);
      }
    constexpr int CH = C::NCB < 8 ? C::NCB : 8;  // channel blocks per accumulator pass
#pragma unroll
    for (int cb0 = 0; cb0 < C::NCB; cb0 += CH) {
      float o[CH][NT][4];
#pragma unroll
      for (int u = 0; u < CH; ++u)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[u][nt][e] = 0.f;
      const int g = (16 * cb0) / Rec<D>::kVGroup;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int t0 = 16 * (2 * warp + j) + 2 * q4;
        const unsigned char* v0 = Rk + R::kVCodes + (t0 + 0) * (D / 4) + 4 * cb0;
        const unsigned char* v1 = Rk + R::kVCodes + (t0 + 1) * (D / 4) + 4 * cb0;
        const unsigned char* v8 = Rk + R::kVCodes + (t0 + 8) * (D / 4) + 4 * cb0;
        const unsigned char* v9 = Rk + R::kVCodes + (t0 + 9) * (D / 4) + 4 * cb0;
#pragma unroll
        for (int u = 0; u < CH; u += 2) {
          const uint2 a0 = reinterpret_cast<const uint2*>(v0)[u / 2];
          const uint2 a1 = reinterpret_cast<const uint2*>(v1)[u / 2];
          const uint2 a8 = reinterpret_cast<const uint2*>(v8)[u / 2];
          const uint2 a9 = reinterpret_cast<const uint2*>(v9)[u / 2];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(o[u][nt], crumb_pair(a0.x, a1.x, sel0, shc), crumb_pair(a0.x, a1.x, sel1, shc),
                     crumb_pair(a8.x, a9.x, sel0, shc), crumb_pair(a8.x, a9.x, sel1, shc),
                     bfr[g][j][nt][0], bfr[g][j][nt][1]);
            mma16816(o[u + 1][nt], crumb_pair(a0.y, a1.y, sel0, shc), crumb_pair(a0.y, a1.y, sel1, shc),
                     crumb_pair(a8.y, a9.y, sel0, shc), crumb_pair(a8.y, a9.y, sel1, shc),
                     bfr[g][j][nt][0], bfr[g][j][nt][1]);
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (4 * nt + q4 < GP) {
#pragma unroll
          for (int u = 0; u < CH; ++u)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int cb = cb0 + u;
              const int c = 16 * cb + g8 + 8 * rr;
              const float O = o[u][nt][2 * rr] + o[u][nt][2 * rr + 1];
              out_acc[cb][rr][nt] = fmaf(vS[c], fmaf(O - swd_o[g][nt], iv_o[g][nt], lw_o[g][nt]),
                                         out_acc[cb][rr][nt]);
            }
        }
      }
    }
  }
  bad = __syncthreads_or(bad);
  if (bad)  // let every copy that was issued land before the CTA exits (bounded)
    for (int kk = 0; kk < nslot; ++kk)
      if (okf[kk]) mbar_wait(&bar[kk], 0);

  // ---------------- cross-warp sum of the value partials, softmax sum ------
  float L[GP];
#pragma unroll
  for (int h = 0; h < GP; ++h) L[h] = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // lsum of head 4nt + hcol: summed over the column's lanes (lo lanes hold 0), then
    // one lane per head adds it
#pragma unroll
    for (int m = 1; m <= 4; m <<= 1) lsum[nt] += __shfl_xor_sync(0xffffffffu, lsum[nt], m);
    const float v = (q4 == 0 && is_hi) ? lsum[nt] : 0.f;
#pragma unroll
    for (int h = 0; h < GP; ++h)
      if (h == 4 * nt + hcol) L[h] += v;
  }
  cta_sum<GP, NW>(L, red, tid);
  float* vred = reinterpret_cast<float*>(smem + C::OFF_PART);  // [NW][GP][D]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = 4 * nt + q4;
    if (h < GP) {
#pragma unroll
      for (int cb = 0; cb < C::NCB; ++cb)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
          vred[(warp * GP + h) * D + 16 * cb + g8 + 8 * rr] = out_acc[cb][rr][nt];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += 128) {
    const int h = idx / D, c = idx % D;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += vred[(w * GP + h) * D + c];
    ws_acc[(part + (int64_t)h * items) * D + c] = bad ? NAN : s;
  }
  if (tid < G) {
    float Mh = M[0], lh = L[0];
#pragma unroll
    for (int h = 1; h < GP; ++h)
      if (h == tid) { Mh = M[h]; lh = L[h]; }
    ws_ml[(part + (int64_t)tid * items) * 2 + 0] = bad ? NAN : Mh * kLn2D;
    ws_ml[(part + (int64_t)tid * items) * 2 + 1] = bad ? NAN : lh;
  }
}

// LSE combine: one CTA of D threads per (query head, sequence). The items'
// (max, sum) pairs are reduced cooperatively, their weights kept in shared
// memory, then each thread sums its channel over the items with independent,
// coalesced loads.
template <int D>
__global__ void __launch_bounds__(D)
decode_combine_kernel(const float* __restrict__ ws_ml, const float* __restrict__ ws_acc, int Hq,
                      int items, int tile_items, float* __restrict__ out) {
  constexpr int NW = D / 32;
  constexpr int CH = 1024;  // items per weight chunk in shared memory
  __shared__ float x[D];
  __shared__ float wgt[CH];
  __shared__ float redf[NW];
  __shared__ int redi[NW];
  const int hq = blockIdx.x, b = blockIdx.y, c = threadIdx.x, lane = c & 31, wid = c >> 5;
  const int64_t base = ((int64_t)b * Hq + hq) * items;
  float M = kNegInf;
  int poison = 0;
  for (int j = c; j < items; j += D) {
    const float lj = ws_ml[(base + j) * 2 + 1];
    if (!(lj >= 0.f)) poison = 1;
    if (lj > 0.f) M = fmaxf(M, ws_ml[(base + j) * 2]);
  }
  M = warp_max(M);
  poison = __any_sync(0xffffffffu, poison);
  if (lane == 0) { redf[wid] = M; redi[wid] = poison; }
  __syncthreads();
  M = redf[0];
  poison = redi[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) { M = fmaxf(M, redf[w]); poison |= redi[w]; }
  __syncthreads();
  float L = 0.f, arot = 0.f, awin = 0.f;
  for (int j0 = 0; j0 < items; j0 += CH) {
    const int n = min(CH, items - j0);
    for (int j = c; j < n; j += D) {
      const float lj = ws_ml[(base + j0 + j) * 2 + 1];
      const float w = lj > 0.f ? expf(ws_ml[(base + j0 + j) * 2] - M) : 0.f;
      wgt[j] = w;
      L = fmaf(lj > 0.f ? lj : 0.f, w, L);
    }
    __syncthreads();
    const float* a = ws_acc + (base + j0) * D + c;
#pragma unroll 8
    for (int j = 0; j < n; ++j) {
      const float w = wgt[j];
      if (w != 0.f) {
        const float v = a[(int64_t)j * D];
        if (j0 + j < tile_items) arot = fmaf(w, v, arot);
        else awin = fmaf(w, v, awin);
      }
    }
    __syncthreads();
  }
  L = warp_sum(L);
  if (lane == 0) redf[wid] = L;
  x[c] = arot;
  __syncthreads();
  L = redf[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) L += redf[w];
#pragma unroll
  for (int h = 1; h < D; h <<= 1) {
    const float v = x[c], o = x[c ^ h];
    __syncthreads();
    x[c] = (c & h) ? (o - v) : (v + o);
    __syncthreads();
  }
  float r = 0.f;
  if (L > 0.f) r = (x[c] * (1.0f / sqrtf((float)D)) + awin) / L;
  if (poison) r = NAN;
  out[((int64_t)b * Hq + hq) * D + c] = r;
}

template <int D, int GP, int TPS>
cudaError_t launch_split_t(const DecodePlan& p, const DecodeArgs& a, float* ws_ml, float* ws_acc,
                           cudaStream_t st) {
  using C = DC<D, GP, TPS>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(decode_split_kernel<D, GP, TPS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  dim3 grid(p.items, a.Hkv, a.B);
  decode_split_kernel<D, GP, TPS><<<grid, 128, C::SMEM, st>>>(
      a.q, a.tiles, a.tile_table, a.n_tiles, a.win_k, a.win_v, a.win_start, a.win_len,
      a.win_capacity, a.Hq, a.Hkv, a.Hq / a.Hkv, a.max_tiles, p.items, p.tile_items, a.scale, ws_ml,
      ws_acc);
  return cudaGetLastError();
}

template <int D, int GP>
cudaError_t launch_split_g(const DecodePlan& p, const DecodeArgs& a, float* ws_ml, float* ws_acc,
                           cudaStream_t st) {
  switch (p.tiles_per_item) {
    case 1: return launch_split_t<D, GP, 1>(p, a, ws_ml, ws_acc, st);
    case 2: return launch_split_t<D, GP, 2>(p, a, ws_ml, ws_acc, st);
    case 4: return launch_split_t<D, GP, 4>(p, a, ws_ml, ws_acc, st);
    default: return cudaErrorInvalidValue;
  }
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

}  // namespace

int decode_plan(int B, int Hq, int Hkv, int D, int max_tiles, int win_capacity, DecodePlan* p) {
  const int G = Hq / Hkv;
  p->g_pad = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8;
  const int cap = D >= 256 ? 2 : 4;  // tiles staged per CTA (shared memory)
  const int64_t total = (int64_t)B * Hkv * max_tiles;
  const int64_t target = 4LL * sm_count();
  int tps = (int)((total + target - 1) / (target > 0 ? target : 1));
  tps = tps <= 1 ? 1 : tps <= 2 ? 2 : 4;
  if (tps > cap) tps = cap;
  p->tiles_per_item = tps;
  p->tile_items = max_tiles > 0 ? (max_tiles + tps - 1) / tps : 0;
  // window rows per warp and chunks per item, as DC<D, GP, TPS>::WCH and its 4 warps
  const int rb = 112 * D + 1024 + 1024 * (D > 128 ? D / 128 : 1);
  const int w0 = (tps * rb) / (4 * 2 * D * 4);
  const int wch = w0 >= 16 ? 16 : w0 >= 8 ? 8 : w0 >= 4 ? 4 : 2;
  p->win_items = win_capacity > 0 ? (win_capacity + 4 * wch - 1) / (4 * wch) : 0;
  p->items = p->tile_items + p->win_items;
  const size_t parts = (size_t)B * Hq * p->items;
  const size_t ml = (parts * 2 * sizeof(float) + 255) / 256 * 256;
  p->ws_bytes = ml + parts * (size_t)D * sizeof(float);
  return 0;
}

cudaError_t launch_decode_split(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                cudaStream_t st) {
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

cudaError_t launch_decode_combine(const DecodePlan& p, int B, int Hq, int D, const void* ws,
                                  float* out, cudaStream_t st) {
  float *ml, *acc;
  ws_split(p, B, Hq, const_cast<void*>(ws), &ml, &acc);
  const dim3 grid(Hq, B);
  switch (D) {
    case 64: decode_combine_kernel<64><<<grid, 64, 0, st>>>(ml, acc, Hq, p.items, p.tile_items, out); break;
    case 128: decode_combine_kernel<128><<<grid, 128, 0, st>>>(ml, acc, Hq, p.items, p.tile_items, out); break;
    case 256: decode_combine_kernel<256><<<grid, 256, 0, st>>>(ml, acc, Hq, p.items, p.tile_items, out); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace kvarn
