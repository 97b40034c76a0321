// decode.cu -- KVarN decode attention over the compressed cache on sm_103a.
//
// Split-tile design (SharpInference issue #433, item 2: a fixed worst-case
// grid over (head, tile range) with early exit, followed by an LSE combine;
// the deferred inverse WHT is applied after combining the rotated partials):
//
//   split kernel   grid (item, KV head, sequence) of TPS warps per CTA. Items
//                  0..tile_items-1 own TPS consecutive packed tiles, one warp
//                  per tile; the remaining items own TPS chunks of 16 (8 at
//                  head_dim 256) FP32 window rows, one per warp, staged by
//                  bulk copies (raw rows, unrotated query).
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
#include <math.h>

#include "kvarn_common.cuh"

namespace kvarn {
namespace {

constexpr float kNegInf = -INFINITY;

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

template <int D, int GP, int TPS>
struct DC {
  static constexpr int RB = Rec<D>::kBytes;
  static constexpr int GV = Rec<D>::kGv;
  static constexpr int WCH = D >= 256 ? 8 : 16;  // window tokens per warp (K+V rows fit a slot)
  static constexpr int WK = (D > 128 * GV ? D : 128 * GV) * GP;  // floats of per-warp scratch
  static constexpr int OFF_SC = TPS * RB;                         // [TPS][128][GP] scores
  static constexpr int OFF_WK = OFF_SC + TPS * 128 * GP * 4;      // [TPS][WK]
  static constexpr int OFF_QS = OFF_WK + TPS * WK * 4;            // [D][GP]
  static constexpr int OFF_RED = OFF_QS + D * GP * 4;             // [2][TPS][GP]
  static constexpr int OFF_FLG = OFF_RED + 2 * TPS * GP * 4;      // int [TPS]
  static constexpr int OFF_BAR = (OFF_FLG + TPS * 4 + 7) / 8 * 8;
  static constexpr int SMEM = (OFF_BAR + TPS * 8 + 15) / 16 * 16;
  static_assert(GP * D * 4 <= RB, "value partials must fit in a record slot");
  static_assert(2 * WCH * D * 4 <= RB, "a window chunk must fit in a record slot");
};

template <int D, int GP, int TPS>
__global__ void __launch_bounds__(32 * TPS)
decode_split_kernel(const float* __restrict__ q, const uint8_t* __restrict__ tiles,
                    const int64_t* __restrict__ tile_table, const int32_t* __restrict__ n_tiles,
                    const float* __restrict__ win_k, const float* __restrict__ win_v,
                    const int32_t* __restrict__ win_start, const int32_t* __restrict__ win_len,
                    int cap, int Hq, int Hkv, int G, int max_tiles, int items, int tile_items,
                    float scale, float* __restrict__ ws_ml, float* __restrict__ ws_acc) {
  using C = DC<D, GP, TPS>;
  using R = Rec<D>;
  extern __shared__ __align__(16) unsigned char smem[];
  const int item = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool is_win = item >= tile_items;
  const int64_t part = ((int64_t)b * Hq + (int64_t)kvh * G) * items + item;

  // slots of this item: packed tiles, or 128-token chunks of the window
  int nslot, wlen = 0, wstart = 0, wj0 = 0;
  if (!is_win) {
    const int nt = min(max(n_tiles[b], 0), max_tiles);
    nslot = min(max(nt - item * TPS, 0), TPS);
  } else {
    wlen = min(max(win_len[b], 0), cap);
    wstart = ((win_start[b] % cap) + cap) % cap;
    wj0 = C::WCH * TPS * (item - tile_items);
    nslot = min(max((wlen - wj0 + C::WCH - 1) / C::WCH, 0), TPS);
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
  float* red_max = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* red_l = red_max + TPS * GP;
  int* okf = reinterpret_cast<int*>(smem + C::OFF_FLG);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

  const int k = warp;
  const bool have = k < nslot;
  bool ok = have;
  const int tw = lane & 15, cs = lane >> 4;
  float zr[4][GP];
  float mx[GP];
#pragma unroll
  for (int h = 0; h < GP; ++h) mx[h] = kNegInf;

  if (!is_win) {
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
    // the rotated, scaled query of every head of the GQA group
    for (int h = warp; h < GP; h += TPS)
      rotate_head_to_smem<D, GP>(q + ((int64_t)b * Hq + (int64_t)kvh * G + h) * D, h < G, scale,
                                 qs, h, lane);
    __syncthreads();
    ok = have && okf[k];
    if (ok) ok = mbar_wait(&bar[k], 0);
  } else {
    // window rows are raw FP32: stage each warp's chunk of WCH rows of K and V
    // (contiguous D-float rows of the ring) into its slot with bulk copies
    const int64_t head_base = ((int64_t)b * Hkv + kvh) * cap;
    if (tid == 0) {
      for (int kk = 0; kk < nslot; ++kk) mbar_init(&bar[kk], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      for (int kk = 0; kk < nslot; ++kk) {
        const int n = min(C::WCH, wlen - (wj0 + C::WCH * kk));
        okf[kk] = 1;
        mbar_expect_tx(&bar[kk], (uint32_t)(n * D * 4 * 2));
        unsigned char* dst = smem + kk * C::RB;
        for (int j = 0; j < n; ++j) {
          const int slot = (wstart + wj0 + C::WCH * kk + j) % cap;
          bulk_g2s(dst + j * D * 4, win_k + (head_base + slot) * D, D * 4, &bar[kk]);
          bulk_g2s(dst + (C::WCH + j) * D * 4, win_v + (head_base + slot) * D, D * 4, &bar[kk]);
        }
      }
    }
    // the unrotated, scaled query
    for (int idx = tid; idx < D * GP; idx += 32 * TPS) {
      const int c = idx / GP, h = idx % GP;
      qs[idx] = h < G ? scale * q[((int64_t)b * Hq + (int64_t)kvh * G + h) * D + c] : 0.f;
    }
    __syncthreads();
    if (ok) ok = mbar_wait(&bar[k], 0);
  }
  const unsigned char* Rk = smem + k * C::RB;
  const int wn = is_win ? min(C::WCH, wlen - (wj0 + C::WCH * k)) : 0;  // tokens in this warp's chunk
  // window chunk: lane owns channels lane*E .. lane*E+E-1; after the row
  // reduction it holds the score of token wtok(lane) (lanes >= WCH repeat)
  constexpr int E = D / 32;
  const int wtok = win_row_of_lane<C::WCH>(lane);
  float zw[GP];

  // ---------------- phase A: scores of this warp's slot -------------------
  if (ok && !is_win) {
    const float* kS = reinterpret_cast<const float*>(Rk + R::kKS);
    const float* kD = reinterpret_cast<const float*>(Rk + R::kKDelta);
    const float* kL = reinterpret_cast<const float*>(Rk + R::kKLo);
    const float* kR = reinterpret_cast<const float*>(Rk + R::kKR);
    float* wd = reinterpret_cast<float*>(smem + C::OFF_WK) + k * C::WK;  // [D][GP]
    float bias[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) bias[h] = 0.f;
    for (int c = lane; c < D; c += 32) {
      const float s = kS[c], d = kD[c], lo = kL[c];
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float w = qs[c * GP + h] * s;
        wd[c * GP + h] = w * d;
        bias[h] = fmaf(w, lo, bias[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < GP; ++h) bias[h] = warp_sum(bias[h]);
    __syncwarp();
    float acc[8][GP];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int h = 0; h < GP; ++h) acc[i][h] = 0.f;
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(Rk + R::kKCodes) + tw;
#pragma unroll 4
    for (int j = 0; j < D / 2; ++j) {
      const int c = cs + 2 * j;
      const uint32_t w = kc[c * (kTile / 8)];
      float wv[GP];
#pragma unroll
      for (int h = 0; h < GP; ++h) wv[h] = wd[c * GP + h];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float f = code_f((w >> (4 * i)) & 15u);
#pragma unroll
        for (int h = 0; h < GP; ++h) acc[i][h] = fmaf(wv[h], f, acc[i][h]);
      }
    }
    // lanes tw and tw+16 hold the two channel halves of the same 8 tokens
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float send = cs ? acc[j][h] : acc[j + 4][h];
        const float keep = cs ? acc[j + 4][h] : acc[j][h];
        acc[j][h] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
      }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = 8 * tw + 4 * cs + j;
      const float r = kR[t];
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float z = r * (acc[j][h] + bias[h]);
        zr[j][h] = z;
        mx[h] = fmaxf(mx[h], z);
      }
    }
  } else if (ok) {
    const float* Kw = reinterpret_cast<const float*>(Rk);
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      float qv[E];
#pragma unroll
      for (int e = 0; e < E; ++e) qv[e] = qs[(lane * E + e) * GP + h];
      float part[C::WCH];
#pragma unroll
      for (int j = 0; j < C::WCH; ++j) {
        float a = 0.f;
        if (j < wn) {
#pragma unroll
          for (int e = 0; e < E; ++e) a = fmaf(qv[e], Kw[j * D + lane * E + e], a);
        }
        part[j] = a;
      }
      zw[h] = warp_reduce_rows<C::WCH>(part, lane);
      if (wtok < wn) mx[h] = zw[h];
    }
  }
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    mx[h] = warp_max(mx[h]);
    if (lane == 0) red_max[k * GP + h] = mx[h];
  }
  __syncthreads();
  bool poison = false;
  for (int kk = 0; kk < nslot; ++kk) poison |= !okf[kk];
  float M[GP];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    M[h] = kNegInf;
    for (int kk = 0; kk < TPS; ++kk) M[h] = fmaxf(M[h], red_max[kk * GP + h]);
  }
  float l[GP];
#pragma unroll
  for (int h = 0; h < GP; ++h) l[h] = 0.f;
  if (ok && !is_win) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = 8 * tw + 4 * cs + j;
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float p = expf(zr[j][h] - M[h]);
        l[h] += p;
        sc[(k * 128 + t) * GP + h] = p;
      }
    }
  } else if (ok && lane < C::WCH) {
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      const float p = wtok < wn ? expf(zw[h] - M[h]) : 0.f;
      l[h] += p;
      sc[(k * 128 + wtok) * GP + h] = p;
    }
  }
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    l[h] = warp_sum(l[h]);
    if (lane == 0) red_l[k * GP + h] = ok ? l[h] : (have ? NAN : 0.f);
  }
  __syncwarp();

  // ---------------- phase B: value aggregate of this warp's slot ----------
  float* vred = reinterpret_cast<float*>(smem + k * C::RB);  // [GP][D] partial of slot k
  if (ok && !is_win) {
    const float* vR = reinterpret_cast<const float*>(Rk + R::kVR);
    const float* vD = reinterpret_cast<const float*>(Rk + R::kVDelta);
    const float* vL = reinterpret_cast<const float*>(Rk + R::kVLo);
    const float* vS = reinterpret_cast<const float*>(Rk + R::kVS);
    float* pd = reinterpret_cast<float*>(smem + C::OFF_WK) + k * C::WK;  // [GV][128][GP]
    constexpr int GV = C::GV;
    float Lg[GV][GP];
#pragma unroll
    for (int g = 0; g < GV; ++g)
#pragma unroll
      for (int h = 0; h < GP; ++h) Lg[g][h] = 0.f;
    for (int t = lane; t < 128; t += 32) {
      const float r = vR[t];
#pragma unroll
      for (int g = 0; g < GV; ++g) {
        const float d = vD[t * GV + g], lo = vL[t * GV + g];
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          const float pv = sc[(k * 128 + t) * GP + h] * r;
          pd[(g * 128 + t) * GP + h] = pv * d;
          Lg[g][h] = fmaf(pv, lo, Lg[g][h]);
        }
      }
    }
#pragma unroll
    for (int g = 0; g < GV; ++g)
#pragma unroll
      for (int h = 0; h < GP; ++h) Lg[g][h] = warp_sum(Lg[g][h]);
    __syncwarp();
    const unsigned char* vc = Rk + R::kVCodes;
    constexpr int COLS = D / 4;                        // bytes per token row
    constexpr int CPL = COLS >= 32 ? COLS / 32 : 1;    // byte columns per lane
    constexpr int TSTEP = COLS >= 32 ? 1 : 32 / COLS;  // lanes sharing a column (token split)
    const int jb0 = COLS >= 32 ? lane : (lane % COLS);
    const int tpar = COLS >= 32 ? 0 : (lane / COLS);
    float acc[CPL][4][GP];
#pragma unroll
    for (int u = 0; u < CPL; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int h = 0; h < GP; ++h) acc[u][e][h] = 0.f;
#pragma unroll 2
    for (int t = tpar; t < 128; t += TSTEP) {
#pragma unroll
      for (int u = 0; u < CPL; ++u) {
        const int jb = jb0 + 32 * u;
        const int g = (4 * jb) / Rec<D>::kVGroup;
        const uint32_t byte = vc[t * COLS + jb];
        float pv[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) pv[h] = pd[(g * 128 + t) * GP + h];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float f = code_f((byte >> (2 * e)) & 3u);
#pragma unroll
          for (int h = 0; h < GP; ++h) acc[u][e][h] = fmaf(pv[h], f, acc[u][e][h]);
        }
      }
    }
    if (TSTEP > 1) {
#pragma unroll
      for (int s = COLS; s < 32; s <<= 1)
#pragma unroll
        for (int u = 0; u < CPL; ++u)
#pragma unroll
          for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int h = 0; h < GP; ++h) acc[u][e][h] += __shfl_xor_sync(0xffffffffu, acc[u][e][h], s);
    }
    float sv[CPL][4];
#pragma unroll
    for (int u = 0; u < CPL; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) sv[u][e] = vS[4 * (jb0 + 32 * u) + e];
    __syncwarp();  // the record slot is reused for this tile's value partials
    if (tpar == 0) {
#pragma unroll
      for (int u = 0; u < CPL; ++u) {
        const int jb = jb0 + 32 * u;
        const int g = (4 * jb) / Rec<D>::kVGroup;
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int h = 0; h < GP; ++h) vred[h * D + 4 * jb + e] = sv[u][e] * (acc[u][e][h] + Lg[g][h]);
      }
    }
  } else if (ok) {
    const float* Vw = reinterpret_cast<const float*>(Rk) + C::WCH * D;
    float acc[E][GP];
#pragma unroll
    for (int e = 0; e < E; ++e)
#pragma unroll
      for (int h = 0; h < GP; ++h) acc[e][h] = 0.f;
    __syncwarp();  // the chunk's probabilities are in sc
#pragma unroll
    for (int j = 0; j < C::WCH; ++j) {
      if (j < wn) {
        float pv[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) pv[h] = sc[(k * 128 + j) * GP + h];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float x = Vw[j * D + lane * E + e];
#pragma unroll
          for (int h = 0; h < GP; ++h) acc[e][h] = fmaf(pv[h], x, acc[e][h]);
        }
      }
    }
    __syncwarp();  // the slot's rows are overwritten by the partials below
#pragma unroll
    for (int e = 0; e < E; ++e)
#pragma unroll
      for (int h = 0; h < GP; ++h) vred[h * D + lane * E + e] = acc[e][h];
  }
  __syncthreads();

  for (int idx = tid; idx < G * D; idx += 32 * TPS) {
    const int h = idx / D, c = idx % D;
    float s = 0.f;
    for (int kk = 0; kk < nslot; ++kk) s += reinterpret_cast<const float*>(smem + kk * C::RB)[h * D + c];
    ws_acc[(part + (int64_t)h * items) * D + c] = poison ? NAN : s;
  }
  if (tid < G) {
    float M0 = kNegInf, L0 = 0.f;
    for (int kk = 0; kk < TPS; ++kk) {
      M0 = fmaxf(M0, red_max[kk * GP + tid]);
      if (kk < nslot) L0 += red_l[kk * GP + tid];
    }
    ws_ml[(part + (int64_t)tid * items) * 2 + 0] = poison ? NAN : M0;
    ws_ml[(part + (int64_t)tid * items) * 2 + 1] = poison ? NAN : L0;
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
  decode_split_kernel<D, GP, TPS><<<grid, 32 * TPS, C::SMEM, st>>>(
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
  const int wch = D >= 256 ? 8 : 16;  // window tokens per warp, as in DC<>::WCH
  p->win_items = win_capacity > 0 ? (win_capacity + wch * tps - 1) / (wch * tps) : 0;
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
