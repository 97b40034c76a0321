/*
 * kvarn_oracle.c -- plain, slow, fp64 CPU oracle of the KVarN hot path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call this code:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Every step follows the method as the pages state it, in their order:
 *   SharpInference issue #180, "Algorithm (per 128-token tile)":
 *     step 1  Hadamard rotation along the channel dim (orthonormal)
 *     step 2  dual-axis "Sinkhorn" variance normalisation, log-space
 *             alternation of per-channel / per-token std normalisation
 *     step 3  asymmetric RTN: per-channel keys, per-token values, group 128
 *     step 4  scales folded at read time; preset k4v2_g128
 *   SharpInference PR #434, commit 82efc4f: 128-token tiles, channel-major K
 *     and token-major V packing, 2-bit bit packing.
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - H is the Sylvester-ordered Walsh-Hadamard matrix scaled by 1/sqrt(D),
 *     no random signs; Y_t = H X_t for every token row.
 *   - Sinkhorn: n rounds (n = 4 by default), channel step first, std is the
 *     population std about the mean; a step whose std is not larger than
 *     2^-20 times the RMS of the same group (a constant or empty group, or a
 *     NaN) is skipped, i.e. ln(sigma) := 0 for that group.
 *   - RTN: lo = min, hi = max, delta = (hi - lo) / (2^b - 1),
 *     code = clamp(floor((y - lo) / delta + 1/2), 0, 2^b - 1); every code is 0
 *     when delta == 0. The zero point is stored as the float offset lo.
 *   - V groups are min(D, 128) channels wide.
 *
 * Parity pins for each function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_T 128

static int orc_pow2_dim(int D) { return D >= 2 && D <= 4096 && (D & (D - 1)) == 0; }

/* Parity (0/1) of the number of set bits of x. */
static int orc_parity(unsigned x) {
  int p = 0;
  while (x) { p ^= 1; x &= x - 1; }
  return p;
}

/* ---------------------------------------------------------------------------
 * c1: Walsh-Hadamard rotation (issue #180, Algorithm step 1).
 * Entry (i, j) of the order-D Sylvester Hadamard matrix is (-1)^popcount(i&j);
 * dividing by sqrt(D) makes it orthonormal. Written as the plain matrix
 * product, O(D^2) per row, no fast transform.
 */
double orc_hadamard_entry(int i, int j, int D) {
  return (orc_parity((unsigned)(i & j)) ? -1.0 : 1.0) / sqrt((double)D);
}

/* y[r][i] = sum_j H[i][j] x[r][j] for r < rows. x and y may not alias. */
int orc_wht_rows(const double* x, double* y, int64_t rows, int D) {
  if (!orc_pow2_dim(D)) return -3;
  for (int64_t r = 0; r < rows; ++r) {
    const double* xr = x + r * D;
    double* yr = y + r * D;
    for (int i = 0; i < D; ++i) {
      double acc = 0.0;
      for (int j = 0; j < D; ++j) acc += orc_hadamard_entry(i, j, D) * xr[j];
      yr[i] = acc;
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * c2: dual-axis log-space Sinkhorn variance normalisation (issue #180,
 * Algorithm step 2; PR #434 commit 82efc4f).
 */

/* Population mean/std/RMS of z[0], z[stride], ..., n values. */
static void orc_moments(const double* z, int n, double* std_out, double* rms_out) {
  double mean = 0.0, ms = 0.0;
  for (int i = 0; i < n; ++i) { mean += z[i]; ms += z[i] * z[i]; }
  mean /= n;
  ms /= n;
  double var = 0.0;
  for (int i = 0; i < n; ++i) var += (z[i] - mean) * (z[i] - mean);
  var /= n;
  *std_out = sqrt(var);
  *rms_out = sqrt(ms);
}

/* The skip rule: a group's std only updates its log factor when it is larger
 * than 2^-20 times the group's RMS (NaN compares false and is skipped too). */
static int orc_sigma_usable(double sigma, double rms) {
  return sigma > ldexp(rms, -20);
}

/*
 * Y: [T][D] rotated rows of one tensor of one tile. Outputs:
 *   s[D] = exp(alpha), r[T] = exp(beta), yn[T][D] = Y * exp(-alpha_c - beta_t).
 * alpha and beta start at 0; each of the n rounds first updates alpha from the
 * per-channel std over tokens of the currently normalised values, then beta
 * from the per-token std over channels, each time adding ln(std).
 */
int orc_sinkhorn(const double* Y, int T, int D, int iters, double* s, double* r,
                 double* yn) {
  if (T <= 0 || D <= 0 || iters < 0) return -4;
  double* alpha = (double*)calloc((size_t)D, sizeof(double));
  double* beta = (double*)calloc((size_t)T, sizeof(double));
  double* z = (double*)malloc(sizeof(double) * (size_t)(T > D ? T : D));
  if (!alpha || !beta || !z) { free(alpha); free(beta); free(z); return -7; }
  for (int it = 0; it < iters; ++it) {
    /* per-channel step: std over the T tokens of channel c */
    for (int c = 0; c < D; ++c) {
      for (int t = 0; t < T; ++t) z[t] = Y[(int64_t)t * D + c] * exp(-alpha[c] - beta[t]);
      double sd, rms;
      orc_moments(z, T, &sd, &rms);
      if (orc_sigma_usable(sd, rms)) alpha[c] += log(sd);
    }
    /* per-token step: std over the D channels of token t */
    for (int t = 0; t < T; ++t) {
      for (int c = 0; c < D; ++c) z[c] = Y[(int64_t)t * D + c] * exp(-alpha[c] - beta[t]);
      double sd, rms;
      orc_moments(z, D, &sd, &rms);
      if (orc_sigma_usable(sd, rms)) beta[t] += log(sd);
    }
  }
  for (int c = 0; c < D; ++c) s[c] = exp(alpha[c]);
  for (int t = 0; t < T; ++t) r[t] = exp(beta[t]);
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < D; ++c)
      yn[(int64_t)t * D + c] = Y[(int64_t)t * D + c] * exp(-alpha[c] - beta[t]);
  free(alpha); free(beta); free(z);
  return 0;
}

/* ---------------------------------------------------------------------------
 * c3: asymmetric round-to-nearest of one group (issue #180, Algorithm step 3).
 * The n values are y[0], y[stride], ...; codes and the pre-rounding values
 * v = (y - lo) / delta are written with the same stride (vpre may be NULL).
 */
int orc_rtn_group(const double* y, int n, int64_t stride, int bits, double* delta_out,
                  double* lo_out, uint8_t* codes, double* vpre) {
  if (n <= 0 || bits < 1 || bits > 8) return -4;
  double lo = y[0], hi = y[0];
  for (int i = 1; i < n; ++i) {
    double v = y[(int64_t)i * stride];
    if (v < lo) lo = v;
    if (v > hi) hi = v;
  }
  const int qmax = (1 << bits) - 1;
  const double delta = (hi - lo) / qmax;
  for (int i = 0; i < n; ++i) {
    double v = 0.0;
    int code = 0;
    if (delta != 0.0) {
      v = (y[(int64_t)i * stride] - lo) / delta;
      code = (int)floor(v + 0.5);
      if (code < 0) code = 0;
      if (code > qmax) code = qmax;
    }
    codes[(int64_t)i * stride] = (uint8_t)code;
    if (vpre) vpre[(int64_t)i * stride] = v;
  }
  *delta_out = delta;
  *lo_out = lo;
  return 0;
}

/* ---------------------------------------------------------------------------
 * One tensor of one tile: rotate, normalise, quantise.
 *   x      : fp32 rows, x[t * row_stride + c], t < 128, c < D.
 *   per_channel != 0 (keys): one group per channel over the 128 tokens,
 *       k_bits; delta/lo have D entries.
 *   per_channel == 0 (values): one group per token and per min(D,128)-channel
 *       block; delta/lo have 128 * Gv entries, index t * Gv + g.
 * Outputs (fp64): s[D], r[128], delta, lo, codes u8 [128][D] (one code per
 * byte, unpacked), vpre [128][D] (pre-rounding values, may be NULL).
 */
int orc_quantize_tensor(const float* x, int64_t row_stride, int D, int iters, int per_channel,
                        int bits, double* s, double* r, double* delta, double* lo,
                        uint8_t* codes, double* vpre) {
  if (!orc_pow2_dim(D)) return -3;
  const int T = ORC_T;
  double* X = (double*)malloc(sizeof(double) * (size_t)T * D);
  double* Y = (double*)malloc(sizeof(double) * (size_t)T * D);
  double* YN = (double*)malloc(sizeof(double) * (size_t)T * D);
  if (!X || !Y || !YN) { free(X); free(Y); free(YN); return -7; }
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < D; ++c) X[(int64_t)t * D + c] = (double)x[(int64_t)t * row_stride + c];
  int rc = orc_wht_rows(X, Y, T, D);
  if (rc == 0) rc = orc_sinkhorn(Y, T, D, iters, s, r, YN);
  if (rc == 0) {
    if (per_channel) {
      for (int c = 0; c < D && rc == 0; ++c)
        rc = orc_rtn_group(YN + c, T, D, bits, &delta[c], &lo[c], codes + c,
                           vpre ? vpre + c : NULL);
    } else {
      const int gw = D < 128 ? D : 128;
      const int ng = D / gw;
      for (int t = 0; t < T && rc == 0; ++t)
        for (int g = 0; g < ng && rc == 0; ++g) {
          const int64_t o = (int64_t)t * D + (int64_t)g * gw;
          rc = orc_rtn_group(YN + o, gw, 1, bits, &delta[t * ng + g], &lo[t * ng + g],
                             codes + o, vpre ? vpre + o : NULL);
        }
    }
  }
  free(X); free(Y); free(YN);
  return rc;
}

/* ---------------------------------------------------------------------------
 * c4: packed record (layout of include/kvarn.h, restated here on purpose so
 * that the oracle does not include the library's header).
 * Scale fields are stored as IEEE binary32 (sw = 4 bytes, the default
 * layout) or as IEEE binary16 (sw = 2: the f16-scale layout that
 * SharpInference issue #433, item 3 names as a later saving). The codes are
 * the same in both: only the stored precision of the scales differs.
 */
typedef struct {
  int64_t bytes, k_codes, v_codes, k_delta, k_lo, k_s, k_r, v_delta, v_lo, v_r, v_s;
  int gv, sw, vb;
} orc_layout;

/* vb: V code width, 2 (the method's k4v2 preset), 3 or 4 (variants with
 * other value widths). Packing: the V codes of token t form a little-endian
 * bit stream of D * vb / 8 bytes starting at byte t * (D vb / 8); channel c
 * occupies stream bits vb*c .. vb*c + vb - 1, stream bit i being bit i % 8 of
 * byte i / 8. For vb = 2 and 4 that is the (c % (8/vb))-th vb-bit field of
 * byte c / (8/vb); a 3-bit code may straddle two bytes. */
static orc_layout orc_record_layout(int D, int sw, int vb) {
  orc_layout L;
  L.gv = D / (D < 128 ? D : 128);
  L.sw = sw;
  L.vb = vb;
  L.k_codes = 0;
  L.v_codes = L.k_codes + (int64_t)D * (ORC_T / 2);     /* 4-bit K codes        */
  L.k_delta = L.v_codes + (int64_t)ORC_T * (D * vb / 8); /* vb-bit V codes      */
  L.k_lo = L.k_delta + (int64_t)sw * D;
  L.k_s = L.k_lo + (int64_t)sw * D;
  L.k_r = L.k_s + (int64_t)sw * D;
  L.v_delta = L.k_r + (int64_t)sw * ORC_T;
  L.v_lo = L.v_delta + (int64_t)sw * ORC_T * L.gv;
  L.v_r = L.v_lo + (int64_t)sw * ORC_T * L.gv;
  L.v_s = L.v_r + (int64_t)sw * ORC_T;
  L.bytes = L.v_s + (int64_t)sw * D;
  return L;
}

static int orc_sw_ok(int sw) { return sw == 4 || sw == 2; }
static int orc_fmt_ok(int D, int sw, int vb) {
  return orc_pow2_dim(D) && D >= 4 && orc_sw_ok(sw) && (vb == 2 || vb == 3 || vb == 4) &&
         (D * vb) % 8 == 0;
}

int64_t orc_record_bytes_fmt(int D, int sw, int vb) {
  if (!orc_fmt_ok(D, sw, vb)) return -3;
  return orc_record_layout(D, sw, vb).bytes;
}
int64_t orc_record_bytes_sw(int D, int sw) { return orc_record_bytes_fmt(D, sw, 2); }
int64_t orc_record_bytes(int D) { return orc_record_bytes_sw(D, 4); }

/* IEEE binary16 encoding of v, rounded to nearest with ties to even, from the
 * format's definition: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits; subnormals have the quantum 2^-24, a normal number 2^E (1 + f/1024)
 * the quantum 2^(E-10); results above 65504 after rounding are infinite. */
uint16_t orc_f64_to_f16_bits(double v) {
  if (isnan(v)) return 0x7E00;
  const uint16_t sign = signbit(v) ? 0x8000 : 0;
  const double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7C00);
  int e;
  frexp(a, &e);                  /* a = m 2^e, m in [0.5, 1): a = 1.f 2^(e-1) */
  int E = e - 1;
  if (E < -14) E = -14;          /* subnormal range shares the quantum 2^-24 */
  const double ulp = ldexp(1.0, E - 10);
  const double n = rint(a / ulp); /* exact scaling; ties to even (default mode) */
  const double bits = ldexp((double)(E + 14), 10) + n;
  if (bits >= 31744.0) return (uint16_t)(sign | 0x7C00); /* 0x7C00: overflow */
  return (uint16_t)(sign | (uint16_t)bits);
}

double orc_f16_bits_to_f64(uint16_t h) {
  const int sign = h >> 15, ex = (h >> 10) & 0x1F, fr = h & 0x3FF;
  double m;
  if (ex == 0x1F) m = fr ? NAN : INFINITY;
  else if (ex == 0) m = ldexp((double)fr, -24);
  else m = ldexp(1024.0 + fr, ex - 25);
  return sign ? -m : m;
}

static void orc_put_scale(uint8_t* dst, double v, int sw) {
  if (sw == 4) {
    float f = (float)v;
    memcpy(dst, &f, 4);
  } else {
    const uint16_t h = orc_f64_to_f16_bits(v);
    memcpy(dst, &h, 2);
  }
}
static double orc_get_scale(const uint8_t* src, int sw) {
  if (sw == 4) {
    float f;
    memcpy(&f, src, 4);
    return (double)f;
  }
  uint16_t h;
  memcpy(&h, src, 2);
  return orc_f16_bits_to_f64(h);
}

/* Writes the record from unpacked codes ([128][D], one per byte) and fp64
 * scales, which are stored rounded to the layout's scale format. */
int orc_pack_record_fmt(int D, int sw, int vb, const uint8_t* k_codes, const uint8_t* v_codes,
                        const double* k_delta, const double* k_lo, const double* k_s,
                        const double* k_r, const double* v_delta, const double* v_lo,
                        const double* v_r, const double* v_s, uint8_t* rec) {
  if (!orc_fmt_ok(D, sw, vb)) return -3;
  const orc_layout L = orc_record_layout(D, sw, vb);
  const int64_t row = (int64_t)D * vb / 8;               /* V code bytes per token */
  memset(rec, 0, (size_t)L.bytes);
  for (int c = 0; c < D; ++c)
    for (int t = 0; t < ORC_T; ++t) {
      const uint8_t code = k_codes[(int64_t)t * D + c] & 0xF;
      rec[L.k_codes + (int64_t)c * (ORC_T / 2) + t / 2] |= (uint8_t)(code << (4 * (t & 1)));
    }
  for (int t = 0; t < ORC_T; ++t)
    for (int c = 0; c < D; ++c) {
      const unsigned code = v_codes[(int64_t)t * D + c] & ((1u << vb) - 1u);
      for (int b = 0; b < vb; ++b) {  /* one stream bit at a time */
        const int64_t bit = (int64_t)vb * c + b;
        rec[L.v_codes + t * row + bit / 8] |= (uint8_t)(((code >> b) & 1u) << (bit % 8));
      }
    }
  for (int c = 0; c < D; ++c) {
    orc_put_scale(rec + L.k_delta + (int64_t)sw * c, k_delta[c], sw);
    orc_put_scale(rec + L.k_lo + (int64_t)sw * c, k_lo[c], sw);
    orc_put_scale(rec + L.k_s + (int64_t)sw * c, k_s[c], sw);
    orc_put_scale(rec + L.v_s + (int64_t)sw * c, v_s[c], sw);
  }
  for (int t = 0; t < ORC_T; ++t) {
    orc_put_scale(rec + L.k_r + (int64_t)sw * t, k_r[t], sw);
    orc_put_scale(rec + L.v_r + (int64_t)sw * t, v_r[t], sw);
    for (int g = 0; g < L.gv; ++g) {
      orc_put_scale(rec + L.v_delta + (int64_t)sw * (t * L.gv + g), v_delta[t * L.gv + g], sw);
      orc_put_scale(rec + L.v_lo + (int64_t)sw * (t * L.gv + g), v_lo[t * L.gv + g], sw);
    }
  }
  return 0;
}
int orc_pack_record_sw(int D, int sw, const uint8_t* k_codes, const uint8_t* v_codes,
                       const double* k_delta, const double* k_lo, const double* k_s,
                       const double* k_r, const double* v_delta, const double* v_lo,
                       const double* v_r, const double* v_s, uint8_t* rec) {
  return orc_pack_record_fmt(D, sw, 2, k_codes, v_codes, k_delta, k_lo, k_s, k_r, v_delta, v_lo,
                             v_r, v_s, rec);
}
int orc_pack_record(int D, const uint8_t* k_codes, const uint8_t* v_codes,
                    const double* k_delta, const double* k_lo, const double* k_s,
                    const double* k_r, const double* v_delta, const double* v_lo,
                    const double* v_r, const double* v_s, uint8_t* rec) {
  return orc_pack_record_sw(D, 4, k_codes, v_codes, k_delta, k_lo, k_s, k_r, v_delta, v_lo,
                            v_r, v_s, rec);
}

/* Inverse of orc_pack_record_sw: unpacked codes and the stored scales. */
int orc_unpack_record_fmt(int D, int sw, int vb, const uint8_t* rec, uint8_t* k_codes,
                          uint8_t* v_codes, double* k_delta, double* k_lo, double* k_s,
                          double* k_r, double* v_delta, double* v_lo, double* v_r, double* v_s) {
  if (!orc_fmt_ok(D, sw, vb)) return -3;
  const orc_layout L = orc_record_layout(D, sw, vb);
  const int64_t row = (int64_t)D * vb / 8;
  for (int c = 0; c < D; ++c)
    for (int t = 0; t < ORC_T; ++t)
      k_codes[(int64_t)t * D + c] =
          (rec[L.k_codes + (int64_t)c * (ORC_T / 2) + t / 2] >> (4 * (t & 1))) & 0xF;
  for (int t = 0; t < ORC_T; ++t)
    for (int c = 0; c < D; ++c) {
      unsigned code = 0;
      for (int b = 0; b < vb; ++b) {
        const int64_t bit = (int64_t)vb * c + b;
        code |= (unsigned)((rec[L.v_codes + t * row + bit / 8] >> (bit % 8)) & 1u) << b;
      }
      v_codes[(int64_t)t * D + c] = (uint8_t)code;
    }
  for (int c = 0; c < D; ++c) {
    k_delta[c] = orc_get_scale(rec + L.k_delta + (int64_t)sw * c, sw);
    k_lo[c] = orc_get_scale(rec + L.k_lo + (int64_t)sw * c, sw);
    k_s[c] = orc_get_scale(rec + L.k_s + (int64_t)sw * c, sw);
    v_s[c] = orc_get_scale(rec + L.v_s + (int64_t)sw * c, sw);
  }
  for (int t = 0; t < ORC_T; ++t) {
    k_r[t] = orc_get_scale(rec + L.k_r + (int64_t)sw * t, sw);
    v_r[t] = orc_get_scale(rec + L.v_r + (int64_t)sw * t, sw);
    for (int g = 0; g < L.gv; ++g) {
      v_delta[t * L.gv + g] = orc_get_scale(rec + L.v_delta + (int64_t)sw * (t * L.gv + g), sw);
      v_lo[t * L.gv + g] = orc_get_scale(rec + L.v_lo + (int64_t)sw * (t * L.gv + g), sw);
    }
  }
  return 0;
}
int orc_unpack_record_sw(int D, int sw, const uint8_t* rec, uint8_t* k_codes, uint8_t* v_codes,
                         double* k_delta, double* k_lo, double* k_s, double* k_r,
                         double* v_delta, double* v_lo, double* v_r, double* v_s) {
  return orc_unpack_record_fmt(D, sw, 2, rec, k_codes, v_codes, k_delta, k_lo, k_s, k_r, v_delta,
                               v_lo, v_r, v_s);
}
int orc_unpack_record(int D, const uint8_t* rec, uint8_t* k_codes, uint8_t* v_codes,
                      double* k_delta, double* k_lo, double* k_s, double* k_r,
                      double* v_delta, double* v_lo, double* v_r, double* v_s) {
  return orc_unpack_record_sw(D, 4, rec, k_codes, v_codes, k_delta, k_lo, k_s, k_r, v_delta,
                              v_lo, v_r, v_s);
}

/* Full compression of one (tile, KV head) unit into a record; also returns the
 * fp64 scales and the pre-rounding values for the parity checks. The codes
 * come from the fp64 scales whatever the stored scale format. */
int orc_compress_unit_fmt(const float* k, const float* v, int64_t row_stride, int D, int iters,
                          int sw, int vb, uint8_t* rec, double* k_s, double* k_r, double* k_delta,
                          double* k_lo, double* k_vpre, double* v_s, double* v_r,
                          double* v_delta, double* v_lo, double* v_vpre) {
  if (!orc_fmt_ok(D, sw, vb)) return -3;
  uint8_t* kc = (uint8_t*)malloc((size_t)ORC_T * D);
  uint8_t* vc = (uint8_t*)malloc((size_t)ORC_T * D);
  if (!kc || !vc) { free(kc); free(vc); return -7; }
  int rc = orc_quantize_tensor(k, row_stride, D, iters, 1, 4, k_s, k_r, k_delta, k_lo, kc,
                               k_vpre);
  if (rc == 0)
    rc = orc_quantize_tensor(v, row_stride, D, iters, 0, vb, v_s, v_r, v_delta, v_lo, vc,
                             v_vpre);
  if (rc == 0)
    rc = orc_pack_record_fmt(D, sw, vb, kc, vc, k_delta, k_lo, k_s, k_r, v_delta, v_lo, v_r,
                             v_s, rec);
  free(kc); free(vc);
  return rc;
}
int orc_compress_unit_sw(const float* k, const float* v, int64_t row_stride, int D, int iters,
                         int sw, uint8_t* rec, double* k_s, double* k_r, double* k_delta,
                         double* k_lo, double* k_vpre, double* v_s, double* v_r,
                         double* v_delta, double* v_lo, double* v_vpre) {
  return orc_compress_unit_fmt(k, v, row_stride, D, iters, sw, 2, rec, k_s, k_r, k_delta, k_lo,
                               k_vpre, v_s, v_r, v_delta, v_lo, v_vpre);
}
int orc_compress_unit(const float* k, const float* v, int64_t row_stride, int D, int iters,
                      uint8_t* rec, double* k_s, double* k_r, double* k_delta, double* k_lo,
                      double* k_vpre, double* v_s, double* v_r, double* v_delta,
                      double* v_lo, double* v_vpre) {
  return orc_compress_unit_sw(k, v, row_stride, D, iters, 4, rec, k_s, k_r, k_delta, k_lo,
                              k_vpre, v_s, v_r, v_delta, v_lo, v_vpre);
}

/* ---------------------------------------------------------------------------
 * c5: reconstruction of one record to unrotated K and V rows ([128][D] each).
 * K~[t][c] = r_t s_c (delta_c code + lo_c), V~[t][c] = r_t s_c (delta_tg code
 * + lo_tg) with the stored scales, then each row is multiplied by H (H is its
 * own inverse).
 */
int orc_dequant_record_fmt(int D, int sw, int vb, const uint8_t* rec, double* k_out,
                           double* v_out) {
  if (!orc_fmt_ok(D, sw, vb)) return -3;
  const orc_layout L = orc_record_layout(D, sw, vb);
  const int T = ORC_T;
  uint8_t* kc = (uint8_t*)malloc((size_t)T * D);
  uint8_t* vc = (uint8_t*)malloc((size_t)T * D);
  double* buf = (double*)malloc(sizeof(double) * (size_t)(6 * D + 2 * T + 4 * T * L.gv));
  double* kt = (double*)malloc(sizeof(double) * (size_t)T * D);
  double* vt = (double*)malloc(sizeof(double) * (size_t)T * D);
  if (!kc || !vc || !buf || !kt || !vt) {
    free(kc); free(vc); free(buf); free(kt); free(vt);
    return -7;
  }
  double *k_delta = buf, *k_lo = k_delta + D, *k_s = k_lo + D, *v_s = k_s + D;
  double *k_r = v_s + D, *v_r = k_r + T, *v_delta = v_r + T, *v_lo = v_delta + T * L.gv;
  orc_unpack_record_fmt(D, sw, vb, rec, kc, vc, k_delta, k_lo, k_s, k_r, v_delta, v_lo, v_r, v_s);
  const int gw = D < 128 ? D : 128;
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < D; ++c) {
      const int64_t i = (int64_t)t * D + c;
      const int g = c / gw;
      kt[i] = k_r[t] * k_s[c] * (k_delta[c] * kc[i] + k_lo[c]);
      vt[i] = v_r[t] * v_s[c] * (v_delta[t * L.gv + g] * vc[i] + v_lo[t * L.gv + g]);
    }
  orc_wht_rows(kt, k_out, T, D);
  orc_wht_rows(vt, v_out, T, D);
  free(kc); free(vc); free(buf); free(kt); free(vt);
  return 0;
}
int orc_dequant_record_sw(int D, int sw, const uint8_t* rec, double* k_out, double* v_out) {
  return orc_dequant_record_fmt(D, sw, 2, rec, k_out, v_out);
}
int orc_dequant_record(int D, const uint8_t* rec, double* k_out, double* v_out) {
  return orc_dequant_record_sw(D, 4, rec, k_out, v_out);
}

/* ---------------------------------------------------------------------------
 * c7/c8: exact softmax attention of one query over n (key, value) rows:
 *   z_j = scale * q . k_j, p = softmax(z) with max subtraction,
 *   out = sum_j p_j v_j. n == 0 gives a zero output.
 */
int orc_attend(const double* q, const double* keys, const double* values, int64_t n, int D,
               double scale, double* out) {
  for (int c = 0; c < D; ++c) out[c] = 0.0;
  if (n <= 0) return 0;
  double* z = (double*)malloc(sizeof(double) * (size_t)n);
  if (!z) return -7;
  double zmax = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int c = 0; c < D; ++c) acc += q[c] * keys[j * D + c];
    z[j] = scale * acc;
    if (z[j] > zmax) zmax = z[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    z[j] = exp(z[j] - zmax);
    l += z[j];
  }
  for (int64_t j = 0; j < n; ++j) {
    const double p = z[j] / l;
    for (int c = 0; c < D; ++c) out[c] += p * values[j * D + c];
  }
  free(z);
  return 0;
}
