// kvarn_common.cuh -- device-side helpers shared by the KVarN kernels.
//
// Nothing here is shared with the CPU oracle; the oracle restates the same
// layout from the method description on its own.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvarn.h"

namespace kvarn {

constexpr int kTile = KVARN_TILE_TOKENS;  // tokens per compressed tile

// Byte offsets of the record fields for head_dim D with scale fields of SB
// bytes, 4 (fp32, layout version 1) or 2 (IEEE binary16, layout version 2),
// and VB-bit value codes, 2 (the k4v2 preset), 3 or 4 (the k4v3 and k4v4
// variants): each token's value codes are a little-endian bit stream, channel
// c at bits VB*c .. (a 3-bit code can straddle two bytes). Same values as
// kvarn_layout_ex(); kept as constexpr so the kernels index without a struct.
template <int D, int SB = 4, int VB = 2>
struct Rec {
  static_assert(SB == 4 || SB == 2, "scale field width");
  static_assert(VB == 2 || VB == 3 || VB == 4, "value code width");
  static constexpr int kSB = SB;
  static constexpr int kVB = VB;
  static constexpr int kGv = D / (D < 128 ? D : 128);     // V groups per token
  static constexpr int kVGroup = D < 128 ? D : 128;        // channels per V group
  static constexpr int kVRow = D * VB / 8;                 // V code bytes per token
  static constexpr int kKCodes = 0;                        // u8 [D][64]
  static constexpr int kVCodes = kKCodes + D * (kTile / 2);  // u8 [128][kVRow]
  static constexpr int kKDelta = kVCodes + kTile * kVRow;
  static constexpr int kKLo = kKDelta + SB * D;
  static constexpr int kKS = kKLo + SB * D;
  static constexpr int kKR = kKS + SB * D;
  static constexpr int kVDelta = kKR + SB * kTile;
  static constexpr int kVLo = kVDelta + SB * kTile * kGv;
  static constexpr int kVR = kVLo + SB * kTile * kGv;
  static constexpr int kVS = kVR + SB * kTile;
  static constexpr int kBytes = kVS + SB * D;
  // stride of a record slot in shared memory (slots start on 1024-byte swizzle atoms)
  static constexpr int kSlot = (kBytes + 1023) / 1024 * 1024;
  static_assert(kBytes == 64 * D + 16 * VB * D + SB * (4 * D + 256 + 256 * kGv), "record size");
  static_assert(kBytes % 128 == 0, "records on 128-byte lines");
};

// Scale fields of a record, fp32 (SB = 4) or binary16 (SB = 2), read as fp32:
// element i, the pair i, i+1 (i even) and the four i..i+3 (i a multiple of 4).
template <int SB>
__device__ __forceinline__ float sc_ld(const unsigned char* base, int i) {
  if constexpr (SB == 4) return reinterpret_cast<const float*>(base)[i];
  else return __half2float(reinterpret_cast<const __half*>(base)[i]);
}
template <int SB>
__device__ __forceinline__ float2 sc_ld2(const unsigned char* base, int i) {
  if constexpr (SB == 4) return *reinterpret_cast<const float2*>(base + 4 * i);
  else return __half22float2(*reinterpret_cast<const __half2*>(base + 2 * i));
}
template <int SB>
__device__ __forceinline__ float4 sc_ld4(const unsigned char* base, int i) {
  if constexpr (SB == 4) {
    return *reinterpret_cast<const float4*>(base + 4 * i);
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(base + 2 * i);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
}
// Stores v into scale field i, rounded to nearest (ties to even) for binary16.
template <int SB>
__device__ __forceinline__ void sc_st(unsigned char* base, int i, float v) {
  if constexpr (SB == 4) reinterpret_cast<float*>(base)[i] = v;
  else reinterpret_cast<__half*>(base)[i] = __float2half_rn(v);
}

__device__ __forceinline__ float shfl_xor(float v, int m) {
  return __shfl_xor_sync(0xffffffffu, v, m);
}

// Chan et al. pairwise merge of two (mean, M2) summaries with counts na, nb.
__device__ __forceinline__ void chan_merge(float& mean, float& m2, float na, float mean_b,
                                           float m2_b, float nb) {
  const float n = na + nb;
  const float d = mean_b - mean;
  mean = fmaf(d, nb / n, mean);
  m2 = m2 + m2_b + d * d * (na * nb / n);
}

// Programmatic dependent launch: wait for the previous grid on the stream
// (no-op when the kernel was launched without the attribute) and let the
// next grid be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Multiprocessor count of the current device (cached per device).
int sm_count();

// Device address of the library's error word on the current device (looked
// up once per device), or NULL if it cannot be found; kernels given NULL
// report nothing.
unsigned* device_error_word();

// cudaLaunchKernelEx configuration honouring the KVARN_LAUNCH_PDL bit of the
// call's launch flags.
struct LaunchCfg {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  LaunchCfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st, unsigned flags) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & KVARN_LAUNCH_PDL) ? 1 : 0;
  }
  LaunchCfg(const LaunchCfg&) = delete;
  LaunchCfg& operator=(const LaunchCfg&) = delete;
};

// ---------------------------------------------------------------------------
// Device-side failure reporting. A kernel that gives up (a wait that ran out
// of time, an input it refuses to touch) sets its KVARN_DEVERR_* bit in the
// library's error word and poisons the affected output with NaN; the word is
// read (and cleared) on the host with kvarn_get_device_error().
__device__ __forceinline__ void report(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Every wait on an mbarrier gives up after this long (a copy or a product of
// the same kernel completes within microseconds).
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;

__device__ __forceinline__ bool mbar_test_parity(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"((uint32_t)__cvta_generic_to_shared(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits until the phase of `bar` with the given parity has completed, for at
// most limit_ns (and a fixed number of polls, should the timer not move);
// returns false, after setting `bit` in *err, when it gives up. If `stop` is
// given, the wait also gives up (without reporting) once *stop is non-zero,
// and a wait that runs out sets *stop.
__device__ __forceinline__ bool mbar_wait_timed(uint64_t* bar, uint32_t parity, unsigned* err,
                                                unsigned bit, volatile int* stop = nullptr,
                                                uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_test_parity(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (int it = 0; it < (1 << 20); ++it) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_test_parity(bar, parity)) return true;
    if (stop && *stop) return false;
    if (global_ns() - t0 > limit_ns) break;
  }
  if (stop) *stop = 1;
  report(err, bit);
  return false;
}

}  // namespace kvarn

// Launchers implemented in the .cu files; kvarn_abi.cu validates arguments
// and calls them. They return a cudaError_t from cudaGetLastError().
namespace kvarn {
cudaError_t launch_compress(int D, int iters, int scale_bytes, int v_bits, const float* k_raw,
                            const float* v_raw, int64_t row_stride, int64_t n_rows,
                            const int64_t* src_row0, uint8_t* tiles, int64_t tiles_bytes,
                            const int64_t* dst_record, int64_t n_units, unsigned* err,
                            cudaStream_t st);
cudaError_t launch_rotate(const float* q, float* q_rot, int64_t n_rows, int D, cudaStream_t st);
cudaError_t launch_append(const float* k_new, const float* v_new, int64_t n_new, float* win_k,
                          float* win_v, int win_capacity, const int32_t* win_start,
                          const int32_t* win_len, int n_seq, int n_kv_heads, int D,
                          unsigned flags, unsigned* err, cudaStream_t st);
cudaError_t launch_selftest_wait(uint64_t timeout_ns, unsigned* err, cudaStream_t st);

struct DecodePlan {
  int tiles_per_round;  // packed tiles a split CTA works on at once (one per warp group)
  int rounds;           // tiles each warp group takes in turn (records double-buffered when > 1)
  int tiles_per_item;   // tiles_per_round * rounds: packed tiles handled by one split CTA
  int warps_per_tile;   // 2 or 4 (64 or 32 tokens per warp)
  int tile_items;       // ceil(max_tiles / tiles_per_item)
  int win_items;       // window items: ceil(win_capacity / window rows per item)
  int items;           // tile_items + win_items
  int g_pad;           // query heads per KV head rounded up to 1, 2, 4 or 8
  size_t ws_bytes;
};
struct DecodeArgs {
  const float* q;
  const uint8_t* tiles;
  const int64_t* tile_table;
  const int32_t* n_tiles;
  const float* win_k;
  const float* win_v;
  const int32_t* win_start;
  const int32_t* win_len;
  int win_capacity, B, Hq, Hkv, D, max_tiles;
  float scale;
  int scale_bytes;  // record scale fields: 4 (fp32) or 2 (binary16)
  int v_bits;       // value code width: 2 or 4
  int64_t tiles_bytes;  // size of the record pool
  unsigned flags;       // KVARN_LAUNCH_* bits of the call
  unsigned* err;        // device error word (may be NULL)
};
int decode_plan(int B, int Hq, int Hkv, int D, int max_tiles, int win_capacity, DecodePlan* p);
cudaError_t launch_decode_split(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                cudaStream_t st);
// the split kernels for records with fp32 (sb4) or binary16 (sb2) scale
// fields and 2-, 3- or 4-bit (v2, v3, v4) value codes, built as six
// translation units of decode.cu
cudaError_t launch_decode_split_sb4_v2(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st);
cudaError_t launch_decode_split_sb2_v2(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st);
cudaError_t launch_decode_split_sb4_v4(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st);
cudaError_t launch_decode_split_sb2_v4(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st);
cudaError_t launch_decode_split_sb4_v3(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st);
cudaError_t launch_decode_split_sb2_v3(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                       cudaStream_t st);
cudaError_t launch_decode_combine(const DecodePlan& p, int B, int Hq, int D, const void* ws,
                                  float* out, unsigned flags, cudaStream_t st);
cudaError_t launch_prefill(const float* q, int C, int64_t pos0, const uint8_t* tiles,
                           int64_t tiles_bytes, const int64_t* tile_table, int table_stride,
                           int n_tiles,
                           const float* win_k, const float* win_v, int win_start, int win_len,
                           int win_capacity, int Hq, int Hkv, int D, float softmax_scale,
                           int scale_bytes, int v_bits, void* ws, int ws_blocks, int cached_tiles,
                           float* out, unsigned* err, cudaStream_t st);
// 128-key blocks a prefill chunk sees (tiles, and tiles + window blocks), and
// the workspace bytes of one (block, KV head) image.
void prefill_blocks(int64_t pos0, int C, int n_tiles, int win_len, int* n_tblk, int* n_blk);
size_t prefill_block_bytes(int D);
cudaError_t launch_window_advance(int32_t* win_start, int32_t* win_len, int32_t* n_tiles,
                                  int n_seq, int d_len, int promote, int win_capacity,
                                  unsigned flags, cudaStream_t st);
}  // namespace kvarn
