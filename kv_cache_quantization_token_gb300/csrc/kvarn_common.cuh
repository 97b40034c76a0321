// kvarn_common.cuh -- device-side helpers shared by the KVarN kernels.
//
// Nothing here is shared with the CPU oracle; the oracle restates the same
// layout from the method description on its own.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvarn.h"

namespace kvarn {

constexpr int kTile = KVARN_TILE_TOKENS;  // tokens per compressed tile

// Byte offsets of the record fields for head_dim D (same values as
// kvarn_layout(); kept as constexpr so the kernels index without a struct).
template <int D>
struct Rec {
  static constexpr int kGv = D / (D < 128 ? D : 128);     // V groups per token
  static constexpr int kVGroup = D < 128 ? D : 128;        // channels per V group
  static constexpr int kKCodes = 0;                        // u8 [D][64]
  static constexpr int kVCodes = kKCodes + D * (kTile / 2);  // u8 [128][D/4]
  static constexpr int kKDelta = kVCodes + kTile * (D / 4);
  static constexpr int kKLo = kKDelta + 4 * D;
  static constexpr int kKS = kKLo + 4 * D;
  static constexpr int kKR = kKS + 4 * D;
  static constexpr int kVDelta = kKR + 4 * kTile;
  static constexpr int kVLo = kVDelta + 4 * kTile * kGv;
  static constexpr int kVR = kVLo + 4 * kTile * kGv;
  static constexpr int kVS = kVR + 4 * kTile;
  static constexpr int kBytes = kVS + 4 * D;
  static_assert(kBytes == 112 * D + 1024 + 1024 * kGv, "record size");
};

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

// Current kvarn_set_launch_flags() value.
unsigned launch_flags();

// cudaLaunchKernelEx configuration honouring KVARN_LAUNCH_PDL.
struct LaunchCfg {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  LaunchCfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & KVARN_LAUNCH_PDL) ? 1 : 0;
  }
  LaunchCfg(const LaunchCfg&) = delete;
  LaunchCfg& operator=(const LaunchCfg&) = delete;
};

}  // namespace kvarn

// Launchers implemented in the .cu files; kvarn_abi.cu validates arguments
// and calls them. They return a cudaError_t from cudaGetLastError().
namespace kvarn {
cudaError_t launch_compress(int D, int iters, const float* k_raw, const float* v_raw,
                            int64_t row_stride, const int64_t* src_row0, uint8_t* tiles,
                            const int64_t* dst_record, int64_t n_units, cudaStream_t st);
cudaError_t launch_rotate(const float* q, float* q_rot, int64_t n_rows, int D, cudaStream_t st);
cudaError_t launch_append(const float* k_new, const float* v_new, int64_t n_new, float* win_k,
                          float* win_v, int win_capacity, const int32_t* win_start,
                          const int32_t* win_len, int n_seq, int n_kv_heads, int D,
                          cudaStream_t st);

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
};
int decode_plan(int B, int Hq, int Hkv, int D, int max_tiles, int win_capacity, DecodePlan* p);
cudaError_t launch_decode_split(const DecodePlan& p, const DecodeArgs& a, void* ws,
                                cudaStream_t st);
cudaError_t launch_decode_combine(const DecodePlan& p, int B, int Hq, int D, const void* ws,
                                  float* out, cudaStream_t st);
cudaError_t launch_prefill(const float* q, int C, int64_t pos0, const uint8_t* tiles,
                           const int64_t* tile_table, int table_stride, int n_tiles,
                           const float* win_k, const float* win_v, int win_start, int win_len,
                           int win_capacity, int Hq, int Hkv, int D, float softmax_scale,
                           void* ws, float* out, cudaStream_t st);
// 128-key blocks a prefill chunk sees (tiles, and tiles + window blocks), and
// the workspace bytes of one (block, KV head) image.
void prefill_blocks(int64_t pos0, int C, int n_tiles, int win_len, int* n_tblk, int* n_blk);
size_t prefill_block_bytes(int D);
cudaError_t launch_window_advance(int32_t* win_start, int32_t* win_len, int32_t* n_tiles,
                                  int n_seq, int d_len, int promote, int win_capacity,
                                  cudaStream_t st);
}  // namespace kvarn
