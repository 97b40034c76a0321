// prefill.cu -- KVarN chunked-prefill attention on sm_103a tensor cores.
//
// Per chunk of C query positions of one sequence (SharpInference PR #434,
// commit 99c3773: a single streaming softmax over the compressed tiles plus
// the FP32 window with a deferred inverse WHT; issue #433 item 1: run the
// K-score and V-aggregate contractions on tensor cores), after the chunk's
// tokens were appended and whole tiles promoted:
//   out[i][h] = sum_j softmax_j(scale * q[i][h] . k_j) v_j  over keys j with
//   position(j) <= pos0 + i,
// tile k holding positions [128k, 128k+128) and window token w position
// 128 * n_tiles + w.
//
// Two kernels per chunk:
//   dequant   one CTA per (visible 128-key block, KV head): a packed tile is
//             dequantised (K~ = r_t s_c (delta code + lo), V~ likewise) or a
//             block of window rows rotated (H k, H v), into fp16 images of
//             K~ [key][channel] and V~^T [channel][key], each as a hi part and
//             a lo part (x - hi), in the 128-byte-swizzled K-major layout the
//             tensor cores read; staged in shared memory in two halves (K~,
//             then V~^T) and written to the workspace with bulk copies. Each
//             block is dequantised once per chunk, not once per query CTA.
//   attention one CTA (10 warps) per KV head and 128 score rows (the G query
//             heads of the GQA group times 128/G positions): 8 softmax warps,
//             one MMA warp, one copy warp, handing off through mbarriers.
//             The rotated, scaled query Q' stays in tensor memory (TMEM) as
//             fp16 hi + lo for the whole CTA, and both contractions take their
//             A operand from TMEM (the "TS" form of tcgen05.mma), so shared
//             memory only feeds the B operands:
//               S  = Q'h K~h + Q'l K~h + Q'h K~l      (fp32 accumulate, TMEM)
//               O += Ph V~h + Pl V~h + Ph V~l
//             A single fp16 rounding of any of the four operands costs 1e-3 to
//             1e-2 in the output (cancellation in q.k with rotated keys; in
//             P V the weights and the values each carry 2^-11 relative), so
//             each is carried as a pair whose sum holds about 22 bits and the
//             lo x lo product (2^-22) is dropped. Scores are double-buffered
//             in TMEM: S of block j+1 is formed while the softmax of block j
//             runs. Two threads per score row apply the causal mask and a
//             base-2 online softmax (the row maximum is exchanged between the
//             pair through shared memory; the reference maximum is only moved,
//             and O rescaled in TMEM, when a score exceeds it by more than 8);
//             P goes back into the TMEM columns its scores came from, as fp16
//             hi and lo, and the P V product reads it there. Row sums are
//             accumulated in fp32 by the softmax threads. At the end one
//             thread per row divides by the row sum and applies the one
//             inverse rotation (H is its own inverse).
// head_dim 256 has its own attention kernel (prefill_kernel_d256: 64-key
// sub-blocks, Q'l in shared memory, optional two-CTA cluster key split); the
// roles and the hand-offs are the same.
// Every wait is bounded; a CTA that gives up writes NaN rows, frees its TMEM
// and returns.
#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <math.h>

#include "kvarn_common.cuh"

namespace kvarn {
namespace {

namespace cg = cooperative_groups;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of element (row, k) of a K-major fp16 operand of `rows` rows in
// the 128-byte-swizzled canonical layout: 64-element K blocks, each `rows`
// x 128 bytes, 16-byte chunks XOR-swizzled by (row & 7).
__device__ __forceinline__ uint32_t sw_off(int row, int k, int rows) {
  return (uint32_t)((k >> 6) * rows * 128 + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) +
                    (k & 7) * 2);
}

// tcgen05 shared-memory matrix descriptor: K-major, SWIZZLE_128B, 8-row
// groups 1024 bytes apart (stride byte offset), version bits 46-48 = 0b001.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// The descriptor of the operand `bytes` further on (16-byte multiple): the
// start address field holds address / 16 in 14 bits, and every shared
// address here stays below 256 KB, so the sum never carries out of the field.
__device__ __forceinline__ uint64_t sdesc_add(uint64_t desc, uint32_t bytes) {
  return desc + (uint64_t)(bytes >> 4);
}
// Instruction descriptor, kind::f16: D f32, A and B f16, both K-major, M = 128.
template <int N>
__device__ __forceinline__ uint32_t idesc() {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t id,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(id), "r"(accumulate));
}
// The same product with the A operand (M = 128 rows, fp16 pairs packed two per
// 32-bit column, element 2k in the low half) read from tensor memory.
__device__ __forceinline__ void mma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t id,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(id), "r"(accumulate));
}
// The TS product that always accumulates into D.
__device__ __forceinline__ void mma_f16_ts_acc(uint32_t tmem_d, uint32_t tmem_a, uint64_t b,
                                               uint32_t id) {
  asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;\n" ::"r"(tmem_d),
               "r"(tmem_a), "l"(b), "r"(id));
}
// One lane of a converged warp (the same lane every time the warp is whole).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
               : "=r"(pred));
  return pred != 0;
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   su32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_init1(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(bar)) : "memory");
}
// Bounded waits (a fixed time limit; running out reports KVARN_DEVERR_WAIT).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned* err) {
  return mbar_wait_timed(bar, parity, err, KVARN_DEVERR_WAIT);
}
// The same wait, which also gives up once another thread of the CTA has
// raised `fail`; a wait that runs out raises it.
__device__ __forceinline__ bool mbar_wait_flag(uint64_t* bar, uint32_t parity, volatile int* fail,
                                               unsigned* err) {
  return mbar_wait_timed(bar, parity, err, KVARN_DEVERR_WAIT, fail);
}
// mbar_wait_flag for a whole warp, which leaves together: true only when
// every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait_flag(uint64_t* bar, uint32_t parity, volatile int* fail,
                                               unsigned* err) {
  return __all_sync(0xffffffffu, mbar_wait_flag(bar, parity, fail, err));
}
// The same for two barriers, one after the other.
__device__ __forceinline__ bool warp_wait_flag2(uint64_t* bar0, uint32_t parity0, uint64_t* bar1,
                                                uint32_t parity1, volatile int* fail, unsigned* err) {
  return warp_wait_flag(bar0, parity0, fail, err) && warp_wait_flag(bar1, parity1, fail, err);
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}
// TMEM lane field of the 32 lanes warp `w` may access (lanes 32 (w % 4) ..).
__device__ __forceinline__ uint32_t lane_base_of(int w) { return (uint32_t)((w & 3) * 32) << 16; }

// Bulk copy whose bytes count against a transaction count announced earlier.
__device__ __forceinline__ void bulk_copy_tx(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(bar))
      : "memory");
}

// Shared -> global bulk copy; the CTA waits until the source has been read.
__device__ __forceinline__ void bulk_store_wait(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(su32(ssrc)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// 32 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// 32 consecutive 32-bit TMEM columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_st32_nowait(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// x = hi + lo with hi, lo fp16: the pair carries about 22 significant bits.
__device__ __forceinline__ void split2(float x0, float x1, __half2& hi, __half2& lo) {
  hi = __floats2half2_rn(x0, x1);
  lo = __floats2half2_rn(x0 - __low2float(hi), x1 - __high2float(hi));
}

// The pair (x0, x1) as two fp16x2 words: hi = (x0, x1) rounded, lo = the
// rounded remainders; x0 in the low halves.
__device__ __forceinline__ void split2w(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  __half2 h, l;
  split2(x0, x1, h, l);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 2^x on the special-function unit (results below 2^-126 flush to zero).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// In-register orthonormal Walsh-Hadamard transform of N values (N a power of 2).
template <int N>
__device__ __forceinline__ void fwht_reg(float (&x)[N]) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1)
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (!(i & h)) {
        const float a = x[i], b = x[i | h];
        x[i] = a + b;
        x[i | h] = a - b;
      }
  const float s = 1.0f / sqrtf((float)N);
#pragma unroll
  for (int i = 0; i < N; ++i) x[i] *= s;
}

template <int D>
struct PC {
  static constexpr int OPB = 128 * D * 2;                // one fp16 operand image: 128 rows x D
  static constexpr int BLK = 4 * OPB;                    // workspace block: K~ hi, K~ lo, V~^T hi, V~^T lo
  // attention kernel shared memory (head_dim <= 128; head_dim 256 uses PA256)
  static constexpr int OFF_K = 0;                        // [2 buffers][K~ hi | K~ lo], [128 keys][D]
  static constexpr int OFF_V = 4 * OPB;                  // V~^T hi | lo, [D][128 keys]
  static constexpr int OFF_BAR = 6 * OPB;                // 10 mbarriers
  static constexpr int OFF_XM = OFF_BAR + 128;           // float [2][2][128]: row-max exchange
  static constexpr int OFF_XB = OFF_XM + 2 * 2 * 128 * 4; // int [2][8]: per-warp stop flags
  static constexpr int OFF_MISC = OFF_XB + 64;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;     // + slack to align the base to 1024
  // tensor memory columns: Q' hi and lo (fp16 pairs), S double buffer, O
  static constexpr int T_QH = 0, T_QL = D / 2, T_S = D, T_O = D + 256;
  static constexpr int TMEM_COLS = 512;
  // dequant kernel shared memory: the record (room for the fp32 layout of its
  // value width), then one half of the block image (K~ hi + lo, then V~^T hi
  // + lo in the same place) and a barrier
  static constexpr int DQ_OUT = 2 * OPB;
  template <int VB>
  struct DQ {
    static constexpr int OFF_OUT = Rec<D, 4, VB>::kSlot;
    static constexpr int OFF_BAR = OFF_OUT + DQ_OUT;
    static constexpr int SMEM = OFF_BAR + 64 + 1024;
  };
  static constexpr int NTHR = 256;                       // dequant: two threads per key row
  static constexpr int NTHR_ATT = 320;                   // attention: 8 softmax warps, MMA, loads
  static_assert(D == 64 || D == 128 || D == 256, "prefill head_dim");
  static_assert(OPB % 1024 == 0, "swizzled images on 1024-byte boundaries");
  static_assert(D == 256 || (T_O + D <= TMEM_COLS && SMEM <= 227 * 1024), "TMEM and shared memory");
};

struct PrefillArgs {
  const float* q;
  const uint8_t* tiles;
  const int64_t* tile_table;  // [Hkv][table_stride]
  const float* win_k;
  const float* win_v;
  uint8_t* ws;                // [Hkv][ws_stride] block images
  float* out;
  int64_t pos0;
  int C, Hq, Hkv, G, n_tiles, table_stride, win_start, win_len, win_cap;
  int n_tblk, n_blk;          // tiles, and tiles + window blocks, visible to the chunk
  int ws_stride;              // block images per KV head in ws (>= n_blk)
  int first_blk;              // first block whose image this call builds (earlier tiles' are kept)
  float qscale;               // softmax_scale * log2(e)
  int64_t tiles_bytes;        // size of the record pool
  unsigned* err;              // device error word (may be NULL)
};

// ---------------------------------------------------------------------------
// dequant: block j (tile j, or window block j - n_tblk) of KV head blockIdx.y
template <int D, int SB, int VB>
__global__ void __launch_bounds__(256, (D == 256) ? 1 : 2) prefill_dequant_kernel(const PrefillArgs a) {
  using P = PC<D>;
  using R = Rec<D, SB, VB>;  // scale fields fp32 (SB 4) or binary16 (SB 2); VB-bit values
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                       ~uintptr_t(1023));
  const unsigned char* rec = sm;
  unsigned char* sH = sm + P::template DQ<VB>::OFF_OUT;  // hi image (K~, then V~^T)
  unsigned char* sL = sH + P::OPB;                        // lo image
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + P::template DQ<VB>::OFF_BAR);
  const int j = a.first_blk + blockIdx.x, kvh = blockIdx.y;
  // the attention kernel may start now: it prepares its query rows and waits
  // for this grid before it reads an image
  pdl_trigger();
  uint8_t* gimg = a.ws + ((int64_t)kvh * a.ws_stride + j) * P::BLK;
  const int tid = threadIdx.x, row = tid & 127, half = tid >> 7;
  const bool is_tile = j < a.n_tblk;  // uniform over the CTA
  bool poison = false;
  if (is_tile) {
    const int64_t off = a.tile_table[(int64_t)kvh * a.table_stride + j];
    const bool aligned = (off & 15) == 0 && off >= 0 && off <= a.tiles_bytes - R::kBytes;
    if (tid == 0) {
      mbar_init1(bar);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      if (!aligned) report(a.err, KVARN_DEVERR_RECORD);
    }
    __syncthreads();
    if (aligned && tid == 0) bulk_load(sm, a.tiles + off, R::kBytes, bar);
    poison = !aligned || !mbar_wait_bounded(bar, 0, a.err);
    poison = __syncthreads_or(poison) != 0;
    // an unusable record: NaN keys make every score of this block NaN
    if (poison && aligned && tid == 0) mbar_wait_bounded(bar, 0, nullptr);  // let the copy land (bounded)
  }
  auto fill_nan = [&](unsigned char* dst, int bytes) {
    for (int o = tid * 16; o < bytes; o += 16 * P::NTHR)
      *reinterpret_cast<uint4*>(dst + o) = make_uint4(0x7E007E00u, 0x7E007E00u, 0x7E007E00u, 0x7E007E00u);
  };
  // the staged half goes out with one bulk copy (async proxy: fence the
  // generic writes first); the CTA waits until the copy has read it
  auto store_half = [&](uint8_t* dst) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) bulk_store_wait(dst, sH, 2 * P::OPB);
    __syncthreads();
  };
  // Tile images are written in blocks of 8 channels x 8 keys, one 16-byte
  // chunk (8 consecutive elements of a swizzled row) per store. Thread ->
  // block maps keep the 8 lanes of each store phase on 8 distinct chunk
  // positions of their rows: the K~ lanes differ in the channel group (rows
  // are keys), the V~^T lanes in the key group (rows are channels).
  constexpr int NCG8 = D / 8;  // 8-channel groups

  // window block: raw rows, rotated (K into K~, V into V~^T); rows past the
  // window's length are zero. Two threads per row (its two channel halves)
  // rotate their half in registers and meet for the butterfly over the top
  // channel bit through a padded fp32 staging area over the (unused) record
  // and image region, which the images then overwrite.
  const int wb = j - a.n_tblk;
  const int nkeys = is_tile ? 128 : min(128, a.win_len - 128 * wb);
  const int64_t slot = ((int64_t)a.win_start + 128 * wb + row) % a.win_cap;
  const int64_t rbase = ((int64_t)kvh * a.win_cap + slot) * D;
  constexpr int HD = D / 2, XS = D + 4;  // half a row; staging row stride (floats)
  static_assert(128 * XS * 4 <= P::template DQ<VB>::OFF_BAR, "window staging fits");
  auto win_rotate = [&](const float* base, float (&x)[HD]) {
    if (row < nkeys) {
      const float4* src = reinterpret_cast<const float4*>(base + rbase + half * HD);
#pragma unroll
      for (int c4 = 0; c4 < HD / 4; ++c4) {
        const float4 v = src[c4];
        x[4 * c4] = v.x; x[4 * c4 + 1] = v.y; x[4 * c4 + 2] = v.z; x[4 * c4 + 3] = v.w;
      }
#pragma unroll
      for (int h = 1; h < HD; h <<= 1)
#pragma unroll
        for (int i = 0; i < HD; ++i)
          if (!(i & h)) {
            const float u = x[i], w = x[i | h];
            x[i] = u + w;
            x[i | h] = u - w;
          }
    } else {
#pragma unroll
      for (int c = 0; c < HD; ++c) x[c] = 0.f;
    }
    float* xb = reinterpret_cast<float*>(sm);
#pragma unroll
    for (int c4 = 0; c4 < HD / 4; ++c4)
      *reinterpret_cast<float4*>(xb + row * XS + half * HD + 4 * c4) =
          make_float4(x[4 * c4], x[4 * c4 + 1], x[4 * c4 + 2], x[4 * c4 + 3]);
    __syncthreads();
    const float sc = 1.0f / sqrtf((float)D);
#pragma unroll
    for (int c4 = 0; c4 < HD / 4; ++c4) {
      const float4 y = *reinterpret_cast<const float4*>(xb + row * XS + (half ^ 1) * HD + 4 * c4);
      const float yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = 4 * c4 + e;
        x[c] = (half == 0 ? x[c] + yv[e] : yv[e] - x[c]) * sc;  // low half: a + b, high: a - b
      }
    }
    __syncthreads();  // the staging area is read before the images overwrite it
  };

  // ---------------- K~ hi / lo  [128 keys][D]
  if (is_tile) {
    if (poison) {
      fill_nan(sH, 2 * P::OPB);
    } else {
      const unsigned char* kS = rec + R::kKS;
      const unsigned char* kD = rec + R::kKDelta;
      const unsigned char* kL = rec + R::kKLo;
      const unsigned char* kR = rec + R::kKR;
      for (int blk = tid; blk < 16 * NCG8; blk += P::NTHR) {
        const int cg = blk % NCG8, kg = blk / NCG8;  // channels 8 cg .., keys 8 kg ..
        float dd[8], ll[8];
        uint32_t cw[8];  // nibble i of cw[e]: the code of key 8 kg + i, channel 8 cg + e
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 8 * cg + e;
          const float sc = sc_ld<SB>(kS, c);
          dd[e] = sc_ld<SB>(kD, c) * sc;
          ll[e] = sc_ld<SB>(kL, c) * sc;
          cw[e] = *reinterpret_cast<const uint32_t*>(rec + R::kKCodes + c * 64 + 4 * kg);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = 8 * kg + i;
          const float r = sc_ld<SB>(kR, t);
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const float v0 = r * fmaf(dd[2 * e2], (float)((cw[2 * e2] >> (4 * i)) & 15u), ll[2 * e2]);
            const float v1 =
                r * fmaf(dd[2 * e2 + 1], (float)((cw[2 * e2 + 1] >> (4 * i)) & 15u), ll[2 * e2 + 1]);
            split2w(v0, v1, hw[e2], lw[e2]);
          }
          const uint32_t o = sw_off(t, 8 * cg, 128);
          *reinterpret_cast<uint4*>(sH + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(sL + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
    }
  } else {
    float x[HD];
    win_rotate(a.win_k, x);
#pragma unroll
    for (int c8 = 0; c8 < HD / 8; ++c8) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) split2w(x[8 * c8 + 2 * e2], x[8 * c8 + 2 * e2 + 1], hw[e2], lw[e2]);
      const uint32_t o = sw_off(row, half * HD + 8 * c8, 128);
      *reinterpret_cast<uint4*>(sH + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(sL + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
  store_half(gimg);

  // ---------------- V~^T hi / lo  [D][128 keys]
  if (is_tile) {
    if (poison) {
      fill_nan(sH, 2 * P::OPB);
    } else {
      const unsigned char* vS = rec + R::kVS;
      const unsigned char* vR = rec + R::kVR;
      const unsigned char* vD = rec + R::kVDelta;
      const unsigned char* vL = rec + R::kVLo;
      constexpr uint32_t kMask = (1u << VB) - 1u;
      for (int blk = tid; blk < 16 * NCG8; blk += P::NTHR) {
        const int tg = blk % 16, cg = blk / 16;  // keys 8 tg .., channels 8 cg ..
        const int g = (8 * cg) / R::kVGroup;     // the channels' value group
        float sv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sv[e] = sc_ld<SB>(vS, 8 * cg + e);
        float vals[8][8];  // [channel e][key i]
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = 8 * tg + i;
          const float r = sc_ld<SB>(vR, t);
          const float d = sc_ld<SB>(vD, t * R::kGv + g) * r, lo = sc_ld<SB>(vL, t * R::kGv + g) * r;
          // the 8 codes of channels 8 cg .. form VB bytes of the row's bit stream
          const unsigned char* cb = rec + R::kVCodes + t * R::kVRow + VB * cg;
          uint32_t w = 0;
#pragma unroll
          for (int q = 0; q < VB; ++q) w |= (uint32_t)cb[q] << (8 * q);
#pragma unroll
          for (int e = 0; e < 8; ++e) vals[e][i] = sv[e] * fmaf(d, (float)((w >> (VB * e)) & kMask), lo);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2) split2w(vals[e][2 * i2], vals[e][2 * i2 + 1], hw[i2], lw[i2]);
          const uint32_t o = sw_off(8 * cg + e, 8 * tg, D);
          *reinterpret_cast<uint4*>(sH + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(sL + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
    }
  } else {  // V row -> column `row` of V~^T (this thread's channel half)
    float x[HD];
    win_rotate(a.win_v, x);
#pragma unroll
    for (int c = 0; c < HD; ++c) {
      const __half h = __float2half_rn(x[c]);
      const uint32_t o = sw_off(half * HD + c, row, D);
      *reinterpret_cast<__half*>(sH + o) = h;
      *reinterpret_cast<__half*>(sL + o) = __float2half_rn(x[c] - __half2float(h));
    }
  }
  store_half(gimg + 2 * P::OPB);
}

// Key blocks visible to some row of a CTA whose query positions span
// [pmin, pmax]: tiles, then 128-token window blocks (a CTA that sees a window
// block sees every tile).
struct Visible {
  int n_tile_blk, n_blk;
};
__device__ __forceinline__ Visible visible_blocks(const PrefillArgs& a, int64_t pmax) {
  const int64_t win_pos0 = 128LL * a.n_tiles;
  int n_tile_blk = a.n_tiles;
  if (n_tile_blk > 0 && 128LL * (n_tile_blk - 1) > pmax) n_tile_blk = (int)(pmax / 128) + 1;
  n_tile_blk = min(n_tile_blk, a.n_tiles);
  int n_win_blk = 0;
  for (int w = 0; 128 * w < a.win_len; ++w)
    if (win_pos0 + 128 * w <= pmax) n_win_blk = w + 1;
  return Visible{n_tile_blk, n_tile_blk + n_win_blk};
}

// Row maximum of a score row split over two threads (warps w and w + 4, the
// same TMEM lanes): each publishes its half's maximum and reads the other's
// after a barrier of the two warps, and the pair agrees on whether to go on:
// false when either warp gave up (`bad` is uniform over a warp). Slots
// alternate with the block parity, so a thread's next write never lands
// before its partner has read this one.
__device__ __forceinline__ bool pair_max(float mloc, bool bad, float* xm, int* xb, int par, int half,
                                         int row, int warp, float& mblk) {
  xm[(par * 2 + half) * 128 + row] = mloc;
  if ((threadIdx.x & 31) == 0) xb[par * 8 + warp] = bad ? 1 : 0;
  asm volatile("bar.sync %0, 64;" ::"r"(2 + (warp & 3)) : "memory");
  mblk = fmaxf(mloc, xm[(par * 2 + (half ^ 1)) * 128 + row]);
  return !bad && xb[par * 8 + (warp ^ 4)] == 0;
}

// ---------------------------------------------------------------------------
// attention over the block images of the chunk (head_dim 64 or 128)
//
// Warp roles: warps 0-7 run the softmax (two threads per score row) and the
// epilogue, warp 8 issues the tcgen05 MMAs (one elected lane), warp 9 the
// bulk copies (one thread). K~ is double-buffered in shared memory, V~^T
// single but in two 64-key halves with barriers of their own: PV(j) commits
// after its first half, and the first half of V~^T(j+1) streams in while the
// second half of PV(j) runs. S is double-buffered in TMEM. The tensor pipe
// runs, in order, S(0), S(1), PV(0), S(2), PV(1), ...; S(j+2) overwrites the
// TMEM columns that held P(j) only after PV(j), which the pipe completes
// first.
template <int D>
__global__ void __launch_bounds__(320, 1) prefill_kernel(const PrefillArgs a) {
  using P = PC<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                       ~uintptr_t(1023));
  unsigned char* sK = sm + P::OFF_K;
  unsigned char* sV = sm + P::OFF_V;
  uint64_t* bar_k = reinterpret_cast<uint64_t*>(sm + P::OFF_BAR);  // [2] K~ of block j in buffer j & 1
  uint64_t* bar_v = bar_k + 2;     // [2] key half h of V~^T(j) landed
  uint64_t* bar_s = bar_k + 4;     // [2] S(j) complete: scores ready, K~ buffer j & 1 free
  uint64_t* bar_o = bar_k + 6;     // PV(j) complete: V~^T free, O current
  uint64_t* bar_vh = bar_k + 7;    // the first half of PV(j) complete: V~^T half 0 free
  // [2] P(j) in TMEM and O rescaled: one arrival per softmax warp, on the
  // barrier of the block's parity (a warp may run one block ahead of the
  // others; its arrival must not count toward the block before)
  uint64_t* bar_p = bar_k + 8;
  float* xm = reinterpret_cast<float*>(sm + P::OFF_XM);
  int* xb = reinterpret_cast<int*>(sm + P::OFF_XB);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + P::OFF_MISC);
  volatile int* fail = reinterpret_cast<volatile int*>(sm + P::OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // score row of a softmax thread and its half of the key block (TMEM lanes of
  // warp w are 32 (w % 4) .. +31, so rows and TMEM lanes agree)
  const int row = tid & 127, half = (tid >> 7) & 1;
  const int kvh = blockIdx.y;
  const int ppc = 128 / a.G;                 // positions per CTA
  const int i0 = blockIdx.x * ppc;           // first chunk row of this CTA
  // score row `row` <-> (head g = row / ppc, chunk position i0 + row % ppc)
  const int my_g = row / ppc, my_i = i0 + row % ppc;
  const bool my_valid = my_i < a.C && my_g < a.G;
  const int64_t my_pos = a.pos0 + my_i;
  const int64_t pmax = a.pos0 + min(a.C, i0 + ppc) - 1;  // largest query position of the CTA
  const int64_t pmin = a.pos0 + i0;                       // smallest
  const int hq = kvh * a.G + min(my_g, a.G - 1);
  const int64_t win_pos0 = 128LL * a.n_tiles;
  const Visible vis_blk = visible_blocks(a, pmax);
  const int n_tile_blk = vis_blk.n_tile_blk, n_blk = vis_blk.n_blk;
  auto image = [&](int jj) -> const uint8_t* {  // workspace image of this CTA's block jj
    const int widx = jj < n_tile_blk ? jj : a.n_tblk + (jj - n_tile_blk);
    return a.ws + ((int64_t)kvh * a.ws_stride + widx) * P::BLK;
  };

  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init1(bar_k + i);
    for (int i = 0; i < 2; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(su32(bar_p + i)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *fail = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(tmem_slot)),
                 "r"(P::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_o = tmem + P::T_O;
  const uint32_t lb = lane_base_of(warp);

  // the first copies go out while the query rows are prepared
  int nk[2] = {0, 0}, nv[2] = {0, 0};  // copies issued per barrier (loader thread)
  auto load_k = [&](int jj) {
    const int b = jj & 1;
    bulk_load(sK + b * 2 * P::OPB, image(jj), 2 * P::OPB, bar_k + b);
    ++nk[b];
  };
  // keys 64 h .. 64 h + 63 of V~^T hi and lo: the h-th 64-key block of each
  constexpr uint32_t kVHalf = D * 128;
  auto load_v = [&](int jj, int h) {
    const uint8_t* src = image(jj) + 2 * P::OPB + h * kVHalf;
    mbar_expect_tx(bar_v + h, 2 * kVHalf);
    bulk_copy_tx(sV + h * kVHalf, src, kVHalf, bar_v + h);
    bulk_copy_tx(sV + P::OPB + h * kVHalf, src + P::OPB, kVHalf, bar_v + h);
    ++nv[h];
  };
  if (warp == 9 && lane == 0 && n_blk > 0) {
    pdl_wait();  // the images of this call's dequantisation grid are complete
    load_k(0);
    if (n_blk > 1) load_k(1);
    load_v(0, 0);
    load_v(0, 1);
  }
  // Q' row into TMEM: rotate, scale, fp16 hi + lo (one thread per row)
  if (tid < 128) {
    float x[D];
    if (my_valid) {
      const float4* src = reinterpret_cast<const float4*>(a.q + ((int64_t)my_i * a.Hq + hq) * D);
#pragma unroll
      for (int c4 = 0; c4 < D / 4; ++c4) {
        const float4 v = src[c4];
        x[4 * c4] = v.x; x[4 * c4 + 1] = v.y; x[4 * c4 + 2] = v.z; x[4 * c4 + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < D; ++c) x[c] = 0.f;
    }
    fwht_reg<D>(x);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 64) {
      uint32_t hw[32], lw[32];
#pragma unroll
      for (int e = 0; e < 32; ++e)
        split2w(x[c0 + 2 * e] * a.qscale, x[c0 + 2 * e + 1] * a.qscale, hw[e], lw[e]);
      tmem_st32_nowait(tmem + lb + P::T_QH + c0 / 2, hw);
      tmem_st32_nowait(tmem + lb + P::T_QL + c0 / 2, lw);
    }
    tmem_wait_st();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  float m_ref = -INFINITY, l_part = 0.f;  // softmax threads: reference max, half-row sum
  if (warp == 9) {
    // ---------------- loader: block images into shared memory
    if (lane == 0 && n_blk > 0) {
      // completion order of the tensor pipe: S(j) before PV(j)
      for (int j = 0; j < n_blk; ++j) {
        if (j + 2 < n_blk) {
          if (!mbar_wait_flag(bar_s + (j & 1), (uint32_t)(j >> 1) & 1u, fail, a.err)) break;
          load_k(j + 2);
        }
        if (j + 1 < n_blk) {
          if (!mbar_wait_flag(bar_vh, (uint32_t)j & 1u, fail, a.err)) break;
          load_v(j + 1, 0);
          if (!mbar_wait_flag(bar_o, (uint32_t)j & 1u, fail, a.err)) break;
          load_v(j + 1, 1);
        }
      }
      // every copy issued has landed before the CTA can retire
      for (int b = 0; b < 2; ++b) {
        if (nk[b] > 0) mbar_wait_bounded(bar_k + b, (uint32_t)(nk[b] - 1) & 1u, a.err);
        if (nv[b] > 0) mbar_wait_bounded(bar_v + b, (uint32_t)(nv[b] - 1) & 1u, a.err);
      }
    }
    __syncwarp();
  } else if (warp == 8) {
    // ---------------- MMA issuer. The whole warp runs the loop, so operand
    // addresses stay warp-uniform, and one elected lane issues each group of
    // products with its commit: a lone lane computing them while two softmax
    // warps share its scheduler falls behind an N = 128 product chain.
    if (n_blk > 0) {
      uint64_t* last = nullptr;  // the most recent commit, drained on the way out
      uint32_t last_par = 0;
      const uint64_t dk = sdesc(su32(sK)), dvh = sdesc(su32(sV)), dvl = sdesc_add(dvh, P::OPB);
      auto issue_s = [&](int j) -> bool {
        const int b = j & 1;
        if (!warp_wait_flag(bar_k + b, (uint32_t)(j >> 1) & 1u, fail, a.err)) return false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t t_s = tmem + P::T_S + 128 * b;
        const uint64_t kh = sdesc_add(dk, b * 2 * P::OPB), kl = sdesc_add(kh, P::OPB);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 128 * 128 + (kk & 3) * 32;
            const uint32_t qh = tmem + P::T_QH + 8 * kk, ql = tmem + P::T_QL + 8 * kk;
            if (kk == 0) mma_f16_ts(t_s, qh, kh, idesc<128>(), 0);
            else mma_f16_ts_acc(t_s, qh, sdesc_add(kh, off), idesc<128>());
            mma_f16_ts_acc(t_s, ql, sdesc_add(kh, off), idesc<128>());
            mma_f16_ts_acc(t_s, qh, sdesc_add(kl, off), idesc<128>());
          }
          mma_commit(bar_s + b);
        }
        __syncwarp();
        last = bar_s + b; last_par = (uint32_t)(j >> 1) & 1u;
        return true;
      };
      bool ok = issue_s(0);
      for (int j = 0; ok && j < n_blk; ++j) {
        // S(j+1) goes in ahead of PV(j): its TMEM buffer held P(j-1), which
        // PV(j-1), issued earlier, reads first
        if (j + 1 < n_blk && !issue_s(j + 1)) break;
        const uint32_t t_p = tmem + P::T_S + 128 * (j & 1);
        bool pv_ok = true;
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // key half h: P columns of thread half h, V~^T half h
          if (!(h == 0 ? warp_wait_flag2(bar_p + (j & 1), (uint32_t)(j >> 1) & 1u, bar_v,
                                         (uint32_t)j & 1u, fail, a.err)
                       : warp_wait_flag(bar_v + 1, (uint32_t)j & 1u, fail, a.err))) {
            pv_ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          if (elect_one()) {
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {  // 16 keys each
              const uint32_t ph = t_p + 64 * h + 8 * kq, pl = ph + 32;
              const uint32_t off = h * kVHalf + kq * 32;
              if (h == 0 && kq == 0) mma_f16_ts(t_o, ph, dvh, idesc<D>(), j > 0);
              else mma_f16_ts_acc(t_o, ph, sdesc_add(dvh, off), idesc<D>());
              mma_f16_ts_acc(t_o, pl, sdesc_add(dvh, off), idesc<D>());
              mma_f16_ts_acc(t_o, ph, sdesc_add(dvl, off), idesc<D>());
            }
            mma_commit(h == 0 ? bar_vh : bar_o);
          }
          __syncwarp();
          last = h == 0 ? bar_vh : bar_o; last_par = (uint32_t)j & 1u;
        }
        if (!pv_ok) break;
      }
      // the tensor pipe completes in order: the last commit covers everything
      if (last != nullptr &&
          !__all_sync(0xffffffffu, mbar_wait_bounded(last, last_par, a.err)))
        *fail = 1;
    }
    __syncwarp();
  } else {
    // ---------------- softmax (warps 0-7): two threads per row, 64 keys each
    for (int j = 0; j < n_blk; ++j) {
      const bool is_tile = j < n_tile_blk;
      const int64_t kpos0 = is_tile ? 128LL * j : win_pos0 + 128LL * (j - n_tile_blk);
      const int nkeys = is_tile ? 128 : min(128, a.win_len - 128 * (j - n_tile_blk));
      const bool full_vis = kpos0 + 127 <= pmin && nkeys == 128;  // uniform over the CTA
      bool bad = !mbar_wait_flag(bar_s + (j & 1), (uint32_t)(j >> 1) & 1u, fail, a.err);
      bad = __any_sync(0xffffffffu, bad || *fail != 0);  // the warp (and its pair) leave together
      const uint32_t t_s = tmem + P::T_S + 128 * (j & 1) + lb + 64 * half;
      float sv[64];
      float mloc = -INFINITY;
      if (!bad) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        tmem_ld32(t_s, *reinterpret_cast<float(*)[32]>(sv));
        tmem_ld32(t_s + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
        if (full_vis) {
#pragma unroll
          for (int u = 0; u < 64; u += 2) mloc = fmax3(mloc, sv[u], sv[u + 1]);
          if (!my_valid) mloc = -INFINITY;
        } else {
#pragma unroll
          for (int u = 0; u < 64; ++u) {
            const int t = 64 * half + u;
            const bool vis = my_valid && t < nkeys && kpos0 + t <= my_pos;
            sv[u] = vis ? sv[u] : -INFINITY;
            mloc = fmaxf(mloc, sv[u]);
          }
        }
      }
      float mblk;
      if (!pair_max(mloc, bad, xm, xb, j & 1, half, row, warp, mblk)) break;
      // move the reference max (and rescale O and the row sum) only when a
      // score exceeds it by more than 8; both threads of a row see the same
      // values
      const bool need = mblk > m_ref + 8.0f;
      const float m_new = need ? mblk : m_ref;
      const float alpha = (need && m_ref != -INFINITY) ? exp2f(m_ref - m_new) : 1.0f;
      m_ref = m_new;
      // exp2 of a non-positive argument (up to +8); results below 2^-126 flush
      // to zero; a row with no visible key yet subtracts +inf and gets 0
      const float msub = m_ref == -INFINITY ? INFINITY : m_ref;
      uint32_t hw[32], lw[32];
      float ls = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float p0 = ex2_ftz(sv[2 * e] - msub), p1 = ex2_ftz(sv[2 * e + 1] - msub);
        ls += p0 + p1;
        split2w(p0, p1, hw[e], lw[e]);
      }
      l_part = fmaf(l_part, alpha, ls);
      // P(j) replaces this thread's scores: hi in the first 32 columns of its
      // half, lo in the next 32
      tmem_st32_nowait(t_s, hw);
      tmem_st32_nowait(t_s + 32, lw);
      // O belongs to PV(j-1) until it completes
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        if (mbar_wait_flag(bar_o, (uint32_t)(j - 1) & 1u, fail, a.err)) {
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
          for (int c0 = 0; c0 < D / 2; c0 += 32) {
            float v[32];
            tmem_ld32(t_o + lb + half * (D / 2) + c0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tmem_st32(t_o + lb + half * (D / 2) + c0, v);
          }
        }
        // (a failed wait leaves O alone; the next block's check stops the warp)
      }
      tmem_wait_st();
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p + (j & 1));
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const bool ok = *fail == 0;
  // row sums of the two halves meet in shared memory
  if (tid < 256) xm[half * 128 + row] = l_part;
  __syncthreads();
  // ---- epilogue: O / l, one inverse rotation, store (one thread per row)
  if (tid < 128) {
    float o[D];
    const float l_row = xm[row] + xm[128 + row];
    if (n_blk > 0 && ok) {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        tmem_ld32(t_o + lb + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c0 + i] = v[i];
      }
    } else {
#pragma unroll
      for (int c = 0; c < D; ++c) o[c] = 0.f;
    }
    const float inv = l_row > 0.f ? 1.0f / l_row : 0.f;
#pragma unroll
    for (int c = 0; c < D; ++c) o[c] *= inv;
    fwht_reg<D>(o);
    if (my_valid) {
      float4* dst = reinterpret_cast<float4*>(a.out + ((int64_t)my_i * a.Hq + hq) * D);
#pragma unroll
      for (int c4 = 0; c4 < D / 4; ++c4) {
        float4 v;
        v.x = ok ? o[4 * c4] : NAN; v.y = ok ? o[4 * c4 + 1] : NAN;
        v.z = ok ? o[4 * c4 + 2] : NAN; v.w = ok ? o[4 * c4 + 3] : NAN;
        dst[c4] = v;
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(P::TMEM_COLS));
}

// ---------------------------------------------------------------------------
// attention at head_dim 256
//
// TMEM cannot hold Q' hi and lo (256 columns each) beside O (256 columns), so
// Q' hi stays in TMEM and Q' lo in shared memory (the Q'l K~h product takes
// both operands from shared memory). Keys stream in 64-key sub-blocks: K~ hi
// and lo of a sub-block (32 KB each, one buffer, each half on its own
// barrier so the next sub-block's hi half streams in while this one's
// Q'h K~l product runs) and V~^T hi and lo (32 KB each). TMEM: Q' hi in
// columns 0-127, S double-buffered in 128-191 and 192-255 (N = 64), O in
// 256-511. Roles, barriers and the tensor-pipe order S(0), S(1), PV(0), S(2),
// PV(1), ... are those of prefill_kernel, per sub-block. The two 128-channel
// halves of a row's rotation (the prologue's H q and the epilogue's H o) meet
// through shared memory: one butterfly over channel bit 7. A chunk whose grid
// would leave more than half of the SMs idle runs as clusters of two CTAs
// (gridDim.z = 2) that take alternate 128-key blocks of the same rows; rank 1
// hands its (m, l, O) to rank 0 through distributed shared memory and rank 0
// merges and stores.
struct PA256 {
  static constexpr int D = 256;
  static constexpr int QB = 128 * D * 2;                 // fp16 Q' lo [128 rows][256]
  static constexpr int KSB = 64 * D * 2;                 // K~ hi or lo of 64 keys: 4 x [64 rows][64 ch]
  static constexpr int VSB = D * 64 * 2;                 // V~^T hi or lo of 64 keys: [256 rows][64 keys]
  static constexpr int OFF_QL = 0;
  static constexpr int OFF_KH = OFF_QL + QB;
  static constexpr int OFF_KL = OFF_KH + KSB;
  static constexpr int OFF_VH = OFF_KL + KSB;
  static constexpr int OFF_VL = OFF_VH + VSB;
  static constexpr int OFF_BAR = OFF_VL + VSB;          // 9 mbarriers
  static constexpr int OFF_XM = OFF_BAR + 128;           // float [2][2][128]
  static constexpr int OFF_XB = OFF_XM + 2 * 2 * 128 * 4; // int [2][8]
  static constexpr int OFF_MISC = OFF_XB + 64;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;
  static constexpr int TMEM_COLS = 512;
  static constexpr int T_QH = 0, T_S = 128, T_O = 256;
  static_assert(OFF_KH % 1024 == 0 && OFF_VH % 1024 == 0 && OFF_VL % 1024 == 0, "swizzle atoms");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(OFF_VH >= 128 * 1024, "epilogue exchange fits Q'l and the K~ buffers");
  static_assert(OFF_BAR - OFF_KH >= 32 * 1024, "prologue exchange fits the K~ buffers");
};

__global__ void __launch_bounds__(320, 1) prefill_kernel_d256(const PrefillArgs a) {
  using P = PA256;
  constexpr int D = P::D;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                       ~uintptr_t(1023));
  unsigned char* sQl = sm + P::OFF_QL;
  unsigned char* sKh = sm + P::OFF_KH;
  unsigned char* sKl = sm + P::OFF_KL;
  unsigned char* sVh = sm + P::OFF_VH;
  uint64_t* bar_kh = reinterpret_cast<uint64_t*>(sm + P::OFF_BAR);  // K~ hi of sub-block landed
  uint64_t* bar_kl = bar_kh + 1;   // K~ lo landed
  uint64_t* bar_v = bar_kh + 2;    // V~^T hi + lo landed
  uint64_t* bar_s = bar_kh + 3;    // [2] S(j) complete (TMEM buffer j & 1); K~ lo free
  uint64_t* bar_khf = bar_kh + 5;  // the K~ hi products of S(j) complete: K~ hi free
  uint64_t* bar_o = bar_kh + 6;    // PV(j) complete: V~^T free, O current
  uint64_t* bar_p = bar_kh + 7;    // [2] P(j) in TMEM, O rescaled (per block parity, as above)
  float* xm = reinterpret_cast<float*>(sm + P::OFF_XM);
  int* xb = reinterpret_cast<int*>(sm + P::OFF_XB);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + P::OFF_MISC);
  volatile int* fail = reinterpret_cast<volatile int*>(sm + P::OFF_MISC + 4);
  float4* xch = reinterpret_cast<float4*>(sm + P::OFF_KH);  // prologue exchange (32 KB)
  float4* ych = reinterpret_cast<float4*>(sm + P::OFF_QL);  // epilogue exchange (128 KB)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127, half = (tid >> 7) & 1;
  const int kvh = blockIdx.y;
  const int ppc = 128 / a.G;
  const int i0 = blockIdx.x * ppc;
  const int my_g = row / ppc, my_i = i0 + row % ppc;
  const bool my_valid = my_i < a.C && my_g < a.G;
  const int64_t my_pos = a.pos0 + my_i;
  const int64_t pmax = a.pos0 + min(a.C, i0 + ppc) - 1;
  const int64_t pmin = a.pos0 + i0;
  const int hq = kvh * a.G + min(my_g, a.G - 1);
  const int64_t win_pos0 = 128LL * a.n_tiles;
  const Visible vis_blk = visible_blocks(a, pmax);
  const int n_tile_blk = vis_blk.n_tile_blk, n_blk = vis_blk.n_blk;
  // key split: with gridDim.z = 2 the two CTAs of a cluster take alternate
  // 128-key blocks of the same rows and merge (m, l, O) at the end
  const int rank = blockIdx.z, nsplit = gridDim.z;
  const int n_loc = n_blk > rank ? (n_blk - rank + nsplit - 1) / nsplit : 0;
  const int n_sub = 2 * n_loc;  // this CTA's 64-key sub-blocks
  auto gblk = [&](int k) { return k * nsplit + rank; };  // local block -> visible block
  auto image = [&](int jj) -> const uint8_t* {
    const int widx = jj < n_tile_blk ? jj : a.n_tblk + (jj - n_tile_blk);
    return a.ws + ((int64_t)kvh * a.ws_stride + widx) * PC<256>::BLK;
  };

  if (tid == 0) {
    for (int i = 0; i < 7; ++i) mbar_init1(bar_kh + i);
    for (int i = 0; i < 2; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(su32(bar_p + i)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *fail = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(tmem_slot)),
                 "r"(P::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_o = tmem + P::T_O;
  const uint32_t lb = lane_base_of(warp);
  const float rs2 = 0.70710678118654752f;
  if (tid < 256) {
    // Q' row: two threads per row, each rotating its 128 channels; the
    // butterfly over channel bit 7 pairs them through shared memory. Q' hi
    // goes to TMEM (columns 64 half ..), Q' lo to shared memory.
    float x[128];
    if (my_valid) {
      const float4* src =
          reinterpret_cast<const float4*>(a.q + ((int64_t)my_i * a.Hq + hq) * D + 128 * half);
#pragma unroll
      for (int c4 = 0; c4 < 32; ++c4) {
        const float4 v = src[c4];
        x[4 * c4] = v.x; x[4 * c4 + 1] = v.y; x[4 * c4 + 2] = v.z; x[4 * c4 + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < 128; ++c) x[c] = 0.f;
    }
    fwht_reg<128>(x);
    const float sc = a.qscale * rs2;
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {  // 32 channels per pass through the 32 KB buffer
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4)
        xch[c4 * 256 + tid] = make_float4(x[32 * pass + 4 * c4], x[32 * pass + 4 * c4 + 1],
                                          x[32 * pass + 4 * c4 + 2], x[32 * pass + 4 * c4 + 3]);
      asm volatile("bar.sync 1, 256;" ::: "memory");
      float y[32];
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 o = xch[c4 * 256 + (tid ^ 128)];
        const float of[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mine = x[32 * pass + 4 * c4 + e];
          // channel c of half 0: (a + b) / sqrt 2; channel 128 + c: (a - b) / sqrt 2
          y[4 * c4 + e] = (half == 0 ? mine + of[e] : of[e] - mine) * sc;
        }
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      uint32_t hw[16];
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split2w(y[8 * c8 + 2 * e], y[8 * c8 + 2 * e + 1], hw[4 * c8 + e], lo[e]);
        const int c = 128 * half + 32 * pass + 8 * c8;
        *reinterpret_cast<uint4*>(sQl + sw_off(row, c, 128)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      tmem_st16_nowait(tmem + lb + P::T_QH + 64 * half + 16 * pass, hw);
    }
    tmem_wait_st();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  float m_ref = -INFINITY, l_part = 0.f;  // softmax threads: reference max, half-row sum
  if (warp == 9) {
    // ---------------- loader
    if (lane == 0 && n_sub > 0) {
      int nkh = 1, nkl = 1, nv = 1;
      auto load_k = [&](unsigned char* dst, int part, int jsub, uint64_t* b) {
        // rows 64 s .. 64 s + 63 of each 64-channel block of the image's K~ part
        const uint8_t* src = image(gblk(jsub >> 1)) + part * PC<256>::OPB + (jsub & 1) * 8192;
        mbar_expect_tx(b, P::KSB);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) bulk_copy_tx(dst + kb * 8192, src + kb * 16384, 8192, b);
      };
      auto load_v = [&](int jsub) {  // key half jsub & 1 of the block's V~^T hi and lo
        const uint8_t* src = image(gblk(jsub >> 1)) + 2 * PC<256>::OPB + (jsub & 1) * P::VSB;
        mbar_expect_tx(bar_v, 2 * P::VSB);
        bulk_copy_tx(sVh, src, P::VSB, bar_v);
        bulk_copy_tx(sVh + P::VSB, src + PC<256>::OPB, P::VSB, bar_v);
      };
      pdl_wait();  // the images of this call's dequantisation grid are complete
      load_k(sKh, 0, 0, bar_kh);
      load_k(sKl, 1, 0, bar_kl);
      load_v(0);
      // in the tensor pipe's completion order -- the K~ hi products of S(j),
      // S(j), then PV(j-1) (S(j+1) goes in ahead of PV(j)) -- so that K~ hi of
      // the next sub-block is requested as soon as its buffer is free, not
      // after the P.V before it
      for (int j = 0; j < n_sub; ++j) {
        if (j + 1 < n_sub) {
          if (!mbar_wait_flag(bar_khf, (uint32_t)j & 1u, fail, a.err)) break;
          load_k(sKh, 0, j + 1, bar_kh);
          ++nkh;
          if (!mbar_wait_flag(bar_s + (j & 1), (uint32_t)(j >> 1) & 1u, fail, a.err)) break;
          load_k(sKl, 1, j + 1, bar_kl);
          ++nkl;
        }
        if (j >= 1) {
          if (!mbar_wait_flag(bar_o, (uint32_t)(j - 1) & 1u, fail, a.err)) break;
          load_v(j);
          ++nv;
        }
      }
      mbar_wait_bounded(bar_kh, (uint32_t)(nkh - 1) & 1u, a.err);
      mbar_wait_bounded(bar_kl, (uint32_t)(nkl - 1) & 1u, a.err);
      mbar_wait_bounded(bar_v, (uint32_t)(nv - 1) & 1u, a.err);
    }
    __syncwarp();
  } else if (warp == 8) {
    // ---------------- MMA issuer: the whole warp runs the loop and one
    // elected lane issues (operand addresses stay warp-uniform)
    if (n_sub > 0) {
      uint64_t* last = nullptr;
      uint32_t last_par = 0;
      const uint64_t dql = sdesc(su32(sQl)), dkh = sdesc(su32(sKh)), dkl = sdesc(su32(sKl));
      const uint64_t dvh = sdesc(su32(sVh)), dvl = sdesc_add(dvh, P::VSB);
      auto issue_s = [&](int j) -> bool {
        const uint32_t t_s = tmem + P::T_S + 64 * (j & 1);
        if (!warp_wait_flag(bar_kh, (uint32_t)j & 1u, fail, a.err)) return false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off_a = (kk >> 2) * 128 * 128 + (kk & 3) * 32;
            const uint32_t off_b = (kk >> 2) * 64 * 128 + (kk & 3) * 32;
            const uint32_t qh = tmem + P::T_QH + 8 * kk;
            if (kk == 0) mma_f16_ts(t_s, qh, dkh, idesc<64>(), 0);
            else mma_f16_ts_acc(t_s, qh, sdesc_add(dkh, off_b), idesc<64>());
            mma_f16(t_s, sdesc_add(dql, off_a), sdesc_add(dkh, off_b), idesc<64>(), 1);
          }
          mma_commit(bar_khf);
        }
        __syncwarp();
        last = bar_khf; last_par = (uint32_t)j & 1u;
        if (!warp_wait_flag(bar_kl, (uint32_t)j & 1u, fail, a.err)) return false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off_b = (kk >> 2) * 64 * 128 + (kk & 3) * 32;
            mma_f16_ts_acc(t_s, tmem + P::T_QH + 8 * kk, sdesc_add(dkl, off_b), idesc<64>());
          }
          mma_commit(bar_s + (j & 1));
        }
        __syncwarp();
        last = bar_s + (j & 1); last_par = (uint32_t)(j >> 1) & 1u;
        return true;
      };
      bool ok = issue_s(0);
      for (int j = 0; ok && j < n_sub; ++j) {
        if (j + 1 < n_sub && !issue_s(j + 1)) break;
        if (!warp_wait_flag2(bar_p + (j & 1), (uint32_t)(j >> 1) & 1u, bar_v, (uint32_t)j & 1u, fail,
                             a.err))
          break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t t_p = tmem + P::T_S + 64 * (j & 1);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 16 keys each; keys 32 h .. are thread half h's
            const uint32_t ph = t_p + 32 * (kk >> 1) + 8 * (kk & 1), pl = ph + 16;
            if (kk == 0) mma_f16_ts(t_o, ph, dvh, idesc<256>(), j > 0);
            else mma_f16_ts_acc(t_o, ph, sdesc_add(dvh, 32 * kk), idesc<256>());
            mma_f16_ts_acc(t_o, pl, sdesc_add(dvh, 32 * kk), idesc<256>());
            mma_f16_ts_acc(t_o, ph, sdesc_add(dvl, 32 * kk), idesc<256>());
          }
          mma_commit(bar_o);
        }
        __syncwarp();
        last = bar_o; last_par = (uint32_t)j & 1u;
      }
      if (last != nullptr &&
          !__all_sync(0xffffffffu, mbar_wait_bounded(last, last_par, a.err)))
        *fail = 1;
    }
    __syncwarp();
  } else {
    // ---------------- softmax (warps 0-7): two threads per row, 32 keys each
    for (int j = 0; j < n_sub; ++j) {
      const int jb = gblk(j >> 1), sb = j & 1;
      const bool is_tile = jb < n_tile_blk;
      const int64_t kpos0 = (is_tile ? 128LL * jb : win_pos0 + 128LL * (jb - n_tile_blk)) + 64 * sb;
      const int nkeys = (is_tile ? 128 : min(128, a.win_len - 128 * (jb - n_tile_blk))) - 64 * sb;
      const bool full_vis = kpos0 + 63 <= pmin && nkeys >= 64;
      bool bad = !mbar_wait_flag(bar_s + (j & 1), (uint32_t)(j >> 1) & 1u, fail, a.err);
      bad = __any_sync(0xffffffffu, bad || *fail != 0);
      const uint32_t t_s = tmem + P::T_S + 64 * (j & 1) + lb + 32 * half;
      float sv[32];
      float mloc = -INFINITY;
      if (!bad) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        tmem_ld32(t_s, sv);
        if (full_vis) {
#pragma unroll
          for (int u = 0; u < 32; u += 2) mloc = fmax3(mloc, sv[u], sv[u + 1]);
          if (!my_valid) mloc = -INFINITY;
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int t = 32 * half + u;
            const bool vis = my_valid && t < nkeys && kpos0 + t <= my_pos;
            sv[u] = vis ? sv[u] : -INFINITY;
            mloc = fmaxf(mloc, sv[u]);
          }
        }
      }
      float mblk;
      if (!pair_max(mloc, bad, xm, xb, j & 1, half, row, warp, mblk)) break;
      const bool need = mblk > m_ref + 8.0f;
      const float m_new = need ? mblk : m_ref;
      const float alpha = (need && m_ref != -INFINITY) ? exp2f(m_ref - m_new) : 1.0f;
      m_ref = m_new;
      const float msub = m_ref == -INFINITY ? INFINITY : m_ref;
      uint32_t hw[16], lw[16];
      float ls = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float p0 = ex2_ftz(sv[2 * e] - msub), p1 = ex2_ftz(sv[2 * e + 1] - msub);
        ls += p0 + p1;
        split2w(p0, p1, hw[e], lw[e]);
      }
      l_part = fmaf(l_part, alpha, ls);
      tmem_st16_nowait(t_s, hw);
      tmem_st16_nowait(t_s + 16, lw);
      // O belongs to PV(j-1) until it completes
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        if (mbar_wait_flag(bar_o, (uint32_t)(j - 1) & 1u, fail, a.err)) {
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
          for (int c0 = 0; c0 < D / 2; c0 += 32) {
            float v[32];
            tmem_ld32(t_o + lb + half * (D / 2) + c0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tmem_st32(t_o + lb + half * (D / 2) + c0, v);
          }
        }
      }
      tmem_wait_st();
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p + (j & 1));
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  bool ok = *fail == 0;
  if (tid < 256) xm[half * 128 + row] = l_part;
  __syncthreads();
  // ---- epilogue: O / l, one inverse rotation (two threads per row), store
  float o[128];
  float l_row = 0.f;
  if (tid < 256) {
    l_row = xm[row] + xm[128 + row];
    if (n_sub > 0 && ok) {
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        float v[32];
        tmem_ld32(t_o + lb + 128 * half + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c0 + i] = v[i];
      }
    } else {
#pragma unroll
      for (int c = 0; c < 128; ++c) o[c] = 0.f;
    }
  }
  if (nsplit > 1) {
    // rank 1's (m, l, O) go to rank 0's shared memory: O in the Q'l and K~
    // region, free once both CTAs' products completed (first cluster barrier)
    cg::cluster_group cluster = cg::this_cluster();
    float2* xml = reinterpret_cast<float2*>(sm + P::OFF_VH);           // [128 rows] (m, l)
    int* xfail = reinterpret_cast<int*>(sm + P::OFF_MISC + 8);
    cluster.sync();
    if (rank == 1) {
      float4* ro = cluster.map_shared_rank(ych, 0);
      if (tid < 256) {
#pragma unroll
        for (int c4 = 0; c4 < 32; ++c4)
          ro[c4 * 256 + tid] = make_float4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
        if (half == 0) cluster.map_shared_rank(xml, 0)[row] = make_float2(m_ref, l_row);
      }
      if (tid == 0) *cluster.map_shared_rank(xfail, 0) = ok ? 0 : 1;
    }
    cluster.sync();
    if (rank == 0 && tid < 256) {
      ok = ok && *xfail == 0;
      const float2 pml = xml[row];
      const float M = fmaxf(m_ref, pml.x);
      const float w0 = M == -INFINITY ? 0.f : exp2f(m_ref - M);
      const float w1 = M == -INFINITY ? 0.f : exp2f(pml.x - M);
#pragma unroll
      for (int c4 = 0; c4 < 32; ++c4) {
        const float4 p = ych[c4 * 256 + tid];
        o[4 * c4] = fmaf(o[4 * c4], w0, p.x * w1);
        o[4 * c4 + 1] = fmaf(o[4 * c4 + 1], w0, p.y * w1);
        o[4 * c4 + 2] = fmaf(o[4 * c4 + 2], w0, p.z * w1);
        o[4 * c4 + 3] = fmaf(o[4 * c4 + 3], w0, p.w * w1);
      }
      l_row = fmaf(l_row, w0, pml.y * w1);
      asm volatile("bar.sync 1, 256;" ::: "memory");  // the partner's O is read before reuse
    }
  }
  if (rank == 0 && tid < 256) {
    const float inv = (l_row > 0.f ? 1.0f / l_row : 0.f) * rs2;
#pragma unroll
    for (int c = 0; c < 128; ++c) o[c] *= inv;
    fwht_reg<128>(o);
    // Q'l and K~ are no longer read (the last MMA completed): they hold the exchange
#pragma unroll
    for (int c4 = 0; c4 < 32; ++c4)
      ych[c4 * 256 + tid] = make_float4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (my_valid) {
      float4* dst = reinterpret_cast<float4*>(a.out + ((int64_t)my_i * a.Hq + hq) * D + 128 * half);
#pragma unroll
      for (int c4 = 0; c4 < 32; ++c4) {
        const float4 p = ych[c4 * 256 + (tid ^ 128)];
        float4 v;
        if (half == 0) {
          v = make_float4(o[4 * c4] + p.x, o[4 * c4 + 1] + p.y, o[4 * c4 + 2] + p.z, o[4 * c4 + 3] + p.w);
        } else {
          v = make_float4(p.x - o[4 * c4], p.y - o[4 * c4 + 1], p.z - o[4 * c4 + 2], p.w - o[4 * c4 + 3]);
        }
        if (!ok) v = make_float4(NAN, NAN, NAN, NAN);
        dst[c4] = v;
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(P::TMEM_COLS));
}

template <int D, int SB, int VB>
cudaError_t launch_prefill_d(const PrefillArgs& a, cudaStream_t st) {
  using P = PC<D>;
  constexpr int att_smem = D == 256 ? PA256::SMEM : P::SMEM;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    if constexpr (D == 256)
      e = cudaFuncSetAttribute(prefill_kernel_d256, cudaFuncAttributeMaxDynamicSharedMemorySize, att_smem);
    else
      e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, att_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_dequant_kernel<D, SB, VB>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, P::template DQ<VB>::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  // With a dequantisation grid in front, the attention kernel is a programmatic
  // dependent of it: its CTAs may take the SMs the dequantisation leaves free
  // and rotate their query rows meanwhile; the loader waits for the grid before
  // its first image copy. The dequantisation grid itself starts only after all
  // earlier work on the stream, so everything else the attention kernel reads
  // (the queries) is complete either way.
  const bool dq = a.n_blk > a.first_blk;
  if (dq) {
    prefill_dequant_kernel<D, SB, VB><<<dim3(a.n_blk - a.first_blk, a.Hkv), P::NTHR,
                                        P::template DQ<VB>::SMEM, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int ppc = 128 / a.G;
  dim3 grid((a.C + ppc - 1) / ppc, a.Hkv);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(P::NTHR_ATT);
  cfg.dynamicSmemBytes = att_smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (dq) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if constexpr (D == 256) {
    // a grid that leaves more than half of the SMs idle splits each row
    // block's keys over a cluster of two CTAs
    const int64_t ctas = (int64_t)grid.x * grid.y;
    const int ns = 2 * ctas <= sm_count() ? 2 : 1;
    cfg.gridDim = dim3(grid.x, grid.y, ns);
    cfg.blockDim = dim3(320);
    if (ns > 1) {
      attr[na].id = cudaLaunchAttributeClusterDimension;
      attr[na].val.clusterDim.x = 1;
      attr[na].val.clusterDim.y = 1;
      attr[na].val.clusterDim.z = ns;
      ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, prefill_kernel_d256, a);
  } else {
    cfg.gridDim = grid;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, prefill_kernel<D>, a);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// Blocks visible to some position of the chunk [pos0, pos0 + C): tiles whose
// first position is <= the last one, then the window's 128-token blocks likewise.
void prefill_blocks(int64_t pos0, int C, int n_tiles, int win_len, int* n_tblk, int* n_blk) {
  const int64_t pmax = pos0 + C - 1;
  int nt = n_tiles;
  if (nt > 0 && 128LL * (nt - 1) > pmax) nt = (int)(pmax / 128) + 1;
  int nw = 0;
  for (int w = 0; 128 * w < win_len; ++w)
    if (128LL * n_tiles + 128 * w <= pmax) nw = w + 1;
  *n_tblk = nt;
  *n_blk = nt + nw;
}

size_t prefill_block_bytes(int D) { return (size_t)4 * 128 * D * 2; }

cudaError_t launch_prefill(const float* q, int C, int64_t pos0, const uint8_t* tiles,
                           int64_t tiles_bytes, const int64_t* tile_table, int table_stride,
                           int n_tiles,
                           const float* win_k, const float* win_v, int win_start, int win_len,
                           int win_capacity, int Hq, int Hkv, int D, float softmax_scale,
                           int scale_bytes, int v_bits, void* ws, int ws_blocks, int cached_tiles,
                           float* out, unsigned* err, cudaStream_t st) {
  PrefillArgs a;
  a.q = q; a.tiles = tiles; a.tile_table = tile_table; a.win_k = win_k; a.win_v = win_v;
  a.ws = reinterpret_cast<uint8_t*>(ws);
  a.out = out; a.pos0 = pos0; a.C = C; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv;
  a.n_tiles = n_tiles; a.table_stride = table_stride; a.win_start = win_start;
  a.win_len = win_len; a.win_cap = win_capacity; a.qscale = softmax_scale * kLog2e;
  a.tiles_bytes = tiles_bytes; a.err = err;
  prefill_blocks(pos0, C, n_tiles, win_len, &a.n_tblk, &a.n_blk);
  a.ws_stride = ws_blocks > 0 ? ws_blocks : a.n_blk;
  a.first_blk = cached_tiles < a.n_tblk ? cached_tiles : a.n_tblk;
  const int key = 100 * D + 10 * scale_bytes + v_bits;
  switch (key) {
    case 6442: return launch_prefill_d<64, 4, 2>(a, st);
    case 6422: return launch_prefill_d<64, 2, 2>(a, st);
    case 6444: return launch_prefill_d<64, 4, 4>(a, st);
    case 6424: return launch_prefill_d<64, 2, 4>(a, st);
    case 12842: return launch_prefill_d<128, 4, 2>(a, st);
    case 12822: return launch_prefill_d<128, 2, 2>(a, st);
    case 12844: return launch_prefill_d<128, 4, 4>(a, st);
    case 12824: return launch_prefill_d<128, 2, 4>(a, st);
    case 25642: return launch_prefill_d<256, 4, 2>(a, st);
    case 25622: return launch_prefill_d<256, 2, 2>(a, st);
    case 25644: return launch_prefill_d<256, 4, 4>(a, st);
    case 25624: return launch_prefill_d<256, 2, 4>(a, st);
    case 6443: return launch_prefill_d<64, 4, 3>(a, st);
    case 6423: return launch_prefill_d<64, 2, 3>(a, st);
    case 12843: return launch_prefill_d<128, 4, 3>(a, st);
    case 12823: return launch_prefill_d<128, 2, 3>(a, st);
    case 25643: return launch_prefill_d<256, 4, 3>(a, st);
    case 25623: return launch_prefill_d<256, 2, 3>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvarn
