// window.cu -- query rotation and FP32 staging-window append.
//
// Query rotation: q' = H q per query head, H the orthonormal Sylvester
// Walsh-Hadamard matrix (SharpInference PR #434, commit 0d7cd28,
// llm_kvarn_rotate_query; issue #180, "Algorithm (per 128-token tile)" step 1).
// Window append: raw K/V rows go into the per-sequence FP32 ring that stages
// tokens until a whole 128-token tile is promoted (PR #434, commit 6040076).
// Window advance: the ring's start/length and the tile count move on the
// device after an append or a promotion.
#include "kvarn_common.cuh"

namespace kvarn {
namespace {

// One warp per row; lane l holds elements l*E .. l*E+E-1 (E = D/32). The
// butterflies of the low log2(E) bits run in registers, the other five across
// lanes with shuffles; the result is scaled by 1/sqrt(D).
template <int D>
__global__ void __launch_bounds__(256) rotate_kernel(const float* q, float* q_rot, int64_t n_rows) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  float x[E];
  const float* src = q + row * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = src[e];
#pragma unroll
  for (int h = 1; h < E; h <<= 1)
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (!(e & h)) {
        const float a = x[e], b = x[e | h];
        x[e] = a + b;
        x[e | h] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = lane & m;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = upper ? (o - x[e]) : (x[e] + o);
    }
  }
  const float sc = 1.0f / sqrtf((float)D);
  float* dst = q_rot + row * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) dst[e] = x[e] * sc;
}

__global__ void append_kernel(const float4* __restrict__ k_new, const float4* __restrict__ v_new,
                              int64_t n_new, float4* __restrict__ win_k, float4* __restrict__ win_v,
                              int cap, const int32_t* __restrict__ win_start,
                              const int32_t* __restrict__ win_len, int n_seq, int hkv, int d4,
                              unsigned* err) {
  pdl_trigger();
  pdl_wait();
  const int64_t total = (int64_t)n_seq * n_new * hkv * d4;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c4 = (int)(idx % d4);
    int64_t r = idx / d4;
    const int h = (int)(r % hkv);
    r /= hkv;
    const int64_t i = r % n_new;
    const int s = (int)(r / n_new);
    // a ring that would overflow keeps its rows (none of them promoted yet)
    const int len = win_len[s];
    if (len < 0 || (int64_t)len + n_new > cap) {
      if (i == 0 && h == 0 && c4 == 0) report(err, KVARN_DEVERR_WINDOW);
      continue;
    }
    int64_t slot = ((int64_t)win_start[s] + len + i) % cap;
    if (slot < 0) slot += cap;
    const int64_t dst = (((int64_t)s * hkv + h) * cap + slot) * d4 + c4;
    win_k[dst] = k_new[idx];
    win_v[dst] = v_new[idx];
  }
}

// Window bookkeeping on the device, so that a decode step (append, attend,
// advance) can be captured in a CUDA graph and replayed.
__global__ void advance_kernel(int32_t* win_start, int32_t* win_len, int32_t* n_tiles, int n_seq,
                               int d_len, int promote, int cap) {
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n_seq) return;
  int len = win_len[s] + d_len;
  if (promote > 0) {
    win_start[s] = (int)(((int64_t)win_start[s] + 128LL * promote) % cap);
    len -= 128 * promote;
    n_tiles[s] += promote;
  }
  win_len[s] = len;
}

// Waits on an mbarrier that nothing completes, for at most timeout_ns, then
// reports KVARN_DEVERR_SELFTEST: the device failure path, run on purpose.
__global__ void selftest_wait_kernel(uint64_t timeout_ns, unsigned* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(&bar))
                 : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_timed(&bar, 0, err, KVARN_DEVERR_SELFTEST, nullptr, timeout_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(uint64_t timeout_ns, unsigned* err, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(timeout_ns, err);
  return cudaGetLastError();
}

cudaError_t launch_window_advance(int32_t* win_start, int32_t* win_len, int32_t* n_tiles,
                                  int n_seq, int d_len, int promote, int win_capacity,
                                  unsigned flags, cudaStream_t st) {
  LaunchCfg L(dim3((n_seq + 127) / 128), dim3(128), 0, st, flags);
  return cudaLaunchKernelEx(&L.cfg, advance_kernel, win_start, win_len, n_tiles, n_seq, d_len,
                            promote, win_capacity);
}

cudaError_t launch_rotate(const float* q, float* q_rot, int64_t n_rows, int D, cudaStream_t st) {
  const unsigned blocks = (unsigned)((n_rows + 7) / 8);
  switch (D) {
    case 64: rotate_kernel<64><<<blocks, 256, 0, st>>>(q, q_rot, n_rows); break;
    case 128: rotate_kernel<128><<<blocks, 256, 0, st>>>(q, q_rot, n_rows); break;
    case 256: rotate_kernel<256><<<blocks, 256, 0, st>>>(q, q_rot, n_rows); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_append(const float* k_new, const float* v_new, int64_t n_new, float* win_k,
                          float* win_v, int win_capacity, const int32_t* win_start,
                          const int32_t* win_len, int n_seq, int n_kv_heads, int D,
                          unsigned flags, unsigned* err, cudaStream_t st) {
  const int64_t total = (int64_t)n_seq * n_new * n_kv_heads * (D / 4);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  LaunchCfg L(dim3((unsigned)blocks), dim3(256), 0, st, flags);
  return cudaLaunchKernelEx(&L.cfg, append_kernel, reinterpret_cast<const float4*>(k_new),
                            reinterpret_cast<const float4*>(v_new), n_new,
                            reinterpret_cast<float4*>(win_k), reinterpret_cast<float4*>(win_v),
                            win_capacity, win_start, win_len, n_seq, n_kv_heads, D / 4, err);
}

}  // namespace kvarn
