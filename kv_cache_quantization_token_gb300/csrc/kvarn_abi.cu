// kvarn_abi.cu -- the extern "C" entry points of libkvarn.so.
//
// Each entry point validates its arguments on the host, returns a
// kvarn_status_t without enqueuing anything when they are wrong, and otherwise
// launches the kernels of compress.cu, window.cu or decode.cu on the stream.
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "kvarn_common.cuh"

namespace {

bool supported_dim(int D) { return D == 64 || D == 128 || D == 256; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
int from_cuda(cudaError_t e) { return e == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA; }

// sb: bytes of each scale field, 4 (fp32, layout version 1) or 2 (binary16,
// layout version 2); vb: value code width, 2 (the k4v2 preset) or 4 (k4v4).
int fill_layout(int D, int iters, int sb, int vb, kvarn_layout_t* L) {
  memset(L, 0, sizeof(*L));
  L->version = sb == 2 ? KVARN_LAYOUT_VERSION_F16_SCALES : KVARN_LAYOUT_VERSION;
  L->head_dim = D;
  L->tile_tokens = KVARN_TILE_TOKENS;
  L->sinkhorn_iters = iters;
  L->k_bits = KVARN_K_BITS;
  L->v_bits = vb;
  L->v_group = D < 128 ? D : 128;
  L->v_groups = D / L->v_group;
  const int64_t T = KVARN_TILE_TOKENS, gv = L->v_groups;
  L->off_k_codes = 0;
  L->off_v_codes = L->off_k_codes + (int64_t)D * (T / 2);
  L->off_k_delta = L->off_v_codes + T * (D * vb / 8);
  L->off_k_lo = L->off_k_delta + (int64_t)sb * D;
  L->off_k_s = L->off_k_lo + (int64_t)sb * D;
  L->off_k_r = L->off_k_s + (int64_t)sb * D;
  L->off_v_delta = L->off_k_r + sb * T;
  L->off_v_lo = L->off_v_delta + sb * T * gv;
  L->off_v_r = L->off_v_lo + sb * T * gv;
  L->off_v_s = L->off_v_r + sb * T;
  L->record_bytes = L->off_v_s + (int64_t)sb * D;
  return KVARN_OK;
}

// Bytes of each scale field of a layout this library produced.
int scale_bytes_of(const kvarn_layout_t* L) {
  return L->version == KVARN_LAYOUT_VERSION_F16_SCALES ? 2 : 4;
}

// A layout handed back by the caller must be one this library produced.
bool layout_ok(const kvarn_layout_t* L) {
  if (!L || !supported_dim(L->head_dim)) return false;
  if (L->version != KVARN_LAYOUT_VERSION && L->version != KVARN_LAYOUT_VERSION_F16_SCALES)
    return false;
  if (L->sinkhorn_iters < 1 || L->sinkhorn_iters > 16) return false;
  if (L->v_bits < 2 || L->v_bits > 4) return false;
  kvarn_layout_t ref;
  fill_layout(L->head_dim, L->sinkhorn_iters, scale_bytes_of(L), L->v_bits, &ref);
  return memcmp(&ref, L, sizeof(ref)) == 0;
}

bool flags_ok(unsigned flags) {
  if (flags & ~(KVARN_LAUNCH_PDL | KVARN_LAUNCH_PREFETCH)) return false;
  return !((flags & KVARN_LAUNCH_PREFETCH) && !(flags & KVARN_LAUNCH_PDL));
}

// The device error word: KVARN_DEVERR_* bits that kernels OR in when they give
// up on something. One word per device (each device that loads the library
// has its own copy of this file-scope variable); kernels get its address as an
// argument.
__device__ unsigned g_device_error;
constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
unsigned* g_err_ptr[kMaxDevices] = {};

}  // namespace

namespace kvarn {
unsigned* device_error_word() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_err_ptr[dev];
}
}  // namespace kvarn

extern "C" {

int kvarn_get_device_error(unsigned* bits, int clear) {
  if (!bits) return KVARN_ERR_NULL;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return KVARN_ERR_CUDA;
  *bits = v;
  if (clear && v) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return KVARN_ERR_CUDA;
  }
  return KVARN_OK;
}

int kvarn_selftest_bounded_wait(unsigned timeout_us, kvarn_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return KVARN_ERR_BAD_ARG;
  unsigned* err = kvarn::device_error_word();
  if (!err) return KVARN_ERR_CUDA;
  return from_cuda(kvarn::launch_selftest_wait((uint64_t)timeout_us * 1000, err, (cudaStream_t)stream));
}

int kvarn_layout(int head_dim, int sinkhorn_iters, kvarn_layout_t* out) {
  return kvarn_layout_ex(head_dim, sinkhorn_iters, 32, KVARN_V_BITS, out);
}

int kvarn_layout_scales(int head_dim, int sinkhorn_iters, int scale_bits, kvarn_layout_t* out) {
  return kvarn_layout_ex(head_dim, sinkhorn_iters, scale_bits, KVARN_V_BITS, out);
}

int kvarn_layout_ex(int head_dim, int sinkhorn_iters, int scale_bits, int v_bits,
                    kvarn_layout_t* out) {
  if (!out) return KVARN_ERR_NULL;
  if (!supported_dim(head_dim) || sinkhorn_iters < 1 || sinkhorn_iters > 16 ||
      (scale_bits != 32 && scale_bits != 16) || v_bits < 2 || v_bits > 4)
    return KVARN_ERR_UNSUPPORTED;
  return fill_layout(head_dim, sinkhorn_iters, scale_bits / 8, v_bits, out);
}

const char* kvarn_status_string(int status) {
  switch (status) {
    case KVARN_OK: return "ok";
    case KVARN_ERR_NULL: return "a required pointer is NULL";
    case KVARN_ERR_ALIGN: return "a pointer, stride or offset is not 16-byte aligned";
    case KVARN_ERR_UNSUPPORTED: return "unsupported head_dim, GQA group or iteration count";
    case KVARN_ERR_BAD_ARG: return "a size or count is negative or inconsistent";
    case KVARN_ERR_WORKSPACE: return "workspace smaller than the _workspace_bytes query";
    case KVARN_ERR_CUDA: return "the CUDA runtime rejected a launch or a copy";
    default: return "unknown kvarn status";
  }
}

int kvarn_rotate_query(const float* q, float* q_rot, int64_t n_rows, int head_dim,
                       kvarn_stream_t stream) {
  if (!supported_dim(head_dim)) return KVARN_ERR_UNSUPPORTED;
  if (n_rows < 0 || n_rows > (int64_t)8 * 0x7fffffff) return KVARN_ERR_BAD_ARG;
  if (n_rows == 0) return KVARN_OK;
  if (!q || !q_rot) return KVARN_ERR_NULL;
  if (!aligned16(q) || !aligned16(q_rot)) return KVARN_ERR_ALIGN;
  if (q != q_rot) {  // only exact in-place use may overlap
    const char *a = reinterpret_cast<const char*>(q), *b = reinterpret_cast<const char*>(q_rot);
    const int64_t bytes = n_rows * head_dim * 4;
    if (a < b + bytes && b < a + bytes) return KVARN_ERR_BAD_ARG;
  }
  return from_cuda(kvarn::launch_rotate(q, q_rot, n_rows, head_dim, (cudaStream_t)stream));
}

int kvarn_compress_tile(const float* k_raw, const float* v_raw, int64_t row_stride,
                        int64_t n_rows, const int64_t* src_row0, uint8_t* tiles,
                        int64_t tiles_bytes, const int64_t* dst_record, int64_t n_units,
                        const kvarn_layout_t* layout, kvarn_stream_t stream) {
  if (!layout) return KVARN_ERR_NULL;
  if (!layout_ok(layout)) return KVARN_ERR_UNSUPPORTED;
  const int D = layout->head_dim;
  if (n_units < 0 || n_units > 0x3fffffff || n_rows < 0 || tiles_bytes < 0) return KVARN_ERR_BAD_ARG;
  if (n_units == 0) return KVARN_OK;
  if (!k_raw || !v_raw || !src_row0 || !tiles || !dst_record) return KVARN_ERR_NULL;
  if (row_stride < D || n_rows < KVARN_TILE_TOKENS || tiles_bytes < layout->record_bytes)
    return KVARN_ERR_BAD_ARG;
  if ((row_stride & 3) || !aligned16(k_raw) || !aligned16(v_raw) || !aligned16(tiles))
    return KVARN_ERR_ALIGN;
  return from_cuda(kvarn::launch_compress(D, layout->sinkhorn_iters, scale_bytes_of(layout),
                                          layout->v_bits, k_raw, v_raw, row_stride, n_rows,
                                          src_row0, tiles, tiles_bytes, dst_record, n_units,
                                          kvarn::device_error_word(), (cudaStream_t)stream));
}

int kvarn_append_window(const float* k_new, const float* v_new, int64_t n_new, float* win_k,
                        float* win_v, int win_capacity, const int32_t* win_start,
                        const int32_t* win_len, int n_seq, int n_kv_heads, int head_dim,
                        unsigned launch_flags, kvarn_stream_t stream) {
  if (!supported_dim(head_dim)) return KVARN_ERR_UNSUPPORTED;
  if (!flags_ok(launch_flags)) return KVARN_ERR_BAD_ARG;
  if (n_new < 0 || n_seq < 0 || n_kv_heads <= 0 || win_capacity <= 0) return KVARN_ERR_BAD_ARG;
  if (n_new > win_capacity) return KVARN_ERR_BAD_ARG;
  if (n_new == 0 || n_seq == 0) return KVARN_OK;
  if (!k_new || !v_new || !win_k || !win_v || !win_start || !win_len) return KVARN_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(win_k) || !aligned16(win_v))
    return KVARN_ERR_ALIGN;
  return from_cuda(kvarn::launch_append(k_new, v_new, n_new, win_k, win_v, win_capacity,
                                        win_start, win_len, n_seq, n_kv_heads, head_dim,
                                        launch_flags, kvarn::device_error_word(),
                                        (cudaStream_t)stream));
}

static int decode_check(int B, int Hq, int Hkv, int D, int max_tiles, int win_capacity) {
  if (!supported_dim(D)) return KVARN_ERR_UNSUPPORTED;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || max_tiles < 0 || win_capacity < 0) return KVARN_ERR_BAD_ARG;
  if (Hq % Hkv) return KVARN_ERR_BAD_ARG;
  if (Hq / Hkv > 8) return KVARN_ERR_UNSUPPORTED;
  if (B > 65535 || Hkv > 65535) return KVARN_ERR_BAD_ARG;
  return KVARN_OK;
}

int kvarn_decode_workspace_bytes(int B, int Hq, int Hkv, int head_dim, int max_tiles,
                                 int win_capacity, size_t* bytes) {
  if (!bytes) return KVARN_ERR_NULL;
  const int rc = decode_check(B, Hq, Hkv, head_dim, max_tiles, win_capacity);
  if (rc != KVARN_OK) return rc;
  kvarn::DecodePlan p;
  kvarn::decode_plan(B, Hq, Hkv, head_dim, max_tiles, win_capacity, &p);
  *bytes = p.ws_bytes;
  return KVARN_OK;
}

static int decode_prepare(const float* q, const uint8_t* tiles, int64_t tiles_bytes,
                          const int64_t* tile_table, const int32_t* n_tiles, const float* win_k,
                          const float* win_v, const int32_t* win_start, const int32_t* win_len,
                          int win_capacity, int B, int Hq, int Hkv, int head_dim, int max_tiles,
                          float softmax_scale, const kvarn_layout_t* layout, void* ws,
                          size_t ws_bytes, unsigned launch_flags, kvarn::DecodePlan* p,
                          kvarn::DecodeArgs* a) {
  int rc = decode_check(B, Hq, Hkv, head_dim, max_tiles, win_capacity);
  if (rc != KVARN_OK) return rc;
  if (!flags_ok(launch_flags) || tiles_bytes < 0) return KVARN_ERR_BAD_ARG;
  if (!layout) return KVARN_ERR_NULL;
  if (!layout_ok(layout) || layout->head_dim != head_dim) return KVARN_ERR_UNSUPPORTED;
  kvarn::decode_plan(B, Hq, Hkv, head_dim, max_tiles, win_capacity, p);
  if (B == 0) return KVARN_OK;
  if (!q || !n_tiles) return KVARN_ERR_NULL;
  if (max_tiles > 0 && (!tiles || !tile_table)) return KVARN_ERR_NULL;
  if (win_capacity > 0 && (!win_k || !win_v || !win_start || !win_len)) return KVARN_ERR_NULL;
  if (p->ws_bytes > 0 && !ws) return KVARN_ERR_NULL;
  if (ws_bytes < p->ws_bytes) return KVARN_ERR_WORKSPACE;
  if (!aligned16(q) || (max_tiles > 0 && !aligned16(tiles)) ||
      (win_capacity > 0 && (!aligned16(win_k) || !aligned16(win_v))) ||
      (reinterpret_cast<uintptr_t>(ws) & 255))
    return KVARN_ERR_ALIGN;
  if (!(softmax_scale == softmax_scale)) return KVARN_ERR_BAD_ARG;
  *a = kvarn::DecodeArgs{q, tiles, tile_table, n_tiles, win_k, win_v, win_start, win_len,
                         win_capacity, B, Hq, Hkv, head_dim, max_tiles, softmax_scale,
                         scale_bytes_of(layout), layout->v_bits, tiles_bytes, launch_flags,
                         kvarn::device_error_word()};
  return KVARN_OK;
}

int kvarn_decode_split(const float* q, const uint8_t* tiles, int64_t tiles_bytes,
                       const int64_t* tile_table, const int32_t* n_tiles, const float* win_k,
                       const float* win_v, const int32_t* win_start, const int32_t* win_len,
                       int win_capacity, int B, int Hq, int Hkv, int head_dim, int max_tiles,
                       float softmax_scale, const kvarn_layout_t* layout, void* ws,
                       size_t ws_bytes, unsigned launch_flags, kvarn_stream_t stream) {
  kvarn::DecodePlan p;
  kvarn::DecodeArgs a;
  const int rc = decode_prepare(q, tiles, tiles_bytes, tile_table, n_tiles, win_k, win_v,
                                win_start, win_len, win_capacity, B, Hq, Hkv, head_dim, max_tiles,
                                softmax_scale, layout, ws, ws_bytes, launch_flags, &p, &a);
  if (rc != KVARN_OK || B == 0) return rc;
  return from_cuda(kvarn::launch_decode_split(p, a, ws, (cudaStream_t)stream));
}

int kvarn_decode_combine(const void* ws, size_t ws_bytes, int B, int Hq, int Hkv, int head_dim,
                         int max_tiles, int win_capacity, float* out, unsigned launch_flags,
                         kvarn_stream_t stream) {
  const int rc = decode_check(B, Hq, Hkv, head_dim, max_tiles, win_capacity);
  if (rc != KVARN_OK) return rc;
  if (!flags_ok(launch_flags)) return KVARN_ERR_BAD_ARG;
  if (B == 0) return KVARN_OK;
  kvarn::DecodePlan p;
  kvarn::decode_plan(B, Hq, Hkv, head_dim, max_tiles, win_capacity, &p);
  if (!out || (p.ws_bytes > 0 && !ws)) return KVARN_ERR_NULL;
  if (ws_bytes < p.ws_bytes) return KVARN_ERR_WORKSPACE;
  if (!aligned16(out) || (reinterpret_cast<uintptr_t>(ws) & 255)) return KVARN_ERR_ALIGN;
  return from_cuda(kvarn::launch_decode_combine(p, B, Hq, head_dim, ws, out, launch_flags,
                                                (cudaStream_t)stream));
}

int kvarn_decode_attention(const float* q, const uint8_t* tiles, int64_t tiles_bytes,
                           const int64_t* tile_table, const int32_t* n_tiles,
                           const float* win_k, const float* win_v, const int32_t* win_start,
                           const int32_t* win_len, int win_capacity, int B, int Hq, int Hkv,
                           int head_dim, int max_tiles, float softmax_scale,
                           const kvarn_layout_t* layout, void* ws, size_t ws_bytes, float* out,
                           unsigned launch_flags, kvarn_stream_t stream) {
  kvarn::DecodePlan p;
  kvarn::DecodeArgs a;
  int rc = decode_prepare(q, tiles, tiles_bytes, tile_table, n_tiles, win_k, win_v, win_start,
                          win_len, win_capacity, B, Hq, Hkv, head_dim, max_tiles, softmax_scale,
                          layout, ws, ws_bytes, launch_flags, &p, &a);
  if (rc != KVARN_OK || B == 0) return rc;
  if (!out) return KVARN_ERR_NULL;
  if (!aligned16(out)) return KVARN_ERR_ALIGN;
  rc = from_cuda(kvarn::launch_decode_split(p, a, ws, (cudaStream_t)stream));
  if (rc != KVARN_OK) return rc;
  return from_cuda(kvarn::launch_decode_combine(p, B, Hq, head_dim, ws, out, launch_flags,
                                                (cudaStream_t)stream));
}

int kvarn_prefill_workspace_bytes(int n_tiles, int win_len, int Hkv, int head_dim, size_t* bytes) {
  if (!bytes) return KVARN_ERR_NULL;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVARN_ERR_UNSUPPORTED;
  if (n_tiles < 0 || win_len < 0 || Hkv <= 0) return KVARN_ERR_BAD_ARG;
  const size_t blocks = (size_t)n_tiles + (size_t)(win_len + KVARN_TILE_TOKENS - 1) / KVARN_TILE_TOKENS;
  *bytes = blocks * (size_t)Hkv * kvarn::prefill_block_bytes(head_dim);
  return KVARN_OK;
}

static int prefill_common(const float* q_chunk, int C, int64_t pos0, const uint8_t* tiles,
                          int64_t tiles_bytes, const int64_t* tile_table, int table_stride,
                          int n_tiles,
                          const float* win_k, const float* win_v, int win_start, int win_len,
                          int win_capacity, int Hq, int Hkv, int head_dim, float softmax_scale,
                          const kvarn_layout_t* layout, void* ws, size_t ws_bytes, int ws_blocks,
                          int cached_tiles, float* out, kvarn_stream_t stream) {
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVARN_ERR_UNSUPPORTED;
  if (!layout) return KVARN_ERR_NULL;
  if (!layout_ok(layout) || layout->head_dim != head_dim) return KVARN_ERR_UNSUPPORTED;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || Hkv > 65535) return KVARN_ERR_BAD_ARG;
  if (Hq / Hkv > 8) return KVARN_ERR_UNSUPPORTED;
  if (C < 0 || pos0 < 0 || n_tiles < 0 || win_len < 0 || win_capacity < 0 || tiles_bytes < 0 ||
      table_stride < n_tiles || win_len > win_capacity)
    return KVARN_ERR_BAD_ARG;
  if (pos0 + C > (int64_t)KVARN_TILE_TOKENS * n_tiles + win_len) return KVARN_ERR_BAD_ARG;
  if (cached_tiles < 0 || cached_tiles > n_tiles || ws_blocks < 0) return KVARN_ERR_BAD_ARG;
  if (C == 0) return KVARN_OK;
  if (!q_chunk || !out) return KVARN_ERR_NULL;
  if (n_tiles > 0 && (!tiles || !tile_table)) return KVARN_ERR_NULL;
  if (win_len > 0 && (!win_k || !win_v)) return KVARN_ERR_NULL;
  int n_tblk = 0, n_blk = 0;
  kvarn::prefill_blocks(pos0, C, n_tiles, win_len, &n_tblk, &n_blk);
  const int stride = ws_blocks > 0 ? ws_blocks : n_blk;
  if (stride < n_blk) return KVARN_ERR_WORKSPACE;
  const size_t need = (size_t)stride * (size_t)Hkv * kvarn::prefill_block_bytes(head_dim);
  if (need > 0 && !ws) return KVARN_ERR_NULL;
  if (ws_bytes < need) return KVARN_ERR_WORKSPACE;
  if (!aligned16(q_chunk) || !aligned16(out) || (n_tiles > 0 && !aligned16(tiles)) ||
      (win_len > 0 && (!aligned16(win_k) || !aligned16(win_v))) ||
      (reinterpret_cast<uintptr_t>(ws) & 255))
    return KVARN_ERR_ALIGN;
  if (!(softmax_scale == softmax_scale)) return KVARN_ERR_BAD_ARG;
  return from_cuda(kvarn::launch_prefill(q_chunk, C, pos0, tiles, tiles_bytes, tile_table,
                                         table_stride, n_tiles, win_k, win_v, win_start, win_len,
                                         win_capacity, Hq, Hkv, head_dim, softmax_scale,
                                         scale_bytes_of(layout), layout->v_bits, ws, stride,
                                         cached_tiles, out, kvarn::device_error_word(),
                                         (cudaStream_t)stream));
}

int kvarn_prefill_attention(const float* q_chunk, int C, int64_t pos0, const uint8_t* tiles,
                            int64_t tiles_bytes, const int64_t* tile_table, int table_stride,
                            int n_tiles, const float* win_k, const float* win_v, int win_start,
                            int win_len, int win_capacity, int Hq, int Hkv, int head_dim,
                            float softmax_scale, const kvarn_layout_t* layout, void* ws,
                            size_t ws_bytes, float* out, kvarn_stream_t stream) {
  return prefill_common(q_chunk, C, pos0, tiles, tiles_bytes, tile_table, table_stride, n_tiles,
                        win_k, win_v,
                        win_start, win_len, win_capacity, Hq, Hkv, head_dim, softmax_scale, layout,
                        ws, ws_bytes, 0, 0, out, stream);
}

int kvarn_prefill_attention_cached(const float* q_chunk, int C, int64_t pos0, const uint8_t* tiles,
                                   int64_t tiles_bytes, const int64_t* tile_table,
                                   int table_stride, int n_tiles, const float* win_k,
                                   const float* win_v, int win_start, int win_len,
                                   int win_capacity, int Hq, int Hkv, int head_dim,
                                   float softmax_scale, const kvarn_layout_t* layout, void* ws,
                                   size_t ws_bytes, int ws_blocks, int cached_tiles, float* out,
                                   kvarn_stream_t stream) {
  if (ws_blocks <= 0) return KVARN_ERR_BAD_ARG;
  return prefill_common(q_chunk, C, pos0, tiles, tiles_bytes, tile_table, table_stride, n_tiles,
                        win_k, win_v,
                        win_start, win_len, win_capacity, Hq, Hkv, head_dim, softmax_scale, layout,
                        ws, ws_bytes, ws_blocks, cached_tiles, out, stream);
}

int kvarn_window_advance(int32_t* win_start, int32_t* win_len, int32_t* n_tiles, int n_seq,
                         int d_len, int promote, int win_capacity, unsigned launch_flags,
                         kvarn_stream_t stream) {
  if (n_seq < 0 || promote < 0 || win_capacity <= 0 || (win_capacity % KVARN_TILE_TOKENS) ||
      !flags_ok(launch_flags))
    return KVARN_ERR_BAD_ARG;
  if (n_seq == 0 || (d_len == 0 && promote == 0)) return KVARN_OK;
  if (!win_start || !win_len || (promote > 0 && !n_tiles)) return KVARN_ERR_NULL;
  return from_cuda(kvarn::launch_window_advance(win_start, win_len, n_tiles, n_seq, d_len, promote,
                                                win_capacity, launch_flags, (cudaStream_t)stream));
}

}  // extern "C"
