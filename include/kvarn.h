/*
 * kvarn.h -- C ABI of the KVarN hot path on GB300 (sm_103a).
 *
 * KVarN stores the KV cache of a transformer as 4-bit keys and 2-bit values.
 * Every 128-token tile of each KV head is compressed on its own:
 *   1. an orthonormal Walsh-Hadamard rotation of every K and V row along
 *      head_dim                       (SharpInference issue #180, "Algorithm
 *                                      (per 128-token tile)" step 1;
 *                                      SharpInference PR #434, commit 82efc4f);
 *   2. a dual-axis "Sinkhorn" variance normalisation that alternates
 *      per-channel and per-token std scaling, accumulated in log space
 *                                     (issue #180, Algorithm step 2);
 *   3. asymmetric round-to-nearest quantisation: keys 4-bit per channel over
 *      the tile's tokens, values 2-bit per token over 128-channel groups,
 *      keys packed channel-major and values token-major
 *                                     (issue #180, Algorithm steps 3-4;
 *                                      PR #434, commit 82efc4f).
 * Attention reads the packed tiles directly: the query is rotated once, the
 * scales are folded into the dequant-dot at read time, one streaming softmax
 * runs over the tiles and the FP32 staging window of not-yet-full tiles, and
 * a single inverse rotation is applied at the end (issue #180 step 4; PR #434,
 * commits 0d7cd28 and 99c3773; SharpInference issue #433, item 2, which
 * describes the split-tile decode with an LSE combine).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every array argument is a DEVICE pointer owned by the caller, unless the
 *    argument says "host". The library never allocates device memory and
 *    keeps no state between calls: scratch space is passed in as a workspace,
 *    and how a call's kernels are launched is an argument of that call
 *    (launch_flags). The two exceptions are the sticky device error word
 *    (kvarn_get_device_error) and the fixed scratch array of
 *    kvarn_decode_attention_noalloc.
 *  - Work is enqueued asynchronously on the given stream; nothing synchronises
 *    except kvarn_get_device_error.
 *  - Calls that read packed records take the record pool's size (tiles_bytes);
 *    a record whose offset is negative, misaligned or runs past the pool is
 *    not read: the kernel poisons what depends on it with NaN and sets
 *    KVARN_DEVERR_RECORD in the device error word. Writes are bounded the
 *    same way (kvarn_compress_tile).
 *  - All floating-point data is IEEE fp32, little-endian.
 *  - The return value is a kvarn_status_t. Argument errors are detected on the
 *    host before anything is launched and nothing is enqueued in that case.
 *    A launch failure reported by the CUDA runtime returns KVARN_ERR_CUDA.
 *    Faults inside a kernel surface at the caller's next synchronisation.
 *  - head_dim D must be a power of two in [64, 256]; the pages' CUDA path
 *    supports power-of-two head dims up to 256 (PR #434, "Scope notes").
 *  - The GQA mapping is contiguous: query head h reads KV head h / G with
 *    G = Hq / Hkv (the pages do not state it; this is the usual grouping).
 */
#ifndef KVARN_H_
#define KVARN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. 0 = legacy default stream. */
typedef struct CUstream_st* kvarn_stream_t;

typedef enum kvarn_status {
  KVARN_OK = 0,
  KVARN_ERR_NULL = -1,        /* a required pointer is NULL                        */
  KVARN_ERR_ALIGN = -2,       /* a pointer, stride or offset breaks 16-byte alignment */
  KVARN_ERR_UNSUPPORTED = -3, /* head_dim, GQA group or iteration count out of range */
  KVARN_ERR_BAD_ARG = -4,     /* a size or count is negative or inconsistent       */
  KVARN_ERR_WORKSPACE = -5,   /* the workspace is smaller than the _workspace_bytes query */
  KVARN_ERR_CUDA = -6         /* the CUDA runtime rejected a launch                */
} kvarn_status_t;

/* Tokens per compressed tile. Tile i of a sequence always covers token
 * positions [128 i, 128 i + 128), whatever chunking produced it, so
 * re-chunking yields byte-identical tiles (PR #434, commit 99c3773; issue #433
 * item 1, "re-chunking oracle"). */
#define KVARN_TILE_TOKENS 128
#define KVARN_K_BITS 4
#define KVARN_V_BITS 2
#define KVARN_LAYOUT_VERSION 1
#define KVARN_LAYOUT_VERSION_F16_SCALES 2
#define KVARN_DEFAULT_SINKHORN_ITERS 4

/*
 * Launch flags of the calls on the decode path (kvarn_append_window,
 * kvarn_window_advance, kvarn_decode_split, kvarn_decode_combine,
 * kvarn_decode_attention, kvarn_decode_attention_noalloc), per call. The pages
 * have no counterpart: this is how the kernels are chained on this GPU.
 *   0                      plain stream-ordered launches.
 *   KVARN_LAUNCH_PDL       programmatic dependent launch: the kernel may be
 *                          scheduled while the previous kernel on the stream
 *                          is still running and waits for it on the device
 *                          before touching memory, which hides the launch
 *                          gap. Results are identical to 0.
 *   KVARN_LAUNCH_PDL | KVARN_LAUNCH_PREFETCH
 *                          as above, and the split kernel reads n_tiles, the
 *                          tile table and the packed records BEFORE that wait
 *                          (so a layer's records stream in while the previous
 *                          kernels finish). The caller guarantees that no
 *                          kernel still running ahead of it on the stream
 *                          writes those three (e.g. promotions are enqueued
 *                          between graph replays, not inside the step).
 * Other bits, or PREFETCH without PDL, give KVARN_ERR_BAD_ARG.
 */
#define KVARN_LAUNCH_PDL 1u
#define KVARN_LAUNCH_PREFETCH 2u

/*
 * Device error bits (kvarn_get_device_error). A kernel that gives up on
 * something sets its bit and writes NaN where the result depends on it; it
 * never traps, so the CUDA context stays usable.
 *   KVARN_DEVERR_WAIT      a wait for an asynchronous copy or tensor-core
 *                          product of the same kernel ran out of time
 *                          (200 ms): the hardware did not complete it.
 *   KVARN_DEVERR_RECORD    a tile-table entry (or a compress destination)
 *                          was negative, misaligned or ran past tiles_bytes;
 *                          a compress source ran past n_rows.
 *   KVARN_DEVERR_WINDOW    kvarn_append_window would have overfilled a
 *                          sequence's ring (win_len + n_new > win_capacity);
 *                          that sequence's rows were not written.
 *   KVARN_DEVERR_SELFTEST  set by kvarn_selftest_bounded_wait.
 */
#define KVARN_DEVERR_WAIT 1u
#define KVARN_DEVERR_RECORD 2u
#define KVARN_DEVERR_WINDOW 4u
#define KVARN_DEVERR_SELFTEST 8u

/*
 * Packed tile record: one record per (tile, KV head), headerless, all fields
 * at 16-byte aligned offsets. The pages fix only channel-major K codes,
 * token-major V codes and fp32 scales stored beside the codes (PR #434,
 * commit 82efc4f; issue #433 item 3 names f16 scales as a later saving);
 * the bit and field order below are this library's own.
 * With T = 128, D = head_dim, Gv = D / min(D, 128) value groups per token:
 *
 *   off_k_codes  u8 [D][T/2]   K code of token t, channel c: byte c*64 + t/2,
 *                              low nibble for even t, high nibble for odd t
 *   off_v_codes  u8 [T][D/4]   V code of token t, channel c: byte t*(D/4) + c/4,
 *                              bits 2*(c%4) .. 2*(c%4)+1
 *   off_k_delta  f32 [D]       K step per channel
 *   off_k_lo     f32 [D]       K offset (zero point, the group minimum) per channel
 *   off_k_s      f32 [D]       K Sinkhorn channel factor s_c = exp(alpha_c)
 *   off_k_r      f32 [T]       K Sinkhorn token factor r_t = exp(beta_t)
 *   off_v_delta  f32 [T][Gv]   V step per token and group
 *   off_v_lo     f32 [T][Gv]   V offset per token and group
 *   off_v_r      f32 [T]       V Sinkhorn token factor
 *   off_v_s      f32 [D]       V Sinkhorn channel factor
 *
 * Reconstruction in the rotated space: K~[t][c] = r_t s_c (delta_c code + lo_c),
 * V~[t][c] = r_t s_c (delta_{t,g(c)} code + lo_{t,g(c)}); the token's K or V
 * row is H times that row, H the orthonormal Sylvester Walsh-Hadamard matrix.
 * record_bytes = 112 D + 1024 + 1024 Gv: 9216 at D=64, 16384 at D=128,
 * 31744 at D=256.
 */
typedef struct kvarn_layout {
  int32_t version;        /* KVARN_LAYOUT_VERSION                           */
  int32_t head_dim;       /* D                                              */
  int32_t tile_tokens;    /* 128                                            */
  int32_t sinkhorn_iters; /* n, the fixed Sinkhorn round count (default 4)  */
  int32_t k_bits;         /* 4                                              */
  int32_t v_bits;         /* 2 (3 or 4 for the variants of kvarn_layout_ex) */
  int32_t v_group;        /* min(D, 128) channels per V quantisation group  */
  int32_t v_groups;       /* D / v_group                                    */
  int64_t record_bytes;
  int64_t off_k_codes, off_v_codes;
  int64_t off_k_delta, off_k_lo, off_k_s, off_k_r;
  int64_t off_v_delta, off_v_lo, off_v_r, off_v_s;
} kvarn_layout_t;

/* Fills *out (host pointer) for head_dim and sinkhorn_iters (1..16).
 * Returns KVARN_ERR_UNSUPPORTED for other head dims or iteration counts. */
int kvarn_layout(int head_dim, int sinkhorn_iters, kvarn_layout_t* out);

/*
 * The record layout with scale fields of scale_bits bits: 32 gives the layout
 * above (version KVARN_LAYOUT_VERSION); 16 gives the f16-scale layout
 * (version KVARN_LAYOUT_VERSION_F16_SCALES; SharpInference issue #433, item 3
 * names f16 scales as a saving of the record): the same fields in the same
 * order, every scale field (delta, lo, s, r of K and V) an IEEE binary16
 * value rounded to nearest from the fp32 one, and the same codes, which are
 * computed from the unrounded scales. record_bytes = 96 D + 2 (4 D + 256 +
 * 256 Gv): 7680 at D=64, 14336 at D=128, 28160 at D=256 (multiples of 128).
 * Reconstruction reads the stored binary16 values. Scales whose magnitude
 * exceeds 65504 (group ranges or stds that large) do not fit the format;
 * use the fp32 layout for such data. Every entry point taking a layout
 * accepts either version.
 * Returns KVARN_ERR_UNSUPPORTED for other head dims, iteration counts or
 * scale_bits.
 */
int kvarn_layout_scales(int head_dim, int sinkhorn_iters, int scale_bits, kvarn_layout_t* out);

/*
 * The record layout with scale fields of scale_bits bits (32 or 16, as in
 * kvarn_layout_scales) and v_bits-bit value codes (other key/value bit
 * widths, gmlx PR #116): 2 gives the k4v2 layouts above; 3 and 4 give k4v3
 * and k4v4 variants, values quantised per token and 128-channel group to
 * 2^v_bits levels (delta = (max - min) / (2^v_bits - 1)). Every width packs
 * a token's value codes as a little-endian bit stream of D * v_bits / 8
 * bytes at off_v_codes + t * D * v_bits / 8: channel c occupies stream bits
 * v_bits * c .. v_bits * c + v_bits - 1, stream bit i being bit i % 8 of
 * byte i / 8 (for 2 and 4 bits: the (c % (8 / v_bits))-th field of byte
 * c / (8 / v_bits); a 3-bit code can straddle two bytes). The keys, the
 * Sinkhorn factors and the field order are unchanged. record_bytes = 64 D +
 * 16 v_bits D + SB (4 D + 256 + 256 Gv), SB = scale_bits / 8: 18432 (k4v3)
 * and 20480 (k4v4) at D=128 with fp32 scales. kvarn_compress_tile, the
 * decode entry points and the prefill entry points accept all of them.
 * Returns KVARN_ERR_UNSUPPORTED for other head dims, iteration counts,
 * scale_bits or v_bits.
 */
int kvarn_layout_ex(int head_dim, int sinkhorn_iters, int scale_bits, int v_bits,
                    kvarn_layout_t* out);

/* Static, NUL-terminated description of a status code. Never NULL. */
const char* kvarn_status_string(int status);

/*
 * Reads the current device's error word (KVARN_DEVERR_* bits set by kernels
 * of this library since it was last cleared) into *bits (host pointer) and,
 * if clear is non-zero, clears it. The pages have no counterpart: it is how
 * a kernel that gave up reports it. Synchronises the current device (a
 * blocking copy), so do not call it inside stream capture. The first call on
 * a device, like the first launch of any call that reports, looks the word's
 * address up once (cudaGetSymbolAddress); make that first call outside
 * stream capture.
 */
int kvarn_get_device_error(unsigned* bits, int clear);

/*
 * Self-check of the device failure path: one kernel waits on an mbarrier
 * that nothing will complete, gives up after timeout_us microseconds
 * (1..1000000), sets KVARN_DEVERR_SELFTEST in the error word and returns
 * normally. Lets a caller (or a test) confirm that a device wait that runs
 * out is reported without faulting the context. No counterpart on the pages.
 */
int kvarn_selftest_bounded_wait(unsigned timeout_us, kvarn_stream_t stream);

/*
 * Query rotation (PR #434, commit 0d7cd28, llm_kvarn_rotate_query; issue #180
 * Algorithm step 1): q_rot[i] = H q[i] for every row i, H the orthonormal
 * Sylvester Walsh-Hadamard matrix of order D (symmetric, so self-inverse).
 * Because H is orthonormal, (H q) . (H k) = q . k.
 *   q, q_rot : fp32 [n_rows][D], contiguous, 16-byte aligned. q_rot == q
 *              (in place) is allowed; any other overlap is not.
 *   n_rows   : >= 0; 0 enqueues nothing.
 */
int kvarn_rotate_query(const float* q, float* q_rot, int64_t n_rows, int head_dim,
                       kvarn_stream_t stream);

/*
 * Tile compression (issue #180, Algorithm steps 1-3; PR #434, commits 82efc4f
 * and 0d7cd28, llm_kvarn_compress_tile). Each unit u turns 128 consecutive raw
 * K rows and the matching 128 V rows into one packed record:
 *   K rows  k_raw[(src_row0[u] + t) * row_stride + c], t < 128, c < D
 *   V rows  v_raw[(same index)]
 *   record  tiles + dst_record[u] (byte offset), layout->record_bytes long.
 * A unit is a pure function of its 256 input rows, so the result does not
 * depend on which other units share the launch or on their order.
 *   k_raw, v_raw  : fp32, n_rows rows of row_stride elements, 16-byte aligned.
 *   row_stride    : elements between rows, >= D and a multiple of 4.
 *   n_rows        : rows in k_raw and v_raw. A unit whose rows run past
 *                   n_rows (src_row0[u] < 0 or src_row0[u] + 128 > n_rows)
 *                   is skipped and KVARN_DEVERR_RECORD set.
 *   src_row0      : int64 [n_units], device.
 *   tiles         : u8 base of the record pool, 16-byte aligned, tiles_bytes
 *                   long.
 *   dst_record    : int64 [n_units] byte offsets, device, multiples of 16;
 *                   records of one launch must not overlap. A unit whose
 *                   record would not lie inside the pool (or is misaligned)
 *                   is skipped and KVARN_DEVERR_RECORD set.
 *   layout        : host pointer from kvarn_layout().
 */
int kvarn_compress_tile(const float* k_raw, const float* v_raw, int64_t row_stride,
                        int64_t n_rows, const int64_t* src_row0, uint8_t* tiles,
                        int64_t tiles_bytes, const int64_t* dst_record, int64_t n_units,
                        const kvarn_layout_t* layout, kvarn_stream_t stream);

/*
 * FP32 staging window append (PR #434, commit 6040076: the FP32 window is the
 * staging area and whole 128-token tiles are promoted out of it). Copies n_new
 * new raw K and V tokens of every sequence into that sequence's ring window:
 *   k_new, v_new  : fp32 [n_seq][n_new][Hkv][D] (the projection's layout).
 *   win_k, win_v  : fp32 [n_seq][Hkv][win_capacity][D] ring buffers.
 *   win_start,
 *   win_len       : int32 [n_seq], device. New token i of sequence s goes to
 *                   ring slot (win_start[s] + win_len[s] + i) % win_capacity.
 *                   win_len[s] + n_new must not exceed win_capacity (the ring
 *                   would overwrite rows not yet promoted): a sequence for
 *                   which it would is left unwritten and KVARN_DEVERR_WINDOW
 *                   is set.
 *   launch_flags  : 0 or KVARN_LAUNCH_PDL (PREFETCH has no effect here).
 * The library does not change win_start or win_len: the caller applies the
 * promotion rule (while win_len >= W, compress the oldest 128 tokens with
 * kvarn_compress_tile, then win_start += 128, win_len -= 128) and advances
 * them. With win_capacity a multiple of 128 and win_start kept a multiple of
 * 128, the oldest 128 tokens are always contiguous rows of the ring.
 */
int kvarn_append_window(const float* k_new, const float* v_new, int64_t n_new,
                        float* win_k, float* win_v, int win_capacity,
                        const int32_t* win_start, const int32_t* win_len,
                        int n_seq, int n_kv_heads, int head_dim, unsigned launch_flags,
                        kvarn_stream_t stream);

/*
 * Device-side window bookkeeping (PR #434, commit 6040076: whole-tile
 * promotion out of the FP32 staging window; commit e43f3f0: promotion is
 * hoisted out of the CUDA-graph decode step). For every sequence s < n_seq:
 *   win_len[s] += d_len                      (tokens appended since the last call)
 *   then, if promote > 0:
 *   win_start[s] = (win_start[s] + 128 * promote) % win_capacity
 *   win_len[s]  -= 128 * promote,  n_tiles[s] += promote
 * The caller decides `promote` under the rule "while win_len >= W, compress
 * the oldest 128 tokens" and has already compressed those tokens with
 * kvarn_compress_tile. win_start, win_len, n_tiles: int32 [n_seq], device
 * (n_tiles may be NULL when promote == 0). win_capacity must be a positive
 * multiple of 128. d_len and promote apply to every sequence of the call: a
 * ragged batch whose sequences promote at different steps advances each
 * sequence with its own call (pointers offset to that sequence, n_seq = 1).
 * One tiny launch; it lets a whole decode step be captured.
 * launch_flags: 0 or KVARN_LAUNCH_PDL.
 */
int kvarn_window_advance(int32_t* win_start, int32_t* win_len, int32_t* n_tiles, int n_seq,
                         int d_len, int promote, int win_capacity, unsigned launch_flags,
                         kvarn_stream_t stream);

/*
 * Decode attention over the compressed cache (PR #434, commits 0d7cd28 and
 * e43f3f0, llm_kvarn_attention; issue #433 item 2: a fixed worst-case grid
 * over (head, tile range) with early exit, followed by an LSE combine, with
 * the deferred inverse rotation applied after combining the rotated
 * partials). Two kernels:
 *   kvarn_decode_split    grid over (item, KV head, sequence): each item is a
 *                         fixed range of packed tiles, or a fixed range of
 *                         128-token chunks of the FP32 window; it writes the
 *                         item's softmax max, sum and (rotated for tiles, raw
 *                         for the window) value accumulator into ws.
 *   kvarn_decode_combine  grid over (query head, sequence): LSE merge of the
 *                         items, one inverse rotation of the merged tile
 *                         accumulator, plus the window accumulator, / sum.
 * kvarn_decode_attention enqueues both.
 *
 * For query head h of sequence b the result is exact softmax attention
 *   out[b][h] = sum_j softmax_j(scale * q[b][h] . k_j) v_j
 * over every cached token j of KV head h / G: the tiles' tokens (k_j, v_j
 * reconstructed as described at kvarn_layout_t) and then the window's raw rows.
 *   q          : fp32 [B][Hq][D], unrotated. Hq / Hkv = G must be 1..8.
 *   tiles      : u8 base of the record pool, tiles_bytes long.
 *   tile_table : int64 [B][Hkv][max_tiles] record byte offsets, multiples of
 *                128 (record_bytes is a multiple of 128, so a pool of whole
 *                records qualifies); an entry that is misaligned, negative or
 *                runs past tiles_bytes makes that head's output NaN and sets
 *                KVARN_DEVERR_RECORD; entries at or past n_tiles[b] are never
 *                read.
 *   n_tiles    : int32 [B], 0 <= n_tiles[b] <= max_tiles (clamped on device).
 *   win_k/v    : fp32 [B][Hkv][win_capacity][D]; win_start/win_len int32 [B]
 *                as in kvarn_append_window (win_len clamped to win_capacity).
 *   out        : fp32 [B][Hq][D]. A head with no tokens at all gets zeros.
 *   softmax_scale : usually 1/sqrt(D) (the pages do not state it).
 *   ws         : device workspace of at least kvarn_decode_workspace_bytes()
 *                bytes, 256-byte aligned; it holds the per-item partials and
 *                needs no initialisation. Calls sharing ws must not overlap.
 *   launch_flags : KVARN_LAUNCH_* bits, see above.
 * The grids depend only on (B, Hq, Hkv, D, max_tiles, win_capacity, device),
 * so the calls can be captured in a CUDA graph and replayed while n_tiles and
 * the windows change. Results are deterministic (bit-identical on repeat).
 */
int kvarn_decode_workspace_bytes(int B, int Hq, int Hkv, int head_dim, int max_tiles,
                                 int win_capacity, size_t* bytes);
int kvarn_decode_split(const float* q, const uint8_t* tiles, int64_t tiles_bytes,
                       const int64_t* tile_table, const int32_t* n_tiles, const float* win_k,
                       const float* win_v, const int32_t* win_start, const int32_t* win_len,
                       int win_capacity, int B, int Hq, int Hkv, int head_dim, int max_tiles,
                       float softmax_scale, const kvarn_layout_t* layout, void* ws,
                       size_t ws_bytes, unsigned launch_flags, kvarn_stream_t stream);
int kvarn_decode_combine(const void* ws, size_t ws_bytes, int B, int Hq, int Hkv, int head_dim,
                         int max_tiles, int win_capacity, float* out, unsigned launch_flags,
                         kvarn_stream_t stream);
int kvarn_decode_attention(const float* q, const uint8_t* tiles, int64_t tiles_bytes,
                           const int64_t* tile_table, const int32_t* n_tiles,
                           const float* win_k, const float* win_v, const int32_t* win_start,
                           const int32_t* win_len, int win_capacity, int B, int Hq, int Hkv,
                           int head_dim, int max_tiles, float softmax_scale,
                           const kvarn_layout_t* layout, void* ws, size_t ws_bytes, float* out,
                           unsigned launch_flags, kvarn_stream_t stream);

/*
 * Chunked-prefill attention (PR #434, commit 99c3773, llm_kvarn_prefill_attention:
 * a single streaming softmax over the compressed tiles plus the FP32 window
 * with a deferred inverse WHT; issue #433 item 1: run the K-score and
 * V-aggregate contractions on tensor cores). For one sequence, after the
 * chunk's K/V were appended to the window and whole tiles promoted:
 *   out[i][h] = sum_j softmax_j(scale * q[i][h] . k_j) v_j
 * over the keys j of KV head h / G whose position is <= pos0 + i, where tile
 * k holds positions [128 k, 128 k + 128) and window token w (w < win_len)
 * sits at position 128 * n_tiles + w.
 * The two contractions run on tcgen05 tensor cores with fp32 accumulation;
 * each operand (rotated query, keys, probabilities, values) is carried as a
 * pair of fp16 values whose sum holds about 22 bits, so the result meets the
 * same 1e-4 relative bound as decode. Two kernels: every 128-key block the
 * chunk sees (packed tiles dequantised, window rows rotated into the same
 * space) is written once per KV head into ws as fp16 operand images, then one
 * attention kernel per (KV head, 128 score rows) streams those images through
 * shared memory; the softmax, causal mask and final inverse rotation run on
 * CUDA cores. The call as a whole is ordered after earlier work on the
 * stream. Within it, the attention kernel is a programmatic dependent of the
 * dequantisation kernel: it may rotate its query rows while the images are
 * being written, and reads an image only after they all are.
 *   q_chunk    : fp32 [C][Hq][D], unrotated; out: fp32 [C][Hq][D].
 *   tiles      : u8 base of the record pool, tiles_bytes long.
 *   tile_table : int64 [Hkv][table_stride] record byte offsets (multiples of
 *                16, inside the pool; another offset makes the keys of that
 *                tile NaN and sets KVARN_DEVERR_RECORD) of this sequence's
 *                tiles; table_stride >= n_tiles.
 *   win_k/v    : fp32 [Hkv][win_capacity][D] ring of this sequence;
 *                win_start, win_len, n_tiles: host integers.
 *   ws         : device workspace of at least kvarn_prefill_workspace_bytes(
 *                n_tiles, win_len, Hkv, head_dim) bytes, 256-byte aligned; no
 *                initialisation needed. Calls sharing ws must not overlap.
 * Requires pos0 + C <= 128 * n_tiles + win_len (the chunk's own keys are in
 * the cache), head_dim 64, 128 or 256 and Hq / Hkv <= 8. At head_dim 256
 * the attention streams keys in 64-key sub-blocks (the query operands fill
 * much of the tensor memory); the result has the same form.
 */
int kvarn_prefill_workspace_bytes(int n_tiles, int win_len, int Hkv, int head_dim, size_t* bytes);
int kvarn_prefill_attention(const float* q_chunk, int C, int64_t pos0, const uint8_t* tiles,
                            int64_t tiles_bytes, const int64_t* tile_table, int table_stride,
                            int n_tiles,
                            const float* win_k, const float* win_v, int win_start, int win_len,
                            int win_capacity, int Hq, int Hkv, int head_dim, float softmax_scale,
                            const kvarn_layout_t* layout, void* ws, size_t ws_bytes, float* out,
                            kvarn_stream_t stream);

/*
 * Chunked prefill that keeps the packed tiles' operand images in ws from one
 * chunk to the next (same result as kvarn_prefill_attention). A prompt's
 * tiles never change once promoted, so a caller that streams the chunks of
 * one sequence in order can keep ws for the whole prompt and let each call
 * convert only the tiles promoted since the previous one, plus the window
 * blocks (which change every chunk).
 *   ws           : [Hkv][ws_blocks] block images of kvarn_prefill_workspace_bytes(
 *                  max_tiles, win_capacity, Hkv, head_dim) / Hkv / ws_blocks bytes
 *                  each; ws_blocks >= the blocks any call of the sequence sees,
 *                  e.g. max_tiles + ceil(win_capacity / 128), and the same for
 *                  every call of the sequence.
 *   cached_tiles : leading tiles whose images ws already holds: 0 on the first
 *                  call, then the n_tiles of the previous call, provided that
 *                  call's chunk was the last one appended (it then saw every
 *                  tile), and that tiles, tile_table, layout and ws_blocks
 *                  are unchanged. 0 <= cached_tiles <= n_tiles. Images of tiles
 *                  [cached_tiles, n_tiles) and of the window blocks are built.
 * Returns KVARN_ERR_BAD_ARG for ws_blocks <= 0, KVARN_ERR_WORKSPACE when
 * ws_blocks is smaller than the blocks this chunk sees or ws_bytes smaller
 * than ws_blocks * Hkv images; otherwise as kvarn_prefill_attention.
 */
int kvarn_prefill_attention_cached(const float* q_chunk, int C, int64_t pos0, const uint8_t* tiles,
                                   int64_t tiles_bytes, const int64_t* tile_table,
                                   int table_stride, int n_tiles,
                                   const float* win_k, const float* win_v, int win_start,
                                   int win_len, int win_capacity, int Hq, int Hkv, int head_dim,
                                   float softmax_scale, const kvarn_layout_t* layout, void* ws,
                                   size_t ws_bytes, int ws_blocks, int cached_tiles, float* out,
                                   kvarn_stream_t stream);

/*
 * Decode attention for callers that cannot allocate device memory. The pages
 * have no counterpart to this entry point; it exists for embedders that may
 * not call cudaMalloc where attention runs (code inside another runtime's
 * memory arena, or a host framework that owns every allocation).
 * Same arguments and result as kvarn_decode_attention, minus the workspace:
 * the partials go to a scratch array of KVARN_NOALLOC_SCRATCH_BYTES that the
 * library keeps in its own device memory. Every GPU that loads the library
 * holds that array until the process exits.
 *  - Returns KVARN_ERR_WORKSPACE (nothing enqueued) when
 *    kvarn_decode_workspace_bytes() for these sizes exceeds the array; with
 *    head_dim 128, 32 query and 8 KV heads that allows about
 *    B * max_tiles <= 16,000 on a 152-SM GB300 (the split plan, and with it
 *    the workspace size, depends on the device's SM count).
 *  - The first call on a device (that device current) looks up the array's
 *    device address with cudaGetSymbolAddress and caches it; make that first
 *    call before any stream capture. It never calls cudaMalloc or cudaFree.
 *  - Every call on a device shares the one array and leaves its last contents
 *    there; nothing in it needs to start at zero. Calls that overlap on the
 *    GPU (different streams, or different host threads) race on it.
 */
#define KVARN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int kvarn_decode_attention_noalloc(const float* q, const uint8_t* tiles, int64_t tiles_bytes,
                                   const int64_t* tile_table, const int32_t* n_tiles,
                                   const float* win_k, const float* win_v,
                                   const int32_t* win_start, const int32_t* win_len,
                                   int win_capacity, int B, int Hq, int Hkv, int head_dim,
                                   int max_tiles, float softmax_scale,
                                   const kvarn_layout_t* layout, float* out,
                                   unsigned launch_flags, kvarn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVARN_H_ */
