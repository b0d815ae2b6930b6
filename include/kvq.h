/*
 * kvq.h -- C ABI of libkvq: low-bit KV-cache append and decode attention,
 * written for NVIDIA GB300 (sm_103a).
 *
 * Method (KV Cache量化技术介绍, developer.horizon.auto/blog/13163):
 *   KVQuant, "Per-Channel Key Quantization"       keys: one scale/zero per
 *                                                  channel over a token block;
 *   KVQuant, "Pre-RoPE Key Quantization"          keys are stored pre-RoPE and
 *                                                  rotated after dequantization;
 *   KVQuant, "Per-Vector Dense-and-Sparse ..."    each vector's largest-|x|
 *                                                  elements kept as fp16 pairs;
 *   Quanto, "Quanto 的量化原理" steps 1-2          block-wise codes with a
 *                                                  scale and zero_point each.
 * Arithmetic of one code (the page's formula image is lost; this is the
 * reading the library implements and its oracle checks bit for bit):
 *   z = min over the group's dense elements (fp16, exact; -0 stored as +0)
 *   s = fp16_round_up(fp32(fp32(max - min) / L)),  L = 2^bits - 1
 *   q = clamp(rint_half_even(fp32(fp32(x - z) / s)), 0, L)   (q = 0 if s = 0)
 *   x_hat = q * s + z, except at outlier positions, which hold the fp16 value.
 *
 * Conventions for every entry point:
 *   - Ownership: the caller allocates and frees every device buffer, using the
 *     sizes kvq_layout() returns. The library allocates nothing, frees
 *     nothing and never synchronizes the device or the stream.
 *   - Pointers: device pointers unless marked "host"; each must be 16-byte
 *     aligned (cudaMalloc and the PyTorch caching allocator return 256-byte
 *     aligned memory). A buffer whose size is 0 may be NULL.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream). Work is enqueued asynchronously; inputs must stay
 *     valid and unmodified until the stream has executed the call.
 *   - Errors: every function returns a kvq_status. Arguments are checked on
 *     the host before anything is launched; on any error nothing is launched
 *     and no output or cache field changes. KVQ_ERR_CUDA reports a launch
 *     error (cudaGetLastError after the launch; no synchronization).
 *   - Devices: calls run on the calling thread's current CUDA device; the
 *     buffers must belong to that device. Device ordinals 0 .. 63 are
 *     supported; a launching call on a higher ordinal returns
 *     KVQ_ERR_UNSUPPORTED before anything is launched.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_ARG = 1,          /* NULL or misaligned pointer, negative count, q_pos out of range */
  KVQ_ERR_UNSUPPORTED = 2,  /* a configuration outside the supported set (see kvq_config) */
  KVQ_ERR_CAPACITY = 3,     /* T_cur + n_new > T_max */
  KVQ_ERR_WORKSPACE = 4,    /* workspace or RoPE table smaller than kvq_layout() says */
  KVQ_ERR_CUDA = 5,         /* the CUDA runtime reported an error at launch */
  KVQ_ERR_TIMEOUT = 6       /* a bounded wait of a kernel expired (read from the status word) */
} kvq_status;

/* Device status word: the first 4 bytes of every decode workspace (the
 * layout's workspace_bytes include a 256-byte header for it; the partials
 * follow). The head_dim-128 decode kernels wait on shared-memory barriers for
 * their TMA copies; every wait is bounded (one second). When one expires
 * the kernel ORs KVQ_STATUS_TIMEOUT into the word, waits (bounded) for its own
 * copies, writes NaN partials for its part of the output and returns, so the
 * context stays usable. The library never clears the word and never reads it
 * back: zero the header when the workspace is allocated, and copy the word to
 * the host (cudaMemcpyAsync, 4 bytes) when a check is wanted; a set bit means
 * the outputs of the calls since it was cleared are not valid
 * (KVQ_ERR_TIMEOUT). */
#define KVQ_STATUS_TIMEOUT 1u

#define KVQ_MAX_OUTLIERS 8  /* largest n_out per vector */

/* kvq_config.flags. KVQ_FLAG_PRECISE_SCORES: decode attention at head_dim
 * 128 dequantizes and rotates the keys in fp32 and splits both q . k operands
 * into fp16 hi + lo parts (three tensor-core products each), so the scores
 * carry about 22 significant bits instead of fp16's 11; P . V takes p * s as
 * hi + lo as well. Without it the scores come from fp16 operands: their error
 * is about 2^-11 of sum_c |q_c k_c| per token, which stays far below the
 * outputs' tolerance while the logits span a few nats but moves the weights
 * of attention whose competing logits are tens of nats apart from the rest.
 * The flag costs decode time (about 2.1-2.3x on GB300). head_dim 64 computes
 * in fp32 and ignores it; a level-table decode (kvq_decode_attn_levels) at
 * head_dim 128 runs on the tensor-core kernel with fp16 operands unless the
 * flag is set, which sends it to the fp32 CUDA-core kernel. Other bits:
 * reserved (0). */
#define KVQ_FLAG_PRECISE_SCORES 1

/* One layer's cache shape. Supported: bits in {2, 3, 4, 8} (8: the 8-bit
 * width of Quanto's block-wise scheme, page 3 "Quanto"); D in {64, 128};
 * key_block in {64, 128}; value_group in {32, 64, 128} dividing D;
 * T_max > 0 a multiple of key_block and < 2^24; B, H_kv >= 1, B*H_kv <= 65535;
 * outlier_frac = 0 (no outliers) or in (0, 1]: n_out = max(1, floor(frac*D)),
 * at most KVQ_MAX_OUTLIERS (frac = 0.01 gives n_out = 1 for D = 64 or 128). */
typedef struct kvq_config {
  int32_t B;            /* sequences in the batch (all hold T_cur tokens) */
  int32_t H_kv;         /* key/value heads */
  int32_t D;            /* head_dim */
  int32_t T_max;        /* token capacity per sequence */
  int32_t bits;         /* code width */
  int32_t key_block;    /* Bk: tokens per key-quantization block */
  int32_t value_group;  /* Gv: channels per value-quantization group */
  float outlier_frac;   /* fraction of each K and V vector kept as fp16 outliers */
  int32_t flags;        /* KVQ_FLAG_* (0: defaults) */
} kvq_config;

/* Cache buffers. Every buffer is [B][H_kv][...] with each (b, h_kv) stream
 * contiguous; "fp16" means IEEE binary16 bits in a uint16.
 *   K_CODES [B][H_kv][T_max][D*bits/8]   packed key codes; row t is an
 *            LSB-first bitstream, element d at bits [bits*d, bits*d + bits)
 *   K_META  [B][H_kv][T_max/Bk][D][2]    fp16 {s, z} per key block and channel
 *   K_TAIL  [B][H_kv][Bk][D]             fp16 keys of the unfinished block,
 *            token t at row t % Bk
 *   K_OUTL  [B][H_kv][T_max][n_out][2]   {uint16 channel, fp16 value} per key
 *            vector of a finished block, descending |x| then ascending channel
 *   V_CODES [B][H_kv][T_max][D*bits/8]   packed value codes (same packing)
 *   V_META  [B][H_kv][T_max][D/Gv][2]    fp16 {s, z} per token and group
 *   V_OUTL  [B][H_kv][T_max][n_out][2]   {channel, fp16 value} per value vector
 * Key codes, metadata and outliers exist only for finished blocks (tokens
 * below Bk * floor(T_cur / Bk)); the last T_cur % Bk keys stay fp16 in K_TAIL.
 */
typedef enum kvq_buffer {
  KVQ_K_CODES = 0, KVQ_K_META, KVQ_K_TAIL, KVQ_K_OUTL,
  KVQ_V_CODES, KVQ_V_META, KVQ_V_OUTL, KVQ_NBUF
} kvq_buffer;

typedef struct kvq_layout_t {
  size_t bytes[KVQ_NBUF];        /* size of each cache buffer, whole batch */
  size_t stream_bytes[KVQ_NBUF]; /* size of one (b, h_kv) stream of each buffer */
  size_t cache_bytes;            /* sum of bytes[] */
  size_t fp16_equiv_bytes;       /* fp16 K and V of the same capacity: 2*B*H_kv*T_max*D*2 */
  size_t rope_bytes;             /* size of the RoPE table (kvq_rope_init) */
  size_t workspace_bytes;        /* decode scratch for the given H_q */
  int32_t n_out;                 /* outliers kept per vector */
  int32_t code_row_bytes;        /* D*bits/8 */
} kvq_layout_t;

/* Device pointers to one layer's cache plus its fill level. */
typedef struct kvq_cache {
  void* k_codes;
  void* k_meta;
  void* k_tail;
  void* k_outl;   /* may be NULL when n_out = 0 */
  void* v_codes;
  void* v_meta;
  void* v_outl;   /* may be NULL when n_out = 0 */
  int32_t T_cur;  /* tokens stored per sequence; kvq_append advances it */
} kvq_cache;

/* Sizes of every buffer for `cfg` and for decode with H_q query heads
 * (H_q a positive multiple of H_kv). Passage: the KV-cache memory formula of
 * the page "TurboQuant ..." (mlqm.cn/news/1002276), §2.1 "KVCache的本质与内存
 * 开销": fp16 K and V take 2 x layers x batch x tokens x hidden x 2 bytes;
 * fp16_equiv_bytes is that size for one layer of this cache's capacity, and
 * cache_bytes what the packed codes, metadata and outliers take instead.
 * Host-only and pure: touches no device.
 * Errors: KVQ_ERR_ARG (NULL), KVQ_ERR_UNSUPPORTED (cfg or H_q). */
KVQ_API int kvq_layout(const kvq_config* cfg, int32_t H_q, kvq_layout_t* out);

/* Fill the RoPE table used by kvq_decode_attn for base `rope_theta` (> 0).
 * Passage: page 3, KVQuant "Pre-RoPE Key Quantization" (keys are cached
 * before the rotary embedding, which is applied to them after
 * dequantization); the table holds that rotation:
 * cos/sin of pos * theta^(-2i/D) (rotate-half pairs (i, i + D/2)), built in
 * binary64 on the device and stored as binary32, for every position the cache
 * can hold. Its contents are private to the library; build it once per
 * (cfg, theta) and reuse it for every decode call and layer of that shape.
 * Errors: KVQ_ERR_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_WORKSPACE (rope_bytes
 * too small), KVQ_ERR_CUDA. */
KVQ_API int kvq_rope_init(const kvq_config* cfg, double rope_theta, void* rope_tab, size_t rope_bytes,
                  void* stream);

/* Append n_new tokens per sequence at positions T_cur .. T_cur + n_new - 1
 * (KVQuant "Pre-RoPE Key Quantization": keys arrive before RoPE).
 *   k_new, v_new: fp16 [B][H_kv][n_new][D], contiguous.
 * Values are quantized per token at once (outliers, then per-group s, z,
 * codes). Keys are quantized per channel when their block of Bk tokens is
 * complete (KVQuant "Per-Channel Key Quantization"; keys of the block read so
 * far come back from K_TAIL); keys of an unfinished block are copied to
 * K_TAIL. One kernel launch covers every (b, h_kv, block) touched; an append
 * that completes the tail's block and also leaves a new unfinished block
 * copies that block's keys to K_TAIL in a second, small launch. On success
 * cache->T_cur += n_new (host field). n_new = 0 is a no-op.
 * Errors: KVQ_ERR_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CAPACITY, KVQ_ERR_CUDA. */
KVQ_API int kvq_append(const kvq_config* cfg, kvq_cache* cache, const void* k_new, const void* v_new,
               int32_t n_new, void* stream);

/* kvq_append with sliding-window key statistics (page mlqm.cn/news/1064729
 * ("UltraQuant ..."), §3.2 "时空自适应量化", sliding-window statistics: the
 * scale and zero follow the most recent `window` tokens instead of the whole
 * sequence). Values are quantized exactly as kvq_append quantizes them. When
 * a key block completes, its (s, z) per channel are the group parameters of
 * the channel's dense elements (outliers excluded) in the last `window`
 * tokens up to the block's end, tokens [max(0, t_end - window), t_end); the
 * block's codes, outliers and K_META entry are then those of kvq_append with
 * these (s, z). window = key_block gives exactly kvq_append's cache.
 *   window:  tokens, a positive multiple of key_block (1024 in the passage);
 *   k_bstat: device buffer of the size of K_META (layout bytes[KVQ_K_META]),
 *            caller-owned and kept with the cache: every finished key block's
 *            dense {min, max} per channel (fp16 pair; +inf / -inf when all of
 *            the channel's elements in the block are outliers), laid out like
 *            K_META. Every append to the cache must go through this call with
 *            the same window and buffer; decode reads the cache unchanged
 *            (kvq_decode_attn).
 * Two launches (statistics, then key codes), plus the deferred tail copy of
 * kvq_append when it applies. Errors: those of kvq_append; KVQ_ERR_ARG for a
 * NULL or misaligned k_bstat; KVQ_ERR_UNSUPPORTED for a bad window. */
KVQ_API int kvq_append_window(const kvq_config* cfg, kvq_cache* cache, const void* k_new, const void* v_new,
                              int32_t n_new, int32_t window, void* k_bstat, void* stream);

/* Decode attention of one query token per sequence over the T_cur cached
 * tokens (GQA: query head h reads kv head h / G, G = H_q / H_kv in
 * {1, 2, 4, 8}). Passages: page 3, Quanto "量化原理" step 3 (the cache is
 * dequantized as it is read) and KVQuant "Pre-RoPE Key Quantization" (RoPE
 * applied to the dequantized keys); the dense-and-sparse outliers of KVQuant
 * "Per-Vector Dense-and-Sparse Quantization" are restored on read.
 *   q:   fp16 [B][H_q][D], pre-RoPE, at position q_pos (0 <= q_pos < T_max);
 *   out: fp16 [B][H_q][D].
 * out_h = sum_t softmax_t(sm_scale * <RoPE(q_h, q_pos), RoPE(k_hat_t, t)>) v_hat_t
 * over t in [0, T_cur); k_hat, v_hat are the dequantized cache with outliers
 * restored, and tail keys are read as fp16. rope_tab = NULL applies no RoPE;
 * otherwise it is a table filled by kvq_rope_init for this cfg. The work is
 * split over T (flash-decode) into partial (max, sum, output) triples in
 * `workspace`, merged by a second kernel. Requires T_cur >= 1.
 * Errors: KVQ_ERR_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_WORKSPACE, KVQ_ERR_CUDA. */
KVQ_API int kvq_decode_attn(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t H_q,
                    int32_t q_pos, const void* rope_tab, float sm_scale, void* out,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Diagnostics of the bounded waits: kvq_decode_attn (head_dim 128) with every
 * ring stage's barrier armed for tx_pad bytes (a multiple of 16) more than its
 * copies deliver. With tx_pad > 0 no stage ever completes, so every wait
 * expires (each after one second of the GPU's global timer): the kernel sets
 * KVQ_STATUS_TIMEOUT in the workspace's status word, drains its copies
 * (bounded waits again), writes NaN partials and returns; a call takes a few
 * seconds. It exists to test the failure path without a fault (no page has a
 * counterpart); tx_pad = 0 gives kvq_decode_attn's results. Errors: those of
 * kvq_decode_attn; KVQ_ERR_UNSUPPORTED for head_dim 64 or a tx_pad that is
 * not a multiple of 16. */
KVQ_API int kvq_decode_attn_diag(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t H_q,
                                 int32_t q_pos, const void* rope_tab, float sm_scale, void* out,
                                 void* workspace, size_t workspace_bytes, uint32_t tx_pad, void* stream);

/* One decode step of one layer in a single stream-ordered call: append the
 * new token of every sequence, then attend its query over all cached tokens
 * including the new one (the serving workflow of mlqm.cn/news/1064729, §3.2
 * and §4.2: a token is quantized as it arrives, a key block once its last
 * token has arrived).
 *   k_new, v_new: fp16 [B][H_kv][1][D], the new token's pre-RoPE key and
 *                 value, stored at position T_cur exactly as kvq_append stores
 *                 it (the value quantized at once; the key kept fp16 in K_TAIL
 *                 until it completes its block, which is then quantized);
 *   q:            fp16 [B][H_q][D], pre-RoPE, at position T_cur (the new token);
 *   out:          fp16 [B][H_q][D], attention over positions 0 .. T_cur.
 * The other arguments are those of kvq_decode_attn. The result and the cache
 * are bit-identical to kvq_append(n_new = 1) followed by kvq_decode_attn with
 * q_pos = T_cur on the same stream, which is what this call enqueues (two or
 * three kernels, no synchronization). On success cache->T_cur += 1.
 * Errors: every check of both operations runs before the first launch:
 * KVQ_ERR_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CAPACITY (T_cur = T_max),
 * KVQ_ERR_WORKSPACE; then nothing is launched and nothing changes.
 * KVQ_ERR_CUDA from the append launch leaves T_cur unchanged; from the
 * attention launch the append is already enqueued, so T_cur has advanced. */
KVQ_API int kvq_decode_step(const kvq_config* cfg, kvq_cache* cache, const void* k_new, const void* v_new,
                            const void* q, int32_t H_q, const void* rope_tab, float sm_scale, void* out,
                            void* workspace, size_t workspace_bytes, void* stream);

/* kvq_decode_attn without a workspace argument, for callers that cannot
 * allocate device memory on the decode path: for example a serving engine
 * that reserves all device memory at start-up and forbids later cudaMalloc
 * calls, or a plain-C host that owns no device allocator from which to hand
 * over scratch. The pages have no counterpart; it is a convenience of this
 * library. Same arguments and errors as kvq_decode_attn. The results are
 * bit-identical to kvq_decode_attn's when the split limit below does not
 * bind; when it does, fewer T splits change the order of the fp32 merge and
 * the results agree within the decode tolerance (2e-3 max-abs, 1e-2
 * relative) instead.
 *   - Scratch: the split partials go to one file-scope device array of
 *     8 MiB that every GPU loading the library keeps until the process
 *     exits. No allocation or free happens in this call.
 *   - Limit: one T split needs B * H_q * (D + 2) * 4 bytes. The call uses at
 *     most 8 MiB / that many splits (at most 256); a shape whose single split
 *     exceeds 8 MiB is rejected with KVQ_ERR_WORKSPACE. Fewer splits can make
 *     it slower than kvq_decode_attn on very wide batches.
 *   - Set-up: the first call on each device looks up the array's device
 *     address with that device current (and again after the device gets a
 *     new context, e.g. after cudaDeviceReset); make that first call before
 *     any stream capture on the device.
 *   - Sharing: every call uses the same array. Each call writes every entry
 *     it later reads, so nothing has to be cleared between calls, but calls
 *     whose kernels overlap on the GPU (different streams, or different host
 *     threads) race on the array and give wrong results. */
KVQ_API int kvq_decode_attn_noalloc(const kvq_config* cfg, const kvq_cache* cache, const void* q,
                                    int32_t H_q, int32_t q_pos, const void* rope_tab,
                                    float sm_scale, void* out, void* stream);

/* ---- Paged, ragged batches (continuous batching; mlqm.cn/news/1002276 §5.2-5.3
 * name continuous batching and PagedAttention as the serving setting of a
 * quantized cache). The sequences of a batch hold different numbers of
 * tokens and share pools of physical key blocks through a block table.
 * Each physical block holds Bk consecutive tokens of one sequence for all
 * H_kv heads, encoded exactly as in the contiguous cache:
 *   K_CODES [n_blocks][H_kv][Bk][D*bits/8]   K_META [n_blocks][H_kv][D][2]
 *   K_OUTL  [n_blocks][H_kv][Bk][n_out][2]   V_CODES [n_blocks][H_kv][Bk][D*bits/8]
 *   V_META  [n_blocks][H_kv][Bk][D/Gv][2]    V_OUTL  [n_blocks][H_kv][Bk][n_out][2]
 *   K_TAIL  [B][H_kv][Bk][D]                 fp16 keys of each sequence's unfinished block
 * For these calls kvq_config.B is the number of sequences (rows of the block
 * table) and T_max the capacity of one sequence (block-table row length
 * T_max / Bk). Token t of sequence b lives in physical block
 * block_table[b][t / Bk], row t % Bk. The caller owns the pools and the
 * table and hands out the blocks (any physical block may serve any
 * sequence); a table entry outside [0, n_blocks) is clamped into the pool,
 * which keeps every access in bounds but gives undefined values. */
typedef struct kvq_paged_cache {
  void* k_codes;                /* pools, layouts above */
  void* k_meta;
  void* k_tail;
  void* k_outl;                 /* may be NULL when n_out = 0 */
  void* v_codes;
  void* v_meta;
  void* v_outl;                 /* may be NULL when n_out = 0 */
  const int32_t* block_table;   /* device [B][T_max / Bk] */
  int32_t* seq_len;             /* device [B]: tokens stored per sequence */
  int32_t n_blocks;             /* physical blocks in each pool */
  int32_t max_len;              /* host: an upper bound of every seq_len[b] (sizes the grids) */
} kvq_paged_cache;

/* Sizes of a paged cache (passage: the paged serving setting of
 * mlqm.cn/news/1002276 §5.2-5.3, with the memory formula of its §2.1 giving
 * fp16_equiv_bytes): the pools for n_blocks physical blocks (bytes[]), per physical
 * block for the pools and per sequence for K_TAIL (stream_bytes[]), and the
 * decode workspace for H_q query heads. fp16_equiv_bytes is the fp16 K and V
 * of the pools' capacity. Host-only and pure.
 * Errors: KVQ_ERR_ARG (NULL), KVQ_ERR_UNSUPPORTED (cfg, H_q, n_blocks < 1 or
 * n_blocks * H_kv >= 2^31). */
KVQ_API int kvq_paged_layout(const kvq_config* cfg, int32_t n_blocks, int32_t H_q, kvq_layout_t* out);

/* kvq_append for a paged cache: n_new tokens for every sequence b, stored at
 * positions seq_len[b] .. seq_len[b] + n_new - 1 (each sequence at its own
 * position, read on the device), with the same encoding as kvq_append; then
 * seq_len[b] += n_new on the device, stream-ordered after the stores, and
 * cache->max_len += n_new. The blocks those positions fall in must already be
 * in the block table. A single sequence can be appended alone by passing
 * B = 1 and pointers to its table row, seq_len entry and K_TAIL stream.
 *   k_new, v_new: fp16 [B][H_kv][n_new][D].
 * Errors: KVQ_ERR_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CAPACITY
 * (max_len + n_new > T_max), KVQ_ERR_CUDA. */
KVQ_API int kvq_paged_append(const kvq_config* cfg, kvq_paged_cache* cache, const void* k_new,
                             const void* v_new, int32_t n_new, void* stream);

/* kvq_decode_attn for a paged cache: sequence b attends over its own
 * seq_len[b] tokens with its query at position seq_len[b] - 1 (the newest
 * token); a sequence with no tokens gets out = 0. Other arguments and the
 * workspace size (kvq_paged_layout or kvq_layout of the same cfg) as for
 * kvq_decode_attn. Errors: KVQ_ERR_ARG, KVQ_ERR_UNSUPPORTED,
 * KVQ_ERR_WORKSPACE, KVQ_ERR_CUDA. */
KVQ_API int kvq_paged_decode_attn(const kvq_config* cfg, const kvq_paged_cache* cache, const void* q,
                                  int32_t H_q, const void* rope_tab, float sm_scale, void* out,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* ---- Non-uniform codes (page 3, KVQuant "Non-Uniform KV Cache Quantization":
 * a calibrated format instead of the uniform grid). A level table holds
 * 2^bits binary32 levels 0 = l_0 < l_1 < ... < l_L = 1 on a group's
 * normalized range. Groups, outliers, buffers and packing are those of
 * kvq_append; per group the scale's slot holds the range
 * r = fp16_round_up(fp32(max) - fp32(min)) of the dense elements, the code of
 * x is the nearest level of u = fp32(fp32(x - z) / r) (the number of binary32
 * midpoints fp32(0.5 (l_k + l_k+1)) below u, ties to the lower level; r = 0
 * gives 0), and x_hat = z + r * l_code. These calls run CUDA-core kernels for
 * caches filled in whole key blocks (no fp16 tail). */

/* Level table (page 3, KVQuant "Non-Uniform KV Cache Quantization": the
 * format is calibrated offline) of 2^bits levels fitted to calibration samples u[0..n) in
 * [0, 1] (normalized dense values, e.g. (x - min) / (max - min) of groups of
 * representative keys or values): one-dimensional k-means (Lloyd) started
 * from the uniform grid k / L, with the end levels held at 0 and 1; a level
 * whose cell is empty stays. Host memory only; touches no device.
 * Errors: KVQ_ERR_ARG (NULL, iters < 0, a sample outside [0, 1]),
 * KVQ_ERR_UNSUPPORTED (bits not in {2, 3, 4, 8}). */
KVQ_API int kvq_fit_levels(const double* u, size_t n, int32_t bits, int32_t iters, float* levels);

/* kvq_append with non-uniform codes (page 3, KVQuant "Non-Uniform KV Cache
 * Quantization"). levels: host pointer to the 2^bits levels of the table
 * (copied into the launch). Any T_cur and n_new, as kvq_append: the keys of an
 * unfinished key block wait as fp16 in K_TAIL and are coded when the block
 * completes; values are coded at once. Errors: those of kvq_append;
 * KVQ_ERR_ARG for a table that does not start at 0, end at 1 and increase. */
KVQ_API int kvq_append_levels(const kvq_config* cfg, kvq_cache* cache, const void* k_new, const void* v_new,
                              int32_t n_new, const float* levels, void* stream);

/* kvq_decode_attn over a cache appended with kvq_append_levels and the same
 * table (page 3, KVQuant "Non-Uniform KV Cache Quantization": x_hat = z + r *
 * l_code on read; any T_cur, the keys of an unfinished block from K_TAIL).
 * head_dim 128 takes the tensor-core kernel (levels as fp16 operands; the
 * workspace then carries the status word of kvq_decode_attn), head_dim 64 and
 * KVQ_FLAG_PRECISE_SCORES the fp32 CUDA-core kernel. Errors: those of
 * kvq_decode_attn; KVQ_ERR_ARG for a bad table. */
KVQ_API int kvq_decode_attn_levels(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t H_q,
                                   int32_t q_pos, const void* rope_tab, float sm_scale, void* out,
                                   void* workspace, size_t workspace_bytes, const float* levels, void* stream);

/* kvq_decode_step for a level-table cache (page 3, KVQuant "Non-Uniform KV
 * Cache Quantization", in the serving workflow of mlqm.cn/news/1064729, §3.2
 * and §4.2): kvq_append_levels of the new token (n_new = 1), then
 * kvq_decode_attn_levels of q at its position T_cur, on one stream, with the
 * same table (levels: host pointer to the 2^bits levels, copied into the
 * launches). Arguments, results, ownership and the T_cur update are those of
 * kvq_decode_step; the result and the cache are bit-identical to the two
 * calls. Errors: those of kvq_decode_step, plus KVQ_ERR_ARG for a table that
 * does not start at 0, end at 1 and increase (checked before any launch). */
KVQ_API int kvq_decode_step_levels(const kvq_config* cfg, kvq_cache* cache, const void* k_new, const void* v_new,
                                   const void* q, int32_t H_q, const void* rope_tab, float sm_scale, void* out,
                                   void* workspace, size_t workspace_bytes, const float* levels, void* stream);

/* Static, human-readable name of a status code (a utility of this library;
 * no passage). */
KVQ_API const char* kvq_status_string(int status);

/* Library version, e.g. "kvq 0.1.0 sm_103a" (a utility; no passage). */
KVQ_API const char* kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
