/*
 * tq.h -- C ABI of the TurboQuant compressed KV-cache library for GB300 (sm_103a).
 *
 * Method sources (cited by page title and section):
 *  [README] "SwiftLM" (nomorevibe.com/p/swiftlm), section "TurboQuantization:
 *           KV Cache Compression" -> "The Algorithm": K-Cache steps 1-5
 *           (4.25 bits/dim) and the V-Cache paragraph (3.125 bits/dim).
 *  [ART]    "SwiftLM ... Swift製LLM推論サーバー" (lilting.ch): "Lloyd-Maxコードブックとは"
 *           (8 levels for N(0,1/d), computed once before inference), "KVキャッシュ圧縮の内訳",
 *           "Walsh-Hadamard Transform（WHT）の役割".
 *  [VLLM]   "論文解説: vLLM-MLX" (0h-n0.github.io), "Paged KVキャッシュ": fixed-size
 *           blocks addressed through a block table.
 *
 * Conventions shared by every entry point
 *  - head_dim d is 128 or 256; a paged block holds TQ_BLOCK_SIZE (16) token slots.
 *  - Device pointers are plain CUDA device addresses owned by the caller; the
 *    library allocates nothing and keeps no state between calls.
 *  - Every call is asynchronous and ordered on `stream` (a cudaStream_t; NULL =
 *    legacy default stream), except tq_codebook_init, which synchronises it.
 *  - Return value: TQ_OK (0) or a negative TQ_ERR_* code.  All argument errors
 *    are detected on the host before anything is launched.  Errors the host
 *    cannot see (a block id or slot outside the pool) are reported by the
 *    kernels in the optional device word `status` (bitwise OR of TQ_STATUS_*);
 *    the offending element is skipped, never trapped.
 *  - A K pool is uint8[num_blocks][n_kv_heads][tq_k_record_bytes(d)], a V pool
 *    uint8[num_blocks][n_kv_heads][tq_v_record_bytes(d)]; both 16-byte aligned.
 *    A record packs the 16 slots of one block for one kv head: three bit-planes
 *    of the 3-bit Lloyd-Max cell index (plus, for K, one plane of QJL sign bits),
 *    followed by fp16 norms (K: ||x|| and ||r|| per slot; V: ||v|| per slot).
 *  - A slot index is block * 16 + offset.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *tq_stream_t;   /* identical to cudaStream_t */

#define TQ_BLOCK_SIZE 16

enum {
    TQ_OK = 0,
    TQ_ERR_INVALID = -1,        /* a size or count out of range, or a NULL required pointer */
    TQ_ERR_HEAD_DIM = -2,       /* d is not 128 or 256 */
    TQ_ERR_GQA = -3,            /* n_q_heads is not a multiple of n_kv_heads, or group > 8 */
    TQ_ERR_WORKSPACE = -4,      /* workspace or params buffer too small */
    TQ_ERR_CUDA = -5,           /* a CUDA runtime call or kernel launch failed */
    TQ_ERR_DTYPE = -6,          /* dtype is not TQ_DTYPE_F32 or TQ_DTYPE_BF16 */
    TQ_ERR_ALIGN = -7           /* a pool, params or workspace pointer is not 16-byte aligned */
};

enum { TQ_DTYPE_F32 = 0, TQ_DTYPE_BF16 = 1 };

enum {
    TQ_STATUS_BAD_SLOT = 1,     /* a slot or block id outside [0, num_blocks) was skipped */
    TQ_STATUS_BAD_PARAMS = 2,   /* the params buffer was not initialised for this d */
    TQ_STATUS_TIMEOUT = 4       /* a device-side wait gave up (bounded); the call's output is invalid */
};

/* Bytes of one packed record (16 slots, one kv head).
 * d=128: K 1088 (= 4.25 bits/dim), V 800 (= 3.125 bits/dim).
 * d=256: K 2112 (4.125 bits/dim), V 1568 (3.0625 bits/dim).  0 for another d. */
size_t tq_k_record_bytes(int d);
size_t tq_v_record_bytes(int d);

/* Size of the device params buffer for head_dim d (0 for an unsupported d). */
size_t tq_params_bytes(int d);

/* tq_codebook_init -- build the device params for head_dim d.
 * [ART "Lloyd-Maxコードブックとは": the 8-level Lloyd-Max codebook of the
 * Gaussian is computed once, before inference, with no calibration data;
 * README K-Cache steps 2 and 5: the random WHT signs and the QJL matrix.]
 *   D_host      host int8[d], the rotation's random sign diagonal (+1/-1).
 *   S_host      host float[d*d], the QJL Gaussian matrix, row-major (row k
 *               produces sign bit k).  It is held at binary16 precision: each
 *               entry is rounded to the nearest binary16 value (ties to even), and
 *               every call uses the rounded matrix.
 *   params_dev  device buffer of >= tq_params_bytes(d) bytes, 16-byte aligned.
 *   centroids_out8  optional host double[8]: the codebook (unit variance).
 * The codebook is solved on the host in fp64 (fixed-point Lloyd-Max, once per
 * process), stored in fp32 with its fp16 lookup tables.  Copies D and S to the
 * device and derives the tables the kernels use (S transposed, the QJL offset
 * weights).  Synchronises `stream`.  Errors: TQ_ERR_HEAD_DIM, TQ_ERR_INVALID (NULL
 * or a D entry not +-1), TQ_ERR_WORKSPACE, TQ_ERR_ALIGN, TQ_ERR_CUDA. */
int tq_codebook_init(int d, const int8_t *D_host, const float *S_host, void *params_dev,
                     size_t params_bytes, double *centroids_out8, tq_stream_t stream);

/* tq_encode_k -- compress keys into a paged K pool.
 * [README K-Cache steps 1-5; ART "KVキャッシュ圧縮の内訳" steps 1-5]
 * For every (token, kv head) vector x (length d): n = ||x||; y = Pi (x/n) with
 * Pi = H diag(D)/sqrt(d); cell_i = number of Lloyd-Max thresholds <= sqrt(d) y_i;
 * r = y - c[cell]/sqrt(d); gamma = ||r||; sign bit k = [(S r)_k >= 0].
 * Stores cells, sign bits, fp16(n), fp16(gamma) at slot slot_mapping[token].
 *   params        device params of head_dim d (tq_codebook_init).
 *   k             device [n_tokens][n_kv_heads][d], dtype TQ_DTYPE_F32 or _BF16, contiguous.
 *   slot_mapping  device int64[n_tokens]; a slot outside the pool is skipped
 *                 and flagged TQ_STATUS_BAD_SLOT; a negative slot is skipped silently
 *                 (padding).
 *   k_pool        device K pool with num_blocks blocks.
 *   status        optional device int32 (may be NULL).
 * n_tokens == 0 is a no-op.  Errors: TQ_ERR_INVALID, TQ_ERR_HEAD_DIM,
 * TQ_ERR_DTYPE, TQ_ERR_ALIGN, TQ_ERR_CUDA. */
int tq_encode_k(const void *params, int d, const void *k, int dtype, int64_t n_tokens,
                int n_kv_heads, const int64_t *slot_mapping, void *k_pool, int64_t num_blocks,
                int32_t *status, tq_stream_t stream);

/* tq_encode_v -- compress values into a paged V pool: steps 1-3 only, no
 * residual and no QJL [README V-Cache paragraph; ART "KVキャッシュ圧縮の内訳", V].
 * Stores cells and fp16(||v||).  Arguments and errors as tq_encode_k. */
int tq_encode_v(const void *params, int d, const void *v, int dtype, int64_t n_tokens,
                int n_kv_heads, const int64_t *slot_mapping, void *v_pool, int64_t num_blocks,
                int32_t *status, tq_stream_t stream);

/* tq_paged_append -- encode one new token per sequence into its next slot.
 * [VLLM "Paged KVキャッシュ"; README K-Cache and V-Cache]
 * For sequence b the slot is block_table[b][ctx_lens[b]/16]*16 + ctx_lens[b]%16,
 * i.e. ctx_lens holds the lengths BEFORE the append (the library does not
 * update them).
 *   k_new, v_new  device [batch][n_kv_heads][d] in dtype.
 *   block_table   device int32[batch][max_blocks].
 *   ctx_lens      device int32[batch]; a sequence with ctx_lens[b] < 0 is skipped,
 *                 one whose slot falls outside its table or the pool is flagged
 *                 TQ_STATUS_BAD_SLOT and skipped.
 * Every byte of a record belongs to one slot, so sequences may share a block;
 * two sequences appending into the same slot race.  One kernel launch.
 * Errors: as tq_encode_k. */
int tq_paged_append(const void *params, int d, const void *k_new, const void *v_new, int dtype,
                    int batch, int n_kv_heads, const int32_t *block_table, int max_blocks,
                    const int32_t *ctx_lens, void *k_pool, void *v_pool, int64_t num_blocks,
                    int32_t *status, tq_stream_t stream);

/* tq_dequant_k / tq_dequant_v -- dense vectors of whole paged blocks, for a prefill (or any
 * dense attention) over a compressed prefix.  [README "TurboQuantization: KV Cache
 * Compression" -> "The Algorithm": the codebook value of each rotated coordinate, plus for K
 * the QJL estimate of the residual; README "Throughput & Inference Memory Profile": prompts
 * are processed in chunks (chunked prefill), each chunk attending the cached prefix]
 * For j < n_ids, slot t < 16 of block block_ids[j] and kv head h:
 *   K: out[16 j + t][h] = n  Pi^T ( c[cell]/sqrt d + sqrt(pi/2)/d gamma S^T (2 sign - 1) )
 *   V: out[16 j + t][h] = nv Pi^T ( c[cell]/sqrt d ),          Pi^T y = D (H y) / sqrt d,
 * so that q . out_K / sqrt d is exactly the score tq_decode_attn computes and a softmax over
 * these vectors is exactly its attention.
 *   block_ids  device int32[n_ids]; an id outside [0, num_blocks) gives zeros for its 16 rows
 *              and sets TQ_STATUS_BAD_SLOT in *status.
 *   out        device [n_ids * 16][n_kv_heads][d] in out_dtype (TQ_DTYPE_F32 or TQ_DTYPE_BF16,
 *              rounded to nearest even).  Slots never written hold whatever the pool held.
 * Errors: TQ_ERR_HEAD_DIM, TQ_ERR_DTYPE, TQ_ERR_INVALID (also n_ids > 0 with num_blocks = 0),
 * TQ_ERR_ALIGN, TQ_ERR_CUDA. */
int tq_dequant_k(const void *params, int d, const void *k_pool, int64_t num_blocks, int n_kv_heads,
                 const int32_t *block_ids, int n_ids, void *out, int out_dtype, int32_t *status,
                 tq_stream_t stream);
int tq_dequant_v(const void *params, int d, const void *v_pool, int64_t num_blocks, int n_kv_heads,
                 const int32_t *block_ids, int n_ids, void *out, int out_dtype, int32_t *status,
                 tq_stream_t stream);

/* Workspace bytes tq_decode_attn needs for this shape (0 for invalid sizes).
 * It depends on d, batch and n_q_heads only (max_ctx is checked, not used). */
size_t tq_decode_workspace_bytes(int d, int batch, int n_q_heads, int max_ctx);

/* tq_decode_attn -- one decode step of attention over the compressed paged cache.
 * [README "The Algorithm" (fused dequantisation inside attention);
 *  VLLM "Paged KVキャッシュ"]
 * For query head h of sequence b (kv head h / (n_q_heads/n_kv_heads)), over the
 * ctx_lens[b] cached tokens (token j in block block_table[b][j/16], slot j%16):
 *   qbar = Pi q,  u = S qbar,
 *   s_j  = (n_j/sqrt d) ( <qbar, c[cell_j]>/sqrt d + gamma_j sqrt(pi/2)/d <u, 2 sign_j - 1> ),
 *   P    = softmax(s),  a = sum_j P_j nv_j c[vcell_j]/sqrt d,  out = Pi^T a.
 * The scores are computed in the rotated domain, so no key or value is
 * reconstructed; one inverse rotation per (b, h) is applied at the end.
 *   q          device [batch][n_q_heads][d] in dtype.
 *   ctx_lens   device int32[batch]; each must be <= max_ctx (larger values are
 *              clamped to max_ctx); 0 gives out = 0.
 *   max_ctx    host upper bound of ctx_lens (larger lengths are clamped to it).
 *   out        device float[batch][n_q_heads][d].
 *   workspace  device scratch of >= tq_decode_workspace_bytes(...) bytes.
 * n_q_heads/n_kv_heads must be 1..8.  Errors: TQ_ERR_INVALID, TQ_ERR_HEAD_DIM,
 * TQ_ERR_GQA, TQ_ERR_DTYPE, TQ_ERR_WORKSPACE, TQ_ERR_ALIGN, TQ_ERR_CUDA. */
int tq_decode_attn(const void *params, int d, const void *q, int dtype, int batch, int n_q_heads,
                   int n_kv_heads, const void *k_pool, const void *v_pool, int64_t num_blocks,
                   const int32_t *block_table, int max_blocks, const int32_t *ctx_lens,
                   int max_ctx, float *out, void *workspace, size_t workspace_bytes,
                   int32_t *status, tq_stream_t stream);

/* The two stages of tq_decode_attn as separate calls, for callers that
 * schedule or time them individually.  Called in this order on one stream with
 * the same shape arguments, ctx_lens contents and workspace, they compute
 * exactly what tq_decode_attn computes; argument meanings and errors are as
 * there.
 *   tq_decode_qprep   qbar = Pi q and u = S qbar for every (sequence, query head),
 *                     written to the workspace as tensor-core operands (ctx_lens and
 *                     max_ctx are checked as by tq_decode_attn; the prep reads neither).
 *   tq_decode_splitk  the pass over the cache.  The context of each (sequence,
 *                     kv head) is cut into chunks of 128 tokens; the chunks of all (sequence,
 *                     kv head) pairs, in that order, are shared out in equal
 *                     contiguous ranges among a fixed set of resident CTAs, each of
 *                     which works out its range from ctx_lens.  A pair whose chunks
 *                     span several CTAs is combined from their online-softmax states
 *                     by a merge kernel after the pass; each pair writes
 *                     out = Pi^T a for its query heads. */
int tq_decode_qprep(const void *params, int d, const void *q, int dtype, int batch, int n_q_heads,
                    int n_kv_heads, const int32_t *ctx_lens, int max_ctx, void *workspace,
                    size_t workspace_bytes, tq_stream_t stream);
int tq_decode_splitk(const void *params, int d, int batch, int n_q_heads, int n_kv_heads,
                     const void *k_pool, const void *v_pool, int64_t num_blocks,
                     const int32_t *block_table, int max_blocks, const int32_t *ctx_lens,
                     int max_ctx, float *out, void *workspace, size_t workspace_bytes,
                     int32_t *status, tq_stream_t stream);

/* tq_decode_step -- one decode step: append one token per sequence, then attend.
 * [VLLM "Paged KVキャッシュ" (the slot of the new token); README "The Algorithm" (its
 *  encoding); then tq_decode_attn over the grown cache]
 * For each sequence b with pre_lens[b] >= 0: K and V of the new token (k_new[b], v_new[b])
 * are encoded into the slot of position pre_lens[b] (as tq_paged_append), and query head h
 * of sequence b attends the pre_lens[b] + 1 tokens (as tq_decode_attn, clamped to
 * max_ctx).  A sequence with pre_lens[b] < 0 appends nothing and gets out = 0.
 * The append and the query preparation run in one launch, followed by the split-K pass and
 * its merge (three launches); the result equals tq_paged_append followed by tq_decode_attn
 * with ctx_lens = pre_lens + 1, bit for bit.
 *   k_new, v_new  device [batch][n_kv_heads][d] in dtype;  q  device [batch][n_q_heads][d].
 *   pre_lens      device int32[batch].
 *   workspace     >= tq_decode_workspace_bytes(d, batch, n_q_heads, max_ctx) bytes.
 * Errors: as tq_paged_append and tq_decode_attn. */
int tq_decode_step(const void *params, int d, const void *k_new, const void *v_new, const void *q, int dtype,
                   int batch, int n_q_heads, int n_kv_heads, const int32_t *block_table, int max_blocks,
                   const int32_t *pre_lens, int max_ctx, void *k_pool, void *v_pool, int64_t num_blocks,
                   float *out, void *workspace, size_t workspace_bytes, int32_t *status,
                   tq_stream_t stream);

/* Multi-query decode: q_len new tokens per sequence are verified in one pass over the
 * cache (speculative or multi-token-prediction decoding), so the compressed records are
 * read once for all of them.  [README "Performance: MTP Speculative Decoding", key
 * takeaways: a verification batch of several draft tokens shares one read of the KV
 * cache; the attention of each query is that of tq_decode_attn]
 * The q_len tokens are the last q_len of the ctx_lens[b] cached tokens, and query i
 * (0-based) sees the tokens up to itself (causal): it attends the first
 * ctx_lens[b] - (q_len - 1 - i) tokens (none if that is <= 0; ctx_lens[b] is clamped to
 * max_ctx first).  Otherwise each query is exactly tq_decode_attn's.
 *   q, out     device [batch][q_len][n_q_heads][d] (q in dtype, out fp32).
 *   workspace  >= tq_decode_workspace_bytes_mq(d, batch, q_len, n_q_heads, max_ctx) bytes.
 * q_len * n_q_heads / n_kv_heads must be <= 8 (TQ_ERR_GQA otherwise); q_len = 1 is
 * tq_decode_attn.  Other arguments and errors as tq_decode_attn. */
size_t tq_decode_workspace_bytes_mq(int d, int batch, int q_len, int n_q_heads, int max_ctx);
int tq_decode_attn_mq(const void *params, int d, const void *q, int dtype, int batch, int q_len,
                      int n_q_heads, int n_kv_heads, const void *k_pool, const void *v_pool,
                      int64_t num_blocks, const int32_t *block_table, int max_blocks,
                      const int32_t *ctx_lens, int max_ctx, float *out, void *workspace,
                      size_t workspace_bytes, int32_t *status, tq_stream_t stream);

/* tq_decode_step_mq -- tq_decode_step for q_len tokens per sequence: K and V of token i
 * (k_new[b][i], v_new[b][i], device [batch][q_len][n_kv_heads][d]) are encoded into the slot
 * of position pre_lens[b] + i, then the q_len queries attend as in tq_decode_attn_mq with
 * ctx_lens = pre_lens + q_len (query i sees pre_lens[b] + 1 + i tokens).  A sequence with
 * pre_lens[b] < 0 appends nothing and gets out = 0.  One launch for the append and the query
 * preparation, one for the pass, one for its merge; the result equals tq_paged_append of each
 * token followed by tq_decode_attn_mq.  Errors as tq_decode_step and tq_decode_attn_mq. */
int tq_decode_step_mq(const void *params, int d, const void *k_new, const void *v_new, const void *q,
                      int dtype, int batch, int q_len, int n_q_heads, int n_kv_heads,
                      const int32_t *block_table, int max_blocks, const int32_t *pre_lens, int max_ctx,
                      void *k_pool, void *v_pool, int64_t num_blocks, float *out, void *workspace,
                      size_t workspace_bytes, int32_t *status, tq_stream_t stream);

/* tq_decode_attn_hybrid -- decode attention over a hybrid cache: the compressed paged history
 * plus a window of recent tokens kept uncompressed, in one softmax.  [README: compression
 * starts past 2048 tokens ("--turbo-kv" in the options table, "After 2048 tokens" in the
 * kv_bits / --turbo-kv comparison), and attention covers the recent hot window together with
 * the compressed history (the "--turbo-kv long-range recall" note)]
 * For query head h of sequence b the attended set is the ctx_lens[b] compressed tokens (scored
 * as in tq_decode_attn) and the win_lens[b] window tokens j < win_lens[b] (row
 * win_k[b][j][kv head], scored q . k / sqrt d in the original domain); out = sum_j P_j v_j
 * over both, with one softmax P.  Window slots are an unordered set, so a ring buffer of the
 * most recent tokens can be passed as it is.
 *   win_k, win_v  device [batch][win_cap][n_kv_heads][d] in win_dtype (TQ_DTYPE_F32 or
 *                 TQ_DTYPE_BF16); win_lens device int32[batch], clamped to [0, win_cap].
 *   workspace     >= tq_decode_workspace_bytes_hybrid(d, batch, n_q_heads, max_ctx, win_cap).
 * Other arguments and errors as tq_decode_attn; win_cap = 0 is tq_decode_attn. */
size_t tq_decode_workspace_bytes_hybrid(int d, int batch, int n_q_heads, int max_ctx, int win_cap);
int tq_decode_attn_hybrid(const void *params, int d, const void *q, int dtype, int batch, int n_q_heads,
                          int n_kv_heads, const void *k_pool, const void *v_pool, int64_t num_blocks,
                          const int32_t *block_table, int max_blocks, const int32_t *ctx_lens, int max_ctx,
                          const void *win_k, const void *win_v, int win_dtype, int win_cap,
                          const int32_t *win_lens, float *out, void *workspace, size_t workspace_bytes,
                          int32_t *status, tq_stream_t stream);

/* tq_hybrid_append -- one new token per sequence into a hybrid cache, compressing the oldest
 * window token once the window is full.  [README, "TurboQuantization: KV Cache Compression":
 * its options table and its kv_bits / --turbo-kv comparison put the start of compression at
 * 2048 tokens; the most recent tokens stay uncompressed and older ones are compressed]
 * Window layout: token p of sequence b, while uncompressed, sits in window slot p mod win_cap.
 * Tokens 0 .. ctx_lens[b] - 1 are in the compressed paged history and tokens ctx_lens[b] ..
 * ctx_lens[b] + win_lens[b] - 1 in the window, so the window fills slots 0, 1, ... first and,
 * once full, every appended token takes the slot of the oldest one.  For each sequence:
 *   - win_lens[b] == win_cap: the window token at position ctx_lens[b] (slot ctx_lens[b] mod
 *     win_cap) is encoded (K and V, every kv head, as tq_paged_append) into the paged pools at
 *     history position ctx_lens[b] through block_table; ctx_lens[b] += 1; the new token takes
 *     the freed slot;
 *   - win_lens[b] < win_cap: the new token goes into slot win_lens[b]; win_lens[b] += 1.
 * The result is the cache tq_decode_attn_hybrid reads (its window slots 0 .. win_lens[b] - 1).
 *   k_new, v_new  device [batch][n_kv_heads][d] in dtype (TQ_DTYPE_F32 or TQ_DTYPE_BF16);
 *   win_k, win_v  device [batch][win_cap][n_kv_heads][d], the same dtype;
 *   win_lens, ctx_lens  device int32[batch], read and updated in place;
 *   scratch       device, >= tq_hybrid_append_scratch_bytes(d, batch, n_kv_heads, dtype)
 *                 bytes (the leaving rows and their positions), overwritten.
 * A sequence whose state is not one this call produces (win_lens outside [0, win_cap],
 * ctx_lens < 0, or a window that is not full while ctx_lens[b] mod win_cap != 0) is left
 * unchanged and sets TQ_STATUS_BAD_SLOT; so is a full window whose leaving token's history
 * position ctx_lens[b] has no valid block (past max_blocks, or a block id outside
 * [0, num_blocks)): nothing moves and neither length changes.
 * Two launches on the stream: the window step (the leaving rows copied to scratch, the new token
 * written, the lengths updated), then the encode of the leaving rows.
 * Errors: TQ_ERR_HEAD_DIM, TQ_ERR_DTYPE, TQ_ERR_INVALID (win_cap <= 0 among others),
 * TQ_ERR_ALIGN (every buffer 16-byte aligned), TQ_ERR_WORKSPACE (scratch too small),
 * TQ_ERR_CUDA. */
size_t tq_hybrid_append_scratch_bytes(int d, int batch, int n_kv_heads, int dtype);
int tq_hybrid_append(const void *params, int d, const void *k_new, const void *v_new, int dtype, int batch,
                     int n_kv_heads, void *win_k, void *win_v, int win_cap, int32_t *win_lens,
                     const int32_t *block_table, int max_blocks, int32_t *ctx_lens, void *k_pool, void *v_pool,
                     int64_t num_blocks, void *scratch, size_t scratch_bytes, int32_t *status, tq_stream_t stream);

/* tq_selftest_wait_timeout -- check of the library's bounded device waits.  The pages have no
 * counterpart to this call.  The bulk encode and dequantisation kernels wait on mbarriers for
 * their tile copies and tensor-core results; every such wait gives up after about 0.5 s, sets
 * TQ_STATUS_TIMEOUT and lets the kernel finish, so a lost arrival can never hang the GPU.  This
 * call launches one CTA that runs the same wait on an mbarrier nothing arrives at: after about
 * 0.5 s it ORs TQ_STATUS_TIMEOUT into the device word *status (required) and exits normally.
 * Errors: TQ_ERR_INVALID (status NULL), TQ_ERR_CUDA. */
int tq_selftest_wait_timeout(int32_t *status, tq_stream_t stream);

/* tq_decode_attn_noalloc -- tq_decode_attn without a caller workspace.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory when they decode: a serving runtime that
 * reserves all free GPU memory for its KV pool at start-up and allows no
 * allocation afterwards, or a latency-bound decode loop that must not call
 * cudaMalloc, which can synchronise the device.
 * Same arguments, result and errors as tq_decode_attn, minus workspace and
 * workspace_bytes.  The scratch is a fixed array of TQ_NOALLOC_SCRATCH_BYTES
 * (16 MiB) compiled into the library; every GPU that loads the library keeps
 * it until the process exits.  A shape whose tq_decode_workspace_bytes()
 * exceeds it is rejected with TQ_ERR_WORKSPACE (16 x 32 query heads at
 * d = 128 need about 8.0 MiB; 64 x 32 need 20.4 MiB).  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library call.
 * The scratch used is that of the device current at the call; the stream must
 * belong to it.  The first call made with a device current looks up the
 * scratch address on that device (cudaGetSymbolAddress); make that first call
 * before any stream capture.  All calls share the one array per device: two
 * calls whose kernels overlap on the GPU (different streams, no ordering) race
 * and corrupt each other's results.  No part of the scratch needs to start at
 * zero, so nothing is cleared between calls. */
#define TQ_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int tq_decode_attn_noalloc(const void *params, int d, const void *q, int dtype, int batch,
                           int n_q_heads, int n_kv_heads, const void *k_pool, const void *v_pool,
                           int64_t num_blocks, const int32_t *block_table, int max_blocks,
                           const int32_t *ctx_lens, int max_ctx, float *out, int32_t *status,
                           tq_stream_t stream);

/* ---- Group-quantised KV cache: the fidelity comparator beside TurboQuant.
 * [README "Per-Request API Parameters": kv_bits (4 or 8) selects MLX-native standard group
 *  quantization of the KV cache from token 0, kv_group_size its group (default 64), "~2-4x vs
 *  FP16"; ART "TurboQuant V2+V3ハイブリッド実装": the V2 route, linear affine quantization.]
 * For each group of `group` consecutive coordinates of a (token, kv head) vector x:
 *   scale = fp16((max - min) / (2^bits - 1)),  bias = fp16(min),
 *   code_i = clamp(rint((x_i - bias) / scale), 0, 2^bits - 1)   (0 when scale is 0),
 * every step in fp32 with round-to-nearest-even; the decoded coordinate is scale * code + bias.
 * K and V use the same format (no rotation, no QJL).  Supported: d 128 or 256, bits 4 or 8,
 * group 32, 64 or 128.
 * Record of one (block, kv head), tq_gq_record_bytes(d, bits, group) bytes:
 *   codes  [16 slots][d * bits / 8]  4-bit: coordinate 2j in the low nibble of byte j
 *   params [16 slots][d / group][2]  fp16 scale, fp16 bias
 * At d = 128, group 64: 1152 B (4.5 bits/dim) at 4 bits, 2176 B (8.5 bits/dim) at 8 bits.
 * 0 for an unsupported combination. */
size_t tq_gq_record_bytes(int d, int bits, int group);

/* tq_gq_encode -- quantise x [n_tokens][n_kv_heads][d] (dtype, contiguous, 16-byte aligned)
 * into slot slot_mapping[token] of `pool` (num_blocks records per kv head, 16-byte aligned).
 * Slots as tq_encode_k: negative skipped silently, >= 16 num_blocks flagged
 * TQ_STATUS_BAD_SLOT and skipped.  Coordinates must be finite and within fp16 range.
 * Errors: TQ_ERR_HEAD_DIM, TQ_ERR_INVALID (also bits or group unsupported), TQ_ERR_DTYPE,
 * TQ_ERR_ALIGN, TQ_ERR_CUDA. */
int tq_gq_encode(int d, int bits, int group, const void *x, int dtype, int64_t n_tokens,
                 int n_kv_heads, const int64_t *slot_mapping, void *pool, int64_t num_blocks,
                 int32_t *status, tq_stream_t stream);

/* Workspace of tq_gq_decode_attn: per (sequence, kv head, 128-token chunk of max_ctx, query
 * head of the group rounded up to 1, 2, 4 or 8) a partial of d + 4 floats.  0 if invalid. */
size_t tq_gq_decode_workspace_bytes(int d, int batch, int n_q_heads, int n_kv_heads, int max_ctx);

/* tq_gq_decode_attn -- decode attention over group-quantised paged K and V pools: for query
 * head h of sequence b (kv head h / G) over its ctx_lens[b] tokens,
 *   s_j = q . k~_j / sqrt d,  P = softmax(s),  out = sum_j P_j v~_j,
 * with k~, v~ the decoded vectors; fp32 arithmetic, out float [batch][n_q_heads][d].
 * Arguments, block-table and ctx_lens semantics, status and errors as tq_decode_attn (no params
 * buffer; workspace from tq_gq_decode_workspace_bytes, 16-byte aligned). */
int tq_gq_decode_attn(int d, int bits, int group, const void *q, int dtype, int batch,
                      int n_q_heads, int n_kv_heads, const void *k_pool, const void *v_pool,
                      int64_t num_blocks, const int32_t *block_table, int max_blocks,
                      const int32_t *ctx_lens, int max_ctx, float *out, void *workspace,
                      size_t workspace_bytes, int32_t *status, tq_stream_t stream);

/* Short English text for a TQ_* return code (static storage). */
const char *tq_error_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H_ */
