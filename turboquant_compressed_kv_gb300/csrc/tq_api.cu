// tq_api.cu -- the C ABI declared in include/tq.h: argument checks on the host,
// then kernel launches on the caller's stream.  Allocates no device memory.
#include <vector>
#include <math.h>
#include <string.h>

#include "tq_gq.cuh"
#include "tq_internal.cuh"

namespace tq {
namespace {

// Lloyd-Max fixed point for the unit Gaussian with 8 levels, in fp64 on the host
// ("Lloyd-Maxコードブックとは", lilting.ch SwiftLM article: computed once before inference,
// no calibration).  The optimum is symmetric (the Gaussian is symmetric and log-concave, so
// the optimum is unique), so only the four positive cells are iterated: edges 0, m1, m2, m3,
// +inf; each level moves to the Gaussian mean of its cell, each inner edge to the midpoint
// of its two levels.
void lloyd_max_positive(double (&lv)[4]) {
    const double inv_sqrt2 = 0.70710678118654752440;
    const double inv_sqrt2pi = 0.39894228040143267794;
    lv[0] = 0.3; lv[1] = 0.8; lv[2] = 1.4; lv[3] = 2.2;
    for (int it = 0; it < 100000; ++it) {
        const double edge[5] = {0.0, 0.5 * (lv[0] + lv[1]), 0.5 * (lv[1] + lv[2]), 0.5 * (lv[2] + lv[3]), 0.0};
        double moved = 0.0;
        for (int k = 0; k < 4; ++k) {
            const double a = edge[k];
            const bool last = (k == 3);
            const double dens_a = inv_sqrt2pi * exp(-0.5 * a * a);
            const double dens_b = last ? 0.0 : inv_sqrt2pi * exp(-0.5 * edge[k + 1] * edge[k + 1]);
            const double tail_a = 0.5 * erfc(a * inv_sqrt2);
            const double tail_b = last ? 0.0 : 0.5 * erfc(edge[k + 1] * inv_sqrt2);
            const double m = (dens_a - dens_b) / (tail_a - tail_b);
            moved = fmax(moved, fabs(m - lv[k]));
            lv[k] = m;
        }
        if (moved < 1e-15) break;
    }
}

// Nearest binary16 value of a positive normal-range double (ties to even), and its bits.
double f16_round_pos(double v, int *ex_out = nullptr) {
    int e;
    frexp(v, &e);                     // v = f 2^e, f in [0.5, 1): spacing 2^(e - 11)
    const double ulp = ldexp(1.0, e - 11);
    if (ex_out) *ex_out = e;
    return nearbyint(v / ulp) * ulp;  // default rounding mode: to nearest, ties to even
}
// Nearest binary16 value of any finite double in the binary16 range (ties to even, subnormals
// included).
double f16_round(double v) {
    const double a = fabs(v);
    if (a == 0.0) return v;
    const double r = a < ldexp(1.0, -14) ? nearbyint(a / ldexp(1.0, -24)) * ldexp(1.0, -24) : f16_round_pos(a);
    return copysign(r, v);
}
uint16_t f16_bits(double v) {
    const bool neg = v < 0;
    int e;
    const double r = f16_round_pos(neg ? -v : v, &e);
    int ex;
    const double f = frexp(r, &ex);   // rounding may carry into the next binade
    const uint32_t mant = (uint32_t)ldexp(f, 11) - 1024u;
    return (uint16_t)((neg ? 0x8000u : 0u) | ((uint32_t)(ex - 1 + 15) << 10) | mant);
}

// The decode kernels read the codebook as eight binary16 values T[j] = f16(alpha c[j]) through
// byte-permute lookups and undo alpha in fp32.  alpha in [1, 2) is chosen to put all four
// magnitudes closest to binary16 values: the worst relative error of T[j] / alpha against
// c[j] is then under 2e-5 (plain f16 rounding would leave up to 3e-4).
double choose_alpha(const double (&lv)[4]) {
    double best = 1.0, best_err = 1e30;
    for (int k = 0; k < 1000000; ++k) {
        const double al = 1.0 + k * 1e-6;
        double err = 0.0;
        for (int j = 0; j < 4 && err < best_err; ++j) {
            const double v = al * lv[j];
            err = fmax(err, fabs(f16_round_pos(v) - v) / v);
        }
        if (err < best_err) {
            best_err = err;
            best = al;
        }
    }
    return best;
}

ParamsHeader make_header() {
    ParamsHeader h;
    memset(&h, 0, sizeof h);
    double lv[4];
    lloyd_max_positive(lv);
    for (int k = 0; k < 4; ++k) {
        h.centroid64[4 + k] = lv[k];
        h.centroid64[3 - k] = -lv[k];
    }
    for (int j = 0; j < 8; ++j) h.centroid[j] = (float)h.centroid64[j];
    for (int j = 0; j < 7; ++j) h.threshold[j] = (float)(0.5 * (h.centroid64[j] + h.centroid64[j + 1]));
    h.threshold[3] = 0.0f;
    h.threshold[7] = INFINITY;
    h.one16x2 = 0x3C003C00u;
    const double al = choose_alpha(lv);
    h.inv_alpha = (float)(1.0 / al);
    for (int j = 0; j < 8; ++j) {
        const uint16_t t = f16_bits(al * h.centroid64[j]);
        h.t16[j] = t;
        h.lut_lo[j >> 2] |= (uint32_t)(t & 0xFFu) << (8 * (j & 3));
        h.lut_hi[j >> 2] |= (uint32_t)(t >> 8) << (8 * (j & 3));
    }
    h.magic = kParamsMagic;
    return h;
}

// The header depends on d only through its d field: solved once per process.
void fill_header(ParamsHeader &h, int d) {
    static const ParamsHeader base = make_header();
    h = base;
    h.d = d;
}

// D signs arrive as int8 in a scratch spot (the start of the S region);
// store them as +-1.0f.
__global__ void signs_kernel(uint8_t *params, int d) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= d) return;
    const int8_t s = reinterpret_cast<const int8_t *>(params + params_off_S(d))[i];
    reinterpret_cast<float *>(params + params_off_D(d))[i] = (s < 0) ? -1.0f : 1.0f;
}

// S^T (column k of S as a contiguous row) for coalesced projections.
__global__ void transpose_kernel(uint8_t *params, int d) {
    const float *S = reinterpret_cast<const float *>(params + params_off_S(d));
    float *ST = reinterpret_cast<float *>(params + params_off_ST(d));
    const int i = blockIdx.x, k = threadIdx.x;
    if (i < d && k < d) ST[(size_t)i * d + k] = S[(size_t)k * d + i];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA; }

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" {

size_t tq_k_record_bytes(int d) { return valid_d(d) ? k_record(d) : 0; }
size_t tq_v_record_bytes(int d) { return valid_d(d) ? v_record(d) : 0; }
size_t tq_params_bytes(int d) { return valid_d(d) ? params_total(d) : 0; }

const char *tq_error_string(int code) {
    switch (code) {
        case TQ_OK: return "ok";
        case TQ_ERR_INVALID: return "invalid argument (size, count or NULL pointer)";
        case TQ_ERR_HEAD_DIM: return "unsupported head_dim (must be 128 or 256)";
        case TQ_ERR_GQA: return "n_q_heads must be a multiple of n_kv_heads with group size 1..8";
        case TQ_ERR_WORKSPACE: return "workspace or params buffer too small";
        case TQ_ERR_CUDA: return "CUDA launch or runtime error";
        case TQ_ERR_DTYPE: return "unsupported dtype (TQ_DTYPE_F32 or TQ_DTYPE_BF16)";
        case TQ_ERR_ALIGN: return "pointer not 16-byte aligned";
        default: return "unknown error";
    }
}

int tq_codebook_init(int d, const int8_t *D_host, const float *S_host, void *params_dev, size_t params_bytes,
                     double *centroids_out8, tq_stream_t stream) {
    if (!valid_d(d)) return TQ_ERR_HEAD_DIM;
    if (!D_host || !S_host || !params_dev) return TQ_ERR_INVALID;
    if (!aligned16(params_dev)) return TQ_ERR_ALIGN;
    if (params_bytes < params_total(d)) return TQ_ERR_WORKSPACE;
    for (int i = 0; i < d; ++i)
        if (D_host[i] != 1 && D_host[i] != -1) return TQ_ERR_INVALID;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *P = static_cast<uint8_t *>(params_dev);
    ParamsHeader h;
    fill_header(h, d);
    cudaError_t e = cudaMemsetAsync(P, 0, sizeof(ParamsHeader), st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(P + params_off_S(d), D_host, (size_t)d, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) { signs_kernel<<<(d + 127) / 128, 128, 0, st>>>(P, d); e = cudaGetLastError(); }
    // S is held at binary16 precision: the QJL projections then need no low-order part of S on
    // the tensor cores (sr stays alive until the stream is synchronised below)
    std::vector<float> sr((size_t)d * d);
    for (size_t i = 0; i < sr.size(); ++i) sr[i] = (float)f16_round((double)S_host[i]);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(P + params_off_S(d), sr.data(), sizeof(float) * (size_t)d * d, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) { transpose_kernel<<<d, d, 0, st>>>(P, d); e = cudaGetLastError(); }
    // the QJL offset weights, summed in fp64 (wv stays alive until the stream is synchronised below)
    std::vector<float> wv((size_t)d);
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int k = 0; k < d; ++k)
            if (qjl_pos(k) < 3) acc += (double)sr[(size_t)k * d + j];
        wv[(size_t)j] = (float)acc;
    }
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(P + params_off_W(d), wv.data(), sizeof(float) * (size_t)d, cudaMemcpyHostToDevice, st);
    // the header (magic last in stream order) once D and S are in place; h stays alive until the
    // stream is synchronised below
    if (e == cudaSuccess) e = cudaMemcpyAsync(P, &h, sizeof h, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && centroids_out8) memcpy(centroids_out8, h.centroid64, 8 * sizeof(double));
    return cuda_status(e);
}

static int check_pool_call(const void *params, int d, const void *x, int dtype, int64_t n_tokens, int n_heads,
                           const void *slots, const void *pool, int64_t num_blocks) {
    if (!valid_d(d)) return TQ_ERR_HEAD_DIM;
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16) return TQ_ERR_DTYPE;
    if (n_tokens < 0 || n_heads <= 0 || num_blocks < 0) return TQ_ERR_INVALID;
    if (n_tokens == 0) return TQ_OK;
    if (!params || !x || !slots || !pool) return TQ_ERR_INVALID;
    if (!aligned16(params) || !aligned16(pool)) return TQ_ERR_ALIGN;
    if (n_tokens > ((int64_t)1 << 40) / n_heads) return TQ_ERR_INVALID;
    return TQ_OK;
}

int tq_encode_k(const void *params, int d, const void *k, int dtype, int64_t n_tokens, int n_kv_heads,
                const int64_t *slot_mapping, void *k_pool, int64_t num_blocks, int32_t *status, tq_stream_t stream) {
    int rc = check_pool_call(params, d, k, dtype, n_tokens, n_kv_heads, slot_mapping, k_pool, num_blocks);
    if (rc != TQ_OK || n_tokens == 0) return rc;
    return cuda_status(launch_encode(true, d, dtype, params, k, n_tokens, n_kv_heads, slot_mapping, k_pool,
                                     num_blocks, status, reinterpret_cast<cudaStream_t>(stream)));
}

int tq_encode_v(const void *params, int d, const void *v, int dtype, int64_t n_tokens, int n_kv_heads,
                const int64_t *slot_mapping, void *v_pool, int64_t num_blocks, int32_t *status, tq_stream_t stream) {
    int rc = check_pool_call(params, d, v, dtype, n_tokens, n_kv_heads, slot_mapping, v_pool, num_blocks);
    if (rc != TQ_OK || n_tokens == 0) return rc;
    return cuda_status(launch_encode(false, d, dtype, params, v, n_tokens, n_kv_heads, slot_mapping, v_pool,
                                     num_blocks, status, reinterpret_cast<cudaStream_t>(stream)));
}

int tq_paged_append(const void *params, int d, const void *k_new, const void *v_new, int dtype, int batch,
                    int n_kv_heads, const int32_t *block_table, int max_blocks, const int32_t *ctx_lens,
                    void *k_pool, void *v_pool, int64_t num_blocks, int32_t *status, tq_stream_t stream) {
    if (!valid_d(d)) return TQ_ERR_HEAD_DIM;
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16) return TQ_ERR_DTYPE;
    if (batch < 0 || n_kv_heads <= 0 || max_blocks <= 0 || num_blocks < 0) return TQ_ERR_INVALID;
    if (batch == 0) return TQ_OK;
    if (!params || !k_new || !v_new || !block_table || !ctx_lens || !k_pool || !v_pool) return TQ_ERR_INVALID;
    if (!aligned16(params) || !aligned16(k_pool) || !aligned16(v_pool)) return TQ_ERR_ALIGN;
    return cuda_status(launch_append(d, dtype, params, k_new, v_new, batch, n_kv_heads, block_table, max_blocks,
                                     ctx_lens, k_pool, v_pool, num_blocks, status,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

static int dequant_call(bool is_k, const void *params, int d, const void *pool, int64_t num_blocks, int n_kv_heads,
                        const int32_t *block_ids, int n_ids, void *out, int out_dtype, int32_t *status,
                        tq_stream_t stream) {
    if (!valid_d(d)) return TQ_ERR_HEAD_DIM;
    if (out_dtype != TQ_DTYPE_F32 && out_dtype != TQ_DTYPE_BF16) return TQ_ERR_DTYPE;
    if (n_ids < 0 || n_kv_heads <= 0 || num_blocks < 0) return TQ_ERR_INVALID;
    if (n_ids == 0) return TQ_OK;
    if (num_blocks == 0) return TQ_ERR_INVALID;   // no block to read
    if (!params || !pool || !block_ids || !out) return TQ_ERR_INVALID;
    if (!aligned16(params) || !aligned16(pool)) return TQ_ERR_ALIGN;
    return cuda_status(launch_dequant(is_k, d, out_dtype, params, pool, num_blocks, n_kv_heads, block_ids, n_ids, out,
                                      status, reinterpret_cast<cudaStream_t>(stream)));
}

int tq_dequant_k(const void *params, int d, const void *k_pool, int64_t num_blocks, int n_kv_heads,
                 const int32_t *block_ids, int n_ids, void *out, int out_dtype, int32_t *status, tq_stream_t stream) {
    return dequant_call(true, params, d, k_pool, num_blocks, n_kv_heads, block_ids, n_ids, out, out_dtype, status,
                        stream);
}

int tq_dequant_v(const void *params, int d, const void *v_pool, int64_t num_blocks, int n_kv_heads,
                 const int32_t *block_ids, int n_ids, void *out, int out_dtype, int32_t *status, tq_stream_t stream) {
    return dequant_call(false, params, d, v_pool, num_blocks, n_kv_heads, block_ids, n_ids, out, out_dtype, status,
                        stream);
}

size_t tq_decode_workspace_bytes(int d, int batch, int n_q_heads, int max_ctx) {
    return decode_workspace_bytes(d, batch, n_q_heads, max_ctx);
}

size_t tq_decode_workspace_bytes_mq(int d, int batch, int q_len, int n_q_heads, int max_ctx) {
    if (q_len <= 0 || q_len > 8 || n_q_heads <= 0) return 0;
    return decode_workspace_bytes(d, batch, q_len * n_q_heads, max_ctx);
}

static int check_decode(const void *params, int d, int batch, int q_len, int hq, int hkv, int max_ctx, void *ws,
                        size_t ws_bytes) {
    if (!valid_d(d)) return TQ_ERR_HEAD_DIM;
    if (batch < 0 || q_len <= 0 || hq <= 0 || hkv <= 0 || max_ctx < 0) return TQ_ERR_INVALID;
    if (hq % hkv != 0 || q_len > 8 || q_len * (hq / hkv) > 8) return TQ_ERR_GQA;
    if (batch > 65535 || hkv > 65535) return TQ_ERR_INVALID;
    if (batch == 0) return TQ_OK;
    if (!params || !ws) return TQ_ERR_INVALID;
    if (!aligned16(params) || !aligned16(ws)) return TQ_ERR_ALIGN;
    if (ws_bytes < decode_workspace_bytes(d, batch, q_len * hq, max_ctx)) return TQ_ERR_WORKSPACE;
    return TQ_OK;
}

int tq_decode_qprep(const void *params, int d, const void *q, int dtype, int batch, int n_q_heads, int n_kv_heads,
                    const int32_t *ctx_lens, int max_ctx, void *workspace, size_t workspace_bytes,
                    tq_stream_t stream) {
    int rc = check_decode(params, d, batch, 1, n_q_heads, n_kv_heads, max_ctx, workspace, workspace_bytes);
    if (rc != TQ_OK || batch == 0) return rc;
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16) return TQ_ERR_DTYPE;
    if (!q) return TQ_ERR_INVALID;
    if (!ctx_lens) return TQ_ERR_INVALID;
    return cuda_status(launch_qprep(d, dtype, params, q, batch, 1, n_q_heads, n_kv_heads, workspace,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int tq_decode_splitk(const void *params, int d, int batch, int n_q_heads, int n_kv_heads, const void *k_pool,
                     const void *v_pool, int64_t num_blocks, const int32_t *block_table, int max_blocks,
                     const int32_t *ctx_lens, int max_ctx, float *out, void *workspace, size_t workspace_bytes,
                     int32_t *status, tq_stream_t stream) {
    int rc = check_decode(params, d, batch, 1, n_q_heads, n_kv_heads, max_ctx, workspace, workspace_bytes);
    if (rc != TQ_OK || batch == 0) return rc;
    if (max_blocks <= 0 || num_blocks < 0) return TQ_ERR_INVALID;
    if (!k_pool || !v_pool || !block_table || !ctx_lens || !out) return TQ_ERR_INVALID;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return TQ_ERR_ALIGN;
    return cuda_status(launch_splitk(d, params, batch, 1, n_q_heads, n_kv_heads, k_pool, v_pool, num_blocks,
                                     block_table, max_blocks, ctx_lens, 0, max_ctx, out, workspace, status,
                                     reinterpret_cast<cudaStream_t>(stream), false));
}

int tq_decode_attn_mq(const void *params, int d, const void *q, int dtype, int batch, int q_len, int n_q_heads,
                      int n_kv_heads, const void *k_pool, const void *v_pool, int64_t num_blocks,
                      const int32_t *block_table, int max_blocks, const int32_t *ctx_lens, int max_ctx, float *out,
                      void *workspace, size_t workspace_bytes, int32_t *status, tq_stream_t stream) {
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16 && valid_d(d)) return TQ_ERR_DTYPE;
    int rc = check_decode(params, d, batch, q_len, n_q_heads, n_kv_heads, max_ctx, workspace, workspace_bytes);
    if (rc != TQ_OK || batch == 0) return rc;
    if (max_blocks <= 0 || num_blocks < 0) return TQ_ERR_INVALID;
    if (!q || !k_pool || !v_pool || !block_table || !ctx_lens || !out) return TQ_ERR_INVALID;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return TQ_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_qprep(d, dtype, params, q, batch, q_len, n_q_heads, n_kv_heads, workspace, st);
    if (e == cudaSuccess)
        e = launch_splitk(d, params, batch, q_len, n_q_heads, n_kv_heads, k_pool, v_pool, num_blocks, block_table,
                          max_blocks, ctx_lens, 0, max_ctx, out, workspace, status, st, true);
    return cuda_status(e);
}

static size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

int tq_selftest_wait_timeout(int32_t *status, tq_stream_t stream) {
    if (!status) return TQ_ERR_INVALID;
    return cuda_status(launch_wait_timeout_selftest(status, reinterpret_cast<cudaStream_t>(stream)));
}

size_t tq_hybrid_append_scratch_bytes(int d, int batch, int n_kv_heads, int dtype) {
    if (!valid_d(d) || batch < 0 || n_kv_heads <= 0) return 0;
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16) return 0;
    return hybrid_append_scratch_bytes(d, batch, n_kv_heads, dtype);
}

int tq_hybrid_append(const void *params, int d, const void *k_new, const void *v_new, int dtype, int batch,
                     int n_kv_heads, void *win_k, void *win_v, int win_cap, int32_t *win_lens,
                     const int32_t *block_table, int max_blocks, int32_t *ctx_lens, void *k_pool, void *v_pool,
                     int64_t num_blocks, void *scratch, size_t scratch_bytes, int32_t *status, tq_stream_t stream) {
    if (!valid_d(d)) return TQ_ERR_HEAD_DIM;
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16) return TQ_ERR_DTYPE;
    if (batch < 0 || n_kv_heads <= 0 || win_cap <= 0 || max_blocks <= 0 || num_blocks < 0) return TQ_ERR_INVALID;
    if (batch == 0) return TQ_OK;
    if (!params || !k_new || !v_new || !win_k || !win_v || !win_lens || !block_table || !ctx_lens || !k_pool ||
        !v_pool || !scratch)
        return TQ_ERR_INVALID;
    if (!aligned16(params) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(win_k) || !aligned16(win_v) ||
        !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(scratch))
        return TQ_ERR_ALIGN;
    if (scratch_bytes < hybrid_append_scratch_bytes(d, batch, n_kv_heads, dtype)) return TQ_ERR_WORKSPACE;
    return cuda_status(launch_hybrid_append(d, dtype, params, k_new, v_new, batch, n_kv_heads, win_k, win_v, win_cap,
                                            win_lens, block_table, max_blocks, ctx_lens, k_pool, v_pool, num_blocks,
                                            scratch, status, reinterpret_cast<cudaStream_t>(stream)));
}

size_t tq_decode_workspace_bytes_hybrid(int d, int batch, int n_q_heads, int max_ctx, int win_cap) {
    const size_t base = decode_workspace_bytes(d, batch, n_q_heads, max_ctx);
    if (base == 0 || win_cap < 0) return 0;
    return al256(base) + al256((size_t)batch * n_q_heads * sizeof(float)) +
           hybrid_part_bytes(d, batch, n_q_heads, win_cap);
}

int tq_decode_attn_hybrid(const void *params, int d, const void *q, int dtype, int batch, int n_q_heads,
                          int n_kv_heads, const void *k_pool, const void *v_pool, int64_t num_blocks,
                          const int32_t *block_table, int max_blocks, const int32_t *ctx_lens, int max_ctx,
                          const void *win_k, const void *win_v, int win_dtype, int win_cap, const int32_t *win_lens,
                          float *out, void *workspace, size_t workspace_bytes, int32_t *status, tq_stream_t stream) {
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16 && valid_d(d)) return TQ_ERR_DTYPE;
    if (win_dtype != TQ_DTYPE_F32 && win_dtype != TQ_DTYPE_BF16 && valid_d(d)) return TQ_ERR_DTYPE;
    int rc = check_decode(params, d, batch, 1, n_q_heads, n_kv_heads, max_ctx, workspace, workspace_bytes);
    if (rc != TQ_OK || batch == 0) return rc;
    if (win_cap < 0 || max_blocks <= 0 || num_blocks < 0) return TQ_ERR_INVALID;
    if (workspace_bytes < tq_decode_workspace_bytes_hybrid(d, batch, n_q_heads, max_ctx, win_cap))
        return TQ_ERR_WORKSPACE;
    if (!q || !k_pool || !v_pool || !block_table || !ctx_lens || !out) return TQ_ERR_INVALID;
    if (win_cap > 0 && (!win_k || !win_v || !win_lens)) return TQ_ERR_INVALID;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return TQ_ERR_ALIGN;
    if (win_cap > 0 && (!aligned16(win_k) || !aligned16(win_v))) return TQ_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    const size_t base = al256(decode_workspace_bytes(d, batch, n_q_heads, max_ctx));
    float *lse = reinterpret_cast<float *>(ws + base);
    float *part = reinterpret_cast<float *>(ws + base + al256((size_t)batch * n_q_heads * sizeof(float)));
    cudaError_t e = launch_qprep(d, dtype, params, q, batch, 1, n_q_heads, n_kv_heads, ws, st);
    if (e == cudaSuccess)
        e = launch_splitk(d, params, batch, 1, n_q_heads, n_kv_heads, k_pool, v_pool, num_blocks, block_table,
                          max_blocks, ctx_lens, 0, max_ctx, out, ws, status, st, true, lse);
    if (e == cudaSuccess)
        e = launch_hybrid_window(d, dtype, win_dtype, q, win_k, win_v, batch, n_q_heads, n_kv_heads, win_cap, win_lens,
                                 part, out, lse, st);
    return cuda_status(e);
}

int tq_decode_attn(const void *params, int d, const void *q, int dtype, int batch, int n_q_heads, int n_kv_heads,
                   const void *k_pool, const void *v_pool, int64_t num_blocks, const int32_t *block_table,
                   int max_blocks, const int32_t *ctx_lens, int max_ctx, float *out, void *workspace,
                   size_t workspace_bytes, int32_t *status, tq_stream_t stream) {
    return tq_decode_attn_mq(params, d, q, dtype, batch, 1, n_q_heads, n_kv_heads, k_pool, v_pool, num_blocks,
                             block_table, max_blocks, ctx_lens, max_ctx, out, workspace, workspace_bytes, status,
                             stream);
}

int tq_decode_step_mq(const void *params, int d, const void *k_new, const void *v_new, const void *q, int dtype,
                      int batch, int q_len, int n_q_heads, int n_kv_heads, const int32_t *block_table,
                      int max_blocks, const int32_t *pre_lens, int max_ctx, void *k_pool, void *v_pool,
                      int64_t num_blocks, float *out, void *workspace, size_t workspace_bytes, int32_t *status,
                      tq_stream_t stream) {
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16 && valid_d(d)) return TQ_ERR_DTYPE;
    int rc = check_decode(params, d, batch, q_len, n_q_heads, n_kv_heads, max_ctx, workspace, workspace_bytes);
    if (rc != TQ_OK || batch == 0) return rc;
    if (max_blocks <= 0 || num_blocks < 0) return TQ_ERR_INVALID;
    if (!k_new || !v_new || !q || !k_pool || !v_pool || !block_table || !pre_lens || !out) return TQ_ERR_INVALID;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return TQ_ERR_ALIGN;
    return cuda_status(launch_step(d, dtype, params, k_new, v_new, q, batch, q_len, n_q_heads, n_kv_heads,
                                   block_table, max_blocks, pre_lens, max_ctx, k_pool, v_pool, num_blocks, out,
                                   workspace, status, reinterpret_cast<cudaStream_t>(stream)));
}

int tq_decode_step(const void *params, int d, const void *k_new, const void *v_new, const void *q, int dtype,
                   int batch, int n_q_heads, int n_kv_heads, const int32_t *block_table, int max_blocks,
                   const int32_t *pre_lens, int max_ctx, void *k_pool, void *v_pool, int64_t num_blocks, float *out,
                   void *workspace, size_t workspace_bytes, int32_t *status, tq_stream_t stream) {
    return tq_decode_step_mq(params, d, k_new, v_new, q, dtype, batch, 1, n_q_heads, n_kv_heads, block_table,
                             max_blocks, pre_lens, max_ctx, k_pool, v_pool, num_blocks, out, workspace,
                             workspace_bytes, status, stream);
}

size_t tq_gq_record_bytes(int d, int bits, int group) { return gq_valid(d, bits, group) ? gq_region_bytes(d, bits, group) : 0; }

static int check_gq(int d, int bits, int group) {
    if (d != 128 && d != 256) return TQ_ERR_HEAD_DIM;
    return gq_valid(d, bits, group) ? TQ_OK : TQ_ERR_INVALID;
}

int tq_gq_encode(int d, int bits, int group, const void *x, int dtype, int64_t n_tokens, int n_kv_heads,
                 const int64_t *slot_mapping, void *pool, int64_t num_blocks, int32_t *status, tq_stream_t stream) {
    int rc = check_gq(d, bits, group);
    if (rc != TQ_OK) return rc;
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16) return TQ_ERR_DTYPE;
    if (n_tokens < 0 || n_kv_heads <= 0 || num_blocks < 0) return TQ_ERR_INVALID;
    if (n_tokens == 0) return TQ_OK;
    if (!x || !slot_mapping || !pool) return TQ_ERR_INVALID;
    if (!aligned16(x) || !aligned16(pool)) return TQ_ERR_ALIGN;
    if (n_tokens > ((int64_t)1 << 40) / n_kv_heads) return TQ_ERR_INVALID;
    return cuda_status(launch_gq_encode(d, bits, group, dtype, x, n_tokens, n_kv_heads, slot_mapping,
                                        static_cast<uint8_t *>(pool), num_blocks, status,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

size_t tq_gq_decode_workspace_bytes(int d, int batch, int n_q_heads, int n_kv_heads, int max_ctx) {
    if ((d != 128 && d != 256) || batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || max_ctx < 0) return 0;
    if (n_q_heads % n_kv_heads != 0 || n_q_heads / n_kv_heads > 8) return 0;
    return gq_workspace_bytes(d, batch, n_q_heads, n_kv_heads, max_ctx);
}

int tq_gq_decode_attn(int d, int bits, int group, const void *q, int dtype, int batch, int n_q_heads, int n_kv_heads,
                      const void *k_pool, const void *v_pool, int64_t num_blocks, const int32_t *block_table,
                      int max_blocks, const int32_t *ctx_lens, int max_ctx, float *out, void *workspace,
                      size_t workspace_bytes, int32_t *status, tq_stream_t stream) {
    int rc = check_gq(d, bits, group);
    if (rc != TQ_OK) return rc;
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16) return TQ_ERR_DTYPE;
    if (batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || max_ctx < 0) return TQ_ERR_INVALID;
    if (n_q_heads % n_kv_heads != 0 || n_q_heads / n_kv_heads > 8) return TQ_ERR_GQA;
    if (batch > 65535 || n_kv_heads > 65535) return TQ_ERR_INVALID;
    if (batch == 0) return TQ_OK;
    if (max_blocks <= 0 || num_blocks < 0) return TQ_ERR_INVALID;
    if (!q || !k_pool || !v_pool || !block_table || !ctx_lens || !out) return TQ_ERR_INVALID;
    if (workspace_bytes < gq_workspace_bytes(d, batch, n_q_heads, n_kv_heads, max_ctx)) return TQ_ERR_WORKSPACE;
    if (max_ctx > 0 && !workspace) return TQ_ERR_INVALID;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(workspace)) return TQ_ERR_ALIGN;
    return cuda_status(launch_gq_decode(d, bits, group, dtype, q, batch, n_q_heads, n_kv_heads,
                                        static_cast<const uint8_t *>(k_pool), static_cast<const uint8_t *>(v_pool),
                                        num_blocks, block_table, max_blocks, ctx_lens, max_ctx, out,
                                        static_cast<float *>(workspace), status, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
