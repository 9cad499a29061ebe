// tq_decode.cu -- decode attention over the compressed paged cache.
//
// Method: scores and the value sum are evaluated in the rotated domain straight
// from the packed cells, signs and fp16 norms (the "fused dequantisation" of
// the SwiftLM README, "TurboQuantization: KV Cache Compression"); blocks are
// found through the block table of the vLLM-MLX explainer, "Paged KVキャッシュ".
// With qbar = Pi q and u = S qbar:
//   s_j = (n_j/sqrt d) (<qbar, c[cell_j]>/sqrt d + gamma_j sqrt(pi/2)/d <u, 2 sign_j - 1>)
//   a   = sum_j softmax(s)_j nv_j c[vcell_j] / sqrt d,    out = Pi^T a.
//
// Tensor-core formulation (this library's design, not the pages'): the scores and the value
// sum are mma.sync (m16n8k16, f16 operands, fp32 accumulation) contractions whose record-side
// operands are built by byte-permute table lookups of the codebook (tq_decode_warp.cu); the
// fp32 query side is carried as f16 hi + lo (relative error about 2^-22), the softmax weights
// as f16 hi + lo (one f16 above 4 heads) with a running power-of-two scale.
//
// Two launches per call: (1) query prep (qbar, u, f16 operand fragments,
// offset constants, and the work schedule of the pass); (2) the split-K pass,
// persistent: the context of every (sequence, kv head) is cut into 128-token
// chunks (256 for groups of more than 4 query heads), and CTA c of P takes
// the c-th of P equal, contiguous ranges of the chunk sequence ordered by
// (sequence, kv head, chunk) ("stream-K").  A (sequence, kv head) inside one
// CTA's range is finished there; one shared by several CTAs leaves an
// online-softmax partial (m, l, acc[d]) per query head from each, and the last
// of them to finish merges the partials.  Either way one inverse rotation per
// (sequence, query head) is applied at the end.
#include <atomic>

#include "tq_split.cuh"

namespace tq {

size_t decode_workspace_bytes(int d, int batch, int hq, int max_ctx) {
    if (!valid_d(d) || batch <= 0 || hq <= 0 || max_ctx < 0) return 0;
    size_t off[5];
    return ws_sizes(d, batch, hq, off);
}

namespace {

// ---------------------------------------------------------------- (1) query prep (body in tq_prep.cuh)
template <int D, int NTK, typename T>
__global__ void __launch_bounds__(128)
qprep_kernel(const uint8_t *__restrict__ params, const T *__restrict__ q, int batch, int q_len, int hq, int hkv,
             const int32_t *__restrict__ ctx_lens, int max_ctx, int chunk, int P, uint8_t *__restrict__ packs,
             unsigned int *__restrict__ counters, int64_t *__restrict__ cpre, int32_t *__restrict__ cta_b) {
    extern __shared__ __align__(16) uint8_t qsm[];
    pdl_launch_dependents();
    if (blockIdx.x == gridDim.x - 1) {   // the last CTA lays out the pass's work
        build_schedule(ctx_lens, 0, batch, hkv, max_ctx, chunk, P, cpre, cta_b);
        return;
    }
    qprep_rows<D, NTK, T>(params, q, batch, q_len, hq, hkv, ctx_lens, 0, max_ctx, chunk, P, packs, counters, cpre, cta_b,
                          blockIdx.x, qsm);
}

// Persistent CTAs of the pass on the current device: up to kCtasPerSm per SM
// (fewer if the kernel's resources allow fewer), for at most kMaxSms SMs.
// Cached per (device, d, G): query prep and the pass must agree on it, and the
// occupancy query is not free.
int pass_ctas_any(int d, int G) {
    constexpr int kDevs = 64;
    static std::atomic<int> cache[kDevs][2][9];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || G < 1 || G > 8) return 0;
    if (dev >= kDevs) return warp_pass_ctas(d, G);
    std::atomic<int> &slot = cache[dev][d == 128 ? 0 : 1][G];
    int n = slot.load(std::memory_order_relaxed);
    if (n == 0) {
        n = warp_pass_ctas(d, G);
        slot.store(n, std::memory_order_relaxed);
    }
    return n;
}

template <int D, int NTK, typename T>
cudaError_t qprep_launch_t(const uint8_t *P, const void *q, int batch, int q_len, int hq, int hkv,
                           const int32_t *ctx_lens, int max_ctx, int nctas, const WsLayout &w, cudaStream_t st) {
    constexpr size_t smem = qprep_smem<D>();
    auto kern = qprep_kernel<D, NTK, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(batch * q_len * hq + kQRows - 1) / kQRows + 1, 128, smem, st>>>(P, (const T *)q, batch, q_len, hq, hkv, ctx_lens,
                                                                       max_ctx, pass_chunk(q_len * hq / hkv), nctas,
                                                                       w.packs, w.counters, w.cpre, w.cta_b);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t qprep_launch(const uint8_t *P, const void *q, int batch, int q_len, int hq, int hkv,
                         const int32_t *ctx_lens, int max_ctx, int nctas, const WsLayout &w, cudaStream_t st) {
    // n-tile count of the K-side operand: (2G + 7) / 8 for G = q_len * hq / hkv columns, as in the passes
    if (q_len * hq / hkv <= 4)
        return qprep_launch_t<D, 1, T>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st);
    return qprep_launch_t<D, 2, T>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st);
}

}  // namespace

cudaError_t launch_qprep(int d, int dtype, const void *params, const void *q, int batch, int q_len, int hq,
                         int hkv, const int32_t *ctx_lens, int max_ctx, void *ws, cudaStream_t st) {
    const WsLayout w = ws_layout(ws, d, batch, q_len * hq);
    const int nctas = pass_ctas_any(d, q_len * hq / hkv);
    if (nctas <= 0) return cudaErrorInvalidConfiguration;
    const uint8_t *P = (const uint8_t *)params;
    if (d == 128)
        return dtype == TQ_DTYPE_BF16
                   ? qprep_launch<128, __nv_bfloat16>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st)
                   : qprep_launch<128, float>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st);
    return dtype == TQ_DTYPE_BF16
               ? qprep_launch<256, __nv_bfloat16>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st)
               : qprep_launch<256, float>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st);
}

cudaError_t launch_splitk(int d, const void *params, int batch, int q_len, int hq, int hkv, const void *k_pool,
                          const void *v_pool, int64_t num_blocks, const int32_t *block_table, int max_blocks,
                          const int32_t *ctx_lens, int ctx_add, int max_ctx, float *out, void *ws, int32_t *status,
                          cudaStream_t st, float *lse) {
    const WsLayout w = ws_layout(ws, d, batch, q_len * hq);
    const int G = q_len * hq / hkv;   // operand columns per kv head
    const int nctas = pass_ctas_any(d, G);
    if (nctas <= 0) return cudaErrorInvalidConfiguration;
    const uint8_t *P = (const uint8_t *)params;
    return warp_pass_launch(d, G, nctas, st, P, batch, q_len, hq, hkv, (const uint8_t *)k_pool, (const uint8_t *)v_pool,
                            num_blocks, block_table, max_blocks, ctx_lens, ctx_add, max_ctx, w, out, lse, status);
}

// ---------------------------------------------------------------- the decode step: append, then attend
// One launch runs the append of one token per sequence (K tiles, V tiles) and the query prep
// side by side; the pass follows.  pre_lens[b] is the position of the new token, and the pass
// attends pre_lens[b] + 1 tokens.
namespace {
// K append tiles hold one vector (all four warps share its QJL projection: 128 FMA per thread),
// V tiles four (no projection)
constexpr int kAppendTileK = 1, kAppendTileV = 4;

template <int D, int NTK, typename T>
__global__ void __launch_bounds__(128)
step_prep_kernel(const uint8_t *__restrict__ params, const T *__restrict__ k_new, const T *__restrict__ v_new,
                 const T *__restrict__ q, int batch, int q_len, int hq, int hkv, SlotMap map, uint8_t *__restrict__ k_pool,
                 uint8_t *__restrict__ v_pool, int n_app_k, int n_app_v, int max_ctx, int chunk, int P,
                 uint8_t *__restrict__ packs,
                 unsigned int *__restrict__ counters, int64_t *__restrict__ cpre, int32_t *__restrict__ cta_b,
                 int32_t *status) {
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_launch_dependents();
    const int blk = blockIdx.x;
    if (blk < n_app_k) {
        encode_tiles<D, kAppendTileK, T>(params, k_new, (int64_t)batch * q_len * hkv, map, k_pool, true, true, blk,
                                         n_app_k, smem, status);
    } else if (blk < n_app_k + n_app_v) {
        encode_tiles<D, kAppendTileV, T>(params, v_new, (int64_t)batch * q_len * hkv, map, v_pool, false, false,
                                         blk - n_app_k, n_app_v, smem, status);
    } else if (blk == gridDim.x - 1) {   // the last CTA lays out the pass's work
        build_schedule(map.ctx_lens, q_len, batch, hkv, max_ctx, chunk, P, cpre, cta_b);
    } else {
        qprep_rows<D, NTK, T>(params, q, batch, q_len, hq, hkv, map.ctx_lens, q_len, max_ctx, chunk, P, packs, counters, cpre,
                              cta_b, blk - n_app_k - n_app_v, smem);
    }
}

template <int D, int NTK, typename T>
cudaError_t step_prep_launch(const uint8_t *P, const void *k_new, const void *v_new, const void *q, int batch,
                             int q_len, int hq, int hkv, const SlotMap &map, void *kp, void *vp, int max_ctx,
                             int nctas, const WsLayout &w, int32_t *status, cudaStream_t st) {
    constexpr size_t ek = EncSmem<D, kAppendTileK>::kBytes, ev = EncSmem<D, kAppendTileV>::kBytes;
    constexpr size_t es = ek > ev ? ek : ev, qs = qprep_smem<D>();
    constexpr size_t smem = es > qs ? es : qs;
    auto kern = step_prep_kernel<D, NTK, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int n_app_k = (batch * q_len * hkv + kAppendTileK - 1) / kAppendTileK;
    const int n_app_v = (batch * q_len * hkv + kAppendTileV - 1) / kAppendTileV;
    const int n_q = (batch * q_len * hq + kQRows - 1) / kQRows;
    kern<<<n_app_k + n_app_v + n_q + 1, 128, smem, st>>>(P, (const T *)k_new, (const T *)v_new, (const T *)q, batch, q_len, hq,
                                             hkv, map, (uint8_t *)kp, (uint8_t *)vp, n_app_k, n_app_v, max_ctx,
                                             pass_chunk(q_len * hq / hkv), nctas, w.packs, w.counters, w.cpre, w.cta_b,
                                             status);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t step_prep_any(const uint8_t *P, const void *k_new, const void *v_new, const void *q, int batch, int q_len,
                          int hq, int hkv, const SlotMap &map, void *kp, void *vp, int max_ctx, int nctas,
                          const WsLayout &w, int32_t *status, cudaStream_t st) {
    if (q_len * hq / hkv <= 4)
        return step_prep_launch<D, 1, T>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, kp, vp, max_ctx, nctas, w,
                                         status, st);
    return step_prep_launch<D, 2, T>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, kp, vp, max_ctx, nctas, w,
                                     status, st);
}
}  // namespace

cudaError_t launch_step(int d, int dtype, const void *params, const void *k_new, const void *v_new, const void *q,
                        int batch, int q_len, int hq, int hkv, const int32_t *block_table, int max_blocks,
                        const int32_t *pre_lens, int max_ctx, void *k_pool, void *v_pool, int64_t num_blocks,
                        float *out, void *ws, int32_t *status, cudaStream_t st) {
    const WsLayout w = ws_layout(ws, d, batch, q_len * hq);
    const int nctas = pass_ctas_any(d, q_len * hq / hkv);
    if (nctas <= 0) return cudaErrorInvalidConfiguration;
    const uint8_t *P = (const uint8_t *)params;
    SlotMap map{nullptr, block_table, pre_lens, max_blocks, num_blocks, hkv};
    map.q_len = q_len;
    cudaError_t e;
    if (d == 128)
        e = dtype == TQ_DTYPE_BF16
                ? step_prep_any<128, __nv_bfloat16>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, k_pool, v_pool,
                                                    max_ctx, nctas, w, status, st)
                : step_prep_any<128, float>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, k_pool, v_pool, max_ctx,
                                            nctas, w, status, st);
    else
        e = dtype == TQ_DTYPE_BF16
                ? step_prep_any<256, __nv_bfloat16>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, k_pool, v_pool,
                                                    max_ctx, nctas, w, status, st)
                : step_prep_any<256, float>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, k_pool, v_pool, max_ctx,
                                            nctas, w, status, st);
    if (e != cudaSuccess) return e;
    return launch_splitk(d, params, batch, q_len, hq, hkv, k_pool, v_pool, num_blocks, block_table, max_blocks,
                         pre_lens, q_len, max_ctx, out, ws, status, st);
}

}  // namespace tq
