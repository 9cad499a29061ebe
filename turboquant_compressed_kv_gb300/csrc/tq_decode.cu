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
// Launches per call: (1) query prep (qbar, u, f16 operand fragments and offset constants),
// or, for the decode step, the append of the new token together with the query prep; (2) the
// split-K pass, persistent: the context of every (sequence, kv head) is cut into 128-token
// chunks, and CTA c of P takes the c-th of P equal, contiguous ranges of the chunk sequence
// ordered by (sequence, kv head, chunk) ("stream-K"), worked out by every CTA from the lengths.
// A (sequence, kv head) inside one CTA's range is finished there; one shared by several CTAs
// leaves an online-softmax partial (m, l, acc[d]) per query head from each, which (3) the merge
// kernel combines.  Either way one inverse rotation per (sequence, query head) is applied at
// the end.
#include <atomic>

#include "tq_split.cuh"

namespace tq {

size_t decode_workspace_bytes(int d, int batch, int hq, int max_ctx) {
    if (!valid_d(d) || batch <= 0 || hq <= 0 || max_ctx < 0) return 0;
    size_t off[3];
    return ws_sizes(d, batch, hq, off);
}

namespace {

// ---------------------------------------------------------------- (1) query prep (body in tq_prep.cuh)
template <int D, int NTK, typename T>
__global__ void __launch_bounds__(128)
qprep_kernel(const uint8_t *__restrict__ params, const T *__restrict__ q, int batch, int q_len, int hq, int hkv,
             uint8_t *__restrict__ packs) {
    extern __shared__ __align__(16) uint8_t qsm[];
    pdl_launch_dependents();
    qprep_slice<D, NTK, T>(params, q, batch, q_len, hq, hkv, packs, blockIdx.x, qsm);
}

// Persistent CTAs of the pass on the current device: up to kCtasPerSm per SM
// (fewer if the kernel's resources allow fewer), for at most kMaxSms SMs.
// Cached per (device, d, G): the occupancy query is not free.
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
cudaError_t qprep_launch_t(const uint8_t *P, const void *q, int batch, int q_len, int hq, int hkv, const WsLayout &w,
                           cudaStream_t st) {
    constexpr size_t smem = qprep_smem<D>();
    auto kern = qprep_kernel<D, NTK, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<qprep_ctas(D, batch * q_len * hq), 128, smem, st>>>(P, (const T *)q, batch, q_len, hq, hkv, w.packs);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t qprep_launch(const uint8_t *P, const void *q, int batch, int q_len, int hq, int hkv, const WsLayout &w,
                         cudaStream_t st) {
    // n-tile count of the K-side operand: (2G + 7) / 8 for G = q_len * hq / hkv columns, as in the passes
    if (q_len * hq / hkv <= 4) return qprep_launch_t<D, 1, T>(P, q, batch, q_len, hq, hkv, w, st);
    return qprep_launch_t<D, 2, T>(P, q, batch, q_len, hq, hkv, w, st);
}

}  // namespace

cudaError_t launch_qprep(int d, int dtype, const void *params, const void *q, int batch, int q_len, int hq, int hkv,
                         void *ws, cudaStream_t st) {
    const WsLayout w = ws_layout(ws, d, batch, q_len * hq);
    const uint8_t *P = (const uint8_t *)params;
    if (d == 128)
        return dtype == TQ_DTYPE_BF16 ? qprep_launch<128, __nv_bfloat16>(P, q, batch, q_len, hq, hkv, w, st)
                                      : qprep_launch<128, float>(P, q, batch, q_len, hq, hkv, w, st);
    return dtype == TQ_DTYPE_BF16 ? qprep_launch<256, __nv_bfloat16>(P, q, batch, q_len, hq, hkv, w, st)
                                  : qprep_launch<256, float>(P, q, batch, q_len, hq, hkv, w, st);
}

cudaError_t launch_splitk(int d, const void *params, int batch, int q_len, int hq, int hkv, const void *k_pool,
                          const void *v_pool, int64_t num_blocks, const int32_t *block_table, int max_blocks,
                          const int32_t *ctx_lens, int ctx_add, int max_ctx, float *out, void *ws, int32_t *status,
                          cudaStream_t st, bool early, float *lse) {
    const WsLayout w = ws_layout(ws, d, batch, q_len * hq);
    const int G = q_len * hq / hkv;   // operand columns per kv head
    const int nctas = pass_ctas_any(d, G);
    if (nctas <= 0) return cudaErrorInvalidConfiguration;
    const uint8_t *P = (const uint8_t *)params;
    return warp_pass_launch(d, G, nctas, st, P, batch, q_len, hq, hkv, (const uint8_t *)k_pool, (const uint8_t *)v_pool,
                            num_blocks, block_table, max_blocks, ctx_lens, ctx_add, max_ctx, early, w, out, lse,
                            status);
}

// ---------------------------------------------------------------- the append and the decode step
// One launch runs the append of the new tokens (K slices, V rows: tq_prep.cuh) and, for the
// step, the query prep side by side; the pass follows.  pre_lens[b] is the position of
// sequence b's first new token, and the pass attends pre_lens[b] + q_len tokens.
namespace {

template <int D> __host__ __device__ constexpr size_t append_smem() {
    return append_k_smem<D>() > append_v_smem<D>() ? append_k_smem<D>() : append_v_smem<D>();
}

template <int D, int NTK, typename T>
__global__ void __launch_bounds__(128)
step_prep_kernel(const uint8_t *__restrict__ params, const T *__restrict__ k_new, const T *__restrict__ v_new,
                 const T *__restrict__ q, int batch, int q_len, int hq, int hkv, SlotMap map, uint8_t *__restrict__ k_pool,
                 uint8_t *__restrict__ v_pool, int n_app_k, int n_app_v, uint8_t *__restrict__ packs, int32_t *status) {
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_launch_dependents();
    const int blk = blockIdx.x;
    const int64_t n_vec = (int64_t)batch * q_len * hkv;
    if (blk < n_app_k)
        append_k_slice<D, T>(params, k_new, n_vec, map, k_pool, blk, smem, status);
    else if (blk < n_app_k + n_app_v)
        append_v_rows<D, T>(params, v_new, n_vec, map, v_pool, false, blk - n_app_k, smem, status);
    else if (q)
        qprep_slice<D, NTK, T>(params, q, batch, q_len, hq, hkv, packs, blk - n_app_k - n_app_v, smem);
}

template <int D, int NTK, typename T>
cudaError_t step_prep_launch(const uint8_t *P, const void *k_new, const void *v_new, const void *q, int batch,
                             int q_len, int hq, int hkv, const SlotMap &map, void *kp, void *vp, uint8_t *packs,
                             int32_t *status, cudaStream_t st) {
    constexpr size_t as = append_smem<D>(), qs = qprep_smem<D>();
    constexpr size_t smem = as > qs ? as : qs;
    auto kern = step_prep_kernel<D, NTK, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t n_vec = (int64_t)batch * q_len * hkv;
    const int n_app_k = append_k_ctas(D, n_vec), n_app_v = append_v_ctas(n_vec);
    const int n_q = q ? qprep_ctas(D, batch * q_len * hq) : 0;
    kern<<<n_app_k + n_app_v + n_q, 128, q ? smem : as, st>>>(P, (const T *)k_new, (const T *)v_new, (const T *)q, batch,
                                                             q_len, hq, hkv, map, (uint8_t *)kp, (uint8_t *)vp, n_app_k,
                                                             n_app_v, packs, status);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t step_prep_any(const uint8_t *P, const void *k_new, const void *v_new, const void *q, int batch, int q_len,
                          int hq, int hkv, const SlotMap &map, void *kp, void *vp, uint8_t *packs, int32_t *status,
                          cudaStream_t st) {
    if (!q || q_len * hq / hkv <= 4)
        return step_prep_launch<D, 1, T>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, kp, vp, packs, status, st);
    return step_prep_launch<D, 2, T>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, kp, vp, packs, status, st);
}

cudaError_t step_prep(int d, int dtype, const void *params, const void *k_new, const void *v_new, const void *q,
                      int batch, int q_len, int hq, int hkv, const SlotMap &map, void *kp, void *vp, uint8_t *packs,
                      int32_t *status, cudaStream_t st) {
    const uint8_t *P = (const uint8_t *)params;
    if (d == 128)
        return dtype == TQ_DTYPE_BF16
                   ? step_prep_any<128, __nv_bfloat16>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, kp, vp, packs,
                                                       status, st)
                   : step_prep_any<128, float>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, kp, vp, packs, status, st);
    return dtype == TQ_DTYPE_BF16
               ? step_prep_any<256, __nv_bfloat16>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, kp, vp, packs,
                                                   status, st)
               : step_prep_any<256, float>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, kp, vp, packs, status, st);
}
}  // namespace

// One new token per sequence (K and V), through the step's prep launch without a query.
cudaError_t launch_append(int d, int dtype, const void *params, const void *k_new, const void *v_new, int batch,
                          int n_heads, const int32_t *bt, int max_blocks, const int32_t *ctx, void *kp, void *vp,
                          int64_t num_blocks, int32_t *status, cudaStream_t st) {
    SlotMap map{nullptr, bt, ctx, max_blocks, num_blocks, n_heads};
    return step_prep(d, dtype, params, k_new, v_new, nullptr, batch, 1, n_heads, n_heads, map, kp, vp, nullptr, status,
                     st);
}

cudaError_t launch_step(int d, int dtype, const void *params, const void *k_new, const void *v_new, const void *q,
                        int batch, int q_len, int hq, int hkv, const int32_t *block_table, int max_blocks,
                        const int32_t *pre_lens, int max_ctx, void *k_pool, void *v_pool, int64_t num_blocks,
                        float *out, void *ws, int32_t *status, cudaStream_t st) {
    const WsLayout w = ws_layout(ws, d, batch, q_len * hq);
    SlotMap map{nullptr, block_table, pre_lens, max_blocks, num_blocks, hkv};
    map.q_len = q_len;
    cudaError_t e = step_prep(d, dtype, params, k_new, v_new, q, batch, q_len, hq, hkv, map, k_pool, v_pool, w.packs,
                              status, st);
    if (e != cudaSuccess) return e;
    return launch_splitk(d, params, batch, q_len, hq, hkv, k_pool, v_pool, num_blocks, block_table, max_blocks,
                         pre_lens, q_len, max_ctx, out, ws, status, st, true);
}

}  // namespace tq
