// tq_split.cuh -- pieces shared by the decode launches (tq_decode.cu: query prep, the fused
// step and the dispatch; tq_decode_warp.cu: the pass): tuning switches, the workspace layout,
// block-table lookup and the final inverse rotation.
#pragma once

#include "tq_internal.cuh"
#include "tq_prep.cuh"

namespace tq {

#ifndef TQ_SPLITK_BPW
#define TQ_SPLITK_BPW 2          // blocks scored per warp per chunk
#endif
#ifndef TQ_SPLITK_CTAS_PER_SM
#define TQ_SPLITK_CTAS_PER_SM 3  // persistent CTAs per SM (at most)
#endif
constexpr int kCtasPerSm = TQ_SPLITK_CTAS_PER_SM;

#ifndef TQ_DECODE_PDL
#define TQ_DECODE_PDL 1          // the pass may launch while the prep launch before it finishes
#endif

// Launch of a decode pass.  With TQ_DECODE_PDL it is a programmatic dependent launch: its CTAs
// may be launched while the prep kernel before it on the stream finishes (the prep signals
// pdl_launch_dependents as it starts), and they wait for that kernel's completion (pdl_wait)
// before touching memory.  After any other kernel it behaves as an ordinary launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pass(void (*kern)(KArgs...), int nctas, int threads, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nctas);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = TQ_DECODE_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace: query packs [B*Hkv] | chunk prefix int64[B+1] (written by the pass for the merge
// kernel) | partials [P][2][G][d+4].  Sized with Hq >= Hkv, G <= min(8, Hq) and
// P <= kCtasPerSm * kMaxSms.
struct WsLayout {
    uint8_t *packs;
    int64_t *cpre;
    float *part;
};
inline size_t ws_sizes(int d, int batch, int hq, size_t *off) {
    const int gmax = hq < 8 ? hq : 8;
    const size_t pmax = (size_t)kCtasPerSm * kMaxSms;
    const size_t per_head = kPackBytes(d);
    off[0] = 0;
    off[1] = off[0] + align256((size_t)batch * hq * per_head);
    off[2] = off[1] + align256(((size_t)batch + 1) * 8);
    return off[2] + pmax * 2 * gmax * kPartStride(d) * sizeof(float);
}
inline WsLayout ws_layout(void *ws, int d, int batch, int hq) {
    size_t off[3];
    ws_sizes(d, batch, hq, off);
    uint8_t *base = reinterpret_cast<uint8_t *>(ws);
    return WsLayout{base + off[0], reinterpret_cast<int64_t *>(base + off[1]), reinterpret_cast<float *>(base + off[2])};
}

// physical block of logical block lb, or -1 (past the table or outside the pool)
__device__ __forceinline__ int64_t block_of(const int32_t *__restrict__ bt, int b, int max_blocks, int lb,
                                            int64_t num_blocks) {
    if (lb >= max_blocks) return -1;
    const int64_t p = bt[(size_t)b * max_blocks + lb];
    return (p >= 0 && p < num_blocks) ? p : -1;
}

// out[row] = Pi^T (v / l): D (H v) / (l sqrt d), v spread over the warp as v[r] at lane
template <int D>
__device__ __forceinline__ void finish_row(float (&v)[D / 32], float l, const uint8_t *params, float *out_row,
                                           int lane) {
    constexpr int R = D / 32;
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] *= inv;
    fwht_warp<R>(v, lane);
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const float inv_sd = rsqrtf((float)D);
#pragma unroll
    for (int r = 0; r < R; ++r) out_row[32 * r + lane] = v[r] * inv_sd * __ldg(Dsign + 32 * r + lane);
}


// The decode pass (tq_decode_warp.cu): persistent CTAs it runs with on the current device, and
// its launch.  G counts operand columns: q_len queries x the query heads of a kv head.
int warp_pass_ctas(int d, int G);
cudaError_t warp_pass_launch(int d, int G, int nctas, cudaStream_t st, const uint8_t *P, int batch, int q_len, int hq,
                             int hkv, const uint8_t *kp, const uint8_t *vp, int64_t nb, const int32_t *bt, int mb,
                             const int32_t *ctx, int ctx_add, int max_ctx, bool early, const WsLayout &w, float *out,
                             float *lse, int32_t *status);

}  // namespace tq
