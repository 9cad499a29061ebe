// tq_encode.cu -- TurboQuant K/V encode kernels (bulk prefill and paged append).
//
// Method: "SwiftLM" README, "TurboQuantization: KV Cache Compression" ->
// "The Algorithm", K-Cache steps 1-5 (norm, WHT rotation, 3-bit Lloyd-Max
// cells, residual, QJL sign bits) and the V-Cache paragraph (steps 1-3, no
// QJL); the lilting.ch SwiftLM article, "KVキャッシュ圧縮の内訳", lists the
// same steps.  Slots follow the paged layout of the vLLM-MLX explainer,
// "Paged KVキャッシュ".
//
// One warp encodes one (token, kv head) vector.  Lane l holds coordinates
// kdim/vdim(l, r) for r < d/32, so the rotation runs in registers and
// shuffles, and every packed word is one __ballot_sync.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kWarps = 4;   // warps per CTA in the encode kernels

struct EncodeSmem {
    float centroid[8];
    float threshold[8];
};

// Encode the vector at x (d contiguous values) into slot `slot` of the pool.
// rho_smem: per-warp scratch of d floats (K only).
template <int D, bool IS_K, typename T>
__device__ __forceinline__ void encode_vector(const uint8_t *__restrict__ params, const EncodeSmem &sm,
                                              const T *__restrict__ x, int64_t slot, int head, int n_heads,
                                              uint8_t *__restrict__ pool, float *rho_smem, int lane) {
    constexpr int R = D / 32;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    float v[R];
    int dims[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        dims[r] = IS_K ? kdim<D>(lane, r) : vdim<D>(lane, r);
        v[r] = to_f32<T>(x[dims[r]]);
    }
    // step 1: L2 norm
    float ss = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) ss = fmaf(v[r], v[r], ss);
    const float n = sqrtf(warp_sum(ss));
    // step 2: randomized WHT; z = sqrt(d) * Pi(x/n) = H(D x) / n
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] *= __ldg(Dsign + dims[r]);
    fwht_warp<R>(v, lane);
    int code[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float z = (n > 0.f) ? v[r] / n : 0.f;
        v[r] = z;
        // step 3: 3-bit Lloyd-Max cell = number of thresholds <= z
        int k = 0;
#pragma unroll
        for (int j = 0; j < 7; ++j) k += (z >= sm.threshold[j]) ? 1 : 0;
        code[r] = k;
    }
    const int64_t blk = slot / kBlock;
    const int off = (int)(slot % kBlock);
    if (IS_K) {
        // step 4: residual in the rotated, unit-variance domain: rho = z - c[cell]
        float g2 = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float rho = v[r] - sm.centroid[code[r]];
            v[r] = rho;
            g2 = fmaf(rho, rho, g2);
            rho_smem[dims[r]] = rho;
        }
        // gamma = ||y - c/sqrt d|| = ||rho|| / sqrt d
        const float gamma = sqrtf(warp_sum(g2)) / sqrtf((float)D);
        __syncwarp();
        // step 5: QJL signs, bit k = [(S rho)_k >= 0]  (sqrt d > 0 does not change a sign)
        const float *S = reinterpret_cast<const float *>(params + params_off_S(D));
        bool sbit[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float4 *row = reinterpret_cast<const float4 *>(S + (size_t)dims[r] * D);
            const float4 *rr = reinterpret_cast<const float4 *>(rho_smem);
            float acc = 0.f;
#pragma unroll 8
            for (int i = 0; i < D / 4; ++i) {
                const float4 a = __ldg(row + i);
                const float4 b = rr[i];
                acc = fmaf(a.x, b.x, acc);
                acc = fmaf(a.y, b.y, acc);
                acc = fmaf(a.z, b.z, acc);
                acc = fmaf(a.w, b.w, acc);
            }
            sbit[r] = acc >= 0.f;
        }
        __syncwarp();
        uint8_t *rec = pool + ((size_t)blk * n_heads + head) * k_record(D);
        uint32_t *planes = reinterpret_cast<uint32_t *>(rec);
        constexpr int NW = D / 128;
        const int gid = off & 7, th = off >> 3;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t w0 = __ballot_sync(0xffffffffu, code[r] & 1);
            const uint32_t w1 = __ballot_sync(0xffffffffu, (code[r] >> 1) & 1);
            const uint32_t w2 = __ballot_sync(0xffffffffu, (code[r] >> 2) & 1);
            const uint32_t ws = __ballot_sync(0xffffffffu, sbit[r]);
            if (lane == r) {
                const int L = 4 * gid + (r & 3);
                const size_t word = (size_t)(L * 2 + th) * NW + (r >> 2);
                const size_t plane_words = 2 * D / 4;
                planes[word] = w0;
                planes[plane_words + word] = w1;
                planes[2 * plane_words + word] = w2;
                planes[3 * plane_words + word] = ws;
            }
        }
        if (lane == 0) {
            __half2 nh = __halves2half2(__float2half_rn(n), __float2half_rn(gamma));
            *reinterpret_cast<__half2 *>(rec + 8 * D + 4 * off) = nh;
        }
    } else {
        uint8_t *rec = pool + ((size_t)blk * n_heads + head) * v_record(D);
        constexpr int NWV = D / 64;
        constexpr int NM = D / 128;
        const int tigv = (off & 7) >> 1, jb = (off >> 3) + 2 * (off & 1);   // lane tig, byte in word
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t w0 = __ballot_sync(0xffffffffu, code[r] & 1);
            const uint32_t w1 = __ballot_sync(0xffffffffu, (code[r] >> 1) & 1);
            const uint32_t w2 = __ballot_sync(0xffffffffu, (code[r] >> 2) & 1);
            if ((lane >> 2) == r) {
                const int beta = lane & 3;
                const int tau = 4 * r + beta;
                const int mhi = tau % NM, rh = (tau / NM) & 1, gid = tau / (2 * NM);
                const int L = 4 * gid + tigv;
                const size_t byte = ((size_t)L * NWV + 2 * mhi + rh) * 4 + jb;
                rec[byte] = (uint8_t)(w0 >> (8 * beta));
                rec[2 * D + byte] = (uint8_t)(w1 >> (8 * beta));
                rec[4 * D + byte] = (uint8_t)(w2 >> (8 * beta));
            }
        }
        if (lane == 0) *reinterpret_cast<__half *>(rec + 6 * D + 2 * off) = __float2half_rn(n);
    }
}

__device__ __forceinline__ void load_codebook(const uint8_t *params, EncodeSmem &sm) {
    const ParamsHeader *h = reinterpret_cast<const ParamsHeader *>(params);
    if (threadIdx.x < 8) {
        sm.centroid[threadIdx.x] = h->centroid[threadIdx.x];
        sm.threshold[threadIdx.x] = h->threshold[threadIdx.x];
    }
    __syncthreads();
}

__device__ __forceinline__ bool params_ok(const uint8_t *params, int d) {
    const ParamsHeader *h = reinterpret_cast<const ParamsHeader *>(params);
    return h->magic == kParamsMagic && h->d == d;
}

template <int D, bool IS_K, typename T>
__global__ void __launch_bounds__(kWarps * 32)
encode_kernel(const uint8_t *__restrict__ params, const T *__restrict__ x, int64_t n_tokens, int n_heads,
              const int64_t *__restrict__ slots, uint8_t *__restrict__ pool, int64_t num_blocks,
              int32_t *status) {
    __shared__ EncodeSmem sm;
    __shared__ __align__(16) float rho[kWarps][D];
    if (!params_ok(params, D)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    load_codebook(params, sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nv = n_tokens * n_heads;
    for (int64_t v = (int64_t)blockIdx.x * kWarps + warp; v < nv; v += (int64_t)gridDim.x * kWarps) {
        const int64_t tok = v / n_heads;
        const int head = (int)(v % n_heads);
        const int64_t slot = slots[tok];
        if (slot < 0) continue;
        if (slot / kBlock >= num_blocks) {
            if (lane == 0) flag_status(status, TQ_STATUS_BAD_SLOT);
            continue;
        }
        encode_vector<D, IS_K, T>(params, sm, x + v * D, slot, head, n_heads, pool, rho[warp], lane);
    }
}

// Paged append: item = (sequence, head, K or V); one warp per item.
template <int D, typename T>
__global__ void __launch_bounds__(kWarps * 32)
append_kernel(const uint8_t *__restrict__ params, const T *__restrict__ k_new, const T *__restrict__ v_new,
              int batch, int n_heads, const int32_t *__restrict__ block_table, int max_blocks,
              const int32_t *__restrict__ ctx_lens, uint8_t *__restrict__ k_pool, uint8_t *__restrict__ v_pool,
              int64_t num_blocks, int32_t *status) {
    __shared__ EncodeSmem sm;
    __shared__ __align__(16) float rho[kWarps][D];
    if (!params_ok(params, D)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    load_codebook(params, sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t items = (int64_t)batch * n_heads * 2;
    for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; it < items; it += (int64_t)gridDim.x * kWarps) {
        const bool is_k = (it & 1) == 0;
        const int64_t bh = it >> 1;
        const int b = (int)(bh / n_heads), head = (int)(bh % n_heads);
        const int L = ctx_lens[b];
        if (L < 0) continue;
        const int lb = L / kBlock;
        int64_t blk = -1;
        if (lb < max_blocks) blk = block_table[(size_t)b * max_blocks + lb];
        if (blk < 0 || blk >= num_blocks) {
            if (lane == 0 && is_k) flag_status(status, TQ_STATUS_BAD_SLOT);
            continue;
        }
        const int64_t slot = blk * kBlock + (L % kBlock);
        if (is_k)
            encode_vector<D, true, T>(params, sm, k_new + bh * D, slot, head, n_heads, k_pool, rho[warp], lane);
        else
            encode_vector<D, false, T>(params, sm, v_new + bh * D, slot, head, n_heads, v_pool, rho[warp], lane);
    }
}

int grid_for(int64_t items) {
    int64_t g = (items + kWarps - 1) / kWarps;
    const int64_t cap = 152 * 16;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

}  // namespace

// ---------------------------------------------------------------- launchers

template <int D, bool IS_K, typename T>
static cudaError_t launch_encode_t(const void *params, const void *x, int64_t n_tokens, int n_heads,
                                   const int64_t *slots, void *pool, int64_t num_blocks, int32_t *status,
                                   cudaStream_t st) {
    encode_kernel<D, IS_K, T><<<grid_for(n_tokens * n_heads), kWarps * 32, 0, st>>>(
        (const uint8_t *)params, (const T *)x, n_tokens, n_heads, slots, (uint8_t *)pool, num_blocks, status);
    return cudaGetLastError();
}

cudaError_t launch_encode(bool is_k, int d, int dtype, const void *params, const void *x, int64_t n_tokens,
                          int n_heads, const int64_t *slots, void *pool, int64_t num_blocks, int32_t *status,
                          cudaStream_t st) {
#define TQ_ENC(DD, K, TT) return launch_encode_t<DD, K, TT>(params, x, n_tokens, n_heads, slots, pool, num_blocks, status, st)
    if (d == 128) {
        if (is_k) { if (dtype == TQ_DTYPE_BF16) TQ_ENC(128, true, __nv_bfloat16); TQ_ENC(128, true, float); }
        if (dtype == TQ_DTYPE_BF16) TQ_ENC(128, false, __nv_bfloat16);
        TQ_ENC(128, false, float);
    }
    if (is_k) { if (dtype == TQ_DTYPE_BF16) TQ_ENC(256, true, __nv_bfloat16); TQ_ENC(256, true, float); }
    if (dtype == TQ_DTYPE_BF16) TQ_ENC(256, false, __nv_bfloat16);
    TQ_ENC(256, false, float);
#undef TQ_ENC
}

template <int D, typename T>
static cudaError_t launch_append_t(const void *params, const void *k_new, const void *v_new, int batch,
                                   int n_heads, const int32_t *bt, int max_blocks, const int32_t *ctx,
                                   void *kp, void *vp, int64_t num_blocks, int32_t *status, cudaStream_t st) {
    append_kernel<D, T><<<grid_for((int64_t)batch * n_heads * 2), kWarps * 32, 0, st>>>(
        (const uint8_t *)params, (const T *)k_new, (const T *)v_new, batch, n_heads, bt, max_blocks, ctx,
        (uint8_t *)kp, (uint8_t *)vp, num_blocks, status);
    return cudaGetLastError();
}

cudaError_t launch_append(int d, int dtype, const void *params, const void *k_new, const void *v_new, int batch,
                          int n_heads, const int32_t *bt, int max_blocks, const int32_t *ctx, void *kp, void *vp,
                          int64_t num_blocks, int32_t *status, cudaStream_t st) {
#define TQ_APP(DD, TT) return launch_append_t<DD, TT>(params, k_new, v_new, batch, n_heads, bt, max_blocks, ctx, kp, vp, num_blocks, status, st)
    if (d == 128) { if (dtype == TQ_DTYPE_BF16) TQ_APP(128, __nv_bfloat16); TQ_APP(128, float); }
    if (dtype == TQ_DTYPE_BF16) TQ_APP(256, __nv_bfloat16);
    TQ_APP(256, float);
#undef TQ_APP
}

}  // namespace tq
