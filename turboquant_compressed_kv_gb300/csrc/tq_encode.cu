// tq_encode.cu -- TurboQuant K/V encode kernels (bulk prefill and paged append).
//
// Method: "SwiftLM" README, "TurboQuantization: KV Cache Compression" ->
// "The Algorithm", K-Cache steps 1-5 (norm, WHT rotation, 3-bit Lloyd-Max
// cells, residual, QJL sign bits) and the V-Cache paragraph (steps 1-3, no
// QJL); the lilting.ch SwiftLM article, "KVキャッシュ圧縮の内訳", lists the
// same steps.  Slots follow the paged layout of the vLLM-MLX explainer,
// "Paged KVキャッシュ".
//
// A CTA of 4 warps encodes tiles of 16 (bulk) or 4 (append) vectors,
// persistent over tiles:
//  1. one warp per vector: norm, rotation (in registers and shuffles), cells,
//     residual (K) written to shared memory;
//  2. K only, all threads: the 16 QJL projections S rho, thread k computing
//     row k for every vector of the tile from S^T in shared memory (resident
//     for d=128, streamed in chunks for d=256); sign bits to shared memory;
//  3. one warp per vector: ballot-pack cells and signs, byte/word stores.
// One launch may carry K (blockIdx.y == 0) and V (blockIdx.y == 1) tiles.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kWarps = 4;                  // warps per CTA

// Where vector v of a launch goes: slot (or -1 to skip) and its input row.
struct SlotMap {
    const int64_t *slots;                  // bulk: slots[token]
    const int32_t *block_table;            // append: slot from the block table and length
    const int32_t *ctx_lens;
    int max_blocks;
    int64_t num_blocks;
    int n_heads;
    __device__ int64_t slot(int64_t token, int32_t *status, bool report) const {
        int64_t s = -1;
        if (slots) {
            s = slots[token];
            if (s < 0) return -1;
        } else {
            const int Lb = ctx_lens[token];
            if (Lb < 0) return -1;
            const int lb = Lb / kBlock;
            const int64_t blk = (lb < max_blocks) ? (int64_t)block_table[(size_t)token * max_blocks + lb] : -1;
            s = (blk >= 0) ? blk * kBlock + (Lb % kBlock) : -2;
            if (s == -2) {   // no block for this position
                if (report) flag_status(status, TQ_STATUS_BAD_SLOT);
                return -1;
            }
        }
        if (s / kBlock >= num_blocks) {
            if (report) flag_status(status, TQ_STATUS_BAD_SLOT);
            return -1;
        }
        return s;
    }
};

// TILE vectors per CTA: 16 for bulk encodes (each S^T read serves 16
// vectors), 4 for the one-token append (more CTAs, shorter latency chains).
template <int D, int TILE>
struct EncSmem {
    static constexpr bool kResident = (D == 128);
    static constexpr size_t kST = kResident ? (size_t)D * D * 4 : (size_t)2 * kProjRows * D * 4;
    static constexpr size_t kRho = (size_t)TILE * D * 4;
    static constexpr size_t kSgn = (size_t)TILE * D;
    static constexpr size_t kBytes = kST + kRho + kSgn;
};

// kinds: 1 = K only, 2 = V only, 3 = K (blockIdx.y 0) and V (blockIdx.y 1).
template <int D, int TILE, typename T>
__global__ void __launch_bounds__(kWarps * 32)
encode_kernel(const uint8_t *__restrict__ params, const T *__restrict__ xk, const T *__restrict__ xv, int64_t n_vec,
              SlotMap map, uint8_t *__restrict__ k_pool, uint8_t *__restrict__ v_pool, int kinds, int32_t *status) {
    constexpr int R = D / 32;
    constexpr int kTile = TILE, kPerWarp = TILE / kWarps;
    using SM = EncSmem<D, TILE>;
    extern __shared__ __align__(16) uint8_t smem[];
    float *sST = reinterpret_cast<float *>(smem);
    float (*s_rho)[D] = reinterpret_cast<float (*)[D]>(smem + SM::kST);
    uint8_t (*s_sgn)[D] = reinterpret_cast<uint8_t (*)[D]>(smem + SM::kST + SM::kRho);
    __shared__ float s_cent[8], s_thr[8];
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const bool is_k = (kinds == 3) ? (blockIdx.y == 0) : (kinds == 1);
    const T *__restrict__ x = is_k ? xk : xv;
    uint8_t *__restrict__ pool = is_k ? k_pool : v_pool;
    const float *gST = reinterpret_cast<const float *>(params + params_off_ST(D));
    if (is_k && SM::kResident) stage_st_rows<D, kWarps * 32>(sST, gST, 0, D);   // waited before first use
    if (threadIdx.x < 8) {
        s_cent[threadIdx.x] = ph->centroid[threadIdx.x];
        s_thr[threadIdx.x] = ph->threshold[threadIdx.x];
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const int64_t ntiles = (n_vec + kTile - 1) / kTile;

#pragma unroll 1
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t v0 = tile * kTile;
        int code[kPerWarp][R];
        float nrm[kPerWarp], gam[kPerWarp];
        int64_t slot[kPerWarp];
        // ---- 1. norm, rotation, cells, residual
#pragma unroll
        for (int j = 0; j < kPerWarp; ++j) {
            const int tv = warp + kWarps * j;              // vector within the tile
            const int64_t v = v0 + tv;
            slot[j] = -1;
            if (v < n_vec)   // a bad slot is reported once per token (by the K tile of an append)
                slot[j] = map.slot(v / map.n_heads, status, (kinds != 3 || is_k) && lane == 0 && (v % map.n_heads) == 0);
            float val[R];
            int dims[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                dims[r] = is_k ? kdim<D>(lane, r) : vdim<D>(lane, r);
                val[r] = (slot[j] >= 0) ? to_f32<T>(x[v * D + dims[r]]) : 0.f;
            }
            float ss = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) ss = fmaf(val[r], val[r], ss);
            const float n = sqrtf(warp_sum(ss));
#pragma unroll
            for (int r = 0; r < R; ++r) val[r] *= __ldg(Dsign + dims[r]);
            fwht_warp<R>(val, lane);                       // z = H(D x) / n = sqrt(d) Pi (x/n)
            float g2 = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float z = (n > 0.f) ? val[r] / n : 0.f;
                int k = 0;
#pragma unroll
                for (int t = 0; t < 7; ++t) k += (z >= s_thr[t]) ? 1 : 0;
                code[j][r] = k;
                if (is_k) {
                    const float rho = z - s_cent[k];     // residual, rotated unit-variance domain
                    g2 = fmaf(rho, rho, g2);
                    s_rho[tv][dims[r]] = rho;
                }
            }
            nrm[j] = n;
            gam[j] = is_k ? sqrtf(warp_sum(g2)) / sqrtf((float)D) : 0.f;   // ||y - c/sqrt d|| = ||rho|| / sqrt d
        }
        // ---- 2. QJL projections of the tile (K only): bit k = [(S rho)_k >= 0]
        if (is_k) {
            constexpr int KPT = D / (kWarps * 32);
            float acc[KPT][kTile];
#pragma unroll
            for (int u = 0; u < KPT; ++u)
#pragma unroll
                for (int t = 0; t < kTile; ++t) acc[u][t] = 0.f;
            if (SM::kResident) {
                cp_async_wait_all();
                __syncthreads();
                project_rows<D, kTile, kWarps * 32>(sST, 0, D, s_rho, acc);
            } else {
                __syncthreads();
                project_streamed<D, kTile, kWarps * 32>(gST, sST, s_rho, acc);
            }
#pragma unroll
            for (int u = 0; u < KPT; ++u)
#pragma unroll
                for (int t = 0; t < kTile; ++t) s_sgn[t][threadIdx.x + 128 * u] = acc[u][t] >= 0.f ? 1 : 0;
            __syncthreads();
        }
        // ---- 3. pack and store
#pragma unroll
        for (int j = 0; j < kPerWarp; ++j) {
            if (slot[j] < 0) continue;                     // warp-uniform
            const int tv = warp + kWarps * j;
            const int head = (int)((v0 + tv) % map.n_heads);
            const int64_t blk = slot[j] / kBlock;
            const int off = (int)(slot[j] % kBlock);
            if (is_k) {
                uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * k_record(D);
                uint32_t *planes = reinterpret_cast<uint32_t *>(rec);
                constexpr int NW = D / 128;
                const int gid = off & 7, th = off >> 3;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t w0 = __ballot_sync(0xffffffffu, code[j][r] & 1);
                    const uint32_t w1 = __ballot_sync(0xffffffffu, (code[j][r] >> 1) & 1);
                    const uint32_t w2 = __ballot_sync(0xffffffffu, (code[j][r] >> 2) & 1);
                    const uint32_t ws = __ballot_sync(0xffffffffu, s_sgn[tv][kdim<D>(lane, r)]);
                    if (lane == r) {
                        const int L = 4 * gid + (r & 3);
                        const size_t word = (size_t)(L * 2 + th) * NW + (r >> 2);
                        constexpr size_t PW = 2 * D / 4;   // words per plane
                        planes[word] = w0;
                        planes[PW + word] = w1;
                        planes[2 * PW + word] = w2;
                        planes[3 * PW + word] = ws;
                    }
                }
                if (lane == 0)
                    *reinterpret_cast<__half2 *>(rec + 8 * D + 4 * off) =
                        __halves2half2(__float2half_rn(nrm[j]), __float2half_rn(gam[j]));
            } else {
                uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * v_record(D);
                constexpr int NWV = D / 64, NM = D / 128;
                const int tigv = (off & 7) >> 1, jb = (off >> 3) + 2 * (off & 1);   // lane tig, byte in word
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t w0 = __ballot_sync(0xffffffffu, code[j][r] & 1);
                    const uint32_t w1 = __ballot_sync(0xffffffffu, (code[j][r] >> 1) & 1);
                    const uint32_t w2 = __ballot_sync(0xffffffffu, (code[j][r] >> 2) & 1);
                    if ((lane >> 2) == r) {
                        const int beta = lane & 3, tau = 4 * r + beta;
                        const int mhi = tau % NM, rh = (tau / NM) & 1, gid = tau / (2 * NM);
                        const size_t byte = ((size_t)(4 * gid + tigv) * NWV + 2 * mhi + rh) * 4 + jb;
                        rec[byte] = (uint8_t)(w0 >> (8 * beta));
                        rec[2 * D + byte] = (uint8_t)(w1 >> (8 * beta));
                        rec[4 * D + byte] = (uint8_t)(w2 >> (8 * beta));
                    }
                }
                if (lane == 0) *reinterpret_cast<__half *>(rec + 6 * D + 2 * off) = __float2half_rn(nrm[j]);
            }
        }
        __syncthreads();   // s_rho / s_sgn are rewritten by the next tile
    }
}

template <int D, int TILE, typename T>
cudaError_t launch_enc(const void *params, const void *xk, const void *xv, int64_t n_vec, const SlotMap &map,
                       void *kp, void *vp, int kinds, int32_t *status, cudaStream_t st) {
    const int64_t ntiles = (n_vec + TILE - 1) / TILE;
    if (ntiles <= 0) return cudaSuccess;
    const int ny = (kinds == 3) ? 2 : 1;
    const int64_t cap = 152 * 2;               // persistent: two CTAs per SM
    const unsigned gx = (unsigned)(ntiles < cap ? ntiles : cap);
    constexpr size_t smem = EncSmem<D, TILE>::kBytes;
    auto kern = encode_kernel<D, TILE, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(gx, ny), kWarps * 32, smem, st>>>((const uint8_t *)params, (const T *)xk, (const T *)xv, n_vec, map,
                                                  (uint8_t *)kp, (uint8_t *)vp, kinds, status);
    return cudaGetLastError();
}

template <int TILE>
cudaError_t launch_any(int d, int dtype, const void *params, const void *xk, const void *xv, int64_t n_vec,
                       const SlotMap &map, void *kp, void *vp, int kinds, int32_t *status, cudaStream_t st) {
    if (d == 128)
        return dtype == TQ_DTYPE_BF16
                   ? launch_enc<128, TILE, __nv_bfloat16>(params, xk, xv, n_vec, map, kp, vp, kinds, status, st)
                   : launch_enc<128, TILE, float>(params, xk, xv, n_vec, map, kp, vp, kinds, status, st);
    return dtype == TQ_DTYPE_BF16
               ? launch_enc<256, TILE, __nv_bfloat16>(params, xk, xv, n_vec, map, kp, vp, kinds, status, st)
               : launch_enc<256, TILE, float>(params, xk, xv, n_vec, map, kp, vp, kinds, status, st);
}

}  // namespace

cudaError_t launch_encode(bool is_k, int d, int dtype, const void *params, const void *x, int64_t n_tokens,
                          int n_heads, const int64_t *slots, void *pool, int64_t num_blocks, int32_t *status,
                          cudaStream_t st) {
    SlotMap map{slots, nullptr, nullptr, 0, num_blocks, n_heads};
    return launch_any<16>(d, dtype, params, is_k ? x : nullptr, is_k ? nullptr : x, n_tokens * n_heads, map,
                          is_k ? pool : nullptr, is_k ? nullptr : pool, is_k ? 1 : 2, status, st);
}

// One new token per sequence, K and V in one launch.
cudaError_t launch_append(int d, int dtype, const void *params, const void *k_new, const void *v_new, int batch,
                          int n_heads, const int32_t *bt, int max_blocks, const int32_t *ctx, void *kp, void *vp,
                          int64_t num_blocks, int32_t *status, cudaStream_t st) {
    SlotMap map{nullptr, bt, ctx, max_blocks, num_blocks, n_heads};
    return launch_any<4>(d, dtype, params, k_new, v_new, (int64_t)batch * n_heads, map, kp, vp, 3, status, st);
}

}  // namespace tq
