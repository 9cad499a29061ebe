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
#include "tq_tc.cuh"
#include "tq_prep.cuh"

namespace tq {
namespace {

// kinds: 1 = K only, 2 = V only, 3 = K (blockIdx.y 0) and V (blockIdx.y 1).
template <int D, int TILE, typename T>
__global__ void __launch_bounds__(kEncWarps * 32)
encode_kernel(const uint8_t *__restrict__ params, const T *__restrict__ xk, const T *__restrict__ xv, int64_t n_vec,
              SlotMap map, uint8_t *__restrict__ k_pool, uint8_t *__restrict__ v_pool, int kinds, int32_t *status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const bool is_k = (kinds == 3) ? (blockIdx.y == 0) : (kinds == 1);
    encode_tiles<D, TILE, T>(params, is_k ? xk : xv, n_vec, map, is_k ? k_pool : v_pool, is_k, kinds != 3 || is_k,
                             blockIdx.x, gridDim.x, smem, status);
}

// ---------------------------------------------------------------- bulk encode at d = 128, QJL on tcgen05
// A persistent CTA (16 warps) encodes tiles of 128 vectors:
//  1. the tile's inputs (contiguous rows) arrive by one bulk copy, two tiles in flight;
//  2. one warp per vector: norm, rotation, cells, residual, ballot-packed cell planes and
//     norms, as in encode_kernel; for K the residual rho (x 256) is written as f16 hi and lo
//     rows of the A operand (128-byte swizzle, K index 4 * lane + r);
//  3. K only: p = S rho for the 128 vectors as three f16 products S_hi rho_hi + S_lo rho_hi +
//     S_hi rho_lo on the tensor cores (M = 128 vectors, N = 128, K = 128, fp32 accumulation),
//     with S's rows permuted so that thread (vector, word) reads 32 consecutive columns in the
//     bit order of one sign-plane word.
namespace enc128 {
constexpr int D = 128, kRows = 128, kThreads = 512, kTileWarps = 16;
constexpr float kRhoScale = 256.f;          // keeps the f16 low parts of rho out of the subnormals
constexpr int oB = 0;                        // S hi, S lo: 2 x 32 KB
constexpr int oA = 65536;                    // rho hi, rho lo: 2 x 32 KB
constexpr int oX = 131072;                   // input tiles
template <typename T> __host__ __device__ constexpr int x_bytes() { return kRows * D * (int)sizeof(T); }
template <typename T> __host__ __device__ constexpr int n_xbuf() { return sizeof(T) == 2 ? 2 : 1; }
template <typename T> __host__ __device__ constexpr int smem_bytes() { return oX + n_xbuf<T>() * x_bytes<T>(); }
}  // namespace enc128

template <typename T>
__global__ void __launch_bounds__(enc128::kThreads, 1)
encode128_tc_kernel(const uint8_t *__restrict__ params, const T *__restrict__ x, int64_t n_vec, SlotMap map,
                    uint8_t *__restrict__ pool, int is_k, int32_t *status) {
    using namespace enc128;
    constexpr int R = D / 32, NXB = n_xbuf<T>(), XB = x_bytes<T>();
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t xfull[2], mmabar;
    __shared__ uint32_t tmem_base;
    __shared__ int64_t sSlot[kRows];
    __shared__ float s_cent[8], s_thr[8];
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ntiles = (n_vec + kRows - 1) / kRows;
    if ((int64_t)blockIdx.x >= ntiles) return;
    if (tid == 0) {
        tc::mbar_init(&xfull[0], 1);
        tc::mbar_init(&xfull[1], 1);
        tc::mbar_init(&mmabar, 1);
    }
    if (is_k && warp == 0) tc::tmem_alloc(&tmem_base, 128);
    if (tid < 8) {
        s_cent[tid] = ph->centroid[tid];
        s_thr[tid] = ph->threshold[tid];
    }
    if (is_k) {
        // B = S with rows permuted to sign-plane bit order and columns to the A operand's K order
        const float *S = reinterpret_cast<const float *>(params + params_off_S(D));
        for (int e = tid; e < D * D; e += kThreads) {
            const int n = e >> 7, k = e & 127;
            const float sv = __ldg(S + kdim<D>(n & 31, n >> 5) * D + kdim<D>(k >> 2, k & 3));
            const __half hi = __float2half_rn(sv);
            const __half lo = __float2half_rn(sv - __half2float(hi));
            const int off = tc::sw128_off(n, k, D);
            *reinterpret_cast<__half *>(smem + oB + off) = hi;
            *reinterpret_cast<__half *>(smem + oB + 32768 + off) = lo;
        }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = is_k ? tmem_base : 0u;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    bool timed_out = false;

    auto issue = [&](int64_t tile, int buf) {
        const int64_t v0 = tile * kRows;
        const int rows = (int)min((int64_t)kRows, n_vec - v0);
        const uint32_t bytes = (uint32_t)rows * D * sizeof(T);
        tc::mbar_arrive_expect_tx(&xfull[buf], bytes);
        tc::bulk_g2s(smem + oX + buf * XB, x + v0 * D, bytes, &xfull[buf]);
    };
    if (tid == 0)
        for (int b2 = 0; b2 < NXB; ++b2) {
            const int64_t t2 = blockIdx.x + (int64_t)b2 * gridDim.x;
            if (t2 < ntiles) issue(t2, b2);
        }

    int it = 0;
#pragma unroll 1
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
        const int buf = (NXB == 2) ? (it & 1) : 0, use = (NXB == 2) ? (it >> 1) : it;
        const int64_t v0 = tile * kRows;
        const int rows = (int)min((int64_t)kRows, n_vec - v0);
        if (tid < kRows) {
            const int64_t v = v0 + tid;
            sSlot[tid] = (tid < rows) ? map.slot(v / map.n_heads, status, (v % map.n_heads) == 0) : -1;
        }
        if (!tc::mbar_wait(&xfull[buf], use & 1)) timed_out = true;
        __syncthreads();
        const T *xt = reinterpret_cast<const T *>(smem + oX + buf * XB);
        // ---- one warp per vector
#pragma unroll 1
        for (int j = 0; j < kRows / kTileWarps; ++j) {
            const int v = warp + kTileWarps * j;
            const bool valid = v < rows;
            int dims[R];
            float val[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                dims[r] = is_k ? kdim<D>(lane, r) : vdim<D>(lane, r);
                val[r] = valid ? to_f32<T>(xt[v * D + dims[r]]) : 0.f;
            }
            float ss = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) ss = fmaf(val[r], val[r], ss);
            const float n = sqrtf(warp_sum(ss));
#pragma unroll
            for (int r = 0; r < R; ++r) val[r] *= __ldg(Dsign + dims[r]);
            fwht_warp<R>(val, lane);                 // z = H(D x) / n = sqrt(d) Pi (x/n)
            int code[R];
            float rho[R], g2 = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float z = (n > 0.f) ? val[r] / n : 0.f;
                int k = 0;
#pragma unroll
                for (int t = 0; t < 7; ++t) k += (z >= s_thr[t]) ? 1 : 0;
                code[r] = k;
                rho[r] = z - s_cent[k];
                g2 = fmaf(rho[r], rho[r], g2);
            }
            const int64_t slot = sSlot[v];
            if (is_k) {
                const float gam = sqrtf(warp_sum(g2)) / sqrtf((float)D);
                __half h[R], l[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float rs = valid ? rho[r] * kRhoScale : 0.f;
                    h[r] = __float2half_rn(rs);
                    l[r] = __float2half_rn(rs - __half2float(h[r]));
                }
                const int off = tc::sw128_off(v, 4 * lane, D);
                uint2 hw, lw;
                hw.x = (uint32_t)__half_as_ushort(h[0]) | ((uint32_t)__half_as_ushort(h[1]) << 16);
                hw.y = (uint32_t)__half_as_ushort(h[2]) | ((uint32_t)__half_as_ushort(h[3]) << 16);
                lw.x = (uint32_t)__half_as_ushort(l[0]) | ((uint32_t)__half_as_ushort(l[1]) << 16);
                lw.y = (uint32_t)__half_as_ushort(l[2]) | ((uint32_t)__half_as_ushort(l[3]) << 16);
                *reinterpret_cast<uint2 *>(smem + oA + off) = hw;
                *reinterpret_cast<uint2 *>(smem + oA + 32768 + off) = lw;
                if (slot >= 0) {
                    const int64_t blk = slot / kBlock;
                    const int o = (int)(slot % kBlock), head = (int)((v0 + v) % map.n_heads);
                    uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * k_record(D);
                    uint32_t *planes = reinterpret_cast<uint32_t *>(rec);
                    const int gid = o & 7, th = o >> 3;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t w0 = __ballot_sync(0xffffffffu, code[r] & 1);
                        const uint32_t w1 = __ballot_sync(0xffffffffu, (code[r] >> 1) & 1);
                        const uint32_t w2 = __ballot_sync(0xffffffffu, (code[r] >> 2) & 1);
                        if (lane == r) {
                            const size_t word = (size_t)(4 * gid + r) * 2 + th;
                            constexpr size_t PW = 2 * D / 4;
                            planes[word] = w0;
                            planes[PW + word] = w1;
                            planes[2 * PW + word] = w2;
                        }
                    }
                    if (lane == 0)
                        *reinterpret_cast<__half2 *>(rec + 8 * D + 4 * o) =
                            __halves2half2(__float2half_rn(n), __float2half_rn(gam));
                }
            } else if (slot >= 0) {
                const int64_t blk = slot / kBlock;
                const int o = (int)(slot % kBlock), head = (int)((v0 + v) % map.n_heads);
                uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * v_record(D);
                constexpr int NWV = D / 64, NM = D / 128;
                const int tigv = (o & 7) >> 1, jb = (o >> 3) + 2 * (o & 1);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t w0 = __ballot_sync(0xffffffffu, code[r] & 1);
                    const uint32_t w1 = __ballot_sync(0xffffffffu, (code[r] >> 1) & 1);
                    const uint32_t w2 = __ballot_sync(0xffffffffu, (code[r] >> 2) & 1);
                    if ((lane >> 2) == r) {
                        const int beta = lane & 3, tau = 4 * r + beta;
                        const int mhi = tau % NM, rh = (tau / NM) & 1, gid = tau / (2 * NM);
                        const size_t byte = ((size_t)(4 * gid + tigv) * NWV + 2 * mhi + rh) * 4 + jb;
                        rec[byte] = (uint8_t)(w0 >> (8 * beta));
                        rec[2 * D + byte] = (uint8_t)(w1 >> (8 * beta));
                        rec[4 * D + byte] = (uint8_t)(w2 >> (8 * beta));
                    }
                }
                if (lane == 0) *reinterpret_cast<__half *>(rec + 6 * D + 2 * o) = __float2half_rn(n);
            }
        }
        // ---- K: QJL projections of the tile on the tensor cores, then the sign plane
        if (is_k) {
            tc::fence_async_smem();
            tc::fence_before_sync();
            __syncthreads();
            if (tid == 0) {
                tc::fence_after_sync();
                const uint32_t bh = tc::smem_u32(smem + oB), bl = bh + 32768;
                const uint32_t ah = tc::smem_u32(smem + oA), al = ah + 32768;
                constexpr uint32_t id = tc::idesc_f16(kRows, D);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    tc::mma_ss_f16(tmem, tc::sw128_desc(ah, ks, kRows), tc::sw128_desc(bh, ks, D), id, ks > 0);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    tc::mma_ss_f16(tmem, tc::sw128_desc(al, ks, kRows), tc::sw128_desc(bh, ks, D), id, true);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    tc::mma_ss_f16(tmem, tc::sw128_desc(ah, ks, kRows), tc::sw128_desc(bl, ks, D), id, true);
                tc::mma_commit(&mmabar);
            }
            if (!tc::mbar_wait(&mmabar, it & 1)) timed_out = true;
            tc::fence_after_sync();
            // thread: vector row 32 (warp % 4) + lane, sign word tig = warp / 4 (columns 32 tig ..)
            const int vrow = 32 * (warp & 3) + lane, tig = warp >> 2;
            const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * tig;
            uint32_t sw = 0u;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float pv[16];
                tc::ld16(taddr + 16 * q, pv);
                tc::wait_ld();
#pragma unroll
                for (int x2 = 0; x2 < 16; ++x2) sw |= (pv[x2] >= 0.f ? 1u : 0u) << (16 * q + x2);
            }
            const int64_t slot = (vrow < rows) ? sSlot[vrow] : -1;
            if (slot >= 0) {
                const int64_t blk = slot / kBlock;
                const int o = (int)(slot % kBlock), head = (int)((v0 + vrow) % map.n_heads);
                uint32_t *planes = reinterpret_cast<uint32_t *>(pool + ((size_t)blk * map.n_heads + head) * k_record(D));
                constexpr size_t PW = 2 * D / 4;
                planes[3 * PW + (size_t)(4 * (o & 7) + tig) * 2 + (o >> 3)] = sw;
            }
            tc::fence_before_sync();
        }
        __syncthreads();   // the input buffer, the A operand and the accumulator are free
        if (tid == 0) {
            const int64_t nt = tile + (int64_t)NXB * gridDim.x;
            if (nt < ntiles) issue(nt, buf);
        }
    }
    if (timed_out) flag_status(status, TQ_STATUS_TIMEOUT);
    if (is_k) {
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::tmem_dealloc(tmem, 128);
    }
}

template <typename T>
cudaError_t launch_enc128(const void *params, const void *x, int64_t n_vec, const SlotMap &map, void *pool, bool is_k,
                          int32_t *status, cudaStream_t st) {
    const int64_t ntiles = (n_vec + enc128::kRows - 1) / enc128::kRows;
    if (ntiles <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    constexpr int smem = enc128::smem_bytes<T>();
    auto kern = encode128_tc_kernel<T>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(ntiles < sms ? ntiles : sms);
    kern<<<grid, enc128::kThreads, smem, st>>>((const uint8_t *)params, (const T *)x, n_vec, map, (uint8_t *)pool,
                                               is_k ? 1 : 0, status);
    return cudaGetLastError();
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
    kern<<<dim3(gx, ny), kEncWarps * 32, smem, st>>>((const uint8_t *)params, (const T *)xk, (const T *)xv, n_vec, map,
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
    if (d == 128 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0)
        return dtype == TQ_DTYPE_BF16
                   ? launch_enc128<__nv_bfloat16>(params, x, n_tokens * n_heads, map, pool, is_k, status, st)
                   : launch_enc128<float>(params, x, n_tokens * n_heads, map, pool, is_k, status, st);
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
