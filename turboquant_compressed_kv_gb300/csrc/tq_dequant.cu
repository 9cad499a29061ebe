// tq_dequant.cu -- bulk dequantisation of paged blocks back to dense K / V vectors, for a
// prefill (or any dense attention) that runs over a compressed prefix.
//
// The reconstruction is the estimator the decode scores with, written out per vector
// (SwiftLM README, "TurboQuantization: KV Cache Compression" -> "The Algorithm": the
// codebook value of each rotated coordinate, plus for K the QJL term of the residual):
//   K: k = n  Pi^T ( c[cell]/sqrt d + sqrt(pi/2)/d * gamma * S^T (2 sign - 1) )
//   V: v = nv Pi^T ( c[cell]/sqrt d )
// with Pi^T y = D (H y) / sqrt d.  Attention over these vectors is exactly the decode's
// attention (q . k = n <Pi q, ...>), which is what makes a dense prefill over them valid.
//
// A CTA of 4 warps takes one (block, kv head) record at a time (16 slots):
//  1. one warp per slot: the cell bits (and for K the sign bits) are read back in the
//     encoder's lane order (the inverse of its ballot packing), the signs go to shared
//     memory as +-1;
//  2. K only, all threads: S^T b for the 16 slots from S's rows in shared memory (resident
//     at d = 128, streamed at d = 256);
//  3. one warp per slot: codebook values plus the QJL term, the inverse rotation in
//     registers and shuffles, the norm, and the store.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kDqWarps = 4, kDqTile = kBlock;   // one record (16 slots) per tile

template <int D>
struct DqSmem {
    static constexpr bool kResident = (D == 128);
    static constexpr size_t kS = kResident ? (size_t)D * D * 4 : (size_t)2 * kProjRows * D * 4;
    static constexpr size_t kB = (size_t)kDqTile * D * 4;   // signs (+-1), then S^T b
    static constexpr size_t kBytes = kS + kB;
};

template <typename TO> __device__ __forceinline__ TO from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <int D, typename TO>
__global__ void __launch_bounds__(kDqWarps * 32)
dequant_kernel(const uint8_t *__restrict__ params, const uint8_t *__restrict__ pool, int64_t num_blocks, int n_heads,
               const int32_t *__restrict__ block_ids, int n_ids, int is_k, TO *__restrict__ out, int32_t *status) {
    constexpr int R = D / 32, NT = kDqWarps * 32, PER_WARP = kDqTile / kDqWarps;
    using SM = DqSmem<D>;
    extern __shared__ __align__(16) uint8_t smem[];
    float *sS = reinterpret_cast<float *>(smem);
    float (*s_b)[D] = reinterpret_cast<float (*)[D]>(smem + SM::kS);
    __shared__ float s_cent[8];
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const float *gS = reinterpret_cast<const float *>(params + params_off_S(D));
    if (is_k && SM::kResident) stage_st_rows<D, NT>(sS, gS, 0, D);   // S's rows; waited before first use
    if (threadIdx.x < 8) s_cent[threadIdx.x] = ph->centroid[threadIdx.x];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const float inv_sd = rsqrtf((float)D);
    const float qjl = 1.2533141373155003f / (float)D;   // sqrt(pi/2) / d
    const size_t rec_bytes = is_k ? k_record(D) : v_record(D);
    const int64_t units = (int64_t)n_ids * n_heads;

#pragma unroll 1
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int j = (int)(u / n_heads), h = (int)(u % n_heads);
        const int64_t blk = block_ids[j];
        const bool good = blk >= 0 && blk < num_blocks;
        if (!good && threadIdx.x == 0) flag_status(status, TQ_STATUS_BAD_SLOT);
        const uint8_t *rec = pool + ((size_t)(good ? blk : 0) * n_heads + h) * rec_bytes;
        float val[PER_WARP][R];
        int dims[R];
#pragma unroll
        for (int r = 0; r < R; ++r) dims[r] = is_k ? kdim<D>(lane, r) : vdim<D>(lane, r);
        float nrm[PER_WARP], gam[PER_WARP];
        // ---- 1. cells (and signs) of this warp's slots, in the encoder's lane order
#pragma unroll
        for (int jj = 0; jj < PER_WARP; ++jj) {
            const int t = warp + kDqWarps * jj;   // slot in the block
            if (is_k) {
                constexpr int NW = D / 128;
                constexpr size_t PW = 2 * D / 4;   // words per plane
                const uint32_t *planes = reinterpret_cast<const uint32_t *>(rec);
                const int gid = t & 7, th = t >> 3;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const size_t word = (size_t)((4 * gid + (r & 3)) * 2 + th) * NW + (r >> 2);
                    const int c = (int)((planes[word] >> lane) & 1u) | (int)(((planes[PW + word] >> lane) & 1u) << 1) |
                                  (int)(((planes[2 * PW + word] >> lane) & 1u) << 2);
                    val[jj][r] = s_cent[c] * inv_sd;
                    s_b[t][dims[r]] = ((planes[3 * PW + word] >> lane) & 1u) ? 1.f : -1.f;
                }
                const __half2 ng = *reinterpret_cast<const __half2 *>(rec + 8 * D + 4 * t);
                nrm[jj] = __low2float(ng);
                gam[jj] = __high2float(ng);
            } else {
                constexpr int NWV = D / 64, NM = D / 128;
                const int tigv = (t & 7) >> 1, jb = (t >> 3) + 2 * (t & 1), beta = lane >> 3;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int tau = 4 * r + beta;
                    const int mhi = tau % NM, rh = (tau / NM) & 1, gid = tau / (2 * NM);
                    const size_t byte = ((size_t)(4 * gid + tigv) * NWV + 2 * mhi + rh) * 4 + jb;
                    const int c = ((rec[byte] >> (lane & 7)) & 1) | (((rec[2 * D + byte] >> (lane & 7)) & 1) << 1) |
                                  (((rec[4 * D + byte] >> (lane & 7)) & 1) << 2);
                    val[jj][r] = s_cent[c] * inv_sd;
                }
                nrm[jj] = __half2float(*reinterpret_cast<const __half *>(rec + 6 * D + 2 * t));
                gam[jj] = 0.f;
            }
        }
        // ---- 2. K: p = S^T b for the 16 slots (thread k computes p_k), into s_b
        if (is_k) {
            constexpr int KPT = D / NT;
            float acc[KPT][kDqTile];
#pragma unroll
            for (int k = 0; k < KPT; ++k)
#pragma unroll
                for (int t = 0; t < kDqTile; ++t) acc[k][t] = 0.f;
            if (SM::kResident) {
                cp_async_wait_all();
                __syncthreads();
                project_rows<D, kDqTile, NT>(sS, 0, D, s_b, acc);
            } else {
                __syncthreads();
                project_streamed<D, kDqTile, NT>(gS, sS, s_b, acc);
            }
            __syncthreads();   // every thread is done reading the signs
#pragma unroll
            for (int k = 0; k < KPT; ++k)
#pragma unroll
                for (int t = 0; t < kDqTile; ++t) s_b[t][threadIdx.x + NT * k] = acc[k][t];
            __syncthreads();
        }
        // ---- 3. y, inverse rotation, norm, store
#pragma unroll
        for (int jj = 0; jj < PER_WARP; ++jj) {
            const int t = warp + kDqWarps * jj;
            float v[R];
#pragma unroll
            for (int r = 0; r < R; ++r) v[r] = is_k ? fmaf(qjl * gam[jj], s_b[t][dims[r]], val[jj][r]) : val[jj][r];
            fwht_warp<R>(v, lane);
            const float sc = nrm[jj] * inv_sd;
            TO *orow = out + (((size_t)j * kBlock + t) * n_heads + h) * D;
#pragma unroll
            for (int r = 0; r < R; ++r) orow[dims[r]] = from_f32<TO>(good ? v[r] * sc * __ldg(Dsign + dims[r]) : 0.f);
        }
        if (is_k) __syncthreads();   // s_b is rewritten by the next tile
    }
}

template <int D, typename TO>
cudaError_t dq_launch(const void *params, const void *pool, int64_t num_blocks, int n_heads, const int32_t *ids,
                      int n_ids, bool is_k, void *out, int32_t *status, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const size_t smem = DqSmem<D>::kBytes;
    auto kern = dequant_kernel<D, TO>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DqSmem<D>::kBytes);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)n_ids * n_heads;
    const int64_t grid = units < (int64_t)sms * 8 ? units : (int64_t)sms * 8;
    kern<<<(unsigned)grid, kDqWarps * 32, smem, st>>>((const uint8_t *)params, (const uint8_t *)pool, num_blocks,
                                                      n_heads, ids, n_ids, is_k ? 1 : 0, (TO *)out, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dequant(bool is_k, int d, int out_dtype, const void *params, const void *pool, int64_t num_blocks,
                           int n_heads, const int32_t *block_ids, int n_ids, void *out, int32_t *status,
                           cudaStream_t st) {
    if (d == 128)
        return out_dtype == TQ_DTYPE_BF16
                   ? dq_launch<128, __nv_bfloat16>(params, pool, num_blocks, n_heads, block_ids, n_ids, is_k, out,
                                                   status, st)
                   : dq_launch<128, float>(params, pool, num_blocks, n_heads, block_ids, n_ids, is_k, out, status, st);
    return out_dtype == TQ_DTYPE_BF16
               ? dq_launch<256, __nv_bfloat16>(params, pool, num_blocks, n_heads, block_ids, n_ids, is_k, out, status,
                                               st)
               : dq_launch<256, float>(params, pool, num_blocks, n_heads, block_ids, n_ids, is_k, out, status, st);
}

}  // namespace tq
