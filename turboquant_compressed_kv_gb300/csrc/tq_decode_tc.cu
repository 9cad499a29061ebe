// tq_decode_tc.cu -- decode attention at head_dim 128 on the tcgen05 tensor cores.
//
// Computes what the split-K pass of tq_decode.cu computes (rotated-domain scores from the
// packed cells, QJL signs and fp16 norms; online softmax; value sums; one inverse rotation
// per head; stream-K work split with partial merges), formulated for tcgen05.mma:
//
//  * Operands from bit planes.  A plane word holds, in each of its 4 bytes, one bit per
//    bit position j = 0..7.  With mask 0x01010101 << j and an e4m3 base byte b_j, one LOP3
//    (w & mask) ^ (b_j * 0x01010101) yields four e4m3 values, each alpha_j (bit clear) or
//    alpha_j + delta_j (bit set); the table below keeps |delta_j| in [0.5, 2].
//  * K side: D_K[token, column] = sum_k A_K[token, k] B_K[k, column].  A_K rows are tokens
//    (written to tensor memory by the thread that owns the token), k runs over the 4
//    level masks (Walsh decomposition of the 8 Lloyd-Max levels, as in tq_decode.cu) and
//    the QJL sign mask, 128 dimensions each.  B_K holds the query side, pre-divided by
//    delta_j and pre-scaled by the level mask's Walsh coefficient, as a sum of e4m3
//    pieces with per-column power-of-two scales (5 pieces for <qbar, c>, 4 for <u, s>).
//  * V side: D_V[coordinate, (mask, head, piece)] = sum_token A_V[coordinate, token]
//    B_V[token, (head, piece)].  A_V rows are coordinates (written by the thread that owns
//    the coordinate); B_V holds the softmax weights as 3 e4m3 pieces (scales 1, 1/16,
//    1/256) with a per-head power-of-two scale 2^-E.
//  * The value accumulator stays in tensor memory across chunks.  A head's reference
//    maximum (and E) changes only when a chunk's maximum exceeds it by more than kTau (or
//    its weights would overflow the e4m3 range); then the accumulator is rescaled.
//
// One persistent CTA per SM, 288 threads:
//   warps 0-3  token rows: expand K, issue the K-side MMAs, scores, softmax, weight pieces;
//   warps 4-7  coordinate rows: expand V, issue the V-side MMAs, own the value accumulator;
//   warp 8     stages the K and V records of each 128-token chunk with bulk copies into a
//              ring of kStages buffers (mbarrier full/empty handshake).
#include "tq_internal.cuh"
#include "tq_tc.cuh"

#include <cuda_fp8.h>

namespace tq {
namespace tcd {

constexpr int D = 128;
constexpr int kCH = 128;                  // tokens per chunk (the MMA's M on the K side)
constexpr int kBPC = kCH / kBlock;        // 8 blocks per chunk
constexpr int kKRec = 8 * D + 64, kVRec = 6 * D + 32;
constexpr int kStageBytes = kBPC * (kKRec + kVRec);
constexpr int kStages = 6;
constexpr int kNP = 5, kNQ = 4, kNPV = 3;
constexpr float kTau = 5.0f;              // lazy-maximum slack (natural log units)
constexpr int kThreads = 288;
constexpr uint32_t kColAK = 0, kColAV = 160, kColDK = 288, kColDV = 384, kTmemCols = 512;

// e4m3 operand values of bit position j (see the header comment)
__host__ __device__ constexpr uint32_t e4_base(int j) {
    return j == 0 ? 0x48u : j == 1 ? 0x40u : j == 2 ? 0x38u : j == 3 ? 0x30u
         : j == 4 ? 0x28u : j == 5 ? 0x18u : j == 6 ? 0x00u : 0x38u;
}
__host__ __device__ constexpr float e4_alpha(int j) {
    return j == 0 ? 4.f : j == 1 ? 2.f : j == 2 ? 1.f : j == 3 ? 0.5f : j == 4 ? 0.25f : j == 5 ? 0.0625f
         : j == 6 ? 0.f : 1.f;
}
__host__ __device__ constexpr float e4_delta(int j) {
    return j <= 3 ? 0.5f : j == 4 ? 0.75f : j == 5 ? 0.9375f : j == 6 ? 2.f : -2.f;
}

template <int G>
struct Cfg {
    static constexpr int NC = 16 * ((G * kNP + 15) / 16);    // K-side columns, <qbar, c> pieces
    static constexpr int NQ = 16 * ((G * kNQ + 15) / 16);    // K-side columns, <u, s> pieces
    static constexpr int NV = 16 * ((G * kNPV + 15) / 16);   // V-side columns per level mask
    static constexpr int codeBytes = NC * 512, qjlBytes = NQ * 128;
    static constexpr int floatOff = codeBytes + qjlBytes;   // scales[NC], scales[NQ], cc[8], cq[8]
    static constexpr int packBytes = ((floatOff + 4 * (NC + NQ + 16)) + 255) & ~255;
    static constexpr int bvBytes = NV * kCH;
    static_assert(kColDK + NC + NQ <= kColDV && kColDV + 4 * NV <= kTmemCols, "tensor memory budget");
};
// bytes of the query pack of one (sequence, kv head), and a bound per query head
__host__ __device__ constexpr int pack_bytes(int G) {
    return G == 1 ? Cfg<1>::packBytes : G == 2 ? Cfg<2>::packBytes : G == 3 ? Cfg<3>::packBytes
         : G == 4 ? Cfg<4>::packBytes : G == 5 ? Cfg<5>::packBytes : G == 6 ? Cfg<6>::packBytes
         : G == 7 ? Cfg<7>::packBytes : Cfg<8>::packBytes;
}
constexpr int kPackPerHead = Cfg<1>::packBytes;   // pack_bytes(G) <= G * kPackPerHead for G = 1..8

// byte offset of element (row n, k) in a no-swizzle K-major operand with N rows
__host__ __device__ constexpr int op_off(int n, int k, int N) {
    return ((k >> 4) * (N >> 3) + (n >> 3)) * 128 + (n & 7) * 16 + (k & 15);
}
// K-side: dimension of K index k within one mask (column c = 8 tig + j, byte b)
__host__ __device__ constexpr int kdim_of(int k) {
    return 16 * ((k >> 2) & 7) + 8 * (k & 1) + 2 * (k >> 5) + ((k >> 1) & 1);
}

__device__ __forceinline__ uint8_t to_e4(float x) {
    return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float from_e4(uint8_t b) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3)));
}

// ---------------------------------------------------------------- query prep (operand packs)
// One warp per (sequence, query head) row, 4 rows per CTA: qbar = Pi q (FWHT), u = S qbar
// (S^T staged in shared memory), then the row's columns of the K-side B operands as e4m3
// pieces, their scales and offset constants.  CTA 0 also lays out the pass's work.
constexpr int kQRows = 4;

template <int G, typename T>
__global__ void __launch_bounds__(128)
qprep_tc_kernel(const uint8_t *__restrict__ params, const T *__restrict__ q, int batch, int hq, int hkv,
                const int32_t *__restrict__ ctx_lens, int max_ctx, int P, uint8_t *__restrict__ packs,
                unsigned int *__restrict__ counters, int64_t *__restrict__ cpre, int32_t *__restrict__ cta_b) {
    using C = Cfg<G>;
    constexpr int R = D / 32;
    extern __shared__ __align__(16) uint8_t qsm[];
    float (*qs)[D] = reinterpret_cast<float (*)[D]>(qsm);
    float (*us)[D] = reinterpret_cast<float (*)[D]>(qsm + kQRows * D * 4);
    float *sbuf = reinterpret_cast<float *>(qsm + 2 * kQRows * D * 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrows = batch * hq, row = blockIdx.x * kQRows + warp;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const float *ST = reinterpret_cast<const float *>(params + params_off_ST(D));
    const float inv_sd = rsqrtf((float)D);
    {
        float v[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            v[r] = (row < nrows) ? to_f32<T>(q[(size_t)row * D + 32 * r + lane]) * __ldg(Dsign + 32 * r + lane) : 0.f;
        fwht_warp<R>(v, lane);
#pragma unroll
        for (int r = 0; r < R; ++r) qs[warp][32 * r + lane] = v[r] * inv_sd;
    }
    {
        float acc[1][kQRows];
#pragma unroll
        for (int rr = 0; rr < kQRows; ++rr) acc[0][rr] = 0.f;
        project_streamed<D, kQRows, 128, 128>(ST, sbuf, qs, acc);     // u = S qbar
#pragma unroll
        for (int rr = 0; rr < kQRows; ++rr) us[rr][threadIdx.x] = acc[0][rr];
    }
    __syncthreads();
    if (row < nrows) {
        const int b = row / hq, h = row % hq, kvh = h / G, hg = h % G;
        if (hg == 0 && lane == 0) counters[b * hkv + kvh] = 0u;
        uint8_t *pack = packs + ((size_t)b * hkv + kvh) * C::packBytes;
        uint8_t *img_c = pack, *img_q = pack + C::codeBytes;
        float *scl_c = reinterpret_cast<float *>(pack + C::floatOff), *scl_q = scl_c + C::NC;
        float *cst = scl_q + C::NQ;                        // cc[8], cq[8]
        const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
        float A[4];
        walsh4(ph->centroid, A);
        // <qbar, c> operand: K index k = 128 m + kk, value A_m * 2 qbar[dim(kk)] / delta_j
        {
            float r[16], bh[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int k = lane + 32 * i, kk = k & 127, j = (kk >> 2) & 7;
                r[i] = A[k >> 7] * 2.f * qs[warp][kdim_of(kk)] / e4_delta(j);
                bh[i] = 0.f;
            }
#pragma unroll 1
            for (int p = 0; p < kNP; ++p) {
                float e = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) e = fmaxf(e, fabsf(r[i]));
                e = warp_max(e);
                int ex = 0;
                if (e > 0.f) frexpf(e, &ex);
                const int sig = (e > 0.f) ? 8 - ex : 0;
                const int n = hg * kNP + p;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int k = lane + 32 * i;
                    const uint8_t by = to_e4(ldexpf(r[i], sig));
                    const float dec = ldexpf(from_e4(by), -sig);
                    r[i] -= dec;
                    bh[i] += dec;
                    img_c[op_off(n, k, C::NC)] = by;
                }
                if (lane == 0) scl_c[n] = ldexpf(1.f, -sig);
            }
            float cs = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int j = (((lane + 32 * i) & 127) >> 2) & 7;
                cs = fmaf(bh[i], e4_alpha(j) + 0.5f * e4_delta(j), cs);
            }
            cs = warp_sum(cs);
            if (lane == 0) cst[hg] = cs;
        }
        // <u, s> operand: K index k (0..127), value 2 u[dim(k)] / delta_j
        {
            float r[4], bh[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int k = lane + 32 * i, j = (k >> 2) & 7;
                r[i] = 2.f * us[warp][kdim_of(k)] / e4_delta(j);
                bh[i] = 0.f;
            }
#pragma unroll 1
            for (int p = 0; p < kNQ; ++p) {
                float e = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) e = fmaxf(e, fabsf(r[i]));
                e = warp_max(e);
                int ex = 0;
                if (e > 0.f) frexpf(e, &ex);
                const int sig = (e > 0.f) ? 8 - ex : 0;
                const int n = hg * kNQ + p;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int k = lane + 32 * i;
                    const uint8_t by = to_e4(ldexpf(r[i], sig));
                    const float dec = ldexpf(from_e4(by), -sig);
                    r[i] -= dec;
                    bh[i] += dec;
                    img_q[op_off(n, k, C::NQ)] = by;
                }
                if (lane == 0) scl_q[n] = ldexpf(1.f, -sig);
            }
            float cs = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = ((lane + 32 * i) >> 2) & 7;
                cs = fmaf(bh[i], e4_alpha(j) + 0.5f * e4_delta(j), cs);
            }
            cs = warp_sum(cs);
            if (lane == 0) cst[8 + hg] = cs;
        }
        // columns beyond the group's heads are zero (written by the group's first head)
        if (hg == 0) {
            for (int n = G * kNP; n < C::NC; ++n) {
                for (int k = lane; k < 512; k += 32) img_c[op_off(n, k, C::NC)] = 0;
                if (lane == 0) scl_c[n] = 0.f;
            }
            for (int n = G * kNQ; n < C::NQ; ++n) {
                for (int k = lane; k < 128; k += 32) img_q[op_off(n, k, C::NQ)] = 0;
                if (lane == 0) scl_q[n] = 0.f;
            }
        }
    }
    if (blockIdx.x == 0) build_schedule(ctx_lens, batch, hkv, max_ctx, kCH, P, cpre, cta_b);
}

// ---------------------------------------------------------------- the pass

// out[row] = Pi^T (v / l), v spread over a warp as v[r] at lane
__device__ __forceinline__ void finish_row128(float (&v)[4], float l, const uint8_t *params, float *out_row, int lane) {
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] *= inv;
    fwht_warp<4>(v, lane);
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const float inv_sd = rsqrtf((float)D);
#pragma unroll
    for (int r = 0; r < 4; ++r) out_row[32 * r + lane] = v[r] * inv_sd * __ldg(Dsign + 32 * r + lane);
}

template <int G>
struct Smem {
    using C = Cfg<G>;
    static constexpr int oStages = 0;
    static constexpr int oBK = oStages + kStages * kStageBytes;        // code image, qjl image, floats
    static constexpr int oBV = oBK + C::packBytes;                      // 2 weight operands
    static constexpr int oAcc = oBV + 2 * C::bvBytes;                   // [G][D] floats (epilogue)
    static constexpr int used = oAcc + G * D * 4;
    static constexpr int bytes = used > 120 * 1024 ? used : 120 * 1024;   // one CTA per SM
};

struct Shared {                       // static shared state
    uint64_t full[kStages], empty[kStages], mma_k, mma_v;
    uint32_t tmem;
    int ok[kStages][kBPC];
    float cm[4][8];                   // per K warp: chunk maxima per head
    float nvm[4];                     // per K warp: maximum value norm
    float pl[4][8];                   // per K warp: sum of p per head
    float pt[4][8][kNPV];             // per K warp: sum of raw weight pieces per head
    float fV[2][8];                   // value-accumulator rescale factor per head (by chunk parity)
    int rescale[2];
    float runL[8], runT[8][kNPV], runM[8];
    int runE[8];
    bool last;
};

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const uint8_t *__restrict__ params, const uint8_t *__restrict__ packs, int batch, int hq, int hkv,
                 const uint8_t *__restrict__ k_pool, const uint8_t *__restrict__ v_pool, int64_t num_blocks,
                 const int32_t *__restrict__ block_table, int max_blocks, const int32_t *__restrict__ ctx_lens,
                 int max_ctx, const int64_t *__restrict__ cpre, const int32_t *__restrict__ cta_b,
                 float *__restrict__ part, unsigned int *__restrict__ counters, float *__restrict__ out,
                 int32_t *status) {
    using C = Cfg<G>;
    using SM = Smem<G>;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ Shared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;

    for (int b = cta; b < batch; b += gridDim.x)
        if (clamp_len(ctx_lens[b], max_ctx) == 0)
            for (int i = tid; i < hq * D; i += kThreads) out[(size_t)b * hq * D + i] = 0.f;

    const int64_t W = cpre[batch];
    const int P = (int)(W < (int64_t)gridDim.x ? W : (int64_t)gridDim.x);
    if (cta >= P) return;
    const int64_t g0 = sk_begin(cta, P, W), g1 = sk_begin(cta + 1, P, W);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&sh.full[s], 1);
            tc::mbar_init(&sh.empty[s], 256);
        }
        tc::mbar_init(&sh.mma_k, 1);
        tc::mbar_init(&sh.mma_v, 1);
    }
    if (warp == 0) tc::tmem_alloc(&sh.tmem, kTmemCols);
    // weight operands start zero (columns of heads >= G are never written)
    for (int i = tid; i < 2 * C::bvBytes / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + SM::oBV)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sh.tmem;
    bool timed_out = false;

    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    float A[4];
    walsh4(ph->centroid, A);
    const float inv_sd = rsqrtf((float)D);

    if (warp == 8) {
        // ---------------- producer: stage the records of every chunk of this CTA's range
        int b = cta_b[cta];
        int64_t ub = cpre[b];
        int nchb = (int)((cpre[b + 1] - ub) / hkv);
        int kh = (int)((g0 - ub) / nchb);
        int64_t g = g0;
        int i = 0;                                // chunk counter of this CTA
#pragma unroll 1
        while (true) {
            const int64_t us = ub + (int64_t)kh * nchb, ue = us + nchb;
            const int64_t se = (g1 < ue) ? g1 : ue;
            const int L = clamp_len(ctx_lens[b], max_ctx);
            const int t1 = min(L, (int)(se - us) * kCH);
#pragma unroll 1
            for (int tc0 = (int)(g - us) * kCH; tc0 < t1; tc0 += kCH, ++i) {
                const int s = i % kStages, k = i / kStages;
                if (k > 0 && !tc::mbar_wait(&sh.empty[s], (k - 1) & 1)) timed_out = true;
                int64_t p = -1;
                if (lane < kBPC) {
                    const bool inrange = tc0 + kBlock * lane < t1;
                    const int lb = tc0 / kBlock + lane;
                    if (inrange && lb < max_blocks) {
                        const int64_t pb = block_table[(size_t)b * max_blocks + lb];
                        p = (pb >= 0 && pb < num_blocks) ? pb : -1;
                    }
                    if (inrange && p < 0) flag_status(status, TQ_STATUS_BAD_SLOT);
                    sh.ok[s][lane] = p >= 0;
                }
                unsigned int bytes = (p >= 0) ? (unsigned)(kKRec + kVRec) : 0u;
#pragma unroll
                for (int m = 16; m > 0; m >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, m);
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_expect_tx(&sh.full[s], bytes);
                __syncwarp();
                if (p >= 0) {
                    uint8_t *st = smem + SM::oStages + s * kStageBytes;
                    tc::bulk_g2s(st + lane * kKRec, k_pool + ((size_t)p * hkv + kh) * kKRec, kKRec, &sh.full[s]);
                    tc::bulk_g2s(st + kBPC * kKRec + lane * kVRec, v_pool + ((size_t)p * hkv + kh) * kVRec, kVRec,
                                 &sh.full[s]);
                }
            }
            g = se;
            if (g >= g1) break;
            if (++kh == hkv) {
                kh = 0;
                do {
                    ++b;
                    ub = cpre[b];
                    nchb = (int)((cpre[b + 1] - ub) / hkv);
                } while (nchb == 0);
            }
        }
    } else {
    // consumers: chunk walk of this CTA's range, one (sequence, kv head) segment at a time
    int b = cta_b[cta];
    int64_t ub = cpre[b];
    int nchb = (int)((cpre[b + 1] - ub) / hkv);
    int kh = (int)((g0 - ub) / nchb);
    int64_t g = g0;
    bool first_seg = true;
    int ci = 0;                                   // chunk counter of this CTA

#pragma unroll 1
    while (true) {
        const int64_t us = ub + (int64_t)kh * nchb, ue = us + nchb;
        const int64_t se = (g1 < ue) ? g1 : ue;
        const int L = clamp_len(ctx_lens[b], max_ctx);
        const int t0 = (int)(g - us) * kCH;
        const int t1 = min(L, (int)(se - us) * kCH);
        const int nchunks = (int)(se - g);

        if (warp < 4) {
            // ---------------- K group: thread t owns token row t of every chunk
            const int t = tid;
            const uint32_t lanebase = (uint32_t)(32 * warp) << 16;
            // the query operand of this (sequence, kv head)
            {
                const uint4 *src = reinterpret_cast<const uint4 *>(packs + ((size_t)b * hkv + kh) * C::packBytes);
                uint4 *dst = reinterpret_cast<uint4 *>(smem + SM::oBK);
                for (int i = t; i < C::packBytes / 16; i += 128) dst[i] = src[i];
                tc::fence_async_smem();
            }
            tc::named_sync(1, 128);
            const float *scl_c = reinterpret_cast<const float *>(smem + SM::oBK + C::floatOff);
            const float *scl_q = scl_c + C::NC;
            const float *cst = scl_q + C::NQ;
            float m_ref[G];
            int E[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                m_ref[h] = -INFINITY;
                E[h] = 0;
            }
            if (t < G) {
                sh.runL[t] = 0.f;
#pragma unroll
                for (int p = 0; p < kNPV; ++p) sh.runT[t][p] = 0.f;
            }
#pragma unroll 1
            for (int c = 0; c < nchunks; ++c) {
                const int i = ci + c, s = i % kStages;
                const int tc0 = t0 + c * kCH;
                if (!tc::mbar_wait(&sh.full[s], (i / kStages) & 1)) timed_out = true;
                const uint8_t *st = smem + SM::oStages + s * kStageBytes;
                const int kb = t >> 4, tt = t & 15;
                const uint32_t *rec = reinterpret_cast<const uint32_t *>(st + kb * kKRec);
                const bool ok = sh.ok[s][kb] != 0 && (tc0 + t < t1);
                uint32_t w[5][4];
#pragma unroll
                for (int pl = 0; pl < 4; ++pl)
#pragma unroll
                    for (int tg = 0; tg < 4; ++tg) w[pl == 3 ? 4 : pl][tg] = rec[pl * 64 + (4 * (tt & 7) + tg) * 2 + (tt >> 3)];
                const __half2 ng = *reinterpret_cast<const __half2 *>(st + kb * kKRec + 8 * D + 4 * tt);
                const float nrm = __low2float(ng), gam = __high2float(ng);
                // (records of blocks that were not copied hold stale bytes: use nothing of them)
                const float nv = ok ? __half2float(*reinterpret_cast<const __half *>(st + kBPC * kKRec + kb * kVRec + 6 * D + 2 * tt)) : 0.f;
                tc::mbar_arrive(&sh.empty[s]);
#pragma unroll
                for (int tg = 0; tg < 4; ++tg) w[3][tg] = w[0][tg] ^ w[1][tg] ^ w[2][tg];
                // expand the 5 masks into A_K (32 columns each)
#pragma unroll
                for (int m = 0; m < 5; ++m) {
                    uint32_t r[32];
#pragma unroll
                    for (int tg = 0; tg < 4; ++tg)
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            r[8 * tg + j] = lop_and_xor(w[m][tg], 0x01010101u << j, e4_base(j) * 0x01010101u);
                    tc::st32(tmem + lanebase + kColAK + 32 * m, r);
                }
                tc::wait_st();
                tc::fence_before_sync();
                tc::named_sync(1, 128);
                if (t == 0) {
                    tc::fence_after_sync();
                    const uint32_t sbk = tc::smem_u32(smem + SM::oBK);
#pragma unroll
                    for (int ks = 0; ks < 16; ++ks)
                        tc::mma_ts(tmem + kColDK, tmem + kColAK + 8 * ks,
                                   tc::smem_desc(sbk + ks * 2 * (C::NC / 8) * 128, (C::NC / 8) * 128, 128),
                                   tc::idesc_e4m3(128, C::NC), ks > 0);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ts(tmem + kColDK + C::NC, tmem + kColAK + 128 + 8 * ks,
                                   tc::smem_desc(sbk + C::codeBytes + ks * 2 * (C::NQ / 8) * 128, (C::NQ / 8) * 128, 128),
                                   tc::idesc_e4m3(128, C::NQ), ks > 0);
                    tc::mma_commit(&sh.mma_k);
                }
                if (!tc::mbar_wait(&sh.mma_k, i & 1)) timed_out = true;
                tc::fence_after_sync();
                // scores of token t for the G heads
                float sc[G];
                {
                    float dk[C::NC + C::NQ];
#pragma unroll
                    for (int c16 = 0; c16 < (C::NC + C::NQ) / 16; ++c16) {
                        float v16[16];
                        tc::ld16(tmem + lanebase + kColDK + 16 * c16, v16);
#pragma unroll
                        for (int x = 0; x < 16; ++x) dk[16 * c16 + x] = v16[x];
                    }
                    tc::wait_ld();
                    const float qjl = 1.2533141373155003f / (float)D;
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        float cd = -cst[h], qd = -cst[8 + h];
#pragma unroll
                        for (int p = 0; p < kNP; ++p) cd = fmaf(scl_c[h * kNP + p], dk[h * kNP + p], cd);
#pragma unroll
                        for (int p = 0; p < kNQ; ++p) qd = fmaf(scl_q[h * kNQ + p], dk[C::NC + h * kNQ + p], qd);
                        sc[h] = ok ? nrm * inv_sd * (cd * inv_sd + gam * qjl * qd) : -INFINITY;
                    }
                }
                // chunk maxima per head and of the value norms
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float mx = warp_max(sc[h]);
                    if (lane == 0) sh.cm[warp][h] = mx;
                }
                {
                    const float mx = warp_max(nv);
                    if (lane == 0) sh.nvm[warp] = mx;
                }
                tc::named_sync(1, 128);
                const float nvmax = fmaxf(fmaxf(sh.nvm[0], sh.nvm[1]), fmaxf(sh.nvm[2], sh.nvm[3]));
                int any_rescale = 0;
                float fV[G], fL[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float cmax = fmaxf(fmaxf(sh.cm[0][h], sh.cm[1][h]), fmaxf(sh.cm[2][h], sh.cm[3][h]));
                    const float m_old = m_ref[h];
                    const int E_old = E[h];
                    float m_new = m_old;
                    if (cmax > m_old + kTau || m_old == -INFINITY) m_new = cmax;
                    int E_new = E_old;
                    if (m_new != -INFINITY) {
                        const float bound = __expf(cmax - m_new) * nvmax * inv_sd;
                        if (bound > 0.f) {
                            int ex;
                            frexpf(bound * (1.f / 256.f), &ex);
                            E_new = (m_old == -INFINITY) ? ex : max(E_old, ex);
                        }
                    }
                    fL[h] = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
                    fV[h] = ldexpf(fL[h], E_old - E_new);
                    if (m_old != -INFINITY && (m_new != m_old || E_new != E_old)) any_rescale = 1;
                    m_ref[h] = m_new;
                    E[h] = E_new;
                }
                // weights of token t, as 3 e4m3 pieces, into the weight operand (token order kappa)
                uint8_t *bv = smem + SM::oBV + (i & 1) * C::bvBytes;
                const int kap = 16 * kb + 4 * ((tt & 7) >> 1) + (tt >> 3) + 2 * (tt & 1);
                float pT[G][kNPV], pp[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float pr = (sc[h] == -INFINITY) ? 0.f : __expf(sc[h] - m_ref[h]);
                    pp[h] = pr;
                    float wv = ldexpf(pr * nv * inv_sd, -E[h]);
#pragma unroll
                    for (int p = 0; p < kNPV; ++p) {
                        const uint8_t by = to_e4(ldexpf(wv, 4 * p));
                        const float dec = from_e4(by);
                        pT[h][p] = dec;
                        wv -= ldexpf(dec, -4 * p);
                        bv[op_off(h * kNPV + p, kap, C::NV)] = by;
                    }
                }
                tc::fence_async_smem();
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float ls = warp_sum(pp[h]);
                    if (lane == 0) sh.pl[warp][h] = ls;
#pragma unroll
                    for (int p = 0; p < kNPV; ++p) {
                        const float ts = warp_sum(pT[h][p]);
                        if (lane == 0) sh.pt[warp][h][p] = ts;
                    }
                }
                if (t == 0) {
#pragma unroll
                    for (int h = 0; h < G; ++h) sh.fV[i & 1][h] = fV[h];
                    sh.rescale[i & 1] = any_rescale;
                }
                // running sums of this segment (thread h keeps head h)
                if (t < G) {
                    float fl = 1.f, fv = 1.f;
#pragma unroll
                    for (int h = 0; h < G; ++h)
                        if (h == t) {
                            fl = fL[h];
                            fv = fV[h];
                        }
                    // partial sums of this chunk are published after the barrier below
                    sh.runL[t] *= fl;
#pragma unroll
                    for (int p = 0; p < kNPV; ++p) sh.runT[t][p] *= fv;
                }
                tc::named_sync(3, 256);        // weight operand, partial sums and rescale factors ready
                if (t < G) {
                    sh.runL[t] += sh.pl[0][t] + sh.pl[1][t] + sh.pl[2][t] + sh.pl[3][t];
#pragma unroll
                    for (int p = 0; p < kNPV; ++p)
                        sh.runT[t][p] += sh.pt[0][t][p] + sh.pt[1][t][p] + sh.pt[2][t][p] + sh.pt[3][t][p];
                }
            }
            if (t < G) {
#pragma unroll
                for (int h = 0; h < G; ++h)
                    if (h == t) {
                        sh.runM[t] = m_ref[h];
                        sh.runE[t] = E[h];
                    }
            }
        } else {
            // ---------------- V group: thread L owns coordinate row L of the value accumulator
            const int Lr = tid - 128, wv = Lr >> 5;
            const uint32_t lanebase = (uint32_t)(32 * wv) << 16;
            const int gid = 4 * (wv & 1) + (lane & 3), rh = (lane >> 2) & 1, mt = 4 * (wv >> 1) + (lane >> 3);
            const uint32_t vmask = 0x01010101u << mt, vbase = e4_base(mt) * 0x01010101u;
#pragma unroll 1
            for (int c = 0; c < nchunks; ++c) {
                const int i = ci + c, s = i % kStages;
                if (!tc::mbar_wait(&sh.full[s], (i / kStages) & 1)) timed_out = true;
                const uint8_t *st = smem + SM::oStages + s * kStageBytes + kBPC * kKRec;
                uint32_t x[3][kBPC][4];
#pragma unroll
                for (int kb = 0; kb < kBPC; ++kb) {
                    const uint32_t *rec = reinterpret_cast<const uint32_t *>(st + kb * kVRec);
#pragma unroll
                    for (int pl = 0; pl < 3; ++pl)
#pragma unroll
                        for (int tg = 0; tg < 4; ++tg) x[pl][kb][tg] = rec[pl * 64 + (4 * gid + tg) * 2 + rh];
                }
                tc::mbar_arrive(&sh.empty[s]);
                if (i > 0 && !tc::mbar_wait(&sh.mma_v, (i - 1) & 1)) timed_out = true;   // A_V is free
                tc::fence_after_sync();
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    uint32_t r[32];
#pragma unroll
                    for (int kb = 0; kb < kBPC; ++kb)
#pragma unroll
                        for (int tg = 0; tg < 4; ++tg) {
                            const uint32_t xw = (m < 3) ? x[m][kb][tg] : (x[0][kb][tg] ^ x[1][kb][tg] ^ x[2][kb][tg]);
                            r[4 * kb + tg] = lop_and_xor(xw, vmask, vbase);
                        }
                    tc::st32(tmem + lanebase + kColAV + 32 * m, r);
                }
                tc::wait_st();
                tc::fence_before_sync();
                tc::named_sync(3, 256);        // the weight operand of this chunk is ready
                tc::fence_after_sync();
                if (c > 0 && sh.rescale[i & 1]) {
                    // rescale the value accumulator (the previous chunk's MMAs are complete)
#pragma unroll
                    for (int c16 = 0; c16 < 4 * C::NV / 16; ++c16) {
                        float v16[16];
                        tc::ld16(tmem + lanebase + kColDV + 16 * c16, v16);
                        tc::wait_ld();
#pragma unroll
                        for (int x2 = 0; x2 < 16; ++x2) {
                            const int col = (16 * c16 + x2) % C::NV, h = col / kNPV;
                            v16[x2] *= (h < G) ? sh.fV[i & 1][h] : 0.f;
                        }
                        tc::st16(tmem + lanebase + kColDV + 16 * c16, v16);
                    }
                    tc::wait_st();
                    tc::fence_before_sync();
                    tc::named_sync(2, 128);
                    tc::fence_after_sync();
                }
                if (Lr == 0) {
                    const uint32_t sbv = tc::smem_u32(smem + SM::oBV + (i & 1) * C::bvBytes);
#pragma unroll
                    for (int m = 0; m < 4; ++m)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc::mma_ts(tmem + kColDV + m * C::NV, tmem + kColAV + 32 * m + 8 * ks,
                                       tc::smem_desc(sbv + ks * 2 * (C::NV / 8) * 128, (C::NV / 8) * 128, 128),
                                       tc::idesc_e4m3(128, C::NV), c > 0 || ks > 0);
                    tc::mma_commit(&sh.mma_v);
                }
            }
            // the segment's value sums: wait for its last MMAs
            if (!tc::mbar_wait(&sh.mma_v, (ci + nchunks - 1) & 1)) timed_out = true;
            tc::fence_after_sync();
        }

        // ---------------- segment epilogue (all 288 threads)
        tc::named_sync(4, 256);               // running sums final; value MMAs complete
        float *sAcc = reinterpret_cast<float *>(smem + SM::oAcc);
        if (warp >= 4) {
            const int Lr = tid - 128, wv = Lr >> 5;
            const uint32_t lanebase = (uint32_t)(32 * wv) << 16;
            const int gid = 4 * (wv & 1) + (lane & 3), rh = (lane >> 2) & 1, mt = 4 * (wv >> 1) + (lane >> 3);
            const int coord = 16 * mt + gid + 8 * rh;
            const float al = e4_alpha(mt), inv_de = 2.f / e4_delta(mt);
            float v[G];
#pragma unroll
            for (int h = 0; h < G; ++h) v[h] = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
                for (int c16 = 0; c16 < C::NV / 16; ++c16) {
                    float d16[16];
                    tc::ld16(tmem + lanebase + kColDV + m * C::NV + 16 * c16, d16);
                    tc::wait_ld();
#pragma unroll
                    for (int x2 = 0; x2 < 16; ++x2) {
                        const int col = 16 * c16 + x2, h = col / kNPV, p = col % kNPV;
                        if (h < G) {
                            const float T = sh.runT[h][p];
                            v[h] += A[m] * ldexpf((d16[x2] - al * T) * inv_de - T, -4 * p);
                        }
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) sAcc[h * D + coord] = ldexpf(v[h], sh.runE[h]);
        }
        tc::named_sync(4, 256);
        const int lo = sk_cta_of(us, P, W), hi = sk_cta_of(ue - 1, P, W);
        const size_t row0 = (size_t)b * hq + (size_t)kh * G;
        if (lo == hi) {
            for (int h = warp; h < G; h += 8) {
                float v[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) v[r] = sAcc[h * D + 32 * r + lane];
                finish_row128(v, sh.runL[h], params, out + (row0 + h) * D, lane);
            }
        } else {
            const int slot = first_seg ? 0 : 1;
            for (int h = 0; h < G; ++h) {
                float *dst = part + (((size_t)cta * 2 + slot) * G + h) * kPartStride(D);
                for (int i = tid; i < D; i += 256) dst[4 + i] = sAcc[h * D + i];
                if (tid == 0) {
                    dst[0] = sh.runM[h];
                    dst[1] = sh.runL[h];
                }
            }
            __threadfence();
            tc::named_sync(4, 256);
            if (tid == 0) {
                const unsigned int nseg = (unsigned int)(hi - lo + 1);
                const unsigned int done = atomicAdd(&counters[b * hkv + kh], 1u) + 1u;
                sh.last = (done == nseg);
                if (sh.last) counters[b * hkv + kh] = 0u;
            }
            tc::named_sync(4, 256);
            if (sh.last) {
                __threadfence();
                const int slot_lo = (sk_begin(lo, P, W) >= us) ? 0 : 1;
                for (int h = warp; h < G; h += 8) {
                    float M = -INFINITY;
                    for (int c2 = lo; c2 <= hi; ++c2) {
                        const int sl = (c2 == lo) ? slot_lo : 0;
                        M = fmaxf(M, __ldcg(part + (((size_t)c2 * 2 + sl) * G + h) * kPartStride(D)));
                    }
                    float v[4] = {0.f, 0.f, 0.f, 0.f};
                    float l = 0.f;
                    for (int c2 = lo; c2 <= hi; ++c2) {
                        const int sl = (c2 == lo) ? slot_lo : 0;
                        const float *ps = part + (((size_t)c2 * 2 + sl) * G + h) * kPartStride(D);
                        const float m = __ldcg(ps);
                        const float wgt = (m == -INFINITY) ? 0.f : __expf(m - M);
                        l = fmaf(__ldcg(ps + 1), wgt, l);
#pragma unroll
                        for (int r = 0; r < 4; ++r) v[r] = fmaf(__ldcg(ps + 4 + 32 * r + lane), wgt, v[r]);
                    }
                    finish_row128(v, l, params, out + (row0 + h) * D, lane);
                }
            }
        }
        tc::named_sync(4, 256);               // sAcc and the running sums are reused by the next segment

        ci += nchunks;
        g = se;
        if (g >= g1) break;
        first_seg = false;
        if (++kh == hkv) {
            kh = 0;
            do {
                ++b;
                ub = cpre[b];
                nchb = (int)((cpre[b + 1] - ub) / hkv);
            } while (nchb == 0);
        }
    }
    }
    if (timed_out) flag_status(status, TQ_STATUS_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- launchers

int pass_ctas() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms > kMaxSms ? kMaxSms : sms;
}

template <int G, typename T>
cudaError_t qprep_launch(const uint8_t *P, const void *q, int batch, int hq, int hkv, const int32_t *ctx_lens,
                         int max_ctx, int nctas, uint8_t *packs, unsigned int *counters, int64_t *cpre, int32_t *cta_b,
                         cudaStream_t st) {
    constexpr size_t smem = (size_t)2 * kQRows * D * 4 + (size_t)128 * D * 4;
    auto kern = qprep_tc_kernel<G, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(batch * hq + kQRows - 1) / kQRows, 128, smem, st>>>(P, (const T *)q, batch, hq, hkv, ctx_lens, max_ctx,
                                                               nctas, packs, counters, cpre, cta_b);
    return cudaGetLastError();
}

template <int G>
cudaError_t pass_launch(int nctas, cudaStream_t st, const uint8_t *P, int batch, int hq, int hkv, const uint8_t *kp,
                        const uint8_t *vp, int64_t nb, const int32_t *bt, int mb, const int32_t *ctx, int max_ctx,
                        const uint8_t *packs, const int64_t *cpre, const int32_t *cta_b, float *part,
                        unsigned int *counters, float *out, int32_t *status) {
    constexpr size_t smem = Smem<G>::bytes;
    auto kern = decode_tc_kernel<G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<nctas, kThreads, smem, st>>>(P, packs, batch, hq, hkv, kp, vp, nb, bt, mb, ctx, max_ctx, cpre, cta_b, part,
                                       counters, out, status);
    return cudaGetLastError();
}

}  // namespace tcd

#define TQ_TC_G(MACRO) \
    switch (G) {       \
        case 1: MACRO(1); \
        case 2: MACRO(2); \
        case 3: MACRO(3); \
        case 4: MACRO(4); \
        case 5: MACRO(5); \
        case 6: MACRO(6); \
        case 7: MACRO(7); \
        default: MACRO(8); \
    }

int tc_pass_ctas() { return tcd::pass_ctas(); }
size_t tc_pack_bytes_per_head() { return (size_t)tcd::kPackPerHead; }
size_t tc_pack_bytes(int G) { return (size_t)tcd::pack_bytes(G); }

cudaError_t launch_qprep_tc(int dtype, const void *params, const void *q, int batch, int hq, int hkv,
                            const int32_t *ctx_lens, int max_ctx, int nctas, uint8_t *packs, unsigned int *counters,
                            int64_t *cpre, int32_t *cta_b, cudaStream_t st) {
    const int G = hq / hkv;
    const uint8_t *P = (const uint8_t *)params;
#define TQ_QP(GG)                                                                                                   \
    return dtype == TQ_DTYPE_BF16                                                                                   \
               ? tcd::qprep_launch<GG, __nv_bfloat16>(P, q, batch, hq, hkv, ctx_lens, max_ctx, nctas, packs, counters, \
                                                       cpre, cta_b, st)                                              \
               : tcd::qprep_launch<GG, float>(P, q, batch, hq, hkv, ctx_lens, max_ctx, nctas, packs, counters, cpre,  \
                                              cta_b, st)
    TQ_TC_G(TQ_QP)
#undef TQ_QP
}

cudaError_t launch_pass_tc(int nctas, const void *params, int batch, int hq, int hkv, const void *k_pool,
                           const void *v_pool, int64_t num_blocks, const int32_t *block_table, int max_blocks,
                           const int32_t *ctx_lens, int max_ctx, const uint8_t *packs, const int64_t *cpre,
                           const int32_t *cta_b, float *part, unsigned int *counters, float *out, int32_t *status,
                           cudaStream_t st) {
    const int G = hq / hkv;
    const uint8_t *P = (const uint8_t *)params;
#define TQ_PS(GG)                                                                                                      \
    return tcd::pass_launch<GG>(nctas, st, P, batch, hq, hkv, (const uint8_t *)k_pool, (const uint8_t *)v_pool,       \
                                num_blocks, block_table, max_blocks, ctx_lens, max_ctx, packs, cpre, cta_b, part,     \
                                counters, out, status)
    TQ_TC_G(TQ_PS)
#undef TQ_PS
}
#undef TQ_TC_G

}  // namespace tq
