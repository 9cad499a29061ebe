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
// Tensor-core formulation (this library's design, not the pages'):
//  * The 8 Lloyd-Max levels are odd in the three cell bits b0,b1,b2, so with
//    sigma_p = 2 b_p - 1 every level is exactly
//      c[cell] = A0 sigma_0 + A1 sigma_1 + A2 sigma_2 + A3 sigma_0 sigma_1 sigma_2,
//    where sigma_0 sigma_1 sigma_2 = 2 (b0^b1^b2) - 1.  A dot product with the
//    levels is therefore four +-1 dot products, and the QJL term a fifth.
//  * A bit plane becomes f16 mma.sync (m16n8k16) operands with one LOP3 per
//    register: for bit position q in 8..15 of each half, (w & bit) ^ base_q is
//    the f16 value alpha_q (bit 0) or alpha_q + delta_q (bit 1), |delta_q| >=
//    1/4; bits at positions 0..7 are first moved up by a shift of the word.
//    The other operand is pre-divided by delta_q and a per-column constant
//    removes alpha_q, so the +-1 product is recovered exactly.
//  * The fp32 query side is carried as f16 hi + lo (relative error about
//    2^-22), the softmax weights as one f16 with a running power-of-two scale;
//    the tensor core accumulates in fp32.
//
// Two launches per call: (1) query prep (qbar, u, f16 operand fragments,
// offset constants); (2) the split-K pass: an online-softmax partial (m, l,
// acc[d]) per (seq, q head, split); the last split of each (seq, kv head) to
// finish merges the partials and applies one inverse rotation per head.
#include <cuda_fp8.h>

#include "tq_internal.cuh"

namespace tq {

constexpr int kMinSplit = 512;             // shortest context split (sizes the workspace)
constexpr int kMaxSplit = 8192;
__host__ __device__ constexpr int kPartStride(int d) { return d + 4; }   // m, l, pad, pad, acc[d]
// Per (sequence, kv head) query pack: f16x2 B-operand fragments
// [2 (qbar, u)][d/16 k-steps][2 n-tiles][32 lanes][2 words], then the offset
// constants [2][8 heads] as floats.
__host__ __device__ constexpr size_t kPackBytes(int d) { return 64 * (size_t)d + 256; }
__host__ __device__ constexpr int kPackFloatOff(int d) { return 16 * d; }   // in floats

// Workspace: query packs [B*Hkv] | split counters [B*Hkv] | partials [B*Hq][nsplit][d+4].
// Sized with Hq >= Hkv and the shortest split, so every layout below fits.
__host__ __device__ constexpr size_t kCounterBytes(int batch, int hq) {
    return ((size_t)batch * hq * 4 + 255) & ~(size_t)255;
}
size_t decode_workspace_bytes(int d, int batch, int hq, int max_ctx) {
    if (!valid_d(d) || batch <= 0 || hq <= 0 || max_ctx < 0) return 0;
    const size_t nsplit = (size_t)((max_ctx + kMinSplit - 1) / kMinSplit);
    const size_t pack = (size_t)batch * hq * kPackBytes(d);
    const size_t part = (size_t)batch * hq * (nsplit ? nsplit : 1) * kPartStride(d) * sizeof(float);
    return pack + kCounterBytes(batch, hq) + part;
}

namespace {

// ---------------------------------------------------------------- f16 operand helpers

// Operand bit position q (8..15 within each f16 half): mask, base, and the
// operand values alpha (bit clear) and alpha + delta (bit set).
__host__ __device__ constexpr uint32_t op_mask(int q) { return 0x00010001u << q; }
__host__ __device__ constexpr uint32_t op_base(int q) { return q == 14 ? 0u : 0x3C003C00u; }
__host__ __device__ constexpr float op_alpha(int q) { return q == 14 ? 0.f : 1.f; }
__host__ __device__ constexpr float op_delta(int q) {
    return q == 8 ? 0.25f : q == 9 ? 0.5f : q == 10 ? -0.5f : q == 11 ? -0.75f
         : q == 12 ? -0.9375f : q == 13 ? -0.99609375f : q == 14 ? 2.0f : -2.0f;
}
// (w & mask) ^ base as a single LOP3 (base held in a register by the caller)
__device__ __forceinline__ uint32_t lop_and_xor(uint32_t w, uint32_t mask, uint32_t base) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(w), "r"(mask), "r"(base));
    return d;
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// exponent e with x * 2^e in [128, 256) for x > 0
__device__ __forceinline__ int scale_exp(float x) {
    int ex;
    frexpf(x, &ex);
    return 8 - ex;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, m));
    return x;
}

// Walsh coefficients A0..A3 of the 8 levels (c[k] = sum_m A_m sigma_m(k)).
__device__ __forceinline__ void walsh4(const float *cen, float (&A)[4]) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float s0 = (k & 1) ? 1.f : -1.f, s1 = (k & 2) ? 1.f : -1.f, s2 = (k & 4) ? 1.f : -1.f;
        a0 += cen[k] * s0;
        a1 += cen[k] * s1;
        a2 += cen[k] * s2;
        a3 += cen[k] * s0 * s1 * s2;
    }
    A[0] = a0 * 0.125f;
    A[1] = a1 * 0.125f;
    A[2] = a2 * 0.125f;
    A[3] = a3 * 0.125f;
}

// ---------------------------------------------------------------- (1) query prep
// A CTA handles kQRows (sequence, query head) rows: each warp rotates its rows
// (qbar = Pi q), then thread k computes u_k = (S qbar)_k for every row from
// S^T (coalesced, each load shared by the rows), then each warp writes its
// rows' hi and lo columns (2*hg, 2*hg+1) of the K-side B operand for qbar
// (qu=0) and u (qu=1) into the pack of the row's (sequence, kv head), and the
// offset constants.
constexpr int kQRows = 8;

template <int D, int NTK, typename T>
__global__ void __launch_bounds__(128)
qprep_kernel(const uint8_t *__restrict__ params, const T *__restrict__ q, int batch, int hq, int hkv,
             uint8_t *__restrict__ packs, unsigned int *__restrict__ counters) {
    constexpr int R = D / 32, NKS = D / 16, KPT = D / 128;
    extern __shared__ __align__(16) uint8_t qsm[];
    float (*qs)[D] = reinterpret_cast<float (*)[D]>(qsm);                       // [kQRows][D] qbar
    float (*us)[D] = reinterpret_cast<float (*)[D]>(qsm + kQRows * D * 4);      // [kQRows][D] u
    float *sbuf = reinterpret_cast<float *>(qsm + 2 * kQRows * D * 4);         // S^T chunks
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrows = batch * hq, row0 = blockIdx.x * kQRows;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const float *ST = reinterpret_cast<const float *>(params + params_off_ST(D));
    const float inv_sd = rsqrtf((float)D);
#pragma unroll
    for (int j = 0; j < kQRows / 4; ++j) {
        const int rr = warp + 4 * j, row = row0 + rr;
        float v[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            v[r] = (row < nrows) ? to_f32<T>(q[(size_t)row * D + 32 * r + lane]) * __ldg(Dsign + 32 * r + lane) : 0.f;
        fwht_warp<R>(v, lane);
#pragma unroll
        for (int r = 0; r < R; ++r) qs[rr][32 * r + lane] = v[r] * inv_sd;   // qbar = H D q / sqrt d
    }
    {
        float acc[KPT][kQRows];
#pragma unroll
        for (int u = 0; u < KPT; ++u)
#pragma unroll
            for (int rr = 0; rr < kQRows; ++rr) acc[u][rr] = 0.f;
        project_streamed<D, kQRows, 128>(ST, sbuf, qs, acc);     // u = S qbar
#pragma unroll
        for (int u = 0; u < KPT; ++u)
#pragma unroll
            for (int rr = 0; rr < kQRows; ++rr) us[rr][threadIdx.x + 128 * u] = acc[u][rr];
    }
    __syncthreads();
#pragma unroll 1
    for (int j = 0; j < kQRows / 4; ++j) {
        const int rr = warp + 4 * j, row = row0 + rr;
        if (row >= nrows) break;
        const int b = row / hq, h = row % hq, G = hq / hkv, kvh = h / G, hg = h % G;
        if (hg == 0 && lane == 0) counters[b * hkv + kvh] = 0u;   // split-K completion counter
        float v[R], u[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            v[r] = qs[rr][32 * r + lane];
            u[r] = us[rr][32 * r + lane];
        }
        uint8_t *pack = packs + ((size_t)b * hkv + kvh) * kPackBytes(D);
        uint16_t *ph = reinterpret_cast<uint16_t *>(pack);
        float *pf = reinterpret_cast<float *>(pack) + kPackFloatOff(D);
#pragma unroll
        for (int qu = 0; qu < 2; ++qu) {
            double cs = 0.0;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int dim = 32 * r + lane, s = dim >> 4, k = dim & 15, qd = 8 + (s & 7);
                const float beta = 2.f * (qu == 0 ? v[r] : u[r]) / op_delta(qd);
                const __half hi = __float2half_rn(beta);
                const __half lo = __float2half_rn(beta - __half2float(hi));
                cs += ((double)__half2float(hi) + (double)__half2float(lo)) * (double)(op_alpha(qd) + 0.5f * op_delta(qd));
                const int reg = k >> 3, tig = (k & 7) >> 1, e = k & 1;
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int col = 2 * hg + x, nt = col >> 3, gid = col & 7;
                    const size_t word = ((size_t)(qu * NKS + s) * NTK + nt) * 64 + (4 * gid + tig) * 2 + reg;
                    ph[word * 2 + e] = __half_as_ushort(x == 0 ? hi : lo);
                }
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, m);
            if (lane == 0) pf[qu * 8 + hg] = (float)cs;
        }
        // columns beyond the group's 2*G are zero (written by the group's first head)
        if (hg == 0) {
            uint32_t *pw = reinterpret_cast<uint32_t *>(pack);
            for (int col = 2 * G; col < 8 * NTK; ++col) {
                const int nt = col >> 3, gid = col & 7;
                for (int i = lane; i < 2 * NKS * 8; i += 32) {
                    const int qu = i / (NKS * 8), s = (i / 8) % NKS, k = i % 8;
                    pw[((size_t)(qu * NKS + s) * NTK + nt) * 64 + (4 * gid + (k >> 1)) * 2 + (k & 1)] = 0u;
                }
            }
        }
    }
}

// ---------------------------------------------------------------- (2) split-K pass
// grid (splits, Hkv, B), NWARP warps (4 for G <= 4, else 8).  The records of
// a chunk of 32*NWARP tokens (2 blocks per warp) are staged in shared memory
// by cp.async one chunk ahead.  Per chunk: warp w scores blocks 2w, 2w+1
// against all G heads (K side); the warps run the online softmax (warp w owns
// heads w, w+NWARP); warp w accumulates values for its D/NWARP coordinates
// over the whole chunk (V side).

// physical block of logical block lb, or -1 (past the table or outside the pool)
__device__ __forceinline__ int64_t block_of(const int32_t *__restrict__ bt, int b, int max_blocks, int lb,
                                            int64_t num_blocks) {
    if (lb >= max_blocks) return -1;
    const int64_t p = bt[(size_t)b * max_blocks + lb];
    return (p >= 0 && p < num_blocks) ? p : -1;
}


#ifndef TQ_SPLITK_BPW
#define TQ_SPLITK_BPW 2          // blocks scored per warp per chunk
#endif
#ifndef TQ_SPLITK_MINBLOCKS
#define TQ_SPLITK_MINBLOCKS 4    // resident CTAs per SM the register budget is sized for (4-warp CTAs)
#endif

template <int D, int NWARP>
struct SplitCfg {
    static constexpr int NT = NWARP * 32;
    static constexpr int BPW = TQ_SPLITK_BPW;        // blocks scored per warp per chunk
    static constexpr int BPC = NWARP * BPW;          // blocks per chunk
    static constexpr int CH = kBlock * BPC;          // tokens per chunk
    static constexpr int KREC = (int)k_record(D), VREC = (int)v_record(D);
    static constexpr size_t kBytes = 2 * (size_t)BPC * KREC;   // double-buffered K records
    static constexpr size_t vBytes = 2 * (size_t)BPC * VREC;
};

template <int D, int G, int NWARP>
constexpr size_t split_smem_bytes() {
    using C = SplitCfg<D, NWARP>;
    return C::kBytes + C::vBytes + (size_t)8 * (C::CH + 8) * 2 + (size_t)C::CH * G * 4;
}

template <int D, int G, int NWARP>
__global__ void __launch_bounds__(NWARP * 32, (NWARP == 4 ? TQ_SPLITK_MINBLOCKS : 1))
decode_mma_kernel(const uint8_t *__restrict__ params, const uint8_t *__restrict__ packs, int hq, int hkv,
                  const uint8_t *__restrict__ k_pool, const uint8_t *__restrict__ v_pool, int64_t num_blocks,
                  const int32_t *__restrict__ block_table, int max_blocks, const int32_t *__restrict__ ctx_lens,
                  int max_ctx, int split, float *__restrict__ part, int nsplit, unsigned int *__restrict__ counters,
                  float *__restrict__ out, int32_t *status) {
    using C = SplitCfg<D, NWARP>;
    constexpr int NT_ = C::NT, BPW = C::BPW, BPC = C::BPC, CH = C::CH;
    constexpr int TPL = CH / 32;               // softmax tokens per lane
    constexpr int NTK = (2 * G + 7) / 8;       // K-side n-tiles (hi, lo x G heads)
    constexpr int NKS = D / 16;                // K-side k16 steps
    constexpr int MTW = D / 16 / NWARP;        // V-side m-tiles per warp
    constexpr int NW = D / 128, NWV = D / 64;
    constexpr int KREC = C::KREC, VREC = C::VREC;
    constexpr int HPW = (G + NWARP - 1) / NWARP;   // heads owned per warp in the softmax
    constexpr int PROW = CH + 8;               // halves per sP row (pad: conflict-free fragment reads)

    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *sK = smem;                                        // [2][BPC][KREC]
    uint8_t *sV = sK + C::kBytes;                              // [2][BPC][VREC]
    __half *sP = reinterpret_cast<__half *>(sV + C::vBytes);   // [8][PROW] weights, head-major
    float *sS = reinterpret_cast<float *>(sP + 8 * PROW);      // [CH][G] scores
    float *sAcc = reinterpret_cast<float *>(sK);               // [G][D], after the loop
    __shared__ int sOk[2][BPC];
    __shared__ float sF[8];
    __shared__ float sM[8], sL[8], sT[8];
    __shared__ int sE[8];

    const int s = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
    int L = ctx_lens[b];
    if (L > max_ctx) L = max_ctx;
    const int t0 = s * split;
    if (t0 >= L) {                             // nothing to attend: split 0 writes out = 0
        if (L <= 0 && s == 0)
            for (int i = tid; i < G * D; i += NT_) out[((size_t)b * hq + kh * G) * D + i] = 0.f;
        return;
    }
    const int t1 = min(L, t0 + split);

    // stage the K and V records of the chunk starting at token tc into buffer buf
    auto issue_chunk = [&](int tc, int buf) {
        const int k = tid % BPC;
        const bool inrange = tc + kBlock * k < t1;
        const int64_t p = inrange ? block_of(block_table, b, max_blocks, tc / kBlock + k, num_blocks) : -1;
        if (tid < BPC) {
            sOk[buf][k] = p >= 0;
            if (inrange && p < 0) flag_status(status, TQ_STATUS_BAD_SLOT);
        }
        if (p >= 0) {
            const uint8_t *gk = k_pool + ((size_t)p * hkv + kh) * KREC;
            const uint8_t *gv = v_pool + ((size_t)p * hkv + kh) * VREC;
            uint8_t *dk = sK + ((size_t)buf * BPC + k) * KREC;
            uint8_t *dv = sV + ((size_t)buf * BPC + k) * VREC;
            for (int j = tid / BPC; j < KREC / 16; j += NT_ / BPC) cp_async16(dk + 16 * j, gk + 16 * j);
            for (int j = tid / BPC; j < VREC / 16; j += NT_ / BPC) cp_async16(dv + 16 * j, gv + 16 * j);
        }
        cp_async_commit();
    };
    issue_chunk(t0, 0);

    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    float A[4];
    walsh4(ph->centroid, A);
    const float Asum = A[0] + A[1] + A[2] + A[3];
    const float inv_sd = rsqrtf((float)D);
    const float qjl = 1.2533141373155003f / (float)D;   // sqrt(pi/2) / d
    // f16x2 {1.0, 1.0}, read at run time so that it stays in a register for LOP3
    const uint32_t one16x2 = (uint32_t)ph->one16x2;

    // weight rows of heads >= G stay zero
    for (int i = tid; i < (8 - G) * PROW; i += NT_) sP[G * PROW + i] = __float2half(0.f);

    // K-side operand fragments and offset constants of this (sequence, kv head)
    const uint8_t *pack = packs + ((size_t)b * hkv + kh) * kPackBytes(D);
    const float *pf = reinterpret_cast<const float *>(pack) + kPackFloatOff(D);
    uint32_t bq[2][NKS][NTK][2];
#pragma unroll
    for (int qu = 0; qu < 2; ++qu)
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks)
#pragma unroll
            for (int nt = 0; nt < NTK; ++nt) {
                const uint2 w = *reinterpret_cast<const uint2 *>(
                    pack + (((size_t)(qu * NKS + ks) * NTK + nt) * 64 + lane * 2) * 4);
                bq[qu][ks][nt][0] = w.x;
                bq[qu][ks][nt][1] = w.y;
            }
    float cq[NTK], cu[NTK];
#pragma unroll
    for (int nt = 0; nt < NTK; ++nt) {
        const int hg = 4 * nt + tig;           // columns 2tig (hi) and 2tig+1 (lo) of n-tile nt
        cq[nt] = hg < G ? pf[hg] * Asum : 0.f;
        cu[nt] = hg < G ? pf[8 + hg] : 0.f;
    }
    // V side: operand mask/base of this warp's m-tiles
    uint32_t vmask[MTW], vbase[MTW];
#pragma unroll
    for (int i = 0; i < MTW; ++i) {
        const int q = 8 + ((warp * MTW + i) & 7);
        vmask[i] = 0x00010001u << q;
        vbase[i] = (q == 14) ? 0u : one16x2;
    }
    const int mhi = (warp * MTW) >> 3;

    float O[4][MTW][4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int i = 0; i < MTW; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k) O[m][i][k] = 0.f;
    float m_run[HPW], l_run[HPW], w_ref[HPW], T_run[HPW];
    int e_run[HPW];
#pragma unroll
    for (int k = 0; k < HPW; ++k) {
        m_run[k] = -INFINITY;
        l_run[k] = 0.f;
        w_ref[k] = 0.f;
        e_run[k] = 0;
        T_run[k] = 0.f;
    }

    int buf = 0;
    for (int tc = t0; tc < t1; tc += CH, buf ^= 1) {
        cp_async_wait_all();
        __syncthreads();   // chunk `buf` staged and visible; the other buffer is free
        if (tc + CH < t1) issue_chunk(tc + CH, buf ^ 1);
        const uint8_t *kb_base = sK + (size_t)buf * BPC * KREC;
        const uint8_t *vb_base = sV + (size_t)buf * BPC * VREC;
        // ---- K side: warp scores blocks BPW*warp .. BPW*warp+BPW-1 of the chunk
#pragma unroll 1
        for (int bw = 0; bw < BPW; ++bw) {
            const int k = BPW * warp + bw;
            const bool ok = sOk[buf][k] != 0;
            const uint8_t *rec = kb_base + (size_t)k * KREC;
            uint32_t W[4][2][NW];
#pragma unroll
            for (int pl = 0; pl < 4; ++pl) {
                if (NW == 1) {
                    const uint2 w = *reinterpret_cast<const uint2 *>(rec + pl * 2 * D + lane * 8);
                    W[pl][0][0] = w.x;
                    W[pl][1][0] = w.y;
                } else {
                    const uint4 w = *reinterpret_cast<const uint4 *>(rec + pl * 2 * D + lane * 16);
                    W[pl][0][0] = w.x;
                    W[pl][0][NW - 1] = w.y;
                    W[pl][1][0] = w.z;
                    W[pl][1][NW - 1] = w.w;
                }
            }
            float nrm[2], gam[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const __half2 ng = *reinterpret_cast<const __half2 *>(rec + 8 * D + 4 * (gid + 8 * r));
                nrm[r] = __low2float(ng);
                gam[r] = __high2float(ng);
            }
            // five masks as independent accumulator chains: code = sum_m A_m (mask m), qjl = mask 4
            uint32_t w[5][2][NW], w8[5][2][NW];
#pragma unroll
            for (int m = 0; m < 5; ++m)
#pragma unroll
                for (int th = 0; th < 2; ++th)
#pragma unroll
                    for (int wj = 0; wj < NW; ++wj) {
                        w[m][th][wj] = (m < 3) ? W[m][th][wj]
                                     : (m == 3) ? (W[0][th][wj] ^ W[1][th][wj] ^ W[2][th][wj]) : W[3][th][wj];
                        w8[m][th][wj] = w[m][th][wj] << 8;
                    }
            float acc[5][NTK][4];
#pragma unroll
            for (int m = 0; m < 5; ++m)
#pragma unroll
                for (int nt = 0; nt < NTK; ++nt)
#pragma unroll
                    for (int x = 0; x < 4; ++x) acc[m][nt][x] = 0.f;
#pragma unroll
            for (int ks = 0; ks < NKS; ++ks) {
                const int q = 8 + (ks & 7), wj = ks >> 3;
                const uint32_t msk = op_mask(q), bas = (q == 14) ? 0u : one16x2;
#pragma unroll
                for (int m = 0; m < 5; ++m) {
                    const uint32_t a0 = lop_and_xor(w8[m][0][wj], msk, bas), a1 = lop_and_xor(w8[m][1][wj], msk, bas);
                    const uint32_t a2 = lop_and_xor(w[m][0][wj], msk, bas), a3 = lop_and_xor(w[m][1][wj], msk, bas);
                    const int qu = (m == 4) ? 1 : 0;
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt)
                        mma_f16(acc[m][nt], a0, a1, a2, a3, bq[qu][ks][nt][0], bq[qu][ks][nt][1]);
                }
            }
            float code[NTK][4], qjv[NTK][4];
#pragma unroll
            for (int nt = 0; nt < NTK; ++nt)
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    code[nt][x] = A[0] * acc[0][nt][x] + A[1] * acc[1][nt][x] + A[2] * acc[2][nt][x] + A[3] * acc[3][nt][x];
                    qjv[nt][x] = acc[4][nt][x];
                }
#pragma unroll
            for (int nt = 0; nt < NTK; ++nt) {
                const int hg = 4 * nt + tig;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float dot_c = code[nt][2 * r] + code[nt][2 * r + 1] - cq[nt];
                    const float dot_q = qjv[nt][2 * r] + qjv[nt][2 * r + 1] - cu[nt];
                    const int tl = kBlock * k + gid + 8 * r;           // token within the chunk
                    const bool valid = ok && (tc + tl < t1);
                    const float sc = nrm[r] * inv_sd * (dot_c * inv_sd + gam[r] * qjl * dot_q);
                    if (hg < G) sS[tl * G + hg] = valid ? sc : -INFINITY;
                }
            }
        }
        __syncthreads();   // scores of the chunk are in sS
        // ---- online softmax: warp owns heads warp, warp + NWARP
#pragma unroll
        for (int hk = 0; hk < HPW; ++hk) {
            const int h = warp + NWARP * hk;
            if (h < G) {
                float sc[TPL], w[TPL], p[TPL];
                float cmax = -INFINITY;
#pragma unroll
                for (int i = 0; i < TPL; ++i) {
                    sc[i] = sS[(lane + 32 * i) * G + h];
                    cmax = fmaxf(cmax, sc[i]);
                }
                cmax = warp_max(cmax);
                const float m_new = fmaxf(m_run[hk], cmax);
                const float alpha = (m_run[hk] == -INFINITY) ? 0.f : __expf(m_run[hk] - m_new);
                float psum = 0.f, wmax = 0.f;
#pragma unroll
                for (int i = 0; i < TPL; ++i) {
                    const int tl = lane + 32 * i;
                    p[i] = (sc[i] == -INFINITY) ? 0.f : __expf(sc[i] - m_new);
                    const float nv = __half2float(*reinterpret_cast<const __half *>(
                        vb_base + (size_t)(tl >> 4) * VREC + 6 * D + 2 * (tl & 15)));
                    w[i] = (p[i] > 0.f) ? p[i] * nv * inv_sd : 0.f;
                    psum += p[i];
                    wmax = fmaxf(wmax, fabsf(w[i]));
                }
                psum = warp_sum(psum);
                wmax = warp_max(wmax);
                const float wr = fmaxf(w_ref[hk] * alpha, wmax);
                const int e_new = wr > 0.f ? scale_exp(wr) : e_run[hk];
                const float f = ldexpf(alpha, e_new - e_run[hk]);
                float tsum = 0.f;
#pragma unroll
                for (int i = 0; i < TPL; ++i) {
                    const __half hv = __float2half_rn(ldexpf(w[i], e_new));
                    sP[h * PROW + lane + 32 * i] = hv;
                    tsum += __half2float(hv);
                }
                T_run[hk] = T_run[hk] * f + warp_sum(tsum);
                l_run[hk] = l_run[hk] * alpha + psum;
                m_run[hk] = m_new;
                w_ref[hk] = wr;
                e_run[hk] = e_new;
                if (lane == 0) sF[h] = f;
            }
        }
        __syncthreads();   // weights of the chunk are in sP, factors in sF
        // ---- V side: coordinates of m-tiles warp*MTW .. warp*MTW+MTW-1 (columns = heads)
        {
            const float f0 = (2 * tig < G) ? sF[2 * tig] : 0.f;
            const float f1 = (2 * tig + 1 < G) ? sF[2 * tig + 1] : 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int i = 0; i < MTW; ++i) {
                    O[m][i][0] *= f0;
                    O[m][i][1] *= f1;
                    O[m][i][2] *= f0;
                    O[m][i][3] *= f1;
                }
        }
#pragma unroll 2
        for (int kb = 0; kb < BPC; ++kb) {
            const uint8_t *rec = vb_base + (size_t)kb * VREC;
            uint32_t x[3][2];
#pragma unroll
            for (int pl = 0; pl < 3; ++pl) {
                const uint2 wv = *reinterpret_cast<const uint2 *>(rec + pl * 2 * D + (lane * NWV + 2 * mhi) * 4);
                x[pl][0] = wv.x;
                x[pl][1] = wv.y;
            }
            const __half *prow = sP + gid * PROW + kBlock * kb + 2 * tig;
            const uint32_t b0 = *reinterpret_cast<const uint32_t *>(prow);
            const uint32_t b1 = *reinterpret_cast<const uint32_t *>(prow + 8);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t x0 = (m < 3) ? x[m][0] : (x[0][0] ^ x[1][0] ^ x[2][0]);
                const uint32_t x1 = (m < 3) ? x[m][1] : (x[0][1] ^ x[1][1] ^ x[2][1]);
                const uint32_t x0s = x0 << 8, x1s = x1 << 8;
#pragma unroll
                for (int i = 0; i < MTW; ++i) {
                    const uint32_t a0 = lop_and_xor(x0s, vmask[i], vbase[i]), a1 = lop_and_xor(x1s, vmask[i], vbase[i]);
                    const uint32_t a2 = lop_and_xor(x0, vmask[i], vbase[i]), a3 = lop_and_xor(x1, vmask[i], vbase[i]);
                    mma_f16(O[m][i], a0, a1, a2, a3, b0, b1);
                }
            }
        }
    }

    // ---- epilogue: combine the masks, undo the operand offsets and the weight scale
#pragma unroll
    for (int hk = 0; hk < HPW; ++hk) {
        const int h = warp + NWARP * hk;
        if (h < G && lane == 0) {
            sM[h] = m_run[hk];
            sL[h] = l_run[hk];
            sE[h] = e_run[hk];
            sT[h] = T_run[hk];
        }
    }
    __syncthreads();   // sK is no longer read; sAcc reuses it
#pragma unroll
    for (int i = 0; i < MTW; ++i) {
        const int mt = warp * MTW + i, q = 8 + (mt & 7);
        const float al = op_alpha(q), inv_de = 2.f / op_delta(q);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * tig + e;
            if (h < G) {
                const float T = sT[h];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    float v = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) v += A[m] * ((O[m][i][2 * r + e] - al * T) * inv_de - T);
                    sAcc[h * D + 16 * mt + gid + 8 * r] = ldexpf(v, -sE[h]);
                }
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float *dst = part + (((size_t)b * hq + kh * G + h) * nsplit + s) * kPartStride(D);
        for (int i = tid; i < D; i += NT_) dst[4 + i] = sAcc[h * D + i];
        if (tid == 0) {
            dst[0] = sM[h];
            dst[1] = sL[h];
        }
    }
    // ---- the last split of this (sequence, kv head) to finish merges all of them
    __shared__ bool s_last;
    __threadfence();                           // every thread publishes its part of the partial
    __syncthreads();
    if (tid == 0) {
        const unsigned int nsb = (unsigned int)((L + split - 1) / split);
        const unsigned int done = atomicAdd(&counters[b * hkv + kh], 1u) + 1u;
        s_last = (done == nsb);
        if (s_last) counters[b * hkv + kh] = 0u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int nsb = (L + split - 1) / split;
    constexpr int R = D / 32;
    for (int h = warp; h < G; h += NWARP) {
        const int row = b * hq + kh * G + h;
        const float *p0 = part + (size_t)row * nsplit * kPartStride(D);
        float M = -INFINITY;
        for (int t = 0; t < nsb; ++t) M = fmaxf(M, __ldcg(p0 + (size_t)t * kPartStride(D)));
        float v[R];
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = 0.f;
        float l = 0.f;
        for (int t = 0; t < nsb; ++t) {
            const float *ps = p0 + (size_t)t * kPartStride(D);
            const float m = __ldcg(ps);
            const float w = (m == -INFINITY) ? 0.f : __expf(m - M);
            l = fmaf(__ldcg(ps + 1), w, l);
#pragma unroll
            for (int r = 0; r < R; ++r) v[r] = fmaf(__ldcg(ps + 4 + 32 * r + lane), w, v[r]);
        }
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] *= inv;
        // out = Pi^T a = D (H a) / sqrt d
        fwht_warp<R>(v, lane);
        const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
#pragma unroll
        for (int r = 0; r < R; ++r) out[(size_t)row * D + 32 * r + lane] = v[r] * inv_sd * __ldg(Dsign + 32 * r + lane);
    }
}

// Context split length: the shortest power-of-two multiple of 512 tokens that
// still gives about 4 waves of CTAs (3 per SM) over the (sequence, kv head) units.
int choose_split(int batch, int hkv, int max_ctx) {
    const long long units = (long long)batch * hkv;
    const long long target = 152LL * 3 * 4;
    int split = kMinSplit;
    while (split < kMaxSplit && units * ((max_ctx + 2LL * split - 1) / (2LL * split)) >= target) split *= 2;
    return split;
}

struct WsLayout {
    uint8_t *packs;
    unsigned int *counters;
    float *part;
    int split;
    int nsplit;
};
WsLayout ws_layout(void *ws, int d, int batch, int hq, int hkv, int max_ctx) {
    WsLayout w;
    w.split = choose_split(batch, hkv, max_ctx);
    w.nsplit = max(1, (max_ctx + w.split - 1) / w.split);
    w.packs = reinterpret_cast<uint8_t *>(ws);
    w.counters = reinterpret_cast<unsigned int *>(w.packs + (size_t)batch * hq * kPackBytes(d));
    w.part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(w.counters) + kCounterBytes(batch, hq));
    return w;
}

template <int D, int NTK, typename T>
cudaError_t qprep_launch_t(const uint8_t *P, const void *q, int batch, int hq, int hkv, uint8_t *packs,
                           unsigned int *counters, cudaStream_t st) {
    constexpr size_t smem = (size_t)2 * kQRows * D * 4 + (size_t)2 * kProjRows * D * 4;
    auto kern = qprep_kernel<D, NTK, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(batch * hq + kQRows - 1) / kQRows, 128, smem, st>>>(P, (const T *)q, batch, hq, hkv, packs, counters);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t qprep_launch(const uint8_t *P, const void *q, int batch, int hq, int hkv, uint8_t *packs,
                         unsigned int *counters, cudaStream_t st) {
    // n-tile count of the K-side operand: (2G + 7) / 8, as in decode_mma_kernel
    if (hq / hkv <= 4) return qprep_launch_t<D, 1, T>(P, q, batch, hq, hkv, packs, counters, st);
    return qprep_launch_t<D, 2, T>(P, q, batch, hq, hkv, packs, counters, st);
}

template <int D, int G>
cudaError_t partial_launch_g(dim3 grid, cudaStream_t st, const uint8_t *P, const uint8_t *packs, int hq, int hkv,
                             const uint8_t *kp, const uint8_t *vp, int64_t nb, const int32_t *bt, int mb,
                             const int32_t *ctx, int max_ctx, int split, float *part, int nsplit,
                             unsigned int *counters, float *out, int32_t *status) {
    constexpr int NWARP = G <= 4 ? 4 : 8;
    constexpr size_t smem = split_smem_bytes<D, G, NWARP>();
    auto kern = decode_mma_kernel<D, G, NWARP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, NWARP * 32, smem, st>>>(P, packs, hq, hkv, kp, vp, nb, bt, mb, ctx, max_ctx, split, part, nsplit,
                                        counters, out, status);
    return cudaGetLastError();
}

template <int D>
cudaError_t partial_launch(int G, dim3 grid, cudaStream_t st, const uint8_t *P, const uint8_t *packs, int hq,
                           int hkv, const uint8_t *kp, const uint8_t *vp, int64_t nb, const int32_t *bt, int mb,
                           const int32_t *ctx, int max_ctx, int split, float *part, int nsplit,
                           unsigned int *counters, float *out, int32_t *status) {
#define TQ_PART(GG) return partial_launch_g<D, GG>(grid, st, P, packs, hq, hkv, kp, vp, nb, bt, mb, ctx, max_ctx, split, part, nsplit, counters, out, status)
    switch (G) {
        case 1: TQ_PART(1);
        case 2: TQ_PART(2);
        case 3: TQ_PART(3);
        case 4: TQ_PART(4);
        case 5: TQ_PART(5);
        case 6: TQ_PART(6);
        case 7: TQ_PART(7);
        default: TQ_PART(8);
    }
#undef TQ_PART
}

}  // namespace

cudaError_t launch_qprep(int d, int dtype, const void *params, const void *q, int batch, int hq, int hkv,
                         int max_ctx, void *ws, cudaStream_t st) {
    const WsLayout w = ws_layout(ws, d, batch, hq, hkv, max_ctx);
    const uint8_t *P = (const uint8_t *)params;
    if (d == 128)
        return dtype == TQ_DTYPE_BF16 ? qprep_launch<128, __nv_bfloat16>(P, q, batch, hq, hkv, w.packs, w.counters, st)
                                      : qprep_launch<128, float>(P, q, batch, hq, hkv, w.packs, w.counters, st);
    return dtype == TQ_DTYPE_BF16 ? qprep_launch<256, __nv_bfloat16>(P, q, batch, hq, hkv, w.packs, w.counters, st)
                                  : qprep_launch<256, float>(P, q, batch, hq, hkv, w.packs, w.counters, st);
}

cudaError_t launch_splitk(int d, const void *params, int batch, int hq, int hkv, const void *k_pool,
                          const void *v_pool, int64_t num_blocks, const int32_t *block_table, int max_blocks,
                          const int32_t *ctx_lens, int max_ctx, float *out, void *ws, int32_t *status,
                          cudaStream_t st) {
    const WsLayout w = ws_layout(ws, d, batch, hq, hkv, max_ctx);
    const dim3 grid(w.nsplit, hkv, batch);
    const int G = hq / hkv;
    const uint8_t *P = (const uint8_t *)params;
    if (d == 128)
        return partial_launch<128>(G, grid, st, P, w.packs, hq, hkv, (const uint8_t *)k_pool, (const uint8_t *)v_pool,
                                   num_blocks, block_table, max_blocks, ctx_lens, max_ctx, w.split, w.part, w.nsplit,
                                   w.counters, out, status);
    return partial_launch<256>(G, grid, st, P, w.packs, hq, hkv, (const uint8_t *)k_pool, (const uint8_t *)v_pool,
                               num_blocks, block_table, max_blocks, ctx_lens, max_ctx, w.split, w.part, w.nsplit,
                               w.counters, out, status);
}

}  // namespace tq
