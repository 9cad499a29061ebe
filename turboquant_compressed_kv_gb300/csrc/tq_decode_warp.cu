// tq_decode_warp.cu -- the decode pass at d = 128: every warp scores, weighs and sums its
// own 16-token blocks end to end.
//
// Method as in tq_decode.cu (scores and value sums in the rotated domain, straight from
// the packed cells, signs and fp16 norms: the "fused dequantisation" of the SwiftLM
// README, "TurboQuantization: KV Cache Compression"; blocks through the block table of
// the vLLM-MLX explainer, "Paged KVキャッシュ"), and the same stream-K schedule,
// workspace and merge.  What differs is the work split inside a CTA:
//  * A CTA of 4 warps takes the same 128-token chunks; warp w owns blocks 2w, 2w+1 of
//    each chunk and stages them itself (cp.async, one pair ahead), so the chunk loop has
//    no CTA-wide barrier.
//  * K side as in the coordinate-split pass: five +-1 planes on f16 mma.sync against
//    the f16 hi/lo query fragments.
//  * Online softmax in registers, per warp and head, with a lazily moved reference:
//    weights are 2^(s - m) * nv with s in log2 units, and m only moves when a block's
//    maximum passes m + 8 (or a weight would leave the f16 range), so the accumulators
//    are rescaled rarely.
//  * V side over all 128 coordinates of the warp's block.  The four Walsh planes share
//    one accumulator per m-tile: plane m's B operand is the weights times A_m in f16 (the
//    value sum sum_t w_t c[cell_t] = sum_m A_m sum_t w_t sigma_m), with an f16 lo part for
//    the planes of the two large coefficients (A_1, A_2; A_0 and A_3 are 3.4 and 15 times
//    smaller than A_2, so their single rounding costs little).
//    One more mma with a constant A = 1 sums those B operands (for the offset of the
//    0/delta operands).  Each block's mma sums start from zero and are added to fp32
//    running sums: chained tensor-core accumulation over thousands of tokens is not
//    accurate enough for the 2 sum(w b) - sum(w) cancellation.
//  * At the end of a (sequence, kv head) segment the 4 warps' (m, l, acc) are merged
//    in shared memory, then the segment is finished or left as a partial exactly as in
//    the coordinate-split pass (m in log2 units here).
#include "tq_split.cuh"

#ifndef TQ_WARP_BQ_SMEM
#define TQ_WARP_BQ_SMEM 0        // 1: K-side query fragments read from shared memory for every group size
#endif
#ifndef TQ_WARP_MINBLOCKS
#define TQ_WARP_MINBLOCKS 3      // resident CTAs per SM the register budget is sized for (G <= 4)
#endif
#ifndef TQ_WARP_MINBLOCKS_WIDE
#define TQ_WARP_MINBLOCKS_WIDE 3 // the same for groups of 5..8 heads (two K-side n-tiles)
#endif

namespace tq {
namespace {

constexpr int kWD = 128, kWWarps = 4, kWBpw = TQ_SPLITK_BPW;
constexpr int kWKrec = (int)k_record(kWD), kWVrec = (int)v_record(kWD), kWRec = kWKrec + kWVrec;
constexpr float kTau = 8.f;          // the reference moves when a block's maximum passes it by this (log2)
constexpr float kWLimit = 32768.f;   // largest weight held (f16 max is 65504)
constexpr float kNoRef = -1e30f;     // softmax reference before the first unmasked score

template <int G>
__host__ __device__ constexpr int w_ntk() { return (2 * G + 7) / 8; }
// K-side query fragments in shared memory rather than registers: needed above 4 heads
// (two n-tiles would take 64 registers)
template <int G>
__host__ __device__ constexpr bool w_bq_smem() { return TQ_WARP_BQ_SMEM || G > 4; }

template <int G>
__host__ __device__ constexpr size_t warp_smem_bytes() {
    const size_t stage = (size_t)kWWarps * 2 * kWBpw * kWRec;                  // per warp: 2 buffers x BPW blocks
    const size_t merge = (size_t)(kWWarps + 1) * G * kWD * 4;                  // sAccW + sAcc
    const size_t bq = w_bq_smem<G>() ? (size_t)2 * (kWD / 16) * w_ntk<G>() * 64 * 4 : 0;
    return stage + merge + bq;
}

// ld.shared of a query fragment at each use: a plain load would be hoisted out of the block
// loop by the compiler and pin 64 registers
__device__ __forceinline__ uint2 lds_u2(const uint32_t *p) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "r"((uint32_t)__cvta_generic_to_shared(p)));
    return v;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int G>
__global__ void __launch_bounds__(kWWarps * 32, G <= 4 ? TQ_WARP_MINBLOCKS : TQ_WARP_MINBLOCKS_WIDE)
decode_warp_kernel(const uint8_t *__restrict__ params, const uint8_t *__restrict__ packs, int batch, int q_len, int hq, int hkv,
                   const uint8_t *__restrict__ k_pool, const uint8_t *__restrict__ v_pool, int64_t num_blocks,
                   const int32_t *__restrict__ block_table, int max_blocks, const int32_t *__restrict__ ctx_lens,
                   int ctx_add, int max_ctx, const int64_t *__restrict__ cpre, const int32_t *__restrict__ cta_b,
                   float *__restrict__ part, unsigned int *__restrict__ counters, float *__restrict__ out,
                   float *__restrict__ lse, int32_t *status) {
    constexpr int D = kWD, NT = kWWarps * 32, NWARP = kWWarps, BPW = kWBpw;
    constexpr int CH = kBlock * NWARP * BPW;    // tokens per chunk (the schedule's unit)
    constexpr int NTK = w_ntk<G>();             // K-side n-tiles; thread holds heads 4*nt + tig
    constexpr int NKS = D / 16, MT = D / 16, R = D / 32;
    constexpr int KREC = kWKrec, VREC = kWVrec, REC = kWRec;
    constexpr size_t kStage = (size_t)NWARP * 2 * BPW * REC;
    constexpr size_t kMerge = (size_t)(NWARP + 1) * G * D * 4;
    constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;

    extern __shared__ __align__(16) uint8_t smem[];
    const int cta = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
    uint8_t *sStage = smem + (size_t)warp * 2 * BPW * REC;     // this warp's [2][BPW][K record | V record]
    float *sAccW = reinterpret_cast<float *>(smem + kStage);     // [NWARP][G][D], segment end only
    float *sAcc = sAccW + NWARP * G * D;                         // [G][D]
    uint32_t *sBq = reinterpret_cast<uint32_t *>(smem + kStage + kMerge);
    __shared__ float sMW[NWARP][8], sLW[NWARP][8];
    __shared__ float sM[8], sL[8];
    __shared__ bool s_last;

    pdl_wait();   // everything before this launch (the prep's schedule, packs, counters) is complete

    for (int b = cta; b < batch; b += gridDim.x)
        if (attended_len(ctx_lens[b], ctx_add, max_ctx) == 0)
        {
            for (int i = tid; i < q_len * hq * D; i += NT) out[(size_t)b * q_len * hq * D + i] = 0.f;
            if (lse)
                for (int i = tid; i < q_len * hq; i += NT) lse[(size_t)b * q_len * hq + i] = -INFINITY;
        }

    const int64_t W = cpre[batch];
    const int P = (int)(W < (int64_t)gridDim.x ? W : (int64_t)gridDim.x);
    if (cta >= P) return;
    const int64_t g0 = sk_begin(cta, P, W), g1 = sk_begin(cta + 1, P, W);

    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    float A[4];
    walsh4(ph->centroid, A);
    const float Asum = A[0] + A[1] + A[2] + A[3];
    const float inv_sd = rsqrtf((float)D);
    const float c_sc = inv_sd * kLog2e;                 // scores in log2 units
    const float qjl = 1.2533141373155003f / (float)D;   // sqrt(pi/2) / d
    const uint32_t one16x2 = (uint32_t)ph->one16x2;

    // The CTA's range [g0, g1) of global chunks, walked one (sequence, kv head) segment at a time.
    struct Seg {
        int b, kh, t0, t1, L;
        int64_t us, ue, se;
    };
    auto make_seg = [&](int b, int kh, int64_t ub, int nchb, int64_t g) {
        Seg s;
        s.b = b;
        s.kh = kh;
        s.us = ub + (int64_t)kh * nchb;
        s.ue = s.us + nchb;
        s.se = (g1 < s.ue) ? g1 : s.ue;
        s.t0 = (int)(g - s.us) * CH;
        s.L = attended_len(ctx_lens[b], ctx_add, max_ctx);
        s.t1 = min(s.L, (int)(s.se - s.us) * CH);
        return s;
    };
    // the segment after s, if the range has one
    auto next_seg = [&](const Seg &s, Seg &n) -> bool {
        if (s.se >= g1) return false;
        int nb = s.b, nkh = s.kh + 1;
        int64_t nub = cpre[nb];
        int nn = (int)((cpre[nb + 1] - nub) / hkv);
        if (nkh == hkv) {
            nkh = 0;
            do {
                ++nb;
                nub = cpre[nb];
                nn = (int)((cpre[nb + 1] - nub) / hkv);
            } while (nn == 0);
        }
        n = make_seg(nb, nkh, nub, nn, s.se);
        return true;
    };
    // stage this warp's blocks of the chunk at token tc of segment s into buffer buf; bit bw
    // of the result is set when block bw is in range and has a valid physical id.  Blocks past
    // the context are not copied; a block with a bad id is replaced by block 0 (its scores are
    // masked), so the copies need no per-lane branch.
    auto stage = [&](const Seg &s, int tc, int buf) -> int {
        int okm = 0;
#pragma unroll
        for (int bw = 0; bw < BPW; ++bw) {
            const int tb = tc + kBlock * (BPW * warp + bw);
            if (tb < s.t1) {
                const int64_t p = block_of(block_table, s.b, max_blocks, tb / kBlock, num_blocks);
                if (p < 0 && lane == 0) flag_status(status, TQ_STATUS_BAD_SLOT);
                okm |= (p >= 0) << bw;
                const size_t row = (size_t)(p < 0 ? 0 : p) * hkv + s.kh;
                const uint8_t *gk = k_pool + row * KREC, *gv = v_pool + row * VREC;
                uint8_t *dk = sStage + (size_t)(buf * BPW + bw) * REC, *dv = dk + KREC;
#pragma unroll
                for (int j = lane; j < KREC / 16; j += 32) cp_async16(dk + 16 * j, gk + 16 * j);
#pragma unroll
                for (int j = lane; j < VREC / 16; j += 32) cp_async16(dv + 16 * j, gv + 16 * j);
            }
        }
        cp_async_commit();
        return okm;
    };

    // the staging area starts zeroed: slots of blocks that are not copied then always hold
    // finite values (old records or zeros), whose weight is exactly 0
    for (int i = tid; i < (int)(kStage / 16); i += NT) reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    Seg s;
    {
        const int b0 = cta_b[cta];
        const int64_t ub0 = cpre[b0];
        const int n0 = (int)((cpre[b0 + 1] - ub0) / hkv);
        s = make_seg(b0, (int)((g0 - ub0) / n0), ub0, n0, g0);
    }
    bool first_seg = true;
    int buf = 0;
    int okm = stage(s, s.t0, 0);

#pragma unroll 1
    while (true) {
        const int b = s.b, kh = s.kh, t0 = s.t0, t1 = s.t1;
        const int64_t us = s.us, ue = s.ue;
        Seg ns;
        const bool more_segs = next_seg(s, ns);

        // K-side query fragments and offset constants of this (sequence, kv head)
        const uint8_t *pack = packs + ((size_t)b * hkv + kh) * kPackBytes(D);
        const float *pf = reinterpret_cast<const float *>(pack) + kPackFloatOff(D);
        constexpr bool BQS = w_bq_smem<G>();
        uint32_t bq[2][NKS][NTK][2];
        if constexpr (BQS) {
            for (int i = tid; i < 2 * NKS * NTK * 64 / 4; i += NT)
                reinterpret_cast<uint4 *>(sBq)[i] = reinterpret_cast<const uint4 *>(pack)[i];
            __syncthreads();
        } else {
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
        }
        float cq[NTK], cu[NTK];
        int tlim[NTK];   // tokens column 4 nt + tig attends in this segment (query i: L - (q_len - 1 - i))
#pragma unroll
        for (int nt = 0; nt < NTK; ++nt) {
            const int hg = 4 * nt + tig;
            cq[nt] = hg < G ? pf[hg] * Asum : 0.f;
            cu[nt] = hg < G ? pf[8 + hg] : 0.f;
            tlim[nt] = hg < G ? min(t1, s.L - (q_len - 1 - hg / (G / q_len))) : 0;
        }

        // running value sums (fp32 adds of the per-block mma results) and offset sums
        float arun[MT][4], Trun[4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int k = 0; k < 4; ++k) arun[mt][k] = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) Trun[k] = 0.f;
        float mref[NTK], lpart[NTK];
#pragma unroll
        for (int nt = 0; nt < NTK; ++nt) {
            mref[nt] = kNoRef;   // finite: exp2(s - mref) is 0 for masked scores (s = -inf) at any time
            lpart[nt] = 0.f;
        }

        // multiply the accumulators and row sums of head h (= 4 nt + tig) by f[nt]
        auto rescale = [&](const float (&f)[NTK]) {
#pragma unroll
            for (int nt = 0; nt < NTK; ++nt) lpart[nt] *= f[nt];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                // accumulator column c holds head c (G > 4) or head c & 3 (G <= 4: hi, then lo parts)
                const int c = 2 * tig + e, hc = (G <= 4) ? (c & 3) : c;
                float fc = 1.f;
#pragma unroll
                for (int nt = 0; nt < NTK; ++nt) {
                    const float v = __shfl_sync(0xffffffffu, f[nt], (lane & ~3) | (hc & 3));
                    if ((hc >> 2) == nt) fc = v;
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    arun[mt][e] *= fc;
                    arun[mt][2 + e] *= fc;
                }
                Trun[e] *= fc;
                Trun[2 + e] *= fc;
            }
        };

#pragma unroll 1
        for (int tc = t0; tc < t1; tc += CH, buf ^= 1) {
            // stage the next chunk of this segment, or the first chunk of the next segment
            const bool ahead = tc + CH < t1 || more_segs;
            if (ahead) {
                const int nxt = (tc + CH < t1) ? stage(s, tc + CH, buf ^ 1) : stage(ns, ns.t0, buf ^ 1);
                okm = (okm & ~(((1 << BPW) - 1) << ((buf ^ 1) * BPW))) | (nxt << ((buf ^ 1) * BPW));
                cp_async_wait_1();
            } else {
                cp_async_wait_all();
            }
            __syncwarp();
#pragma unroll 1
            for (int bw = 0; bw < BPW; ++bw) {
                const int tb = tc + kBlock * (BPW * warp + bw);   // first token of the block
                if (tb >= t1) break;
                const bool ok = (okm >> (buf * BPW + bw)) & 1;
                const uint8_t *krec = sStage + (size_t)(buf * BPW + bw) * REC;
                const uint8_t *vrec = krec + KREC;

                // ---- K side: scores of tokens tb + gid + 8r for heads 4 nt + tig (log2 units)
                float s2[NTK][2];
                {
                    uint32_t Wd[4][2];
#pragma unroll
                    for (int pl = 0; pl < 4; ++pl) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(krec + pl * 2 * D + lane * 8);
                        Wd[pl][0] = w.x;
                        Wd[pl][1] = w.y;
                    }
                    float nrm[2], gam[2];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const __half2 ng = *reinterpret_cast<const __half2 *>(krec + 8 * D + 4 * (gid + 8 * r));
                        nrm[r] = __low2float(ng);
                        gam[r] = __high2float(ng);
                    }
                    uint32_t w[5][2], w8[5][2];
#pragma unroll
                    for (int m = 0; m < 5; ++m)
#pragma unroll
                        for (int th = 0; th < 2; ++th) {
                            w[m][th] = (m < 3) ? Wd[m][th] : (m == 3) ? (Wd[0][th] ^ Wd[1][th] ^ Wd[2][th]) : Wd[3][th];
                            w8[m][th] = w[m][th] << 8;
                        }
                    float acc[5][NTK][4];   // started by the first k-step's zero-accumulator mma
#pragma unroll
                    for (int ks = 0; ks < NKS; ++ks) {
                        const int q = 8 + ks;
                        const uint32_t msk = op_mask(q), bas = (q == 14) ? 0u : one16x2;
                        uint2 bsm[2][NTK];   // this k-step's fragments of q-bar (0) and u (1), shared-memory case
                        if constexpr (BQS) {
#pragma unroll
                            for (int qu = 0; qu < 2; ++qu)
#pragma unroll
                                for (int nt = 0; nt < NTK; ++nt)
                                    bsm[qu][nt] = lds_u2(sBq + ((qu * NKS + ks) * NTK + nt) * 64 + lane * 2);
                        }
#pragma unroll
                        for (int m = 0; m < 5; ++m) {
                            const uint32_t a0 = lop_and_xor(w8[m][0], msk, bas), a1 = lop_and_xor(w8[m][1], msk, bas);
                            const uint32_t a2 = lop_and_xor(w[m][0], msk, bas), a3 = lop_and_xor(w[m][1], msk, bas);
                            const int qu = (m == 4) ? 1 : 0;
#pragma unroll
                            for (int nt = 0; nt < NTK; ++nt) {
                                const uint32_t b0 = BQS ? bsm[qu][nt].x : bq[qu][ks][nt][0];
                                const uint32_t b1 = BQS ? bsm[qu][nt].y : bq[qu][ks][nt][1];
                                if (ks == 0) mma_f16_z(acc[m][nt], a0, a1, a2, a3, b0, b1);
                                else mma_f16(acc[m][nt], a0, a1, a2, a3, b0, b1);
                            }
                        }
                    }
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt) {
                        const int hg = 4 * nt + tig;
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            float code2 = 0.f;
#pragma unroll
                            for (int m = 0; m < 4; ++m)
                                code2 = fmaf(A[m], acc[m][nt][2 * r] + acc[m][nt][2 * r + 1], code2);
                            const float dot_c = code2 - cq[nt];
                            const float dot_q = acc[4][nt][2 * r] + acc[4][nt][2 * r + 1] - cu[nt];
                            const bool valid = ok && (tb + gid + 8 * r < tlim[nt]);
                            s2[nt][r] = valid ? nrm[r] * c_sc * (dot_c * inv_sd + gam[r] * qjl * dot_q) : -INFINITY;
                        }
                    }
                }

                // ---- online softmax: move the reference when the block's maximum passes it
                {
                    float f[NTK];
                    bool need = false;
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt) {
                        float bm = fmaxf(s2[nt][0], s2[nt][1]);
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
                        const bool up = bm > mref[nt] + kTau;
                        f[nt] = up ? exp2f(mref[nt] - bm) : 1.f;
                        if (up) mref[nt] = bm;
                        need |= up;
                    }
                    if (__any_sync(0xffffffffu, need)) rescale(f);
                }
                float wv[NTK][2], pr[NTK][2];
                {
                    float nv[2];
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        nv[r] = __half2float(*reinterpret_cast<const __half *>(vrec + 6 * D + 2 * (gid + 8 * r)));
                    float wmax = 0.f;
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt)
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const float p = exp2f(s2[nt][r] - mref[nt]);
                            pr[nt][r] = p;
                            wv[nt][r] = p * nv[r];
                            wmax = fmaxf(wmax, wv[nt][r]);
                        }
                    if (__any_sync(0xffffffffu, wmax > kWLimit)) {
                        // a weight would leave the f16 range: raise the reference of that head
                        float f[NTK];
#pragma unroll
                        for (int nt = 0; nt < NTK; ++nt) {
                            float hm = fmaxf(wv[nt][0], wv[nt][1]);
                            hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 4));
                            hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 8));
                            hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 16));
                            const float sh = hm > kWLimit ? ceilf(log2f(hm / kWLimit)) : 0.f;
                            f[nt] = exp2f(-sh);
                            mref[nt] += sh;
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                pr[nt][r] *= f[nt];
                                wv[nt][r] *= f[nt];
                            }
                        }
                        rescale(f);
                    }
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt) lpart[nt] += pr[nt][0] + pr[nt][1];
                }

                // ---- weights to the V-side B layout: thread (gid, tig) takes head gid & 3 (G <= 4)
                // or gid (G > 4), tokens 2 tig, 2 tig + 1 (b0) and 2 tig + 8, 2 tig + 9 (b1); token
                // t < 8 of head h sits in lane 4 t + (h & 3), slot 0 (t + 8: slot 1), n-tile h >> 2.
                // Planes 1 and 2 carry w A_m as f16 hi + lo (2^-22): for G <= 4 the lo parts fill
                // columns 4..7 of the same mma, for G > 4 they take a second mma.  Planes 0 and 3
                // carry one f16 (columns 4..7 zero).
                uint32_t Bh[4][2], Bl[4][2];
                {
                    const int srcA = 8 * tig + (gid & 3), srcB = srcA + 4;
                    const int hcol = (G <= 4) ? (gid & 3) : gid;     // head this thread's column carries
                    float u[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt) {
                        const float x0 = __shfl_sync(0xffffffffu, wv[nt][0], srcA);
                        const float x1 = __shfl_sync(0xffffffffu, wv[nt][0], srcB);
                        const float x2 = __shfl_sync(0xffffffffu, wv[nt][1], srcA);
                        const float x3 = __shfl_sync(0xffffffffu, wv[nt][1], srcB);
                        if ((hcol >> 2) == nt) {
                            u[0] = x0;
                            u[1] = x1;
                            u[2] = x2;
                            u[3] = x3;
                        }
                    }
                    if (hcol >= G) u[0] = u[1] = u[2] = u[3] = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float x0 = u[0] * A[m], x1 = u[1] * A[m], x2 = u[2] * A[m], x3 = u[3] * A[m];
                        const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
                        Bh[m][0] = *reinterpret_cast<const uint32_t *>(&h01);
                        Bh[m][1] = *reinterpret_cast<const uint32_t *>(&h23);
                        if (m == 1 || m == 2) {
                            const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                            Bl[m][0] = pack_h2(x0 - f01.x, x1 - f01.y);
                            Bl[m][1] = pack_h2(x2 - f23.x, x3 - f23.y);
                        } else {
                            Bl[m][0] = Bl[m][1] = 0u;
                        }
                        if (G <= 4) {   // columns 4..7: the lo parts (or zero)
                            Bh[m][0] = gid >= 4 ? Bl[m][0] : Bh[m][0];
                            Bh[m][1] = gid >= 4 ? Bl[m][1] : Bh[m][1];
                        }
                    }
                }

                // ---- V side: all 8 m-tiles, the four planes into one accumulator per m-tile
                {
                    uint32_t x[4][2];
#pragma unroll
                    for (int pl = 0; pl < 3; ++pl) {
                        const uint2 v = *reinterpret_cast<const uint2 *>(vrec + pl * 2 * D + lane * 8);
                        x[pl][0] = v.x;
                        x[pl][1] = v.y;
                    }
                    x[3][0] = x[0][0] ^ x[1][0] ^ x[2][0];
                    x[3][1] = x[0][1] ^ x[1][1] ^ x[2][1];
                    float O[MT][4], Tacc[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t xs0 = x[m][0] << 8, xs1 = x[m][1] << 8;
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const int q = 8 + mt;
                            const uint32_t msk = 0x00010001u << q, bas = vop_base(q);
                            const uint32_t a0 = lop_and_xor(xs0, msk, bas), a1 = lop_and_xor(xs1, msk, bas);
                            const uint32_t a2 = lop_and_xor(x[m][0], msk, bas), a3 = lop_and_xor(x[m][1], msk, bas);
                            if (m == 0) mma_f16_z(O[mt], a0, a1, a2, a3, Bh[m][0], Bh[m][1]);
                            else mma_f16(O[mt], a0, a1, a2, a3, Bh[m][0], Bh[m][1]);
                            if constexpr (G > 4) {
                                if (m == 1 || m == 2) mma_f16(O[mt], a0, a1, a2, a3, Bl[m][0], Bl[m][1]);
                            }
                        }
                        if (m == 0) mma_f16_z(Tacc, one16x2, one16x2, one16x2, one16x2, Bh[m][0], Bh[m][1]);
                        else mma_f16(Tacc, one16x2, one16x2, one16x2, one16x2, Bh[m][0], Bh[m][1]);
                        if constexpr (G > 4) {
                            if (m == 1 || m == 2) mma_f16(Tacc, one16x2, one16x2, one16x2, one16x2, Bl[m][0], Bl[m][1]);
                        }
                    }
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int k = 0; k < 4; ++k) arun[mt][k] += O[mt][k];
#pragma unroll
                    for (int k = 0; k < 4; ++k) Trun[k] += Tacc[k];
                }
            }
            __syncwarp();   // buffer `buf` is restaged in the next iteration
        }

        // ---- segment end: merge the warps' (m, l, acc) in shared memory
        float lh[NTK];
#pragma unroll
        for (int nt = 0; nt < NTK; ++nt) {
            float l = lpart[nt];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            lh[nt] = l;
        }
        __syncthreads();   // the previous segment's merge is done with sAccW / sAcc
        if (gid == 0) {
#pragma unroll
            for (int nt = 0; nt < NTK; ++nt) {
                const int h = 4 * nt + tig;
                if (h < G) {
                    sMW[warp][h] = mref[nt];
                    sLW[warp][h] = lh[nt];
                }
            }
        }
        if constexpr (G <= 4) {
            // columns 4..7 (tig 2, 3) carry the lo parts of heads 0..3 (tig 0, 1): add them in
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float t = __shfl_xor_sync(0xffffffffu, Trun[k], 2);
                if (tig < 2) Trun[k] += t;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const float o = __shfl_xor_sync(0xffffffffu, arun[mt][k], 2);
                    if (tig < 2) arun[mt][k] += o;
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int q = 8 + mt;
            const float al = vop_alpha(q), inv_de = 2.f / vop_delta(q);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = 2 * tig + e;
                if (h < G && (G > 4 || tig < 2)) {
                    const float T = Trun[e];
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        sAccW[(warp * G + h) * D + 16 * mt + gid + 8 * r] = (arun[mt][2 * r + e] - al * T) * inv_de - T;
                }
            }
        }
        __syncthreads();
        for (int i = tid; i < G * D; i += NT) {
            const int h = i / D;
            float M = -INFINITY;
#pragma unroll
            for (int w2 = 0; w2 < NWARP; ++w2) M = fmaxf(M, sMW[w2][h]);
            float v = 0.f, l = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < NWARP; ++w2) {
                const float fw = (sMW[w2][h] == -INFINITY) ? 0.f : exp2f(sMW[w2][h] - M);
                v = fmaf(fw, sAccW[(w2 * G + h) * D + (i % D)], v);
                l = fmaf(fw, sLW[w2][h], l);
            }
            sAcc[i] = v * inv_sd;
            if (i % D == 0) {
                sM[h] = M;
                sL[h] = l;
            }
        }
        __syncthreads();

        const int lo = sk_cta_of(us, P, W), hi = sk_cta_of(ue - 1, P, W);
        // output row of operand column h: query h / gq of head kh * gq + h % gq
        const int gq = G / q_len;
        auto out_row = [&](int h) { return ((size_t)b * q_len + h / gq) * hq + (size_t)kh * gq + h % gq; };
        if (lo == hi) {
            for (int h = warp; h < G; h += NWARP) {
                float v[R];
#pragma unroll
                for (int r = 0; r < R; ++r) v[r] = sAcc[h * D + 32 * r + lane];
                finish_row<D>(v, sL[h], params, out + out_row(h) * D, lane);
                if (lse && lane == 0) lse[out_row(h)] = sL[h] > 0.f ? sM[h] * kLn2 + logf(sL[h]) : -INFINITY;
            }
        } else {
            const int slot = first_seg ? 0 : 1;
#pragma unroll 1
            for (int h = 0; h < G; ++h) {
                float *dst = part + (((size_t)cta * 2 + slot) * G + h) * kPartStride(D);
                for (int i = tid; i < D; i += NT) dst[4 + i] = sAcc[h * D + i];
                if (tid == 0) {
                    dst[0] = sM[h];
                    dst[1] = sL[h];
                }
            }
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const unsigned int nseg = (unsigned int)(hi - lo + 1);
                const unsigned int done = atomicAdd(&counters[b * hkv + kh], 1u) + 1u;
                s_last = (done == nseg);
                if (s_last) counters[b * hkv + kh] = 0u;
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                const int slot_lo = (sk_begin(lo, P, W) >= us) ? 0 : 1;
                for (int h = warp; h < G; h += NWARP) {
                    float M = -INFINITY;
                    for (int c2 = lo; c2 <= hi; ++c2) {
                        const int sl = (c2 == lo) ? slot_lo : 0;
                        M = fmaxf(M, __ldcg(part + (((size_t)c2 * 2 + sl) * G + h) * kPartStride(D)));
                    }
                    float v[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) v[r] = 0.f;
                    float l = 0.f;
                    for (int c2 = lo; c2 <= hi; ++c2) {
                        const int sl = (c2 == lo) ? slot_lo : 0;
                        const float *ps = part + (((size_t)c2 * 2 + sl) * G + h) * kPartStride(D);
                        const float m = __ldcg(ps);
                        const float wgt = (m == -INFINITY) ? 0.f : exp2f(m - M);
                        l = fmaf(__ldcg(ps + 1), wgt, l);
#pragma unroll
                        for (int r = 0; r < R; ++r) v[r] = fmaf(__ldcg(ps + 4 + 32 * r + lane), wgt, v[r]);
                    }
                    finish_row<D>(v, l, params, out + out_row(h) * D, lane);
                    if (lse && lane == 0) lse[out_row(h)] = l > 0.f ? M * kLn2 + logf(l) : -INFINITY;
                }
            }
        }
        if (!more_segs) break;
        first_seg = false;
        s = ns;   // its first chunk is already staged in `buf`
    }
}

template <int G>
int warp_ctas_g() {
    int dev = 0, sms = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    constexpr size_t smem = warp_smem_bytes<G>();
    auto kern = decode_warp_kernel<G>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kWWarps * 32, smem) != cudaSuccess) return 0;
    occ = occ < 1 ? 1 : (occ > kCtasPerSm ? kCtasPerSm : occ);
    sms = sms > kMaxSms ? kMaxSms : sms;
    return occ * sms;
}

template <int G>
cudaError_t warp_launch_g(int nctas, cudaStream_t st, const uint8_t *P, int batch, int q_len, int hq, int hkv,
                          const uint8_t *kp, const uint8_t *vp, int64_t nb, const int32_t *bt, int mb,
                          const int32_t *ctx, int ctx_add, int max_ctx, const WsLayout &w, float *out,
                          float *lse, int32_t *status) {
    constexpr size_t smem = warp_smem_bytes<G>();
    auto kern = decode_warp_kernel<G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pass(kern, nctas, kWWarps * 32, smem, st, P, w.packs, batch, q_len, hq, hkv, kp, vp, nb, bt, mb, ctx,
                       ctx_add, max_ctx, w.cpre, w.cta_b, w.part, w.counters, out, lse, status);
}

}  // namespace

int warp_pass_ctas(int G) {
    switch (G) {
        case 1: return warp_ctas_g<1>();
        case 2: return warp_ctas_g<2>();
        case 3: return warp_ctas_g<3>();
        case 4: return warp_ctas_g<4>();
        case 5: return warp_ctas_g<5>();
        case 6: return warp_ctas_g<6>();
        case 7: return warp_ctas_g<7>();
        default: return warp_ctas_g<8>();
    }
}

cudaError_t warp_pass_launch(int G, int nctas, cudaStream_t st, const uint8_t *P, int batch, int q_len, int hq, int hkv,
                             const uint8_t *kp, const uint8_t *vp, int64_t nb, const int32_t *bt, int mb,
                             const int32_t *ctx, int ctx_add, int max_ctx, const WsLayout &w, float *out,
                             float *lse, int32_t *status) {
#define TQ_WPASS(GG) return warp_launch_g<GG>(nctas, st, P, batch, q_len, hq, hkv, kp, vp, nb, bt, mb, ctx, ctx_add, max_ctx, w, out, lse, status)
    switch (G) {
        case 1: TQ_WPASS(1);
        case 2: TQ_WPASS(2);
        case 3: TQ_WPASS(3);
        case 4: TQ_WPASS(4);
        case 5: TQ_WPASS(5);
        case 6: TQ_WPASS(6);
        case 7: TQ_WPASS(7);
        default: TQ_WPASS(8);
    }
#undef TQ_WPASS
}

}  // namespace tq
