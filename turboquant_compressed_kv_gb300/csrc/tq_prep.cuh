// tq_prep.cuh -- the two small kernels that precede the decode pass, as device functions so
// that they can run in one launch: the paged append's encode (tiles of vectors) and the
// query prep (rotation, S projection, operand packs, work schedule).
#pragma once

#include "tq_internal.cuh"

namespace tq {

constexpr int kEncWarps = 4;               // warps per encode CTA

// Where vector v of a launch goes: slot (or -1 to skip) and its input row.
struct SlotMap {
    const int64_t *slots;                  // bulk: slots[token]
    const int32_t *block_table;            // append: slot from the block table and length
    const int32_t *ctx_lens;
    int max_blocks;
    int64_t num_blocks;
    int n_heads;
    int q_len = 1;                         // append: tokens per sequence (token t is number t % q_len of sequence t / q_len)
    __device__ int64_t slot(int64_t token, int32_t *status, bool report) const {
        int64_t s = -1;
        if (slots) {
            s = slots[token];
            if (s < 0) return -1;
        } else {
            const int64_t seq = token / q_len;
            const int L0 = ctx_lens[seq];
            if (L0 < 0) return -1;
            const int Lb = L0 + (int)(token - seq * q_len);
            const int lb = Lb / kBlock;
            const int64_t blk = (lb < max_blocks) ? (int64_t)block_table[(size_t)seq * max_blocks + lb] : -1;
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
    static constexpr size_t kCode = (size_t)TILE * D;
    static constexpr size_t kBytes = kST + kRho + kSgn + kCode;
};


// Encode tiles blk, blk + nblk, ... of TILE vectors (K if is_k, else V) with one CTA of
// 4 warps; `smem` holds EncSmem<D, TILE>::kBytes.  A bad slot is reported by the K tiles
// (or, without K tiles, by the V tiles) when report_bad is set.
template <int D, int TILE, typename T>
__device__ __forceinline__ void encode_tiles(const uint8_t *__restrict__ params, const T *__restrict__ x,
                                             int64_t n_vec, const SlotMap &map, uint8_t *__restrict__ pool, bool is_k,
                                             bool report_bad, int blk, int nblk, uint8_t *smem, int32_t *status) {
    constexpr int R = D / 32;
    constexpr int kTile = TILE, kPerWarp = (TILE + kEncWarps - 1) / kEncWarps;   // tiles below 4 leave warps idle in 1 and 3
    using SM = EncSmem<D, TILE>;
    float *sST = reinterpret_cast<float *>(smem);
    float (*s_rho)[D] = reinterpret_cast<float (*)[D]>(smem + SM::kST);
    uint8_t (*s_sgn)[D] = reinterpret_cast<uint8_t (*)[D]>(smem + SM::kST + SM::kRho);
    uint8_t (*s_code)[D] = reinterpret_cast<uint8_t (*)[D]>(smem + SM::kST + SM::kRho + SM::kSgn);
    __shared__ float s_cent[8], s_thr[8];
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    const float *gST = reinterpret_cast<const float *>(params + params_off_ST(D));
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blk == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    if (threadIdx.x < 8) {
        s_cent[threadIdx.x] = ph->centroid[threadIdx.x];
        s_thr[threadIdx.x] = ph->threshold[threadIdx.x];
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const int64_t ntiles = (n_vec + kTile - 1) / kTile;

#pragma unroll 1
    for (int64_t tile = blk; tile < ntiles; tile += nblk) {
        const int64_t v0 = tile * kTile;
        float nrm[kPerWarp], gam[kPerWarp];
        int64_t slot[kPerWarp];
        // ---- 1. norm, rotation, cells, residual
#pragma unroll
        for (int j = 0; j < kPerWarp; ++j) {
            const int tv = warp + kEncWarps * j;              // vector within the tile
            const bool mine = tv < kTile;                     // warp-uniform
            const int64_t v = v0 + tv;
            float val[R];
            int dims[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {   // the input row does not depend on the slot: load it first
                dims[r] = is_k ? kdim<D>(lane, r) : vdim<D>(lane, r);
                val[r] = (mine && v < n_vec) ? to_f32<T>(x[v * D + dims[r]]) : 0.f;
            }
            // the slot (block-table lookups) is needed only by the stores: a vector without one is
            // encoded from whatever it holds and not stored, so nothing here waits for the lookup
            slot[j] = -1;
            if (mine && v < n_vec)   // a bad slot is reported once per token
                slot[j] = map.slot(v / map.n_heads, status, report_bad && lane == 0 && (v % map.n_heads) == 0);
            // S^T (64 KB at d = 128) is copied once, after the first rows are requested, so that
            // those small loads are not queued behind it; it is waited for before the projection
            if (is_k && SM::kResident && j == 0 && tile == blk) stage_st_rows<D, kEncWarps * 32>(sST, gST, 0, D);
            nrm[j] = 0.f;
            gam[j] = 0.f;
            if (!mine) continue;
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
                s_code[tv][dims[r]] = (uint8_t)k;
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
            constexpr int KPT = D / (kEncWarps * 32);
            float acc[KPT][kTile];
#pragma unroll
            for (int u = 0; u < KPT; ++u)
#pragma unroll
                for (int t = 0; t < kTile; ++t) acc[u][t] = 0.f;
            if (SM::kResident) {
                cp_async_wait_all();
                __syncthreads();
                project_rows<D, kTile, kEncWarps * 32>(sST, 0, D, s_rho, acc);
            } else {
                __syncthreads();
                project_streamed<D, kTile, kEncWarps * 32>(gST, sST, s_rho, acc);
            }
#pragma unroll
            for (int u = 0; u < KPT; ++u)
#pragma unroll
                for (int t = 0; t < kTile; ++t) s_sgn[t][threadIdx.x + 128 * u] = acc[u][t] >= 0.f ? 1 : 0;
            __syncthreads();
        }
        // ---- 3. pack and store (the layout of tq_internal.cuh); a warp packs the vectors it encoded
        __syncwarp();
#pragma unroll
        for (int j = 0; j < kPerWarp; ++j) {
            if (slot[j] < 0) continue;                     // warp-uniform (also for a warp without a vector)
            const int tv = warp + kEncWarps * j;
            const int head = (int)((v0 + tv) % map.n_heads);
            const int64_t blk = slot[j] / kBlock;
            const int off = (int)(slot[j] % kBlock);
            const uint8_t *cd = s_code[tv];
            if (is_k) {
                // 4 D/32 words of 8 fields: word (tig, w) holds columns 2tig, 2tig+1, 2tig+8, 2tig+9 of
                // k-steps 2w (fields 0..3) and 2w+1 (fields 4..7)
                constexpr int NW = D / 32;
                uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * k_record(D);
                const uint8_t *sg = s_sgn[tv];
                const int gid = off & 7, rr = off >> 3;
                for (int wi = lane; wi < 4 * NW; wi += 32) {
                    const int tg = wi / NW, w = wi % NW;
                    uint32_t word = 0;
#pragma unroll
                    for (int f = 0; f < 8; ++f) {
                        const int cs = f & 3, x = 16 * (2 * w + (f >> 2)) + 2 * tg + (cs & 1) + 8 * (cs >> 1);
                        word |= (uint32_t)(cd[x] | (sg[x] << 3)) << (4 * f);
                    }
                    reinterpret_cast<uint32_t *>(rec)[((4 * gid + tg) * 2 + rr) * NW + w] = word;
                }
                if (lane == 0)
                    *reinterpret_cast<__half2 *>(rec + 8 * D + 4 * off) =
                        __halves2half2(__float2half_rn(nrm[j]), __float2half_rn(gam[j]));
            } else {
                // the slot's bytes: per lane gid, group g, word k and half hf, the cells of lane slots
                // 16g + 4k + 2hf + ab (ab = 0, 1: the byte's two fields) with bit k of the cells of lane
                // slots 16g + 12 + 2hf + ab in bit 3 of the fields
                constexpr int NG = D / 128;
                uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * v_record(D);
                const int tg = (off & 7) >> 1, pr = off >> 3, e = off & 1;
                for (int bi = lane; bi < 48 * NG; bi += 32) {
                    const int hf = bi & 1, k = (bi >> 1) % 3, g = ((bi >> 1) / 3) % NG, gid = (bi >> 1) / (3 * NG);
                    uint32_t byte = 0;
#pragma unroll
                    for (int ab = 0; ab < 2; ++ab) {
                        const int sd = 16 * g + 4 * k + 2 * hf + ab, ss = 16 * g + 12 + 2 * hf + ab;
                        const int xd = 16 * (sd >> 1) + gid + 8 * (sd & 1), xs = 16 * (ss >> 1) + gid + 8 * (ss & 1);
                        byte |= (uint32_t)(cd[xd] | (((cd[xs] >> k) & 1) << 3)) << (4 * ab);
                    }
                    rec[((size_t)((4 * gid + tg) * 2 + pr) * 3 * NG + 3 * g + k) * 4 + 2 * hf + e] = (uint8_t)byte;
                }
                if (lane == 0) *reinterpret_cast<__half *>(rec + 6 * D + 2 * off) = __float2half_rn(nrm[j]);
            }
        }
        __syncthreads();   // s_rho / s_sgn are rewritten by the next tile
    }
}


// ---------------------------------------------------------------- f16 operand helpers

// QJL operand of field position i (0..3) of a K record word: bit 4i+3 of each f16 half.
// Positions 3, 7, 11 give 0 or delta_i (2^-21, 2^-17, 2^-13; the first two subnormal, which
// the tensor core keeps); position 15 is the sign bit of 2^-14 (base 0x0400), so that operand
// is -2^-14 sigma.  The B operand is u * qjl_bscale(i), so that every product is
// 2^-16 (u sigma + u) for i < 3 and 2^-16 u sigma for i = 3; the 2^-16 sum of u over the i < 3
// coordinates (delta_i / 2 times the B values) is removed afterwards.
__host__ __device__ constexpr uint32_t qjl_base(int i) { return i == 3 ? 0x04000400u : 0u; }
__host__ __device__ constexpr float qjl_bscale(int i) { return i == 0 ? 64.f : i == 1 ? 4.f : i == 2 ? 0.25f : -0.25f; }
__host__ __device__ constexpr float qjl_half_delta(int i) {
    return i == 0 ? 2.384185791015625e-07f : i == 1 ? 3.814697265625e-06f : i == 2 ? 6.103515625e-05f : 0.f;
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = a b with a zero accumulator.  Long chains of mma.sync accumulation lose precision (the
// tensor core's fp32 accumulation is not rounded to nearest: measured on GB300, 235 ulp of the
// sum after 1024 chained m16n8k16 and 1439 after 4096), so sums over many tokens start each
// block from zero and are added up with FADD.
__device__ __forceinline__ void mma_f16_z(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// Per (sequence, kv head) query pack: f16x2 B-operand fragments
// [2 (qbar / alpha, QJL-scaled u)][d/16 k-steps][n-tiles][32 lanes][2 words], then floats:
// [8] unused, [8 heads] the QJL offset constant.
__host__ __device__ constexpr size_t kPackBytes(int d) { return 64 * (size_t)d + 256; }
__host__ __device__ constexpr int kPackFloatOff(int d) { return 16 * d; }   // in floats

// ---------------------------------------------------------------- (1) query prep
// A CTA handles kQRows (sequence, query head) rows, one per warp: each warp
// rotates its row (qbar = Pi q), then thread k computes u_k = (S qbar)_k for
// every row from S^T staged in shared memory (all of it in one copy at d=128,
// two 64-row chunks in flight at d=256), then each warp writes its row's hi
// and lo columns (2*hg, 2*hg+1) of the K-side B operand for qbar (qu=0) and
// u (qu=1) into the pack of the row's (sequence, kv head), and the offset
// constants.  The pass's work schedule (build_schedule) is laid out by a CTA of its own, in
// parallel with the rows.
constexpr int kQRows = 4;
template <int D> __host__ __device__ constexpr int qprep_st_rows() { return D == 128 ? 128 : 64; }
template <int D> __host__ __device__ constexpr size_t qprep_smem() {
    return (size_t)2 * kQRows * D * 4 + (size_t)(D / qprep_st_rows<D>() > 1 ? 2 : 1) * qprep_st_rows<D>() * D * 4;
}


// Rows 4*blk .. 4*blk+3 of the query prep, one CTA of 128 threads; `qsm` holds
// qprep_smem<D>() bytes.  ctx_add is added to every non-negative length (the number of tokens the
// step appends first).  With q_len > 1
// queries per sequence (q[b][i][h]), query i of head hg of a kv head is operand column
// i * G + hg of the kv head's pack.
template <int D, int NTK, typename T>
__device__ __forceinline__ void qprep_rows(const uint8_t *__restrict__ params, const T *__restrict__ q, int batch,
                                           int q_len, int hq, int hkv, const int32_t *__restrict__ ctx_lens,
                                           int ctx_add, int max_ctx, int chunk, int P, uint8_t *__restrict__ packs,
                                           unsigned int *__restrict__ counters, int64_t *__restrict__ cpre,
                                           int32_t *__restrict__ cta_b, int blk, uint8_t *qsm) {
    constexpr int R = D / 32, NKS = D / 16, KPT = D / 128;
    float (*qs)[D] = reinterpret_cast<float (*)[D]>(qsm);                       // [kQRows][D] qbar
    float (*us)[D] = reinterpret_cast<float (*)[D]>(qsm + kQRows * D * 4);      // [kQRows][D] u
    float *sbuf = reinterpret_cast<float *>(qsm + 2 * kQRows * D * 4);         // S^T rows
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrows = batch * q_len * hq, row0 = blk * kQRows;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const float *ST = reinterpret_cast<const float *>(params + params_off_ST(D));
    const float inv_sd = rsqrtf((float)D);
    constexpr bool kOneCopy = qprep_st_rows<D>() == D;
    {
        const int row = row0 + warp;
        float v[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            v[r] = (row < nrows) ? to_f32<T>(q[(size_t)row * D + 32 * r + lane]) * __ldg(Dsign + 32 * r + lane) : 0.f;
        // S^T (64 KB at d = 128) is requested after the rows, so they are not queued behind it; it
        // arrives while the rows rotate
        if constexpr (kOneCopy) stage_st_rows<D, 128>(sbuf, ST, 0, D);
        fwht_warp<R>(v, lane);
#pragma unroll
        for (int r = 0; r < R; ++r) qs[warp][32 * r + lane] = v[r] * inv_sd;   // qbar = H D q / sqrt d
    }
    {
        float acc[KPT][kQRows];
#pragma unroll
        for (int u = 0; u < KPT; ++u)
#pragma unroll
            for (int rr = 0; rr < kQRows; ++rr) acc[u][rr] = 0.f;
        if constexpr (kOneCopy) {                                              // u = S qbar
            cp_async_wait_all();
            __syncthreads();
            project_rows<D, kQRows, 128>(sbuf, 0, D, qs, acc);
        } else {
            project_streamed<D, kQRows, 128, qprep_st_rows<D>()>(ST, sbuf, qs, acc);
        }
#pragma unroll
        for (int u = 0; u < KPT; ++u)
#pragma unroll
            for (int rr = 0; rr < kQRows; ++rr) us[rr][threadIdx.x + 128 * u] = acc[u][rr];
    }
    __syncthreads();
    const int row = row0 + warp;
    if (row < nrows) {
        const int b = row / (hq * q_len), qi = (row / hq) % q_len, h = row % hq, G = hq / hkv, kvh = h / G;
        const int hg = qi * G + h % G;                            // operand column of this query row
        const int GQ = G * q_len;
        if (hg == 0 && lane == 0) counters[b * hkv + kvh] = 0u;   // completion counter of the pass
        float v[R], u[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            v[r] = qs[warp][32 * r + lane];
            u[r] = us[warp][32 * r + lane];
        }
        uint8_t *pack = packs + ((size_t)b * hkv + kvh) * kPackBytes(D);
        uint16_t *ph = reinterpret_cast<uint16_t *>(pack);
        float *pf = reinterpret_cast<float *>(pack) + kPackFloatOff(D);
        const float inv_alpha = reinterpret_cast<const ParamsHeader *>(params)->inv_alpha;
#pragma unroll
        for (int qu = 0; qu < 2; ++qu) {
            float cs = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int dim = 32 * r + lane;
                // operand row (k-step s, row k) of the coordinate, and its B value
                int s = dim >> 4, k = dim & 15;
                float beta = v[r] * inv_alpha;             // codebook plane: natural order, qbar / alpha
                float hd = 0.f;
                if (qu == 1) {                              // QJL plane: the K record's field position
                    const int c = dim & 15, tg = (c & 7) >> 1, h = c >> 3;
                    const int f = 4 * (s & 1) + (c & 1) + 2 * h, i = f & 3;
                    k = 2 * tg + 8 * (i & 1) + (f >> 2);
                    s = 2 * (s >> 1) + (i >> 1);
                    beta = u[r] * qjl_bscale(i);
                    hd = qjl_half_delta(i);
                }
                const __half hi = __float2half_rn(beta);
                const __half lo = __float2half_rn(beta - __half2float(hi));
                cs = fmaf(__half2float(hi) + __half2float(lo), hd, cs);
                const int reg = k >> 3, tig = (k & 7) >> 1, e = k & 1;
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int col = 2 * hg + x, nt = col >> 3, gid = col & 7;
                    const size_t word = ((size_t)(qu * NKS + s) * NTK + nt) * 64 + (4 * gid + tig) * 2 + reg;
                    ph[word * 2 + e] = __half_as_ushort(x == 0 ? hi : lo);
                }
            }
            if (qu == 1) {
                cs = warp_sum(cs);
                if (lane == 0) pf[8 + hg] = cs;
            }
        }
        // columns beyond the group's 2*G*q_len are zero (written by the group's first row)
        if (hg == 0) {
            uint32_t *pw = reinterpret_cast<uint32_t *>(pack);
            for (int col = 2 * GQ; col < 8 * NTK; ++col) {
                const int nt = col >> 3, gid = col & 7;
                for (int i = lane; i < 2 * NKS * 8; i += 32) {
                    const int qu = i / (NKS * 8), s = (i / 8) % NKS, k = i % 8;
                    pw[((size_t)(qu * NKS + s) * NTK + nt) * 64 + (4 * gid + (k >> 1)) * 2 + (k & 1)] = 0u;
                }
            }
        }
    }
}


}  // namespace tq
