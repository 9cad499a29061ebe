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
// At d = 128 both have one-thread-per-row paths with the rotation in registers (below): K on
// tcgen05, where S^T b for 128 vectors is one 128 x 128 x 128 product, and V.
#include "tq_internal.cuh"
#include "tq_tc.cuh"

#ifndef TQ_DEQUANT_TC
#define TQ_DEQUANT_TC 1          // d = 128: K through the tcgen05 path, V through the row-per-thread path
#endif

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
            const uint32_t *words = reinterpret_cast<const uint32_t *>(rec);
            if (is_k) {
                // field of coordinate x: bits 4f .. 4f+3 of word (L * 2 + row) * d/32 + ks / 2
                constexpr int NW = D / 32;
                const int gid = t & 7, th = t >> 3;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int x = dims[r], ks = x >> 4, c = x & 15;
                    const int f = 4 * (ks & 1) + (c & 1) + 2 * (c >> 3);
                    const uint32_t nib = (words[((4 * gid + ((c & 7) >> 1)) * 2 + th) * NW + (ks >> 1)] >> (4 * f)) & 15u;
                    val[jj][r] = s_cent[nib & 7u] * inv_sd;
                    s_b[t][x] = (nib & 8u) ? 1.f : -1.f;
                }
                const __half2 ng = *reinterpret_cast<const __half2 *>(rec + 8 * D + 4 * t);
                nrm[jj] = __low2float(ng);
                gam[jj] = __high2float(ng);
            } else {
                // lane slot s = 2 mt + rr of coordinate x, groups of 16 slots: 12 fields, then 4 cells kept
                // in bit 3 of the fields of the group's three words
                constexpr int NG = D / 128;
                const int tigv = (t & 7) >> 1, pr = t >> 3, e = t & 1;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int x = dims[r], sl = 2 * (x >> 4) + ((x >> 3) & 1), g = sl >> 4, sg = sl & 15;
                    const int base = ((4 * (x & 7) + tigv) * 2 + pr) * 3 * NG + 3 * g;
                    int c;
                    if (sg < 12) {
                        const int f = 4 * ((sg >> 1) & 1) + 2 * e + (sg & 1);
                        c = (int)((words[base + (sg >> 2)] >> (4 * f)) & 7u);
                    } else {
                        const int f = 4 * ((sg - 12) >> 1) + 2 * e + (sg & 1);
                        c = 0;
#pragma unroll
                        for (int q = 0; q < 3; ++q) c |= (int)((words[base + q] >> (4 * f + 3)) & 1u) << q;
                    }
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

// ---------------------------------------------------------------- K at d = 128 on tcgen05
// kWg warpgroups take alternate tiles of 128 rows (8 records x 16 slots); thread r of a
// warpgroup owns row r:
//  1. the tile's records arrive by bulk copy (two tiles in flight per warpgroup), one record per
//     lane of the warpgroup's second warp, so that the copies leave together and the thread that
//     issues the MMA does nothing else;
//  2. the row's 128 sign bits become the A operand (f16 +-1, 128-byte swizzle) with one shift
//     and one LOP3 per two elements: K index 32 tig + 8 w + 2 p + e holds the sign bit of field
//     p + 4 e of the slot's word (tig, w), bit 4 (p + 4 e) + 3;
//  3. one thread issues p = S^T b with S as one f16 operand (S is held at binary16 precision;
//     B rows = output coordinates, K-major, 8
//     f16 MMAs of K = 16) into the warpgroup's 128 tensor-memory columns;
//  4. the thread reads its row back (tcgen05.ld), adds the codebook values, runs the 128-point
//     inverse transform in registers, and stores the row.
namespace dq128 {
#ifndef TQ_DQ128K_WG
#define TQ_DQ128K_WG 2           // warpgroups per CTA (they share S in shared memory; 3 measured slower)
#endif
constexpr int D = 128, kRows = 128, kUnits = kRows / kBlock, kWg = TQ_DQ128K_WG, kThreads = 128 * kWg;
constexpr int kRec = (int)k_record(D);
constexpr int oB = 0;          // S as f16 (exact: S is held at binary16 precision): 32 KB
constexpr int oA = 32768;      // A operand of each warpgroup: kWg x 32 KB
constexpr int oR = oA + kWg * 32768;   // records: [warpgroup][buffer][unit][kRec]
constexpr int kSmem = oR + kWg * 2 * kUnits * kRec;
}  // namespace dq128

template <typename TO>
__global__ void __launch_bounds__(dq128::kThreads, 1)
dequant128k_tc_kernel(const uint8_t *__restrict__ params, const uint8_t *__restrict__ pool, int64_t num_blocks,
                      int n_heads, const int32_t *__restrict__ block_ids, int n_ids, TO *__restrict__ out,
                      int32_t *status) {
    using namespace dq128;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t recbar[kWg][2], mmabar[kWg];
    __shared__ uint32_t tmem_base;
    __shared__ __align__(16) float s_D[D];
    __shared__ __align__(16) uint32_t s_dsg[D / 2];   // bf16 pair sign masks of D (bit 15 / 31: D_2j / D_2j+1 < 0)
    // centroid pairs (x 1/sqrt d) of two fields, by a record byte masked to its cell bits (0x77):
    // entry i holds c[i & 7], c[i >> 4]; one copy per lane ([index][lane]), so that a half-warp's
    // lookups never share a bank
    __shared__ float2 s_pair[128][32];
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const int tid = threadIdx.x, wg = tid >> 7, row = tid & 127, warp = tid >> 5;
    const int64_t units = (int64_t)n_ids * n_heads, ntiles = (units + kUnits - 1) / kUnits;
    if ((int64_t)blockIdx.x >= ntiles) return;
    if (tid == 0) {
        for (int i = 0; i < kWg; ++i) {
            tc::mbar_init(&recbar[i][0], 1);
            tc::mbar_init(&recbar[i][1], 1);
            tc::mbar_init(&mmabar[i], 1);
        }
    }
    constexpr uint32_t kTmemCols = kWg <= 2 ? 256 : 512;   // 128 columns per warpgroup, a power of two
    if (warp == 0) tc::tmem_alloc(&tmem_base, kTmemCols);
    for (int e = tid; e < 128 * 32; e += kThreads) {
        const int i = e >> 5;
        const float isd = rsqrtf((float)D);
        s_pair[i][e & 31] = make_float2(ph->centroid[i & 7] * isd, ph->centroid[(i >> 4) & 7] * isd);
    }
    if (tid < D) s_D[tid] = reinterpret_cast<const float *>(params + params_off_D(D))[tid];
    if (tid < D / 2) {
        const float *Dp = reinterpret_cast<const float *>(params + params_off_D(D));
        s_dsg[tid] = (Dp[2 * tid] < 0.f ? 0x8000u : 0u) | (Dp[2 * tid + 1] < 0.f ? 0x80000000u : 0u);
    }
    {   // B: row n = output coordinate n, K index k' as in the A operand; S as f16 (exact)
        const float *S = reinterpret_cast<const float *>(params + params_off_S(D));
        for (int e = tid; e < D * D; e += kThreads) {
            const int n = e >> 7, k = e & 127;
            const int tig = k >> 5, w = (k >> 3) & 3, f = ((k >> 1) & 3) + 4 * (k & 1);
            const int coord = 16 * (2 * w + (f >> 2)) + 2 * tig + (f & 1) + 8 * ((f >> 1) & 1);
            // S is held at binary16 precision: one exact f16 operand
            *reinterpret_cast<__half *>(smem + oB + tc::sw128_off(n, k, D)) = __float2half_rn(__ldg(S + coord * D + n));
        }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base + 128u * wg;
    const float inv_sd = rsqrtf((float)D);
    const float qjl = 1.2533141373155003f / (float)D;   // sqrt(pi/2) / d
    bool timed_out = false;

    // tiles of this warpgroup: blockIdx.x + (2 i + wg) * gridDim.x
    auto tile_of = [&](int i) { return (int64_t)blockIdx.x + (int64_t)(kWg * i + wg) * gridDim.x; };
    // Warp 1 of the warpgroup moves the records, lane k < kUnits the record of unit k, while row 0
    // (warp 0) issues the MMA.  A lane reads its block id one tile before the copy that uses it.
    const int lane = tid & 31;
    const bool mover = (warp & 3) == 1;
    auto load_id = [&](int i) -> int32_t {
        const int64_t u = tile_of(i) * kUnits + lane;
        return (lane < kUnits && u < units) ? block_ids[u / n_heads] : 0;
    };
    auto issue = [&](int i, int buf, int32_t id) {   // warp 1: tile i's records into buffer buf
        const int64_t left = units - tile_of(i) * kUnits;
        const int n = left < kUnits ? (int)left : kUnits;
        if (lane == 0) tc::mbar_arrive_expect_tx(&recbar[wg][buf], (uint32_t)(n * kRec));
        __syncwarp();
        if (lane < n) {
            const int64_t u = tile_of(i) * kUnits + lane;
            const int64_t bc = (id >= 0 && id < num_blocks) ? id : 0;   // a bad id reads block 0, output zeroed
            tc::bulk_g2s(smem + oR + ((wg * 2 + buf) * kUnits + lane) * kRec,
                         pool + ((size_t)bc * n_heads + (u % n_heads)) * kRec, kRec, &recbar[wg][buf]);
        }
    };
    int32_t nid = 0;   // warp 1: this lane's block id of the tile two ahead
    if (mover) {
        if (tile_of(0) < ntiles) issue(0, 0, load_id(0));
        if (tile_of(1) < ntiles) issue(1, 1, load_id(1));
    }
    uint8_t *sA = smem + oA + wg * 32768;
    const int bar_id = 1 + wg;   // named barrier of this warpgroup's 128 threads

#pragma unroll 1
    for (int i = 0; tile_of(i) < ntiles; ++i) {
        const int64_t tile = tile_of(i);
        const int buf = i & 1;
        if (mover && tile_of(i + 2) < ntiles) nid = load_id(i + 2);
        if (!tc::mbar_wait(&recbar[wg][buf], (i >> 1) & 1)) timed_out = true;
        // row 32 q + l holds slot (l >> 2) + 8 (bit 1 of l) of unit 2 q + (l & 1): a quarter-warp's
        // record reads fall on 4 different 16-byte bank groups (units are 1088 bytes apart), where
        // a unit per 16 rows put 8 lanes on one group
        const int lq = row & 31, unit_k = 2 * (row >> 5) + (lq & 1), t = (lq >> 2) + 8 * ((lq >> 1) & 1);
        const int64_t u = tile * kUnits + unit_k;
        const bool live = u < units;
        const int64_t blk = live ? block_ids[u / n_heads] : -1;   // checked at the store
        const uint8_t *rec = smem + oR + ((wg * 2 + buf) * kUnits + unit_k) * kRec;
        const int gid = t & 7, th = t >> 3;
        uint32_t kw[4][4];   // the slot's words [tig][w]
#pragma unroll
        for (int tig = 0; tig < 4; ++tig) {
            const uint4 v = live ? reinterpret_cast<const uint4 *>(rec)[(4 * gid + tig) * 2 + th] : make_uint4(0u, 0u, 0u, 0u);
            kw[tig][0] = v.x;
            kw[tig][1] = v.y;
            kw[tig][2] = v.z;
            kw[tig][3] = v.w;
        }
        const __half2 ng = live ? *reinterpret_cast<const __half2 *>(rec + 8 * D + 4 * t) : __floats2half2_rn(0.f, 0.f);
        const float nrm = __low2float(ng), gam = __high2float(ng);
        // A operand: 16-byte chunks of 8 K elements (four f16x2 registers)
#pragma unroll
        for (int tig = 0; tig < 4; ++tig)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r4[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) r4[q] = ((kw[tig][c] << (12 - 4 * q)) & 0x80008000u) ^ 0xBC00BC00u;
                *reinterpret_cast<uint4 *>(sA + tc::sw128_off(row, 32 * tig + 8 * c, kRows)) =
                    make_uint4(r4[0], r4[1], r4[2], r4[3]);
            }
        tc::fence_async_smem();
        tc::fence_before_sync();
        tc::named_sync(bar_id, 128);   // A built, the records read: the buffer can be refilled
        tc::fence_after_sync();
        if (row == 0) {
            const uint32_t bh = tc::smem_u32(smem + oB), a = tc::smem_u32(sA);
            constexpr uint32_t id = tc::idesc_f16(kRows, D);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                tc::mma_ss_f16(tmem, tc::sw128_desc(a, ks, kRows), tc::sw128_desc(bh, ks, D), id, ks > 0);
            tc::mma_commit(&mmabar[wg]);
        }
        if (mover && tile_of(i + 2) < ntiles) issue(i + 2, buf, nid);
        if (!tc::mbar_wait(&mmabar[wg], i & 1)) timed_out = true;
        tc::fence_after_sync();
        // y = c[cell] / sqrt d + sqrt(pi/2)/d gamma p on pairs Y[j] = (y_2j, y_2j+1): coordinate n in
        // column n
        float2 Y[D / 2];
        const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        {
            uint32_t pv[D / 16][16];   // the eight loads share one wait
#pragma unroll
            for (int j = 0; j < D / 16; ++j) tc::ld16_raw(taddr + 16 * j, pv[j]);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < D / 16; ++j)
#pragma unroll
                for (int x = 0; x < 16; ++x) tc::reg_fence(pv[j][x]);
#pragma unroll
            for (int j = 0; j < D / 16; ++j)
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    Y[8 * j + x] = make_float2(__uint_as_float(pv[j][2 * x]), __uint_as_float(pv[j][2 * x + 1]));
        }
        tc::fence_before_sync();
        const float gq = qjl * gam;
        const float2 gq2 = make_float2(gq, gq);
        // byte q of word (tig, w) holds fields 2q, 2q + 1: coordinates x and x + 1 with
        // x = 16 (2 w + (q >> 1)) + 2 tig + 8 (q & 1); one table lookup per byte
#pragma unroll
        for (int tig = 0; tig < 4; ++tig)
#pragma unroll
            for (int w = 0; w < 4; ++w)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 cc = s_pair[(kw[tig][w] >> (8 * q)) & 0x77u][tid & 31];
                    const int x = 16 * (2 * w + (q >> 1)) + 2 * tig + 8 * (q & 1);
                    Y[x >> 1] = __ffma2_rn(gq2, Y[x >> 1], cc);
                }
        // inverse rotation D (H y) / sqrt d: the stage on index bit 0 inside the pairs, bits 1..6
        // between them (f32x2)
#pragma unroll
        for (int j = 0; j < D / 2; ++j) Y[j] = make_float2(Y[j].x + Y[j].y, Y[j].x - Y[j].y);
        {
            const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int st = 1; st < D / 2; st <<= 1)
#pragma unroll
                for (int j = 0; j < D / 2; ++j)
                    if ((j & st) == 0) {
                        const float2 a = Y[j], b = Y[j | st];
                        Y[j] = __fadd2_rn(a, b);
                        Y[j | st] = __ffma2_rn(b, m1, a);   // a - b
                    }
        }
        const bool good = live && blk >= 0 && blk < num_blocks;
        if (live && !good && t == 0) flag_status(status, TQ_STATUS_BAD_SLOT);
        const float sc = good ? nrm * inv_sd : 0.f;
        const float2 sc2 = make_float2(sc, sc);
        if constexpr (sizeof(TO) == 4) {
            if (live) {
                TO *orow = out + (((size_t)(u / n_heads) * kBlock + t) * n_heads + (u % n_heads)) * D;
#pragma unroll
                for (int n = 0; n < D; n += 8) {
                    float2 o[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) o[x] = __fmul2_rn(Y[n / 2 + x], sc2);
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const float4 dv = *reinterpret_cast<const float4 *>(&s_D[n + 4 * x]);
                        *reinterpret_cast<float4 *>(orow + n + 4 * x) =
                            make_float4(o[2 * x].x * dv.x, o[2 * x].y * dv.y, o[2 * x + 1].x * dv.z, o[2 * x + 1].y * dv.w);
                    }
                }
            }
        } else {
            // bf16, the signs D by an XOR of the packed words.  The row (256 bytes) goes to its own
            // bytes of the A operand, free once the MMA has completed (16-byte chunk c to half c >> 3,
            // position (c & 7) ^ (row & 7)); then each store of the warp writes two whole rows.
#pragma unroll
            for (int n = 0; n < D; n += 8) {
                float2 o[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) o[x] = __fmul2_rn(Y[n / 2 + x], sc2);
                const uint4 sm = *reinterpret_cast<const uint4 *>(&s_dsg[n / 2]);
                const uint32_t smw[4] = {sm.x, sm.y, sm.z, sm.w};
                uint32_t pk[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const __nv_bfloat162 b = __floats2bfloat162_rn(o[x].x, o[x].y);
                    pk[x] = *reinterpret_cast<const uint32_t *>(&b) ^ smw[x];
                }
                const int c = n >> 3;
                *reinterpret_cast<uint4 *>(sA + (c >> 3) * (kRows * 128) + row * 128 + (((c & 7) ^ (row & 7)) << 4)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            __syncwarp();
            // store j: lanes 0..15 write slot j of the warp's first unit, lanes 16..31 of its second
            // (rows 32 q + 4 (j & 7) + 2 (j >> 3) + e, e = lane >> 4), chunk lane & 15 each
            const int e = lane >> 4, c = lane & 15;
            const int64_t ue = tile * kUnits + 2 * (warp & 3) + e;
            if (ue < units) {
                TO *obase = out + (((size_t)(ue / n_heads) * kBlock) * n_heads + (ue % n_heads)) * D + 8 * c;
#pragma unroll
                for (int j = 0; j < kBlock; ++j) {
                    const int r = 32 * (warp & 3) + 4 * (j & 7) + 2 * (j >> 3) + e;
                    const uint4 v = *reinterpret_cast<const uint4 *>(sA + (c >> 3) * (kRows * 128) + r * 128 +
                                                                     (((c & 7) ^ (r & 7)) << 4));
                    *reinterpret_cast<uint4 *>(obase + (size_t)j * n_heads * D) = v;
                }
            }
        }
        tc::named_sync(bar_id, 128);   // every row of the accumulator is read before the next MMA
        tc::fence_after_sync();
    }
    if (timed_out) flag_status(status, TQ_STATUS_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------- V at d = 128, one thread per row
// A CTA of 128 threads walks tiles of 8 records (128 rows); thread r owns row r:
//  1. the tile's records arrive by bulk copy, two tiles in flight, one record per lane of warp 0,
//     which also leaves the records' block ids in shared memory for the rows' stores;
//  2. the row's cells are read back word by word (each V byte holds two cells of one slot and one
//     bit of two more), y = c[cell] / sqrt d by one table lookup per byte;
//  3. the 128-point inverse transform in registers, the norm and D, and 16-byte stores.
namespace dq128v {
constexpr int D = 128, kRows = 128, kUnits = kRows / kBlock, kThreads = 128, kMinCtas = 3;
constexpr int kRec = (int)v_record(D);
constexpr int oStage = 2 * kUnits * kRec;                 // records: two buffers of 8
constexpr int kSmem = oStage + (kThreads / 32) * 32 * 256;   // bf16 rows of each warp, staged for the stores
}  // namespace dq128v

template <typename TO>
__global__ void __launch_bounds__(dq128v::kThreads, dq128v::kMinCtas)
dequant128v_rows_kernel(const uint8_t *__restrict__ params, const uint8_t *__restrict__ pool, int64_t num_blocks,
                        int n_heads, const int32_t *__restrict__ block_ids, int n_ids, TO *__restrict__ out,
                        int32_t *status) {
    using namespace dq128v;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint64_t recbar[2], recfree[2];
    __shared__ int32_t s_ids[2][kUnits];   // block ids of the records in each buffer
    __shared__ __align__(16) float s_D[D];
    __shared__ __align__(16) uint32_t s_dsg[D / 2];   // bf16 pair sign masks of D (bit 15 / 31: D_2j / D_2j+1 < 0)
    // centroid pairs (x 1/sqrt d) of two fields, by a record byte masked to its cell bits (0x77):
    // entry i holds c[i & 7], c[i >> 4]; one copy per lane of a half-warp ([index][lane & 15]): an
    // 8-byte load is served a half-warp at a time, so its lookups never share a bank
    __shared__ float2 s_pair[128][16];
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const int row = threadIdx.x;
    const int64_t units = (int64_t)n_ids * n_heads, ntiles = (units + kUnits - 1) / kUnits;
    if ((int64_t)blockIdx.x >= ntiles) return;
    if (row == 0) {
        tc::mbar_init(&recbar[0], 1);
        tc::mbar_init(&recbar[1], 1);
        tc::mbar_init(&recfree[0], kThreads / 32);   // one arrival per warp once its rows are read
        tc::mbar_init(&recfree[1], kThreads / 32);
    }
    const float inv_sd = rsqrtf((float)D);
    for (int e = row; e < 128 * 16; e += kThreads) {
        const int i = e >> 4;
        s_pair[i][e & 15] = make_float2(ph->centroid[i & 7] * inv_sd, ph->centroid[(i >> 4) & 7] * inv_sd);
    }
    const int lane = row & 31;
    s_D[row] = reinterpret_cast<const float *>(params + params_off_D(D))[row];
    if (row < D / 2) {
        const float *Dp = reinterpret_cast<const float *>(params + params_off_D(D));
        s_dsg[row] = (Dp[2 * row] < 0.f ? 0x8000u : 0u) | (Dp[2 * row + 1] < 0.f ? 0x80000000u : 0u);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    bool timed_out = false;
    auto tile_of = [&](int i) { return (int64_t)blockIdx.x + (int64_t)i * gridDim.x; };
    // Warp 0 moves the records: lane k < kUnits reads the block id of unit k one tile ahead and
    // copies that unit's record.
    auto load_id = [&](int i) -> int32_t {
        const int64_t u = tile_of(i) * kUnits + lane;
        return (lane < kUnits && u < units) ? block_ids[u / n_heads] : 0;
    };
    auto issue = [&](int i, int buf, int32_t id) {   // warp 0: tile i's records into buffer buf
        const int64_t left = units - tile_of(i) * kUnits;
        const int n = left < kUnits ? (int)left : kUnits;
        if (lane < kUnits) s_ids[buf][lane] = id;   // for the rows' stores, visible once the buffer is full
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_expect_tx(&recbar[buf], (uint32_t)(n * kRec));
        if (lane < n) {
            const int64_t u = tile_of(i) * kUnits + lane;
            const int64_t bc = (id >= 0 && id < num_blocks) ? id : 0;   // a bad id reads block 0, output zeroed
            tc::bulk_g2s(smem + (buf * kUnits + lane) * kRec, pool + ((size_t)bc * n_heads + (u % n_heads)) * kRec,
                         kRec, &recbar[buf]);
        }
    };
    const bool mover = row < 32;
    int32_t nid = 0;   // warp 0: this lane's block id of the tile two ahead
    if (mover) {
        if (tile_of(0) < ntiles) issue(0, 0, load_id(0));
        if (tile_of(1) < ntiles) issue(1, 1, load_id(1));
    }

#pragma unroll 1
    for (int i = 0; tile_of(i) < ntiles; ++i) {
        const int64_t tile = tile_of(i);
        const int buf = i & 1;
        if (mover && tile_of(i + 2) < ntiles) nid = load_id(i + 2);
        if (!tc::mbar_wait(&recbar[buf], (i >> 1) & 1)) timed_out = true;
        const int unit_k = row >> 4, t = row & 15;
        const int64_t u = tile * kUnits + unit_k;
        const bool live = u < units;
        const int64_t blk = live ? s_ids[buf][unit_k] : -1;   // checked at the store
        const uint8_t *rec = smem + (buf * kUnits + unit_k) * kRec;
        const uint32_t *words = reinterpret_cast<const uint32_t *>(rec);
        // the slot's bytes: per lane gid, words 3 (L * 2 + pair) + k (k = 0..2), bytes 2 hf + e.
        // Byte (k, hf) holds the cells of lane slots 4k + 2hf + ab (ab = 0, 1: coordinates
        // 16 (2k + hf) + gid + 8 ab) in bits 4ab .. 4ab + 2, and in bit 4ab + 3 bit k of the cell of
        // lane slot 12 + 2hf + ab (coordinate 16 (6 + hf) + gid + 8 ab)
        const int a = (t & 7) >> 1, pr = t >> 3, e = t & 1;
        // pairs P[8 m + g] = (y_{16 m + g}, y_{16 m + g + 8}): one table lookup fills one pair
        float2 P[D / 2];
#pragma unroll
        for (int gid = 0; gid < 8; ++gid) {
            uint32_t bt[3][2];
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const uint32_t w = words[((4 * gid + a) * 2 + pr) * 3 + k];
                bt[k][0] = (w >> (8 * e)) & 0xFFu;
                bt[k][1] = (w >> (16 + 8 * e)) & 0xFFu;
            }
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                for (int k = 0; k < 3; ++k) P[8 * (2 * k + hf) + gid] = s_pair[bt[k][hf] & 0x77u][lane & 15];
                // bit 3 (ab = 0) and bit 7 (ab = 1) of the three bytes: the cells of slots 12 + 2hf + ab
                const uint32_t sp = ((bt[0][hf] >> 3) & 0x11u) | ((bt[1][hf] >> 2) & 0x22u) | ((bt[2][hf] >> 1) & 0x44u);
                P[8 * (6 + hf) + gid] = s_pair[sp][lane & 15];
            }
        }
        const __half nh = *reinterpret_cast<const __half *>(rec + 6 * D + 2 * t);
        tc::fence_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&recfree[buf]);   // this warp's rows of the buffer are read
        // warp 0 refills the buffer with the tile two ahead once every warp has read it (after
        // this tile's work, when they are long done; nobody else waits)
        auto refill = [&]() {
            if (mover && tile_of(i + 2) < ntiles) {
                if (!tc::mbar_wait(&recfree[buf], (i >> 1) & 1)) timed_out = true;
                issue(i + 2, buf, nid);
            }
        };
        // inverse rotation D (H y) / sqrt d: index bit 3 inside the pairs; bits 0..2 and 4..6 between
        // them (pair index bits 0..2 and 3..5), on f32x2
#pragma unroll
        for (int j = 0; j < D / 2; ++j) P[j] = make_float2(P[j].x + P[j].y, P[j].x - P[j].y);
        {
            const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int st = 1; st < D / 2; st <<= 1)
#pragma unroll
                for (int j = 0; j < D / 2; ++j)
                    if ((j & st) == 0) {
                        const float2 a2 = P[j], b2 = P[j | st];
                        P[j] = __fadd2_rn(a2, b2);
                        P[j | st] = __ffma2_rn(b2, m1, a2);   // a - b
                    }
        }
        const bool good = live && blk >= 0 && blk < num_blocks;
        if (live && !good && t == 0) flag_status(status, TQ_STATUS_BAD_SLOT);
        const float sc = good ? __half2float(nh) * inv_sd : 0.f;
        const float2 sc2 = make_float2(sc, sc);
        // coordinate n is component (n >> 3) & 1 of pair 8 (n >> 4) + (n & 7)
        auto yv = [&](int n) -> float { return ((n >> 3) & 1) ? P[8 * (n >> 4) + (n & 7)].y : P[8 * (n >> 4) + (n & 7)].x; };
        if constexpr (sizeof(TO) == 4) {
            if (live) {
                TO *orow = out + (((size_t)(u / n_heads) * kBlock + t) * n_heads + (u % n_heads)) * D;
#pragma unroll
                for (int n = 0; n < D; n += 8) {
                    float2 o[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) o[x] = __fmul2_rn(make_float2(yv(n + 2 * x), yv(n + 2 * x + 1)), sc2);
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const float4 dv = *reinterpret_cast<const float4 *>(&s_D[n + 4 * x]);
                        *reinterpret_cast<float4 *>(orow + n + 4 * x) =
                            make_float4(o[2 * x].x * dv.x, o[2 * x].y * dv.y, o[2 * x + 1].x * dv.z, o[2 * x + 1].y * dv.w);
                    }
                }
            }
        } else {
            // bf16, the signs D by an XOR of the packed words.  The row (256 bytes) goes to the
            // warp's staging area (16-byte chunk c at position c ^ (row & 15)); then each store of
            // the warp writes two whole rows.
            uint8_t *stg = smem + oStage + (row >> 5) * (32 * 256);
#pragma unroll
            for (int n = 0; n < D; n += 8) {
                float2 o[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) o[x] = __fmul2_rn(make_float2(yv(n + 2 * x), yv(n + 2 * x + 1)), sc2);
                const uint4 sm = *reinterpret_cast<const uint4 *>(&s_dsg[n / 2]);
                const uint32_t smw[4] = {sm.x, sm.y, sm.z, sm.w};
                uint32_t pk[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const __nv_bfloat162 b = __floats2bfloat162_rn(o[x].x, o[x].y);
                    pk[x] = *reinterpret_cast<const uint32_t *>(&b) ^ smw[x];
                }
                *reinterpret_cast<uint4 *>(stg + lane * 256 + (((n >> 3) ^ (lane & 15)) << 4)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            __syncwarp();
            // store j: lanes 0..15 write slot j of the warp's first unit (its lane j), lanes 16..31
            // of its second (lane 16 + j), chunk lane & 15 each
            const int e = lane >> 4, c = lane & 15;
            const int64_t ue = tile * kUnits + 2 * (row >> 5) + e;
            if (ue < units) {
                TO *obase = out + (((size_t)(ue / n_heads) * kBlock) * n_heads + (ue % n_heads)) * D + 8 * c;
#pragma unroll
                for (int j = 0; j < kBlock; ++j) {
                    const int r = 16 * e + j;
                    const uint4 v = *reinterpret_cast<const uint4 *>(stg + r * 256 + ((c ^ (r & 15)) << 4));
                    *reinterpret_cast<uint4 *>(obase + (size_t)j * n_heads * D) = v;
                }
            }
            __syncwarp();   // the staging area is read before the next tile's rows overwrite it
        }
        refill();
    }
    if (timed_out) flag_status(status, TQ_STATUS_TIMEOUT);
}

template <typename TO>
cudaError_t dq128v_launch(const void *params, const void *pool, int64_t num_blocks, int n_heads, const int32_t *ids,
                          int n_ids, void *out, int32_t *status, cudaStream_t st) {
    const int64_t ntiles = ((int64_t)n_ids * n_heads + dq128v::kUnits - 1) / dq128v::kUnits;
    if (ntiles <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    auto kern = dequant128v_rows_kernel<TO>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dq128v::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t want = (int64_t)sms * dq128v::kMinCtas;
    const int64_t grid = ntiles < want ? ntiles : want;
    kern<<<(unsigned)grid, dq128v::kThreads, dq128v::kSmem, st>>>((const uint8_t *)params, (const uint8_t *)pool,
                                                                num_blocks, n_heads, ids, n_ids, (TO *)out, status);
    return cudaGetLastError();
}

template <typename TO>
cudaError_t dq128k_launch(const void *params, const void *pool, int64_t num_blocks, int n_heads, const int32_t *ids,
                          int n_ids, void *out, int32_t *status, cudaStream_t st) {
    const int64_t ntiles = ((int64_t)n_ids * n_heads + dq128::kUnits - 1) / dq128::kUnits;
    if (ntiles <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    auto kern = dequant128k_tc_kernel<TO>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dq128::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t grid = ntiles < sms ? ntiles : sms;
    kern<<<(unsigned)grid, dq128::kThreads, dq128::kSmem, st>>>((const uint8_t *)params, (const uint8_t *)pool,
                                                              num_blocks, n_heads, ids, n_ids, (TO *)out, status);
    return cudaGetLastError();
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
    if (d == 128 && is_k && TQ_DEQUANT_TC)
        return out_dtype == TQ_DTYPE_BF16
                   ? dq128k_launch<__nv_bfloat16>(params, pool, num_blocks, n_heads, block_ids, n_ids, out, status, st)
                   : dq128k_launch<float>(params, pool, num_blocks, n_heads, block_ids, n_ids, out, status, st);
    if (d == 128 && !is_k && TQ_DEQUANT_TC)
        return out_dtype == TQ_DTYPE_BF16
                   ? dq128v_launch<__nv_bfloat16>(params, pool, num_blocks, n_heads, block_ids, n_ids, out, status, st)
                   : dq128v_launch<float>(params, pool, num_blocks, n_heads, block_ids, n_ids, out, status, st);
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
