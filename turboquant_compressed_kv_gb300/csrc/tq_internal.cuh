// tq_internal.cuh -- layout constants and device helpers shared by the kernels.
//
// Packed layout of one record (16 token slots of one block, one kv head):
//   K: planes 0..2 (bit p of the 3-bit cell), plane 3 (QJL sign bits), each
//      2*d bytes, then 16 x {fp16 ||x||, fp16 ||r||}.
//   V: planes 0..2, each 2*d bytes, then 16 x fp16 ||v||.
// Each plane is an array of 32-bit words indexed by a lane L = 4*gid + tig.
//   K: coordinate i = 16*s + 8*h + 2*tig + e of slot t = gid + 8*th sits in
//      word (L*2 + th)*NW + (s>>3), NW = d/128, at bit 8*h + (s&7) + 16*e.
//   V: coordinate i = 16*mt + gid + 8*rh of slot t = 2*tig + 8*tp + e sits in
//      word L*NWV + 2*(mt>>3) + rh, NWV = d/64, at bit 8*tp + (mt&7) + 16*e.
// In both layouts one byte of a word belongs to one token slot, so slots can
// be written independently with byte stores.  Bits p and p+16 of a word are
// the two halves of one f16x2 operand register of the m16n8k16 mma.sync used
// by decode attention (K: token rows x coordinate columns; V: coordinate rows
// x token columns), so one LOP3 turns them into two f16 operands.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

constexpr uint32_t kParamsMagic = 0x31505154u;   // "TQP1"
constexpr int kBlock = 16;

// Device params header (256 bytes); D signs and S follow.
struct ParamsHeader {
    uint32_t magic;
    int32_t d;
    int32_t reserved[2];
    float centroid[8];     // ascending, unit variance
    float threshold[8];    // 7 used: midpoints of neighbouring centroids
    double centroid64[8];  // the same centroids before rounding to fp32
    float pad[28];
};
static_assert(sizeof(ParamsHeader) == 256, "params header must be 256 bytes");

__host__ __device__ constexpr size_t params_off_D(int /*d*/) { return 256; }
__host__ __device__ constexpr size_t params_off_S(int d) { return 256 + 4 * (size_t)d; }
__host__ __device__ constexpr size_t params_total(int d) { return params_off_S(d) + 4 * (size_t)d * d; }

__host__ __device__ constexpr size_t k_record(int d) { return 8 * (size_t)d + 4 * kBlock; }
__host__ __device__ constexpr size_t v_record(int d) { return 6 * (size_t)d + 2 * kBlock; }

inline bool valid_d(int d) { return d == 128 || d == 256; }

// ---------------------------------------------------------------- value loads

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------- lane -> coordinate maps
// Warp-per-vector encoders hold R = d/32 coordinates per lane; coordinate
// kdim(lane, r) / vdim(lane, r) is chosen so that __ballot_sync over register r
// yields one packed word (K) or four packed bytes (V) directly.

template <int D>
__device__ __forceinline__ int kdim(int lane, int r) {
    const int e = lane >> 4, h = (lane >> 3) & 1, s = 8 * (r >> 2) + (lane & 7), tig = r & 3;
    return 16 * s + 8 * h + 2 * tig + e;
}

template <int D>
__device__ __forceinline__ int vdim(int lane, int r) {
    constexpr int NM = D / 128;
    int beta = lane >> 3, q = lane & 7;
    int tau = 4 * r + beta;
    int mhi = tau % NM, rh = (tau / NM) & 1, gid = tau / (2 * NM);
    int mt = 8 * mhi + q;
    return 16 * mt + gid + 8 * rh;
}

// In-register fast Walsh-Hadamard transform (Sylvester order, unnormalised)
// of a d-vector spread over a warp as v[r] at lane l.  Each index bit of the
// coordinate is either a lane bit (butterfly through a shuffle) or a register
// bit (butterfly inside the thread); since H is the Kronecker product of one
// 2x2 butterfly per index bit, any bijective lane/register map is handled by
// running every lane-bit stage and every register-bit stage once.
template <int R>
__device__ __forceinline__ void fwht_warp(float (&v)[R], int lane) {
#pragma unroll
    for (int x = 0; x < 5; ++x) {
        const int m = 1 << x;
        const bool upper = (lane >> x) & 1;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float w = __shfl_xor_sync(0xffffffffu, v[r], m);
            v[r] = upper ? (w - v[r]) : (v[r] + w);
        }
    }
#pragma unroll
    for (int y = 1; y < R; y <<= 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if ((r & y) == 0) {
                float a = v[r], b = v[r | y];
                v[r] = a + b;
                v[r | y] = a - b;
            }
        }
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

__device__ __forceinline__ void flag_status(int32_t *status, int bits) {
    if (status) atomicOr(status, bits);
}

}  // namespace tq
