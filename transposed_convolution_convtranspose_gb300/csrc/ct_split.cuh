// ct_split.cuh -- the operand split shared by the FP32 tensor-core kernels of
// ct_tc3d_split.cu and ct_tc3s_split.cu: one prep launch that writes x
// channels-last as (t, l) tf32 parts or (hi, lo) bf16 parts, and the weights
// as run panels.  Device code and small host helpers; included into each
// translation unit's anonymous namespace.
//
// Every value v is split as t = tf32(v) (cvt.rna: nearest, ties away) and
// l = tf32(v - t) -- v - t is exact in fp32, |v - t - l| <= 2^-22 |v| -- or,
// for the opt-in pair, hi = bf16(v) (nearest even) and lo = bf16(v - hi).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ct_tma.h"

namespace ct {
namespace {

constexpr int kMaxBlk = 256;     // C_out-row blocks of the weight panels

// Weight panel rows: block b (C_out rows) holds tap blk_tap[b]: tf32x3 its
// t parts (blk_lo 0) or its l parts (blk_lo 1), one fp32 word per input
// channel; bf16x2 its bf16 hi parts (blk_lo 0) or its lo parts (blk_lo 1),
// each twice per K step (a pair per word).
struct WPanels {
    int C_in, C_out, ntap, nblk, tf;
    int16_t blk_tap[kMaxBlk];
    int8_t blk_lo[kMaxBlk];
};

__device__ __forceinline__ float bf16_round(float v)
{
    return __bfloat162float(__float2bfloat16_rn(v));
}
__device__ __forceinline__ uint32_t bf16_bits(float v)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
}
// v rounded to tf32 (10 fraction bits, nearest, ties away from zero): the low
// 13 bits of the result are zero, so the tensor cores read it exactly
__device__ __forceinline__ float tf32_round(float v)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// The split of 4 consecutive channels c .. c + 3 of one position, stored at
// the channel's place in x_c.  tf32x3: per 32 channels [t x 32 | l x 32], 64
// words; bf16x2: per K step of 8 channels [hi x 8 | lo x 8], 16 bf16 per 8
// channels.  `pos` points at the position's x_c row (its element 0) in 4-byte
// units; c is a multiple of 4.
__device__ __forceinline__ void store_split4(uint32_t *pos, int c, const float (&v)[4], bool tf)
{
    if (tf) {
        float t[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            t[i] = tf32_round(v[i]);
            l[i] = tf32_round(v[i] - t[i]);       // v - t is exact in fp32
        }
        uint32_t *r = pos + (c >> 5) * 64 + (c & 31);
        *reinterpret_cast<float4 *>(r) = make_float4(t[0], t[1], t[2], t[3]);
        *reinterpret_cast<float4 *>(r + 32) = make_float4(l[0], l[1], l[2], l[3]);
    } else {
        uint32_t hb[4], lb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float h = bf16_round(v[i]);
            hb[i] = bf16_bits(h);
            lb[i] = bf16_bits(v[i] - h);          // v - h is exact in fp32
        }
        // K step c / 8 of the row (32 bytes = 8 words each), elements c mod 8 ..
        uint16_t *r = reinterpret_cast<uint16_t *>(pos) + (c >> 3) * 16 + (c & 4);
        *reinterpret_cast<uint2 *>(r) = make_uint2(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16));
        *reinterpret_cast<uint2 *>(r + 8) = make_uint2(lb[0] | (lb[1] << 16), lb[2] | (lb[3] << 16));
    }
}

// x (N, C, S) -> x_c (N, S, 2C x 4 bytes (tf32x3) or 2C x 2 bytes (bf16x2));
// S = D*H*W a multiple of 4, C of 32.  Block = 32 channels x 64 positions:
// 16-byte loads of 4 positions of one channel (a warp reads 2 x 256
// contiguous bytes), a shared tile of pitch 33, then per thread 4 channels
// of one position.
__device__ __forceinline__ void prep_x_block(const float *__restrict__ x, uint32_t *__restrict__ xc, int C,
                                             int64_t SP, int bx, int by, int n, bool tf)
{
    __shared__ float tile[64][33];
    const int c0 = by * 32;
    const int64_t s0 = (int64_t)bx * 64;
    const int ncols = (int)((SP - s0) < 64 ? (SP - s0) : 64);
    const float *xs = x + ((int64_t)n * C + c0) * SP + s0;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = threadIdx.x + 256 * it;
        const int c = idx >> 4, p4 = idx & 15;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p4 * 4 < ncols) v = __ldcs(reinterpret_cast<const float4 *>(xs + (int64_t)c * SP + p4 * 4));
        tile[p4 * 4 + 0][c] = v.x;
        tile[p4 * 4 + 1][c] = v.y;
        tile[p4 * 4 + 2][c] = v.z;
        tile[p4 * 4 + 3][c] = v.w;
    }
    __syncthreads();
    // 4-byte words of x_c per position: 2C (tf32x3) or C (bf16x2)
    const int64_t wpp = tf ? 2 * (int64_t)C : (int64_t)C;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = threadIdx.x + 256 * it;
        const int q = idx & 7, pos = idx >> 3;
        if (pos < ncols) {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = tile[pos][4 * q + i];
            store_split4(xc + ((int64_t)n * SP + s0 + pos) * wpp, c0 + 4 * q, v, tf);
        }
    }
}

// w (C_in, C_out, K0, K1, K2) -> weight panels [block][C_out rows][C_in
// words]: tf32x3 the t (blk_lo 0) or l (blk_lo 1) part of each weight;
// bf16x2 rows of [hi | hi] (blk_lo 0) or [lo | lo] (blk_lo 1) per K step of 8
// input channels.
__device__ __forceinline__ void prep_w_block(const float *__restrict__ w, float *__restrict__ wp, const WPanels &q,
                                             int bw, int nbw)
{
    const int64_t per = (int64_t)q.C_out * q.C_in;
    const int64_t total = (int64_t)q.nblk * per;
    for (int64_t e = (int64_t)bw * blockDim.x + threadIdx.x; e < total; e += (int64_t)nbw * blockDim.x) {
        const int b = (int)(e / per);
        const int64_t r = e % per;
        const int oc = (int)(r / q.C_in), ic = (int)(r % q.C_in);
        const float v = __ldg(w + ((int64_t)ic * q.C_out + oc) * q.ntap + q.blk_tap[b]);
        if (q.tf) {
            const float t = tf32_round(v);
            wp[e] = q.blk_lo[b] ? tf32_round(v - t) : t;
        } else {
            const float h = bf16_round(v);
            const uint16_t t = (uint16_t)bf16_bits(q.blk_lo[b] ? v - h : h);
            // the row's bf16 view: K step ic / 8 of its 32-channel block
            uint16_t *row = reinterpret_cast<uint16_t *>(wp + (e - ic));
            const int kb = ic >> 5, kk = (ic & 31) >> 3, el = ic & 7;
            row[kb * 64 + kk * 16 + el] = t;
            row[kb * 64 + kk * 16 + 8 + el] = t;
        }
    }
}

// Channels-last x (N, S, C) -> x_c: the same split, no transpose.  Block =
// 1024 consecutive values (256 threads x 4 channels: one 16-byte load each);
// C a multiple of 32, so 4 channels never cross a position.
__device__ __forceinline__ void prep_x_cl_block(const float *__restrict__ x, uint32_t *__restrict__ xc, int C,
                                                int64_t total, int bx, bool tf)
{
    const int64_t e = ((int64_t)bx * 256 + threadIdx.x) * 4;    // first of 4 values
    if (e >= total) return;
    const float4 v4 = __ldcs(reinterpret_cast<const float4 *>(x + e));
    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
    const int c = (int)(e % C);
    const int64_t pos = e / C;
    store_split4(xc + pos * (tf ? 2 * (int64_t)C : (int64_t)C), c, v, tf);
}

// Both preps in one launch: blocks [0, nxb) move x (nbx x nby per image; or,
// channels last, 1024 consecutive values each), the remaining nbw blocks build
// the panels.  The GEMM kernel is launched as its programmatic dependent.  The
// x blocks run from the end of x backwards: the GEMM consumes x_c from the
// first image on, so its first reads are the lines written last, the ones
// still in L2.
__global__ void __launch_bounds__(256)
prep_kernel(const float *__restrict__ x, uint32_t *__restrict__ xc, int C, int64_t SP,
            int nbx, int nby, int nxb, const float *__restrict__ w, float *__restrict__ wp,
            const __grid_constant__ WPanels q, int nbw, int64_t cl_total)
{
    dev::griddep_launch_dependents();
    const int b = (int)blockIdx.x;
    const bool tf = q.tf != 0;
    if (b < nxb && cl_total > 0) {
        prep_x_cl_block(x, xc, C, cl_total, nxb - 1 - b, tf);
    } else if (b < nxb) {
        const int per = nbx * nby, rb = nxb - 1 - b;
        prep_x_block(x, xc, C, SP, (rb % per) % nbx, (rb % per) / nbx, rb / per, tf);
    } else {
        prep_w_block(w, wp, q, b - nxb, nbw);
    }
}


size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Taps of residue r in one dimension of stride S and dilation DL: the k with
// (r + P - k DL) divisible by S, input offset (r + P - k DL) / S (exact).
int split_dim_taps(int K, int S, int P, int DL, int r, int *k_out, int *d_out, int max)
{
    int n = 0;
    for (int k = 0; k < K; ++k) {
        const int num = r + P - k * DL;
        if (((num % S) + S) % S != 0) continue;
        if (n >= max) return -1;
        k_out[n] = k;
        d_out[n] = num / S;     // divisible: exact for negative values too
        ++n;
    }
    return n;
}

}  // namespace
}  // namespace ct
