// ct_umma_bf16.cu -- bf16-input / fp32-accumulate ConvTranspose3d on the
// 5th-generation tensor cores (tcgen05 + TMEM), as an implicit GEMM per
// stride phase.
//
// Method ([l1_p72] stride-phase classes; [l2_p26] "what cuDNN does": the
// dense C_in x C_out contraction per output): with stride 2 in every
// dimension and an even kernel extent, every output residue class
// (rD, rH, rW) receives the same number of taps per dimension, and
//     y[n, oc, 2q + r] = bias[oc] + sum_{taps t, ic} x[n, ic, q + delta_t] * w[ic, oc, k_t]
// is a GEMM per phase: M = positions q (N*QD*QH*QW), N = C_out,
// K = taps x C_in.  Two repack kernels prepare the operands in the caller's
// workspace:
//   x  (N, C, D, H, W)  ->  x_cl (N, D, H, W, C)           channels-last, bf16
//   w  (C, C_out, kD, kH, kW) -> w_p [phase][oc][tap][ic]   K-major, bf16
// The GEMM kernel (one CTA = 128 positions x C_out channels x both W phases)
// gathers A tiles straight from x_cl with 5-D TMA loads at the tap's input
// offset -- boxes that reach outside the input read zeros, which is the
// boundary handling -- and B tiles from w_p with 2-D TMA loads, both into
// 128-byte-swizzled shared memory, through a 3-stage mbarrier pipeline.
// One thread issues tcgen05.mma (M=128, N=C_out, K=16, bf16 -> fp32) into
// two TMEM accumulators (rW = 0 and 1); the epilogue reads them with
// tcgen05.ld and writes each output row's even and odd W positions as one
// float2, bias added.  Every mbarrier wait is bounded: a timeout records
// CT_ERR_DEVICE_TIMEOUT in the device status word and the CTA unwinds
// (waiting, bounded, for its own TMA copies and freeing its TMEM).
#include <string.h>

#include "ct_internal.h"
#include "ct_device.cuh"
#include "ct_tma.h"

namespace ct {
namespace {

constexpr int BM = 128;      // positions per tile (UMMA M)
constexpr int BK = 64;       // bf16 elements of K per stage (one 128-byte swizzle row)
constexpr int UK = 16;       // K of one tcgen05.mma kind::f16
constexpr int NST = 3;       // pipeline stages (2 CTAs per SM fit in shared memory)
constexpr int kThreads = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct UParams {
    int N, C_in, C_out;
    int Lo0, Lo1, Lo2;
    int QD, QH, QW, MH, n_qhb;
    int nT;                  // taps per dimension and class (kernel extent / 2)
    int n_kb;                // C_in / BK
    int nit;                 // pipeline iterations per tile
    int ntiles;
    uint32_t idesc;          // tcgen05 instruction descriptor
    uint32_t tmem_cols;      // allocated TMEM columns (power of 2 >= 2*C_out)
    uint32_t stage_bytes;    // A + B bytes per stage
    uint32_t b_bytes;        // B bytes per stage
    int delta[3][2][4];      // input offset of tap j for residue r, per dimension
};

// ---- tcgen05 wrappers --------------------------------------------------------
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    // K-major, 128-byte swizzle: 8-row atoms of 128-byte rows, atoms 1024 B apart
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);          // start address
    d |= (uint64_t)1 << 16;                            // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;                  // stride byte offset
    d |= (uint64_t)1 << 46;                            // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                            // swizzle: 128 B
    return d;
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                     dev::smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// ---- GEMM kernel -------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 2)
umma_ct3d_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const float *__restrict__ bias, float *__restrict__ y, UParams p, unsigned int *status)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[NST], empty_bar[NST], done_bar;
    __shared__ uint32_t tmem_slot;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // tile -> (n, qd, qh block, rD, rH); the four (rD, rH) phases of one input
    // region are neighbours so their A tiles are reused from L2
    int t = blockIdx.x;
    const int rH = t & 1; t >>= 1;
    const int rD = t & 1; t >>= 1;
    const int qhb = t % p.n_qhb; t /= p.n_qhb;
    const int qd = t % p.QD; t /= p.QD;
    const int n = t;
    const int qh0 = qhb * p.MH;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&tmA);
        dev::prefetch_tensormap(&tmB);
        for (int s = 0; s < NST; ++s) {
            dev::mbar_init(&full_bar[s], 1);
            dev::mbar_init(&empty_bar[s], 1);
        }
        dev::mbar_init(&done_bar, 1);
        dev::fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         dev::smem_u32(&tmem_slot)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    const int per_dh = p.n_kb * 2 * p.nT;      // iterations per (D tap, H tap)
    bool failed = false;
    int issued = 0;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        for (int it = 0; it < p.nit; ++it) {
            const int s = it % NST;
            if (it >= NST && !dev::mbar_wait_bounded(&empty_bar[s], ((it / NST) - 1) & 1, kWaitLimitNs)) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                failed = true;
                break;
            }
            const int dh = it / per_dh;
            const int rem = it % per_dh;
            const int kb = rem / (2 * p.nT);
            const int j = rem % (2 * p.nT);
            const int rW = j / p.nT, jw = j % p.nT;
            const int jd = dh / p.nT, jh = dh % p.nT;
            uint8_t *a_s = smem + (size_t)s * p.stage_bytes;
            uint8_t *b_s = a_s + BM * BK * 2;
            dev::mbar_arrive_expect_tx(&full_bar[s], p.stage_bytes);
            dev::tma_load_5d(a_s, &tmA, &full_bar[s], kb * BK, p.delta[2][rW][jw],
                             qh0 + p.delta[1][rH][jh], qd + p.delta[0][rD][jd], n);
            const int phase = (rD * 2 + rH) * 2 + rW;
            const int tap = (jd * p.nT + jh) * p.nT + jw;
            dev::tma_load_2d(b_s, &tmB, &full_bar[s], tap * p.C_in + kb * BK, phase * p.C_out);
            ++issued;
        }
        if (failed) {
            // let this CTA's copies still in flight land before its shared memory goes away
            for (int it = issued - NST > 0 ? issued - NST : 0; it < issued; ++it)
                dev::mbar_wait_bounded(&full_bar[it % NST], (it / NST) & 1, kWaitLimitNs);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        for (int it = 0; it < p.nit; ++it) {
            const int s = it % NST;
            if (!dev::mbar_wait_bounded(&full_bar[s], (it / NST) & 1, kWaitLimitNs)) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                failed = true;
                break;
            }
            tc_fence_after();
            const int rem = it % per_dh;
            const int j = rem % (2 * p.nT);
            const int rW = j / p.nT;
            const bool first = it < per_dh && rem < 2 * p.nT && (j % p.nT) == 0;
            const uint32_t a_addr = dev::smem_u32(smem + (size_t)s * p.stage_bytes);
            const uint32_t b_addr = a_addr + BM * BK * 2;
            const uint64_t da = smem_desc_sw128(a_addr), db = smem_desc_sw128(b_addr);
#pragma unroll
            for (int k = 0; k < BK / UK; ++k) {
                // advance 16 bf16 = 32 bytes along K inside the swizzle atom
                umma_bf16(tmem + (uint32_t)(rW * p.C_out), da + (uint64_t)(k * 2), db + (uint64_t)(k * 2),
                          p.idesc, (first && k == 0) ? 0u : 1u);
            }
            umma_commit(&empty_bar[s]);
        }
        if (!failed) umma_commit(&done_bar);
    }
    __syncwarp();

    // ---- epilogue: TMEM -> registers -> y (both W phases of a position as one float2)
    const bool ok = dev::mbar_wait_bounded(&done_bar, 0, kWaitLimitNs);
    if (!ok && threadIdx.x == 0) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
    if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const int m = warp * 32 + lane;
        const int qh = qh0 + m / p.QW, qw = m % p.QW;
        const int od = 2 * qd + rD, oh = 2 * qh + rH;
        const bool valid = od < p.Lo0 && oh < p.Lo1;
        const int64_t sp = (int64_t)p.Lo0 * p.Lo1 * p.Lo2;
        float *yrow = y + (int64_t)n * p.C_out * sp + ((int64_t)od * p.Lo1 + oh) * p.Lo2 + 2 * qw;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        for (int c0 = 0; c0 < p.C_out; c0 += 16) {
            float a0[16], a1[16];
            tmem_ld16(lane_base + (uint32_t)c0, a0);
            tmem_ld16(lane_base + (uint32_t)(p.C_out + c0), a1);
            tmem_ld_wait();
            if (valid) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int oc = c0 + i;
                    const float b = bias ? __ldg(bias + oc) : 0.f;
                    __stcs(reinterpret_cast<float2 *>(yrow + (int64_t)oc * sp), make_float2(a0[i] + b, a1[i] + b));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(p.tmem_cols)
                     : "memory");
    }
}

// ---- repack kernels ------------------------------------------------------------
// x (N, C, S) -> x_cl (N, S, C), S = D*H*W, through a 64 x 64 shared tile.
__global__ void __launch_bounds__(256)
repack_x_kernel(const bf16_t *__restrict__ x, bf16_t *__restrict__ xcl, int C, int64_t SP)
{
    __shared__ bf16_t tile[64][66];
    const int n = blockIdx.z;
    const int c0 = blockIdx.y * 64;
    const int64_t s0 = (int64_t)blockIdx.x * 64;
    const bf16_t *xs = x + (int64_t)n * C * SP;
    bf16_t *xd = xcl + (int64_t)n * C * SP;
    for (int e = threadIdx.x; e < 64 * 64; e += 256) {
        const int c = e >> 6, s = e & 63;
        tile[c][s] = (c0 + c < C && s0 + s < SP) ? xs[(int64_t)(c0 + c) * SP + s0 + s] : (bf16_t)0;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * 64; e += 256) {
        const int s = e >> 6, c = e & 63;
        if (c0 + c < C && s0 + s < SP) xd[(s0 + s) * C + c0 + c] = tile[c][s];
    }
}

struct WPackParams {
    int C_in, C_out, K0, K1, K2, nT;
    int k[3][2][4];          // tap k of index j for residue r, per dimension
};

// w (C_in, C_out, K0, K1, K2) -> w_p[phase][oc][tap][ic], phase = (rD, rH, rW),
// tap = (jd, jh, jw), ic fastest.
__global__ void __launch_bounds__(256)
repack_w_kernel(const bf16_t *__restrict__ w, bf16_t *__restrict__ wp, WPackParams q)
{
    const int ntap = q.nT * q.nT * q.nT;
    const int64_t total = (int64_t)8 * q.C_out * ntap * q.C_in;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = e;
        const int ic = (int)(r % q.C_in); r /= q.C_in;
        const int tap = (int)(r % ntap); r /= ntap;
        const int oc = (int)(r % q.C_out); r /= q.C_out;
        const int ph = (int)r;
        const int rW = ph & 1, rH = (ph >> 1) & 1, rD = (ph >> 2) & 1;
        const int jw = tap % q.nT, jh = (tap / q.nT) % q.nT, jd = tap / (q.nT * q.nT);
        const int kd = q.k[0][rD][jd], kh = q.k[1][rH][jh], kw = q.k[2][rW][jw];
        wp[e] = w[((((int64_t)ic * q.C_out + oc) * q.K0 + kd) * q.K1 + kh) * q.K2 + kw];
    }
}

// ---- host side ------------------------------------------------------------------
struct UPlan {
    UParams p;
    WPackParams wq;
    size_t x_bytes, w_bytes, smem;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

bool make_uplan(const Problem &pb, UPlan *out)
{
    if (pb.nd != 3 || pb.dtype != CT_BF16 || pb.G != 1) return false;
    for (int d = 0; d < 3; ++d) {
        if (pb.S[d] != 2 || pb.DL[d] != 1) return false;
        if (pb.K[d] % 2 != 0 || pb.K[d] / 2 > 4) return false;
        if (pb.K[d] != pb.K[0]) return false;
    }
    if (pb.C_in % BK != 0 || pb.C_out % 16 != 0 || pb.C_out < 16 || pb.C_out > 256) return false;
    if (pb.Lo[2] % 2 != 0) return false;
    UParams p;
    memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C_in = pb.C_in; p.C_out = pb.C_out;
    p.Lo0 = pb.Lo[0]; p.Lo1 = pb.Lo[1]; p.Lo2 = pb.Lo[2];
    p.QW = p.Lo2 / 2;
    if (p.QW > BM || BM % p.QW != 0) return false;
    p.MH = BM / p.QW;
    p.QD = (p.Lo0 + 1) / 2;
    p.QH = (p.Lo1 + 1) / 2;
    p.n_qhb = (p.QH + p.MH - 1) / p.MH;
    p.nT = pb.K[0] / 2;
    p.n_kb = pb.C_in / BK;
    p.nit = p.nT * p.nT * p.n_kb * 2 * p.nT;
    const int64_t tiles = (int64_t)pb.N * p.QD * p.n_qhb * 4;
    if (tiles > 0x7fffffff || tiles == 0) return false;
    p.ntiles = (int)tiles;
    // residue r of a stride-2 dimension takes the taps k == (r + p) mod 2, i.e.
    // k = c + 2j, reading input q + floor((r + p)/2) - j
    WPackParams wq;
    memset(&wq, 0, sizeof(wq));
    for (int d = 0; d < 3; ++d) {
        for (int r = 0; r < 2; ++r) {
            const int c = (r + pb.P[d]) % 2;
            const int base = (r + pb.P[d] - c) / 2;
            for (int j = 0; j < p.nT; ++j) {
                p.delta[d][r][j] = base - j;
                wq.k[d][r][j] = c + 2 * j;
            }
        }
    }
    wq.C_in = pb.C_in; wq.C_out = pb.C_out; wq.nT = p.nT;
    wq.K0 = pb.K[0]; wq.K1 = pb.K[1]; wq.K2 = pb.K[2];
    // tcgen05 instruction descriptor: D fp32, A/B bf16, both K-major, N, M
    p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(pb.C_out >> 3) << 17) |
              ((uint32_t)(BM >> 4) << 24);
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * pb.C_out)) cols <<= 1;
    p.tmem_cols = cols;
    p.b_bytes = (uint32_t)pb.C_out * BK * 2;
    p.stage_bytes = (uint32_t)(BM * BK * 2) + p.b_bytes;
    out->p = p;
    out->wq = wq;
    out->x_bytes = align256((size_t)pb.N * pb.C_in * pb.in_sp() * 2);
    out->w_bytes = align256((size_t)8 * pb.C_out * p.nT * p.nT * p.nT * pb.C_in * 2);
    out->smem = (size_t)NST * p.stage_bytes + 1024;
    if (out->smem > 227 * 1024) return false;
    return true;
}

}  // namespace

bool umma_supported(const Problem &pb, const Args *a)
{
    UPlan pl;
    if (!make_uplan(pb, &pl)) return false;
    if (a && (((uintptr_t)a->y % 8) || ((uintptr_t)a->x % 16) || ((uintptr_t)a->w % 16))) return false;
    return true;
}

size_t umma_workspace_bytes(const Problem &pb)
{
    UPlan pl;
    if (!make_uplan(pb, &pl)) return 0;
    return pl.x_bytes + pl.w_bytes;
}

cudaError_t launch_umma(const Problem &pb, const Args &a)
{
    UPlan pl;
    if (!make_uplan(pb, &pl)) return cudaErrorNotSupported;
    const UParams &p = pl.p;
    bf16_t *xcl = static_cast<bf16_t *>(a.ws);
    bf16_t *wp = reinterpret_cast<bf16_t *>(static_cast<uint8_t *>(a.ws) + pl.x_bytes);

    // 1) x -> channels-last
    const int64_t SP = pb.in_sp();
    dim3 gx((unsigned)((SP + 63) / 64), (unsigned)((pb.C_in + 63) / 64), (unsigned)pb.N);
    if (gx.x > 0x7fffffffu || gx.y > 65535 || gx.z > 65535) return cudaErrorInvalidConfiguration;
    repack_x_kernel<<<gx, 256, 0, a.stream>>>(static_cast<const bf16_t *>(a.x), xcl, pb.C_in, SP);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2) weights -> per-phase K-major
    const int64_t wtot = (int64_t)8 * pb.C_out * p.nT * p.nT * p.nT * pb.C_in;
    int wblocks = (int)((wtot + 255) / 256);
    if (wblocks > 4 * sm_count()) wblocks = 4 * sm_count();
    repack_w_kernel<<<wblocks, 256, 0, a.stream>>>(static_cast<const bf16_t *>(a.w), wp, pl.wq);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // 3) tensor maps: A over x_cl (C, W, H, D, N), B over w_p (K, 8*C_out)
    CUtensorMap tmA, tmB;
    const uint64_t adims[5] = {(uint64_t)pb.C_in, (uint64_t)pb.Li[2], (uint64_t)pb.Li[1],
                               (uint64_t)pb.Li[0], (uint64_t)pb.N};
    const uint64_t astr[4] = {(uint64_t)pb.C_in * 2, (uint64_t)pb.C_in * pb.Li[2] * 2,
                              (uint64_t)pb.C_in * pb.Li[2] * pb.Li[1] * 2,
                              (uint64_t)pb.C_in * pb.Li[2] * pb.Li[1] * pb.Li[0] * 2};
    const uint32_t abox[5] = {(uint32_t)BK, (uint32_t)p.QW, (uint32_t)p.MH, 1u, 1u};
    if (!encode_tiled(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, xcl, adims, astr, abox,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int ntap = p.nT * p.nT * p.nT;
    const uint64_t bdims[2] = {(uint64_t)ntap * pb.C_in, (uint64_t)8 * pb.C_out};
    const uint64_t bstr[1] = {(uint64_t)ntap * pb.C_in * 2};
    const uint32_t bbox[2] = {(uint32_t)BK, (uint32_t)pb.C_out};
    if (!encode_tiled(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wp, bdims, bstr, bbox,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    int per_sm = 0;
    e = prepare_kernel((const void *)&umma_ct3d_kernel, kThreads, pl.smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    unsigned int *status = device_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    umma_ct3d_kernel<<<p.ntiles, kThreads, pl.smem, a.stream>>>(tmA, tmB, a.bias, a.y, p, status);
    return cudaGetLastError();
}

}  // namespace ct
