// ct_tc3d_tf32.cu -- FP32 ConvTranspose3d, plain or with the fused
// add + t*hardswish(t) epilogue, on the tensor cores (tcgen05 kind::tf32)
// with a 3-term split that keeps fp32-level accuracy.
//
// Method ([l1_p72] stride-phase classes: residue r of a dimension receives
// the taps k with (r + p - k) even, reading input q + (r + p - k)/2;
// [l2_p26] the fused epilogue t = conv + bias + add, out = t*hardswish(t)):
// with stride 2 and dilation 1 in every dimension, output (2qd+rD, 2qh+rH,
// 2qw+rW) of channel oc is
//     bias[oc] + sum over the phase's taps (kd, kh, kw) and ic of
//                x[ic][qd+dd][qh+dh][qw+dw] * w[ic][oc][kd][kh][kw]
// -- for 128 positions q a GEMM with M = 128, N = C_out, K = C_in per tap.
//
// Operands (caller's workspace, written by the two prep kernels):
//   x (N, C_in, D, H, W) -> x_hi, x_lo (N, D, H, W, C_in), channels-last
//   w (C_in, C_out, kD, kH, kW) -> w_p [tap][hi, lo][C_out][C_in]
// with hi = v rounded to tf32 (cvt.rna) and lo = v - hi (exact in fp32);
// three MMAs per product accumulate hi*hi + hi*lo + lo*hi in fp32 in TMEM;
// the dropped lo*lo term and the tf32 truncation of lo are each below 2^-21
// of a product.
//
// GEMM kernel: persistent, one CTA per SM, warp-specialised.  A unit of work
// is 128 positions (whole W rows of MH H rows of one D plane) and one D
// residue rD, with all four (rH, rW) phases as four accumulators of C_out
// TMEM columns; two such sets alternate across units when they fit, so the
// epilogue of one unit overlaps the MMAs of the next.
//   warps 0-3  TMA producers, two per ring, taking turns stage by stage (one
//              thread's TMA stream completes about one box at a time).  For
//              every distinct input offset (dd, dh, dw) the unit reads, an A
//              stage (the hi and lo tiles: 5-D boxes of 128 positions x 32
//              channels at that offset; boxes reaching outside the input read
//              zeros, which is the boundary handling), then one B stage (one
//              box: the hi and lo C_out x 32 weight tiles) per phase tap that
//              reads that offset.  A and B stages have separate rings.
//   warp 4     TMEM allocation and MMA issue: per B stage, for each 8-wide
//              K step, three tcgen05.mma (M = 128, N = C_out, K = 8) into the
//              phase's accumulator.
//   warps 5-12 epilogue, two per TMEM lane quarter taking alternate
//              16-channel chunks, one H phase at a time: the add values are
//              loaded first, then tcgen05.ld of the two W phases, bias, the
//              fused epilogue, and each position's even and odd W outputs
//              stored as one float2 (a warp writes two whole output rows per
//              channel and H phase).
// Every mbarrier wait is bounded: a timeout records CT_ERR_DEVICE_TIMEOUT in
// the device status word and the roles unwind (each producer waits, bounded,
// for its own TMA copies and the MMA issuer for its own MMAs before the TMEM
// is freed).
#include <string.h>

#include "ct_internal.h"
#include "ct_device.cuh"
#include "ct_tma.h"
#include "ct_tcgen05.cuh"

namespace ct {
namespace {

constexpr int BM = 128;          // positions per unit (UMMA M)
constexpr int CK = 32;           // fp32 K per stage: one 128-byte swizzle row
constexpr int MAXE = 18;         // A stages of a unit per K block at most (2 x 3 x 3)
constexpr int NA = 4;            // A stages
constexpr int MAXB = 8;          // B stages at most
constexpr int NPA = 2;           // producer warps of the A ring (stage g loaded by warp g mod NPA)
constexpr int NPB = 2;           // producer warps of the B ring
constexpr int EPW = 2;           // epilogue warps per TMEM lane quarter
constexpr int kMmaWarp = NPA + NPB;
constexpr int kEpiWarp0 = kMmaWarp + 1;
constexpr int kThreads = 32 * (kEpiWarp0 + 4 * EPW);
// Every stage slot has exactly one producer warp (ring sizes are multiples of
// the producer counts), which refills it only after waiting for the slot's
// previous round, so a parity wait never has to tell two phases apart.
static_assert(NA % NPA == 0, "one producer per A slot");
static_assert(MAXB % NPB == 0, "one producer per B slot");
constexpr uint32_t kATile = BM * CK * 4;       // one of hi / lo: 16 KB
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// One input offset read by a unit and the phase taps that read it.
struct AEntry {
    int8_t dd, dh, dw, nuse;
    int8_t tap[4];               // weight tap (kd*K1 + kh)*K2 + kw
    int8_t ph[4];                // accumulator rH*2 + rW
};

struct T3Params {
    int N, C_in, C_out;
    int Lo0, Lo1, Lo2;
    int QD, QH, QW, MH, n_qhb;
    int n_kb;                    // C_in / 32
    int nunits;
    int nb;                      // B stages
    int nacc;                    // accumulator sets (1 or 2)
    uint32_t acc_cols;           // 4 x C_out
    uint32_t tmem_cols;
    uint32_t idesc;
    uint32_t b_bytes;            // one of hi / lo: C_out x 128
    int nA[2];                   // entries per D residue
    AEntry ent[2][MAXE];
};

__device__ __forceinline__ float tf32_hi(float v)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// ---- prep kernels ------------------------------------------------------------
// x (N, C, S) -> x_hi, x_lo (N, S, C); S = D*H*W a multiple of 4, C of 32.
// Block = 32 channels x 64 positions: 16-byte loads of 4 positions of one
// channel (a warp reads 2 x 256 contiguous bytes), a shared tile of pitch 33,
// 16-byte stores of 4 channels of one position (a warp writes 4 x 128 bytes).
__global__ void __launch_bounds__(256)
prep_x_kernel(const float *__restrict__ x, float *__restrict__ xhi, float *__restrict__ xlo, int C, int64_t SP)
{
    __shared__ float tile[64][33];
    const int n = blockIdx.z;
    const int c0 = blockIdx.y * 32;
    const int64_t s0 = (int64_t)blockIdx.x * 64;
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
    const int64_t ob = ((int64_t)n * SP + s0) * C + c0;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = threadIdx.x + 256 * it;
        const int q = idx & 7, pos = idx >> 3;
        if (pos < ncols) {
            float h[4], l[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float v = tile[pos][4 * q + i];
                h[i] = tf32_hi(v);
                l[i] = v - h[i];
            }
            const int64_t o = ob + (int64_t)pos * C + 4 * q;
            *reinterpret_cast<float4 *>(xhi + o) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(xlo + o) = make_float4(l[0], l[1], l[2], l[3]);
        }
    }
}

// w (C_in, C_out, K0, K1, K2) -> w_p [tap][hi, lo][C_out][C_in], tap = (kd*K1 + kh)*K2 + kw:
// the hi and lo panels of a tap are adjacent, so one box of 2*C_out rows
// brings both.
__global__ void __launch_bounds__(256)
prep_w_kernel(const float *__restrict__ w, float *__restrict__ wp, int C_in, int C_out, int ntap)
{
    const int64_t total = (int64_t)ntap * C_out * C_in;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int ic = (int)(e % C_in);
        const int64_t r = e / C_in;
        const int oc = (int)(r % C_out);
        const int tap = (int)(r / C_out);
        const float v = __ldg(w + ((int64_t)ic * C_out + oc) * ntap + tap);
        const float h = tf32_hi(v);
        const int64_t o = ((int64_t)tap * 2 * C_out + oc) * C_in + ic;
        wp[o] = h;
        wp[o + (int64_t)C_out * C_in] = v - h;
    }
}

// ---- GEMM kernel ----------------------------------------------------------------
// unit -> (n, qd, qh block, rD); the two D residues of one position block are
// neighbours, so the A tiles they share are reused from L2
struct UnitCoord {
    int n, qd, qhb, rd;
};
__device__ __forceinline__ UnitCoord unit_coord(int u, const T3Params &p)
{
    UnitCoord c;
    c.rd = u & 1;
    u >>= 1;
    c.qhb = u % p.n_qhb;
    u /= p.n_qhb;
    c.qd = u % p.QD;
    c.n = u / p.QD;
    return c;
}

template <bool ADD>
__global__ void __launch_bounds__(kThreads, 1)
tc3d_tf32_kernel(const __grid_constant__ CUtensorMap tmXh, const __grid_constant__ CUtensorMap tmXl,
                 const __grid_constant__ CUtensorMap tmW, const float *__restrict__ bias, const float *add,
                 float *y, T3Params p, unsigned int *status)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t a_full[NA], a_empty[NA], b_full[MAXB], b_empty[MAXB], acc_full[2],
        acc_empty[2], drain_bar;
    __shared__ uint32_t tmem_slot;
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = sm;                                  // NA x (hi, lo)
    uint8_t *sB = sm + NA * 2 * kATile;                // nb x (hi, lo)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&tmXh);
        dev::prefetch_tensormap(&tmXl);
        dev::prefetch_tensormap(&tmW);
        for (int s = 0; s < NA; ++s) {
            dev::mbar_init(&a_full[s], 1);
            dev::mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < p.nb; ++s) {
            dev::mbar_init(&b_full[s], 1);
            dev::mbar_init(&b_empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            dev::mbar_init(&acc_full[a], 1);
            dev::mbar_init(&acc_empty[a], 32 * 4 * EPW);   // every epilogue thread
        }
        dev::mbar_init(&drain_bar, 1);
        dev::fence_mbar_init();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(&tmem_slot, p.tmem_cols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = tmem_slot;
    const int nunit_cta =
        p.nunits > (int)blockIdx.x ? (p.nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const uint32_t b_stage = 2 * p.b_bytes;

    if (warp < NPA + NPB) {
        // ---------------- TMA producers.  One thread's TMA stream completes about one
        // box at a time, so the A ring has NPA producer warps and the B ring NPB,
        // warp q of a ring loading its stages q, q + NP, ... in the ring's order.
        if (lane == 0) {
            const bool isA = warp < NPA;
            const int q = isA ? warp : warp - NPA;
            const int np = isA ? NPA : NPB;
            const int nst = isA ? NA : p.nb;
            uint64_t *fullb = isA ? a_full : b_full;
            uint64_t *emptyb = isA ? a_empty : b_empty;
            int g = 0, last = -1;                     // position in the ring's sequence
            bool failed = false;
            for (int k = 0; k < nunit_cta && !failed; ++k) {
                const UnitCoord u = unit_coord((int)blockIdx.x + k * (int)gridDim.x, p);
                const int qh0 = u.qhb * p.MH;
                const int ne = p.nA[u.rd];
                for (int e = 0; e < ne && !failed; ++e) {
                    const AEntry &en = p.ent[u.rd][e];
                    for (int kb = 0; kb < p.n_kb && !failed; ++kb) {
                        const int nload = isA ? 1 : en.nuse;
                        for (int j = 0; j < nload; ++j, ++g) {
                            if (g % np != q) continue;
                            const int s = g % nst;
                            if (g >= nst && !dev::mbar_wait_bounded(&emptyb[s], ((g / nst) - 1) & 1, kWaitLimitNs)) {
                                failed = true;
                                break;
                            }
                            if (isA) {
                                uint8_t *ah = sA + (size_t)s * 2 * kATile;
                                dev::mbar_arrive_expect_tx(&fullb[s], 2 * kATile);
                                dev::tma_load_5d(ah, &tmXh, &fullb[s], kb * CK, en.dw, qh0 + en.dh, u.qd + en.dd, u.n);
                                dev::tma_load_5d(ah + kATile, &tmXl, &fullb[s], kb * CK, en.dw, qh0 + en.dh,
                                                 u.qd + en.dd, u.n);
                            } else {
                                dev::mbar_arrive_expect_tx(&fullb[s], b_stage);
                                dev::tma_load_2d(sB + (size_t)s * b_stage, &tmW, &fullb[s], kb * CK,
                                                 en.tap[j] * 2 * p.C_out);
                            }
                            last = g;
                        }
                    }
                }
            }
            if (failed) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                // let this warp's copies still in flight land before shared memory goes away
                for (int r = last; r >= 0 && r > last - nst; r -= np)
                    dev::mbar_wait_bounded(&fullb[r % nst], (r / nst) & 1, kWaitLimitNs);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            int ga = 0, gb = 0;
            for (int k = 0; k < nunit_cta && ok; ++k) {
                const UnitCoord u = unit_coord((int)blockIdx.x + k * (int)gridDim.x, p);
                const int a = p.nacc == 2 ? (k & 1) : 0;
                const int use = p.nacc == 2 ? (k >> 1) : k;     // earlier units in accumulator set a
                if (use > 0 && !dev::mbar_wait_bounded(&acc_empty[a], (use - 1) & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)a * p.acc_cols;
                uint32_t init = 0;                              // accumulators written so far
                const int ne = p.nA[u.rd];
                for (int e = 0; e < ne && ok; ++e) {
                    const AEntry &en = p.ent[u.rd][e];
                    for (int kb = 0; kb < p.n_kb && ok; ++kb) {
                        const int sa = ga % NA;
                        if (!dev::mbar_wait_bounded(&a_full[sa], (ga / NA) & 1, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after();
                        const uint32_t ah = dev::smem_u32(sA + (size_t)sa * 2 * kATile);
                        const uint64_t dah = tc::desc_sw128(ah), dal = tc::desc_sw128(ah + kATile);
                        for (int j = 0; j < en.nuse; ++j) {
                            const int sb = gb % p.nb;
                            if (!dev::mbar_wait_bounded(&b_full[sb], (gb / p.nb) & 1, kWaitLimitNs)) {
                                ok = false;
                                break;
                            }
                            tc::fence_after();
                            const uint32_t bh = dev::smem_u32(sB + (size_t)sb * b_stage);
                            const uint64_t dbh = tc::desc_sw128(bh), dbl = tc::desc_sw128(bh + p.b_bytes);
                            const int ph = en.ph[j];
                            const uint32_t dd = d + (uint32_t)(ph * p.C_out);
                            const bool first = !((init >> ph) & 1u);
#pragma unroll
                            for (int kk = 0; kk < CK / 8; ++kk) {
                                // advance 8 tf32 = 32 bytes along K inside the swizzle atom
                                const uint64_t ko = (uint64_t)(kk * 2);
                                tc::mma_tf32(dd, dah + ko, dbh + ko, p.idesc, (first && kk == 0) ? 0u : 1u);
                                tc::mma_tf32(dd, dah + ko, dbl + ko, p.idesc, 1u);
                                tc::mma_tf32(dd, dal + ko, dbh + ko, p.idesc, 1u);
                            }
                            init |= 1u << ph;
                            tc::commit(&b_empty[sb]);
                            ++gb;
                        }
                        tc::commit(&a_empty[sa]);
                        ++ga;
                    }
                }
                if (ok) tc::commit(&acc_full[a]);
            }
            // every MMA issued has to complete before the TMEM is freed
            tc::commit(&drain_bar);
            if (!dev::mbar_wait_bounded(&drain_bar, 0, kWaitLimitNs)) ok = false;
            if (!ok) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
        }
    } else {
        // ---------------- epilogue: EPW warps per TMEM lane quarter (32 positions); a
        // warp reaches the lanes of quarter warp mod 4
        const int ew = warp & 3;
        const int half = (warp - kEpiWarp0) >> 2;
        const int nchunk = p.C_out / 16;
        const int64_t sp = (int64_t)p.Lo0 * p.Lo1 * p.Lo2;
        bool ok = true;
        for (int k = 0; k < nunit_cta; ++k) {
            const UnitCoord u = unit_coord((int)blockIdx.x + k * (int)gridDim.x, p);
            const int a = p.nacc == 2 ? (k & 1) : 0;
            const int use = p.nacc == 2 ? (k >> 1) : k;
            if (ok && !dev::mbar_wait_bounded(&acc_full[a], use & 1, kWaitLimitNs)) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);        // warp-uniform before .sync.aligned loads
            tc::fence_after();
            const int m = ew * 32 + lane;
            const int qh = u.qhb * p.MH + m / p.QW, qw = m % p.QW;
            const int od = 2 * u.qd + u.rd;
            const uint32_t tbase = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)a * p.acc_cols;
            bool released = false;
            for (int ci = half; ci < nchunk; ci += EPW) {
                const int c0 = ci * 16;
#pragma unroll
                for (int rh = 0; rh < 2; ++rh) {
                    const int oh = 2 * qh + rh;
                    const bool valid = od < p.Lo0 && oh < p.Lo1;
                    const int64_t off =
                        (int64_t)u.n * p.C_out * sp + ((int64_t)od * p.Lo1 + oh) * p.Lo2 + 2 * qw + (int64_t)c0 * sp;
                    float2 av[16];
                    if (ADD) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            av[i] = (ok && valid) ? __ldcs(reinterpret_cast<const float2 *>(add + off + (int64_t)i * sp))
                                                  : make_float2(0.f, 0.f);
                    }
                    float v0[16], v1[16];
                    if (ok) {
                        tc::tmem_ld16(tbase + (uint32_t)((rh * 2) * p.C_out + c0), v0);
                        tc::tmem_ld16(tbase + (uint32_t)((rh * 2 + 1) * p.C_out + c0), v1);
                        tc::tmem_wait_ld();
                    }
                    if (rh == 1 && ci + EPW >= nchunk) {   // the warp's last loads: free the accumulators
                        tc::fence_before();
                        dev::mbar_arrive(&acc_empty[a]);
                        released = true;
                    }
                    if (ok && valid) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float bb = bias ? __ldg(bias + c0 + i) : 0.f;
                            float t0 = v0[i] + bb, t1 = v1[i] + bb;
                            if (ADD) {
                                t0 = add_hswish(t0, av[i].x);
                                t1 = add_hswish(t1, av[i].y);
                            }
                            __stcs(reinterpret_cast<float2 *>(y + off + (int64_t)i * sp), make_float2(t0, t1));
                        }
                    }
                }
            }
            if (!released) {                          // a warp without chunks (C_out < 32)
                tc::fence_before();
                dev::mbar_arrive(&acc_empty[a]);
            }
        }
    }

    __syncwarp();
    tc::fence_before();
    __syncthreads();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, p.tmem_cols);
}

// ---- host side ------------------------------------------------------------------
struct T3Plan {
    T3Params p;
    size_t x_bytes, w_bytes, smem;
    int ntap;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Taps of residue r in one stride-2, dilation-1 dimension: k with (r + P - k)
// even, input offset (r + P - k) / 2 (exact).
int dim_taps(int K, int P, int r, int *k_out, int *d_out)
{
    int n = 0;
    for (int k = 0; k < K; ++k) {
        const int num = r + P - k;
        if (((num % 2) + 2) % 2 != 0) continue;
        k_out[n] = k;
        d_out[n] = num / 2;     // even numerator: exact for negative values too
        ++n;
    }
    return n;
}

bool make_t3plan(const Problem &pb, const Args *a, T3Plan *out)
{
    if (pb.nd != 3 || pb.dtype != CT_F32 || pb.G != 1) return false;
    for (int d = 0; d < 3; ++d)
        if (pb.S[d] != 2 || pb.DL[d] != 1 || pb.K[d] < 2 || pb.K[d] > 4) return false;
    if (pb.C_in % CK != 0 || pb.C_out % 16 != 0 || pb.C_out < 16 || pb.C_out > 128) return false;
    if (pb.Lo[2] % 2 != 0 || pb.in_sp() % 4 != 0) return false;
    if (a && (((uintptr_t)a->x % 16) || ((uintptr_t)a->y % 8) || (a->add && ((uintptr_t)a->add % 8))))
        return false;
    T3Params p;
    memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C_in = pb.C_in; p.C_out = pb.C_out;
    p.Lo0 = pb.Lo[0]; p.Lo1 = pb.Lo[1]; p.Lo2 = pb.Lo[2];
    p.QW = p.Lo2 / 2;
    if (p.QW > BM || BM % p.QW != 0) return false;
    p.MH = BM / p.QW;
    p.QD = (p.Lo0 + 1) / 2;
    p.QH = (p.Lo1 + 1) / 2;
    p.n_qhb = (p.QH + p.MH - 1) / p.MH;
    p.n_kb = pb.C_in / CK;
    const int64_t units = (int64_t)pb.N * p.QD * p.n_qhb * 2;
    if (units > 0x7fffffff || units == 0) return false;
    p.nunits = (int)units;

    // per dimension and residue: taps and input offsets
    int tk[3][2][4], td[3][2][4], nt[3][2];
    for (int d = 0; d < 3; ++d)
        for (int r = 0; r < 2; ++r) {
            nt[d][r] = dim_taps(pb.K[d], pb.P[d], r, tk[d][r], td[d][r]);
            if (nt[d][r] < 1) return false;       // every phase must receive a tap
        }
    // distinct offsets of H and W over both residues
    int uo[3][4], nu[3] = {0, 0, 0};
    for (int d = 1; d < 3; ++d)
        for (int r = 0; r < 2; ++r)
            for (int j = 0; j < nt[d][r]; ++j) {
                bool seen = false;
                for (int i = 0; i < nu[d]; ++i) seen = seen || uo[d][i] == td[d][r][j];
                if (!seen) {
                    if (nu[d] >= 4) return false;
                    uo[d][nu[d]++] = td[d][r][j];
                }
            }
    for (int rd = 0; rd < 2; ++rd) {
        int ne = 0;
        for (int jd = 0; jd < nt[0][rd]; ++jd)
            for (int ih = 0; ih < nu[1]; ++ih)
                for (int iw = 0; iw < nu[2]; ++iw) {
                    AEntry en;
                    memset(&en, 0, sizeof(en));
                    en.dd = (int8_t)td[0][rd][jd];
                    en.dh = (int8_t)uo[1][ih];
                    en.dw = (int8_t)uo[2][iw];
                    for (int rh = 0; rh < 2; ++rh)
                        for (int jh = 0; jh < nt[1][rh]; ++jh) {
                            if (td[1][rh][jh] != en.dh) continue;
                            for (int rw = 0; rw < 2; ++rw)
                                for (int jw = 0; jw < nt[2][rw]; ++jw) {
                                    if (td[2][rw][jw] != en.dw) continue;
                                    if (en.nuse >= 4) return false;
                                    const int tap = (tk[0][rd][jd] * pb.K[1] + tk[1][rh][jh]) * pb.K[2] + tk[2][rw][jw];
                                    en.tap[en.nuse] = (int8_t)tap;
                                    en.ph[en.nuse] = (int8_t)(rh * 2 + rw);
                                    ++en.nuse;
                                }
                        }
                    if (en.nuse == 0) continue;
                    if (ne >= MAXE) return false;
                    p.ent[rd][ne++] = en;
                }
        p.nA[rd] = ne;
    }
    p.acc_cols = (uint32_t)(4 * pb.C_out);
    p.nacc = 8 * pb.C_out <= 512 ? 2 : 1;
    uint32_t cols = 32;
    while (cols < (uint32_t)p.nacc * p.acc_cols) cols <<= 1;
    p.tmem_cols = cols;
    p.idesc = tc::idesc(2, pb.C_out, BM);
    p.b_bytes = (uint32_t)pb.C_out * CK * 4;
    const size_t budget = 227 * 1024 - 2048;           // alignment slack, static shared memory
    const size_t a_area = (size_t)NA * 2 * kATile;
    if (budget < a_area) return false;
    int nb = (int)((budget - a_area) / (2 * p.b_bytes));
    if (nb > MAXB) nb = MAXB;
    nb -= nb % NPB;                                     // one producer per B slot
    if (nb < NPB || nb < 2) return false;
    p.nb = nb;
    out->p = p;
    out->ntap = pb.kvol();
    out->x_bytes = align256((size_t)pb.N * pb.C_in * pb.in_sp() * 4);
    out->w_bytes = align256((size_t)out->ntap * 2 * pb.C_out * pb.C_in * 4);   // hi and lo panels
    out->smem = a_area + (size_t)nb * 2 * p.b_bytes + 1024;
    return true;
}

}  // namespace

bool tc3d_supported(const Problem &pb, const Args *a)
{
    T3Plan pl;
    return make_t3plan(pb, a, &pl);
}

size_t tc3d_workspace_bytes(const Problem &pb)
{
    T3Plan pl;
    if (!make_t3plan(pb, nullptr, &pl)) return 0;
    return 2 * pl.x_bytes + pl.w_bytes;
}

cudaError_t launch_tc3d(const Problem &pb, const Args &a)
{
    T3Plan pl;
    if (!make_t3plan(pb, &a, &pl)) return cudaErrorNotSupported;
    const T3Params &p = pl.p;
    uint8_t *ws = static_cast<uint8_t *>(a.ws);
    float *xhi = reinterpret_cast<float *>(ws);
    float *xlo = reinterpret_cast<float *>(ws + pl.x_bytes);
    float *wp = reinterpret_cast<float *>(ws + 2 * pl.x_bytes);

    // 1) x -> channels-last hi / lo
    const int64_t SP = pb.in_sp();
    dim3 gx((unsigned)((SP + 63) / 64), (unsigned)(pb.C_in / 32), (unsigned)pb.N);
    if (gx.x > 0x7fffffffu || gx.y > 65535 || gx.z > 65535) return cudaErrorInvalidConfiguration;
    prep_x_kernel<<<gx, 256, 0, a.stream>>>(static_cast<const float *>(a.x), xhi, xlo, pb.C_in, SP);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2) weights -> per-tap K-major hi / lo
    const int64_t wtot = (int64_t)pl.ntap * pb.C_out * pb.C_in;
    int wblocks = (int)((wtot + 255) / 256);
    if (wblocks > 4 * sm_count()) wblocks = 4 * sm_count();
    prep_w_kernel<<<wblocks, 256, 0, a.stream>>>(static_cast<const float *>(a.w), wp, pb.C_in, pb.C_out, pl.ntap);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // 3) tensor maps: A over x_hi / x_lo (C, W, H, D, N), B over w_p (C_in, ntap*2*C_out)
    CUtensorMap tmXh, tmXl, tmW;
    const uint64_t adims[5] = {(uint64_t)pb.C_in, (uint64_t)pb.Li[2], (uint64_t)pb.Li[1], (uint64_t)pb.Li[0],
                               (uint64_t)pb.N};
    const uint64_t astr[4] = {(uint64_t)pb.C_in * 4, (uint64_t)pb.C_in * pb.Li[2] * 4,
                              (uint64_t)pb.C_in * pb.Li[2] * pb.Li[1] * 4,
                              (uint64_t)pb.C_in * pb.Li[2] * pb.Li[1] * pb.Li[0] * 4};
    const uint32_t abox[5] = {(uint32_t)CK, (uint32_t)p.QW, (uint32_t)p.MH, 1u, 1u};
    const uint64_t bdims[2] = {(uint64_t)pb.C_in, (uint64_t)pl.ntap * 2 * pb.C_out};
    const uint64_t bstr[1] = {(uint64_t)pb.C_in * 4};
    const uint32_t bbox[2] = {(uint32_t)CK, (uint32_t)(2 * pb.C_out)};
    if (!encode_tiled(&tmXh, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, xhi, adims, astr, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmXl, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, xlo, adims, astr, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, wp, bdims, bstr, bbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    const void *fn = a.add ? (const void *)&tc3d_tf32_kernel<true> : (const void *)&tc3d_tf32_kernel<false>;
    int per_sm = 0;
    e = prepare_kernel(fn, kThreads, pl.smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    unsigned int *status = device_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    int grid = sm_count();
    if (grid > p.nunits) grid = p.nunits;
    if (a.add)
        tc3d_tf32_kernel<true><<<grid, kThreads, pl.smem, a.stream>>>(tmXh, tmXl, tmW, a.bias, a.add, a.y, p,
                                                                      status);
    else
        tc3d_tf32_kernel<false><<<grid, kThreads, pl.smem, a.stream>>>(tmXh, tmXl, tmW, a.bias, nullptr, a.y, p,
                                                                       status);
    return cudaGetLastError();
}

}  // namespace ct
