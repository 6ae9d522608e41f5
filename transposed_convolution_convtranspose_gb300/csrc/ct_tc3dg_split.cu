// ct_tc3dg_split.cu -- FP32 ConvTranspose3d with 32 input channels in 1, 2
// or 4 groups (asymmetric kernels up to 8 per dimension, any padding) on the
// tensor cores (tcgen05), every operand split into parts whose products the
// tensor cores form exactly.  Two splits, chosen by the caller:
//  * tf32x3 (CT_F32, the default): v = t + l with t = tf32(v) (cvt.rna) and
//    l = tf32(v - t), |v - t - l| <= 2^-22 |v|; per K step of 8 channels
//    three kind::tf32 MMAs accumulate a_t b_t + a_t b_l + a_l b_t, so an
//    output lies within about 2^-20 of sum |x||w| of the exact sum, the
//    accuracy of fp32 arithmetic over the same terms.  x_c holds per position
//    the t parts of the 32 channels (one 128-byte row), then their l parts
//    (a second row); a panel row holds the t (or l) parts of the weights.
//  * bf16x2 (CT_F32_BF16X2, opt-in): v = hi + lo with hi = bf16(v) and
//    lo = bf16(v - hi), leaving less than 2^-17 |v|.  Per K step the A row
//    holds [a_hi | a_lo] of 8 (or 16) channels and two MMAs multiply it by
//    [b_hi | b_hi] and by [b_lo | b_lo]: together (a_hi + a_lo)(b_hi + b_lo),
//    a relative error of about 2^-16 per product at most.
//
// Method ([l1_p72] stride-phase classes: residue r of a stride-2 dimension
// receives the taps k with (r + p - k) even, reading input q + (r + p - k)/2;
// and its grouped layer: output channel oc of group g sums over the input
// channels of group g only):
//     y[n, oc, 2q + r] = bias[oc] + sum over the phase's taps t and the group's
//                        input channels ic of x[n, ic, q + delta_t] * w[ic, oc_l, k_t]
// For one input offset (dd, dh, dw) every output phase (rD, rH, rW) that reads
// it with some tap contributes; with 128 positions q as the M rows, a group's
// contraction over its Cig = 32 / G channels is Cig / 8 K steps, each of
// three tf32 MMAs of K = 8 (or two bf16 MMAs of K = 16 over the hi and lo
// parts).
//
// Groups without block-diagonal zeros.  All 32 input channels of a position
// are one 128-byte row of the A operand (K-major, 128-byte swizzle), so group
// g's values are the K steps g * Cig/8 .. of that row: the MMAs of group g
// start their A and B descriptors Cig * 4 * g bytes into the rows.  The
// weight panels hold, in the same K positions of one row, the weights of
// every group for that row's (phase, output channel within the group).  One
// MMA-issuing warp per group owns that group's TMEM columns; all of them
// read the same operand stages.
//
// Accumulators: per group, the 8 phases x Cog channels, ordered (rD, rH, rW,
// oc_l), so the phases of one (rD, rH) pair -- both W residues -- are 2 x Cog
// adjacent columns.  An input offset is read by the pairs of a product set
// {rD reading dd} x {rH reading dh}; one MMA of N = 2 x Cog x pairs covers
// the range of pairs from the first to the last of the set (the W residue
// that does not read the offset, and a pair inside the range that does not,
// have zero weights in the panel: the issue rate of MMA instructions, not
// their width, bounds this kernel).  Two sets of accumulators (8 x C_out columns each)
// alternate across units; the epilogue clears a set after draining it, so
// every MMA accumulates.
//
// Operand A without shifted copies (the 128-byte swizzle is a function of the
// absolute shared-memory address): x is repacked channels-last with H fastest
// after the channels, (N, D, W, H, channels); per D offset one TMA box (two
// for tf32x3: the t rows, then the l rows) brings the unit's input window,
// (8 + H halo) x (16 + W halo) positions of 128 bytes, rows ordered (w, h).
// The A operand of offset (dh, dw) is that window read from row (dw - dw_lo)
// * hspan + (dh - dh_lo) with a stride of hspan rows between 8-row groups.  A
// unit is 16 qw x 8 qh positions of one D plane; TMEM row m holds (qw, qh) =
// (m / 8, m mod 8).
//
// Roles (persistent CTA, one per SM):
//   warp 0      TMA producer of the A ring (the window of a D offset)
//   warps 1-4   TMA producers of the B ring (one input offset's panel: hi
//               rows, then lo rows), one per slot
//   warps 5-12  MMA issue, two warps per group, each taking alternate entries
//               of every stage (one thread issues an MMA only every ~100
//               clocks, so the MMAs run from separate threads; the MMAs of a
//               group's two warps all accumulate into its columns, so their
//               order does not matter); TMEM allocation by warp 5
//   warps 13-20 epilogue, two per TMEM lane quarter: tcgen05.ld of a (group,
//               pair) block, zeros stored back, bias added.  When the output
//               has an even H extent, each 8-channel chunk (8 output rows of
//               the pair's H residue x 32 W outputs) is written into one of the
//               half's two staging buffers (128-byte rows, 128-byte swizzle);
//               otherwise each position's even and odd W outputs go out as one
//               float2 (a warp's store then covers 8 rows x 32 bytes)
//   warp 21     store warp (staged epilogue): one TMA store per chunk through
//               the map of y's rows of one H residue, then frees the buffer
// Every ring slot has exactly one producer, which refills it only after
// waiting for its previous round.  Every mbarrier wait is bounded: a timeout
// records CT_ERR_DEVICE_TIMEOUT in the device status word and the roles
// unwind (producers wait, bounded, for their own copies and the issuers for
// their own MMAs before the TMEM is freed).
#include <cuda_bf16.h>
#include <string.h>

#include "ct_internal.h"
#include "ct_device.cuh"
#include "ct_tma.h"
#include "ct_tcgen05.cuh"

namespace ct {
namespace {

constexpr int BM = 128;          // positions per unit (UMMA M)
constexpr int QWT = 16;          // qw per unit (TMEM row m: qw = m / 8)
constexpr int MHT = 8;           // qh per unit (one 8-row swizzle group per qw)
constexpr int CK = 32;           // input channels: one 128-byte row of tf32 parts or of bf16 (hi, lo) pairs
constexpr int NA = 3;            // A ring slots at most (one window each)
constexpr int MAXB = 8;          // B ring slots at most
constexpr int BROWS = 256;       // rows of a B stage at most (one 32 KB slot)
constexpr int NPB = 4;           // B producer warps at most
constexpr int MAXG = 4;          // groups at most
constexpr int IPG = 2;           // MMA-issuing warps per group: p.ipg of them take alternate entries of every stage
constexpr int MAXE = 64;         // input offsets per unit at most
constexpr int MAXDD = 5;         // distinct D offsets at most
constexpr int EPW = 2;           // epilogue warps per TMEM lane quarter
constexpr int kAWarp = 0;
constexpr int kBWarp0 = 1;
constexpr int kMmaWarp0 = kBWarp0 + NPB;
constexpr int kEpiWarp0 = kMmaWarp0 + MAXG * IPG;
constexpr int kStoreWarp = kEpiWarp0 + 4 * EPW;
constexpr int kThreads = 32 * (kStoreWarp + 1);
constexpr int kEpiThreads = 32 * 4 * EPW;
constexpr int NSB = 2;           // staging buffers per epilogue half
constexpr uint32_t kSChunk = 8 * MHT * 2 * QWT * 4;   // 8 channels x 8 rows x 32 W outputs, fp32: 8 KB
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// One input offset of a unit: the pairs (rD, rH) q0 .. q0 + nq - 1 receive
// its MMAs; its panel is 2 x R rows from row0 (hi rows, then lo rows),
// R = nq x 2 x Cog.
struct GEntry {
    int8_t dh, dw, q0, nq;
    int row0;
};

struct GParams {
    int N, C_out, G, Cig, Cog;
    int Lo0, Lo1, Lo2;
    int QD, QH, QW, n_qhb, n_qwb;
    int nunits;
    int ndd;                     // A stages per unit (distinct D offsets)
    int dd[MAXDD];               // D offset of A stage i
    int s0[MAXDD + 1];           // B stages of A stage i: s0[i] .. s0[i + 1]
    int ne;                      // input offsets (entries)
    int nbs;                     // B stages per unit: consecutive entries of one D offset
    int bs_e0[MAXE + 1];         // entries of B stage j: bs_e0[j] .. bs_e0[j + 1]
    int bs_units[MAXE];          // rows of B stage j in units of 4 x Cog rows
    int nb, npb;                 // B ring slots and producers (nb a multiple of npb)
    int hspan, wspan, dh_lo, dw_lo;
    uint32_t a_half;             // bytes of the window's rows of one kind (t or l; all of bf16x2), 1024-aligned
    uint32_t a_slot;             // bytes of one window: a_half (bf16x2) or 2 a_half (tf32x3: t rows, then l rows)
    uint32_t bslot;              // bytes of a B ring slot (the widest panel)
    uint32_t set_cols;           // 8 x C_out
    uint32_t tmem_cols;
    uint32_t idesc_b[5];         // instruction descriptor, N = 2 x Cog x pairs, pairs 1..4
    int na;                      // A ring slots
    int ipg;                     // issuers per group that issue MMAs (1: reproducible order; up to IPG)
    int stg;                     // staged epilogue: 8-channel chunks stored by TMA (else direct stores)
    GEntry ent[MAXE];
};

// Weight panel description for the prep kernel.
struct GPanels {
    int Cig, Cog, K0, K1, K2, ne, tf;
    int off_lo[3];               // smallest input offset per dimension
    int8_t tap[3][2][8];         // tap of residue r reading offset off_lo + i (-1: none)
    int8_t edd[MAXE], edh[MAXE], edw[MAXE], eq0[MAXE], enq[MAXE], emask[MAXE];   // emask: pairs reading it
    int erow0[MAXE];
};

__device__ __forceinline__ uint32_t bf16_bits(float v)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float bf16_round(float v)
{
    return __bfloat162float(__float2bfloat16_rn(v));
}
// v rounded to tf32 (10 fraction bits, nearest, ties away from zero): the low
// 13 bits are zero, so the tensor cores read it exactly
__device__ __forceinline__ float tf32_round(float v)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// K-major, 128-byte swizzled operand with 8-row groups `sbo` bytes apart
__device__ __forceinline__ uint64_t desc_sbo(uint32_t saddr, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;                       // leading byte offset (unused)
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;   // stride byte offset
    d |= (uint64_t)1 << 46;                       // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                       // 128-byte swizzle
    return d;
}

// ---- prep kernels --------------------------------------------------------------
// x (N, 32, D, H, W) -> x_c (N, D, W, H, channels): tf32x3 64 fp32 words
// per position, [t of the 32 channels | l of them]; bf16x2 64 bf16, per group
// [hi of its Cig channels | lo of them].  Block = 32 channels x 64
// consecutive source positions (16-byte loads along W, a shared tile of pitch
// 33); a thread then writes 4 channels of one position: two stores of their
// two parts.  D*H*W is a multiple of 4.
__device__ __forceinline__ void prepg_x_block(const float *__restrict__ x, uint16_t *__restrict__ xc, int D, int H,
                                              int W, int Cig, int bx, int n, bool tf)
{
    __shared__ float tile[64][33];
    const int64_t SP = (int64_t)D * H * W;
    const int64_t s0 = (int64_t)bx * 64;
    const int ncols = (int)((SP - s0) < 64 ? (SP - s0) : 64);
    const float *xs = x + (int64_t)n * CK * SP + s0;
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
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = threadIdx.x + 256 * it;
        const int q = idx & 7, pos = idx >> 3;
        if (pos < ncols) {
            const int64_t s = s0 + pos;
            int w, h, d;
            if (SP <= 0x7fffffff) {                 // 32-bit divisions where the image allows
                const int si = (int)s;
                w = si % W;
                h = (si / W) % H;
                d = si / (W * H);
            } else {
                w = (int)(s % W);
                h = (int)((s / W) % H);
                d = (int)(s / ((int64_t)W * H));
            }
            const int64_t prow = (((int64_t)n * D + d) * W + w) * H + h;
            if (tf) {
                float t[4], l[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float v = tile[pos][4 * q + i];
                    t[i] = tf32_round(v);
                    l[i] = tf32_round(v - t[i]);    // v - t is exact in fp32
                }
                float *cr = reinterpret_cast<float *>(xc) + prow * (2 * CK) + 4 * q;
                *reinterpret_cast<float4 *>(cr) = make_float4(t[0], t[1], t[2], t[3]);
                *reinterpret_cast<float4 *>(cr + CK) = make_float4(l[0], l[1], l[2], l[3]);
                continue;
            }
            uint32_t hb[4], lb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float v = tile[pos][4 * q + i];
                const float hv = bf16_round(v);
                hb[i] = bf16_bits(hv);
                lb[i] = bf16_bits(v - hv);      // v - hv is exact in fp32
            }
            // channels 4q..4q+3 lie in one group g: hi at g*2Cig + i, lo Cig further
            const int c0 = 4 * q, g = c0 / Cig, i0 = c0 % Cig;
            uint16_t *cr = xc + prow * (2 * CK) + g * 2 * Cig + i0;
            *reinterpret_cast<uint2 *>(cr) = make_uint2(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16));
            *reinterpret_cast<uint2 *>(cr + Cig) = make_uint2(lb[0] | (lb[1] << 16), lb[2] | (lb[3] << 16));
        }
    }
}

// w (32, Cog, K0, K1, K2) -> panels.  Blocks (entry e, part hl, slice z), rows
// rr = (pair index i, rW, oc_l) of the entry; the weight of a row for input
// channel ic is w[ic][oc_l][kd][kh][kw] for the tap of phase (q0 + i, rW)
// reading the entry's offset, zero where that phase reads none.  tf32x3: 32
// fp32 words per row, the t parts (part 0) or l parts (part 1) of the 32
// input channels.  bf16x2: 64 bf16 per row, per group: part 0 [hi of its Cig
// channels | hi again], part 1 [lo | lo], the partners of the [hi | lo] order
// of x_c.
constexpr int kWSlices = 8;      // blocks per (entry, part) of the panel prep

__device__ __forceinline__ void prepg_w_block(const float *__restrict__ w, uint8_t *__restrict__ wp,
                                              const GPanels &q, int e, int hl, int z)
{
    const int R = q.enq[e] * 2 * q.Cog;
    const int ncol = q.tf ? CK : 2 * CK;
    for (int idx = threadIdx.x + z * blockDim.x; idx < R * ncol; idx += blockDim.x * kWSlices) {
        const int rr = idx / ncol, k = idx % ncol;
        const int i = rr / (2 * q.Cog);
        const int rW = (rr / q.Cog) & 1, oc_l = rr % q.Cog;
        const int pq = q.eq0[e] + i;
        const int rD = pq >> 1, rH = pq & 1;
        const int kd = q.tap[0][rD][q.edd[e] - q.off_lo[0]];
        const int kh = q.tap[1][rH][q.edh[e] - q.off_lo[1]];
        const int kw = q.tap[2][rW][q.edw[e] - q.off_lo[2]];
        const int g = k / (2 * q.Cig), within = k % (2 * q.Cig);
        const int ic = q.tf ? k : g * q.Cig + (within % q.Cig);
        float v = 0.f;
        if (((q.emask[e] >> pq) & 1) && kd >= 0 && kh >= 0 && kw >= 0)
            v = __ldg(w + (((int64_t)ic * q.Cog + oc_l) * q.K0 + kd) * (q.K1 * q.K2) + kh * q.K2 + kw);
        uint8_t *row = wp + ((int64_t)q.erow0[e] + hl * R + rr) * 128;
        if (q.tf) {
            const float t = tf32_round(v);
            reinterpret_cast<float *>(row)[k] = hl ? tf32_round(v - t) : t;
        } else {
            const float hv = bf16_round(v);
            reinterpret_cast<uint16_t *>(row)[k] = (uint16_t)bf16_bits(hl ? v - hv : hv);
        }
    }
}

// Both preps in one launch: blocks [0, nxb) move x (nbx per image), the rest
// build the panels (kWSlices per (entry, part)).  The GEMM kernel is launched
// as its programmatic dependent, so its CTAs may be scheduled while this
// kernel drains.
__global__ void __launch_bounds__(256)
prepg_kernel(const float *__restrict__ x, uint16_t *__restrict__ xc, int D, int H, int W,
             int Cig, int nbx, int nxb, const float *__restrict__ w, uint8_t *__restrict__ wp,
             const __grid_constant__ GPanels q)
{
    dev::griddep_launch_dependents();
    const int b = (int)blockIdx.x;
    if (b < nxb) {
        prepg_x_block(x, xc, D, H, W, Cig, b % nbx, b / nbx, q.tf != 0);
    } else {
        const int r = b - nxb;
        prepg_w_block(w, wp, q, r / (2 * kWSlices), (r / kWSlices) & 1, r % kWSlices);
    }
}

// ---- GEMM kernel -----------------------------------------------------------------
// unit -> (n, qd, qh block, qw block)
struct GUnit {
    int n, qd, qhb, qwb;
};
__device__ __forceinline__ GUnit g_unit(int u, const GParams &p)
{
    GUnit c;
    c.qwb = u % p.n_qwb;
    u /= p.n_qwb;
    c.qhb = u % p.n_qhb;
    u /= p.n_qhb;
    c.qd = u % p.QD;
    c.n = u / p.QD;
    return c;
}

template <bool TF>
__global__ void __launch_bounds__(kThreads, 1)
tc3dg_split_kernel(const __grid_constant__ CUtensorMap tmXc,
                  const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW4,
                  const __grid_constant__ CUtensorMap tmY, const float *__restrict__ bias,
                  float *__restrict__ y, const __grid_constant__ GParams p, unsigned int *status)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t a_full[NA], a_empty[NA], b_full[MAXB], b_empty[MAXB], acc_full[2],
        acc_empty[2], drain_bar[MAXG * IPG], c_done[2][NSB], e_free[2][NSB];
    __shared__ uint32_t tmem_slot;
    __shared__ float s_bias[64];
    // per entry: A window offset, B offset in its stage, hi -> lo rows, TMEM
    // column within the group; instruction descriptor
    __shared__ uint4 s_ent[MAXE];
    __shared__ uint32_t s_id[MAXE];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = sm;                                  // na x a_slot
    uint8_t *sB = sm + (size_t)p.na * p.a_slot;        // nb x bslot
    uint8_t *sE = sB + (size_t)p.nb * p.bslot;         // 2 x NSB x kSChunk (staged epilogue)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&tmXc);
        dev::prefetch_tensormap(&tmW1);
        dev::prefetch_tensormap(&tmW4);
        if (p.stg) dev::prefetch_tensormap(&tmY);
        // a stage is released by every group's issuer, a set of accumulators by
        // every epilogue thread; a staged chunk is written by the 128 threads of
        // its epilogue half and freed by the store warp
        for (int h = 0; h < 2; ++h)
            for (int b = 0; b < NSB; ++b) {
                dev::mbar_init(&c_done[h][b], 32 * 4);
                dev::mbar_init(&e_free[h][b], 1);
            }
        for (int s = 0; s < p.na; ++s) {
            dev::mbar_init(&a_full[s], 1);
            dev::mbar_init(&a_empty[s], G * IPG);
        }
        for (int s = 0; s < p.nb; ++s) {
            dev::mbar_init(&b_full[s], 1);
            dev::mbar_init(&b_empty[s], G * IPG);
        }
        for (int a = 0; a < 2; ++a) {
            dev::mbar_init(&acc_full[a], G * IPG);
            dev::mbar_init(&acc_empty[a], kEpiThreads);
        }
        for (int j = 0; j < MAXG * IPG; ++j) dev::mbar_init(&drain_bar[j], 1);
        dev::fence_mbar_init();
    }
    if (warp == kMmaWarp0) tc::tmem_alloc(&tmem_slot, p.tmem_cols);
    for (int i = threadIdx.x; i < p.C_out; i += blockDim.x) s_bias[i] = bias ? bias[i] : 0.f;
    for (int j = threadIdx.x; j < p.nbs; j += blockDim.x) {
        const int rb = p.ent[p.bs_e0[j]].row0;
        for (int e = p.bs_e0[j]; e < p.bs_e0[j + 1]; ++e) {
            const GEntry &en = p.ent[e];
            s_ent[e] = make_uint4((uint32_t)((en.dw - p.dw_lo) * p.hspan + (en.dh - p.dh_lo)) * 128u,
                                  (uint32_t)(en.row0 - rb) * 128u, (uint32_t)(en.nq * 2 * p.Cog) * 128u,
                                  (uint32_t)(en.q0 * 2 * p.Cog));
            s_id[e] = p.idesc_b[en.nq];
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = tmem_slot;
    const int nunit_cta =
        p.nunits > (int)blockIdx.x ? (p.nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    // the operands in the workspace come from the prep kernel
    dev::griddep_wait();

    if (warp == kAWarp || (warp >= kBWarp0 && warp < kBWarp0 + NPB)) {
        // ---------------- TMA producers
        const bool isA = warp == kAWarp;
        const int q = isA ? 0 : warp - kBWarp0;
        if (lane == 0 && (isA || q < p.npb)) {
            const int np = isA ? 1 : p.npb;
            const int nst = isA ? p.na : p.nb;
            const int sp = isA ? p.ndd : p.nbs;
            uint64_t *fullb = isA ? a_full : b_full;
            uint64_t *emptyb = isA ? a_empty : b_empty;
            const int total = nunit_cta * sp;
            int last = -1, kc = -1;
            bool failed = false;
            GUnit u;
            u.n = u.qd = u.qhb = u.qwb = 0;
            for (int gi = q; gi < total; gi += np) {
                const int k = gi / sp, i = gi % sp;
                if (k != kc) {
                    kc = k;
                    u = g_unit((int)blockIdx.x + k * (int)gridDim.x, p);
                }
                const int s = gi % nst;
                if (gi >= nst && !dev::mbar_wait_bounded(&emptyb[s], ((gi / nst) - 1) & 1, kWaitLimitNs)) {
                    failed = true;
                    break;
                }
                if (isA) {
                    // x_c viewed as (C, H, W, D, N): the window of D offset dd[i] (tf32x3:
                    // the t rows, then the l rows a_half further)
                    const int h0 = u.qhb * MHT + p.dh_lo, w0 = u.qwb * QWT + p.dw_lo, d0 = u.qd + p.dd[i];
                    dev::mbar_arrive_expect_tx(&fullb[s], (uint32_t)((TF ? 2 : 1) * p.hspan * p.wspan) * 128u);
                    dev::tma_load_5d(sA + (size_t)s * p.a_slot, &tmXc, &fullb[s], 0, h0, w0, d0, u.n);
                    if (TF)
                        dev::tma_load_5d(sA + (size_t)s * p.a_slot + p.a_half, &tmXc, &fullb[s], CK, h0, w0, d0,
                                         u.n);
                } else {
                    // the stage's panels (consecutive rows): boxes of 4 and of 1 unit
                    const int units = p.bs_units[i];
                    const int row0 = p.ent[p.bs_e0[i]].row0;
                    const int ur = 4 * p.Cog;
                    dev::mbar_arrive_expect_tx(&fullb[s], (uint32_t)(units * ur) * 128u);
                    uint8_t *dst = sB + (size_t)s * p.bslot;
                    int uu = 0;
                    for (; uu + 4 <= units; uu += 4)
                        dev::tma_load_2d(dst + (size_t)uu * ur * 128, &tmW4, &fullb[s], 0, row0 + uu * ur);
                    for (; uu < units; ++uu)
                        dev::tma_load_2d(dst + (size_t)uu * ur * 128, &tmW1, &fullb[s], 0, row0 + uu * ur);
                }
                last = gi;
            }
            if (failed) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                // let this warp's copies still in flight land before shared memory goes away
                for (int r = last; r >= 0 && r > last - nst; r -= np)
                    dev::mbar_wait_bounded(&fullb[r % nst], (r / nst) & 1, kWaitLimitNs);
            }
        }
    } else if (warp < kMmaWarp0 + MAXG * IPG) {
        // ---------------- MMA issuers, IPG warps per group; p.ipg of them issue, each
        // taking the entries e with e mod p.ipg == its index (the others only keep
        // the barrier protocol): every MMA accumulates (the epilogue leaves the set
        // cleared)
        const int wi = warp - kMmaWarp0, g = wi / IPG, sub = wi % IPG;
        if (lane == 0 && g < G) {
            bool ok = true;
            const uint32_t sAb = dev::smem_u32(sA), sBb = dev::smem_u32(sB);
            const uint32_t a_slot = p.a_slot, bslot = p.bslot, sbo = (uint32_t)p.hspan * 128u;
            const int Cog = p.Cog, ksteps = p.Cig / 8, nb = p.nb;
            // K step j of group g (tf32x3: 8 channels, 32 bytes of t or of l parts;
            // bf16x2: 16 bf16, hi or lo parts) sits (g * ksteps + j) * 32 bytes into
            // every row
            const uint64_t kgrp = (uint64_t)(g * ksteps * 2);         // in 16-byte units
            int sa = 0, sb = 0;
            uint32_t pa = 0, pb = 0;
            for (int k = 0; k < nunit_cta && ok; ++k) {
                const int set = k & 1;
                if (!dev::mbar_wait_bounded(&acc_empty[set], (k >> 1) & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t dg = tmem + (uint32_t)set * p.set_cols + (uint32_t)(g * 8 * Cog);
                for (int i = 0; i < p.ndd && ok; ++i) {
                    if (!dev::mbar_wait_bounded(&a_full[sa], pa, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t wc = sAb + (uint32_t)sa * a_slot;
                    for (int j = p.s0[i]; j < p.s0[i + 1] && ok; ++j) {
                        if (!dev::mbar_wait_bounded(&b_full[sb], pb, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after();
                        const uint32_t bb = sBb + (uint32_t)sb * bslot;
                        // with one issuing warp per group the MMAs into a column run in a fixed
                        // order (bitwise reproducible results); with two, in no fixed order
                        for (int e = p.bs_e0[j] + sub; sub < p.ipg && e < p.bs_e0[j + 1]; e += p.ipg) {
                            const uint4 t0 = s_ent[e];      // A offset, B offset, hi -> lo rows, column
                            const uint32_t id = s_id[e];    // instruction descriptor
                            const uint64_t da = desc_sbo(wc + t0.x, sbo) + kgrp;
                            const uint64_t dbh = tc::desc_sw128(bb + t0.y) + kgrp;
                            const uint64_t dbl = tc::desc_sw128(bb + t0.y + t0.z) + kgrp;
                            const uint32_t d = dg + t0.w;
                            if (TF) {
                                const uint64_t dal = desc_sbo(wc + p.a_half + t0.x, sbo) + kgrp;
                                for (int kk = 0; kk < ksteps; ++kk) {
                                    const uint64_t kj = (uint64_t)(2 * kk);   // 32 bytes: 8 channels
                                    tc::mma_tf32(d, da + kj, dbh + kj, id, 1u);    // a_t b_t
                                    tc::mma_tf32(d, da + kj, dbl + kj, id, 1u);    // a_t b_l
                                    tc::mma_tf32(d, dal + kj, dbh + kj, id, 1u);   // a_l b_t
                                }
                            } else {
                                for (int kk = 0; kk < ksteps; ++kk) {
                                    const uint64_t kj = (uint64_t)(2 * kk);   // 32 bytes: 16 bf16
                                    tc::mma_bf16(d, da + kj, dbh + kj, id, 1u);   // [a_hi|a_lo] x [b_hi|b_hi]
                                    tc::mma_bf16(d, da + kj, dbl + kj, id, 1u);   // [a_hi|a_lo] x [b_lo|b_lo]
                                }
                            }
                        }
                        tc::commit(&b_empty[sb]);
                        if (++sb == nb) {
                            sb = 0;
                            pb ^= 1u;
                        }
                    }
                    tc::commit(&a_empty[sa]);
                    if (++sa == p.na) {
                        sa = 0;
                        pa ^= 1u;
                    }
                }
                if (ok) tc::commit(&acc_full[set]);
            }
            // every MMA issued has to complete before the TMEM is freed
            tc::commit(&drain_bar[wi]);
            if (!dev::mbar_wait_bounded(&drain_bar[wi], 0, kWaitLimitNs)) ok = false;
            if (!ok) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
        }
    } else if (warp == kStoreWarp) {
        // ---------------- store warp (staged epilogue): each epilogue half writes its
        // chunks (8 channels of one (group, pair) block: 8 output rows of the pair's
        // H residue x 32 W outputs) into its two buffers in turn; this warp stores a
        // written chunk with one TMA store through the map of the rows of one H
        // residue (rows, planes and columns past the output are clipped) and frees
        // a buffer once its store has read it.  Chunks are taken in the order
        // (chunk index, half), the order the halves produce them.
        if (p.stg && lane == 0) {
            const int Cog = p.Cog, ncc = Cog / 8, nch = (G * 4 / 2) * ncc;   // chunks per half and unit
            bool ok = true;
            int issued = 0;
            for (int k = 0; k < nunit_cta && ok; ++k) {
                const GUnit u = g_unit((int)blockIdx.x + k * (int)gridDim.x, p);
                for (int jj = 0; jj < nch && ok; ++jj) {
                    const int gc = k * nch + jj;                 // the half's chunk counter
                    const int bi = gc % NSB;
                    for (int h = 0; h < 2; ++h) {
                        if (!dev::mbar_wait_bounded(&c_done[h][bi], (gc / NSB) & 1, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        const int b = h + 2 * (jj / ncc), c = (jj % ncc) * 8;   // block (group, pair), channels
                        const int g = b >> 2, pq = b & 3;
                        dev::tma_store_5d(&tmY, sE + (size_t)(h * NSB + bi) * kSChunk, 2 * u.qwb * QWT,
                                          u.qhb * MHT, pq & 1, 2 * u.qd + (pq >> 1),
                                          u.n * p.C_out + g * Cog + c);
                        dev::bulk_commit();
                        ++issued;
                        // the store issued two before this one (the same half's previous
                        // chunk) has read its buffer
                        dev::bulk_wait_read<2>();
                        if (gc >= 1) dev::mbar_arrive(&e_free[h][(gc - 1) % NSB]);
                    }
                }
            }
            dev::bulk_wait_all();
            if (!ok) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
            (void)issued;
        }
    } else {
        // ---------------- epilogue: EPW warps per TMEM lane quarter (32 positions:
        // 4 qw x 8 qh); half h of the warps takes the (group, pair) blocks of
        // parity h.  A block is 2 x Cog columns: W residue 0's channels, then W
        // residue 1's.  Both sets are cleared once before the first unit.
        // Staged: per 8 channels the half's four warps write the chunk's 8 KB (8
        // channels x 8 rows x 32 W outputs, 128-byte rows in the 128-byte swizzle)
        // into the half's next buffer and the store warp stores it: whole
        // 128-byte lines instead of a warp's 8 rows x 32 bytes.  Otherwise each
        // position's even and odd W outputs go out as one float2.
        const int ew = warp & 3;
        const int half = (warp - kEpiWarp0) >> 2;
        const int Cog = p.Cog, nblk = G * 4;
        const uint32_t lane_base = tmem + ((uint32_t)(ew * 32) << 16);
        const int64_t sp = (int64_t)p.Lo0 * p.Lo1 * p.Lo2;
        for (int set = 0; set < 2; ++set) {
            for (int b = half; b < nblk; b += 2)
                for (int c = 0; c < 2 * Cog; c += 8)
                    tc::tmem_st8_zero(lane_base + (uint32_t)set * p.set_cols + (uint32_t)(b * 2 * Cog + c));
            tc::tmem_wait_st();
            tc::fence_before();
            dev::mbar_arrive(&acc_empty[set]);
        }
        bool ok = true;
        int gc = 0;                                  // staged: this half's chunk counter
        for (int k = 0; k < nunit_cta; ++k) {
            const int set = k & 1;
            const GUnit u = g_unit((int)blockIdx.x + k * (int)gridDim.x, p);
            if (ok && !dev::mbar_wait_bounded(&acc_full[set], (k >> 1) & 1, kWaitLimitNs)) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);        // warp-uniform before .sync.aligned loads
            tc::fence_after();
            const int m = ew * 32 + lane;
            const int qwl = m >> 3, qhl = m & 7;
            const int qw = u.qwb * QWT + qwl, qh = u.qhb * MHT + qhl;
            const bool inw = qw < p.QW && qh < p.QH;
            const uint32_t sbase = lane_base + (uint32_t)set * p.set_cols;
            for (int b = half; b < nblk; b += 2) {
                const int g = b >> 2, pq = b & 3;
                const int od = 2 * u.qd + (pq >> 1), oh = 2 * qh + (pq & 1);
                const bool valid = inw && od < p.Lo0 && oh < p.Lo1;
                float *yrow = y + ((int64_t)u.n * p.C_out + g * Cog) * sp + ((int64_t)od * p.Lo1 + oh) * p.Lo2 + 2 * qw;
                for (int c = 0; c < Cog; c += 8) {
                    float v0[8], v1[8];
                    const uint32_t t0 = sbase + (uint32_t)(b * 2 * Cog + c);
                    if (ok) {
                        tc::tmem_ld8(t0, v0);
                        tc::tmem_ld8(t0 + (uint32_t)Cog, v1);
                        tc::tmem_wait_ld();
                        tc::tmem_st8_zero(t0);
                        tc::tmem_st8_zero(t0 + (uint32_t)Cog);
                    }
                    if (p.stg) {
                        // the buffer's previous chunk (two before) has been stored
                        const int bi = gc % NSB;
                        if (gc >= NSB && ok &&
                            !dev::mbar_wait_bounded(&e_free[half][bi], ((gc / NSB) - 1) & 1, kWaitLimitNs)) {
                            atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                            ok = false;
                        }
                        if (ok) {
                            // row qhl of channel i: 16-byte unit (qwl / 2) ^ qhl, the float2 of
                            // qwl at byte 8 (qwl & 1) within it
                            uint8_t *buf = sE + (size_t)(half * NSB + bi) * kSChunk;
                            const uint32_t off = (uint32_t)((((qwl >> 1) ^ qhl) << 4) + ((qwl & 1) << 3));
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float bb = s_bias[g * Cog + c + i];
                                *reinterpret_cast<float2 *>(buf + (size_t)(i * MHT + qhl) * 128 + off) =
                                    make_float2(v0[i] + bb, v1[i] + bb);
                            }
                        }
                        dev::fence_proxy_async();
                        dev::mbar_arrive(&c_done[half][bi]);
                        ++gc;
                    } else if (ok && valid) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float bb = s_bias[g * Cog + c + i];
                            __stcs(reinterpret_cast<float2 *>(yrow + (int64_t)(c + i) * sp),
                                   make_float2(v0[i] + bb, v1[i] + bb));
                        }
                    }
                }
            }
            tc::tmem_wait_st();
            tc::fence_before();
            dev::mbar_arrive(&acc_empty[set]);
        }
    }

    __syncwarp();
    tc::fence_before();
    __syncthreads();
    if (warp == kMmaWarp0) tc::tmem_dealloc(tmem, p.tmem_cols);
}

// ---- host side ---------------------------------------------------------------------
struct GPlan {
    GParams p;
    GPanels wq;
    int rows;                    // panel rows in all
    size_t x_bytes, w_bytes, smem;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Taps of residue r in one stride-2, dilation-1 dimension: k with (r + P - k)
// even, input offset (r + P - k) / 2 (exact).
int taps_of(int K, int P, int r, int *k_out, int *d_out)
{
    int n = 0;
    for (int k = 0; k < K; ++k) {
        const int num = r + P - k;
        if (((num % 2) + 2) % 2 != 0) continue;
        k_out[n] = k;
        d_out[n] = num / 2;
        ++n;
    }
    return n;
}

bool make_gplan_3d(const Problem &pb, const Args *a, GPlan *out);

// A unit D dimension (a 2-D call: one input plane, extent 1, stride 1, no
// padding) is the same operator as a D dimension of stride 2 and extent 1:
// one output plane, residue 0 takes tap 0 at offset 0, residue 1 no tap (its
// plane lies past the output).  The 2-D call is planned as that 3-D one.
bool make_gplan(const Problem &pb, const Args *a, GPlan *out)
{
    if (pb.cl) return false;
    if (pb.nd == 2 || (pb.S[0] == 1 && pb.Li[0] == 1)) {
        if (pb.Li[0] != 1 || pb.K[0] != 1 || pb.S[0] != 1 || pb.P[0] != 0 || pb.OP[0] != 0) return false;
        Problem q = pb;
        q.nd = 3;
        q.S[0] = 2;
        return make_gplan_3d(q, a, out);
    }
    return make_gplan_3d(pb, a, out);
}

bool make_gplan_3d(const Problem &pb, const Args *a, GPlan *out)
{
    if (pb.nd != 3 || pb.dtype != CT_F32 || pb.has_add) return false;
    const bool tf = !pb.split2;          // tf32x3 unless the caller opted into the bf16 pair
    for (int d = 0; d < 3; ++d)
        if (pb.S[d] != 2 || pb.DL[d] != 1 || pb.K[d] < 1 || pb.K[d] > 8) return false;
    if (pb.C_in != CK || (pb.G != 1 && pb.G != 2 && pb.G != 4)) return false;
    if (pb.Cog % 8 != 0 || pb.Cog > 16 || 16 * pb.C_out > 512) return false;
    if (pb.Lo[2] % 2 != 0 || pb.in_sp() % 4 != 0) return false;
    if (a && (((uintptr_t)a->x % 16) || ((uintptr_t)a->y % 8))) return false;
    GParams p;
    memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C_out = pb.C_out; p.G = pb.G; p.Cig = pb.Cig; p.Cog = pb.Cog;
    p.Lo0 = pb.Lo[0]; p.Lo1 = pb.Lo[1]; p.Lo2 = pb.Lo[2];
    p.QW = p.Lo2 / 2;
    p.QD = (p.Lo0 + 1) / 2;
    p.QH = (p.Lo1 + 1) / 2;
    p.n_qwb = (p.QW + QWT - 1) / QWT;
    p.n_qhb = (p.QH + MHT - 1) / MHT;
    const int64_t units = (int64_t)pb.N * p.QD * p.n_qhb * p.n_qwb;
    if (units > 0x7fffffff || units == 0) return false;
    p.nunits = (int)units;

    // per dimension and residue: taps and offsets; offsets per dimension
    int tk[3][2][4], td[3][2][4], nt[3][2], lo[3], hi[3];
    for (int d = 0; d < 3; ++d) {
        lo[d] = 1 << 20;
        hi[d] = -(1 << 20);
        for (int r = 0; r < 2; ++r) {
            nt[d][r] = taps_of(pb.K[d], pb.P[d], r, tk[d][r], td[d][r]);
            for (int j = 0; j < nt[d][r]; ++j) {
                lo[d] = td[d][r][j] < lo[d] ? td[d][r][j] : lo[d];
                hi[d] = td[d][r][j] > hi[d] ? td[d][r][j] : hi[d];
            }
        }
        if (hi[d] < lo[d] || hi[d] - lo[d] > 7) return false;
    }
    GPanels wq;
    memset(&wq, 0, sizeof(wq));
    memset(wq.tap, -1, sizeof(wq.tap));
    for (int d = 0; d < 3; ++d) {
        wq.off_lo[d] = lo[d];
        for (int r = 0; r < 2; ++r)
            for (int j = 0; j < nt[d][r]; ++j) wq.tap[d][r][td[d][r][j] - lo[d]] = (int8_t)tk[d][r][j];
    }
    // residues reading each offset: bit r of rd_mask[d][offset - lo]
    int rmask[3][8];
    memset(rmask, 0, sizeof(rmask));
    for (int d = 0; d < 3; ++d)
        for (int r = 0; r < 2; ++r)
            for (int j = 0; j < nt[d][r]; ++j) rmask[d][td[d][r][j] - lo[d]] |= 1 << r;
    // entries, grouped by D offset (one A stage each)
    int row = 0;
    int ent_first[MAXDD + 1];
    for (int od = 0; od <= hi[0] - lo[0]; ++od) {
        if (!rmask[0][od]) continue;
        if (p.ndd >= MAXDD) return false;
        p.dd[p.ndd] = lo[0] + od;
        ent_first[p.ndd] = p.ne;
        for (int oh = 0; oh <= hi[1] - lo[1]; ++oh) {
            if (!rmask[1][oh]) continue;
            for (int ow = 0; ow <= hi[2] - lo[2]; ++ow) {
                if (!rmask[2][ow]) continue;
                if (p.ne >= MAXE) return false;
                GEntry en;
                memset(&en, 0, sizeof(en));
                en.dh = (int8_t)(lo[1] + oh);
                en.dw = (int8_t)(lo[2] + ow);
                // pairs (rD, rH) reading the offset; the MMAs cover the range from
                // the first to the last (pairs inside it that do not read it get
                // zero weights)
                int mask = 0;
                for (int pq = 0; pq < 4; ++pq)
                    if (((rmask[0][od] >> (pq >> 1)) & 1) && ((rmask[1][oh] >> (pq & 1)) & 1)) mask |= 1 << pq;
                int q0 = 0, q1 = 3;
                while (!((mask >> q0) & 1)) ++q0;
                while (!((mask >> q1) & 1)) --q1;
                en.q0 = (int8_t)q0;
                en.nq = (int8_t)(q1 - q0 + 1);
                en.row0 = row;
                wq.edd[p.ne] = (int8_t)(lo[0] + od);
                wq.edh[p.ne] = en.dh;
                wq.edw[p.ne] = en.dw;
                wq.eq0[p.ne] = en.q0;
                wq.enq[p.ne] = en.nq;
                wq.emask[p.ne] = (int8_t)mask;
                wq.erow0[p.ne] = row;
                row += 2 * en.nq * 2 * pb.Cog;
                p.ent[p.ne++] = en;
            }
        }
        ++p.ndd;
        ent_first[p.ndd] = p.ne;
    }
    if (p.ne == 0) return false;
    // B stages: consecutive entries of one D offset, at most BROWS rows
    for (int i = 0; i < p.ndd; ++i) {
        p.s0[i] = p.nbs;
        int e = ent_first[i];
        while (e < ent_first[i + 1]) {
            p.bs_e0[p.nbs] = e;
            int rows = 0;
            while (e < ent_first[i + 1] && rows + 4 * p.ent[e].nq * pb.Cog <= BROWS) rows += 4 * p.ent[e].nq * pb.Cog, ++e;
            if (rows == 0) return false;
            p.bs_units[p.nbs] = rows / (4 * pb.Cog);
            ++p.nbs;
        }
    }
    p.s0[p.ndd] = p.nbs;
    p.bs_e0[p.nbs] = p.ne;
    wq.Cig = pb.Cig; wq.Cog = pb.Cog;
    wq.tf = tf ? 1 : 0;
    wq.K0 = pb.K[0]; wq.K1 = pb.K[1]; wq.K2 = pb.K[2];
    wq.ne = p.ne;
    // input windows
    p.dh_lo = lo[1];
    p.dw_lo = lo[2];
    p.hspan = MHT + hi[1] - lo[1];
    p.wspan = QWT + hi[2] - lo[2];
    p.a_half = (uint32_t)((p.hspan * p.wspan * 128 + 1023) & ~1023);
    p.a_slot = (tf ? 2 : 1) * p.a_half;
    for (int nq = 1; nq <= 4; ++nq) p.idesc_b[nq] = tc::idesc(tf ? 2 : 1, 2 * nq * pb.Cog, BM);
    p.set_cols = (uint32_t)(8 * pb.C_out);
    uint32_t cols = 32;
    while (cols < 2 * p.set_cols) cols <<= 1;
    p.tmem_cols = cols;
    p.bslot = (uint32_t)BROWS * 128u;
    const size_t budget = 227 * 1024 - 2048;
    // staged epilogue (TMA stores of whole 128-byte lines): the output rows of
    // one H residue as a tensor dimension need an even H extent, and rows of
    // 16-byte multiples; its 32 KB of buffers take the third A slot
    const bool stg = pb.Lo[1] % 2 == 0 && pb.Lo[2] % 4 == 0 && (!a || ((uintptr_t)a->y % 16) == 0);
    p.stg = stg ? 1 : 0;
    p.ipg = IPG;                 // the launch lowers it to 1 for reproducible results
    p.na = stg ? 2 : NA;
    const size_t e_area = stg ? (size_t)2 * NSB * kSChunk : 0;
    const size_t a_area = (size_t)p.na * p.a_slot;
    if (a_area + e_area + 2 * (size_t)p.bslot > budget) return false;
    int nb = (int)((budget - a_area - e_area) / p.bslot);
    if (nb >= 8) { nb = 8; p.npb = 4; }
    else if (nb >= 6) { nb = 6; p.npb = 3; }
    else if (nb >= 4) { nb = 4; p.npb = 4; }
    else p.npb = nb;
    p.nb = nb;
    out->p = p;
    out->wq = wq;
    out->rows = row;
    out->x_bytes = align256((size_t)pb.N * CK * pb.in_sp() * (tf ? 8 : 4));
    out->w_bytes = align256((size_t)row * CK * 4);
    out->smem = a_area + (size_t)nb * p.bslot + e_area + 1024;
    return true;
}

}  // namespace

bool tc3dg_supported(const Problem &pb, const Args *a)
{
    GPlan pl;
    return make_gplan(pb, a, &pl);
}

size_t tc3dg_workspace_bytes(const Problem &pb)
{
    GPlan pl;
    if (!make_gplan(pb, nullptr, &pl)) return 0;
    return pl.x_bytes + pl.w_bytes;
}

cudaError_t launch_tc3dg(const Problem &pb, const Args &a)
{
    GPlan pl;
    if (!make_gplan(pb, &a, &pl)) return cudaErrorNotSupported;
    const GParams &p = pl.p;
    uint8_t *ws = static_cast<uint8_t *>(a.ws);
    uint16_t *xc = reinterpret_cast<uint16_t *>(ws);
    uint8_t *wp = ws + pl.x_bytes;

    const bool tf = pl.wq.tf != 0;
    // 1) one launch: x -> (N, D, W, H, channels) split (tf32 [t x 32 | l x 32] or
    // bf16 [hi | lo] per group); weights -> one panel per input offset (hi / t
    // rows, then lo / l rows)
    const int64_t SP = pb.in_sp();
    const int64_t nbx = (SP + 63) / 64;
    const int64_t nxb = nbx * pb.N;
    const int64_t nblocks = nxb + (int64_t)p.ne * 2 * kWSlices;
    if (nblocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    prepg_kernel<<<(unsigned)nblocks, 256, 0, a.stream>>>(static_cast<const float *>(a.x), xc, pb.Li[0],
                                                         pb.Li[1], pb.Li[2], pb.Cig, (int)nbx, (int)nxb,
                                                         static_cast<const float *>(a.w), wp, pl.wq);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // 2) tensor maps: A over x_c viewed as (C, H, W, D, N), one window per box
    // (tf32x3: 64 fp32 words per position, a box of 32, the t or the l rows;
    // bf16x2: 64 bf16, one box), 128-byte rows; B over the panels (32 x 4
    // bytes, rows), boxes of 4 x Cog and 16 x Cog rows
    CUtensorMap tmXc, tmW[2];
    const uint64_t pb_bytes = tf ? 8 * CK : 4 * CK;     // bytes of x_c per position
    const uint64_t cdims[5] = {(uint64_t)(2 * CK), (uint64_t)pb.Li[1], (uint64_t)pb.Li[2], (uint64_t)pb.Li[0],
                               (uint64_t)pb.N};
    const uint64_t astr[4] = {pb_bytes, pb_bytes * pb.Li[1], pb_bytes * pb.Li[1] * pb.Li[2],
                              pb_bytes * pb.Li[1] * pb.Li[2] * pb.Li[0]};
    const uint32_t cbox[5] = {tf ? (uint32_t)CK : (uint32_t)(2 * CK), (uint32_t)p.hspan, (uint32_t)p.wspan, 1u, 1u};
    if (!encode_tiled(&tmXc, tf ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, xc, cdims,
                      astr, cbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const uint64_t bdims[2] = {(uint64_t)CK, (uint64_t)pl.rows};
    const uint64_t bstr[1] = {(uint64_t)CK * 4};
    for (int i = 0; i < 2; ++i) {
        // one unit (4 x Cog rows) and four units
        const uint32_t bbox[2] = {(uint32_t)CK, (uint32_t)(4 * (i == 0 ? 1 : 4) * pb.Cog)};
        if (!encode_tiled(&tmW[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, wp, bdims, bstr, bbox,
                          CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }

    // y for the staged epilogue: (W, H / 2, H residue, D, N x C_out), a box of a
    // chunk: 32 W outputs x 8 rows of one residue x 8 channels, 128-byte swizzle
    CUtensorMap tmY;
    memset(&tmY, 0, sizeof(tmY));
    if (p.stg) {
        const uint64_t ydims[5] = {(uint64_t)pb.Lo[2], (uint64_t)(pb.Lo[1] / 2), 2u, (uint64_t)pb.Lo[0],
                                   (uint64_t)pb.N * pb.C_out};
        const uint64_t ystr[4] = {(uint64_t)pb.Lo[2] * 8, (uint64_t)pb.Lo[2] * 4, (uint64_t)pb.Lo[2] * pb.Lo[1] * 4,
                                  (uint64_t)pb.out_sp() * 4};
        const uint32_t ybox[5] = {(uint32_t)(2 * QWT), (uint32_t)MHT, 1u, 1u, 8u};
        if (!encode_tiled(&tmY, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, a.y, ydims, ystr, ybox,
                          CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    int per_sm = 0;
    const void *fn = tf ? (const void *)&tc3dg_split_kernel<true> : (const void *)&tc3dg_split_kernel<false>;
    e = prepare_kernel(fn, kThreads, pl.smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    unsigned int *status = device_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    int grid = sm_count();
    if (grid > p.nunits) grid = p.nunits;
    // two issuing warps per group unless the caller asked for reproducible results
    GParams pk = p;
    pk.ipg = deterministic() ? 1 : IPG;
    if (tf)
        return launch_dependent(tc3dg_split_kernel<true>, dim3((unsigned)grid), dim3(kThreads), pl.smem, a.stream,
                                tmXc, tmW[0], tmW[1], tmY, a.bias, a.y, pk, status);
    return launch_dependent(tc3dg_split_kernel<false>, dim3((unsigned)grid), dim3(kThreads), pl.smem, a.stream,
                            tmXc, tmW[0], tmW[1], tmY, a.bias, a.y, pk, status);
}

}  // namespace ct
