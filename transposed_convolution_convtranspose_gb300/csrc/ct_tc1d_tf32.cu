// ct_tc1d_tf32.cu -- FP32 ConvTranspose1d on the tensor cores (tcgen05,
// kind::tf32) with a 3-term split that keeps fp32-level accuracy.
//
// Method ([l1_p79]: for k3 s2 p1 d2 every tap lands on the odd outputs, the
// even ones hold the bias; the gather index relation i = (o + p - k*d)/s):
// when the dilation is a multiple of the stride, every tap belongs to one
// residue class r* and output q of that class reads input i = q + e_j with
// e_j = base - j*(d/s).  Per tile of 128 outputs the sum over taps and input
// channels is one GEMM with K = taps x C_in:
//     y[s*q + r*][oc] = bias[oc] + sum_j sum_ic x[ic][q + e_j] * w[ic][oc][k_j]
// A tile is stored once, position-major, for positions q0-4 .. q0+131; the
// A operand of tap j is the same tile read from row 4 + e_j on: only the
// shared-memory descriptor's start address moves (the 128-byte swizzle
// follows absolute address bits, so the base-offset field stays 0), and no
// shifted copy is made.  The other residues hold the bias.
//
// Precision: each fp32 operand is split as v = hi + lo with hi = v rounded to
// tf32 (cvt.rna) and lo = v - hi (exact in fp32); three MMAs accumulate
// hi*hi + hi*lo + lo*hi in fp32 in TMEM.  The dropped lo*lo term and the
// tf32 rounding of lo are each below 2^-21 of a product.
//
// Roles (persistent CTA of 32 * (7 + 4 * EPW) threads, one per SM):
//   warp 0      TMA producer: x box [C_in = 32][136 positions] per tile (no
//               swizzle); positions outside the input read zeros
//   warps 1, 6  MMA issue (warp 1 also allocates the TMEM): taps x 4 K-steps
//               x 3 split terms of tcgen05.mma M=128, N=C_out, K=8 per tile
//               into one of two TMEM accumulators; warp 1 issues the even
//               tiles, warp 6 the odd ones, each with its own split stage and
//               accumulator (one issuing thread manages an MMA only every
//               ~140 clocks, which bounded the kernel with a single issuer)
//   warps 2-5   split + transpose: x box -> position-major (K-major) hi and lo
//               tiles, 128-byte swizzled; the weights once, per tap, the same way
//   warps 7..   epilogue, EPW warps per TMEM lane quarter (32 outputs q)
//               taking interleaved 16-channel chunks: tcgen05.ld, bias, and per channel
//               the s*32 consecutive outputs rebuilt by two warp shuffles and
//               written as two coalesced 128-byte stores
//               (y rows start at arbitrary 4-byte offsets, so no vector or
//               tensor store applies; every store instruction still covers
//               whole sectors except at its two ends)
// Every mbarrier wait is bounded; a timeout records CT_ERR_DEVICE_TIMEOUT in
// the device status word and the roles unwind.
#include <string.h>

#include "ct_internal.h"
#include "ct_device.cuh"
#include "ct_tma.h"

namespace ct {
namespace {

constexpr int EPW = 4;           // epilogue warps per TMEM lane quarter
constexpr int kEpiWarp0 = 7;     // warps 0-6: producer, MMA issuer 0, transposers, MMA issuer 1
constexpr int kThreads = 32 * (kEpiWarp0 + 4 * EPW);
constexpr int BM = 128;          // outputs per tile (UMMA M)
constexpr int PAD = 4;           // stored rows before the first output (16-byte TMA start)
constexpr int XR = BM + 2 * PAD; // stored input positions per tile
constexpr int CI = 32;           // input channels (one 128-byte K row)
constexpr int NS = 2;            // raw x-box stages (TMA destinations)
constexpr int NSS = 2;           // split (hi / lo K-major) stages: one per MMA issuer
constexpr int NACC = 2;          // TMEM accumulators: one per MMA issuer
constexpr int MAXT = 4;          // taps
constexpr int MAXS = 2;          // stride (an output run is s*128 long)
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct TParams {
    int N, C_in, C_out, Cog, K;
    int L_in, L_out, S;
    int nT;                      // taps
    int e[MAXT];                 // input offset of tap j: output q reads q + e_j
    int k_of[MAXT];              // kernel index of tap j
    int rstar;                   // residue receiving the taps
    int ntq;                     // tiles per row
    int ntiles;
    uint32_t tmem_cols;          // allocated TMEM columns (nacc accumulators of C_out)
    uint32_t idesc;
};

// ---- PTX wrappers ---------------------------------------------------------------
__device__ __forceinline__ float tf32_hi(float v)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// K-major, 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;                       // leading byte offset (unused)
    d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset
    d |= (uint64_t)1 << 46;                       // descriptor version (sm_100 family)
    // base offset 0: the swizzle follows the absolute shared-memory address, so a
    // start row inside an atom needs no phase correction
    d |= (uint64_t)2 << 61;                       // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                     dev::smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

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
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }


// byte offset of element (row, k) in a K-major 128-byte-swizzled tile of
// 32-bit elements (the 16-byte chunk index is XORed with the row's phase)
__device__ __forceinline__ uint32_t sw128_off(int row, int k)
{
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((k >> 2) ^ row) & 7) << 4) + (k & 3) * 4);
}

// ---- shared memory layout (offsets from a 1024-byte aligned base) ---------------
constexpr uint32_t kXRaw = CI * XR * 4;                  // TMA box [32][136] fp32
constexpr uint32_t kXK = XR * 128;                       // K-major 136 rows (17 atoms)
constexpr int kWRows = 256;                              // taps * C_out at most
constexpr uint32_t kWTile = kWRows * 128;
constexpr int kChunk = 16;                               // output channels per TMEM load

constexpr uint32_t OFF_XT = 0;
constexpr uint32_t OFF_XHI = OFF_XT + NS * kXRaw;     // NSS stages
constexpr uint32_t OFF_XLO = OFF_XHI + NSS * kXK;
constexpr uint32_t OFF_WHI = OFF_XLO + NSS * kXK;
constexpr uint32_t OFF_WLO = OFF_WHI + kWTile;
constexpr uint32_t kSmemBytes = OFF_WLO + kWTile + 1024;   // + alignment slack
static_assert(kXRaw % 1024 == 0 && kXK % 1024 == 0, "1024-byte aligned tiles");
static_assert(kSmemBytes <= 227 * 1024 - 256, "shared memory budget");
static_assert(NSS % 2 == 0 && NACC % 2 == 0, "issuer k mod 2 owns the split stages and accumulators of its parity");

__global__ void __launch_bounds__(kThreads, 1)
tc1d_tf32_kernel(const __grid_constant__ CUtensorMap tmx, const float *__restrict__ w,
                 const float *__restrict__ bias, float *__restrict__ y, const __grid_constant__ TParams p,
                 unsigned int *status)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_x[NS], xt_free[NS], split_x[NSS], empty_x[NSS], acc_full[NACC],
        acc_empty[NACC], w_ready;
    __shared__ uint32_t tmem_slot;
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&tmx);
        for (int s = 0; s < NS; ++s) {
            dev::mbar_init(&full_x[s], 1);
            dev::mbar_init(&xt_free[s], 128);
        }
        for (int s = 0; s < NSS; ++s) {
            dev::mbar_init(&split_x[s], 128);
            dev::mbar_init(&empty_x[s], 1);
        }
        for (int a = 0; a < NACC; ++a) {
            dev::mbar_init(&acc_full[a], 1);
            dev::mbar_init(&acc_empty[a], 128 * EPW);   // every epilogue thread
        }
        dev::mbar_init(&w_ready, 128);
        dev::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         dev::smem_u32(&tmem_slot)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = tmem_slot;
    const int ntile_cta =
        p.ntiles > (int)blockIdx.x ? (p.ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int issued = 0;
            bool failed = false;
            for (int k = 0; k < ntile_cta; ++k) {
                const int tile = blockIdx.x + k * gridDim.x;
                const int s = k % NS;
                if (k >= NS && !dev::mbar_wait_bounded(&xt_free[s], ((k / NS) - 1) & 1, kWaitLimitNs)) {
                    atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                    failed = true;
                    break;
                }
                const int n = tile / p.ntq, qt = tile % p.ntq;
                dev::mbar_arrive_expect_tx(&full_x[s], kXRaw);
                // x viewed as (L_in, C_in, N): positions q0 - PAD .. q0 + BM + PAD - 1
                dev::tma_load_3d(sm + OFF_XT + s * kXRaw, &tmx, &full_x[s], qt * BM - PAD, 0, n);
                ++issued;
            }
            if (failed)
                for (int k = issued - NS > 0 ? issued - NS : 0; k < issued; ++k)
                    dev::mbar_wait_bounded(&full_x[k % NS], (k / NS) & 1, kWaitLimitNs);
        }
    } else if (warp == 1 || warp == 6) {
        // ---------------- MMA issuers: warp 1 takes the even tiles of this CTA,
        // warp 6 the odd ones -- each owns the split stages and accumulators of
        // its parity; one thread issues an MMA only every ~140 clocks, so the two
        // issue streams run side by side.  (Two accumulators and two split
        // stages per issuer measured slower than one of each.)
        if (lane == 0) {
            bool ok = dev::mbar_wait_bounded(&w_ready, 0, kWaitLimitNs);
            const uint32_t whi = dev::smem_u32(sm + OFF_WHI), wlo = dev::smem_u32(sm + OFF_WLO);
            for (int k = warp == 1 ? 0 : 1; k < ntile_cta && ok; k += 2) {
                // tile k: x stage k mod 2 (this issuer's), accumulator k mod 4 (this
                // issuer alternates between its two)
                const int s = k % NSS, a = k % NACC;
                if (k >= NACC && !dev::mbar_wait_bounded(&acc_empty[a], ((k / NACC) - 1) & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                if (!dev::mbar_wait_bounded(&split_x[s], (k / NSS) & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_after();
                const uint32_t xhi = dev::smem_u32(sm + OFF_XHI + s * kXK);
                const uint32_t xlo = dev::smem_u32(sm + OFF_XLO + s * kXK);
                const uint32_t d = tmem + (uint32_t)(a * p.Cog);
                for (int j = 0; j < p.nT; ++j) {
                    const uint32_t arow = (uint32_t)(PAD + p.e[j]) * 128u;   // tap j's first row
                    const uint32_t boff = (uint32_t)(j * p.Cog) * 128u;        // tap j's weight rows
#pragma unroll
                    for (int kk = 0; kk < CI / 8; ++kk) {
                        const uint64_t ahi = desc_sw128(xhi + arow + kk * 32);
                        const uint64_t alo = desc_sw128(xlo + arow + kk * 32);
                        const uint64_t bhi = desc_sw128(whi + boff + kk * 32);
                        const uint64_t blo = desc_sw128(wlo + boff + kk * 32);
                        mma_tf32(d, ahi, bhi, p.idesc, (j > 0 || kk > 0) ? 1u : 0u);
                        mma_tf32(d, ahi, blo, p.idesc, 1u);
                        mma_tf32(d, alo, bhi, p.idesc, 1u);
                    }
                }
                mma_commit(&empty_x[s]);
                mma_commit(&acc_full[a]);
            }
            if (!ok) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
        }
    } else if (warp < 6) {
        // ---------------- split + transpose warps (128 threads: warps 2-5)
        const int st = threadIdx.x - 64;
        // weights once: tap j's rows j*Cog + oc, K = ic; hi/lo, K-major swizzled
        for (int e = st; e < p.nT * p.Cog * CI; e += 128) {
            const int n = e / CI, ic = e % CI;
            const int j = n / p.Cog, oc = n % p.Cog;
            const float v = __ldg(w + ((int64_t)ic * p.Cog + oc) * p.K + p.k_of[j]);
            const float hi = tf32_hi(v);
            const uint32_t off = sw128_off(n, ic);
            *reinterpret_cast<float *>(sm + OFF_WHI + off) = hi;
            *reinterpret_cast<float *>(sm + OFF_WLO + off) = v - hi;
        }
        fence_async_smem();
        dev::mbar_arrive(&w_ready);
        bool ok = true;
        for (int k = 0; k < ntile_cta; ++k) {
            const int s = k % NS, ss = k % NSS;
            if (ok && !dev::mbar_wait_bounded(&full_x[s], (k / NS) & 1, kWaitLimitNs)) ok = false;
            // the MMAs of tile k - NSS must be done reading split stage ss
            if (ok && k >= NSS && !dev::mbar_wait_bounded(&empty_x[ss], ((k / NSS) - 1) & 1, kWaitLimitNs))
                ok = false;
            if (!ok) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
            if (ok) {
                const float *xt = reinterpret_cast<const float *>(sm + OFF_XT + s * kXRaw);   // [ic][pos]
                uint8_t *xh = sm + OFF_XHI + ss * kXK;
                uint8_t *xl = sm + OFF_XLO + ss * kXK;
                for (int e = st; e < XR * (CI / 4); e += 128) {
                    const int pos = e % XR, cg = e / XR;
                    float4 hv, lv;
                    float *hp = &hv.x, *lp = &lv.x;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float v = xt[(4 * cg + u) * XR + pos];
                        const float hi = tf32_hi(v);
                        hp[u] = hi;
                        lp[u] = v - hi;
                    }
                    const uint32_t off = sw128_off(pos, 4 * cg);
                    *reinterpret_cast<float4 *>(xh + off) = hv;
                    *reinterpret_cast<float4 *>(xl + off) = lv;
                }
                fence_async_smem();
            }
            dev::mbar_arrive(&xt_free[s]);
            dev::mbar_arrive(&split_x[ss]);
        }
    } else {
        // ---------------- epilogue: EPW warps per TMEM lane quarter (32 rows =
        // 32 consecutive outputs q) taking interleaved 16-channel chunks; the
        // accumulator is released once the warp's last chunk is in registers,
        // then the stores run from registers.
        const int ew = warp & 3;                    // lanes 32*ew .. 32*ew + 31
        const int half = (warp - kEpiWarp0) >> 2;   // 0 .. EPW-1
        const int nchunk = p.Cog / kChunk;
        bool ok = true;
        for (int k = 0; k < ntile_cta; ++k) {
            const int tile = blockIdx.x + k * gridDim.x;
            const int n = tile / p.ntq, qt = tile % p.ntq;
            const int a = k % NACC;
            if (ok && !dev::mbar_wait_bounded(&acc_full[a], (k / NACC) & 1, kWaitLimitNs)) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);      // warp-uniform before .sync.aligned loads
            tc_after();
            // this warp's outputs: positions o_w .. o_w + s*32 - 1 of every channel row
            const int o_w = p.S * (qt * BM + 32 * ew);
            const int nv = min(p.S * 32, p.L_out - o_w);   // may be <= 0 past the end
            float *yw = y + (int64_t)n * p.C_out * p.L_out + o_w;
            // chunks half, half + EPW, ...: one TMEM load of 16 channels at a time
            // (compile-time register indices throughout: a runtime index into
            // the value array would put it in local memory)
            for (int ci = half; ci < nchunk; ci += EPW) {
                float v[16];
                if (ok) {
                    tmem_ld16(tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)(a * p.Cog + ci * kChunk), v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                }
                if (ci + EPW >= nchunk) {             // done with accumulator a
                    tc_before();
                    dev::mbar_arrive(&acc_empty[a]);
                }
                const int c0 = ci * kChunk;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int oc = c0 + i;
                    const float bb = bias ? __ldg(bias + oc) : 0.f;
                    float *row = yw + (int64_t)oc * p.L_out;
                    if (p.S == 2) {
                        // lane l writes positions o_w + l and o_w + 32 + l: output q
                        // (l >> 1) resp. 16 + (l >> 1) of this warp, residue l & 1
                        const float s0 = __shfl_sync(0xffffffffu, v[i], lane >> 1);
                        const float s1 = __shfl_sync(0xffffffffu, v[i], 16 + (lane >> 1));
                        const bool hit = (lane & 1) == p.rstar;
                        if (lane < nv) __stcs(row + lane, (hit ? s0 : 0.f) + bb);
                        if (32 + lane < nv) __stcs(row + 32 + lane, (hit ? s1 : 0.f) + bb);
                    } else {
                        if (lane < nv) __stcs(row + lane, v[i] + bb);
                    }
                }
            }
            if (half >= nchunk) {                     // a warp without chunks
                tc_before();
                dev::mbar_arrive(&acc_empty[a]);
            }
        }
    }

    tc_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(p.tmem_cols)
                     : "memory");
    }
}

// ---- host side --------------------------------------------------------------------
bool make_tplan(const Problem &pb, const Args *a, TParams *out)
{
    if (pb.nd != 1 || pb.dtype != CT_F32 || pb.G != 1) return false;
    const int S = pb.S[2], K = pb.K[2], DL = pb.DL[2], P = pb.P[2];
    if (S < 1 || S > MAXS || DL % S != 0 || K > MAXT) return false;
    if (pb.Cig != CI || pb.Cog % kChunk != 0 || pb.Cog > 256 || K * pb.Cog > kWRows) return false;
    if (pb.Li[2] % 4 != 0) return false;                 // TMA: 16-byte row strides of x
    if (a && (((uintptr_t)a->x % 16) || ((uintptr_t)a->y % 16))) return false;
    TParams p;
    memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C_in = pb.C_in; p.C_out = pb.C_out; p.Cog = pb.Cog; p.K = K;
    p.L_in = pb.Li[2]; p.L_out = pb.Lo[2]; p.S = S; p.nT = K;
    // every tap has k*dl == 0 (mod s): residue r* = (-p) mod s receives them,
    // tap k reads q + floor((r* + p)/s) - k*dl/s
    p.rstar = ((-P) % S + S) % S;
    const int base = (p.rstar + P) / S;
    for (int j = 0; j < K; ++j) {
        p.k_of[j] = j;
        p.e[j] = base - j * (DL / S);
        if (p.e[j] < -PAD || p.e[j] > PAD) return false;
    }
    const int nq = (p.L_out + S - 1) / S;
    p.ntq = (nq + BM - 1) / BM;
    const int64_t tiles = (int64_t)pb.N * p.ntq;
    if (tiles > 0x7fffffff) return false;
    p.ntiles = (int)tiles;
    uint32_t cols = 32;
    while (cols < (uint32_t)(NACC * pb.Cog)) cols <<= 1;
    p.tmem_cols = cols;
    // tcgen05 instruction descriptor: D fp32, A/B tf32, both K-major, N = C_out, M = 128
    p.idesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(pb.Cog >> 3) << 17) |
              ((uint32_t)(BM >> 4) << 24);
    *out = p;
    return true;
}

}  // namespace

bool tc1d_supported(const Problem &pb, const Args *a)
{
    TParams p;
    return make_tplan(pb, a, &p);
}

cudaError_t launch_tc1d(const Problem &pb, const Args &a)
{
    TParams p;
    if (!make_tplan(pb, &a, &p)) return cudaErrorNotSupported;
    CUtensorMap tmx;
    const uint64_t dims[3] = {(uint64_t)p.L_in, (uint64_t)p.C_in, (uint64_t)p.N};
    const uint64_t strides[2] = {(uint64_t)p.L_in * 4, (uint64_t)p.L_in * p.C_in * 4};
    const uint32_t box[3] = {(uint32_t)XR, (uint32_t)CI, 1u};
    if (!encode_tiled(&tmx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.x, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    int per_sm = 0;
    cudaError_t e = prepare_kernel((const void *)&tc1d_tf32_kernel, kThreads, kSmemBytes, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int grid = sm_count();
    if (grid > p.ntiles) grid = p.ntiles;
    unsigned int *status = device_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    tc1d_tf32_kernel<<<grid, kThreads, kSmemBytes, a.stream>>>(tmx, static_cast<const float *>(a.w), a.bias,
                                                               a.y, p, status);
    return cudaGetLastError();
}

}  // namespace ct
