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
//
// GEMM kernel: persistent, one CTA per SM, warp-specialised.  A tile is 128
// output positions (whole W rows of one D plane) of one (rD, rH) phase pair,
// with both W phases side by side along N (2 x C_out TMEM columns; two such
// accumulators alternate across tiles when they fit, so the epilogue of one
// tile overlaps the MMAs of the next).
//   warps 0-3  TMA producers, taking turns stage by stage (one thread's TMA
//              stream completes about one box at a time, so one producer
//              cannot keep the tensor cores fed).  A stage holds one A tile -- 128 positions x 64
//              input channels, a 5-D box of x_cl at the tap's input offset;
//              boxes reaching outside the input read zeros, which is the
//              boundary handling -- plus the B tiles (C_out x 64 of w_p) of
//              every W phase whose tap reads that same input offset, so an
//              input W offset both W phases read is fetched once for both.
//   warps 4-5  TMEM allocation and MMA issue, one warp per accumulator taking
//              alternate tiles (one thread issues an MMA only every ~100+
//              clocks; two warps nearly double the rate): tcgen05.mma
//              kind::f16 (M = 128, K = 16); one N = 2 x C_out MMA where both
//              W phases share the A tile, else N = C_out into the phase's half
//              of the accumulator.
//   warps 6-13 epilogue, two per TMEM lane quarter taking alternate
//              16-channel chunks: tcgen05.ld, bias, and each position's even
//              and odd W outputs written as one float2 (a warp writes two
//              whole 128-byte output rows per channel).
// Every mbarrier wait is bounded: a timeout records CT_ERR_DEVICE_TIMEOUT in
// the device status word and the roles unwind (the producer waits, bounded,
// for its own TMA copies and the MMA issuer for its own MMAs before the TMEM
// is freed).
#include <string.h>

#include "ct_internal.h"
#include "ct_device.cuh"
#include "ct_tma.h"
#include "ct_tcgen05.cuh"

namespace ct {
namespace {

constexpr int BM = 128;      // positions per tile (UMMA M)
constexpr int BK = 64;       // bf16 elements of K per stage (one 128-byte swizzle row)
constexpr int UK = 16;       // K of one tcgen05.mma kind::f16
constexpr int MAXST = 8;     // pipeline stages at most
constexpr int MAXWE = 5;     // distinct input W offsets of a tile at most (taps per dimension + 1)
constexpr int NPROD = 4;     // TMA producer warps at most (stage g is loaded by warp g mod nprod)
constexpr int EPW = 2;       // epilogue warps per TMEM lane quarter
constexpr int NMMA = 2;      // MMA-issuing warps at most (one per TMEM accumulator)
constexpr int kMmaWarp0 = NPROD;
constexpr int kEpiWarp0 = NPROD + NMMA;
constexpr int kThreads = 32 * (NPROD + NMMA + 4 * EPW);
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct UParams {
    int N, C_in, C_out;
    int Lo0, Lo1, Lo2;
    int QD, QH, QW, MH, n_qhb;
    int nT;                  // taps per dimension and class (kernel extent / 2)
    int n_kb;                // C_in / BK
    int ntiles;
    int nst;                 // pipeline stages (a multiple of nprod and of nacc)
    int nprod;               // producer warps in use: stage slot s is loaded only by warp s mod nprod
    int nacc;                // TMEM accumulators (1 or 2)
    uint32_t acc_cols;       // columns of one accumulator (2 x C_out)
    uint32_t tmem_cols;      // allocated TMEM columns (power of 2 >= nacc x acc_cols)
    uint32_t idesc1;         // instruction descriptor, N = C_out
    uint32_t idesc2;         // instruction descriptor, N = 2 x C_out (0: too wide)
    uint32_t a_bytes;        // A tile bytes
    uint32_t b_bytes;        // B tile bytes (one W phase)
    uint32_t stage_bytes;    // A + two B tiles
    int delta[3][2][4];      // input offset of tap j for residue r, per dimension
    // distinct input W offsets of a tile: offset we_delta[e] is read by tap
    // we_j[r][e] of W phase r (-1: phase r does not read it)
    int nwe;
    int we_delta[MAXWE];
    int we_j[2][MAXWE];
};

// tile -> (n, qd, qh block, rD, rH); the four (rD, rH) phases of one input
// region are neighbours, so their A tiles are reused from L2
struct TileCoord {
    int n, qd, qhb, rD, rH;
};
__device__ __forceinline__ TileCoord tile_coord(int t, const UParams &p)
{
    TileCoord c;
    c.rH = t & 1; t >>= 1;
    c.rD = t & 1; t >>= 1;
    c.qhb = t % p.n_qhb; t /= p.n_qhb;
    c.qd = t % p.QD; t /= p.QD;
    c.n = t;
    return c;
}

// ---- GEMM kernel -------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
umma_ct3d_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const float *__restrict__ bias, float *__restrict__ y, UParams p, unsigned int *status)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[MAXST], empty_bar[MAXST], acc_full[2], acc_empty[2], drain_bar[NMMA];
    __shared__ uint32_t tmem_slot;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&tmA);
        dev::prefetch_tensormap(&tmB);
        for (int s = 0; s < p.nst; ++s) {
            dev::mbar_init(&full_bar[s], 1);
            dev::mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            dev::mbar_init(&acc_full[a], 1);
            dev::mbar_init(&acc_empty[a], 32 * 4 * EPW);   // every epilogue thread
        }
        for (int j = 0; j < NMMA; ++j) dev::mbar_init(&drain_bar[j], 1);
        dev::fence_mbar_init();
    }
    if (warp == kMmaWarp0) tc::tmem_alloc(&tmem_slot, p.tmem_cols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = tmem_slot;
    const int ntile_cta =
        p.ntiles > (int)blockIdx.x ? (p.ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int stages_per_tile = p.nT * p.nT * p.n_kb * p.nwe;
    // With two accumulators, two warps issue MMAs, each for alternate tiles (one
    // thread issues an MMA only every ~100+ clocks, two nearly double the rate).
    // The ring then carries the two tiles of a pair interleaved stage by stage:
    // stage i of tile k sits at g = (k / ni) * ni * spt + i * ni + k mod ni.
    const int ni = p.nacc;

    if (warp < NPROD) {
        // ---------------- TMA producers: a TMA stream of one thread completes about
        // one box at a time, so nprod warps take turns, warp q loading the stages
        // g = q, q + nprod, ... of this CTA's sequence.  nst is a multiple of nprod,
        // so every stage slot has one producer, which reuses it only after waiting
        // for the slot's previous round: a parity wait never skips a phase.
        if (lane == 0 && warp < p.nprod) {
            const int total = (ntile_cta + ni - 1) / ni * ni * stages_per_tile;
            int g = warp, last = -1;
            bool failed = false;
            int kc = -1, qh0 = 0, ph0 = 0;
            TileCoord tcd;
            for (; g < total; g += p.nprod) {
                const int pr = g / (ni * stages_per_tile), rr = g % (ni * stages_per_tile);
                const int i = rr / ni, k = pr * ni + rr % ni;
                if (k >= ntile_cta) continue;          // the missing partner of a last, lone tile
                if (k != kc) {
                    kc = k;
                    tcd = tile_coord((int)blockIdx.x + k * (int)gridDim.x, p);
                    qh0 = tcd.qhb * p.MH;
                    ph0 = (tcd.rD * 2 + tcd.rH) * 2;
                }
                const int e = i % p.nwe;
                int r = i / p.nwe;
                const int kb = r % p.n_kb; r /= p.n_kb;
                const int jh = r % p.nT, jd = r / p.nT;
                const int s = g % p.nst;
                if (g >= p.nst && !dev::mbar_wait_bounded(&empty_bar[s], ((g / p.nst) - 1) & 1, kWaitLimitNs)) {
                    atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                    failed = true;
                    break;
                }
                const int j0 = p.we_j[0][e], j1 = p.we_j[1][e];
                uint8_t *a_s = smem + (size_t)s * p.stage_bytes;
                uint8_t *b_s = a_s + p.a_bytes;
                dev::mbar_arrive_expect_tx(&full_bar[s], p.a_bytes + p.b_bytes * (uint32_t)((j0 >= 0) + (j1 >= 0)));
                dev::tma_load_5d(a_s, &tmA, &full_bar[s], kb * BK, p.we_delta[e],
                                 qh0 + p.delta[1][tcd.rH][jh], tcd.qd + p.delta[0][tcd.rD][jd], tcd.n);
                const int tap0 = (jd * p.nT + jh) * p.nT;
                if (j0 >= 0)
                    dev::tma_load_2d(b_s, &tmB, &full_bar[s], (tap0 + j0) * p.C_in + kb * BK, ph0 * p.C_out);
                if (j1 >= 0)
                    dev::tma_load_2d(b_s + p.b_bytes, &tmB, &full_bar[s], (tap0 + j1) * p.C_in + kb * BK,
                                     (ph0 + 1) * p.C_out);
                last = g;
            }
            if (failed)   // let this warp's copies still in flight land before shared memory goes away
                for (int q = last; q >= 0 && q > last - p.nst; q -= p.nprod)
                    dev::mbar_wait_bounded(&full_bar[q % p.nst], (q / p.nst) & 1, kWaitLimitNs);
        }
    } else if (warp < kMmaWarp0 + NMMA) {
        // ---------------- MMA issuers.  An MMA costs the issuing thread about 100
        // clocks at best, so the loop carries its ring slot, parity and W-offset
        // index as counters (no division) and keeps the per-offset flags in registers.
        const int j = warp - kMmaWarp0;
        if (lane == 0 && j < ni) {
            bool ok = true;
            uint32_t m0 = 0, m1 = 0;                    // W offsets read by phase 0 / phase 1
            for (int e = 0; e < p.nwe; ++e) {
                if (p.we_j[0][e] >= 0) m0 |= 1u << e;
                if (p.we_j[1][e] >= 0) m1 |= 1u << e;
            }
            const uint32_t sbase = dev::smem_u32(smem);
            const uint32_t idesc1 = p.idesc1, idesc2 = p.idesc2, stage_bytes = p.stage_bytes;
            const uint32_t a_bytes = p.a_bytes, b_bytes = p.b_bytes, c_out = (uint32_t)p.C_out;
            const int nst = p.nst, nwe = p.nwe;
            int s = j;                                  // ring position g = j, j + ni, ...
            uint32_t par = 0;
            for (int k = j; k < ntile_cta && ok; k += ni) {
                const int a = j;
                const int use = k / ni;                        // earlier tiles in accumulator a
                if (use > 0 && !dev::mbar_wait_bounded(&acc_empty[a], (use - 1) & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t d0 = tmem + (uint32_t)a * p.acc_cols;
                const uint32_t d1 = d0 + c_out;
                bool init0 = false, init1 = false;
                int e = 0;
                for (int i = 0; i < stages_per_tile; ++i) {
                    if (!dev::mbar_wait_bounded(&full_bar[s], par, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const bool h0 = (m0 >> e) & 1u, h1 = (m1 >> e) & 1u;
                    const uint32_t a_addr = sbase + (uint32_t)s * stage_bytes;
                    const uint64_t da = tc::desc_sw128(a_addr);
                    const uint64_t db0 = tc::desc_sw128(a_addr + a_bytes);
                    const uint64_t db1 = tc::desc_sw128(a_addr + a_bytes + b_bytes);
                    if (h0 && h1 && idesc2 && init0 == init1) {
                        // both halves in one MMA (they hold the same number of terms)
#pragma unroll
                        for (int kk = 0; kk < BK / UK; ++kk)   // 16 bf16 = 32 bytes along K per step
                            tc::mma_bf16(d0, da + 2 * kk, db0 + 2 * kk, idesc2, (init0 || kk) ? 1u : 0u);
                    } else {
                        if (h0)
#pragma unroll
                            for (int kk = 0; kk < BK / UK; ++kk)
                                tc::mma_bf16(d0, da + 2 * kk, db0 + 2 * kk, idesc1, (init0 || kk) ? 1u : 0u);
                        if (h1)
#pragma unroll
                            for (int kk = 0; kk < BK / UK; ++kk)
                                tc::mma_bf16(d1, da + 2 * kk, db1 + 2 * kk, idesc1, (init1 || kk) ? 1u : 0u);
                    }
                    init0 = init0 || h0;
                    init1 = init1 || h1;
                    tc::commit(&empty_bar[s]);
                    s += ni;                                   // nst is a multiple of ni
                    if (s >= nst) {
                        s -= nst;
                        par ^= 1u;
                    }
                    if (++e == nwe) e = 0;
                }
                if (ok) tc::commit(&acc_full[a]);
            }
            // every MMA issued has to complete before the TMEM is freed
            tc::commit(&drain_bar[j]);
            if (!dev::mbar_wait_bounded(&drain_bar[j], 0, kWaitLimitNs)) ok = false;
            if (!ok) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
        }
    } else {
        // ---------------- epilogue: EPW warps per TMEM lane quarter (32 positions);
        // a warp reaches the lanes of quarter warp mod 4
        const int ew = warp & 3;
        const int half = (warp - kEpiWarp0) >> 2;
        const int nchunk = p.C_out / 16;
        const int64_t sp = (int64_t)p.Lo0 * p.Lo1 * p.Lo2;
        bool ok = true;
        for (int k = 0; k < ntile_cta; ++k) {
            const TileCoord tcd = tile_coord((int)blockIdx.x + k * (int)gridDim.x, p);
            const int a = p.nacc == 2 ? (k & 1) : 0;
            const int use = p.nacc == 2 ? (k >> 1) : k;
            if (ok && !dev::mbar_wait_bounded(&acc_full[a], use & 1, kWaitLimitNs)) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);        // warp-uniform before .sync.aligned loads
            tc::fence_after();
            const int m = ew * 32 + lane;
            const int qh = tcd.qhb * p.MH + m / p.QW, qw = m % p.QW;
            const int od = 2 * tcd.qd + tcd.rD, oh = 2 * qh + tcd.rH;
            const bool valid = od < p.Lo0 && oh < p.Lo1;
            float *yrow = y + (int64_t)tcd.n * p.C_out * sp + ((int64_t)od * p.Lo1 + oh) * p.Lo2 + 2 * qw;
            const uint32_t tbase = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)a * p.acc_cols;
            // chunks half, half + EPW, ..., two per batch; the accumulator is
            // released as soon as the warp's last batch is in registers
            bool released = false;
            for (int ci = half; ci < nchunk; ci += 2 * EPW) {
                const bool two = ci + EPW < nchunk;
                float v0[2][16], v1[2][16];
                if (ok) {
                    tc::tmem_ld16(tbase + (uint32_t)(ci * 16), v0[0]);
                    tc::tmem_ld16(tbase + (uint32_t)(p.C_out + ci * 16), v1[0]);
                    if (two) {
                        tc::tmem_ld16(tbase + (uint32_t)((ci + EPW) * 16), v0[1]);
                        tc::tmem_ld16(tbase + (uint32_t)(p.C_out + (ci + EPW) * 16), v1[1]);
                    }
                    tc::tmem_wait_ld();
                }
                if (ci + 2 * EPW >= nchunk) {
                    tc::fence_before();
                    dev::mbar_arrive(&acc_empty[a]);
                    released = true;
                }
                if (ok && valid) {
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        if (b == 1 && !two) break;
                        const int c0 = (ci + b * EPW) * 16;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int oc = c0 + i;
                            const float bb = bias ? __ldg(bias + oc) : 0.f;
                            __stcs(reinterpret_cast<float2 *>(yrow + (int64_t)oc * sp),
                                   make_float2(v0[b][i] + bb, v1[b][i] + bb));
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
    if (warp == kMmaWarp0) tc::tmem_dealloc(tmem, p.tmem_cols);
}

// ---- repack kernels ------------------------------------------------------------
// Both operands are moved from channel-major rows (one row per channel, the
// other index contiguous) to position-major rows of 64 channels (128 bytes).
// One CTA moves a block of 64 channels x 64 columns with 16-byte loads and
// stores: each thread loads 8 columns of two neighbouring channels, pairs
// them into 32-bit words (channel c in the low half, as it sits in memory),
// and parks the words in shared memory by column; the store side reads four
// words (8 channels) of one column and writes them as one 16-byte store.
// Warps load 4 channels x 128 contiguous bytes and store 4 columns x 128
// contiguous bytes; the tile pitch of 33 words keeps the store side free of
// bank conflicts.
constexpr int RB = 64;                    // channels and columns per repack block

__device__ __forceinline__ void repack_load_pairs(const bf16_t *__restrict__ src, int64_t row_stride,
                                                  int ncols, uint32_t (*tile)[33])
{
    const int icp = threadIdx.x >> 3, k8 = threadIdx.x & 7;
    uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
    if (k8 * 8 < ncols) {
        v0 = __ldcs(reinterpret_cast<const uint4 *>(src + (int64_t)(2 * icp) * row_stride + k8 * 8));
        v1 = __ldcs(reinterpret_cast<const uint4 *>(src + (int64_t)(2 * icp + 1) * row_stride + k8 * 8));
    }
    const uint32_t a[4] = {v0.x, v0.y, v0.z, v0.w};
    const uint32_t b[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        tile[k8 * 8 + 2 * j][icp] = __byte_perm(a[j], b[j], 0x5410);
        tile[k8 * 8 + 2 * j + 1][icp] = __byte_perm(a[j], b[j], 0x7632);
    }
}

// x (N, C, S) -> x_cl (N, S, C), S = D*H*W; S a multiple of 8, C of 64.
__global__ void __launch_bounds__(256)
repack_x_kernel(const bf16_t *__restrict__ x, bf16_t *__restrict__ xcl, int C, int64_t SP)
{
    __shared__ uint32_t tile[RB][33];
    const int n = blockIdx.z;
    const int c0 = blockIdx.y * RB;
    const int64_t s0 = (int64_t)blockIdx.x * RB;
    const int ncols = (int)((SP - s0) < RB ? (SP - s0) : RB);
    repack_load_pairs(x + ((int64_t)n * C + c0) * SP + s0, SP, ncols, tile);
    __syncthreads();
    bf16_t *xd = xcl + ((int64_t)n * SP + s0) * C + c0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int o = threadIdx.x + 256 * t;
        const int q = o & 7, row = o >> 3;
        if (row < ncols) {
            const uint4 v = make_uint4(tile[row][4 * q], tile[row][4 * q + 1], tile[row][4 * q + 2],
                                       tile[row][4 * q + 3]);
            *reinterpret_cast<uint4 *>(xd + (int64_t)row * C + 8 * q) = v;
        }
    }
}

// The same move, one bf16 at a time, for S not a multiple of 8.
__global__ void __launch_bounds__(256)
repack_x_scalar_kernel(const bf16_t *__restrict__ x, bf16_t *__restrict__ xcl, int C, int64_t SP)
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
    int r_of[3][8];          // residue and tap index that kernel index k belongs to
    int j_of[3][8];
};

// w (C_in, C_out, K0, K1, K2) -> w_p[phase][oc][tap][ic], phase = (rD, rH, rW),
// tap = (jd, jh, jw), ic fastest.  Every kernel index (kd, kh, kw) belongs to
// exactly one (phase, tap), so each (ic, oc) row of kD*kH*kW weights is
// scattered once.  Block = (64 input channels, one oc); columns = kernel
// indices in chunks of 64 (kD*kH*kW is a multiple of 8: even extents).
__global__ void __launch_bounds__(256)
repack_w_kernel(const bf16_t *__restrict__ w, bf16_t *__restrict__ wp, WPackParams q)
{
    __shared__ uint32_t tile[RB][33];
    const int ic0 = blockIdx.x * RB;
    const int oc = blockIdx.y;
    const int kvol = q.K0 * q.K1 * q.K2;
    const int ntap = q.nT * q.nT * q.nT;
    const int64_t row_stride = (int64_t)q.C_out * kvol;
    for (int kc = 0; kc < kvol; kc += RB) {
        const int ncols = (kvol - kc) < RB ? (kvol - kc) : RB;
        if (kc) __syncthreads();
        repack_load_pairs(w + ((int64_t)ic0 * q.C_out + oc) * kvol + kc, row_stride, ncols, tile);
        __syncthreads();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int o = threadIdx.x + 256 * t;
            const int qq = o & 7, row = o >> 3;
            if (row < ncols) {
                const int k = kc + row;
                const int kw = k % q.K2, kh = (k / q.K2) % q.K1, kd = k / (q.K1 * q.K2);
                const int ph = (q.r_of[0][kd] << 2) | (q.r_of[1][kh] << 1) | q.r_of[2][kw];
                const int tap = (q.j_of[0][kd] * q.nT + q.j_of[1][kh]) * q.nT + q.j_of[2][kw];
                const uint4 v = make_uint4(tile[row][4 * qq], tile[row][4 * qq + 1],
                                           tile[row][4 * qq + 2], tile[row][4 * qq + 3]);
                *reinterpret_cast<uint4 *>(wp + (((int64_t)ph * q.C_out + oc) * ntap + tap) * q.C_in +
                                           ic0 + 8 * qq) = v;
            }
        }
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
                wq.r_of[d][c + 2 * j] = r;
                wq.j_of[d][c + 2 * j] = j;
            }
        }
    }
    wq.C_in = pb.C_in; wq.C_out = pb.C_out; wq.nT = p.nT;
    wq.K0 = pb.K[0]; wq.K1 = pb.K[1]; wq.K2 = pb.K[2];
    // distinct input W offsets: the two W residues' offsets differ by 0 or 1, so
    // there are at most nT + 1; offsets both phases read come first, so the first
    // MMA of a tile initialises both halves of the accumulator at once
    int lo = p.delta[2][0][0], hi = p.delta[2][0][0];
    for (int r = 0; r < 2; ++r)
        for (int j = 0; j < p.nT; ++j) {
            lo = p.delta[2][r][j] < lo ? p.delta[2][r][j] : lo;
            hi = p.delta[2][r][j] > hi ? p.delta[2][r][j] : hi;
        }
    for (int pass = 0; pass < 3; ++pass)
        for (int dv = lo; dv <= hi; ++dv) {
            int jr[2] = {-1, -1};
            for (int r = 0; r < 2; ++r)
                for (int j = 0; j < p.nT; ++j)
                    if (p.delta[2][r][j] == dv) jr[r] = j;
            const int cat = (jr[0] >= 0 && jr[1] >= 0) ? 0 : (jr[0] >= 0 ? 1 : (jr[1] >= 0 ? 2 : 3));
            if (cat != pass) continue;
            if (p.nwe >= MAXWE) return false;
            p.we_delta[p.nwe] = dv;
            p.we_j[0][p.nwe] = jr[0];
            p.we_j[1][p.nwe] = jr[1];
            ++p.nwe;
        }
    p.idesc1 = tc::idesc(1, pb.C_out, BM);
    p.idesc2 = 2 * pb.C_out <= 256 ? tc::idesc(1, 2 * pb.C_out, BM) : 0u;
    p.acc_cols = (uint32_t)(2 * pb.C_out);
    p.nacc = 4 * pb.C_out <= 512 ? 2 : 1;
    uint32_t cols = 32;
    while (cols < (uint32_t)p.nacc * p.acc_cols) cols <<= 1;
    p.tmem_cols = cols;
    p.a_bytes = (uint32_t)(BM * BK * 2);
    p.b_bytes = (uint32_t)pb.C_out * BK * 2;
    p.stage_bytes = p.a_bytes + 2 * p.b_bytes;
    const size_t budget = 227 * 1024 - 2048;     // alignment slack, static shared memory
    p.nst = (int)(budget / p.stage_bytes);
    if (p.nst > MAXST) p.nst = MAXST;
    if (p.nst < 2) return false;
    p.nprod = p.nst < NPROD ? p.nst : NPROD;
    {
        // one producer per stage slot, and the issuers' interleaved stages on fixed slots
        const int l = (p.nacc == 2 && p.nprod % 2) ? 2 * p.nprod : p.nprod;
        p.nst -= p.nst % l;
        if (p.nst < l) return false;
    }
    out->p = p;
    out->wq = wq;
    out->x_bytes = align256((size_t)pb.N * pb.C_in * pb.in_sp() * 2);
    out->w_bytes = align256((size_t)8 * pb.C_out * p.nT * p.nT * p.nT * pb.C_in * 2);
    out->smem = (size_t)p.nst * p.stage_bytes + 1024;
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
    if (SP % 8 == 0)
        repack_x_kernel<<<gx, 256, 0, a.stream>>>(static_cast<const bf16_t *>(a.x), xcl, pb.C_in, SP);
    else
        repack_x_scalar_kernel<<<gx, 256, 0, a.stream>>>(static_cast<const bf16_t *>(a.x), xcl, pb.C_in, SP);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2) weights -> per-phase K-major
    dim3 gw((unsigned)(pb.C_in / RB), (unsigned)pb.C_out);
    repack_w_kernel<<<gw, 256, 0, a.stream>>>(static_cast<const bf16_t *>(a.w), wp, pl.wq);
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
    int grid = sm_count();
    if (grid > p.ntiles) grid = p.ntiles;
    umma_ct3d_kernel<<<grid, kThreads, pl.smem, a.stream>>>(tmA, tmB, a.bias, a.y, p, status);
    return cudaGetLastError();
}

}  // namespace ct
