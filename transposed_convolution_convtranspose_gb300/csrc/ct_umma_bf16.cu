// ct_umma_bf16.cu -- bf16-input / fp32-accumulate ConvTranspose3d on the
// 5th-generation tensor cores (tcgen05 + TMEM), as an implicit GEMM per
// stride phase.
//
// Method ([l1_p72] stride-phase classes; [l2_p26] "what cuDNN does": the
// dense C_in x C_out contraction per output): with stride 2 in every
// dimension and an even kernel extent, every output residue class
// (rD, rH, rW) receives the same number of taps per dimension, and
//     y[n, oc, 2q + r] = bias[oc] + sum_{taps t, ic} x[n, ic, q + delta_t] * w[ic, oc, k_t]
// is a GEMM per phase: M = positions q, N = C_out, K = taps x C_in.  Two
// repack kernels prepare the operands in the caller's workspace:
//   x (N, C, D, H, W)          ->  x_t (N, D, H, W, C)   bf16, channels fastest
//   w (C, C_out, kD, kH, kW)   ->  weight panels, K-major (C_in fastest)
//
// Tile: 128 output positions q = 8 consecutive qw x 16 consecutive qh of
// one D plane, for one (rD, rH) phase pair; its accumulator is two halves of
// C_out TMEM columns, one per W phase.  TMEM row m holds position
// (qw, qh) = (m mod 8, m / 8), so each 8-row swizzle group of the A operand
// is 8 consecutive qw of one qh row -- contiguous in x_t -- and a warp's 32
// TMEM lanes are 4 qh rows of 8 qw: its stores cover 4 rows x 64 bytes.
// When two accumulators fit, a unit of work is a pair of tiles (two
// neighbouring 8-column qw blocks): they share every input window and weight
// panel, and each of two MMA-issuing warps computes one of them.  When the
// pairs fill whole rounds of the grid but the last round would leave more
// than half the CTAs idle, that round's pairs run as single tiles (twice as
// many units, each a little over half a pair's time): the other issuer and
// epilogue half keep the barrier protocol without MMAs or stores (the SPLIT
// instantiation; without it the issue loop carries no such test).
//
// Order within a unit: all of W phase 0, then all of W phase 1.  The TMEM
// holds no second accumulator to switch to while one is drained, so the
// halves take turns instead: phase 0's half is drained while phase 1 is
// computed, and phase 1's half while the next unit's phase 0 is computed.
//
// Operand A without shifted copies: per (W phase, D tap, K block) one TMA
// box brings the unit's input window, (16 + H halo) x (8 x tiles + nT - 1)
// positions x 64 channels, 128-byte swizzled, rows ordered (h, w).  The A
// operand of input offset (dh, dw) for tile j is that window read from start
// row (dh - dh_lo) * wspan + (dw - wlo) + 8 j with a stride of wspan rows
// between groups: only the shared-memory descriptor's start address and
// stride-byte-offset change (the 128-byte swizzle is a function of the
// absolute shared-memory address, so rows read from any start line up with
// how the TMA wrote them).  Boxes reaching outside the input read zeros,
// which is the boundary handling.
//
// Operand B: for every (phase pair, D tap, H tap, W phase, W tap) one panel
// of C_out rows, K-major, one box each.
//
// Roles (persistent CTA, one per SM):
//   warp 0      TMA producer of the A ring (input windows)
//   warps 1-4   TMA producers of the B ring (weight panels), one per slot
//               (one thread's TMA stream completes about one box at a time)
//   warps 5-6   TMEM allocation and MMA issue, one warp per tile of the
//               pair and its accumulator (one thread issues an MMA only every
//               ~100+ clocks; two warps nearly double the rate); both consume
//               every stage
//   warps 7-22  epilogue, four per TMEM lane quarter: with a tile pair, two
//               of them drain each tile, taking alternate 16-channel chunks;
//               with single tiles the four take alternate chunks.
//               tcgen05.ld, bias; W phase 0 written as (output, 0) float2
//               pairs, W phase 1 into the odd slots
// Every ring slot has exactly one producer, which refills it only after
// waiting for its previous round, so a parity wait never has to tell two
// phases apart.  Every mbarrier wait is bounded: a timeout records
// CT_ERR_DEVICE_TIMEOUT in the device status word and the roles unwind (the
// producers wait, bounded, for their own TMA copies and the MMA issuers for
// their own MMAs before the TMEM is freed).
#include <string.h>

#include "ct_internal.h"
#include "ct_device.cuh"
#include "ct_tma.h"
#include "ct_tcgen05.cuh"

namespace ct {
namespace {

constexpr int BM = 128;      // positions per tile (UMMA M)
constexpr int QWT = 8;       // qw per tile (one 8-row swizzle group per qh; TMEM row m: qw = m mod 8)
constexpr int MHT = 16;      // qh per tile (TMEM row m: qh = m / 8)
constexpr int BK = 64;       // bf16 elements of K per stage (one 128-byte swizzle row)
constexpr int UK = 16;       // K of one tcgen05.mma kind::f16
constexpr int MAXA = 3;      // A ring slots at most (input windows of a tile pair)
constexpr int MAXB = 8;      // B ring slots at most
constexpr int NPB = 4;       // B producer warps at most (slot s loaded by warp s mod npb)
constexpr int NMMA = 2;      // MMA-issuing warps at most (one per TMEM accumulator)
constexpr int EPW = 4;       // epilogue warps per TMEM lane quarter
constexpr int EB = 2;        // 16-channel chunks per epilogue batch (registers)
constexpr int kAWarp = 0;
constexpr int kBWarp0 = 1;
constexpr int kMmaWarp0 = kBWarp0 + NPB;
constexpr int kEpiWarp0 = kMmaWarp0 + NMMA;
constexpr int kThreads = 32 * (kEpiWarp0 + 4 * EPW);
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct UParams {
    int N, C_in, C_out;
    int Lo0, Lo1, Lo2;
    int QD, QH, QW, n_qhb, n_qwp;   // n_qwp: pairs of 8-column qw blocks
    int nT;                  // taps per class of H and W (kernel extent / 2)
    int SD, nTD;             // D: stride 2 and nT taps, or a unit dimension (stride 1, one tap)
    int cl;                  // channels-last y (N, D, H, W, C_out); x is then the caller's own
    int n_kb;                // C_in / BK
    int ntiles;              // units of work: tile pairs (or single tiles when nacc = 1)
    // the last, partial round of pairs split into single tiles: units
    // [0, npair) are pairs, the next nunits - npair are single tiles, two per
    // remaining pair (nunits = ntiles when no pair is split)
    int npair, nunits;
    int nacc;                // TMEM accumulators = MMA issuers = tiles per pair (1 or 2)
    int na, nb, npb;         // A ring slots, B ring slots, B producers (nb a multiple of npb)
    uint32_t acc_cols;       // columns of one accumulator (2 x C_out: W phase 0, then W phase 1)
    uint32_t tmem_cols;      // allocated TMEM columns (power of 2 >= nacc x acc_cols)
    uint32_t idesc;          // instruction descriptor, N = C_out
    uint32_t a_slot;         // bytes of an A ring slot (one input window, 1024-aligned)
    uint32_t b_bytes;        // bytes of one weight panel (C_out rows x 128)
    int wg;                  // W taps per B stage (nT when nT x C_out rows fit one box, else 1)
    uint32_t sbo;            // A descriptor stride between 8-row groups (qh): wspan x 128
    int hspan, wspan;        // input window extents (H, W) of a tile pair and one W phase
    int dh_lo;               // smallest H input offset
    int wlo[2];              // smallest W input offset of each W phase (its window's start)
    int delta[3][2][4];      // input offset of tap j for residue r, per dimension
    int blk_units;           // C_out-row units of one (phase pair, D tap, H tap) block
};

// unit -> (n, qd, qh block, qw block pair, rD, rH); tile j of the pair is qw
// block 2 * qwp + j.  The four (rD, rH) phases of one position block are
// neighbours, so their input windows are reused from L2
struct TileCoord {
    int n, qd, qhb, qwp, rD, rH;
};
__device__ __forceinline__ TileCoord tile_coord(int t, const UParams &p);

// Unit u of the schedule: its pair's coordinates, and for a single-tile unit
// the tile of the pair it computes (*js = 0 or 1; -1 for a whole pair).
// Without SPLIT every unit is a pair (the issue loop keeps no test).
template <bool SPLIT>
__device__ __forceinline__ TileCoord unit_tiles(int u, const UParams &p, int *js)
{
    if (!SPLIT || u < p.npair) {
        *js = -1;
        return tile_coord(u, p);
    }
    const int s = u - p.npair;
    *js = s & 1;
    return tile_coord(p.npair + (s >> 1), p);
}

__device__ __forceinline__ TileCoord tile_coord(int t, const UParams &p)
{
    TileCoord c;
    c.rH = t & 1; t >>= 1;
    c.rD = 0;
    if (p.SD == 2) {
        c.rD = t & 1;
        t >>= 1;
    }
    c.qwp = t % p.n_qwp; t /= p.n_qwp;
    c.qhb = t % p.n_qhb; t /= p.n_qhb;
    c.qd = t % p.QD; t /= p.QD;
    c.n = t;
    return c;
}

// K-major, 128-byte swizzled operand with 8-row groups `sbo` bytes apart
__device__ __forceinline__ uint64_t desc_sw128_sbo(uint32_t saddr, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;                       // leading byte offset (unused)
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;   // stride byte offset
    d |= (uint64_t)1 << 46;                       // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                       // 128-byte swizzle
    return d;
}

// ---- GEMM kernel -------------------------------------------------------------
// SPLIT: the last round's pairs run as single tiles.  CL: channels-last y (a
// template parameter so that each layout's epilogue is compiled alone: the
// two share the kernel's 80 registers).
template <bool SPLIT, bool CL>
__global__ void __launch_bounds__(kThreads, 1)
umma_ct3d_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const float *__restrict__ bias, float *__restrict__ y, const __grid_constant__ UParams p,
                 unsigned int *status)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t a_full[MAXA], a_empty[MAXA], b_full[MAXB], b_empty[MAXB], acc_full[2][2],
        acc_empty[2][2], drain_bar[NMMA];
    __shared__ uint32_t tmem_slot;
    // channels last, the epilogue reads 4 bias values per 16-byte load
    __shared__ alignas(CL ? 16 : 4) float s_bias[256];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                                // na x a_slot
    uint8_t *sB = smem + (size_t)p.na * p.a_slot;      // nb x (wg x b_bytes)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&tmA);
        dev::prefetch_tensormap(&tmB);
        // a stage is released by every issuer, an accumulator half by the
        // epilogue threads that read it (all of them with one tile per unit,
        // half with two)
        for (int s = 0; s < p.na; ++s) {
            dev::mbar_init(&a_full[s], 1);
            dev::mbar_init(&a_empty[s], p.nacc);
        }
        for (int s = 0; s < p.nb; ++s) {
            dev::mbar_init(&b_full[s], 1);
            dev::mbar_init(&b_empty[s], p.nacc);
        }
        for (int a = 0; a < 2; ++a)
            for (int r = 0; r < 2; ++r) {
                dev::mbar_init(&acc_full[a][r], 1);
                dev::mbar_init(&acc_empty[a][r], 32 * 4 * EPW / p.nacc);
            }
        for (int j = 0; j < NMMA; ++j) dev::mbar_init(&drain_bar[j], 1);
        dev::fence_mbar_init();
    }
    if (warp == kMmaWarp0) tc::tmem_alloc(&tmem_slot, p.tmem_cols);
    for (int i = threadIdx.x; i < p.C_out; i += blockDim.x) s_bias[i] = bias ? bias[i] : 0.f;
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // the operands in the workspace come from the repack kernel(s)
    dev::griddep_wait();
    const uint32_t tmem = tmem_slot;
    const int ntile_cta =
        p.nunits > (int)blockIdx.x ? (p.nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    // stages per unit, W phase 0 first, then W phase 1:
    //   A = (W phase, D tap, K block), B = (W phase, D tap, K block, H tap, W tap).
    // A unit is a pair of tiles (two 8-row qh blocks) when two accumulators fit:
    // both issuers consume every stage, issuer j computing tile j from the shared
    // input window (8 rows further down for tile 1) and the shared weight panel.
    const int nT = p.nT, nTD = p.nTD, n_kb = p.n_kb;
    const int spa = 2 * nTD * n_kb;
    const int spb = spa * nT * (nT / p.wg);
    const uint32_t b_slot = (uint32_t)p.wg * p.b_bytes;
    const int ni = p.nacc;

    if (warp == kAWarp || (warp >= kBWarp0 && warp < kBWarp0 + NPB)) {
        // ---------------- TMA producers
        const bool isA = warp == kAWarp;
        const int q = isA ? 0 : warp - kBWarp0;
        if (lane == 0 && (isA || q < p.npb)) {
            const int np = isA ? 1 : p.npb;
            const int nst = isA ? p.na : p.nb;
            const int sp = isA ? spa : spb;
            uint64_t *fullb = isA ? a_full : b_full;
            uint64_t *emptyb = isA ? a_empty : b_empty;
            const int total = ntile_cta * sp;
            int last = -1, kc = -1;
            bool failed = false;
            TileCoord tcd;
            tcd.n = tcd.qd = tcd.qhb = tcd.qwp = tcd.rD = tcd.rH = 0;
            for (int g = q; g < total; g += np) {
                const int k = g / sp, i = g % sp;
                if (k != kc) {
                    kc = k;
                    int js;
                    tcd = unit_tiles<SPLIT>((int)blockIdx.x + k * (int)gridDim.x, p, &js);   // a single tile loads its pair's operands
                }
                const int s = g % nst;
                if (g >= nst && !dev::mbar_wait_bounded(&emptyb[s], ((g / nst) - 1) & 1, kWaitLimitNs)) {
                    failed = true;
                    break;
                }
                if (isA) {
                    const int wr = i / (nTD * n_kb), r = i % (nTD * n_kb);
                    const int jd = r / n_kb, kb = r % n_kb;
                    dev::mbar_arrive_expect_tx(&fullb[s], (uint32_t)(p.hspan * p.wspan) * 128u);
                    // x_t viewed as (C, W, H, D, N): W phase wr's window from
                    // (qw0 + wlo[wr], qh0 + dh_lo)
                    dev::tma_load_5d(sA + (size_t)s * p.a_slot, &tmA, &fullb[s], kb * BK,
                                     tcd.qwp * ni * QWT + p.wlo[wr], tcd.qhb * MHT + p.dh_lo,
                                     tcd.qd + p.delta[0][tcd.rD][jd], tcd.n);
                } else {
                    int r = i;
                    const int jw = (r % (nT / p.wg)) * p.wg;
                    r /= nT / p.wg;
                    const int jh = r % nT;
                    r /= nT;
                    const int kb = r % n_kb;
                    r /= n_kb;
                    const int jd = r % nTD, wr = r / nTD;
                    const int ph2 = tcd.rD * 2 + tcd.rH;
                    const int brow = (((ph2 * nTD + jd) * nT + jh) * p.blk_units + wr * nT + jw) * p.C_out;
                    // the panels of W taps jw .. jw + wg - 1 are consecutive rows
                    dev::mbar_arrive_expect_tx(&fullb[s], b_slot);
                    dev::tma_load_2d(sB + (size_t)s * b_slot, &tmB, &fullb[s], kb * BK, brow);
                }
                last = g;
            }
            if (failed) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                // let this warp's copies still in flight land before shared memory goes away
                for (int r = last; r >= 0 && r > last - nst; r -= np)
                    dev::mbar_wait_bounded(&fullb[r % nst], (r / nst) & 1, kWaitLimitNs);
            }
        }
    } else if (warp < kMmaWarp0 + NMMA) {
        // ---------------- MMA issuers.  An MMA costs the issuing thread about 100
        // clocks at best, so the loop carries ring slots, parities and indices as
        // counters and keeps the per-offset data in registers.  A tile's
        // accumulator is two halves of C_out columns, one per W phase; W phase 0
        // is computed first, so its half is drained while W phase 1 runs, and
        // phase 1's half while the next unit's phase 0 runs.
        const int j = warp - kMmaWarp0;
        if (lane == 0 && j < ni) {
            bool ok = true;
            const uint32_t sAb = dev::smem_u32(sA), sBb = dev::smem_u32(sB);
            const uint32_t idesc = p.idesc, a_slot = p.a_slot, b_bytes = p.b_bytes;
            const int wg = p.wg;
            const uint32_t sbo = p.sbo, c_out = (uint32_t)p.C_out;
            const int na = p.na, nb = p.nb;
            const uint32_t trow = (uint32_t)(j * QWT) * 128u;   // tile j's columns in the window
            int sa = 0, sb = 0;
            uint32_t pa = 0, pb = 0;
            for (int k = 0; k < ntile_cta && ok; ++k) {
                int js;
                const TileCoord tcd = unit_tiles<SPLIT>((int)blockIdx.x + k * (int)gridDim.x, p, &js);
                // a single-tile unit: the other issuer keeps the protocol (waits,
                // commits) but issues no MMAs
                const bool act = !SPLIT || js < 0 || js == j;
                for (int wr = 0; wr < 2 && ok; ++wr) {
                    if (k > 0 && !dev::mbar_wait_bounded(&acc_empty[j][wr], (k - 1) & 1, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t d = tmem + (uint32_t)j * p.acc_cols + (uint32_t)wr * c_out;
                    // W tap jw reads window column nT - 1 - jw: that many rows in
                    const uint32_t awstep = 128u;
                    const uint32_t aw0 = (uint32_t)(nT - 1) * awstep;
                    bool init = false;
                    for (int jd = 0; jd < nTD && ok; ++jd)
                        for (int kb = 0; kb < n_kb && ok; ++kb) {
                            if (!dev::mbar_wait_bounded(&a_full[sa], pa, kWaitLimitNs)) {
                                ok = false;
                                break;
                            }
                            tc::fence_after();
                            const uint32_t wbase = sAb + (uint32_t)sa * a_slot + trow;
                            for (int jh = 0; jh < nT && ok; ++jh) {
                                const uint32_t hoff = (uint32_t)((p.delta[1][tcd.rH][jh] - p.dh_lo) * p.wspan) * 128u;
                                for (int jw0 = 0; jw0 < nT; jw0 += wg) {
                                    if (!dev::mbar_wait_bounded(&b_full[sb], pb, kWaitLimitNs)) {
                                        ok = false;
                                        break;
                                    }
                                    tc::fence_after();
                                    const uint32_t bslot = sBb + (uint32_t)sb * (uint32_t)wg * b_bytes;
                                    for (int t = 0; t < wg; ++t) {
                                        const int jw = jw0 + t;
                                        const uint64_t da =
                                            desc_sw128_sbo(wbase + aw0 - (uint32_t)jw * awstep + hoff, sbo);
                                        const uint64_t db = tc::desc_sw128(bslot + (uint32_t)t * b_bytes);
                                        if (act) {
#pragma unroll
                                            for (int kk = 0; kk < BK / UK; ++kk)   // 16 bf16 = 32 bytes along K
                                                tc::mma_bf16(d, da + 2 * kk, db + 2 * kk, idesc, (init || kk) ? 1u : 0u);
                                        }
                                        init = true;
                                    }
                                    tc::commit(&b_empty[sb]);
                                    if (++sb == nb) {
                                        sb = 0;
                                        pb ^= 1u;
                                    }
                                }
                            }
                            tc::commit(&a_empty[sa]);
                            if (++sa == na) {
                                sa = 0;
                                pa ^= 1u;
                            }
                        }
                    if (ok) tc::commit(&acc_full[j][wr]);
                }
            }
            // every MMA issued has to complete before the TMEM is freed
            tc::commit(&drain_bar[j]);
            if (!dev::mbar_wait_bounded(&drain_bar[j], 0, kWaitLimitNs)) ok = false;
            if (!ok) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
        }
    } else {
        // ---------------- epilogue: EPW warps per TMEM lane quarter (32 positions:
        // 4 qw x 8 qh); a warp reaches the lanes of quarter warp mod 4.  With two
        // tiles per unit, half j of the warps drains tile j (accumulator j) and
        // takes every 16-channel chunk; with one, the halves take alternate chunks.
        // Each W phase half is drained as soon as it is complete.  W phase 0
        // writes each position's pair (even output, 0) as one float2 -- whole
        // 32-byte sectors, so L2 need not fetch the rest of a sector from DRAM,
        // and ordinary stores keep the lines in L2 -- and W phase 1, about half a
        // unit later, overwrites the odd outputs with 4-byte streaming stores.
        // Both stores of a position come from the same thread, in that order.
        const int ew = warp & 3;
        const int grp = (warp - kEpiWarp0) >> 2;            // 0 .. EPW - 1
        // two tiles: groups of even index drain tile 0, odd tile 1, and split its
        // chunks EPW / 2 ways; one tile: the EPW groups split the chunks
        const int a = ni == 2 ? (grp & 1) : 0;
        const int cfirst = ni == 2 ? (grp >> 1) : grp, cstep = ni == 2 ? EPW / 2 : EPW;
        const int nchunk = p.C_out / 16;
        const int64_t sp = (int64_t)p.Lo0 * p.Lo1 * p.Lo2;
        bool ok = true;
        for (int k = 0; k < ntile_cta; ++k) {
            int js;
            const TileCoord tcd = unit_tiles<SPLIT>((int)blockIdx.x + k * (int)gridDim.x, p, &js);
            const bool act = !SPLIT || js < 0 || js == a;   // a single-tile unit: the other half only releases
            const int m = ew * 32 + lane;
            const int qw = (tcd.qwp * ni + a) * QWT + (m & 7), qh = tcd.qhb * MHT + (m >> 3);
            const int od = p.SD * tcd.qd + tcd.rD, oh = 2 * qh + tcd.rH;
            const bool valid = act && qw < p.QW && od < p.Lo0 && oh < p.Lo1;
            for (int wr = 0; wr < 2; ++wr) {
                if (ok && !dev::mbar_wait_bounded(&acc_full[a][wr], k & 1, kWaitLimitNs)) {
                    atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                    ok = false;
                }
                ok = __all_sync(0xffffffffu, ok);    // warp-uniform before .sync.aligned loads
                tc::fence_after();
                float *yrow = y + (int64_t)tcd.n * p.C_out * sp + ((int64_t)od * p.Lo1 + oh) * p.Lo2 + 2 * qw;
                // channels last: output position 2 qw + wr holds C_out consecutive values
                float *ycl = y + ((((int64_t)tcd.n * p.Lo0 + od) * p.Lo1 + oh) * p.Lo2 + 2 * qw + wr) * p.C_out;
                const uint32_t tbase =
                    tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)a * p.acc_cols + (uint32_t)wr * p.C_out;
                // one chunk a batch in the split and channels-last instances: their
                // registers then need no spills
                constexpr int EBK = (SPLIT || CL) ? 1 : EB;
                // EBK chunks per batch; the half is released as soon as the warp's
                // last batch is in registers
                bool released = false;
                for (int ci = cfirst; ci < nchunk; ci += EBK * cstep) {
                    float v[EBK][16];
                    int nc = 0;
                    if (ok && act) {
#pragma unroll
                        for (int b = 0; b < EBK; ++b)
                            if (ci + b * cstep < nchunk) {
                                tc::tmem_ld16(tbase + (uint32_t)((ci + b * cstep) * 16), v[b]);
                                nc = b + 1;
                            }
                        tc::tmem_wait_ld();
                    }
                    if (ci + EBK * cstep >= nchunk) {
                        tc::fence_before();
                        dev::mbar_arrive(&acc_empty[a][wr]);
                        released = true;
                    }
                    if (ok && valid && CL) {
                        // 16 channels of one position: 64 contiguous bytes
#pragma unroll
                        for (int b = 0; b < EBK; ++b) {
                            if (b >= nc) break;
                            const int c0 = (ci + b * cstep) * 16;
                            float4 *dst = reinterpret_cast<float4 *>(ycl + c0);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                __stcs(dst + i, make_float4(v[b][4 * i] + s_bias[c0 + 4 * i],
                                                            v[b][4 * i + 1] + s_bias[c0 + 4 * i + 1],
                                                            v[b][4 * i + 2] + s_bias[c0 + 4 * i + 2],
                                                            v[b][4 * i + 3] + s_bias[c0 + 4 * i + 3]));
                        }
                    } else if (ok && valid) {
#pragma unroll
                        for (int b = 0; b < EBK; ++b) {
                            if (b >= nc) break;
                            const int c0 = (ci + b * cstep) * 16;
                            float *yc = yrow + (int64_t)c0 * sp;
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float bb = s_bias[c0 + i];
                                if (wr == 0)
                                    *reinterpret_cast<float2 *>(yc) = make_float2(v[b][i] + bb, 0.f);
                                else
                                    __stcs(yc + 1, v[b][i] + bb);
                                yc += sp;
                            }
                        }
                    }
                }
                if (!released) {                      // a warp without chunks
                    tc::fence_before();
                    dev::mbar_arrive(&acc_empty[a][wr]);
                }
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
constexpr int RX = 128;                   // x positions per repack block: two halves of RB

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

// x (N, C, D, H, W) -> x_t (N, D, H, W, C); D*H*W a multiple of 8, C of 64.
// Block (bx, by, n): positions bx*128.., channels by*64..: each channel row
// is read as 256 contiguous bytes, and all four 16-byte loads of a thread are
// in flight before the first shared-memory store.
__device__ __forceinline__ void repack_x_block(const bf16_t *__restrict__ x, bf16_t *__restrict__ xt, int C, int D,
                                               int H, int W, int bx, int by, int n)
{
    __shared__ uint32_t tile[RX][33];
    const int64_t SP = (int64_t)D * H * W;
    const int c0 = by * RB;
    const int64_t s0 = (int64_t)bx * RX;
    const int ncols = (int)((SP - s0) < RX ? (SP - s0) : RX);
    const bf16_t *src = x + ((int64_t)n * C + c0) * SP + s0;
    const int icp = threadIdx.x >> 3, k8 = threadIdx.x & 7;
    uint4 v[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int col = h * RB + k8 * 8;
        v[h][0] = v[h][1] = make_uint4(0, 0, 0, 0);
        if (col < ncols) {
            v[h][0] = __ldcs(reinterpret_cast<const uint4 *>(src + (int64_t)(2 * icp) * SP + col));
            v[h][1] = __ldcs(reinterpret_cast<const uint4 *>(src + (int64_t)(2 * icp + 1) * SP + col));
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int col = h * RB + k8 * 8;
        const uint32_t a[4] = {v[h][0].x, v[h][0].y, v[h][0].z, v[h][0].w};
        const uint32_t b[4] = {v[h][1].x, v[h][1].y, v[h][1].z, v[h][1].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            tile[col + 2 * j][icp] = __byte_perm(a[j], b[j], 0x5410);
            tile[col + 2 * j + 1][icp] = __byte_perm(a[j], b[j], 0x7632);
        }
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int o = threadIdx.x + 256 * t;
        const int q = o & 7, row = o >> 3;
        if (row < ncols) {
            // x_t's position index is the flat spatial index of x
            const int64_t dst = ((int64_t)n * SP + s0 + row) * C + c0 + 8 * q;
            const uint4 v = make_uint4(tile[row][4 * q], tile[row][4 * q + 1], tile[row][4 * q + 2],
                                       tile[row][4 * q + 3]);
            *reinterpret_cast<uint4 *>(xt + dst) = v;
        }
    }
}

// The same move, one bf16 at a time, for D*H*W not a multiple of 8.
__global__ void __launch_bounds__(256)
repack_x_scalar_kernel(const bf16_t *__restrict__ x, bf16_t *__restrict__ xt, int C, int D, int H, int W)
{
    __shared__ bf16_t tile[64][66];
    const int64_t SP = (int64_t)D * H * W;
    const int n = blockIdx.z;
    const int c0 = blockIdx.y * 64;
    const int64_t s0 = (int64_t)blockIdx.x * 64;
    const bf16_t *xs = x + (int64_t)n * C * SP;
    for (int e = threadIdx.x; e < 64 * 64; e += 256) {
        const int c = e >> 6, s = e & 63;
        tile[c][s] = (c0 + c < C && s0 + s < SP) ? xs[(int64_t)(c0 + c) * SP + s0 + s] : (bf16_t)0;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * 64; e += 256) {
        const int s = e >> 6, c = e & 63;
        if (c0 + c < C && s0 + s < SP) {
            const int64_t ss = s0 + s;
            const int w = (int)(ss % W), h = (int)((ss / W) % H), d = (int)(ss / ((int64_t)W * H));
            xt[((((int64_t)n * D + d) * H + h) * W + w) * C + c0 + c] = tile[c][s];
        }
    }
}

struct WPackParams {
    int C_in, C_out, K0, K1, K2, nT, nTD;
    int r_of[3][8];          // residue and tap index that kernel index k belongs to
    int j_of[3][8];
    int blk_units;
};

// w (C_in, C_out, K0, K1, K2) -> weight panels: for every (phase pair, D tap,
// H tap), the C_out rows of each (W phase, W tap), C_in fastest.  Every kernel index (kd, kh, kw) belongs to
// exactly one (phase, tap), so each (ic, oc) row of kD*kH*kW weights is
// scattered once.  Block = (64 input channels, one oc); columns = kernel
// indices in chunks of 64 (kD*kH*kW a multiple of 8: rows of 16-byte loads).
__device__ __forceinline__ void repack_w_block(const bf16_t *__restrict__ w, bf16_t *__restrict__ wp,
                                               const WPackParams &q, int bx, int oc)
{
    __shared__ uint32_t tile[RB][33];
    const int ic0 = bx * RB;
    const int kvol = q.K0 * q.K1 * q.K2;
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
                const int ph2 = (q.r_of[0][kd] << 1) | q.r_of[1][kh];
                const int rw = q.r_of[2][kw], jw = q.j_of[2][kw];
                const int unit = ((ph2 * q.nTD + q.j_of[0][kd]) * q.nT + q.j_of[1][kh]) * q.blk_units +
                                 rw * q.nT + jw;
                const uint4 v = make_uint4(tile[row][4 * qq], tile[row][4 * qq + 1],
                                           tile[row][4 * qq + 2], tile[row][4 * qq + 3]);
                *reinterpret_cast<uint4 *>(wp + ((int64_t)unit * q.C_out + oc) * q.C_in + ic0 + 8 * qq) = v;
            }
        }
    }
}

// Both repacks in one launch: blocks [0, nxb) move x (nbx x nby per image),
// the rest the weights (C_in / 64 per output channel).  The GEMM kernel is
// launched as its programmatic dependent once every block has done its work
// (a trigger at the blocks' start let GEMM CTAs take SMs, and wait, while
// repack blocks still needed them: 0.2184 against 0.2006 ms a step).
__global__ void __launch_bounds__(256)
repack_kernel(const bf16_t *__restrict__ x, bf16_t *__restrict__ xt, int C, int D, int H, int W, int nbx, int nby,
              int nxb, const bf16_t *__restrict__ w, bf16_t *__restrict__ wp, const __grid_constant__ WPackParams q)
{
    const int b = (int)blockIdx.x;
    if (b < nxb) {
        const int per = nbx * nby;
        repack_x_block(x, xt, C, D, H, W, (b % per) % nbx, (b % per) / nbx, b / per);
    } else {
        const int r = b - nxb, nwx = q.C_in / RB;
        repack_w_block(w, wp, q, r % nwx, r / nwx);
    }
    dev::griddep_launch_dependents();
}

// The weight repack alone (after the scalar x repack).
__global__ void __launch_bounds__(256)
repack_w_kernel(const bf16_t *__restrict__ w, bf16_t *__restrict__ wp, const __grid_constant__ WPackParams q)
{
    repack_w_block(w, wp, q, (int)blockIdx.x, (int)blockIdx.y);
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
    if ((pb.nd != 3 && pb.nd != 2) || pb.dtype != CT_BF16 || pb.G != 1) return false;
    // D has stride 2 and the extent of H and W, or is a unit dimension (extent 1,
    // stride 1, no padding: a 2-D problem), whose single residue takes tap 0 at
    // offset 0
    const int SD = pb.S[0];
    if (SD == 1 && (pb.K[0] != 1 || pb.P[0] != 0 || pb.OP[0] != 0)) return false;
    for (int d = SD == 1 ? 1 : 0; d < 3; ++d) {
        if (pb.S[d] != 2 || pb.DL[d] != 1) return false;
        if (pb.K[d] % 2 != 0 || pb.K[d] / 2 > 4) return false;
        if (pb.K[d] != pb.K[2]) return false;
    }
    if (pb.kvol() % 8 != 0) return false;     // the weight repack moves 16-byte pieces of a row
    if (pb.C_in % BK != 0 || pb.C_out % 16 != 0 || pb.C_out < 16 || pb.C_out > 256) return false;
    if (pb.Lo[2] % 2 != 0) return false;
    UParams p;
    memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C_in = pb.C_in; p.C_out = pb.C_out;
    p.Lo0 = pb.Lo[0]; p.Lo1 = pb.Lo[1]; p.Lo2 = pb.Lo[2];
    p.QW = p.Lo2 / 2;
    p.SD = SD;
    p.cl = pb.cl ? 1 : 0;
    p.QD = (p.Lo0 + SD - 1) / SD;
    p.QH = (p.Lo1 + 1) / 2;
    p.nacc = 4 * pb.C_out <= 512 ? 2 : 1;     // tiles per unit
    p.n_qhb = (p.QH + MHT - 1) / MHT;
    p.n_qwp = ((p.QW + QWT - 1) / QWT + p.nacc - 1) / p.nacc;
    p.nT = pb.K[2] / 2;
    p.nTD = SD == 2 ? p.nT : 1;
    p.n_kb = pb.C_in / BK;
    const int64_t tiles = (int64_t)pb.N * p.QD * p.n_qhb * p.n_qwp * 2 * SD;
    if (tiles > 0x7fffffff || tiles == 0) return false;
    p.ntiles = (int)tiles;
    p.npair = p.nunits = p.ntiles;           // the launch may split the last round
    // residue r of a stride-2 dimension takes the taps k == (r + p) mod 2, i.e.
    // k = c + 2j, reading input q + floor((r + p)/2) - j
    WPackParams wq;
    memset(&wq, 0, sizeof(wq));
    for (int d = SD == 1 ? 1 : 0; d < 3; ++d) {
        for (int r = 0; r < 2; ++r) {
            const int c = (r + pb.P[d]) % 2;
            const int base = (r + pb.P[d] - c) / 2;
            for (int j = 0; j < p.nT; ++j) {
                p.delta[d][r][j] = base - j;
                wq.r_of[d][c + 2 * j] = r;
                wq.j_of[d][c + 2 * j] = j;
            }
        }
    }
    // input windows: H offsets span [lo, hi] for both H phases; each W phase
    // reads nT consecutive W offsets, its window starting at the lowest
    int lo = p.delta[1][0][0], hi = lo;
    for (int r = 0; r < 2; ++r)
        for (int j = 0; j < p.nT; ++j) {
            lo = p.delta[1][r][j] < lo ? p.delta[1][r][j] : lo;
            hi = p.delta[1][r][j] > hi ? p.delta[1][r][j] : hi;
        }
    p.dh_lo = lo;
    p.hspan = MHT + hi - lo;
    p.wspan = p.nacc * QWT + p.nT - 1;
    if (p.hspan > 256 || p.wspan > 256) return false;
    // W tap j of a phase reads offset wlo + nT - 1 - j: window column nT - 1 - j
    for (int r = 0; r < 2; ++r) p.wlo[r] = p.delta[2][r][p.nT - 1];
    p.sbo = (uint32_t)p.wspan * 128u;
    p.a_slot = (uint32_t)((p.hspan * p.wspan * 128 + 1023) & ~1023);
    // panels: per (phase pair, D tap, H tap) block, the C_out rows of each
    // (W phase, W tap)
    p.blk_units = 2 * p.nT;
    wq.blk_units = p.blk_units;
    wq.C_in = pb.C_in; wq.C_out = pb.C_out; wq.nT = p.nT; wq.nTD = p.nTD;
    wq.K0 = pb.K[0]; wq.K1 = pb.K[1]; wq.K2 = pb.K[2];
    p.idesc = tc::idesc(1, pb.C_out, BM);
    p.acc_cols = (uint32_t)(2 * pb.C_out);
    uint32_t cols = 32;
    while (cols < (uint32_t)p.nacc * p.acc_cols) cols <<= 1;
    p.tmem_cols = cols;
    p.b_bytes = (uint32_t)pb.C_out * BK * 2;
    p.wg = p.nT * pb.C_out <= 256 ? p.nT : 1;
    const size_t b_slot = (size_t)p.wg * p.b_bytes;
    // three A slots when at least four B slots still fit, else two; then 8, 6 or
    // 3 B slots, one producer per slot (3 measured faster than 4 when 4 fit:
    // fewer panels in flight)
    const size_t budget = 227 * 1024 - 3072;
    p.na = MAXA;
    while (p.na > 2 && (size_t)p.na * p.a_slot + 4 * b_slot > budget) --p.na;
    const size_t a_area = (size_t)p.na * p.a_slot;
    if (budget < a_area) return false;
    int nb = (int)((budget - a_area) / b_slot);
    if (nb > MAXB) nb = MAXB;
    if (nb < 2) return false;
    if (nb >= 8) { nb = 8; p.npb = 4; }
    else if (nb >= 6) { nb = 6; p.npb = 3; }
    else if (nb >= 3) { nb = 3; p.npb = 3; }
    else p.npb = nb;
    p.nb = nb;
    const size_t smem = a_area + (size_t)nb * b_slot + 1024;
    out->p = p;
    out->wq = wq;
    // channels-last x is read in place: no repacked copy
    out->x_bytes = pb.cl ? 0 : align256((size_t)pb.N * pb.C_in * pb.in_sp() * 2);
    out->w_bytes = align256((size_t)4 * SD * p.nTD * p.nT * p.nT * pb.C_out * pb.C_in * 2);
    out->smem = smem;
    return true;
}

}  // namespace

bool umma_supported(const Problem &pb, const Args *a)
{
    UPlan pl;
    if (!make_uplan(pb, &pl)) return false;
    if (a && (((uintptr_t)a->y % (pb.cl ? 16 : 8)) || ((uintptr_t)a->x % 16) || ((uintptr_t)a->w % 16)))
        return false;
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
    // channels last: x is already (N, D, H, W, C), the layout the A operand reads
    bf16_t *xt = pb.cl ? const_cast<bf16_t *>(static_cast<const bf16_t *>(a.x)) : static_cast<bf16_t *>(a.ws);
    bf16_t *wp = reinterpret_cast<bf16_t *>(static_cast<uint8_t *>(a.ws) + pl.x_bytes);

    // 1) x -> (N, D, H, W, C) and weights -> panels: one launch when D*H*W is
    // a multiple of 8, else the scalar x repack and the weight repack
    const int64_t SP = pb.in_sp();
    const int64_t nby = (pb.C_in + 63) / 64;
    cudaError_t e;
    if (pb.cl) {
        repack_w_kernel<<<dim3((unsigned)(pb.C_in / RB), (unsigned)pb.C_out), 256, 0, a.stream>>>(
            static_cast<const bf16_t *>(a.w), wp, pl.wq);
    } else if (SP % 8 == 0) {
        const int64_t nbx = (SP + RX - 1) / RX;
        const int64_t nxb = nbx * nby * pb.N;
        const int64_t nblocks = nxb + (int64_t)(pb.C_in / RB) * pb.C_out;
        if (nblocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
        repack_kernel<<<(unsigned)nblocks, 256, 0, a.stream>>>(static_cast<const bf16_t *>(a.x), xt, pb.C_in,
                                                              pb.Li[0], pb.Li[1], pb.Li[2], (int)nbx, (int)nby,
                                                              (int)nxb, static_cast<const bf16_t *>(a.w), wp, pl.wq);
    } else {
        const int64_t nbx = (SP + 63) / 64;
        dim3 gx((unsigned)nbx, (unsigned)nby, (unsigned)pb.N);
        if (gx.x > 0x7fffffffu || gx.y > 65535 || gx.z > 65535) return cudaErrorInvalidConfiguration;
        repack_x_scalar_kernel<<<gx, 256, 0, a.stream>>>(static_cast<const bf16_t *>(a.x), xt, pb.C_in, pb.Li[0],
                                                         pb.Li[1], pb.Li[2]);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        repack_w_kernel<<<dim3((unsigned)(pb.C_in / RB), (unsigned)pb.C_out), 256, 0, a.stream>>>(
            static_cast<const bf16_t *>(a.w), wp, pl.wq);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // 3) tensor maps: A over x_t viewed as (C, W, H, D, N), one input window per
    // box; B over the panels (K = C_in, rows), boxes of wg x C_out rows
    CUtensorMap tmA, tmB;
    const uint64_t adims[5] = {(uint64_t)pb.C_in, (uint64_t)pb.Li[2], (uint64_t)pb.Li[1], (uint64_t)pb.Li[0],
                               (uint64_t)pb.N};
    const uint64_t astr[4] = {(uint64_t)pb.C_in * 2, (uint64_t)pb.C_in * pb.Li[2] * 2,
                              (uint64_t)pb.C_in * pb.Li[2] * pb.Li[1] * 2,
                              (uint64_t)pb.C_in * pb.Li[2] * pb.Li[1] * pb.Li[0] * 2};
    const uint32_t abox[5] = {(uint32_t)BK, (uint32_t)p.wspan, (uint32_t)p.hspan, 1u, 1u};
    if (!encode_tiled(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, xt, adims, astr, abox,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const uint64_t bdims[2] = {(uint64_t)pb.C_in, (uint64_t)4 * p.SD * p.nTD * p.nT * p.nT * pb.C_out};
    const uint64_t bstr[1] = {(uint64_t)pb.C_in * 2};
    const uint32_t bbox[2] = {(uint32_t)BK, (uint32_t)(p.wg * pb.C_out)};
    if (!encode_tiled(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wp, bdims, bstr, bbox,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    int per_sm = 0;
    const void *fn_pair = pb.cl ? (const void *)&umma_ct3d_kernel<false, true>
                                : (const void *)&umma_ct3d_kernel<false, false>;
    const void *fn_split = pb.cl ? (const void *)&umma_ct3d_kernel<true, true>
                                 : (const void *)&umma_ct3d_kernel<true, false>;
    e = prepare_kernel(fn_pair, kThreads, pl.smem, &per_sm);
    if (e == cudaSuccess) e = prepare_kernel(fn_split, kThreads, pl.smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    unsigned int *status = device_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    int grid = sm_count();
    if (grid > p.ntiles) grid = p.ntiles;
    // tile pairs fill whole rounds of the grid; when the last round would leave
    // more than half the CTAs idle, its pairs are split into single tiles (a
    // single takes a little over half a pair's time), one round of them
    UParams pk = p;
    const int rem = grid > 0 ? p.ntiles % grid : 0;
    if (p.nacc == 2 && rem > 0 && 2 * rem <= grid) {
        pk.npair = p.ntiles - rem;
        pk.nunits = pk.npair + 2 * rem;
        if (pb.cl)
            return launch_dependent(umma_ct3d_kernel<true, true>, dim3((unsigned)grid), dim3(kThreads), pl.smem,
                                    a.stream, tmA, tmB, a.bias, a.y, pk, status);
        return launch_dependent(umma_ct3d_kernel<true, false>, dim3((unsigned)grid), dim3(kThreads), pl.smem,
                                a.stream, tmA, tmB, a.bias, a.y, pk, status);
    }
    if (pb.cl)
        return launch_dependent(umma_ct3d_kernel<false, true>, dim3((unsigned)grid), dim3(kThreads), pl.smem,
                                a.stream, tmA, tmB, a.bias, a.y, pk, status);
    return launch_dependent(umma_ct3d_kernel<false, false>, dim3((unsigned)grid), dim3(kThreads), pl.smem, a.stream,
                            tmA, tmB, a.bias, a.y, pk, status);
}

}  // namespace ct
