// ct_tc3d_split.cu -- FP32 ConvTranspose3d (and 2-D: a unit D dimension),
// plain or with the fused add + t*hardswish(t) epilogue, on the tensor cores
// (tcgen05), every operand split into parts whose products the tensor cores
// form exactly.
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
// Two splits, chosen by the caller:
//  * tf32x3 (CT_F32, the default).  v = t + l with t = tf32(v) (cvt.rna) and
//    l = tf32(v - t); v - t is exact in fp32, |v - t| <= 2^-11 |v| and
//    |v - t - l| <= 2^-22 |v|.  Per K step of 8 channels three kind::tf32
//    MMAs accumulate x_t w_t + x_t w_l + x_l w_t, every product exact in the
//    fp32 accumulator; the dropped x_l w_l and the two remainders are each
//    at most 2^-22 |x||w|, so an output lies within about 2^-20 of
//    sum |x||w| of the exact sum -- the accuracy of fp32 arithmetic over the
//    same terms.  A K block is 32 channels: the A stage holds, per position,
//    a 128-byte row of their t parts and one of their l parts (two TMA boxes,
//    two 16 KB halves); a run's panel its t rows, then its l rows.
//  * bf16x2 (CT_F32_BF16X2, opt-in).  hi = bf16(v) (round to nearest even),
//    lo = bf16(v - hi); the dropped remainder is below 2^-17 |v|.  Per K step
//    of 8 input channels the A row holds [x_hi | x_lo] of the 8 (16 bf16 =
//    32 bytes), and two kind::f16 MMAs of K = 16 multiply it by [w_hi | w_hi]
//    and by [w_lo | w_lo]: together (x_hi + x_lo)(w_hi + w_lo), so a product
//    carries a relative error of about 2^-16 at most.  An A row holds 32
//    channels; a run's panel is its hi rows, then its lo rows.
//
// Schedule.  A unit of work is 128 positions (whole W rows of MH H rows of
// one D plane) and one D residue rD, with the four (rH, rW) phases as four
// accumulators of C_out TMEM columns side by side (two such sets alternate
// across units when they fit, so the epilogue of one unit overlaps the MMAs
// of the next).  Every distinct input offset (dd, dh, dw) the unit reads is
// one A tile per K block; the phases that read it with some tap form runs of
// adjacent accumulators, and the weights of a run are stored as one panel, so
// that one MMA with N = run length x C_out serves the whole run.  The host
// orders the four accumulators so that the phases sharing an offset are
// adjacent as often as possible (with a 3-tap kernel the order (0,0), (0,1),
// (1,1), (1,0) makes every offset one run).  An MMA instruction costs the
// issuing thread about 100 clocks whatever its N, so wide runs are what keeps
// the tensor cores busy; the issue loop carries ring slots and parities as
// counters.
//
// Roles (persistent CTA, one per SM):
//   warps 0-2   TMA producers of the A ring (x_c 5-D boxes of 128 positions
//               x 128 bytes of channels at the offset; boxes reaching outside
//               the input read zeros, which is the boundary handling): three
//               for a ring of three slots, else two of them
//   warps 3-4   TMA producers of the B ring (a run's panel is two boxes: its
//               hi / t rows, then its lo / l rows).  Each ring slot has
//               exactly one producer, which refills it only after waiting for
//               its previous round, so a parity wait never has to tell two
//               phases apart
//   warp 5      TMEM allocation and MMA issue
//   warps 6-21  epilogue, in chunks of 16 channels of a unit; warp w reads TMEM
//               lane quarter w mod 4 for one H phase and 8 channels and adds
//               bias (and applies the fused epilogue) to each position's even
//               and odd W outputs, one float2.  Fused and channels first, the
//               warps load the add values from global memory a chunk ahead and
//               store y straight from registers (a warp's store covers whole
//               128-byte segments), so the kernel needs no staging buffers and
//               its B slots hold runs of N = 256.  Otherwise each chunk (16
//               channels x the unit's 2 MH output rows x the whole W extent,
//               32 KB) is staged in one of two or three shared-memory buffers,
//               the add values arriving there by a TMA load two chunks ahead
//   warp 22     chunk mover (staged epilogue): makes chunks ready one or two
//               ahead (the TMA load of the add values, or the release of the
//               buffer) and stores each written chunk with one TMA store (rows
//               and planes past the output are clipped)
// Every mbarrier wait is bounded: a timeout records CT_ERR_DEVICE_TIMEOUT in
// the device status word and the roles unwind (each producer waits, bounded,
// for its own TMA copies and the MMA issuer for its own MMAs before the TMEM
// is freed).
#include <cuda_bf16.h>
#include <string.h>

#include "ct_internal.h"
#include "ct_device.cuh"
#include "ct_tma.h"
#include "ct_tcgen05.cuh"
#include "ct_split.cuh"

namespace ct {
namespace {

constexpr int BM = 128;          // positions per unit (UMMA M)
constexpr int CK = 32;           // input channels per K block: one 128-byte row of bf16 (hi, lo) pairs, or
                                 // of tf32 t parts plus one of l parts
constexpr int NA = 4;            // A ring slots at most (bf16x2: up to 4 of 16 KB; tf32x3: 2 or 3 of 32 KB)
constexpr int NB = 2;            // B stages
constexpr int NE = 3;            // epilogue chunk buffers at most (16 channels of a unit, 32 KB each)
constexpr int NPA = 3;           // A producer warps: p.npa of them, warp q loading the A stages g with
                                 // g mod p.npa == q (p.npa divides the ring's p.na slots)
constexpr int NPB = 2;           // B producer warps: warp q loads the B stages g with g mod NPB == q
constexpr int MAXE = 18;         // input offsets per D residue (2 x 3 x 3 for extents <= 4)
constexpr int MAXR = 64;         // runs per D residue
constexpr int MAXSTEP = 320;     // MMA steps (B stages) per D residue
constexpr int EPW = 4;           // epilogue warps per TMEM lane quarter (H phase x channel half)
constexpr int kAWarp0 = 0;
constexpr int kBWarp0 = kAWarp0 + NPA;
constexpr int kMmaWarp = kBWarp0 + NPB;
constexpr int kEpiWarp0 = kMmaWarp + 1;
constexpr int kStoreWarp = kEpiWarp0 + 4 * EPW;
constexpr int kThreads = 32 * (kStoreWarp + 1);
constexpr uint32_t kAHalf = BM * 128;          // 128 positions x one 128-byte row: 16 KB
constexpr uint32_t kEChunk = 16 * 4 * BM * 4;  // 16 channels x 4 phases x 128 positions, fp32: 32 KB
constexpr int kEpiThreads = 32 * 4 * EPW;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
static_assert(NB % NPB == 0, "one producer per ring slot");

// One input offset a unit reads; its runs are run[rd][run0 .. run0 + nrun).
struct Entry {
    int8_t dd, dh, dw, nrun;
    int16_t run0, pad;
};
// Adjacent accumulators p0 .. p0 + len - 1 served by one weight panel whose
// hi rows start at row brow (lo rows follow after len x C_out rows).  fresh:
// the first MMA of the run writes (rather than adds to) its accumulators.
struct Run {
    int8_t p0, len, fresh, pad;
    int brow;
};
// One B stage of the issuer's schedule, in issue order (entries, then K
// blocks, then runs): flags bit 0 -- a new A stage starts here (wait for it),
// bit 1 -- the A stage is done after this one (release it), bit 2 -- the first
// MMA writes its accumulators; len: run length; col: first TMEM column.
struct Step {
    uint8_t flags, len;
    uint16_t col;
};

struct T3Params {
    int N, C_in, C_out;
    int SD;                      // D stride: 2, or 1 for a unit D dimension (a 2-D problem)
    int Lo0, Lo1, Lo2;
    int QD, QH, QW, MH, n_qhb;
    int n_kb;                    // K blocks: C_in / 32
    int na;                      // A ring slots
    int npa;                     // A producers (3 for a ring of 3 slots, else 2)
    int ne;                      // epilogue chunk buffers (staged epilogue: 2 or 3)
    uint32_t aslot;              // bytes of an A ring slot: 16 KB (bf16x2) or 32 KB (tf32x3: t rows, l rows)
    int nunits;
    int nacc;                    // accumulator sets (1 or 2)
    uint32_t acc_cols;           // 4 x C_out
    uint32_t tmem_cols;
    uint32_t bslot;              // bytes of a B ring slot
    uint32_t idesc_b[5];         // instruction descriptor for N = len x C_out, len 1..4
    int8_t slot[4];              // accumulator slot of phase (rH, rW) = index 2 rH + rW
    int nE[2];
    int nstep[2];
    Entry ent[2][MAXE];
    Run run[2][MAXR];
    Step step[2][MAXSTEP];
};


// ---- GEMM kernel ----------------------------------------------------------------
// unit -> (n, qd, qh block, rD); a unit D dimension (stride 1) has the one residue
// 0 and the unit index is (n, qd, qh block).  The two D residues of one position block are
// neighbours (their shared A tiles are reused from L2).  Units are dealt to the
// CTAs round-robin; rD = 1 has more taps than rD = 0 when the kernel extent is
// odd, and with an even grid a CTA would see one residue only, so the residue
// bit is flipped on every other round (each round's block of grid-size units is
// closed under flipping its low bit, so this permutes the units) and every CTA
// gets both residues in turn.
struct UnitCoord {
    int n, qd, qhb, rd;
};
__device__ __forceinline__ UnitCoord unit_coord(int u, const T3Params &p)
{
    UnitCoord c;
    c.rd = 0;
    if (p.SD == 2) {
        c.rd = (u ^ (u / (int)gridDim.x)) & 1;
        u >>= 1;
    }
    c.qhb = u % p.n_qhb;
    u /= p.n_qhb;
    c.qd = u % p.QD;
    c.n = u / p.QD;
    return c;
}

template <bool ADD, bool CL, bool TF>
__global__ void __launch_bounds__(kThreads, 1)
tc3d_split_kernel(const __grid_constant__ CUtensorMap tmXc,
                 const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW2,
                 const __grid_constant__ CUtensorMap tmW3, const __grid_constant__ CUtensorMap tmW4,
                 const __grid_constant__ CUtensorMap tmAdd, const __grid_constant__ CUtensorMap tmY,
                 const float *__restrict__ bias, const float *add_g, float *y_g,
                 const __grid_constant__ T3Params p, unsigned int *status)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t a_full[NA], a_empty[NA], b_full[NB], b_empty[NB], acc_full[2],
        acc_empty[2], drain_bar, e_full[NE], c_full[NE];
    __shared__ uint32_t tmem_slot;
    __shared__ float s_bias[128];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = sm;                                  // na x aslot
    uint8_t *sB = sm + (size_t)p.na * p.aslot;         // NB x bslot
    uint8_t *sE = sB + NB * p.bslot;                   // ne x kEChunk (staged epilogue only)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&tmXc);
        dev::prefetch_tensormap(&tmW1);
        dev::prefetch_tensormap(&tmW2);
        dev::prefetch_tensormap(&tmW3);
        dev::prefetch_tensormap(&tmW4);
        dev::prefetch_tensormap(&tmY);
        if (ADD) dev::prefetch_tensormap(&tmAdd);
        for (int s = 0; s < p.na; ++s) {
            dev::mbar_init(&a_full[s], 1);
            dev::mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < NB; ++s) {
            dev::mbar_init(&b_full[s], 1);
            dev::mbar_init(&b_empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            dev::mbar_init(&acc_full[a], 1);
            dev::mbar_init(&acc_empty[a], 32 * 4 * EPW);   // every epilogue thread
        }
        dev::mbar_init(&drain_bar, 1);
        for (int b = 0; b < NE; ++b) {
            dev::mbar_init(&e_full[b], 1);               // buffer ready for its chunk
            dev::mbar_init(&c_full[b], kEpiThreads);     // chunk written by every epilogue thread
        }
        dev::fence_mbar_init();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(&tmem_slot, p.tmem_cols);
    for (int i = threadIdx.x; i < p.C_out; i += blockDim.x) s_bias[i] = bias ? bias[i] : 0.f;
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // the operands in the workspace come from the prep kernel
    dev::griddep_wait();
    const uint32_t tmem = tmem_slot;
    const int nunit_cta =
        p.nunits > (int)blockIdx.x ? (p.nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int C_out = p.C_out, n_kb = p.n_kb;

    if (warp < kBWarp0 + NPB) {
        // ---------------- TMA producers.  One thread streams TMA boxes at about one
        // per 400 ns however deep the ring, so each ring has several producers,
        // warp q of a ring taking the stages g with g mod (producers) == q: the
        // ring slots g mod nst of one producer are its own.
        const bool isA = warp < kBWarp0;
        const int q = isA ? warp - kAWarp0 : warp - kBWarp0;
        if (lane == 0 && (!isA || q < p.npa)) {
            const int np = isA ? p.npa : NPB;
            const int nst = isA ? p.na : NB;
            uint64_t *fullb = isA ? a_full : b_full;
            uint64_t *emptyb = isA ? a_empty : b_empty;
            int g = 0, s = 0, last = -1;             // ring position, slot
            uint32_t round_par = 0;                  // parity of g / nst
            bool failed = false;
            for (int k = 0; k < nunit_cta && !failed; ++k) {
                const UnitCoord u = unit_coord((int)blockIdx.x + k * (int)gridDim.x, p);
                const int qh0 = u.qhb * p.MH;
                const int ne = p.nE[u.rd];
                for (int e = 0; e < ne && !failed; ++e) {
                    const Entry &en = p.ent[u.rd][e];
                    for (int kb = 0; kb < n_kb && !failed; ++kb) {
                        const int nload = isA ? 1 : en.nrun;
                        for (int j = 0; j < nload; ++j) {
                            if (g % np == q) {
                                if (g >= nst &&
                                    !dev::mbar_wait_bounded(&emptyb[s], round_par ^ 1u, kWaitLimitNs)) {
                                    failed = true;
                                    break;
                                }
                                if (isA) {
                                    // the K block's 128-byte rows (tf32x3: the t rows, then
                                    // the l rows 16 KB further)
                                    uint8_t *dst = sA + (size_t)s * p.aslot;
                                    dev::mbar_arrive_expect_tx(&fullb[s], p.aslot);
                                    dev::tma_load_5d(dst, &tmXc, &fullb[s], kb * 64, en.dw, qh0 + en.dh,
                                                     u.qd + en.dd, u.n);
                                    if (TF)
                                        dev::tma_load_5d(dst + kAHalf, &tmXc, &fullb[s], kb * 64 + 32, en.dw,
                                                         qh0 + en.dh, u.qd + en.dd, u.n);
                                } else {
                                    // the run's panel exactly: two boxes of len x C_out rows of the
                                    // K block's 128 bytes, the hi / t rows, then the lo / l rows
                                    const Run &ru = p.run[u.rd][en.run0 + j];
                                    const CUtensorMap *tm = ru.len == 1 ? &tmW1 : ru.len == 2 ? &tmW2
                                                          : ru.len == 3 ? &tmW3 : &tmW4;
                                    const uint32_t half = (uint32_t)(ru.len * C_out) * 128u;
                                    uint8_t *dst = sB + (size_t)s * p.bslot;
                                    dev::mbar_arrive_expect_tx(&fullb[s], 2 * half);
                                    dev::tma_load_2d(dst, tm, &fullb[s], kb * CK, ru.brow);
                                    dev::tma_load_2d(dst + half, tm, &fullb[s], kb * CK, ru.brow + ru.len * C_out);
                                }
                                last = g;
                            }
                            ++g;
                            if (++s == nst) {
                                s = 0;
                                round_par ^= 1u;
                            }
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
            const uint32_t sAb = dev::smem_u32(sA), sBb = dev::smem_u32(sB);
            const uint32_t bslot = p.bslot, aslot = p.aslot;
            const int na = p.na;
            int sa = 0, sb = 0;
            uint32_t pa = 0, pb = 0;
            // instruction descriptors by run length, held in registers
            const uint32_t id1 = p.idesc_b[1], id2 = p.idesc_b[2], id3 = p.idesc_b[3], id4 = p.idesc_b[4];
            for (int k = 0; k < nunit_cta && ok; ++k) {
                const int rd = unit_coord((int)blockIdx.x + k * (int)gridDim.x, p).rd;
                const int a = p.nacc == 2 ? (k & 1) : 0;
                const int use = p.nacc == 2 ? (k >> 1) : k;     // earlier units in accumulator set a
                const int nst = p.nstep[rd];
                Step nxt = p.step[rd][0];
                if (use > 0 && !dev::mbar_wait_bounded(&acc_empty[a], (use - 1) & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)a * p.acc_cols;
                uint64_t da = 0;
                // one flat schedule per residue; the next step's record is read while
                // this one waits and issues
                for (int i = 0; i < nst && ok; ++i) {
                    const Step st = nxt;
                    if (i + 1 < nst) nxt = p.step[rd][i + 1];
                    if (st.flags & 1u) {
                        if (!dev::mbar_wait_bounded(&a_full[sa], pa, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after();
                        da = tc::desc_sw128(sAb + (uint32_t)sa * aslot);
                    }
                    if (!dev::mbar_wait_bounded(&b_full[sb], pb, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t bh = sBb + (uint32_t)sb * bslot;
                    const uint64_t dbh = tc::desc_sw128(bh);
                    const uint64_t dbl = tc::desc_sw128(bh + (uint32_t)(st.len * C_out) * 128u);
                    const uint32_t idb = st.len == 1 ? id1 : st.len == 2 ? id2 : st.len == 3 ? id3 : id4;
                    const uint32_t dd = d + (uint32_t)st.col;
                    const uint32_t acc0 = (st.flags & 4u) ? 0u : 1u;
                    if (TF) {
                        // K step kk: 8 channels, 32 bytes of the t rows (A, and the
                        // panel's t rows) and of the l rows (A 16 KB further, the
                        // panel's l rows after its t rows); descriptor units of 16 bytes
                        const uint64_t dal = da + (kAHalf >> 4);
#pragma unroll
                        for (int kk = 0; kk < CK / 8; ++kk) {
                            tc::mma_tf32(dd, da + 2 * kk, dbh + 2 * kk, idb, kk ? 1u : acc0);   // x_t w_t
                            tc::mma_tf32(dd, da + 2 * kk, dbl + 2 * kk, idb, 1u);             // x_t w_l
                            tc::mma_tf32(dd, dal + 2 * kk, dbh + 2 * kk, idb, 1u);            // x_l w_t
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < CK / 8; ++kk) {
                            // 32 bytes along K inside the swizzle atom: 16 bf16, the
                            // hi and lo parts of 8 channels
                            tc::mma_bf16(dd, da + 2 * kk, dbh + 2 * kk, idb, kk ? 1u : acc0);   // x * w_hi
                            tc::mma_bf16(dd, da + 2 * kk, dbl + 2 * kk, idb, 1u);             // x * w_lo
                        }
                    }
                    tc::commit(&b_empty[sb]);
                    if (++sb == NB) {
                        sb = 0;
                        pb ^= 1u;
                    }
                    if (st.flags & 2u) {
                        tc::commit(&a_empty[sa]);
                        if (++sa == na) {
                            sa = 0;
                            pa ^= 1u;
                        }
                    }
                }
                if (ok) tc::commit(&acc_full[a]);
            }
            // every MMA issued has to complete before the TMEM is freed
            tc::commit(&drain_bar);
            if (!dev::mbar_wait_bounded(&drain_bar, 0, kWaitLimitNs)) ok = false;
            if (!ok) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
        }
    } else if (warp == kStoreWarp) {
        if (ADD && !CL) goto done;                  // fused, channels first: the epilogue warps store directly
        // ---------------- chunk mover (staged epilogue).  Buffer gc mod ne holds chunk gc (16 channels of a
        // unit: 16 x 2 MH rows x the whole W extent, 32 KB).  Chunk gc is made ready
        // ne - 1 chunks ahead -- its add values loaded by TMA, or (no add) the buffer
        // released -- and stored by TMA once the epilogue warps have written it.
        const int nchunk = C_out / 16;
        const int total = nunit_cta * nchunk;
        const int ne = p.ne;
        bool ok = true;
        auto ready = [&](int gc) {
            const int b = gc % ne;
            if (ADD) {
                const UnitCoord v = unit_coord((int)blockIdx.x + (gc / nchunk) * (int)gridDim.x, p);
                dev::mbar_arrive_expect_tx(&e_full[b], kEChunk);
                if (CL)    // (C_out, W, H, D, N): 16 channels of every position of the chunk
                    dev::tma_load_5d(sE + (size_t)b * kEChunk, &tmAdd, &e_full[b], (gc % nchunk) * 16, 0,
                                     2 * v.qhb * p.MH, p.SD * v.qd + v.rd, v.n);
                else
                    dev::tma_load_4d(sE + (size_t)b * kEChunk, &tmAdd, &e_full[b], 0, 2 * v.qhb * p.MH,
                                     p.SD * v.qd + v.rd, v.n * C_out + (gc % nchunk) * 16);
            } else {
                dev::mbar_arrive(&e_full[b]);
            }
        };
        if (lane == 0) {
            for (int gc = 0; gc < ne - 1 && gc < total; ++gc) ready(gc);
            for (int gc = 0; gc < total && ok; ++gc) {
                // the epilogue threads wrote chunk gc (they run at most ne - 1 chunks ahead,
                // so the parity of a buffer's barrier is unambiguous)
                if (!dev::mbar_wait_bounded(&c_full[gc % ne], (gc / ne) & 1, kWaitLimitNs)) {
                    atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                    ok = false;
                    break;
                }
                const UnitCoord u = unit_coord((int)blockIdx.x + (gc / nchunk) * (int)gridDim.x, p);
                // rows and planes past the output are clipped by the store
                if (CL)
                    dev::tma_store_5d(&tmY, sE + (size_t)(gc % ne) * kEChunk, (gc % nchunk) * 16, 0,
                                      2 * u.qhb * p.MH, p.SD * u.qd + u.rd, u.n);
                else
                    dev::tma_store_4d(&tmY, sE + (size_t)(gc % ne) * kEChunk, 0, 2 * u.qhb * p.MH,
                                      p.SD * u.qd + u.rd, u.n * C_out + (gc % nchunk) * 16);
                dev::bulk_commit();
                dev::bulk_wait_read<1>();               // chunk gc - 1's store has read its buffer
                if (gc + ne - 1 < total) ready(gc + ne - 1);   // into that buffer
            }
            dev::bulk_wait_all();
            // loads this thread issued that nobody consumed (only after a timeout)
            if (ADD)
                for (int r = total - (ne - 1) > 0 ? total - (ne - 1) : 0; r < total; ++r)
                    dev::mbar_wait_bounded(&e_full[r % ne], (r / ne) & 1, kWaitLimitNs);
        }
    } else {
        // ---------------- epilogue: warp w reads TMEM lane quarter w mod 4; the four
        // warps of a quarter take (H phase, channel half) = ((e >> 2) & 1, e >> 3),
        // e = w - first epilogue warp.  Per chunk a warp waits for the buffer, adds
        // bias (and applies the fused epilogue) in place for its 8 channels, and
        // signals the chunk mover.
        const int ew = warp & 3;
        const int ei = warp - kEpiWarp0;
        const int rh = (ei >> 2) & 1, ch = ei >> 3;
        const int nchunk = C_out / 16;
        const int Lo2 = p.Lo2;
        const int cstride = 2 * p.MH * Lo2 / 2;         // float2 between channels of a chunk
        bool ok = true;
        int gc = 0;
        if (ADD && !CL) {
            // fused, channels first, straight from the accumulators to y: a thread holds
            // position m, output row 2 qh + rh, and for 8 channels of a 16-channel
            // chunk its two W outputs 2 qw, 2 qw + 1 -- one float2 per channel; a
            // warp's 32 positions are whole runs of a row (QW >= 16), so every store
            // instruction covers whole 128-byte segments.  The add values of the
            // next chunk are loaded while this one is computed (and the chunk after
            // is prefetched into L2), so the add stream keeps a chunk in flight.
            const int m = ew * 32 + lane;
            const int qwp = m % p.QW, qhl = m / p.QW;
            const int64_t sp = (int64_t)p.Lo0 * p.Lo1 * Lo2;
            // output offset (floats) of the thread's first channel for unit k, or -1
            auto out_off = [&](int k2) -> int64_t {
                const UnitCoord v = unit_coord((int)blockIdx.x + k2 * (int)gridDim.x, p);
                const int od = p.SD * v.qd + v.rd, oh = 2 * (v.qhb * p.MH + qhl) + rh;
                if (od >= p.Lo0 || oh >= p.Lo1) return -1;
                return ((int64_t)v.n * C_out * p.Lo0 + od) * p.Lo1 * (int64_t)Lo2 + (int64_t)oh * Lo2 + 2 * qwp;
            };
            float2 av[8], an[8];
            int64_t off = nunit_cta > 0 ? out_off(0) : -1;
            if (ADD && off >= 0) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    av[i] = __ldcs(reinterpret_cast<const float2 *>(add_g + off + (int64_t)(ch * 8 + i) * sp));
            }
            for (int k = 0; k < nunit_cta; ++k) {
                const int a = p.nacc == 2 ? (k & 1) : 0;
                const int use = p.nacc == 2 ? (k >> 1) : k;
                const int64_t off_next = k + 1 < nunit_cta ? out_off(k + 1) : -1;
                if (ok && !dev::mbar_wait_bounded(&acc_full[a], use & 1, kWaitLimitNs)) {
                    atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                    ok = false;
                }
                ok = __all_sync(0xffffffffu, ok);        // warp-uniform before .sync.aligned loads
                tc::fence_after();
                const uint32_t tbase = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)a * p.acc_cols;
                for (int c = 0; c < nchunk; ++c) {
                    const int c0 = c * 16 + ch * 8;             // this warp's first channel
                    float v0[8], v1[8];
                    if (ok) {
                        // the accumulators of phases (rh, 0) and (rh, 1)
                        tc::tmem_ld8(tbase + (uint32_t)(p.slot[rh * 2] * C_out + c0), v0);
                        tc::tmem_ld8(tbase + (uint32_t)(p.slot[rh * 2 + 1] * C_out + c0), v1);
                    }
                    // the next chunk's add values (this unit's, or the next unit's first)
                    const int64_t noff = c + 1 < nchunk ? (off >= 0 ? off + (int64_t)16 * sp : -1) : off_next;
                    const int nc0 = c + 1 < nchunk ? c0 + 16 : ch * 8;
                    if (ADD && noff >= 0) {
                        const int64_t base = c + 1 < nchunk ? off : off_next;
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            an[i] = __ldcs(reinterpret_cast<const float2 *>(add_g + base + (int64_t)(nc0 + i) * sp));
                    }
                    if (ADD && c + 2 < nchunk) {
                        // two chunks ahead, into L2: the warp's 8 channels cover two
                        // 128-byte lines each (positions of lanes 0-15 and 16-31); lane l
                        // < 16 prefetches line l & 1 of channel l >> 1
                        const int64_t src = __shfl_sync(0xffffffffu, off, (lane & 1) * 16);
                        if (lane < 16 && src >= 0)
                            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(add_g + src + (int64_t)(c0 + 32 + (lane >> 1)) * sp));
                    }
                    tc::tmem_wait_ld();
                    if (c == nchunk - 1) {                  // the unit's last loads: free the accumulators
                        tc::fence_before();
                        dev::mbar_arrive(&acc_empty[a]);
                    }
                    if (ok && off >= 0) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float bb = s_bias[c0 + i];
                            float t0 = v0[i] + bb, t1 = v1[i] + bb;
                            if (ADD) {
                                t0 = add_hswish(t0, av[i].x);
                                t1 = add_hswish(t1, av[i].y);
                            }
                            __stcs(reinterpret_cast<float2 *>(y_g + off + (int64_t)(c0 + i) * sp), make_float2(t0, t1));
                        }
                    }
                    if (ADD) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) av[i] = an[i];
                    }
                    if (c + 1 == nchunk) off = off_next;
                }
            }
        } else {
        for (int k = 0; k < nunit_cta; ++k) {
            const int a = p.nacc == 2 ? (k & 1) : 0;
            const int use = p.nacc == 2 ? (k >> 1) : k;
            if (ok && !dev::mbar_wait_bounded(&acc_full[a], use & 1, kWaitLimitNs)) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);        // warp-uniform before .sync.aligned loads
            tc::fence_after();
            const int m = ew * 32 + lane;
            const int row = 2 * (m / p.QW) + rh, qw = m % p.QW;
            const uint32_t tbase = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)a * p.acc_cols;
            for (int c = 0; c < nchunk; ++c, ++gc) {
                const int b = gc % p.ne;
                const int c0 = c * 16 + ch * 8;             // this warp's first channel
                float2 *q = reinterpret_cast<float2 *>(sE + (size_t)b * kEChunk) + (row * Lo2 + 2 * qw) / 2 +
                            ch * 8 * cstride;
                float v0[8], v1[8];
                if (ok) {
                    // the accumulators of phases (rh, 0) and (rh, 1)
                    tc::tmem_ld8(tbase + (uint32_t)(p.slot[rh * 2] * C_out + c0), v0);
                    tc::tmem_ld8(tbase + (uint32_t)(p.slot[rh * 2 + 1] * C_out + c0), v1);
                }
                if (ok && !dev::mbar_wait_bounded(&e_full[b], (gc / p.ne) & 1, kWaitLimitNs)) {
                    atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                    ok = false;
                }
                ok = __all_sync(0xffffffffu, ok);
                tc::tmem_wait_ld();
                if (c == nchunk - 1) {                  // the unit's last loads: free the accumulators
                    tc::fence_before();
                    dev::mbar_arrive(&acc_empty[a]);
                }
                if (CL) {
                    // channels last: the chunk buffer is the (16 channels, W, 2 MH rows)
                    // box of the 5-D maps, 64-byte rows (one position's 16 channels) in
                    // the 64-byte swizzle -- the 16-byte unit index (address bits 4-5)
                    // XORed with address bits 7-8 -- which spreads a warp's accesses
                    // (positions 128 bytes apart) over four bank groups.  This warp's
                    // 8 channels of positions 2 qw and 2 qw + 1: two 16-byte units each.
                    if (ok) {
                        uint8_t *buf = sE + (size_t)b * kEChunk;
#pragma unroll
                        for (int w2 = 0; w2 < 2; ++w2) {
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const uint32_t L = (uint32_t)(((row * Lo2 + 2 * qw + w2) * 16 + ch * 8 + 4 * j) * 4);
                                float4 *ptr = reinterpret_cast<float4 *>(buf + (L ^ (((L >> 7) & 3u) << 4)));
                                const int cc = c0 + 4 * j;
                                const float e0 = w2 ? v1[4 * j] : v0[4 * j], e1 = w2 ? v1[4 * j + 1] : v0[4 * j + 1];
                                const float e2 = w2 ? v1[4 * j + 2] : v0[4 * j + 2], e3 = w2 ? v1[4 * j + 3] : v0[4 * j + 3];
                                float4 t = make_float4(e0 + s_bias[cc], e1 + s_bias[cc + 1], e2 + s_bias[cc + 2],
                                                       e3 + s_bias[cc + 3]);
                                if (ADD) {
                                    const float4 av = *ptr;
                                    t = make_float4(add_hswish(t.x, av.x), add_hswish(t.y, av.y), add_hswish(t.z, av.z),
                                                    add_hswish(t.w, av.w));
                                }
                                *ptr = t;
                            }
                        }
                    }
                    dev::fence_proxy_async();
                    dev::mbar_arrive(&c_full[b]);
                    continue;
                }
                if (ok) {
                    // all loads first, then the arithmetic and the stores
                    float2 av[8];
                    if (ADD) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) av[i] = q[i * cstride];
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float bb = s_bias[c0 + i];
                        float t0 = v0[i] + bb, t1 = v1[i] + bb;
                        if (ADD) {
                            t0 = add_hswish(t0, av[i].x);
                            t1 = add_hswish(t1, av[i].y);
                        }
                        q[i * cstride] = make_float2(t0, t1);
                    }
                }
                dev::fence_proxy_async();
                dev::mbar_arrive(&c_full[b]);
            }
        }
        }
    }

done:
    __syncwarp();
    tc::fence_before();
    __syncthreads();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, p.tmem_cols);
}

// ---- host side ------------------------------------------------------------------
struct T3Plan {
    T3Params p;
    WPanels wq;
    int maxlen;                  // longest run
    size_t x_bytes, w_bytes, smem;
};

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

// Entries and runs of both D residues for one order of the accumulators
// (phase_of_slot[s] = phase 2 rH + rW held in slot s).  Fills p.ent, p.run,
// p.nE and the panel blocks of wq; *cost estimates the MMA-issue time of a
// unit pair: per run and K block a B stage (~150 clocks of waits and a
// commit) and its MMAs (~80 clocks each up to N = 128, the tensor-pipe time
// beyond).
bool plan_runs(const Problem &pb, int SD, const int (&nt)[3][2], const int (&tk)[3][2][4],
               const int (&td)[3][2][4], const int (&uo)[3][4], const int (&nu)[3], const int *phase_of_slot,
               int maxlen, int bmul, int mma_per_stage, T3Params *pp, WPanels *wq, double *cost)
{
    T3Params &p = *pp;
    int nblk = 0;
    double c = 0;
    for (int rd = 0; rd < SD; ++rd) {
        int ne = 0, nr = 0;
        uint32_t init = 0;                        // accumulator slots written by earlier runs
        for (int jd = 0; jd < nt[0][rd]; ++jd)
            for (int ih = 0; ih < nu[1]; ++ih)
                for (int iw = 0; iw < nu[2]; ++iw) {
                    // phases reading offset (dd, dh, dw), with their taps
                    int tap_ph[4] = {-1, -1, -1, -1};
                    for (int rh = 0; rh < 2; ++rh)
                        for (int jh = 0; jh < nt[1][rh]; ++jh) {
                            if (td[1][rh][jh] != uo[1][ih]) continue;
                            for (int rw = 0; rw < 2; ++rw)
                                for (int jw = 0; jw < nt[2][rw]; ++jw) {
                                    if (td[2][rw][jw] != uo[2][iw]) continue;
                                    tap_ph[rh * 2 + rw] =
                                        (tk[0][rd][jd] * pb.K[1] + tk[1][rh][jh]) * pb.K[2] + tk[2][rw][jw];
                                }
                        }
                    int tap_of[4];
                    for (int sl = 0; sl < 4; ++sl) tap_of[sl] = tap_ph[phase_of_slot[sl]];
                    Entry en;
                    memset(&en, 0, sizeof(en));
                    en.dd = (int8_t)td[0][rd][jd];
                    en.dh = (int8_t)uo[1][ih];
                    en.dw = (int8_t)uo[2][iw];
                    en.run0 = (int16_t)nr;
                    int ph = 0;
                    while (ph < 4) {
                        if (tap_of[ph] < 0) {
                            ++ph;
                            continue;
                        }
                        // a run: adjacent slots with a tap here, the same written state,
                        // at most maxlen long
                        const bool st = (init >> ph) & 1u;
                        int len = 1;
                        while (ph + len < 4 && len < maxlen && tap_of[ph + len] >= 0 &&
                               (((init >> (ph + len)) & 1u) != 0) == st)
                            ++len;
                        if (nr >= MAXR || nblk + bmul * len > kMaxBlk) return false;
                        Run ru;
                        memset(&ru, 0, sizeof(ru));
                        ru.p0 = (int8_t)ph;
                        ru.len = (int8_t)len;
                        ru.fresh = st ? 0 : 1;
                        ru.brow = nblk * pb.C_out;
                        for (int hl = 0; hl < bmul; ++hl)
                            for (int i = 0; i < len; ++i) {
                                wq->blk_tap[nblk] = (int16_t)tap_of[ph + i];
                                wq->blk_lo[nblk] = (int8_t)hl;
                                ++nblk;
                            }
                        for (int i = 0; i < len; ++i) init |= 1u << (ph + i);
                        p.run[rd][nr++] = ru;
                        ++en.nrun;
                        const double n = (double)(len * pb.C_out);
                        c += 150.0 + mma_per_stage * (n <= 128 ? 80.0 : 80.0 * n / 128.0);
                        ph += len;
                    }
                    if (en.nrun == 0) continue;
                    if (ne >= MAXE) return false;
                    p.ent[rd][ne++] = en;
                }
        if (init != 0xFu) return false;           // every accumulator of the unit is written
        p.nE[rd] = ne;
    }
    wq->nblk = nblk;
    *cost = c;
    return true;
}

bool make_t3plan(const Problem &pb, const Args *a, T3Plan *out)
{
    if ((pb.nd != 3 && pb.nd != 2) || pb.dtype != CT_F32 || pb.G != 1) return false;
    const bool tf = !pb.split2;          // tf32x3 unless the caller opted into the bf16 pair
    // D has stride 2 like H and W, or is a unit dimension (extent 1, stride 1, no
    // padding: a 2-D problem, or a 3-D one that maps planes to planes), whose
    // single residue takes tap 0 at offset 0
    const int SD = pb.S[0];
    if (SD == 1 && (pb.K[0] != 1 || pb.P[0] != 0 || pb.OP[0] != 0)) return false;
    for (int d = SD == 1 ? 1 : 0; d < 3; ++d)
        if (pb.S[d] != 2 || pb.DL[d] != 1 || pb.K[d] < 2 || pb.K[d] > 4) return false;
    if (pb.C_in % 32 != 0 || pb.C_out % 16 != 0 || pb.C_out < 16 || pb.C_out > 128) return false;
    // the epilogue moves whole output rows by TMA: 16-byte rows and bases
    if (pb.Lo[2] % 4 != 0 || pb.in_sp() % 4 != 0) return false;
    if (a && (((uintptr_t)a->x % 16) || ((uintptr_t)a->y % 16) || (a->add && ((uintptr_t)a->add % 16))))
        return false;
    T3Params p;
    memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C_in = pb.C_in; p.C_out = pb.C_out;
    p.SD = SD;
    p.Lo0 = pb.Lo[0]; p.Lo1 = pb.Lo[1]; p.Lo2 = pb.Lo[2];
    p.QW = p.Lo2 / 2;
    if (p.QW > BM || BM % p.QW != 0) return false;
    p.MH = BM / p.QW;
    p.QD = (p.Lo0 + SD - 1) / SD;
    p.QH = (p.Lo1 + 1) / 2;
    p.n_qhb = (p.QH + p.MH - 1) / p.MH;
    p.n_kb = pb.C_in / CK;
    p.na = NA;                   // reduced to fit below
    p.aslot = (tf ? 2 : 1) * kAHalf;
    const int64_t units = (int64_t)pb.N * p.QD * p.n_qhb * SD;
    if (units > 0x7fffffff || units == 0) return false;
    p.nunits = (int)units;

    // per dimension and residue: taps and input offsets
    int tk[3][2][4], td[3][2][4], nt[3][2];
    for (int d = 0; d < 3; ++d)
        for (int r = 0; r < 2; ++r) {
            if (d == 0 && SD == 1) {
                nt[0][r] = r == 0 ? 1 : 0;
                tk[0][r][0] = td[0][r][0] = 0;
                continue;
            }
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
    // runs of adjacent accumulators: at most 4 phases, N = len x C_out <= 256 (a
    // panel is two boxes of len x C_out rows).
    // fused and channels first, the epilogue stores from registers (no staging
    // buffers): B slots of 256 panel rows (runs of N = 256); otherwise the
    // staging buffers leave room for 128 rows
    const bool direct = pb.has_add && !pb.cl;
    int maxlen = (direct ? 256 : 128) / pb.C_out;
    if (maxlen > 4) maxlen = 4;
    // shared memory: A ring, B ring (slots of the longest run's panel) and, staged,
    // the epilogue's chunk buffers.  Without an add, a ring of four A slots
    // gives way to three and the third chunk buffer goes next (the A loads'
    // latency, not the stores', holds the MMAs up there: 2-D 0.303 against
    // 0.317 ms); with one, four A slots give way to two (three measured 5 %
    // slower on the fused workload).  Then runs get shorter, until they fit
    int ne = direct ? 0 : NE;
    {
        const size_t budget = 227 * 1024 - 2048;   // room for the alignment pad and the static barriers
        while ((size_t)p.na * p.aslot + (size_t)NB * (2 * maxlen * pb.C_out) * 128 + (size_t)ne * kEChunk >
               budget) {
            if (p.na > 3) p.na = pb.has_add ? 2 : 3;
            else if (!pb.has_add && ne > 2) ne = 2;
            else if (p.na > 2) p.na = 2;
            else if (maxlen > 1) --maxlen;
            else return false;
        }
    }
    p.npa = p.na == 3 ? 3 : 2;
    p.ne = direct ? 1 : ne;
    // the order of the four accumulators with the cheapest MMA schedule (the
    // first of equal ones, so the natural order when it is as good)
    static const int kPerm[24][4] = {
        {0, 1, 2, 3}, {0, 1, 3, 2}, {0, 2, 1, 3}, {0, 2, 3, 1}, {0, 3, 1, 2}, {0, 3, 2, 1},
        {1, 0, 2, 3}, {1, 0, 3, 2}, {1, 2, 0, 3}, {1, 2, 3, 0}, {1, 3, 0, 2}, {1, 3, 2, 0},
        {2, 0, 1, 3}, {2, 0, 3, 1}, {2, 1, 0, 3}, {2, 1, 3, 0}, {2, 3, 0, 1}, {2, 3, 1, 0},
        {3, 0, 1, 2}, {3, 0, 2, 1}, {3, 1, 0, 2}, {3, 1, 2, 0}, {3, 2, 0, 1}, {3, 2, 1, 0}};
    WPanels wq;
    double best = 0;
    int bi = -1;
    for (int i = 0; i < 24; ++i) {
        WPanels wt;
        memset(&wt, 0, sizeof(wt));
        double c = 0;
        if (!plan_runs(pb, SD, nt, tk, td, uo, nu, kPerm[i], maxlen, 2, tf ? 12 : 8, &p, &wt, &c)) continue;
        if (bi < 0 || c < best - 1e-9) {
            best = c;
            bi = i;
        }
    }
    if (bi < 0) return false;
    memset(&wq, 0, sizeof(wq));
    double c = 0;
    if (!plan_runs(pb, SD, nt, tk, td, uo, nu, kPerm[bi], maxlen, 2, tf ? 12 : 8, &p, &wq, &c)) return false;
    for (int sl = 0; sl < 4; ++sl) p.slot[kPerm[bi][sl]] = (int8_t)sl;
    // the issuer's flat schedule per residue: entries, K blocks, runs
    for (int rd = 0; rd < SD; ++rd) {
        int ns = 0;
        for (int e = 0; e < p.nE[rd]; ++e) {
            const Entry &en = p.ent[rd][e];
            for (int kb = 0; kb < p.n_kb; ++kb)
                for (int j = 0; j < en.nrun; ++j) {
                    if (ns >= MAXSTEP) return false;
                    const Run &ru = p.run[rd][en.run0 + j];
                    Step st;
                    st.flags = (uint8_t)((j == 0 ? 1 : 0) | (j == en.nrun - 1 ? 2 : 0) |
                                         ((ru.fresh && kb == 0) ? 4 : 0));
                    st.len = (uint8_t)ru.len;
                    st.col = (uint16_t)(ru.p0 * pb.C_out);
                    p.step[rd][ns++] = st;
                }
        }
        p.nstep[rd] = ns;
    }
    wq.C_in = pb.C_in;
    wq.C_out = pb.C_out;
    wq.ntap = pb.kvol();
    wq.tf = tf ? 1 : 0;
    for (int len = 1; len <= 4; ++len)
        p.idesc_b[len] = len * pb.C_out <= 256 ? tc::idesc(tf ? 2 : 1, len * pb.C_out, BM) : 0u;
    p.acc_cols = (uint32_t)(4 * pb.C_out);
    p.nacc = 8 * pb.C_out <= 512 ? 2 : 1;
    uint32_t cols = 32;
    while (cols < (uint32_t)p.nacc * p.acc_cols) cols <<= 1;
    p.tmem_cols = cols;
    p.bslot = (uint32_t)(2 * maxlen * pb.C_out) * 128u;
    const size_t smem = (size_t)p.na * p.aslot + (size_t)NB * p.bslot + (size_t)ne * kEChunk + 1024;
    if (smem > 227 * 1024 - 1024) return false;   // room for the static barriers
    out->p = p;
    out->wq = wq;
    out->maxlen = maxlen;
    // x_c: 8 bytes per value (tf32 t and l) or 4 (bf16 hi and lo); a panel row 4
    // bytes per input channel (a tf32 part, or a pair of bf16 parts)
    out->x_bytes = align256((size_t)pb.N * pb.C_in * pb.in_sp() * (tf ? 8 : 4));
    out->w_bytes = align256((size_t)wq.nblk * pb.C_out * pb.C_in * 4);
    out->smem = smem;
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
    return pl.x_bytes + pl.w_bytes;
}

cudaError_t launch_tc3d(const Problem &pb, const Args &a)
{
    T3Plan pl;
    if (!make_t3plan(pb, &a, &pl)) return cudaErrorNotSupported;
    const T3Params &p = pl.p;
    const bool tf = pl.wq.tf != 0;
    uint8_t *ws = static_cast<uint8_t *>(a.ws);
    uint32_t *xc = reinterpret_cast<uint32_t *>(ws);
    float *wp = reinterpret_cast<float *>(ws + pl.x_bytes);

    // 1) one launch: x -> channels-last split (tf32 t, l or bf16 hi, lo), weights ->
    // run panels (channels-last x: the split alone, 1024 values per block)
    const int64_t SP = pb.in_sp();
    const int64_t nbx = (SP + 63) / 64, nby = pb.C_in / 32;
    const int64_t cl_total = pb.cl ? (int64_t)pb.N * SP * pb.C_in : 0;
    const int64_t nxb = pb.cl ? (cl_total + 1023) / 1024 : nbx * nby * pb.N;
    const int64_t wtot = (int64_t)pl.wq.nblk * pb.C_out * pb.C_in;
    int nbw = (int)((wtot + 255) / 256);
    if (nbw > 4 * sm_count()) nbw = 4 * sm_count();
    if (nxb + nbw > 0x7fffffff) return cudaErrorInvalidConfiguration;
    prep_kernel<<<(unsigned)(nxb + nbw), 256, 0, a.stream>>>(static_cast<const float *>(a.x), xc, pb.C_in, SP,
                                                            (int)nbx, (int)nby, (int)nxb,
                                                            static_cast<const float *>(a.w), wp, pl.wq, nbw,
                                                            cl_total);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // 2) tensor maps: A over x_c (2C, W, H, D, N) of fp32 words (tf32x3) or bf16
    // (bf16x2), a box of one 128-byte row per position; B over the panels (rows
    // of C_in words), one map per run length len (a box of 2 x len x C_out
    // rows: the run's panel)
    CUtensorMap tmXc, tmW[4];
    const uint64_t vb = tf ? 8 : 4;          // bytes of x_c per input channel
    const uint64_t astr[4] = {(uint64_t)pb.C_in * vb, (uint64_t)pb.C_in * pb.Li[2] * vb,
                              (uint64_t)pb.C_in * pb.Li[2] * pb.Li[1] * vb,
                              (uint64_t)pb.C_in * pb.Li[2] * pb.Li[1] * pb.Li[0] * vb};
    const uint64_t cdims[5] = {(uint64_t)pb.C_in * 2, (uint64_t)pb.Li[2], (uint64_t)pb.Li[1], (uint64_t)pb.Li[0],
                               (uint64_t)pb.N};
    const uint32_t cbox[5] = {tf ? 32u : 64u, (uint32_t)p.QW, (uint32_t)p.MH, 1u, 1u};
    const uint64_t bdims[2] = {(uint64_t)pb.C_in, (uint64_t)pl.wq.nblk * pb.C_out};
    const uint64_t bstr[1] = {(uint64_t)pb.C_in * 4};
    if (!encode_tiled(&tmXc, tf ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, xc,
                      cdims, astr, cbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    for (int len = 1; len <= 4; ++len) {
        // lengths beyond the longest run keep a valid map of the longest box
        const int l = len <= pl.maxlen ? len : pl.maxlen;
        const uint32_t bbox[2] = {32u, (uint32_t)(l * pb.C_out)};
        if (!encode_tiled(&tmW[len - 1], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, wp, bdims, bstr, bbox,
                          CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }

    // add and y viewed as (W, H, D, N*C_out); a box is one chunk: the whole W
    // extent, the unit's 2 MH rows, one D plane, 16 channels
    CUtensorMap tmAdd, tmY;
    const uint64_t ydims[4] = {(uint64_t)pb.Lo[2], (uint64_t)pb.Lo[1], (uint64_t)pb.Lo[0],
                               (uint64_t)pb.N * pb.C_out};
    const uint64_t ystr[3] = {(uint64_t)pb.Lo[2] * 4, (uint64_t)pb.Lo[2] * pb.Lo[1] * 4,
                              (uint64_t)pb.out_sp() * 4};
    const uint32_t ybox[4] = {(uint32_t)pb.Lo[2], (uint32_t)(2 * p.MH), 1u, 16u};
    if (pb.cl) {
        // channels last: (C_out, W, H, D, N), a box of 16 channels x the whole W
        // extent x the unit's 2 MH rows, 64-byte rows in the 64-byte swizzle
        const uint64_t cdims[5] = {(uint64_t)pb.C_out, (uint64_t)pb.Lo[2], (uint64_t)pb.Lo[1], (uint64_t)pb.Lo[0],
                                   (uint64_t)pb.N};
        const uint64_t cstr[4] = {(uint64_t)pb.C_out * 4, (uint64_t)pb.C_out * pb.Lo[2] * 4,
                                  (uint64_t)pb.C_out * pb.Lo[2] * pb.Lo[1] * 4, (uint64_t)pb.C_out * pb.out_sp() * 4};
        const uint32_t cbox5[5] = {16u, (uint32_t)pb.Lo[2], (uint32_t)(2 * p.MH), 1u, 1u};
        if (!encode_tiled(&tmY, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, a.y, cdims, cstr, cbox5,
                          CU_TENSOR_MAP_SWIZZLE_64B) ||
            !encode_tiled(&tmAdd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, a.add ? a.add : a.y, cdims, cstr, cbox5,
                          CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    } else if (!encode_tiled(&tmY, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.y, ydims, ystr, ybox,
                             CU_TENSOR_MAP_SWIZZLE_NONE) ||
               !encode_tiled(&tmAdd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.add ? a.add : a.y, ydims, ystr, ybox,
                             CU_TENSOR_MAP_SWIZZLE_NONE)) {
        return cudaErrorInvalidValue;
    }

    const void *fn;
#define CT_TC3D_FN(ADD_, CL_) (tf ? (const void *)&tc3d_split_kernel<ADD_, CL_, true> \
                                  : (const void *)&tc3d_split_kernel<ADD_, CL_, false>)
    if (pb.cl)
        fn = a.add ? CT_TC3D_FN(true, true) : CT_TC3D_FN(false, true);
    else
        fn = a.add ? CT_TC3D_FN(true, false) : CT_TC3D_FN(false, false);
#undef CT_TC3D_FN
    int per_sm = 0;
    e = prepare_kernel(fn, kThreads, pl.smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    unsigned int *status = device_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    int grid = sm_count();
    if (grid > p.nunits) grid = p.nunits;
    if (p.SD == 2 && grid > 1 && (grid & 1)) --grid;   // an even grid: the residue flip of unit_coord permutes units
    const dim3 gd((unsigned)grid), bd(kThreads);
#define CT_TC3D_LAUNCH(ADD_, CL_, TF_)                                                                       \
    launch_dependent(tc3d_split_kernel<ADD_, CL_, TF_>, gd, bd, pl.smem, a.stream, tmXc, tmW[0], tmW[1], tmW[2], \
                     tmW[3], tmAdd, tmY, a.bias, a.add, a.y, p, status)
    if (tf) {
        if (pb.cl) return a.add ? CT_TC3D_LAUNCH(true, true, true) : CT_TC3D_LAUNCH(false, true, true);
        return a.add ? CT_TC3D_LAUNCH(true, false, true) : CT_TC3D_LAUNCH(false, false, true);
    }
    if (pb.cl) return a.add ? CT_TC3D_LAUNCH(true, true, false) : CT_TC3D_LAUNCH(false, true, false);
    return a.add ? CT_TC3D_LAUNCH(true, false, false) : CT_TC3D_LAUNCH(false, false, false);
#undef CT_TC3D_LAUNCH
}

}  // namespace ct
