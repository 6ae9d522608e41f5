// ct_tc3s_split.cu -- FP32 ConvTranspose (1-D, 2-D, 3-D) with strides 1 to 4
// in every dimension and any dilation, plain or with the fused add +
// t*hardswish(t) epilogue, on the tensor cores (tcgen05), with the operand
// split of ct_split.cuh (tf32x3 by default, the bf16 pair when opted into).
//
// Method ([l1_p79] "wavefronts": for stride s an output residue class r
// receives exactly the taps k with (r + p - k d) divisible by s, reading input
// q + (r + p - k d)/s, so the operator splits into s phases per dimension
// whose writes are disjoint -- no atomics; when s > (k - 1) d a residue
// receives one tap or none; [l1_p72] the same phase classes in 3-D; [l2_p26]
// the fused epilogue): output (s_D qd + rD, s_H qh + rH, s_W qw + rW) of
// channel oc is
//     bias[oc] + sum over the phase's taps (kd, kh, kw) and ic of
//                x[ic][qd + dd][qh + dh][qw + dw] * w[ic][oc][kd][kh][kw].
// A unit of work is 128 positions q (MH rows of QWp positions: a block of one
// W row range, a block of H rows, one D plane) of one residue pair (rD, rH),
// with the s_W W phases as s_W accumulators of C_out TMEM columns side by side
// (two sets alternate across units when they fit).  Every distinct input
// offset the pair's phases read is one A tile per K block of 32 channels, and
// the W phases reading it form runs of adjacent accumulators served by one
// weight panel and one MMA of N = run length x C_out; the host orders the
// accumulators so that runs are as long as possible.  A residue that receives
// no tap (s > (k - 1) d) leaves its accumulators unwritten, or a whole pair
// without MMAs: the epilogue writes the bias there.
//
// Stride 2 with kernel extents 2 to 4 and at most 128 output channels takes
// the kernel of ct_tc3d_split.cu, which keeps both H residues in one unit;
// this one serves the other strides, and larger kernels and dilations.
//
// Roles (persistent CTA, one per SM):
//   warps 0-1   TMA producers of the A ring (x_c 5-D boxes of the unit's
//               positions at the offset, zero-filled outside the input)
//   warps 2-3   TMA producers of the B ring (a run's panel is one box); each
//               ring slot has exactly one producer
//   warp 4      TMEM allocation and MMA issue
//   warps 5-20  epilogue: 16-channel chunks of a unit (16 channels x MH rows x
//               s_W QWp outputs), in two groups of 8 warps that take alternate
//               chunks, so that two are written at once; warp w reads TMEM lane
//               quarter w mod 4 for 8 channels of every W phase, adds bias (and
//               applies the fused epilogue) in the chunk buffer
//   warp 21     chunk mover: makes chunks ready two ahead (TMA load of the add
//               values, or the release of the buffer) and stores each written
//               chunk with one TMA store through the tensor map of the unit's H
//               residue (rows s_H qh + rH; rows, planes and columns past the
//               output are clipped)
// Every mbarrier wait is bounded: a timeout records CT_ERR_DEVICE_TIMEOUT in
// the status word and the roles unwind (producers wait, bounded, for their own
// TMA copies and the MMA issuer for its own MMAs before the TMEM is freed).
#include <string.h>

#include "ct_internal.h"
#include "ct_device.cuh"
#include "ct_tma.h"
#include "ct_tcgen05.cuh"
#include "ct_split.cuh"

namespace ct {
namespace {

constexpr int BM = 128;          // positions per unit (UMMA M)
constexpr int CK = 32;           // input channels per K block
constexpr int NA = 4;            // A ring slots at most (bf16x2: 4 of 16 KB; tf32x3: 2 of 32 KB)
constexpr int NB = 2;            // B ring slots
constexpr int NE = 3;            // epilogue chunk buffers
constexpr int NPA = 2;           // A producer warps (warp q loads the stages g with g mod NPA == q)
constexpr int NPB = 2;           // B producer warps
constexpr int MAXS = 4;          // largest stride of a dimension
constexpr int MAXT = 8;          // taps of one residue of one dimension at most
constexpr int MAXP = MAXS * MAXS;    // residue pairs (rD, rH)
constexpr int MAXE = 128;        // input offsets over all pairs
constexpr int MAXR = 192;        // runs over all pairs
constexpr int MAXSTEP = 768;     // MMA steps (B stages) over all pairs
constexpr int kAWarp0 = 0;
constexpr int kBWarp0 = kAWarp0 + NPA;
constexpr int kMmaWarp = kBWarp0 + NPB;
constexpr int kEpiWarp0 = kMmaWarp + 1;
constexpr int kStoreWarp = kEpiWarp0 + 16;
constexpr int kThreads = 32 * (kStoreWarp + 1);
constexpr int kEpiThreads = 32 * 16;
constexpr uint32_t kAHalf = BM * 128;   // 128 positions x one 128-byte row: 16 KB
constexpr uint64_t kWaitLimitNs = 2000000000ull;
static_assert(NB % NPB == 0 && NA % NPA == 0 && 2 % NPA == 0, "one producer per ring slot");

// One input offset of a residue pair; its runs are run[run0 .. run0 + nrun).
struct SEntry {
    int8_t dd, dh, dw, nrun;
    int16_t run0, pad;
};
// Adjacent accumulator slots p0 .. p0 + len - 1 served by one panel (hi / t
// rows from row brow, lo / l rows len x C_out rows further).  fresh: the
// run's first MMA writes its accumulators instead of adding to them.
struct SRun {
    int8_t p0, len, fresh, pad;
    int brow;
};
// One B stage of the issuer's schedule, in issue order (entries, then K
// blocks, then runs): flags bit 0 -- a new A stage starts here, bit 1 -- the
// A stage is done after this one, bit 2 -- the first MMA writes its
// accumulators; len: run length; col: first TMEM column.
struct SStep {
    uint8_t flags, len;
    uint16_t col;
};

struct SParams {
    int N, C_in, C_out;
    int SD, SH, SW;              // strides
    int Lo0, Lo1, Lo2;
    int QD;                      // D planes per residue at most: ceil(Lo0 / SD)
    int QWp, MH, n_qhb, n_qwb;   // unit: MH rows of QWp positions; blocks along H and W
    int n_kb;                    // C_in / 32
    int na;                      // A ring slots
    uint32_t aslot, bslot;       // bytes of an A / B ring slot
    uint32_t echunk;             // bytes of an epilogue chunk: 16 x MH x SW QWp floats
    int nrp;                     // residue pairs SD x SH
    int nunits;
    int nacc;                    // accumulator sets (1 or 2)
    uint32_t acc_cols;           // SW x C_out
    uint32_t tmem_cols;
    uint32_t idesc_b[5];         // instruction descriptor for N = len x C_out
    int8_t slot[MAXS];           // accumulator slot of W phase rW
    uint8_t wmask[MAXP];         // W phases of pair k that receive a tap (bit rW)
    uint8_t hrows[MAXS];         // 1 if H residue rH has output rows
    int e0[MAXP + 1];            // entries of pair k: ent[e0[k] .. e0[k + 1])
    int s0[MAXP + 1];            // steps of pair k: step[s0[k] .. s0[k + 1])
    SEntry ent[MAXE];
    SRun run[MAXR];
    SStep step[MAXSTEP];
};

struct SUnit {
    int n, qd, qhb, qwb, rp;
};
__device__ __forceinline__ SUnit s_unit(int u, const SParams &p)
{
    SUnit c;
    c.rp = u % p.nrp;
    u /= p.nrp;
    c.qwb = u % p.n_qwb;
    u /= p.n_qwb;
    c.qhb = u % p.n_qhb;
    u /= p.n_qhb;
    c.qd = u % p.QD;
    c.n = u / p.QD;
    return c;
}

// Warp-wide: 4 consecutive 32-bit TMEM columns of the warp's 32 lanes.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4])
{
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

template <bool ADD, bool TF>
__global__ void __launch_bounds__(kThreads, 1)
tc3s_split_kernel(const __grid_constant__ CUtensorMap tmXc,
                  const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW2,
                  const __grid_constant__ CUtensorMap tmW3, const __grid_constant__ CUtensorMap tmW4,
                  const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                  const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmA3,
                  const __grid_constant__ CUtensorMap tmY0, const __grid_constant__ CUtensorMap tmY1,
                  const __grid_constant__ CUtensorMap tmY2, const __grid_constant__ CUtensorMap tmY3,
                  const float *__restrict__ bias, const __grid_constant__ SParams p, unsigned int *status)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t a_full[NA], a_empty[NA], b_full[NB], b_empty[NB], acc_full[2],
        acc_empty[2], drain_bar, e_full[NE], c_full[NE];
    __shared__ uint32_t tmem_slot;
    __shared__ float s_bias[128];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = sm;                                  // na x aslot
    uint8_t *sB = sA + (size_t)p.na * p.aslot;         // NB x bslot
    uint8_t *sE = sB + (size_t)NB * p.bslot;           // NE x echunk
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&tmXc);
        dev::prefetch_tensormap(&tmW1);
        dev::prefetch_tensormap(&tmW2);
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
            dev::mbar_init(&acc_empty[a], kEpiThreads);
        }
        dev::mbar_init(&drain_bar, 1);
        for (int b = 0; b < NE; ++b) {
            dev::mbar_init(&e_full[b], 1);
            dev::mbar_init(&c_full[b], kEpiThreads / 2);   // one group of epilogue warps writes a chunk
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
        // ---------------- TMA producers: warp q of a ring takes the stages g with
        // g mod (producers) == q, so the ring slots it fills are its own
        if (lane == 0) {
            const bool isA = warp < kBWarp0;
            const int q = isA ? warp - kAWarp0 : warp - kBWarp0;
            const int np = isA ? NPA : NPB;
            const int nst = isA ? p.na : NB;
            uint64_t *fullb = isA ? a_full : b_full;
            uint64_t *emptyb = isA ? a_empty : b_empty;
            int g = 0, s = 0, last = -1;
            uint32_t round_par = 0;
            bool failed = false;
            for (int k = 0; k < nunit_cta && !failed; ++k) {
                const SUnit u = s_unit((int)blockIdx.x + k * (int)gridDim.x, p);
                const int qh0 = u.qhb * p.MH, qw0 = u.qwb * p.QWp;
                for (int e = p.e0[u.rp]; e < p.e0[u.rp + 1] && !failed; ++e) {
                    const SEntry &en = p.ent[e];
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
                                    uint8_t *dst = sA + (size_t)s * p.aslot;
                                    dev::mbar_arrive_expect_tx(&fullb[s], p.aslot);
                                    dev::tma_load_5d(dst, &tmXc, &fullb[s], kb * 64, qw0 + en.dw, qh0 + en.dh,
                                                     u.qd + en.dd, u.n);
                                    if (TF)
                                        dev::tma_load_5d(dst + kAHalf, &tmXc, &fullb[s], kb * 64 + 32, qw0 + en.dw,
                                                         qh0 + en.dh, u.qd + en.dd, u.n);
                                } else {
                                    const SRun &ru = p.run[en.run0 + j];
                                    const CUtensorMap *tm = ru.len == 1 ? &tmW1 : ru.len == 2 ? &tmW2
                                                          : ru.len == 3 ? &tmW3 : &tmW4;
                                    dev::mbar_arrive_expect_tx(&fullb[s], (uint32_t)(2 * ru.len * C_out) * 128u);
                                    dev::tma_load_2d(sB + (size_t)s * p.bslot, tm, &fullb[s], kb * CK, ru.brow);
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
            const uint32_t id1 = p.idesc_b[1], id2 = p.idesc_b[2], id3 = p.idesc_b[3], id4 = p.idesc_b[4];
            for (int k = 0; k < nunit_cta && ok; ++k) {
                const int rp = s_unit((int)blockIdx.x + k * (int)gridDim.x, p).rp;
                const int a = p.nacc == 2 ? (k & 1) : 0;
                const int use = p.nacc == 2 ? (k >> 1) : k;
                const int i0 = p.s0[rp], i1 = p.s0[rp + 1];
                SStep nxt = p.step[i0 < i1 ? i0 : 0];
                if (use > 0 && !dev::mbar_wait_bounded(&acc_empty[a], (use - 1) & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)a * p.acc_cols;
                uint64_t da = 0;
                // the pair's flat schedule; the next step's record is read while this
                // one waits and issues
                for (int i = i0; i < i1 && ok; ++i) {
                    const SStep st = nxt;
                    if (i + 1 < i1) nxt = p.step[i + 1];
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
                        // panel's l rows after its t rows)
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
                // a pair without taps issues no MMA: the commit still arrives once the
                // earlier MMAs have completed, and the epilogue writes the bias
                if (ok) tc::commit(&acc_full[a]);
            }
            tc::commit(&drain_bar);
            if (!dev::mbar_wait_bounded(&drain_bar, 0, kWaitLimitNs)) ok = false;
            if (!ok) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
        }
    } else if (warp == kStoreWarp) {
        // ---------------- chunk mover.  Buffer gc mod NE holds chunk gc (16 channels of a
        // unit); chunk gc is made ready two chunks ahead and stored by TMA once the
        // epilogue warps have written it.
        const int nchunk = C_out / 16;
        const int total = nunit_cta * nchunk;
        bool ok = true;
        auto map_of = [&](int rh, bool add) -> const CUtensorMap * {
            if (add) return rh == 0 ? &tmA0 : rh == 1 ? &tmA1 : rh == 2 ? &tmA2 : &tmA3;
            return rh == 0 ? &tmY0 : rh == 1 ? &tmY1 : rh == 2 ? &tmY2 : &tmY3;
        };
        auto ready = [&](int gc) {
            const int b = gc % NE;
            const SUnit v = s_unit((int)blockIdx.x + (gc / nchunk) * (int)gridDim.x, p);
            const int rd = v.rp / p.SH, rh = v.rp % p.SH;
            if (ADD && p.hrows[rh]) {
                dev::mbar_arrive_expect_tx(&e_full[b], p.echunk);
                dev::tma_load_4d(sE + (size_t)b * p.echunk, map_of(rh, true), &e_full[b], v.qwb * p.QWp * p.SW,
                                 v.qhb * p.MH, p.SD * v.qd + rd, v.n * C_out + (gc % nchunk) * 16);
            } else {
                dev::mbar_arrive(&e_full[b]);
            }
        };
        if (lane == 0) {
            for (int gc = 0; gc < 2 && gc < total; ++gc) ready(gc);
            for (int gc = 0; gc < total && ok; ++gc) {
                if (!dev::mbar_wait_bounded(&c_full[gc % NE], (gc / NE) & 1, kWaitLimitNs)) {
                    atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                    ok = false;
                    break;
                }
                const SUnit u = s_unit((int)blockIdx.x + (gc / nchunk) * (int)gridDim.x, p);
                const int rd = u.rp / p.SH, rh = u.rp % p.SH;
                // rows, planes and columns past the output are clipped by the store
                if (p.hrows[rh])
                    dev::tma_store_4d(map_of(rh, false), sE + (size_t)(gc % NE) * p.echunk, u.qwb * p.QWp * p.SW,
                                      u.qhb * p.MH, p.SD * u.qd + rd, u.n * C_out + (gc % nchunk) * 16);
                dev::bulk_commit();
                dev::bulk_wait_read<1>();               // chunk gc - 1's store has read its buffer
                if (gc + 2 < total) ready(gc + 2);
            }
            dev::bulk_wait_all();
            if (ADD)
                for (int r = total - 2 > 0 ? total - 2 : 0; r < total; ++r)
                    dev::mbar_wait_bounded(&e_full[r % NE], (r / NE) & 1, kWaitLimitNs);
        }
    } else {
        // ---------------- epilogue: warp w reads TMEM lane quarter w mod 4.  The
        // warps form two groups that take alternate chunks (chunk gc goes to group
        // gc mod 2), so two chunks are written at once; the two warps of a group
        // and lane quarter take 8 channels each of the chunk's 16.  A thread holds
        // position m = 32 (w mod 4) + lane: row m / QWp, q m mod QWp, whose s_W
        // outputs s_W q + rW are consecutive in the chunk's row.
        const int ew = warp & 3;
        const int e = (warp - kEpiWarp0) >> 2;          // 0 .. 3
        const int grp = e >> 1, ch = e & 1;
        const int nchunk = C_out / 16;
        const int SW = p.SW;
        const int rowlen = SW * p.QWp;                  // floats of a chunk row
        const int m = ew * 32 + lane;
        const int qh_l = m / p.QWp, qw = m % p.QWp;
        bool ok = true;
        int gc = 0;
        for (int k = 0; k < nunit_cta; ++k) {
            const int a = p.nacc == 2 ? (k & 1) : 0;
            const int use = p.nacc == 2 ? (k >> 1) : k;
            const int rp = s_unit((int)blockIdx.x + k * (int)gridDim.x, p).rp;
            const uint32_t wm = p.wmask[rp];
            // every thread waits for every unit, so that no arrival on acc_empty
            // runs a phase ahead
            if (ok && !dev::mbar_wait_bounded(&acc_full[a], use & 1, kWaitLimitNs)) {
                atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);        // warp-uniform before .sync.aligned loads
            tc::fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)a * p.acc_cols;
            // this group's chunks of the unit: gc0 + c with (gc0 + c) mod 2 == grp
            const int gc0 = gc;
            const int cfirst = (gc0 & 1) == grp ? 0 : 1;
            int clast = -1;
            for (int c = cfirst; c < nchunk; c += 2) clast = c;
            if (clast < 0) {                           // no chunk of this unit: release at once
                tc::fence_before();
                dev::mbar_arrive(&acc_empty[a]);
            }
            for (int c = cfirst; c < nchunk; c += 2) {
                const int g2 = gc0 + c;
                const int b = g2 % NE;
                const int c0 = c * 16 + ch * 8;            // this warp's first channel
                float v[MAXS][8];
#pragma unroll
                for (int rw = 0; rw < MAXS; ++rw) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[rw][i] = 0.f;
                    if (ok && rw < SW && ((wm >> rw) & 1u))   // unit-uniform: the warp loads or skips together
                        tc::tmem_ld8(tbase + (uint32_t)(p.slot[rw] * C_out + c0), v[rw]);
                }
                if (ok && !dev::mbar_wait_bounded(&e_full[b], (g2 / NE) & 1, kWaitLimitNs)) {
                    atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
                    ok = false;
                }
                ok = __all_sync(0xffffffffu, ok);
                tc::tmem_wait_ld();
                if (c == clast) {                       // this thread's last loads of the unit
                    tc::fence_before();
                    dev::mbar_arrive(&acc_empty[a]);
                }
                if (ok) {
                    float *buf = reinterpret_cast<float *>(sE + (size_t)b * p.echunk);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float bb = s_bias[c0 + i];
                        float *row = buf + ((ch * 8 + i) * p.MH + qh_l) * rowlen + SW * qw;
#pragma unroll
                        for (int rw = 0; rw < MAXS; ++rw) {
                            if (rw < SW) {
                                float t = v[rw][i] + bb;
                                if (ADD) t = add_hswish(t, row[rw]);
                                row[rw] = t;
                            }
                        }
                    }
                }
                dev::fence_proxy_async();
                dev::mbar_arrive(&c_full[b]);
            }
            gc = gc0 + nchunk;
        }
    }

    __syncwarp();
    tc::fence_before();
    __syncthreads();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, p.tmem_cols);
}

// ---- host side ------------------------------------------------------------------
struct SPlan {
    SParams p;
    WPanels wq;
    int maxlen;
    size_t x_bytes, w_bytes, smem;
};

// Entries and runs of every residue pair for one order of the W-phase
// accumulators (phase_of_slot[s] = W phase held in slot s); *cost estimates
// the MMA-issue time (per run and K block a B stage of ~150 clocks plus its
// MMAs at ~80 clocks each up to N = 128, the tensor-pipe time beyond).
struct DimTaps {
    int n[MAXS];
    int k[MAXS][MAXT], d[MAXS][MAXT];
};

bool plan_pairs(const Problem &pb, const DimTaps (&dt)[3], const int *uo, int nuo, const int *phase_of_slot,
                int maxlen, int mma_per_stage, SParams *pp, WPanels *wq, double *cost)
{
    SParams &p = *pp;
    const int SW = p.SW;
    int nblk = 0, ne = 0, nr = 0;
    double c = 0;
    for (int rp = 0; rp < p.nrp; ++rp) {
        const int rd = rp / p.SH, rh = rp % p.SH;
        p.e0[rp] = ne;
        uint32_t init = 0;
        for (int jd = 0; jd < dt[0].n[rd]; ++jd)
            for (int jh = 0; jh < dt[1].n[rh]; ++jh)
                for (int iw = 0; iw < nuo; ++iw) {
                    int tap_of[MAXS] = {-1, -1, -1, -1};
                    for (int sl = 0; sl < SW; ++sl) {
                        const int rw = phase_of_slot[sl];
                        for (int jw = 0; jw < dt[2].n[rw]; ++jw)
                            if (dt[2].d[rw][jw] == uo[iw])
                                tap_of[sl] = (dt[0].k[rd][jd] * pb.K[1] + dt[1].k[rh][jh]) * pb.K[2] + dt[2].k[rw][jw];
                    }
                    SEntry en;
                    memset(&en, 0, sizeof(en));
                    en.dd = (int8_t)dt[0].d[rd][jd];
                    en.dh = (int8_t)dt[1].d[rh][jh];
                    en.dw = (int8_t)uo[iw];
                    en.run0 = (int16_t)nr;
                    int ph = 0;
                    while (ph < SW) {
                        if (tap_of[ph] < 0) {
                            ++ph;
                            continue;
                        }
                        const bool st = (init >> ph) & 1u;
                        int len = 1;
                        while (ph + len < SW && len < maxlen && tap_of[ph + len] >= 0 &&
                               (((init >> (ph + len)) & 1u) != 0) == st)
                            ++len;
                        if (nr >= MAXR || nblk + 2 * len > kMaxBlk) return false;
                        SRun ru;
                        memset(&ru, 0, sizeof(ru));
                        ru.p0 = (int8_t)ph;
                        ru.len = (int8_t)len;
                        ru.fresh = st ? 0 : 1;
                        ru.brow = nblk * pb.C_out;
                        for (int hl = 0; hl < 2; ++hl)
                            for (int i = 0; i < len; ++i) {
                                wq->blk_tap[nblk] = (int16_t)tap_of[ph + i];
                                wq->blk_lo[nblk] = (int8_t)hl;
                                ++nblk;
                            }
                        for (int i = 0; i < len; ++i) init |= 1u << (ph + i);
                        p.run[nr++] = ru;
                        ++en.nrun;
                        const double n = (double)(len * pb.C_out);
                        c += 150.0 + mma_per_stage * (n <= 128 ? 80.0 : 80.0 * n / 128.0);
                        ph += len;
                    }
                    if (en.nrun == 0) continue;
                    if (ne >= MAXE) return false;
                    p.ent[ne++] = en;
                }
        uint8_t wm = 0;
        for (int sl = 0; sl < SW; ++sl)
            if ((init >> sl) & 1u) wm |= (uint8_t)(1u << phase_of_slot[sl]);
        p.wmask[rp] = wm;
    }
    p.e0[p.nrp] = ne;
    wq->nblk = nblk;
    *cost = c;
    return true;
}

bool make_splan(const Problem &pb, const Args *a, SPlan *out)
{
    if (pb.dtype != CT_F32 || pb.G != 1 || pb.cl) return false;
    const bool tf = !pb.split2;
    for (int d = 0; d < 3; ++d)
        if (pb.S[d] < 1 || pb.S[d] > MAXS) return false;
    if (pb.C_in % CK != 0 || pb.C_out % 16 != 0 || pb.C_out < 16 || pb.C_out > 128) return false;
    if (pb.S[2] * pb.C_out > 512) return false;
    // the epilogue stores whole 16-byte pieces of output rows by TMA; the prep
    // reads x in 16-byte pieces
    if (pb.Lo[2] % 4 != 0 || pb.in_sp() % 4 != 0) return false;
    if (a && (((uintptr_t)a->x % 16) || ((uintptr_t)a->y % 16) || (a->add && ((uintptr_t)a->add % 16))))
        return false;
    SParams p;
    memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C_in = pb.C_in; p.C_out = pb.C_out;
    p.SD = pb.S[0]; p.SH = pb.S[1]; p.SW = pb.S[2];
    p.Lo0 = pb.Lo[0]; p.Lo1 = pb.Lo[1]; p.Lo2 = pb.Lo[2];
    const int QW = (p.Lo2 + p.SW - 1) / p.SW;
    p.QWp = 1;
    while (p.QWp < QW && p.QWp < BM) p.QWp <<= 1;
    if (p.SW * p.QWp > 256) p.QWp = 256 / p.SW;        // a TMA box extent is at most 256
    // the output box's W extent in whole 16-byte pieces; a unit block's first
    // column (qwb s_W QWp, several blocks only when QWp is at its cap of 64 or
    // more) then starts on a 16-byte boundary too
    if ((p.SW * p.QWp * 4) % 16 != 0) return false;
    p.MH = BM / p.QWp;
    p.n_qwb = (QW + p.QWp - 1) / p.QWp;
    p.QD = (p.Lo0 + p.SD - 1) / p.SD;
    const int QH = (p.Lo1 + p.SH - 1) / p.SH;
    p.n_qhb = (QH + p.MH - 1) / p.MH;
    if (p.MH > 256) return false;
    p.n_kb = pb.C_in / CK;
    p.na = tf ? 2 : NA;
    p.aslot = (tf ? 2 : 1) * kAHalf;
    p.nrp = p.SD * p.SH;
    for (int rh = 0; rh < p.SH; ++rh) p.hrows[rh] = rh < p.Lo1 ? 1 : 0;
    const int64_t units = (int64_t)pb.N * p.QD * p.n_qhb * p.n_qwb * p.nrp;
    if (units > 0x7fffffff || units == 0) return false;
    p.nunits = (int)units;

    // taps and offsets of every residue of every dimension
    DimTaps dt[3];
    for (int d = 0; d < 3; ++d)
        for (int r = 0; r < pb.S[d]; ++r) {
            const int n = split_dim_taps(pb.K[d], pb.S[d], pb.P[d], pb.DL[d], r, dt[d].k[r], dt[d].d[r], MAXT);
            if (n < 0) return false;
            dt[d].n[r] = n;
            for (int j = 0; j < n; ++j)
                if (dt[d].d[r][j] < -100 || dt[d].d[r][j] > 100) return false;
        }
    // distinct W offsets over all W residues
    int uo[MAXS * MAXT], nuo = 0;
    for (int r = 0; r < p.SW; ++r)
        for (int j = 0; j < dt[2].n[r]; ++j) {
            bool seen = false;
            for (int i = 0; i < nuo; ++i) seen = seen || uo[i] == dt[2].d[r][j];
            if (!seen) uo[nuo++] = dt[2].d[r][j];
        }
    // runs: at most s_W phases, N = len x C_out <= 256, a panel of 2 x len x C_out
    // rows <= 256 (one TMA box)
    int maxlen = 128 / pb.C_out;
    if (maxlen > p.SW) maxlen = p.SW;
    static const int kPerm[24][4] = {
        {0, 1, 2, 3}, {0, 1, 3, 2}, {0, 2, 1, 3}, {0, 2, 3, 1}, {0, 3, 1, 2}, {0, 3, 2, 1},
        {1, 0, 2, 3}, {1, 0, 3, 2}, {1, 2, 0, 3}, {1, 2, 3, 0}, {1, 3, 0, 2}, {1, 3, 2, 0},
        {2, 0, 1, 3}, {2, 0, 3, 1}, {2, 1, 0, 3}, {2, 1, 3, 0}, {2, 3, 0, 1}, {2, 3, 1, 0},
        {3, 0, 1, 2}, {3, 0, 2, 1}, {3, 1, 0, 2}, {3, 1, 2, 0}, {3, 2, 0, 1}, {3, 2, 1, 0}};
    WPanels wq;
    double best = 0;
    int bi = -1;
    for (int i = 0; i < 24; ++i) {
        bool valid = true;                   // a permutation of 0 .. s_W - 1 in its first s_W places
        for (int sl = 0; sl < p.SW; ++sl) valid = valid && kPerm[i][sl] < p.SW;
        if (!valid) continue;
        WPanels wt;
        memset(&wt, 0, sizeof(wt));
        double c = 0;
        if (!plan_pairs(pb, dt, uo, nuo, kPerm[i], maxlen, tf ? 12 : 8, &p, &wt, &c)) continue;
        if (bi < 0 || c < best - 1e-9) {
            best = c;
            bi = i;
        }
    }
    if (bi < 0) return false;
    memset(&wq, 0, sizeof(wq));
    double c = 0;
    if (!plan_pairs(pb, dt, uo, nuo, kPerm[bi], maxlen, tf ? 12 : 8, &p, &wq, &c)) return false;
    for (int sl = 0; sl < p.SW; ++sl) p.slot[kPerm[bi][sl]] = (int8_t)sl;
    // the issuer's flat schedule per pair: entries, K blocks, runs
    int ns = 0;
    for (int rp = 0; rp < p.nrp; ++rp) {
        p.s0[rp] = ns;
        for (int e = p.e0[rp]; e < p.e0[rp + 1]; ++e) {
            const SEntry &en = p.ent[e];
            for (int kb = 0; kb < p.n_kb; ++kb)
                for (int j = 0; j < en.nrun; ++j) {
                    if (ns >= MAXSTEP) return false;
                    const SRun &ru = p.run[en.run0 + j];
                    SStep st;
                    st.flags = (uint8_t)((j == 0 ? 1 : 0) | (j == en.nrun - 1 ? 2 : 0) |
                                         ((ru.fresh && kb == 0) ? 4 : 0));
                    st.len = (uint8_t)ru.len;
                    st.col = (uint16_t)(ru.p0 * pb.C_out);
                    p.step[ns++] = st;
                }
        }
    }
    p.s0[p.nrp] = ns;
    wq.C_in = pb.C_in;
    wq.C_out = pb.C_out;
    wq.ntap = pb.kvol();
    wq.tf = tf ? 1 : 0;
    for (int len = 1; len <= 4; ++len)
        p.idesc_b[len] = len * pb.C_out <= 256 ? tc::idesc(tf ? 2 : 1, len * pb.C_out, BM) : 0u;
    p.acc_cols = (uint32_t)(p.SW * pb.C_out);
    p.nacc = 2 * p.acc_cols <= 512 ? 2 : 1;
    uint32_t cols = 32;
    while (cols < (uint32_t)p.nacc * p.acc_cols) cols <<= 1;
    p.tmem_cols = cols;
    p.bslot = (uint32_t)(2 * maxlen * pb.C_out) * 128u;
    p.echunk = (uint32_t)(16 * p.MH * p.SW * p.QWp) * 4u;
    const size_t smem = (size_t)p.na * p.aslot + (size_t)NB * p.bslot + (size_t)NE * p.echunk + 1024;
    if (smem > 227 * 1024 - 1024) return false;
    out->p = p;
    out->wq = wq;
    out->maxlen = maxlen;
    out->x_bytes = align256((size_t)pb.N * pb.C_in * pb.in_sp() * (tf ? 8 : 4));
    out->w_bytes = align256((size_t)(wq.nblk > 0 ? wq.nblk : 1) * pb.C_out * pb.C_in * 4);
    out->smem = smem;
    return true;
}

}  // namespace

bool tc3s_supported(const Problem &pb, const Args *a)
{
    SPlan pl;
    return make_splan(pb, a, &pl);
}

size_t tc3s_workspace_bytes(const Problem &pb)
{
    SPlan pl;
    if (!make_splan(pb, nullptr, &pl)) return 0;
    return pl.x_bytes + pl.w_bytes;
}

cudaError_t launch_tc3s(const Problem &pb, const Args &a)
{
    SPlan pl;
    if (!make_splan(pb, &a, &pl)) return cudaErrorNotSupported;
    const SParams &p = pl.p;
    const bool tf = pl.wq.tf != 0;
    uint8_t *ws = static_cast<uint8_t *>(a.ws);
    uint32_t *xc = reinterpret_cast<uint32_t *>(ws);
    float *wp = reinterpret_cast<float *>(ws + pl.x_bytes);

    // 1) one launch: x -> channels-last split, weights -> run panels
    const int64_t SP = pb.in_sp();
    const int64_t nbx = (SP + 63) / 64, nby = pb.C_in / 32;
    const int64_t nxb = nbx * nby * pb.N;
    const int64_t wtot = (int64_t)pl.wq.nblk * pb.C_out * pb.C_in;
    int nbw = (int)((wtot + 255) / 256);
    if (nbw < 1) nbw = 1;
    if (nbw > 4 * sm_count()) nbw = 4 * sm_count();
    if (nxb + nbw > 0x7fffffff) return cudaErrorInvalidConfiguration;
    prep_kernel<<<(unsigned)(nxb + nbw), 256, 0, a.stream>>>(static_cast<const float *>(a.x), xc, pb.C_in, SP,
                                                            (int)nbx, (int)nby, (int)nxb,
                                                            static_cast<const float *>(a.w), wp, pl.wq, nbw, 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // 2) tensor maps: A over x_c (2C, W, H, D, N), a box of one 128-byte row per
    // position (QWp x MH positions); B over the panels (rows of C_in words), one
    // map per run length; add and y per H residue rH: the rows s_H qh + rH of
    // the output, (W, rows of rH, D, N x C_out), a box of one chunk
    CUtensorMap tmXc, tmW[4], tmA[4], tmY[4];
    const uint64_t vb = tf ? 8 : 4;
    const uint64_t astr[4] = {(uint64_t)pb.C_in * vb, (uint64_t)pb.C_in * pb.Li[2] * vb,
                              (uint64_t)pb.C_in * pb.Li[2] * pb.Li[1] * vb,
                              (uint64_t)pb.C_in * pb.Li[2] * pb.Li[1] * pb.Li[0] * vb};
    const uint64_t cdims[5] = {(uint64_t)pb.C_in * 2, (uint64_t)pb.Li[2], (uint64_t)pb.Li[1], (uint64_t)pb.Li[0],
                               (uint64_t)pb.N};
    const uint32_t cbox[5] = {tf ? 32u : 64u, (uint32_t)p.QWp, (uint32_t)p.MH, 1u, 1u};
    if (!encode_tiled(&tmXc, tf ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, xc,
                      cdims, astr, cbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const uint64_t bdims[2] = {(uint64_t)pb.C_in, (uint64_t)(pl.wq.nblk > 0 ? pl.wq.nblk : 1) * pb.C_out};
    const uint64_t bstr[1] = {(uint64_t)pb.C_in * 4};
    for (int len = 1; len <= 4; ++len) {
        const int l = len <= pl.maxlen ? len : pl.maxlen;
        const uint32_t bbox[2] = {32u, (uint32_t)(2 * l * pb.C_out)};
        if (!encode_tiled(&tmW[len - 1], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, wp, bdims, bstr, bbox,
                          CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    const uint32_t ybox[4] = {(uint32_t)(p.SW * p.QWp), (uint32_t)p.MH, 1u, 16u};
    for (int rh = 0; rh < 4; ++rh) {
        // residues beyond s_H (and one without rows) keep a valid map of residue 0
        const int r = (rh < p.SH && p.hrows[rh]) ? rh : 0;
        const uint64_t rows = (uint64_t)((p.Lo1 - r + p.SH - 1) / p.SH);
        const uint64_t ydims[4] = {(uint64_t)p.Lo2, rows, (uint64_t)p.Lo0, (uint64_t)pb.N * pb.C_out};
        const uint64_t ystr[3] = {(uint64_t)p.SH * p.Lo2 * 4, (uint64_t)p.Lo1 * p.Lo2 * 4, (uint64_t)pb.out_sp() * 4};
        float *ybase = a.y + (size_t)r * p.Lo2;
        const float *abase = (a.add ? a.add : a.y) + (size_t)r * p.Lo2;
        if (!encode_tiled(&tmY[rh], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ybase, ydims, ystr, ybox,
                          CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_tiled(&tmA[rh], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, abase, ydims, ystr, ybox,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }

    const void *fn = a.add ? (tf ? (const void *)&tc3s_split_kernel<true, true>
                                 : (const void *)&tc3s_split_kernel<true, false>)
                           : (tf ? (const void *)&tc3s_split_kernel<false, true>
                                 : (const void *)&tc3s_split_kernel<false, false>);
    int per_sm = 0;
    e = prepare_kernel(fn, kThreads, pl.smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    unsigned int *status = device_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    // a grid coprime with the number of residue pairs, so that every CTA meets
    // every pair in turn (pairs with more taps cost more)
    int grid = sm_count();
    if (grid > p.nunits) grid = p.nunits;
    auto gcd = [](int x, int y) {
        while (y) {
            const int t = x % y;
            x = y;
            y = t;
        }
        return x;
    };
    while (grid > 1 && p.nunits > grid && gcd(grid, p.nrp) != 1) --grid;
    const dim3 gd((unsigned)grid), bd(kThreads);
#define CT_TC3S_LAUNCH(ADD_, TF_)                                                                              \
    launch_dependent(tc3s_split_kernel<ADD_, TF_>, gd, bd, pl.smem, a.stream, tmXc, tmW[0], tmW[1], tmW[2],     \
                     tmW[3], tmA[0], tmA[1], tmA[2], tmA[3], tmY[0], tmY[1], tmY[2], tmY[3], a.bias, p, status)
    if (tf) return a.add ? CT_TC3S_LAUNCH(true, true) : CT_TC3S_LAUNCH(false, true);
    return a.add ? CT_TC3S_LAUNCH(true, false) : CT_TC3S_LAUNCH(false, false);
#undef CT_TC3S_LAUNCH
}

}  // namespace ct
