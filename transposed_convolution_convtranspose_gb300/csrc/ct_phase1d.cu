// ct_phase1d.cu -- stride-phase-decomposed FP32 ConvTranspose1d.
//
// Method ([l1_p79]: odd-only support for k3 s2 p1 d2 and the gather index
// relation; [l1_p72]: phase classes with uniform tap counts):
// write every output as o = s*q + r.  The taps that reach residue r are the
// k with k*dl == (r + p) (mod s); each reads input i = q + delta_k with
//     delta_k = floor((r + p) / s) + (c - k*dl) / s,   c = (r + p) mod s.
// For a fixed class c the tap list and the relative offsets (c - k*dl)/s are
// compile-time constants (template on s, k, dl); only the base
// floor((r + p)/s) depends on the runtime padding.  Each residue class is a
// dense stride-1 correlation over q with a fixed tap list; classes with no
// tap hold the bias (or zero) and cost only stores.
//
// Work split (persistent CTAs, 256 threads = 8 warps, 1 CTA per SM):
//   tile = (n, group, oc block of OCB = OCT*WOC channels, q block of
//   QEXT = WQ*32*QT positions); warp (wo, wq) owns OCT channels and 32*QT
//   q values, lane l the q values qw0 + l + 32*t (t < QT); all non-empty
//   classes are accumulated in one pass (acc[NC][OCT][QT] in registers).
//   The x tile [C_in/G][XT] (all input channels of the group, q range plus
//   halo) is double-buffered in shared memory with cp.async (zero-filled
//   outside [0, L_in)); the next tile's copy is in flight while this one
//   computes.  Weights of the oc block are staged as [ic][k][oc] so a warp
//   reads each as a broadcast float4.
//   Epilogue: per output channel a warp assembles its contiguous run of
//   s*32*QT outputs (every residue, bias added) in a shared-memory staging
//   buffer laid out with the global address's 16-byte phase, then one lane
//   writes the aligned body with a TMA bulk copy (cp.async.bulk) and the
//   lanes store the unaligned head and tail.  Rows of y start at arbitrary
//   4-byte offsets (L_out is odd for the l1_p79 shape), so this is what
//   keeps every DRAM write a full sector.
#include <string.h>

#include "ct_internal.h"
#include "ct_device.cuh"
#include "ct_tma.h"

namespace ct {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int S, int K, int DL>
struct Taps1 {
    __host__ __device__ static constexpr int count(int c)
    {
        int n = 0;
        for (int k = 0; k < K; ++k)
            if ((k * DL) % S == c) ++n;
        return n;
    }
    __host__ __device__ static constexpr int tap(int c, int j)
    {
        int n = 0;
        for (int k = 0; k < K; ++k)
            if ((k * DL) % S == c) {
                if (n == j) return k;
                ++n;
            }
        return 0;
    }
    // relative input offset (c - k*dl)/s, exact, <= 0
    __host__ __device__ static constexpr int rel(int c, int j) { return (c - tap(c, j) * DL) / S; }
    // number of non-empty classes and the accumulator slot of class c
    __host__ __device__ static constexpr int nclasses()
    {
        int n = 0;
        for (int c = 0; c < S; ++c)
            if (count(c) > 0) ++n;
        return n;
    }
    __host__ __device__ static constexpr int slot(int c)
    {
        int n = 0;
        for (int cc = 0; cc < c; ++cc)
            if (count(cc) > 0) ++n;
        return n;
    }
};

struct P1Params {
    int N, C_in, C_out, G, Cig, Cog;
    int L_in, L_out;
    int WOC, WQ, OCB, QEXT;      // warps along oc / q; oc and q extent of a tile
    int n_ocb, n_qt;             // oc blocks per group; q tiles per row
    int XT;                      // x tile row length (floats, multiple of 4)
    int x_lo;                    // x tile start relative to q0 (multiple of 4, <= 0)
    int ntiles;
    int seg_pad;                 // floats per staging buffer (multiple of 4)
    int w_floats;                // staged weight floats (multiple of 4)
    int r_of_c[kMaxS];           // residue r of class c
    int base_of_c[kMaxS];        // floor((r + p) / s) of class c
    int vec_ok;                  // rows 16-B aligned: cp.async 16-B path
};

__device__ __forceinline__ void cp_async4(float *dst, const float *src, bool valid)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(src),
                 "r"(valid ? 4 : 0));
}
__device__ __forceinline__ void cp_async16(float *dst, const float *src, int bytes)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(src), "r"(bytes));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// TMA bulk store (shared -> global), its group bookkeeping and the proxy fence
__device__ __forceinline__ void bulk_store(float *gdst, const float *ssrc, unsigned bytes)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(ssrc);
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gdst), "r"(s),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

struct TileId {
    int n, g, ocb, qt;
};

__device__ __forceinline__ TileId decode(int t, const P1Params &p)
{
    TileId id;
    id.qt = t % p.n_qt; t /= p.n_qt;
    id.n = t % p.N; t /= p.N;
    id.ocb = t % p.n_ocb; t /= p.n_ocb;
    id.g = t;
    return id;
}

// Issue the cp.async copies of one x tile: rows ic of group g, positions
// [q0 + x_lo, q0 + x_lo + XT), zero outside [0, L_in).  Warp w copies rows
// w, w + 8, ...; lanes walk the row.
__device__ __forceinline__ void load_x_tile(float *xs, const float *__restrict__ x, const TileId &id,
                                            const P1Params &p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int start = id.qt * p.QEXT + p.x_lo;
    const float *xrow0 = x + ((int64_t)id.n * p.C_in + (int64_t)id.g * p.Cig) * p.L_in;
    if (p.vec_ok) {
        const int nv = p.XT >> 2;
        for (int ic = warp; ic < p.Cig; ic += kWarps) {
            const float *row = xrow0 + (int64_t)ic * p.L_in;
            float *dst = xs + ic * p.XT;
            for (int v = lane; v < nv; v += 32) {
                const int pos = start + 4 * v;
                int bytes = 0;
                const float *src = row;
                if (pos >= 0 && pos < p.L_in) {
                    const int rem = p.L_in - pos;
                    bytes = rem >= 4 ? 16 : 4 * rem;
                    src = row + pos;
                }
                cp_async16(dst + 4 * v, src, bytes);
            }
        }
    } else {
        for (int ic = warp; ic < p.Cig; ic += kWarps) {
            const float *row = xrow0 + (int64_t)ic * p.L_in;
            float *dst = xs + ic * p.XT;
            for (int v = lane; v < p.XT; v += 32) {
                const int pos = start + v;
                const bool ok = pos >= 0 && pos < p.L_in;
                cp_async4(dst + v, ok ? row + pos : row, ok);
            }
        }
    }
}

// Stage w[g*Cig + ic][ocb*OCB + o][k] as ws[(ic*K + k)*OCB + o].
template <int K>
__device__ __forceinline__ void load_w(float *ws, const float *__restrict__ w, int g, int ocb,
                                       const P1Params &p)
{
    const int tot = p.Cig * K * p.OCB;
    for (int e = threadIdx.x; e < tot; e += kThreads) {
        const int o = e % p.OCB;
        const int t = e / p.OCB;
        const int k = t % K;
        const int ic = t / K;
        ws[e] = __ldg(w + ((int64_t)(g * p.Cig + ic) * p.Cog + ocb * p.OCB + o) * K + k);
    }
}

template <int S, int K, int DL, int OCT, int QT>
__global__ void __launch_bounds__(kThreads, 1)
phase1d_kernel(const float *__restrict__ x, const float *__restrict__ w,
               const float *__restrict__ bias, float *__restrict__ y, P1Params p)
{
    using T = Taps1<S, K, DL>;
    constexpr int NC = T::nclasses() > 0 ? T::nclasses() : 1;
    constexpr int SEG = S * 32 * QT;                    // outputs of one warp row segment
    extern __shared__ __align__(16) float smem[];
    float *ws = smem;                                   // w_floats
    float *stg = smem + p.w_floats;                     // kWarps x 2 x seg_pad
    float *xs0 = stg + kWarps * 2 * p.seg_pad;          // 2 x Cig*XT
    const int xtile = p.Cig * p.XT;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wo = warp % p.WOC, wq = warp / p.WOC;
    const int oc_in_blk = wo * OCT;
    const int qw_in_tile = wq * 32 * QT;                // first q of this warp in the tile
    float *my_stg = stg + warp * 2 * p.seg_pad;

    int tile = blockIdx.x;
    if (tile >= p.ntiles) return;
    TileId id = decode(tile, p);
    load_x_tile(xs0, x, id, p);
    cp_commit();
    int cur_g = id.g, cur_ocb = id.ocb;
    load_w<K>(ws, w, cur_g, cur_ocb, p);
    int buf = 0;

    while (true) {
        const int next = tile + gridDim.x;
        TileId nid;
        if (next < p.ntiles) {
            nid = decode(next, p);
            load_x_tile(xs0 + (buf ^ 1) * xtile, x, nid, p);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();

        const float *xs = xs0 + buf * xtile;
        float acc[NC][OCT][QT];
#pragma unroll
        for (int s = 0; s < NC; ++s)
#pragma unroll
            for (int i = 0; i < OCT; ++i)
#pragma unroll
                for (int t = 0; t < QT; ++t) acc[s][i][t] = 0.f;

        if (T::nclasses() > 0) {
            const float *xq = xs + qw_in_tile + lane - p.x_lo;
            const float *wq4 = ws + oc_in_blk;
#pragma unroll 1
            for (int ic = 0; ic < p.Cig; ++ic) {
                const float *xr = xq + ic * p.XT;
                const float *wr = wq4 + ic * K * p.OCB;
#pragma unroll
                for (int c = 0; c < S; ++c) {
                    const int base = p.base_of_c[c];
#pragma unroll
                    for (int j = 0; j < T::count(c); ++j) {
                        float xv[QT];
#pragma unroll
                        for (int t = 0; t < QT; ++t) xv[t] = xr[base + T::rel(c, j) + 32 * t];
                        const float4 *w4 = reinterpret_cast<const float4 *>(wr + T::tap(c, j) * p.OCB);
                        const int sl = T::slot(c);
#pragma unroll
                        for (int u = 0; u < OCT / 4; ++u) {
                            const float4 wv = w4[u];
#pragma unroll
                            for (int t = 0; t < QT; ++t) {
                                acc[sl][4 * u + 0][t] = fmaf(wv.x, xv[t], acc[sl][4 * u + 0][t]);
                                acc[sl][4 * u + 1][t] = fmaf(wv.y, xv[t], acc[sl][4 * u + 1][t]);
                                acc[sl][4 * u + 2][t] = fmaf(wv.z, xv[t], acc[sl][4 * u + 2][t]);
                                acc[sl][4 * u + 3][t] = fmaf(wv.w, xv[t], acc[sl][4 * u + 3][t]);
                            }
                        }
                    }
                }
            }
        }

        // ---- epilogue: per output channel, stage the warp's run and bulk-store it
        const int q0w = id.qt * p.QEXT + qw_in_tile;
        const int o0 = S * q0w;                            // first output of the run
        const int nvalid = min(SEG, p.L_out - o0);          // may be <= 0 past the end
        const int oc_base = id.g * p.Cog + id.ocb * p.OCB + oc_in_blk;
#pragma unroll
        for (int i = 0; i < OCT; ++i) {
            float *sb = my_stg + (i & 1) * p.seg_pad;
            if (lane == 0) bulk_wait_read<1>();             // buffer (i & 1) is free again
            __syncwarp();
            const int64_t g0 = ((int64_t)id.n * p.C_out + oc_base + i) * p.L_out + o0;
            const int e = (int)(g0 & 3);
            const float bv = bias ? __ldg(bias + oc_base + i) : 0.f;
#pragma unroll
            for (int c = 0; c < S; ++c) {
                const int r = p.r_of_c[c];
                const int sl = T::count(c) > 0 ? T::slot(c) : 0;
#pragma unroll
                for (int t = 0; t < QT; ++t)
                    sb[e + S * (lane + 32 * t) + r] = (T::count(c) > 0 ? acc[sl][i][t] : 0.f) + bv;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (nvalid > 0) {
                const int head = min((4 - e) & 3, nvalid);
                const int body = ((nvalid - head) >> 2) << 2;
                const int tail = nvalid - head - body;
                if (lane == 0 && body > 0) bulk_store(y + g0 + head, sb + e + head, (unsigned)body * 4u);
                if (lane < head) y[g0 + lane] = sb[e + lane];
                if (lane < tail) y[g0 + head + body + lane] = sb[e + head + body + lane];
            }
            if (lane == 0) bulk_commit();
        }

        __syncthreads();   // every warp is done with xs[buf] and ws
        if (next >= p.ntiles) break;
        tile = next;
        id = nid;
        buf ^= 1;
        if (id.g != cur_g || id.ocb != cur_ocb) {
            cur_g = id.g;
            cur_ocb = id.ocb;
            load_w<K>(ws, w, cur_g, cur_ocb, p);
        }
    }
    cp_wait<0>();
    if (lane == 0) bulk_wait_all();
}

// ---- host side --------------------------------------------------------------
struct Variant {
    int S, K, DL, OCT, QT;
    const void *fn;
};

template <int S, int K, int DL, int OCT>
Variant V()
{
    // registers: NC * OCT * QT accumulators, about 128
    constexpr int nc = Taps1<S, K, DL>::nclasses() > 0 ? Taps1<S, K, DL>::nclasses() : 1;
    constexpr int QT = (128 / (nc * OCT)) >= 8 ? 8 : (128 / (nc * OCT)) >= 4 ? 4 : 2;
    return Variant{S, K, DL, OCT, QT, (const void *)&phase1d_kernel<S, K, DL, OCT, QT>};
}

const Variant *variants(int *n)
{
    static const Variant v[] = {
        V<2, 3, 2, 16>(), V<2, 3, 2, 8>(),   // the l1_p79 shape (k3 s2 d2)
        V<2, 3, 1, 16>(), V<2, 3, 1, 8>(),
        V<2, 4, 1, 16>(), V<2, 4, 1, 8>(),
        V<1, 3, 1, 16>(), V<1, 3, 1, 8>(),
    };
    *n = (int)(sizeof(v) / sizeof(v[0]));
    return v;
}

// The largest dynamic shared memory a CTA may opt into on sm_103a (227 KB);
// a fixed constant so that host-only queries give the same answer as launches.
constexpr int kSmemOptin = 227 * 1024;

struct Plan1 {
    const Variant *v;
    P1Params p;
    size_t smem;
};

bool make_plan(const Problem &pb, const Args *a, Plan1 *out)
{
    if (pb.nd != 1 || pb.dtype != CT_F32) return false;
    const int S = pb.S[2], K = pb.K[2], DL = pb.DL[2];
    int nvar = 0;
    const Variant *vs = variants(&nvar);
    const Variant *v = nullptr;
    for (int i = 0; i < nvar; ++i) {
        const Variant &c = vs[i];
        if (c.S == S && c.K == K && c.DL == DL && pb.Cog % c.OCT == 0) { v = &c; break; }
    }
    if (!v) return false;
    if (a && ((uintptr_t)a->y % 16)) return false;   // bulk stores need a 16-B aligned y
    P1Params p;
    memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C_in = pb.C_in; p.C_out = pb.C_out; p.G = pb.G; p.Cig = pb.Cig; p.Cog = pb.Cog;
    p.L_in = pb.Li[2]; p.L_out = pb.Lo[2];
    const int P = pb.P[2];
    const int blocks_oc = pb.Cog / v->OCT;           // OCT-channel blocks in the group
    p.WOC = 1;
    while (p.WOC * 2 <= kWarps && blocks_oc % (p.WOC * 2) == 0) p.WOC *= 2;
    p.WQ = kWarps / p.WOC;
    p.OCB = p.WOC * v->OCT;
    p.n_ocb = pb.Cog / p.OCB;
    p.QEXT = p.WQ * 32 * v->QT;
    // per class: residue and base offset; overall input offset range
    int dmin = 1 << 30, dmax = -(1 << 30);
    for (int c = 0; c < S; ++c) {
        const int r = ((c - P) % S + S) % S;
        const int base = (r + P - c) / S;     // exact: (r + p) == c (mod s)
        p.r_of_c[c] = r;
        p.base_of_c[c] = base;
        for (int k = 0; k < K; ++k) {
            if ((k * DL) % S != c) continue;
            const int d = base + (c - k * DL) / S;
            dmin = d < dmin ? d : dmin;
            dmax = d > dmax ? d : dmax;
        }
    }
    if (dmin > dmax) { dmin = 0; dmax = 0; }     // no taps at all: bias-only output
    const int qmax = (p.L_out + S - 1) / S;       // largest class size (residue 0)
    p.n_qt = (qmax + p.QEXT - 1) / p.QEXT;
    p.x_lo = dmin >= 0 ? (dmin / 4) * 4 : -(((-dmin) + 3) / 4) * 4;
    p.XT = ((p.QEXT - 1 + dmax - p.x_lo + 1) + 3) & ~3;
    const int64_t tiles = (int64_t)pb.G * p.n_ocb * pb.N * p.n_qt;
    if (tiles > 0x7fffffff) return false;
    p.ntiles = (int)tiles;
    p.seg_pad = S * 32 * v->QT + 4;               // +4: room for the 16-byte phase shift
    p.w_floats = (p.Cig * K * p.OCB + 3) & ~3;
    const size_t smem =
        ((size_t)p.w_floats + (size_t)kWarps * 2 * p.seg_pad + 2 * (size_t)p.Cig * p.XT) * sizeof(float);
    if (smem > (size_t)kSmemOptin) return false;
    p.vec_ok = (p.L_in % 4 == 0) && (!a || ((uintptr_t)a->x % 16) == 0);
    out->v = v;
    out->p = p;
    out->smem = smem;
    return true;
}

}  // namespace

bool phase1d_supported(const Problem &pb, const Args *a)
{
    Plan1 pl;
    return make_plan(pb, a, &pl);
}

cudaError_t launch_phase1d(const Problem &pb, const Args &a)
{
    Plan1 pl;
    if (!make_plan(pb, &a, &pl)) return cudaErrorNotSupported;
    int per_sm = 0;
    cudaError_t e = prepare_kernel(pl.v->fn, kThreads, pl.smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int grid = sm_count() * per_sm;
    if (grid > pl.p.ntiles) grid = pl.p.ntiles;
    const float *x = static_cast<const float *>(a.x);
    const float *w = static_cast<const float *>(a.w);
    void *args[] = {(void *)&x, (void *)&w, (void *)&a.bias, (void *)&a.y, (void *)&pl.p};
    return cudaLaunchKernel(pl.v->fn, dim3(grid), dim3(kThreads), args, pl.smem, a.stream);
}

}  // namespace ct
