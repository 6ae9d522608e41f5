// ct_phase3d.cu -- stride-phase-decomposed FP32 ConvTranspose3d with a
// bias or bias + add + t*hardswish(t) epilogue fused into the stores.
//
// Method ([l1_p72] phase classes and per-output tap ranges; [l2_p26] fused
// epilogue): every output is o = s*q + r per dimension.  A (D, H) residue
// class (cD, cH) fixes the D and H tap lists; both W classes are computed
// together so each thread owns 4*s consecutive W outputs and stores them as
// float4 (the W tap lists and offsets are compile-time: template on s, the
// kernel extents and the W padding; D/H offsets carry a runtime base).
//
// Work split (persistent CTAs of 256 threads, 1 per SM):
//   tile = (group, block of OCT output channels, batch n, block of
//   RB_D x RB_H q-rows); a tile runs every (D,H) class in turn, so all tiles
//   cost the same.  Lanes: QWG = QW/4 lanes per q-row, each with 4
//   consecutive qw; a thread holds RT rows.  Accumulators acc[s][OCT][RT][4]
//   stay in registers for a whole class of a tile.
//   The input channels of the group are streamed in chunks of ICC: each
//   stage brings the x halo box [ICC][XD][XH][XW] into shared memory with one
//   4-D TMA load (boxes reaching outside the input read zeros) and the
//   class's weights [ICC][nD][nH][KW][OCT] with cp.async; stages are
//   double-buffered across channel chunks, classes and tiles, and every
//   mbarrier wait is bounded (a timeout sets the device status word and
//   unwinds).
//   Per (channel, D/H tap) a thread loads its x window (XWIN floats per row)
//   once and reuses it for every W tap of both W classes; weights are read
//   as broadcast float4.
#include <string.h>

#include "ct_internal.h"
#include "ct_device.cuh"
#include "ct_tma.h"

namespace ct {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Taps of one dimension with dilation 1 and stride S: class c (= k mod S)
// holds the taps k == c (mod S), i.e. c, c+S, ...; relative input offset (c - k)/S.
template <int S, int K>
struct Cls {
    __host__ __device__ static constexpr int count(int c)
    {
        int n = 0;
        for (int k = 0; k < K; ++k)
            if (k % S == c) ++n;
        return n;
    }
    __host__ __device__ static constexpr int tap(int c, int j)
    {
        int n = 0;
        for (int k = 0; k < K; ++k)
            if (k % S == c) {
                if (n == j) return k;
                ++n;
            }
        return 0;
    }
    __host__ __device__ static constexpr int rel(int c, int j) { return (c - tap(c, j)) / S; }
};

// W dimension fully at compile time (padding PW known): residue of class c,
// base offset floor((r + PW)/S), and absolute input offsets of each tap.
template <int S, int KW, int PW>
struct WDim {
    using C = Cls<S, KW>;
    __host__ __device__ static constexpr int r(int c) { return ((c - PW) % S + S) % S; }
    __host__ __device__ static constexpr int base(int c) { return (r(c) + PW - c) / S; }
    __host__ __device__ static constexpr int delta(int c, int j) { return base(c) + C::rel(c, j); }
    __host__ __device__ static constexpr int dmin()
    {
        int m = 1 << 20;
        for (int c = 0; c < S; ++c)
            for (int j = 0; j < C::count(c); ++j) m = delta(c, j) < m ? delta(c, j) : m;
        return m;
    }
    __host__ __device__ static constexpr int dmax()
    {
        int m = -(1 << 20);
        for (int c = 0; c < S; ++c)
            for (int j = 0; j < C::count(c); ++j) m = delta(c, j) > m ? delta(c, j) : m;
        return m;
    }
    __host__ __device__ static constexpr int cls_of_r(int rr) { return (rr + PW) % S; }
    static constexpr int kWin = 4 + (dmax() - dmin());   // x window of 4 consecutive qw
};

struct P3Params {
    int N, C_in, C_out, G, Cig, Cog;
    int Li0, Li1, Li2, Lo0, Lo1, Lo2;
    int QD, QH, QW;               // q extents (ceil(Lo/S)) used for tiling
    int QWG, RWI;                 // lanes per q-row, q-rows per warp layer (32/QWG)
    int RB_D, RB_H;               // q-row block of a tile
    int n_rbd, n_rbh, n_ocb, n_cls;
    int ICC, n_icc;               // input channels per stage, stages per class
    int XD, XH, XWB;              // x stage box: D, H extents and W row length
    int iw0, wshift;              // box start along W (multiple of 4) and W::dmin() - iw0
    int dlo, hlo;                 // smallest D/H input offset over all classes
    int xbytes;                   // bytes of one x stage box
    int xfl, stage;               // floats: x part (1024-B multiple), whole stage
    int ntiles;
    // D and H class tables (runtime padding): residue, base, q count, taps
    int rD[kMaxS], bD[kMaxS], QDc[kMaxS], nD[kMaxS], tD[kMaxS][kMaxTaps];
    int rH[kMaxS], bH[kMaxS], QHc[kMaxS], nH[kMaxS], tH[kMaxS][kMaxTaps];
};

__device__ __forceinline__ void cp_async4(float *dst, const float *src)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(src));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

struct Tile3 {
    int g, ocb, n, cls, rbd, rbh;
};

__device__ __forceinline__ Tile3 decode3(int tile, int cls, const P3Params &p)
{
    Tile3 d;
    int t = tile;
    d.rbh = t % p.n_rbh; t /= p.n_rbh;
    d.rbd = t % p.n_rbd; t /= p.n_rbd;
    d.n = t % p.N; t /= p.N;
    d.ocb = t % p.n_ocb; t /= p.n_ocb;
    d.g = t;
    d.cls = cls;
    return d;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far beyond any legitimate wait

// Weights of class (CD, CH) for one channel chunk: ws[ic][jd][jh][kw][oc]
// (compile-time extents, so the index decode is multiplies and shifts).
template <int S, int KD, int KH, int KW, int OCT, int CD, int CH>
__device__ __forceinline__ void load_w_cls(float *ws, const float *__restrict__ w, const Tile3 &t,
                                           int chunk, const P3Params &p)
{
    using DC = Cls<S, KD>;
    using HC = Cls<S, KH>;
    constexpr int ND = DC::count(CD), NH = HC::count(CH);
    const int ic0 = t.g * p.Cig + chunk * p.ICC;
    const int tot = p.ICC * ND * NH * KW * OCT;
    for (int e = threadIdx.x; e < tot; e += kThreads) {
        const int oc = e % OCT;
        int r = e / OCT;
        const int kw = r % KW; r /= KW;
        const int jh = r % NH; r /= NH;
        const int jd = r % ND;
        const int ic = r / ND;
        const int kd = CD + S * jd, kh = CH + S * jh;    // class c holds taps c, c+S, ...
        const int ocl = t.ocb * OCT + oc;
        cp_async4(ws + e, w + ((((int64_t)(ic0 + ic) * p.Cog + ocl) * KD + kd) * KH + kh) * KW + kw);
    }
}

// Issue stage (tile, class, chunk) into buffer `buf`: the x box by TMA
// (thread 0), the class's weights by cp.async (all threads).
template <int S, int KD, int KH, int KW, int OCT>
__device__ __forceinline__ void issue_stage(float *buf, uint64_t *bar, const CUtensorMap *tmx,
                                            const float *__restrict__ w, int tile, int cls, int chunk,
                                            const P3Params &p)
{
    const Tile3 t = decode3(tile, cls, p);
    if (threadIdx.x == 0) {
        dev::mbar_arrive_expect_tx(bar, (uint32_t)p.xbytes);
        dev::tma_load_4d(buf, tmx, bar, p.iw0, t.rbh * p.RB_H + p.hlo, t.rbd * p.RB_D + p.dlo,
                         t.n * p.C_in + t.g * p.Cig + chunk * p.ICC);
    }
    float *ws = buf + p.xfl;
    switch (cls) {
    case 0: load_w_cls<S, KD, KH, KW, OCT, 0, 0>(ws, w, t, chunk, p); break;
    case 1: load_w_cls<S, KD, KH, KW, OCT, 0, 1>(ws, w, t, chunk, p); break;
    case 2: load_w_cls<S, KD, KH, KW, OCT, 1, 0>(ws, w, t, chunk, p); break;
    default: load_w_cls<S, KD, KH, KW, OCT, 1, 1>(ws, w, t, chunk, p); break;
    }
}

// Accumulate one stage for the (compile-time) class (CD, CH).
template <int S, int KD, int KH, int KW, int PW, int OCT, int RT, int CD, int CH>
__device__ __forceinline__ void compute_stage(const float *buf, float (&acc)[S][OCT][RT][4],
                                              const int (&xrow)[RT], const P3Params &p)
{
    using W = WDim<S, KW, PW>;
    using DC = Cls<S, KD>;
    using HC = Cls<S, KH>;
    constexpr int ND = DC::count(CD), NH = HC::count(CH);
    constexpr int WIN = W::kWin;
    const float *ws = buf + p.xfl;
    const int hstride = p.XWB, dstride = p.XH * p.XWB, cstride = p.XD * p.XH * p.XWB;
    const int bd = p.bD[CD] - p.dlo, bh = p.bH[CH] - p.hlo;
#pragma unroll 1
    for (int ic = 0; ic < p.ICC; ++ic) {
        const float *xc = buf + ic * cstride;
        const float *wc = ws + ic * ND * NH * KW * OCT;
#pragma unroll 1
        for (int jd = 0; jd < ND; ++jd) {
#pragma unroll 1
            for (int jh = 0; jh < NH; ++jh) {
                // class c holds taps c + S*j, whose relative offset is -j
                const int off = (bd - jd) * dstride + (bh - jh) * hstride;
                float xv[RT][WIN];
#pragma unroll
                for (int t = 0; t < RT; ++t)
#pragma unroll
                    for (int m = 0; m < WIN; ++m) xv[t][m] = xc[xrow[t] + off + m];
                const float *wt = wc + (jd * NH + jh) * KW * OCT;
#pragma unroll
                for (int c = 0; c < S; ++c) {
#pragma unroll
                    for (int j = 0; j < W::C::count(c); ++j) {
                        const int kw = W::C::tap(c, j);
                        const int xo = W::delta(c, j) - W::dmin();
                        const float4 *w4 = reinterpret_cast<const float4 *>(wt + kw * OCT);
#pragma unroll
                        for (int u = 0; u < OCT / 4; ++u) {
                            const float4 wv = w4[u];
#pragma unroll
                            for (int t = 0; t < RT; ++t)
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const float xq = xv[t][q + xo];
                                    acc[c][4 * u + 0][t][q] = fmaf(wv.x, xq, acc[c][4 * u + 0][t][q]);
                                    acc[c][4 * u + 1][t][q] = fmaf(wv.y, xq, acc[c][4 * u + 1][t][q]);
                                    acc[c][4 * u + 2][t][q] = fmaf(wv.z, xq, acc[c][4 * u + 2][t][q]);
                                    acc[c][4 * u + 3][t][q] = fmaf(wv.w, xq, acc[c][4 * u + 3][t][q]);
                                }
                        }
                    }
                }
            }
        }
    }
}

template <int S, int KD, int KH, int KW, int PW, int OCT, int RT, bool ADD, int MB>
__global__ void __launch_bounds__(kThreads, MB)
phase3d_kernel(const __grid_constant__ CUtensorMap tmx, const float *__restrict__ w,
               const float *__restrict__ bias, const float *add, float *y, P3Params p,
               unsigned int *status)
{
    static_assert(S == 2, "the class dispatch below is written for stride 2");
    using W = WDim<S, KW, PW>;
    extern __shared__ __align__(1024) float smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[2];
    // 1024-byte aligned stage buffers (TMA destinations)
    float *smem = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = lane % p.QWG;          // qw group: qw = 4*wg .. 4*wg+3
    int rloc[RT];
#pragma unroll
    for (int t = 0; t < RT; ++t) rloc[t] = (warp * RT + t) * p.RWI + lane / p.QWG;
    int xrow[RT];   // smem offset of (row, first x column of the window) in a channel slice
#pragma unroll
    for (int t = 0; t < RT; ++t) {
        const int qd_l = rloc[t] / p.RB_H, qh_l = rloc[t] % p.RB_H;
        xrow[t] = (qd_l * p.XH + qh_l) * p.XWB + 4 * wg + p.wshift;
    }

    if ((int)blockIdx.x >= p.ntiles) return;
    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&tmx);
        dev::mbar_init(&full_bar[0], 1);
        dev::mbar_init(&full_bar[1], 1);
        dev::fence_mbar_init();
    }
    __syncthreads();
    // stage k -> (tile blockIdx.x + (k / per_tile) * gridDim.x, class, chunk)
    const int per_tile = p.n_cls * p.n_icc;
    issue_stage<S, KD, KH, KW, OCT>(smem, &full_bar[0], &tmx, w, blockIdx.x, 0, 0, p);
    cp_commit();
    int buf = 0;
    uint32_t phases = 0u;   // bit b: parity of the next completion of full_bar[b]
    bool failed = false;
    float acc[S][OCT][RT][4];

    for (int k = 0;; ++k) {
        const int tile = blockIdx.x + (k / per_tile) * gridDim.x;
        if (tile >= p.ntiles) break;
        const int cls = (k % per_tile) / p.n_icc;
        const int ch = k % p.n_icc;
        if (ch == 0) {
#pragma unroll
            for (int c = 0; c < S; ++c)
#pragma unroll
                for (int i = 0; i < OCT; ++i)
#pragma unroll
                    for (int t = 0; t < RT; ++t)
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[c][i][t][q] = 0.f;
        }
        {
            const int k1 = k + 1;
            const int nt = blockIdx.x + (k1 / per_tile) * gridDim.x;
            if (nt < p.ntiles)
                issue_stage<S, KD, KH, KW, OCT>(smem + (buf ^ 1) * p.stage, &full_bar[buf ^ 1], &tmx, w,
                                                nt, (k1 % per_tile) / p.n_icc, k1 % p.n_icc, p);
        }
        cp_commit();
        cp_wait<1>();
        const bool ok = dev::mbar_wait_bounded(&full_bar[buf], (phases >> buf) & 1u, kWaitLimitNs);
        phases ^= 1u << buf;
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
            failed = true;
            break;
        }
        const float *b = smem + buf * p.stage;
        switch (cls) {
        case 0: compute_stage<S, KD, KH, KW, PW, OCT, RT, 0, 0>(b, acc, xrow, p); break;
        case 1: compute_stage<S, KD, KH, KW, PW, OCT, RT, 0, 1>(b, acc, xrow, p); break;
        case 2: compute_stage<S, KD, KH, KW, PW, OCT, RT, 1, 0>(b, acc, xrow, p); break;
        default: compute_stage<S, KD, KH, KW, PW, OCT, RT, 1, 1>(b, acc, xrow, p); break;
        }
        __syncthreads();
        buf ^= 1;
        if (ch != p.n_icc - 1) continue;

        // epilogue of class (cD, cH): 4*S consecutive W outputs per thread
        const Tile3 td = decode3(tile, cls, p);
        const int cD = cls / S, cH = cls % S;
        const int rD = p.rD[cD], rH = p.rH[cH];
        const int oc0 = td.g * p.Cog + td.ocb * OCT;
        const int64_t sp = (int64_t)p.Lo0 * p.Lo1 * p.Lo2;
#pragma unroll
        for (int t = 0; t < RT; ++t) {
            const int qd = td.rbd * p.RB_D + rloc[t] / p.RB_H;
            const int qh = td.rbh * p.RB_H + rloc[t] % p.RB_H;
            if (qd >= p.QDc[cD] || qh >= p.QHc[cH]) continue;
            const int od = S * qd + rD, oh = S * qh + rH;
            const int64_t rowoff = ((int64_t)od * p.Lo1 + oh) * p.Lo2 + S * 4 * wg;
#pragma unroll
            for (int i = 0; i < OCT; ++i) {
                const int oc = oc0 + i;
                const int64_t off = ((int64_t)td.n * p.C_out + oc) * sp + rowoff;
                const float bv = bias ? __ldg(bias + oc) : 0.f;
                float v[4 * S];
#pragma unroll
                for (int e = 0; e < 4 * S; ++e) v[e] = acc[W::cls_of_r(e % S)][i][t][e / S] + bv;
#pragma unroll
                for (int e4 = 0; e4 < S; ++e4) {
                    float4 o = make_float4(v[4 * e4], v[4 * e4 + 1], v[4 * e4 + 2], v[4 * e4 + 3]);
                    if (ADD) {
                        const float4 a = __ldcs(reinterpret_cast<const float4 *>(add + off + 4 * e4));
                        o.x = add_hswish(o.x, a.x);
                        o.y = add_hswish(o.y, a.y);
                        o.z = add_hswish(o.z, a.z);
                        o.w = add_hswish(o.w, a.w);
                    }
                    __stcs(reinterpret_cast<float4 *>(y + off + 4 * e4), o);
                }
            }
        }
    }
    cp_wait<0>();
    if (failed && threadIdx.x == 0) {
        // let the TMA copies this CTA issued land before its shared memory is released
        dev::mbar_wait_bounded(&full_bar[0], phases & 1u, kWaitLimitNs);
        dev::mbar_wait_bounded(&full_bar[1], (phases >> 1) & 1u, kWaitLimitNs);
    }
}

// ---- host side --------------------------------------------------------------
struct Variant3 {
    int S, KD, KH, KW, PW, OCT, RT;
    int MB;                       // CTAs per SM the variant is built for (registers, shared memory)
    const void *fn_plain, *fn_add;
    int dmin_w, dmax_w;
};

template <int S, int KD, int KH, int KW, int PW, int OCT, int RT, int MB>
Variant3 V3()
{
    using W = WDim<S, KW, PW>;
    return Variant3{S, KD, KH, KW, PW, OCT, RT, MB,
                    (const void *)&phase3d_kernel<S, KD, KH, KW, PW, OCT, RT, false, MB>,
                    (const void *)&phase3d_kernel<S, KD, KH, KW, PW, OCT, RT, true, MB>,
                    W::dmin(), W::dmax()};
}

const Variant3 &variant(int i)
{
    static const Variant3 v[] = {
        V3<2, 3, 3, 3, 1, 16, 1, 1>(),   // k3 s2 p1 (the fused l2_p26 shape)
        V3<2, 3, 5, 7, 3, 8, 1, 2>(),    // k(3,5,7) s2 p(.,.,3) (the grouped l1_p72 shape): 2 CTAs per SM
    };
    return v[i];
}
constexpr int kNumVariants = 2;
constexpr int kSmemOptin = 227 * 1024;   // sm_103a opt-in limit per CTA

struct Plan3 {
    const Variant3 *v;
    P3Params p;
    size_t smem;
};

bool fill_class_tables(int L_out, int K, int S, int P, int *r, int *b, int *Q, int *n,
                       int (*taps)[kMaxTaps], int *lo, int *hi)
{
    // classes c = k mod S (dilation 1): residue r = (c - P) mod S,
    // base floor((r + P)/S), input offset base + (c - k)/S
    int mn = 1 << 30, mx = -(1 << 30);
    for (int c = 0; c < S; ++c) {
        r[c] = ((c - P) % S + S) % S;
        b[c] = (r[c] + P - c) / S;
        Q[c] = r[c] < L_out ? (L_out - r[c] + S - 1) / S : 0;
        n[c] = 0;
        for (int k = c; k < K; k += S) {
            if (n[c] >= kMaxTaps) return false;
            taps[c][n[c]++] = k;
            const int d = b[c] + (c - k) / S;
            mn = d < mn ? d : mn;
            mx = d > mx ? d : mx;
        }
        if (n[c] == 0) return false;   // empty class: leave to the generic kernel
    }
    *lo = mn;
    *hi = mx;
    return true;
}

int floor4(int v) { return v >= 0 ? (v / 4) * 4 : -((-v + 3) / 4) * 4; }

bool make_plan3(const Problem &pb, const Args *a, Plan3 *out)
{
    if (pb.nd != 3 || pb.dtype != CT_F32) return false;
    for (int d = 0; d < 3; ++d)
        if (pb.DL[d] != 1 || pb.S[d] != 2) return false;
    const Variant3 *v = nullptr;
    for (int i = 0; i < kNumVariants; ++i) {
        const Variant3 &c = variant(i);
        if (c.KD == pb.K[0] && c.KH == pb.K[1] && c.KW == pb.K[2] && c.PW == pb.P[2] &&
            pb.Cog % c.OCT == 0) {
            v = &c;
            break;
        }
    }
    if (!v) return false;
    const int S = 2;
    P3Params p;
    memset(&p, 0, sizeof(p));
    p.N = pb.N; p.C_in = pb.C_in; p.C_out = pb.C_out; p.G = pb.G; p.Cig = pb.Cig; p.Cog = pb.Cog;
    p.Li0 = pb.Li[0]; p.Li1 = pb.Li[1]; p.Li2 = pb.Li[2];
    p.Lo0 = pb.Lo[0]; p.Lo1 = pb.Lo[1]; p.Lo2 = pb.Lo[2];
    // the TMA tensor map needs 16-byte row strides of x
    if ((p.Li2 * 4) % 16 != 0) return false;
    if ((int64_t)pb.N * pb.C_in > 0x7fffffff) return false;
    // W: every thread owns 4 consecutive qw of both classes, stored as float4
    if (p.Lo2 % (4 * S) != 0) return false;
    p.QW = p.Lo2 / S;
    p.QWG = p.QW / 4;
    if (p.QWG < 1 || 32 % p.QWG != 0) return false;
    p.RWI = 32 / p.QWG;
    p.QD = (p.Lo0 + S - 1) / S;
    p.QH = (p.Lo1 + S - 1) / S;
    const int RB = kWarps * v->RT * p.RWI;
    p.RB_H = p.QH < RB ? p.QH : RB;
    while (p.RB_H > 1 && (RB % p.RB_H != 0)) --p.RB_H;
    p.RB_D = RB / p.RB_H;
    if (p.RB_D * p.RB_H != RB) return false;
    p.n_rbh = (p.QH + p.RB_H - 1) / p.RB_H;
    p.n_rbd = (p.QD + p.RB_D - 1) / p.RB_D;
    int dlo, dhi, hlo, hhi;
    if (!fill_class_tables(p.Lo0, pb.K[0], S, pb.P[0], p.rD, p.bD, p.QDc, p.nD, p.tD, &dlo, &dhi))
        return false;
    if (!fill_class_tables(p.Lo1, pb.K[1], S, pb.P[1], p.rH, p.bH, p.QHc, p.nH, p.tH, &hlo, &hhi))
        return false;
    p.dlo = dlo;
    p.hlo = hlo;
    p.XD = p.RB_D + dhi - dlo;
    p.XH = p.RB_H + hhi - hlo;
    p.iw0 = floor4(v->dmin_w);               // TMA: innermost start coordinate 16-B aligned
    p.wshift = v->dmin_w - p.iw0;
    p.XWB = ((p.QW + v->dmax_w - p.iw0) + 3) & ~3;
    if (p.XWB > 256 || p.XH > 256 || p.XD > 256) return false;
    p.n_ocb = pb.Cog / v->OCT;
    p.n_cls = S * S;
    int ndmax = 0, nhmax = 0;
    for (int c = 0; c < S; ++c) {
        ndmax = p.nD[c] > ndmax ? p.nD[c] : ndmax;
        nhmax = p.nH[c] > nhmax ? p.nH[c] : nhmax;
    }
    // largest channel chunk (dividing C_in/G, at most 256) whose two stages fit
    size_t smem = 0;
    int icc = 0;
    for (int c = pb.Cig < 256 ? pb.Cig : 256; c >= 1; --c) {
        if (pb.Cig % c) continue;
        const size_t xfl = (((size_t)c * p.XD * p.XH * p.XWB) + 255) & ~(size_t)255;  // 1 KB multiple
        const size_t wch = (size_t)c * ndmax * nhmax * v->KW * v->OCT;
        const size_t st = (xfl + wch + 255) & ~(size_t)255;
        const size_t tot = 2 * st * sizeof(float) + 1024;
        if (tot <= (size_t)(kSmemOptin / v->MB - (v->MB > 1 ? 1024 : 0))) {
            icc = c;
            p.xfl = (int)xfl;
            p.stage = (int)st;
            p.xbytes = c * p.XD * p.XH * p.XWB * 4;
            smem = tot;
            break;
        }
    }
    if (!icc) return false;
    p.ICC = icc;
    p.n_icc = pb.Cig / icc;
    const int64_t tiles = (int64_t)pb.G * p.n_ocb * pb.N * p.n_rbd * p.n_rbh;
    if (tiles > 0x7fffffff) return false;
    p.ntiles = (int)tiles;
    if (a) {
        if (((uintptr_t)a->x % 16) || ((uintptr_t)a->y % 16) || (a->add && ((uintptr_t)a->add % 16)))
            return false;
    }
    out->v = v;
    out->p = p;
    out->smem = smem;
    return true;
}

}  // namespace

bool phase3d_supported(const Problem &pb, const Args *a)
{
    Plan3 pl;
    return make_plan3(pb, a, &pl);
}

cudaError_t launch_phase3d(const Problem &pb, const Args &a)
{
    Plan3 pl;
    if (!make_plan3(pb, &a, &pl)) return cudaErrorNotSupported;
    const P3Params &p = pl.p;
    // x viewed as 4-D (W, H, D, N*C_in), fp32, no swizzle; out-of-range boxes read zeros
    CUtensorMap tmx;
    const uint64_t dims[4] = {(uint64_t)p.Li2, (uint64_t)p.Li1, (uint64_t)p.Li0,
                              (uint64_t)p.N * p.C_in};
    const uint64_t strides[3] = {(uint64_t)p.Li2 * 4, (uint64_t)p.Li2 * p.Li1 * 4,
                                 (uint64_t)p.Li2 * p.Li1 * p.Li0 * 4};
    const uint32_t box[4] = {(uint32_t)p.XWB, (uint32_t)p.XH, (uint32_t)p.XD, (uint32_t)p.ICC};
    if (!encode_tiled(&tmx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.x, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const void *fn = a.add ? pl.v->fn_add : pl.v->fn_plain;
    int per_sm = 0;
    cudaError_t e = prepare_kernel(fn, kThreads, pl.smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int grid = sm_count() * per_sm;
    if (grid > p.ntiles) grid = p.ntiles;
    unsigned int *status = device_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    const float *w = static_cast<const float *>(a.w);
    void *args[] = {(void *)&tmx, (void *)&w, (void *)&a.bias, (void *)&a.add, (void *)&a.y,
                    (void *)&pl.p, (void *)&status};
    return cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, pl.smem, a.stream);
}

}  // namespace ct
