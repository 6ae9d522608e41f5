// ct_gather_generic.cu -- gather ("output-stationary") transposed convolution
// for any valid problem: 1-D, 2-D or 3-D, any groups, stride, padding,
// output_padding, dilation, fp32 or bf16 inputs, optional bias, optional
// add + t*hardswish(t) epilogue, channels-first or channels-last layouts.
//
// Formulation ([l1_p79] gather check, [l1_p72] tap-range analysis): output o
// of one dimension receives tap k from input i = (o + p - k*dl) / s when that
// numerator is non-negative, divisible by s, and i < L_in.  No atomics.
//
// Work split: one thread per (n, group, block of OCV output channels, od, oh,
// qw) computes the outputs ow = s_w*qw + r for every residue r in [0, s_w),
// so a warp's threads (consecutive qw) share od and oh -- hence the same D/H
// taps -- and together cover a contiguous run of ow.  Weights and x are read
// through the read-only cache; the tuned phase kernels stage them in shared
// memory instead.  This kernel is the correctness baseline and the path for
// shapes the tuned kernels do not cover.
#include "ct_internal.h"
#include "ct_device.cuh"

namespace ct {
namespace {

struct GenParams {
    int N, C_in, C_out, G, Cig, Cog, n_occ;
    int Li0, Li1, Li2, Lo0, Lo1, Lo2;
    int K0, K1, K2, S0, S1, S2, P0, P1, P2, D0, D1, D2;
    int QW;
    // element strides of x and y (and add): image, channel, position.  Channels
    // first (N, C, spatial): C*sp, sp, 1; channels last (N, spatial, C): sp*C, 1, C
    int64_t xs_n, xs_c, xs_p, ys_n, ys_c, ys_p;
};

template <typename TIN, int OCV, bool ADD>
__global__ void __launch_bounds__(256)
gather_generic_kernel(const TIN *__restrict__ x, const TIN *__restrict__ w,
                      const float *__restrict__ bias, const float *add,
                      float *y, GenParams g)
{
    const int64_t total = (int64_t)g.N * g.G * g.n_occ * g.Lo0 * g.Lo1 * g.QW;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    int64_t t = idx;
    const int qw = (int)(t % g.QW); t /= g.QW;
    const int oh = (int)(t % g.Lo1); t /= g.Lo1;
    const int od = (int)(t % g.Lo0); t /= g.Lo0;
    const int occ = (int)(t % g.n_occ); t /= g.n_occ;
    const int grp = (int)(t % g.G);
    const int n = (int)(t / g.G);

    const int ocl0 = occ * OCV;
    const int jmax = min(OCV, g.Cog - ocl0);
    const int kvol = g.K0 * g.K1 * g.K2;
    const TIN *xg = x + (int64_t)n * g.xs_n + (int64_t)grp * g.Cig * g.xs_c;
    const TIN *wg = w + ((int64_t)grp * g.Cig * g.Cog + ocl0) * kvol;

    for (int r = 0; r < g.S2; ++r) {
        const int ow = qw * g.S2 + r;
        if (ow >= g.Lo2) break;
        float acc[OCV];
#pragma unroll
        for (int j = 0; j < OCV; ++j) acc[j] = 0.f;

        for (int kd = 0; kd < g.K0; ++kd) {
            const int nd_ = od + g.P0 - kd * g.D0;
            if (nd_ < 0 || nd_ % g.S0) continue;
            const int id = nd_ / g.S0;
            if (id >= g.Li0) continue;
            for (int kh = 0; kh < g.K1; ++kh) {
                const int nh = oh + g.P1 - kh * g.D1;
                if (nh < 0 || nh % g.S1) continue;
                const int ih = nh / g.S1;
                if (ih >= g.Li1) continue;
                for (int kw = 0; kw < g.K2; ++kw) {
                    const int nw = ow + g.P2 - kw * g.D2;
                    if (nw < 0 || nw % g.S2) continue;
                    const int iw = nw / g.S2;
                    if (iw >= g.Li2) continue;
                    const int tap = (kd * g.K1 + kh) * g.K2 + kw;
                    const TIN *xp = xg + (((int64_t)id * g.Li1 + ih) * g.Li2 + iw) * g.xs_p;
                    const TIN *wp = wg + tap;
                    for (int ic = 0; ic < g.Cig; ++ic) {
                        const float xv = to_float(ldg(xp + (int64_t)ic * g.xs_c));
                        const TIN *wr = wp + (int64_t)ic * g.Cog * kvol;
#pragma unroll
                        for (int j = 0; j < OCV; ++j)
                            if (j < jmax) acc[j] = fmaf(xv, to_float(ldg(wr + j * kvol)), acc[j]);
                    }
                }
            }
        }
        const int64_t sp = ((int64_t)od * g.Lo1 + oh) * g.Lo2 + ow;
#pragma unroll
        for (int j = 0; j < OCV; ++j) {
            if (j < jmax) {
                const int oc = grp * g.Cog + ocl0 + j;
                const int64_t off = (int64_t)n * g.ys_n + (int64_t)oc * g.ys_c + sp * g.ys_p;
                float v = acc[j] + (bias ? __ldg(bias + oc) : 0.f);
                if (ADD) v = add_hswish(v, add[off]);
                y[off] = v;
            }
        }
    }
}

template <typename TIN, int OCV>
cudaError_t launch_t(const Problem &pb, const Args &a)
{
    GenParams g;
    g.N = pb.N; g.C_in = pb.C_in; g.C_out = pb.C_out; g.G = pb.G; g.Cig = pb.Cig; g.Cog = pb.Cog;
    g.n_occ = (pb.Cog + OCV - 1) / OCV;
    g.Li0 = pb.Li[0]; g.Li1 = pb.Li[1]; g.Li2 = pb.Li[2];
    g.Lo0 = pb.Lo[0]; g.Lo1 = pb.Lo[1]; g.Lo2 = pb.Lo[2];
    g.K0 = pb.K[0]; g.K1 = pb.K[1]; g.K2 = pb.K[2];
    g.S0 = pb.S[0]; g.S1 = pb.S[1]; g.S2 = pb.S[2];
    g.P0 = pb.P[0]; g.P1 = pb.P[1]; g.P2 = pb.P[2];
    g.D0 = pb.DL[0]; g.D1 = pb.DL[1]; g.D2 = pb.DL[2];
    g.QW = (pb.Lo[2] + pb.S[2] - 1) / pb.S[2];
    const int64_t in_sp = pb.in_sp(), out_sp = pb.out_sp();
    g.xs_n = (int64_t)pb.C_in * in_sp;
    g.ys_n = (int64_t)pb.C_out * out_sp;
    g.xs_c = pb.cl ? 1 : in_sp;
    g.xs_p = pb.cl ? pb.C_in : 1;
    g.ys_c = pb.cl ? 1 : out_sp;
    g.ys_p = pb.cl ? pb.C_out : 1;
    const int64_t total = (int64_t)g.N * g.G * g.n_occ * g.Lo0 * g.Lo1 * g.QW;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const TIN *x = static_cast<const TIN *>(a.x);
    const TIN *w = static_cast<const TIN *>(a.w);
    if (a.add)
        gather_generic_kernel<TIN, OCV, true><<<(unsigned)blocks, threads, 0, a.stream>>>(
            x, w, a.bias, a.add, a.y, g);
    else
        gather_generic_kernel<TIN, OCV, false><<<(unsigned)blocks, threads, 0, a.stream>>>(
            x, w, a.bias, nullptr, a.y, g);
    return cudaGetLastError();
}

template <typename TIN>
cudaError_t launch_dtype(const Problem &pb, const Args &a)
{
    if (pb.Cog >= 8) return launch_t<TIN, 8>(pb, a);
    if (pb.Cog >= 4) return launch_t<TIN, 4>(pb, a);
    return launch_t<TIN, 1>(pb, a);
}

}  // namespace

cudaError_t launch_gather_generic(const Problem &pb, const Args &a)
{
    if (pb.dtype == CT_BF16) return launch_dtype<bf16_t>(pb, a);
    return launch_dtype<float>(pb, a);
}

}  // namespace ct
