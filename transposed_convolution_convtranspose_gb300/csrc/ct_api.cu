// ct_api.cu -- the C ABI of libct.so: argument validation, output shapes,
// stride-phase tables, kernel selection and launch.  Declarations and the
// contract of every entry point are in include/ct.h.
#include <string.h>

#include <atomic>
#include <mutex>

#include "ct_internal.h"
#include "ct_introspect.h"

namespace ct {

namespace {
// The status word (element 0: CT_OK or CT_ERR_DEVICE_TIMEOUT) lives in static
// host memory that is page-locked and mapped into the devices' address space
// (cudaHostRegister, on first use): a kernel whose bounded wait runs out
// writes the timeout there, and the host reads it without synchronising --
// every forward call checks it before launching, ct_last_device_error after
// synchronising.  A whole 64 KB page of its own, so that registering it pins
// nothing else of the library on hosts with pages of up to 64 KB.
alignas(65536) unsigned int g_status_page[65536 / sizeof(unsigned int)];
std::mutex g_status_mu;
}  // namespace

unsigned int *device_status_ptr()
{
    // Looked up on every launch, under a lock: the registration and the device
    // address belong to the current context, which a cudaDeviceReset (or a
    // caller's own context) replaces; a page found unregistered is registered
    // again.
    std::lock_guard<std::mutex> lk(g_status_mu);
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, g_status_page);
    if (e != cudaSuccess || at.type == cudaMemoryTypeUnregistered || !at.devicePointer) {
        (void)cudaGetLastError();
        e = cudaHostRegister(g_status_page, sizeof(g_status_page), cudaHostRegisterMapped | cudaHostRegisterPortable);
        if (e != cudaSuccess && e != cudaErrorHostMemoryAlreadyRegistered) {
            (void)cudaGetLastError();
            return nullptr;
        }
        (void)cudaGetLastError();
        if (cudaPointerGetAttributes(&at, g_status_page) != cudaSuccess || !at.devicePointer) {
            (void)cudaGetLastError();
            return nullptr;
        }
    }
    return static_cast<unsigned int *>(at.devicePointer);
}

// Take (read and clear) a timeout recorded by an earlier launch.
ct_status take_device_status()
{
    const unsigned int v = __atomic_exchange_n(&g_status_page[0], 0u, __ATOMIC_ACQ_REL);
    return v != 0 ? CT_ERR_DEVICE_TIMEOUT : CT_OK;
}

// Output length of one dimension ([l1_p79] output-length formula).
static int64_t out_len(int64_t L_in, int64_t k, int64_t s, int64_t p, int64_t op, int64_t dl)
{
    return (L_in - 1) * s - 2 * p + dl * (k - 1) + op + 1;
}

bool build_phase_dim(int L_out, int K, int S, int P, int DL, PhaseDim *pd)
{
    if (S < 1 || S > kMaxS) return false;
    memset(pd, 0, sizeof(*pd));
    pd->S = S;
    for (int r = 0; r < S; ++r) {
        pd->Q[r] = (r < L_out) ? (L_out - r + S - 1) / S : 0;
        for (int k = 0; k < K; ++k) {
            const int num = r + P - k * DL;
            // floor-exact divisibility test, also for negative numerators
            const int rem = ((num % S) + S) % S;
            if (rem != 0) continue;
            if (pd->ntap[r] >= kMaxTaps) return false;
            pd->k[r][pd->ntap[r]] = k;
            pd->delta[r][pd->ntap[r]] = (num - rem) / S;
            ++pd->ntap[r];
        }
    }
    return true;
}

static std::atomic<int> g_override{0};
static std::atomic<int> g_deterministic{0};

bool deterministic() { return g_deterministic.load() != 0; }

}  // namespace ct

using namespace ct;

namespace {

constexpr int64_t kMaxDim = 1 << 30;

ct_status make_problem(int nd, int N, int C_in, int C_out, const int *Li, const int *K, int G,
                       const int *S, const int *P, const int *OP, const int *DL, ct_dtype dtype,
                       bool has_bias, bool has_add, Problem *pb)
{
    if (nd < 1 || nd > 3) return CT_ERR_ARG;
    if (dtype != CT_F32 && dtype != CT_BF16 && dtype != CT_F32_BF16X2) return CT_ERR_ARG;
    // CT_F32_BF16X2 stores x and w as fp32 like CT_F32; only the split the FP32
    // tensor-core kernels use differs
    const bool split2 = dtype == CT_F32_BF16X2;
    if (split2) dtype = CT_F32;
    if (N < 0 || C_in < 1 || C_out < 1 || G < 1) return CT_ERR_ARG;
    if (C_in % G || C_out % G) return CT_ERR_SHAPE;
    Problem p;
    p.nd = nd; p.N = N; p.C_in = C_in; p.C_out = C_out; p.G = G;
    p.Cig = C_in / G; p.Cog = C_out / G;
    p.dtype = dtype; p.split2 = split2; p.has_bias = has_bias; p.has_add = has_add;
    for (int d = 0; d < 3; ++d) {
        p.Li[d] = 1; p.K[d] = 1; p.S[d] = 1; p.P[d] = 0; p.OP[d] = 0; p.DL[d] = 1; p.Lo[d] = 1;
    }
    for (int d = 0; d < nd; ++d) {
        const int e = 3 - nd + d;
        if (Li[d] < 1 || K[d] < 1 || S[d] < 1 || DL[d] < 1) return CT_ERR_SHAPE;
        if (P[d] < 0 || OP[d] < 0) return CT_ERR_SHAPE;
        if (OP[d] >= (S[d] > DL[d] ? S[d] : DL[d])) return CT_ERR_SHAPE;
        const int64_t lo = out_len(Li[d], K[d], S[d], P[d], OP[d], DL[d]);
        if (lo < 1) return CT_ERR_SHAPE;
        if (lo > kMaxDim || Li[d] > kMaxDim) return CT_ERR_UNSUPPORTED;
        p.Li[e] = Li[d]; p.K[e] = K[d]; p.S[e] = S[d]; p.P[e] = P[d]; p.OP[e] = OP[d];
        p.DL[e] = DL[d]; p.Lo[e] = (int)lo;
    }
    // element counts must fit int64 comfortably
    const double ye = (double)N * C_out * (double)p.Lo[0] * p.Lo[1] * p.Lo[2];
    const double xe = (double)N * C_in * (double)p.Li[0] * p.Li[1] * p.Li[2];
    if (ye > 4e18 || xe > 4e18) return CT_ERR_UNSUPPORTED;
    *pb = p;
    return CT_OK;
}

enum class Path { Generic, Phase1d, Phase3d, Umma, Tc1d, Tc3d, Tc3dg, Tc3s };

Path choose_path(const Problem &pb, const Args *a)
{
    const int ov = g_override.load();
    if (ov == 1) return Path::Generic;
    if (pb.cl) {
        // channels-last layouts: the bf16 tensor-core kernel reads x in place and
        // writes y channels-last; the dense FP32 one splits x without a transpose
        // and stores y channels-last; every other shape takes the generic kernel
        if (pb.dtype == CT_BF16 && pb.nd >= 2 && !pb.has_add && umma_supported(pb, a)) return Path::Umma;
        if (pb.dtype == CT_F32 && ov != 2 && pb.nd >= 2 && tc3d_supported(pb, a) &&
            (!a || (a->ws && ((uintptr_t)a->ws % 256) == 0 && a->ws_bytes >= tc3d_workspace_bytes(pb))))
            return Path::Tc3d;
        return Path::Generic;
    }
    // the FP32 tensor-core paths with scratch need the caller's workspace: a call
    // without it takes the kernels that need none (a query without arguments,
    // a == NULL, reports the tensor-core path and its workspace size)
    auto has_ws = [&](size_t need) {
        return !a || (a->ws && ((uintptr_t)a->ws % 256) == 0 && a->ws_bytes >= need);
    };
    if (pb.dtype == CT_F32) {
        if (ov != 2 && pb.nd == 1 && tc1d_supported(pb, a)) return Path::Tc1d;
        if (ov != 2 && pb.nd == 1 && tc3s_supported(pb, a) && has_ws(tc3s_workspace_bytes(pb))) return Path::Tc3s;
        if (pb.nd == 1 && phase1d_supported(pb, a)) return Path::Phase1d;
        // the 3-D tensor-core path works in the caller's workspace: a call without
        // enough of it takes the FFMA kernel (a query without arguments, a == NULL,
        // reports the tensor-core path and its workspace size)
        // a 2-D problem is a 3-D one with a unit D dimension (same layouts)
        if (ov != 2 && pb.nd >= 2 && tc3d_supported(pb, a) &&
            (!a || (a->ws && ((uintptr_t)a->ws % 256) == 0 && a->ws_bytes >= tc3d_workspace_bytes(pb))))
            return Path::Tc3d;
        if (ov != 2 && pb.nd >= 2 && tc3dg_supported(pb, a) &&
            (!a || (a->ws && ((uintptr_t)a->ws % 256) == 0 && a->ws_bytes >= tc3dg_workspace_bytes(pb))))
            return Path::Tc3dg;
        // strides 1 to 4, any dilation, groups 1
        if (ov != 2 && pb.nd >= 2 && tc3s_supported(pb, a) && has_ws(tc3s_workspace_bytes(pb))) return Path::Tc3s;
        if (pb.nd >= 2 && phase3d_supported(pb, a)) return Path::Phase3d;
    } else {
        if (pb.nd >= 2 && umma_supported(pb, a)) return Path::Umma;
    }
    return Path::Generic;
}

const char *path_name(Path p, const Problem &pb)
{
    switch (p) {
    case Path::Generic: return "gather_generic";
    case Path::Phase1d: return "phase1d_f32";
    case Path::Phase3d: return "phase3d_f32";
    case Path::Umma: return "umma_bf16";
    case Path::Tc1d: return "tc1d_tf32x3";
    case Path::Tc3d: return pb.split2 ? "tc3d_bf16x2" : "tc3d_tf32x3";
    case Path::Tc3dg: return pb.split2 ? "tc3dg_bf16x2" : "tc3dg_tf32x3";
    case Path::Tc3s: return pb.split2 ? "tc3s_bf16x2" : "tc3s_tf32x3";
    }
    return "gather_generic";
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Scratch bytes of the path a call with these arguments takes when given it.
size_t workspace_bytes(const Problem &pb)
{
    switch (choose_path(pb, nullptr)) {
    case Path::Umma: return umma_workspace_bytes(pb);
    case Path::Tc3d: return tc3d_workspace_bytes(pb);
    case Path::Tc3dg: return tc3dg_workspace_bytes(pb);
    case Path::Tc3s: return tc3s_workspace_bytes(pb);
    default: return 0;
    }
}

bool overlaps(const void *a, size_t an, const void *b, size_t bn)
{
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + bn && b0 < a0 + an;
}

ct_status run(const Problem &pb, Args a)
{
    const size_t esz = pb.dtype == CT_BF16 ? 2 : 4;
    if (pb.N == 0) return CT_OK;   // empty batch: nothing to compute, x/y may be NULL
    if (!a.x || !a.w || !a.y) return CT_ERR_ARG;
    if (pb.has_add && !a.add) return CT_ERR_ARG;
    if (!aligned(a.x, esz) || !aligned(a.w, esz) || !aligned(a.y, 4) ||
        (a.bias && !aligned(a.bias, 4)) || (a.add && !aligned(a.add, 4)))
        return CT_ERR_ALIGN;
    const size_t yb = (size_t)pb.y_elems() * 4;
    const size_t xb = (size_t)pb.x_elems() * esz;
    const size_t wb = (size_t)pb.C_in * pb.Cog * pb.kvol() * esz;
    if (overlaps(a.y, yb, a.x, xb) || overlaps(a.y, yb, a.w, wb) ||
        (a.bias && overlaps(a.y, yb, a.bias, (size_t)pb.C_out * 4)))
        return CT_ERR_ARG;
    if (a.add && a.add != a.y && overlaps(a.y, yb, a.add, yb)) return CT_ERR_ARG;

    // A workspace is either absent (NULL or 0 bytes: then the kernels that need
    // none run) or at least as large as ct_workspace_size_* reports for these
    // arguments, and 256-byte aligned; anything in between is an error rather
    // than a silent change of kernel.
    if (!a.ws && a.ws_bytes != 0) return CT_ERR_WORKSPACE;
    if (a.ws_bytes == 0) a.ws = nullptr;
    if (a.ws && (!aligned(a.ws, 256) || a.ws_bytes < workspace_bytes(pb))) return CT_ERR_WORKSPACE;
    const Path path = choose_path(pb, &a);
    if (path == Path::Umma) {
        const size_t need = umma_workspace_bytes(pb);
        if (a.ws_bytes < need || !a.ws || !aligned(a.ws, 256)) return CT_ERR_WORKSPACE;
    }
    // a bounded wait of an earlier launch that ran out is reported here, before
    // this call launches anything
    const ct_status pending = take_device_status();
    if (pending != CT_OK) return pending;
    cudaError_t e = cudaSuccess;
    switch (path) {
    case Path::Generic: e = launch_gather_generic(pb, a); break;
    case Path::Phase1d: e = launch_phase1d(pb, a); break;
    case Path::Phase3d: e = launch_phase3d(pb, a); break;
    case Path::Umma: e = launch_umma(pb, a); break;
    case Path::Tc1d: e = launch_tc1d(pb, a); break;
    case Path::Tc3d: e = launch_tc3d(pb, a); break;
    case Path::Tc3dg: e = launch_tc3dg(pb, a); break;
    case Path::Tc3s: e = launch_tc3s(pb, a); break;
    }
    if (e == cudaSuccess) return CT_OK;
    // the failure is reported as CT_ERR_CUDA; clear the runtime's last-error slot
    // so that the caller's next error check does not take it for its own
    (void)cudaGetLastError();
    return CT_ERR_CUDA;
}

}  // namespace

// Internal access for other translation units (declared in ct_internal.h).
namespace ct {
ct_status make_problem_3d(int N, int C_in, int C_out, const int *in_dhw, const int *k_dhw, int groups,
                          const int *stride, const int *padding, const int *output_padding,
                          const int *dilation, ct_dtype dtype, bool has_bias, Problem *pb)
{
    return make_problem(3, N, C_in, C_out, in_dhw, k_dhw, groups, stride, padding, output_padding,
                        dilation, dtype, has_bias, false, pb);
}
bool takes_umma_path(const Problem &pb, const Args *a) { return choose_path(pb, a) == Path::Umma; }
ct_status run_problem(const Problem &pb, const Args &a) { return run(pb, a); }
}  // namespace ct

extern "C" {

int64_t ct_out_len(int64_t L_in, int k, int s, int p, int op, int dl)
{
    if (L_in < 1 || k < 1 || s < 1 || dl < 1 || p < 0 || op < 0) return -1;
    const int64_t lo = out_len(L_in, k, s, p, op, dl);
    return lo >= 1 ? lo : -1;
}

ct_status ct_workspace_size_1d(int N, int C_in, int C_out, int L_in, int k, int groups,
                               int stride, int padding, int output_padding, int dilation,
                               ct_dtype dtype, size_t *bytes)
{
    if (!bytes) return CT_ERR_ARG;
    Problem pb;
    ct_status st = make_problem(1, N, C_in, C_out, &L_in, &k, groups, &stride, &padding,
                                &output_padding, &dilation, dtype, false, false, &pb);
    if (st != CT_OK) return st;
    *bytes = workspace_bytes(pb);
    return CT_OK;
}

ct_status ct_workspace_size_3d(int N, int C_in, int C_out, const int in_dhw[3],
                               const int k_dhw[3], int groups, const int stride[3],
                               const int padding[3], const int output_padding[3],
                               const int dilation[3], ct_dtype dtype, size_t *bytes)
{
    if (!bytes || !in_dhw || !k_dhw || !stride || !padding || !output_padding || !dilation)
        return CT_ERR_ARG;
    Problem pb;
    ct_status st = make_problem(3, N, C_in, C_out, in_dhw, k_dhw, groups, stride, padding,
                                output_padding, dilation, dtype, false, false, &pb);
    if (st != CT_OK) return st;
    *bytes = workspace_bytes(pb);
    return CT_OK;
}

ct_status ct_workspace_size_2d(int N, int C_in, int C_out, const int in_hw[2], const int k_hw[2],
                               int groups, const int stride[2], const int padding[2],
                               const int output_padding[2], const int dilation[2], ct_dtype dtype,
                               size_t *bytes)
{
    if (!bytes || !in_hw || !k_hw || !stride || !padding || !output_padding || !dilation)
        return CT_ERR_ARG;
    Problem pb;
    ct_status st = make_problem(2, N, C_in, C_out, in_hw, k_hw, groups, stride, padding,
                                output_padding, dilation, dtype, false, false, &pb);
    if (st != CT_OK) return st;
    *bytes = workspace_bytes(pb);
    return CT_OK;
}

ct_status ct_forward_1d(const void *x, const void *w, const float *bias, float *y,
                        int N, int C_in, int C_out, int L_in, int k, int groups,
                        int stride, int padding, int output_padding, int dilation,
                        ct_dtype dtype, void *workspace, size_t ws_bytes, void *stream)
{
    Problem pb;
    ct_status st = make_problem(1, N, C_in, C_out, &L_in, &k, groups, &stride, &padding,
                                &output_padding, &dilation, dtype, bias != nullptr, false, &pb);
    if (st != CT_OK) return st;
    Args a{x, w, bias, nullptr, y, workspace, ws_bytes, (cudaStream_t)stream};
    return run(pb, a);
}

ct_status ct_forward_3d(const void *x, const void *w, const float *bias, float *y,
                        int N, int C_in, int C_out, const int in_dhw[3], const int k_dhw[3],
                        int groups, const int stride[3], const int padding[3],
                        const int output_padding[3], const int dilation[3],
                        ct_dtype dtype, void *workspace, size_t ws_bytes, void *stream)
{
    if (!in_dhw || !k_dhw || !stride || !padding || !output_padding || !dilation)
        return CT_ERR_ARG;
    Problem pb;
    ct_status st = make_problem(3, N, C_in, C_out, in_dhw, k_dhw, groups, stride, padding,
                                output_padding, dilation, dtype, bias != nullptr, false, &pb);
    if (st != CT_OK) return st;
    Args a{x, w, bias, nullptr, y, workspace, ws_bytes, (cudaStream_t)stream};
    return run(pb, a);
}

ct_status ct_forward_3d_add_hswish(const void *x, const void *w, const float *bias,
                                   const float *add, float *y,
                                   int N, int C_in, int C_out, const int in_dhw[3],
                                   const int k_dhw[3], int groups, const int stride[3],
                                   const int padding[3], const int output_padding[3],
                                   const int dilation[3], ct_dtype dtype,
                                   void *workspace, size_t ws_bytes, void *stream)
{
    if (!in_dhw || !k_dhw || !stride || !padding || !output_padding || !dilation)
        return CT_ERR_ARG;
    if (!add) return CT_ERR_ARG;
    Problem pb;
    ct_status st = make_problem(3, N, C_in, C_out, in_dhw, k_dhw, groups, stride, padding,
                                output_padding, dilation, dtype, bias != nullptr, true, &pb);
    if (st != CT_OK) return st;
    Args a{x, w, bias, add, y, workspace, ws_bytes, (cudaStream_t)stream};
    return run(pb, a);
}

ct_status ct_forward_2d(const void *x, const void *w, const float *bias, float *y,
                        int N, int C_in, int C_out, const int in_hw[2], const int k_hw[2],
                        int groups, const int stride[2], const int padding[2],
                        const int output_padding[2], const int dilation[2],
                        ct_dtype dtype, void *workspace, size_t ws_bytes, void *stream)
{
    if (!in_hw || !k_hw || !stride || !padding || !output_padding || !dilation)
        return CT_ERR_ARG;
    Problem pb;
    ct_status st = make_problem(2, N, C_in, C_out, in_hw, k_hw, groups, stride, padding,
                                output_padding, dilation, dtype, bias != nullptr, false, &pb);
    if (st != CT_OK) return st;
    Args a{x, w, bias, nullptr, y, workspace, ws_bytes, (cudaStream_t)stream};
    return run(pb, a);
}

ct_status ct_forward_2d_add_hswish(const void *x, const void *w, const float *bias,
                                   const float *add, float *y,
                                   int N, int C_in, int C_out, const int in_hw[2],
                                   const int k_hw[2], int groups, const int stride[2],
                                   const int padding[2], const int output_padding[2],
                                   const int dilation[2], ct_dtype dtype,
                                   void *workspace, size_t ws_bytes, void *stream)
{
    if (!in_hw || !k_hw || !stride || !padding || !output_padding || !dilation)
        return CT_ERR_ARG;
    if (!add) return CT_ERR_ARG;
    Problem pb;
    ct_status st = make_problem(2, N, C_in, C_out, in_hw, k_hw, groups, stride, padding,
                                output_padding, dilation, dtype, bias != nullptr, true, &pb);
    if (st != CT_OK) return st;
    Args a{x, w, bias, add, y, workspace, ws_bytes, (cudaStream_t)stream};
    return run(pb, a);
}

const char *ct_path_1d(int N, int C_in, int C_out, int L_in, int k, int groups, int stride,
                       int padding, int output_padding, int dilation, ct_dtype dtype)
{
    Problem pb;
    if (make_problem(1, N, C_in, C_out, &L_in, &k, groups, &stride, &padding, &output_padding,
                     &dilation, dtype, false, false, &pb) != CT_OK)
        return nullptr;
    return path_name(choose_path(pb, nullptr), pb);
}

const char *ct_path_3d(int N, int C_in, int C_out, const int in_dhw[3], const int k_dhw[3],
                       int groups, const int stride[3], const int padding[3],
                       const int output_padding[3], const int dilation[3], ct_dtype dtype,
                       int fused)
{
    if (!in_dhw || !k_dhw || !stride || !padding || !output_padding || !dilation) return nullptr;
    Problem pb;
    if (make_problem(3, N, C_in, C_out, in_dhw, k_dhw, groups, stride, padding, output_padding,
                     dilation, dtype, false, fused != 0, &pb) != CT_OK)
        return nullptr;
    return path_name(choose_path(pb, nullptr), pb);
}

ct_status ct_workspace_size_cl(int nd, int N, int C_in, int C_out, const int *in_size, const int *k,
                               int groups, const int *stride, const int *padding,
                               const int *output_padding, const int *dilation, ct_dtype dtype,
                               size_t *bytes)
{
    if (!bytes || !in_size || !k || !stride || !padding || !output_padding || !dilation) return CT_ERR_ARG;
    Problem pb;
    ct_status st = make_problem(nd, N, C_in, C_out, in_size, k, groups, stride, padding, output_padding,
                                dilation, dtype, false, false, &pb);
    if (st != CT_OK) return st;
    pb.cl = true;
    *bytes = workspace_bytes(pb);
    return CT_OK;
}

ct_status ct_forward_cl(int nd, const void *x, const void *w, const float *bias, const float *add,
                        float *y, int N, int C_in, int C_out, const int *in_size, const int *k,
                        int groups, const int *stride, const int *padding,
                        const int *output_padding, const int *dilation, ct_dtype dtype,
                        void *workspace, size_t ws_bytes, void *stream)
{
    if (!in_size || !k || !stride || !padding || !output_padding || !dilation) return CT_ERR_ARG;
    Problem pb;
    ct_status st = make_problem(nd, N, C_in, C_out, in_size, k, groups, stride, padding, output_padding,
                                dilation, dtype, bias != nullptr, add != nullptr, &pb);
    if (st != CT_OK) return st;
    pb.cl = true;
    Args a{x, w, bias, add, y, workspace, ws_bytes, (cudaStream_t)stream};
    return run(pb, a);
}

const char *ct_path_cl(int nd, int N, int C_in, int C_out, const int *in_size, const int *k, int groups,
                       const int *stride, const int *padding, const int *output_padding,
                       const int *dilation, ct_dtype dtype, int fused)
{
    if (!in_size || !k || !stride || !padding || !output_padding || !dilation) return nullptr;
    Problem pb;
    if (make_problem(nd, N, C_in, C_out, in_size, k, groups, stride, padding, output_padding, dilation,
                     dtype, false, fused != 0, &pb) != CT_OK)
        return nullptr;
    pb.cl = true;
    return path_name(choose_path(pb, nullptr), pb);
}

const char *ct_path_2d(int N, int C_in, int C_out, const int in_hw[2], const int k_hw[2],
                       int groups, const int stride[2], const int padding[2],
                       const int output_padding[2], const int dilation[2], ct_dtype dtype,
                       int fused)
{
    if (!in_hw || !k_hw || !stride || !padding || !output_padding || !dilation) return nullptr;
    Problem pb;
    if (make_problem(2, N, C_in, C_out, in_hw, k_hw, groups, stride, padding, output_padding,
                     dilation, dtype, false, fused != 0, &pb) != CT_OK)
        return nullptr;
    return path_name(choose_path(pb, nullptr), pb);
}

const char *ct_path_call(int nd, int channels_last, int N, int C_in, int C_out, const int *in_size, const int *k,
                         int groups, const int *stride, const int *padding, const int *output_padding,
                         const int *dilation, ct_dtype dtype, int fused, size_t ws_bytes)
{
    if (!in_size || !k || !stride || !padding || !output_padding || !dilation) return nullptr;
    Problem pb;
    if (make_problem(nd, N, C_in, C_out, in_size, k, groups, stride, padding, output_padding, dilation, dtype,
                     false, fused != 0, &pb) != CT_OK)
        return nullptr;
    pb.cl = channels_last != 0;
    if (ws_bytes > 0 && ws_bytes < workspace_bytes(pb)) return nullptr;     // the call returns CT_ERR_WORKSPACE
    // 256-byte aligned stand-ins for the tensors (never dereferenced: the path
    // checks look at alignment only)
    void *const any = reinterpret_cast<void *>((uintptr_t)1 << 20);
    Args a{any, any, nullptr, fused ? static_cast<const float *>(any) : nullptr, static_cast<float *>(any),
           ws_bytes ? any : nullptr, ws_bytes, nullptr};
    const Path path = choose_path(pb, &a);
    if (path == Path::Umma && ws_bytes < umma_workspace_bytes(pb)) return nullptr;
    return path_name(path, pb);
}

void ct_set_path_override(int mode) { g_override.store(mode == 1 || mode == 2 ? mode : 0); }

void ct_set_deterministic(int on) { g_deterministic.store(on ? 1 : 0); }

int ct_get_deterministic(void) { return g_deterministic.load(); }

const char *ct_status_str(ct_status s)
{
    switch (s) {
    case CT_OK: return "CT_OK";
    case CT_ERR_ARG: return "CT_ERR_ARG: invalid argument (null pointer, bad size, dtype or overlap)";
    case CT_ERR_SHAPE: return "CT_ERR_SHAPE: inconsistent shape or convolution parameters";
    case CT_ERR_ALIGN: return "CT_ERR_ALIGN: pointer not aligned to its element size";
    case CT_ERR_WORKSPACE: return "CT_ERR_WORKSPACE: workspace missing, too small or misaligned";
    case CT_ERR_UNSUPPORTED: return "CT_ERR_UNSUPPORTED: valid operator not supported by this build";
    case CT_ERR_CUDA: return "CT_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    case CT_ERR_DEVICE_TIMEOUT: return "CT_ERR_DEVICE_TIMEOUT: a bounded device-side wait ran out";
    }
    return "unknown ct_status";
}

ct_status ct_last_device_error(void *stream)
{
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CT_ERR_CUDA;
    return take_device_status();
}

}  // extern "C"
