// ct_noalloc.cu -- ct_forward_3d_noalloc: the bf16 tensor-core
// ConvTranspose3d for callers that cannot allocate device memory.
//
// The bf16 path needs scratch memory (the channels-last copy of x and the
// per-phase packed weights).  ct_forward_3d takes that scratch from the
// caller as a workspace; some callers cannot provide one because they may
// not allocate device memory at all (see include/ct.h).  This entry point
// uses instead a fixed buffer that the library owns: the file-scope device
// array below, CT_NOALLOC_SCRATCH_BYTES large, which every GPU that loads
// the library keeps until the process exits.  Nothing here calls cudaMalloc,
// cudaFree or any other allocating routine.
//
// Host code must not use the array's name as a device pointer: in host code
// it only stands for the symbol.  The device address belongs to the context
// that is current when it is looked up (the module is loaded per context),
// so every call looks it up with cudaGetSymbolAddress, with the caller's
// device and context current, and checks the result.  A cached address
// could outlive its context (cudaDeviceReset, or a context the caller made
// current); the lookup costs microseconds once the module is loaded.  The
// first call on a device sets the module up there.
#include "ct_internal.h"

namespace ct {
namespace {

static_assert(CT_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// The library-owned scratch of ct_forward_3d_noalloc (one per device).
static __device__ __align__(256) unsigned char g_noalloc_scratch[CT_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context.
cudaError_t scratch_address(void **out)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (!p || ((uintptr_t)p % 256) != 0) return cudaErrorInvalidValue;
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace ct

using namespace ct;

extern "C" ct_status ct_forward_3d_noalloc(const void *x, const void *w, const float *bias, float *y,
                                           int N, int C_in, int C_out, const int in_dhw[3],
                                           const int k_dhw[3], int groups, const int stride[3],
                                           const int padding[3], const int output_padding[3],
                                           const int dilation[3], ct_dtype dtype, void *stream)
{
    if (!in_dhw || !k_dhw || !stride || !padding || !output_padding || !dilation) return CT_ERR_ARG;
    Problem pb;
    ct_status st = make_problem_3d(N, C_in, C_out, in_dhw, k_dhw, groups, stride, padding,
                                   output_padding, dilation, dtype, bias != nullptr, &pb);
    if (st != CT_OK) return st;
    if (pb.N == 0) return CT_OK;
    Args a{x, w, bias, nullptr, y, nullptr, 0, (cudaStream_t)stream};
    // only the bf16 tensor-core path uses scratch; it is the one this entry point runs
    if (!takes_umma_path(pb, &a)) return CT_ERR_UNSUPPORTED;
    if (umma_workspace_bytes(pb) > (size_t)CT_NOALLOC_SCRATCH_BYTES) return CT_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return CT_ERR_CUDA;
    a.ws = scratch;
    a.ws_bytes = (size_t)CT_NOALLOC_SCRATCH_BYTES;
    return run_problem(pb, a);
}
