// ct_internal.h -- shared host-side description of one forward call and the
// launcher entry points of the kernel translation units.  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ct.h"

namespace ct {

// One validated forward problem.  Spatial dims are right-aligned into three
// slots (D, H, W); a 1-D problem has D = H = 1 with unit kernel/stride.
struct Problem {
    int nd;                                  // 1, 2 or 3 (as called; dims right-aligned in 3 slots)
    int N, C_in, C_out, G, Cig, Cog;         // Cig = C_in/G, Cog = C_out/G
    int Li[3], K[3], S[3], P[3], OP[3], DL[3], Lo[3];
    ct_dtype dtype;                          // storage type of x and w: CT_F32 or CT_BF16
    bool split2 = false;                     // CT_F32_BF16X2: fp32 storage, two-term bf16 split opted into
    bool has_bias, has_add;
    bool cl = false;                         // channels-last x, y, add: (N, spatial..., C)

    int64_t in_sp() const { return (int64_t)Li[0] * Li[1] * Li[2]; }
    int64_t out_sp() const { return (int64_t)Lo[0] * Lo[1] * Lo[2]; }
    int kvol() const { return K[0] * K[1] * K[2]; }
    int64_t y_elems() const { return (int64_t)N * C_out * out_sp(); }
    int64_t x_elems() const { return (int64_t)N * C_in * in_sp(); }
};

// Pointers of one call (device memory, owned by the caller).
struct Args {
    const void *x;
    const void *w;
    const float *bias;   // may be null
    const float *add;    // null unless the fused entry point
    float *y;
    void *ws;            // scratch (bf16 tensor-core path only)
    size_t ws_bytes;
    cudaStream_t stream;
};

// Stride-phase table of one spatial dimension: for an output o = s*q + r the
// taps that land on it are {k : (r + p - k*dl) divisible by s}, reading input
// i = q + delta_k with delta_k = (r + p - k*dl) / s (exact division).
constexpr int kMaxS = 8;
constexpr int kMaxTaps = 16;
struct PhaseDim {
    int S;
    int ntap[kMaxS];
    int k[kMaxS][kMaxTaps];
    int delta[kMaxS][kMaxTaps];
    int Q[kMaxS];            // number of outputs o < L_out with o mod S == r
};
bool build_phase_dim(int L_out, int K, int S, int P, int DL, PhaseDim *pd);

// Device address of the library's device status word (timeouts of bounded
// waits).  Valid on the current device after the first call.
unsigned int *device_status_ptr();
// Process-wide: results must be bitwise reproducible (ct_set_deterministic).
bool deterministic();

// Validation, path choice and launch of ct_api.cu, for other entry points.
ct_status make_problem_3d(int N, int C_in, int C_out, const int *in_dhw, const int *k_dhw, int groups,
                          const int *stride, const int *padding, const int *output_padding,
                          const int *dilation, ct_dtype dtype, bool has_bias, Problem *pb);
bool takes_umma_path(const Problem &pb, const Args *a);
ct_status run_problem(const Problem &pb, const Args &a);

// ---- generic gather kernel (any valid problem; fp32 or bf16 inputs) ----
cudaError_t launch_gather_generic(const Problem &pb, const Args &a);

// ---- FP32 1-D on the tensor cores (3-term tf32 split) ----
bool tc1d_supported(const Problem &pb, const Args *a);
cudaError_t launch_tc1d(const Problem &pb, const Args &a);

// ---- FP32 3-D / 2-D on the tensor cores (3-term tf32 split, or the two-term
// bf16 split when opted into; workspace) ----
bool tc3d_supported(const Problem &pb, const Args *a);
size_t tc3d_workspace_bytes(const Problem &pb);
cudaError_t launch_tc3d(const Problem &pb, const Args &a);

// ---- FP32 1-D / 2-D / 3-D with strides 1 to 4 and any dilation (groups 1) on
// the tensor cores (3-term tf32 split, or the two-term bf16 split when opted
// into; one residue pair (rD, rH) per unit; workspace) ----
bool tc3s_supported(const Problem &pb, const Args *a);
size_t tc3s_workspace_bytes(const Problem &pb);
cudaError_t launch_tc3s(const Problem &pb, const Args &a);

// ---- FP32 3-D, 32 input channels in 1/2/4 groups, on the tensor cores
// (3-term tf32 split, or the two-term bf16 split when opted into; one
// MMA-issuing warp per group; workspace) ----
bool tc3dg_supported(const Problem &pb, const Args *a);
size_t tc3dg_workspace_bytes(const Problem &pb);
cudaError_t launch_tc3dg(const Problem &pb, const Args &a);

// ---- phase-decomposed FP32 1-D kernel ----
bool phase1d_supported(const Problem &pb, const Args *a);
cudaError_t launch_phase1d(const Problem &pb, const Args &a);

// ---- phase-decomposed FP32 3-D kernel (bias / add + hardswish epilogue) ----
bool phase3d_supported(const Problem &pb, const Args *a);
cudaError_t launch_phase3d(const Problem &pb, const Args &a);

// ---- bf16 tcgen05 implicit-GEMM path ----
bool umma_supported(const Problem &pb, const Args *a);
size_t umma_workspace_bytes(const Problem &pb);
cudaError_t launch_umma(const Problem &pb, const Args &a);

}  // namespace ct
