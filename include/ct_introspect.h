/*
 * ct_introspect.h -- host-only introspection and test hooks of libct.so.
 *
 * Nothing here computes: these calls report which kernel family a forward
 * call of include/ct.h would launch, and let tests force the dispatcher onto
 * a given family.  A program that only computes needs ct.h alone.
 *
 * Kernel family names:
 *   "gather_generic"  any valid problem (one thread per output block)
 *   "phase1d_f32"     FP32 1-D, stride-phase FFMA kernel
 *   "tc1d_tf32x3"     FP32 1-D on the tensor cores (three-term tf32 split)
 *   "phase3d_f32"     FP32 2-D / 3-D, stride-phase FFMA kernel
 *   "tc3d_tf32x3"     FP32 2-D / 3-D, dense channels, tensor cores, tf32 split
 *   "tc3d_bf16x2"     the same with the opt-in two-term bf16 split (CT_F32_BF16X2)
 *   "tc3dg_tf32x3"    FP32 2-D / 3-D, 32 input channels in 1, 2 or 4 groups,
 *                     tensor cores, tf32 split
 *   "tc3dg_bf16x2"    the same with the opt-in two-term bf16 split
 *   "tc3s_tf32x3"     FP32 1-D / 2-D / 3-D with strides 1 to 4 and any
 *                     dilation (groups 1), tensor cores, tf32 split
 *   "tc3s_bf16x2"     the same with the opt-in two-term bf16 split
 *   "umma_bf16"       bf16 2-D / 3-D on the tensor cores
 */
#ifndef CT_INTROSPECT_H
#define CT_INTROSPECT_H

#include <stddef.h>

#include "ct.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Kernel family the 1-D / 2-D / 3-D / fused call with these arguments
 * (ct_path_cl: in channels-last layouts) would launch when given the workspace
 * ct_workspace_size_* reports, or NULL if the arguments are invalid.  Host
 * only; launches nothing.  `fused` selects the add + hardswish variant for the
 * 2-D and 3-D queries. */
const char *ct_path_1d(int N, int C_in, int C_out, int L_in, int k, int groups, int stride,
                       int padding, int output_padding, int dilation, ct_dtype dtype);
const char *ct_path_2d(int N, int C_in, int C_out, const int in_hw[2], const int k_hw[2],
                       int groups, const int stride[2], const int padding[2],
                       const int output_padding[2], const int dilation[2], ct_dtype dtype,
                       int fused);
const char *ct_path_cl(int nd, int N, int C_in, int C_out, const int *in_size, const int *k, int groups,
                       const int *stride, const int *padding, const int *output_padding,
                       const int *dilation, ct_dtype dtype, int fused);
const char *ct_path_3d(int N, int C_in, int C_out, const int in_dhw[3], const int k_dhw[3],
                       int groups, const int stride[3], const int padding[3],
                       const int output_padding[3], const int dilation[3], ct_dtype dtype,
                       int fused);

/* Kernel family a forward call would launch given exactly `ws_bytes` of
 * (256-byte aligned, 16-byte aligned tensors) workspace: ws_bytes = 0 is a
 * call without workspace, which takes the kernels that need none (the FFMA or
 * generic kernel for FP32 2-D / 3-D shapes whose tensor-core path needs
 * scratch).  NULL if the arguments are invalid or if the call would return
 * CT_ERR_WORKSPACE (0 < ws_bytes < the reported size, or a bf16 tensor-core
 * shape without workspace).  nd = 1, 2, 3 (array arguments of nd entries,
 * outermost spatial dimension first); channels_last selects the layouts of
 * ct_forward_cl. */
const char *ct_path_call(int nd, int channels_last, int N, int C_in, int C_out, const int *in_size, const int *k,
                         int groups, const int *stride, const int *padding, const int *output_padding,
                         const int *dilation, ct_dtype dtype, int fused, size_t ws_bytes);

/* Test hook: process-wide path override of the dispatcher.  0 = automatic
 * (default), 1 = always the generic gather kernel, 2 = automatic but without
 * the FP32 tensor-core paths (the FFMA phase kernels instead).  Not
 * thread-safe against concurrent forward calls; meant for tests only. */
void ct_set_path_override(int mode);

#ifdef __cplusplus
}
#endif

#endif /* CT_INTROSPECT_H */
