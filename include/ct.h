/*
 * ct.h -- C ABI of the GB300 (sm_103a) forward transposed-convolution library
 * (libct.so).
 *
 * What it computes (POPCORNBENCH reasoning traces, cited by task id):
 *   [l1_p79] trace Kimi-K2.6__l1_p79, ConvTranspose1d with dilation 2: the
 *            output-length formula and the scatter rule
 *            y[n, oc, i*s - p + k*d] += x[n, ic, i] * w[ic, oc, k].
 *   [l1_p72] trace Kimi-K2.6__l1_p72, ConvTranspose3d with groups=4 and an
 *            asymmetric kernel: weight layout (C_in, C_out/groups, kD, kH, kW),
 *            grouped channel mapping, direct accumulation without flipping.
 *   [l2_p26] trace Kimi-K2.6__l2_p26, ConvTranspose3d + add + x*hardswish(x):
 *            t = convT(x) + bias + add;  out = t * hardswish(t),
 *            hardswish(t) = t * clamp(t + 3, 0, 6) / 6.
 *
 * For every spatial dimension d:
 *     L_out[d] = (L_in[d] - 1)*s[d] - 2*p[d] + dl[d]*(k[d] - 1) + op[d] + 1
 * and
 *     y[n, oc, o] = bias[oc] + sum over ic in oc's group, taps k with
 *                   o = i*s - p + k*dl for an input position 0 <= i < L_in
 *                   of x[n, ic, i] * w[ic, oc mod (C_out/groups), k]
 * (per-dimension relations, product over dimensions).  An output no tap
 * reaches holds bias[oc] (or 0 without bias); the output_padding tail is
 * computed by the same rule.
 *
 * Layouts (all contiguous, row-major, owned by the caller, device memory):
 *     x    (N, C_in, L)              or (N, C_in, D, H, W)       dtype CT_F32 or CT_BF16
 *     w    (C_in, C_out/groups, k)   or (C_in, C_out/groups, kD, kH, kW)   same dtype as x
 *     bias (C_out,)  fp32, may be NULL
 *     add  shape of y, fp32 (fused entry point only)
 *     y    (N, C_out, L_out) or (N, C_out, D_out, H_out, W_out), always fp32
 * N may be 0: the call then validates the other arguments, launches nothing
 * and accepts NULL x, y and add.
 * y must not overlap x, w or bias.  y may be the same buffer as add (each
 * element of add is read before the same thread writes that element of y).
 *
 * Execution: every forward call only validates its arguments on the host,
 * then enqueues kernels on `stream` (a cudaStream_t; NULL = the legacy
 * default stream) and returns; nothing is synchronised and no device memory
 * is allocated.  The tensor-core paths keep repacked operands in scratch
 * memory taken from the caller-supplied `workspace`.  A workspace is either
 * absent (workspace = NULL or ws_bytes = 0) or at least the size that
 * ct_workspace_size_* reports for the same arguments and 256-byte aligned;
 * anything in between returns CT_ERR_WORKSPACE.  The bf16 tensor-core path
 * requires it (CT_ERR_WORKSPACE without); an FP32 2-D or 3-D call without a
 * workspace runs the kernels that need none (the FFMA or generic kernel,
 * same results up to rounding, slower) -- ct_path_call in ct_introspect.h
 * reports which.  The workspace is overwritten; calls that share one must
 * not overlap on the GPU.
 *
 * Errors: argument and shape errors are returned synchronously before any
 * launch and leave y untouched.  A failed launch returns CT_ERR_CUDA.  Every
 * wait of the pipelined kernels is bounded; a wait that runs out records
 * CT_ERR_DEVICE_TIMEOUT in a status word in page-locked host memory that the
 * kernels write directly.  The next forward call that finds it set returns
 * CT_ERR_DEVICE_TIMEOUT without launching (and clears it), as does
 * ct_last_device_error(), which synchronises the stream first.  The word is
 * registered with cudaHostRegister on the first launch; make that first call
 * before any stream capture.
 */
#ifndef CT_H
#define CT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CT_OK = 0,
    CT_ERR_ARG = 1,            /* NULL pointer, non-positive size, bad dtype        */
    CT_ERR_SHAPE = 2,          /* groups do not divide channels, L_out <= 0,        */
                               /* output_padding >= max(stride, dilation), p < 0 ... */
    CT_ERR_ALIGN = 3,          /* a pointer is not aligned to its element size      */
    CT_ERR_WORKSPACE = 4,      /* workspace missing, too small or not 256-B aligned */
    CT_ERR_UNSUPPORTED = 5,    /* valid operator this build does not run            */
    CT_ERR_CUDA = 6,           /* a CUDA runtime call or launch failed              */
    CT_ERR_DEVICE_TIMEOUT = 7  /* a bounded device-side wait ran out                */
} ct_status;

/* dtype of x and w (bias, add and y are always fp32):
 *   CT_F32         fp32.  The result is FP32-accurate: every path computes in
 *                  fp32, or on the tensor cores from a three-term tf32 split of
 *                  each operand (error within about 2^-20 of sum |x||w| per
 *                  output, the accuracy of fp32 arithmetic over the same sum).
 *   CT_BF16        bf16 x and w, fp32 accumulation.
 *   CT_F32_BF16X2  fp32 x and w, as CT_F32, for callers that accept about
 *                  16-bit operand precision: the 2-D and 3-D FP32 tensor-core
 *                  paths multiply a two-term bf16 split of each operand
 *                  (relative error up to about 2^-16 of sum |x||w| per output)
 *                  and issue fewer MMAs.  Opt-in only; every other path computes
 *                  as with CT_F32. */
typedef enum { CT_F32 = 0, CT_BF16 = 1, CT_F32_BF16X2 = 2 } ct_dtype;

/* Output length of one spatial dimension ([l1_p79] output-length formula),
 * or -1 if the parameters are invalid (k, s, dl < 1; p, op < 0; result < 1). */
int64_t ct_out_len(int64_t L_in, int k, int s, int p, int op, int dl);

/* Scratch bytes a forward call with these arguments needs to take its
 * fastest path (0 when that path needs none).  Same argument meaning as the
 * forward calls below. */
ct_status ct_workspace_size_1d(int N, int C_in, int C_out, int L_in, int k, int groups,
                               int stride, int padding, int output_padding, int dilation,
                               ct_dtype dtype, size_t *bytes);
ct_status ct_workspace_size_3d(int N, int C_in, int C_out, const int in_dhw[3],
                               const int k_dhw[3], int groups, const int stride[3],
                               const int padding[3], const int output_padding[3],
                               const int dilation[3], ct_dtype dtype, size_t *bytes);
ct_status ct_workspace_size_2d(int N, int C_in, int C_out, const int in_hw[2], const int k_hw[2],
                               int groups, const int stride[2], const int padding[2],
                               const int output_padding[2], const int dilation[2], ct_dtype dtype,
                               size_t *bytes);

/* ConvTranspose1d forward ([l1_p79]).  x (N, C_in, L_in), w (C_in,
 * C_out/groups, k), bias (C_out) or NULL, y (N, C_out, L_out) fp32. */
ct_status ct_forward_1d(const void *x, const void *w, const float *bias, float *y,
                        int N, int C_in, int C_out, int L_in, int k, int groups,
                        int stride, int padding, int output_padding, int dilation,
                        ct_dtype dtype, void *workspace, size_t ws_bytes, void *stream);

/* ConvTranspose3d forward ([l1_p72]).  in_dhw = (D, H, W) of x, k_dhw the
 * kernel extent; stride, padding, output_padding, dilation per (D, H, W). */
ct_status ct_forward_3d(const void *x, const void *w, const float *bias, float *y,
                        int N, int C_in, int C_out, const int in_dhw[3], const int k_dhw[3],
                        int groups, const int stride[3], const int padding[3],
                        const int output_padding[3], const int dilation[3],
                        ct_dtype dtype, void *workspace, size_t ws_bytes, void *stream);

/* ConvTranspose2d forward ([l1_p72]: its ConvTranspose2d asides -- every input
 * element scatter-adds weight x value into the output, unflipped, and the
 * output size (H - 1)s - 2p + d(k - 1) + op + 1 per dimension).  x (N, C_in, H,
 * W), w (C_in, C_out/groups, kH, kW), bias (C_out) or NULL, y (N, C_out, H_out,
 * W_out) fp32; in_hw = (H, W), the other arrays per (H, W).  Computed as the 3-D
 * operator with a unit D dimension (extent 1, stride 1, no padding), which has
 * the same memory layouts, so it takes the same kernels; workspace as
 * ct_workspace_size_2d reports.  Errors as ct_forward_3d. */
ct_status ct_forward_2d(const void *x, const void *w, const float *bias, float *y,
                        int N, int C_in, int C_out, const int in_hw[2], const int k_hw[2],
                        int groups, const int stride[2], const int padding[2],
                        const int output_padding[2], const int dilation[2],
                        ct_dtype dtype, void *workspace, size_t ws_bytes, void *stream);

/* ConvTranspose2d + add + x*hardswish(x): the epilogue of
 * ct_forward_3d_add_hswish on the 2-D operator of ct_forward_2d.  add has the
 * shape of y (fp32) and must not be NULL; y may equal add. */
ct_status ct_forward_2d_add_hswish(const void *x, const void *w, const float *bias,
                                   const float *add, float *y,
                                   int N, int C_in, int C_out, const int in_hw[2],
                                   const int k_hw[2], int groups, const int stride[2],
                                   const int padding[2], const int output_padding[2],
                                   const int dilation[2], ct_dtype dtype,
                                   void *workspace, size_t ws_bytes, void *stream);

/* Channels-last layouts, for 1-D, 2-D or 3-D (nd = 1, 2, 3; the array
 * arguments have nd entries, outermost spatial dimension first): x (N,
 * spatial..., C_in), y and add (N, spatial out..., C_out), w (C_in,
 * C_out/groups, k...) as in the other calls.  The same operator as
 * ct_forward_1d/2d/3d (and, with add != NULL, the fused epilogue of
 * ct_forward_3d_add_hswish; add may equal y), only the memory order of x, y
 * and add differs: channels are the fastest index.  A bf16 call of a shape
 * the bf16 tensor-core kernel takes (stride 2, even kernel extents, ...) reads
 * x in place -- no repacked copy -- and needs workspace only for the weight
 * panels (ct_workspace_size_cl); x and y then need 16-byte alignment.  Other
 * shapes run the generic kernel.  Errors as ct_forward_3d. */
ct_status ct_workspace_size_cl(int nd, int N, int C_in, int C_out, const int *in_size, const int *k,
                               int groups, const int *stride, const int *padding,
                               const int *output_padding, const int *dilation, ct_dtype dtype,
                               size_t *bytes);
ct_status ct_forward_cl(int nd, const void *x, const void *w, const float *bias, const float *add,
                        float *y, int N, int C_in, int C_out, const int *in_size, const int *k,
                        int groups, const int *stride, const int *padding,
                        const int *output_padding, const int *dilation, ct_dtype dtype,
                        void *workspace, size_t ws_bytes, void *stream);

/* Fused ConvTranspose3d + add + x*hardswish(x) ([l2_p26]):
 *     t = convT(x) + bias + add;  y = t * (t * clamp(t + 3, 0, 6) / 6).
 * add has the shape of y (fp32) and must not be NULL; y may equal add. */
ct_status ct_forward_3d_add_hswish(const void *x, const void *w, const float *bias,
                                   const float *add, float *y,
                                   int N, int C_in, int C_out, const int in_dhw[3],
                                   const int k_dhw[3], int groups, const int stride[3],
                                   const int padding[3], const int output_padding[3],
                                   const int dilation[3], ct_dtype dtype,
                                   void *workspace, size_t ws_bytes, void *stream);

/* The same bf16 ConvTranspose3d as ct_forward_3d, for callers that cannot
 * allocate device memory: no workspace argument, and no cudaMalloc, cudaFree
 * or other allocating call inside.  The pages have no counterpart of this
 * entry point; it serves callers such as an engine that reserves all device
 * memory at start-up and forbids allocation afterwards, a plugin running
 * inside a host framework that owns the device memory pool, or an
 * allocation-free real-time loop -- none of them can hand ct_forward_3d a
 * freshly allocated workspace.
 *
 * Scratch: a buffer of CT_NOALLOC_SCRATCH_BYTES (48 MiB) that the library
 * owns, a static device array that every GPU which loads libct.so keeps
 * until the process exits.  Every call looks up the buffer's device address
 * (cudaGetSymbolAddress) with the caller's device and context current, so
 * the address is always that of the current context, also after a
 * cudaDeviceReset; the first call on a device loads the library's module
 * there, so make that first call before any stream capture.  Every call on a
 * device shares the one buffer, so calls that overlap on the GPU (different
 * streams, or other threads) race and must be serialised by the caller.
 * Each call rewrites every scratch byte it reads, so no state carries over
 * from the last call and nothing needs clearing.
 *
 * Arguments and layouts as ct_forward_3d with dtype CT_BF16.  Returns
 * CT_ERR_UNSUPPORTED when the arguments do not take the bf16 tensor-core
 * path (other paths need no scratch: use ct_forward_3d), CT_ERR_WORKSPACE
 * when the problem needs more scratch than CT_NOALLOC_SCRATCH_BYTES (the
 * size ct_workspace_size_3d reports for the same arguments), CT_ERR_CUDA
 * when the address lookup or a launch fails. */
#define CT_NOALLOC_SCRATCH_BYTES (48u * 1024u * 1024u)
ct_status ct_forward_3d_noalloc(const void *x, const void *w, const float *bias, float *y,
                                int N, int C_in, int C_out, const int in_dhw[3], const int k_dhw[3],
                                int groups, const int stride[3], const int padding[3],
                                const int output_padding[3], const int dilation[3],
                                ct_dtype dtype, void *stream);

/* Bitwise reproducibility (process-wide, read at each forward call's launch).
 * Every path computes each output in a fixed order, so repeated calls on the
 * same inputs give identical bits, except the grouped FP32 tensor-core path
 * ("tc3dg_*" in ct_introspect.h), which by default issues each group's MMAs
 * from two threads whose contributions to an output accumulate in no fixed
 * order (results then differ between calls in the last bits, within the
 * path's stated error).  ct_set_deterministic(1) makes that path issue from
 * one thread per group (about 12 % slower on the grouped workload) and every
 * call reproducible; 0 (the default) restores it.  Not synchronised with
 * forward calls in flight on other threads. */
void ct_set_deterministic(int on);
int ct_get_deterministic(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *ct_status_str(ct_status s);

/* Synchronises `stream`, then returns and clears the status word: CT_OK, or
 * CT_ERR_DEVICE_TIMEOUT if a bounded wait in a kernel ran out since the last
 * query (by this call or by a forward call); CT_ERR_CUDA if synchronising
 * failed. */
ct_status ct_last_device_error(void *stream);

/* Failure-detection self-test: launches on `stream` a one-thread kernel that
 * waits on an mbarrier nothing arrives at, with a limit of `limit_ns`
 * nanoseconds (1 .. 1e9), the same bounded wait every pipelined kernel of the
 * library uses.  The wait runs out, CT_ERR_DEVICE_TIMEOUT is recorded in the
 * device status word, and the kernel returns normally: the context stays
 * usable and the next ct_last_device_error() reports the timeout.  No
 * fault, no hang.  Returns CT_ERR_ARG for a limit out of range, CT_ERR_CUDA
 * if the launch fails. */
ct_status ct_selftest_wait_timeout(uint64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CT_H */
