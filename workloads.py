"""Seeded synthetic workloads for the transposed-convolution path.

This module holds the benchmark configurations (shapes, hyper-parameters,
value distributions, seeds) and the random-number generation for their
inputs.  It holds none of the convolution's arithmetic: no output-length
formula, no index mapping, no epilogue.  Both the CUDA path's tests/bench and
the CPU oracle draw their inputs from here, so the two sides always consume
identical values.

Distributions follow the workload descriptions: x ~ N(0, 1); weights and bias
~ U(-b, b) with the stated bound b; the fused workload's add tensor ~ N(0, 1).
The bf16 workload rounds x and w to bf16 once, here (round to nearest even),
and both sides consume the same bf16 values.  Generator: numpy PCG64 via
``numpy.random.default_rng(seed)``; draw order is x, w, bias, add.
"""
import math

import numpy as np

# Workload descriptions.  `out_shape` is stated only where the workload
# description states it (the fused add tensor); elsewhere callers derive it.
CONFIGS = {
    "convT1d_tiny": dict(
        desc="ConvTranspose1d fp32 N=2 C_in=4 C_out=8 k=3 s=2 p=1 d=2 L_in=64 bias",
        nd=1, N=2, C_in=4, C_out=8, groups=1, L_in=(64,), k=(3,), stride=(2,),
        padding=(1,), output_padding=(0,), dilation=(2,), bias=True, add=False,
        dtype="f32", bound=1.0 / math.sqrt(8 * 3), seed=1),
    "convT1d_L131072": dict(
        desc="ConvTranspose1d fp32 N=16 C_in=32 C_out=64 k=3 s=2 p=1 d=2 L_in=131072 no bias",
        nd=1, N=16, C_in=32, C_out=64, groups=1, L_in=(131072,), k=(3,), stride=(2,),
        padding=(1,), output_padding=(0,), dilation=(2,), bias=False, add=False,
        dtype="f32", bound=1.0 / math.sqrt(192), seed=2),
    "convT3d_grouped": dict(
        desc=("ConvTranspose3d fp32 N=8 C_in=32 C_out=32 groups=4 k=(3,5,7) s=2 "
              "p=(1,2,3) op=1 in=16x32x32 bias"),
        nd=3, N=8, C_in=32, C_out=32, groups=4, L_in=(16, 32, 32), k=(3, 5, 7),
        stride=(2, 2, 2), padding=(1, 2, 3), output_padding=(1, 1, 1), dilation=(1, 1, 1),
        bias=True, add=False, dtype="f32", bound=1.0 / math.sqrt(8 * 105), seed=3),
    "convT3d_add_hswish": dict(
        desc=("ConvTranspose3d fp32 N=128 C_in=32 C_out=64 k=3 s=2 p=1 op=1 in=16^3 bias, "
              "+ add (128,64,32,32,32), out = t*hardswish(t)"),
        nd=3, N=128, C_in=32, C_out=64, groups=1, L_in=(16, 16, 16), k=(3, 3, 3),
        stride=(2, 2, 2), padding=(1, 1, 1), output_padding=(1, 1, 1), dilation=(1, 1, 1),
        bias=True, add=True, out_shape=(128, 64, 32, 32, 32), dtype="f32",
        bound=1.0 / math.sqrt(64 * 27), seed=4),
    "convT3d_bf16_dense": dict(
        desc=("ConvTranspose3d bf16-in/fp32-accumulate N=16 C_in=256 C_out=128 k=4 s=2 p=1 "
              "in=16^3 bias"),
        nd=3, N=16, C_in=256, C_out=128, groups=1, L_in=(16, 16, 16), k=(4, 4, 4),
        stride=(2, 2, 2), padding=(1, 1, 1), output_padding=(0, 0, 0), dilation=(1, 1, 1),
        bias=True, add=False, dtype="bf16", bound=1.0 / math.sqrt(128 * 64), seed=5),
    # ConvTranspose2d: the fused workload's layer (32 -> 64, k3 s2 p1 op1) and
    # the bf16 workload's layer (256 -> 128, k4 s2 p1) on 2-D images; no page
    # states a 2-D size, so these take the 3-D workloads' channel counts,
    # kernels and output bytes (1.07 GB and 134 MB of fp32 output)
    "convT2d_f32": dict(
        desc="ConvTranspose2d fp32 N=64 C_in=32 C_out=64 k=3 s=2 p=1 op=1 in=128x128 bias",
        nd=2, N=64, C_in=32, C_out=64, groups=1, L_in=(128, 128), k=(3, 3), stride=(2, 2),
        padding=(1, 1), output_padding=(1, 1), dilation=(1, 1), bias=True, add=False,
        dtype="f32", bound=1.0 / math.sqrt(64 * 9), seed=6),
    "convT2d_bf16_dense": dict(
        desc=("ConvTranspose2d bf16-in/fp32-accumulate N=16 C_in=256 C_out=128 k=4 s=2 p=1 "
              "in=64x64 bias"),
        nd=2, N=16, C_in=256, C_out=128, groups=1, L_in=(64, 64), k=(4, 4), stride=(2, 2),
        padding=(1, 1), output_padding=(0, 0), dilation=(1, 1), bias=True, add=False,
        dtype="bf16", bound=1.0 / math.sqrt(128 * 16), seed=7),
    # the bf16 workload with channels-last x and y (N, D, H, W, C): the same
    # draws, stored channels-last
    "convT3d_bf16_dense_cl": dict(
        desc=("ConvTranspose3d bf16-in/fp32-accumulate N=16 C_in=256 C_out=128 k=4 s=2 p=1 "
              "in=16^3 bias, channels-last x and y"),
        nd=3, N=16, C_in=256, C_out=128, groups=1, L_in=(16, 16, 16), k=(4, 4, 4),
        stride=(2, 2, 2), padding=(1, 1, 1), output_padding=(0, 0, 0), dilation=(1, 1, 1),
        bias=True, add=False, dtype="bf16", bound=1.0 / math.sqrt(128 * 64), seed=5, layout="cl"),
    # the fused workload with channels-last x, add and y (N, D, H, W, C)
    "convT3d_add_hswish_cl": dict(
        desc=("ConvTranspose3d fp32 N=128 C_in=32 C_out=64 k=3 s=2 p=1 op=1 in=16^3 bias, "
              "+ add, out = t*hardswish(t), channels-last x, add and y"),
        nd=3, N=128, C_in=32, C_out=64, groups=1, L_in=(16, 16, 16), k=(3, 3, 3),
        stride=(2, 2, 2), padding=(1, 1, 1), output_padding=(1, 1, 1), dilation=(1, 1, 1),
        bias=True, add=True, out_shape=(128, 64, 32, 32, 32), dtype="f32",
        bound=1.0 / math.sqrt(64 * 27), seed=4, layout="cl"),
    # strides other than 2 (the l1_p79 "wavefronts" passage: s phases per
    # dimension with disjoint writes): no page states such a size, so these
    # take the grouped workload's 16^3 input with 32 -> 32 channels.  k = s = 3
    # lies in the disjoint regime s > (k - 1) d (every output receives exactly
    # one tap per dimension); k = 5, s = 3, p = 1 has overlapping phases (1 or
    # 2 taps per dimension)
    "convT3d_s3_disjoint": dict(
        desc="ConvTranspose3d fp32 N=16 C_in=32 C_out=32 k=3 s=3 p=0 in=16^3 (out 48^3) bias",
        nd=3, N=16, C_in=32, C_out=32, groups=1, L_in=(16, 16, 16), k=(3, 3, 3),
        stride=(3, 3, 3), padding=(0, 0, 0), output_padding=(0, 0, 0), dilation=(1, 1, 1),
        bias=True, add=False, dtype="f32", bound=1.0 / math.sqrt(32 * 27), seed=8),
    "convT3d_s3_k5": dict(
        desc="ConvTranspose3d fp32 N=16 C_in=32 C_out=32 k=5 s=3 p=1 in=16^3 (out 48^3) bias",
        nd=3, N=16, C_in=32, C_out=32, groups=1, L_in=(16, 16, 16), k=(5, 5, 5),
        stride=(3, 3, 3), padding=(1, 1, 1), output_padding=(0, 0, 0), dilation=(1, 1, 1),
        bias=True, add=False, dtype="f32", bound=1.0 / math.sqrt(32 * 125), seed=9),
}

CONFIG_ORDER = ["convT1d_tiny", "convT1d_L131072", "convT3d_grouped",
                "convT3d_add_hswish", "convT3d_bf16_dense", "convT2d_f32", "convT2d_bf16_dense",
                "convT3d_bf16_dense_cl", "convT3d_add_hswish_cl", "convT3d_s3_disjoint", "convT3d_s3_k5"]


def bf16_round(a):
    """Round float32 values to bf16 (nearest, ties to even).

    Returns (bits: uint16 array, values: float32 array holding the bf16 values).
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32)
    lsb = (bits >> np.uint32(16)) & np.uint32(1)
    hi = ((bits + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    vals = (hi.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return hi, vals


def _uniform(rng, shape, bound):
    u = rng.random(shape, dtype=np.float32)
    return ((u * np.float32(2.0) - np.float32(1.0)) * np.float32(bound)).astype(np.float32)


def make_tensors(seed, x_shape, w_shape, bound, bias_len=None, add_shape=None,
                 dtype="f32", x_kind="normal", int_range=None):
    """Draw one set of inputs.

    x_kind "normal": x ~ N(0,1), w/bias ~ U(-bound, bound), add ~ N(0,1).
    int_range=r: every tensor holds integers drawn uniformly from [-r, r]
    (exactly representable in fp32 and bf16), for order-independent checks.
    Returns a dict with float32 arrays x, w, bias (or None), add (or None);
    for dtype "bf16" also x_bits, w_bits (uint16) and x, w hold the bf16 values.
    """
    rng = np.random.default_rng(seed)
    if int_range is not None:
        r = int(int_range)
        x = rng.integers(-r, r + 1, size=x_shape).astype(np.float32)
        w = rng.integers(-r, r + 1, size=w_shape).astype(np.float32)
        bias = (rng.integers(-r, r + 1, size=(bias_len,)).astype(np.float32)
                if bias_len else None)
        add = (rng.integers(-r, r + 1, size=add_shape).astype(np.float32)
               if add_shape is not None else None)
    else:
        x = rng.standard_normal(x_shape, dtype=np.float32)
        w = _uniform(rng, w_shape, bound)
        bias = _uniform(rng, (bias_len,), bound) if bias_len else None
        add = (rng.standard_normal(add_shape, dtype=np.float32)
               if add_shape is not None else None)
    out = dict(x=x, w=w, bias=bias, add=add)
    if dtype == "bf16":
        out["x_bits"], out["x"] = bf16_round(x)
        out["w_bits"], out["w"] = bf16_round(w)
    return out


def config_shapes(cfg, N=None):
    """x and w shapes of a configuration (optionally with another batch size)."""
    n = cfg["N"] if N is None else N
    x_shape = (n, cfg["C_in"]) + tuple(cfg["L_in"])
    w_shape = (cfg["C_in"], cfg["C_out"] // cfg["groups"]) + tuple(cfg["k"])
    return x_shape, w_shape


def config_inputs(name, N=None, int_range=None, seed=None):
    """Inputs of a named configuration.  N overrides the batch size (the
    first N batch items of a draw are NOT the same as a smaller draw; callers
    that sample compare both sides on the same draw)."""
    cfg = CONFIGS[name]
    x_shape, w_shape = config_shapes(cfg, N)
    add_shape = None
    if cfg["add"]:
        add_shape = (x_shape[0],) + tuple(cfg["out_shape"][1:])
    return make_tensors(cfg["seed"] if seed is None else seed, x_shape, w_shape, cfg["bound"],
                        bias_len=cfg["C_out"] if cfg["bias"] else None,
                        add_shape=add_shape, dtype=cfg["dtype"], int_range=int_range)
