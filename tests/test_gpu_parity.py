"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  fp32: |err| <= 1e-4 (1 + |ref|); bf16 inputs with fp32
accumulation: |err| <= 2e-2 (|ref| + rms(ref)); integer-valued inputs: exact."""
import numpy as np
import pytest

import ctcase as cc
import oracle_pins
import workloads

pytestmark = pytest.mark.gpu

CONFIGS = workloads.CONFIG_ORDER


@pytest.fixture(scope="module", autouse=True)
def gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transposed_convolution_convtranspose_gb300 import build
    build.build()
    import transposed_convolution_convtranspose_gb300 as ct
    ct.load()
    torch.cuda.set_device(0)
    yield
    ct.ct_last_device_error(torch.cuda.current_stream())


def _sync():
    import torch
    torch.cuda.synchronize()


def path_of(c):
    import transposed_convolution_convtranspose_gb300 as ct
    dt = ct.CT_BF16 if c["dtype"] == "bf16" else (ct.CT_F32_BF16X2 if c.get("split2") else ct.CT_F32)
    if c.get("layout", "cf") == "cl":
        return ct.ct_path_cl(c["nd"], c["N"], c["C_in"], c["C_out"], c["L"], c["K"], c["G"], c["S"],
                             c["P"], c["OP"], c["DL"], dt, c["add"])
    if c["nd"] == 1:
        return ct.ct_path_1d(c["N"], c["C_in"], c["C_out"], c["L"][0], c["K"][0], c["G"], c["S"][0],
                             c["P"][0], c["OP"][0], c["DL"][0], dt)
    if c["nd"] == 2:
        return ct.ct_path_2d(c["N"], c["C_in"], c["C_out"], c["L"], c["K"], c["G"], c["S"], c["P"],
                             c["OP"], c["DL"], dt, c["add"])
    return ct.ct_path_3d(c["N"], c["C_in"], c["C_out"], c["L"], c["K"], c["G"], c["S"], c["P"],
                         c["OP"], c["DL"], dt, c["add"])


# Reduced-batch versions of every workload, compared element by element.  The
# bf16 workloads are also reduced in space (8^3 and 32^2 inputs) so the scatter
# oracle finishes in seconds; their full spatial size is covered by the sampled
# test.
REDUCED = {"convT1d_tiny": dict(N=2), "convT1d_L131072": dict(N=1),
           "convT3d_grouped": dict(N=2), "convT3d_add_hswish": dict(N=2),
           "convT3d_bf16_dense": dict(N=1, L=[8, 8, 8]), "convT2d_f32": dict(N=1),
           "convT2d_bf16_dense": dict(N=1, L=[32, 32]), "convT3d_bf16_dense_cl": dict(N=1, L=[8, 8, 8]),
           "convT3d_add_hswish_cl": dict(N=2), "convT3d_s3_disjoint": dict(N=1, L=[8, 8, 8]),
           "convT3d_s3_k5": dict(N=1, L=[8, 8, 8])}


@pytest.mark.parametrize("name", CONFIGS)
def test_config_reduced_full_compare(name):
    c = cc.case_from_config(name, N=REDUCED[name]["N"])
    if "L" in REDUCED[name]:
        c["L"] = REDUCED[name]["L"]
    t = cc.make_inputs(c, seed=100 + CONFIGS.index(name), bound=workloads.CONFIGS[name]["bound"])
    y = cc.run_gpu(c, t).cpu().numpy()
    ref = cc.run_oracle(c, t)
    cc.assert_close(y, ref, c["dtype"], "%s reduced (%s)" % (name, path_of(c)))


@pytest.mark.parametrize("name", CONFIGS)
def test_config_integer_exact(name):
    """Integer inputs in [-3, 3]: every partial sum is an integer below 2^24,
    so the conv + bias result is exact in any order (the fused epilogue's
    division by 6 is compared at fp32 tolerance instead)."""
    c = cc.case_from_config(name, N=1)
    if name in ("convT3d_bf16_dense", "convT3d_bf16_dense_cl"):
        c["L"] = [8, 8, 8]
    elif name == "convT2d_bf16_dense":
        c["L"] = [32, 32]
    t = cc.make_inputs(c, seed=200 + CONFIGS.index(name), int_range=3)
    y = cc.run_gpu(c, t).cpu().numpy()
    ref = cc.run_oracle(c, t)
    if c["add"]:
        cc.assert_close(y, ref, "f32", name)
    else:
        assert y.shape == ref.shape
        assert np.array_equal(y.astype(np.float64), ref), "%s: not bit-exact (%s)" % (name, path_of(c))


@pytest.mark.parametrize("name", CONFIGS)
def test_config_full_size_sampled(name):
    """The exact workload shapes, through the same entry point the benchmark
    times, checked on sampled outputs (plus corners) by the pointwise oracle."""
    import torch
    c = cc.case_from_config(name)
    t = workloads.config_inputs(name)
    y = cc.run_gpu(c, t)
    _sync()
    shape = cc.out_shape(c)
    assert list(y.shape) == shape
    idx = cc.sample_indices(shape, 3000, seed=7)
    got = y.reshape(-1)[torch.from_numpy(idx).to(y.device)].cpu().numpy()
    ref = cc.oracle_at(c, t, idx)
    cc.assert_close(got, ref, c["dtype"], "%s full size sampled (%s)" % (name, path_of(c)))
    assert bool(torch.isfinite(y).all())
    if name in ("convT1d_tiny", "convT1d_L131072"):
        # no tap lands on an even output for (k3, s2, p1, d2): bias or exactly 0
        ev = y[:, :, 0::2]
        want = (torch.from_numpy(t["bias"]).to(y.device)[None, :, None].expand_as(ev)
                if t["bias"] is not None else torch.zeros_like(ev))
        assert torch.equal(ev, want)
    del y
    torch.cuda.empty_cache()


def _random_cases(n, seed, nd_choices=(1, 3), scale=1):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        nd = nd_choices[i % len(nd_choices)]
        r = oracle_pins.random_case(rng, nd)
        c = dict(nd=nd, N=r["N"], C_in=r["C_in"] * scale, C_out=r["C_out"] * scale, G=r["G"],
                 L=[v * (3 if nd == 1 else 1) for v in r["L"]], K=r["K"], S=r["S"], P=r["P"],
                 OP=r["OP"], DL=r["DL"], bias=bool(i % 2), add=False, dtype="f32")
        # recheck validity after scaling L
        Lo = cc.out_shape(c)
        if min(Lo[2:]) >= 1:
            out.append(c)
    return out


@pytest.mark.parametrize("forced_generic", [False, True])
def test_random_small_shapes(forced_generic):
    import transposed_convolution_convtranspose_gb300 as ct
    cases = (_random_cases(80, seed=31) + _random_cases(20, seed=32, scale=4)
             + _random_cases(30, seed=33, nd_choices=(2,)))
    ct.ct_set_path_override(1 if forced_generic else 0)
    try:
        for k, c in enumerate(cases):
            t = cc.make_inputs(c, seed=300 + k)
            y = cc.run_gpu(c, t).cpu().numpy()
            cc.assert_close(y, cc.run_oracle(c, t), "f32", "random case %d %r" % (k, c))
    finally:
        ct.ct_set_path_override(0)


def test_random_fused_and_bf16_generic():
    cases = []
    for k, c in enumerate(_random_cases(30, seed=41, nd_choices=(3,))):
        c = dict(c)
        if k % 2:
            c["add"] = True
        else:
            c["dtype"] = "bf16"
        cases.append(c)
    for k, c in enumerate(cases):
        t = cc.make_inputs(c, seed=400 + k)
        y = cc.run_gpu(c, t).cpu().numpy()
        cc.assert_close(y, cc.run_oracle(c, t), c["dtype"], "case %d %r" % (k, c))


# Shapes for the bf16 tensor-core path: stride 2, even kernel extents (taps
# per dimension 1..4), even and odd padding (input W offsets shared by both W
# phases or not), C_out from 16 (one 16-channel chunk, N = 2 C_out = 32) to
# 256 (N = 2 C_out too wide for one MMA, a single TMEM accumulator), ragged
# H blocks and odd D, one case with several tiles per persistent CTA, and 160
# tile pairs (on 152 SMs the last round's 8 pairs run as 16 single tiles).
UMMA = [
    dict(N=1, C_in=64, C_out=16, L=[2, 3, 8], K=[4] * 3, P=[1] * 3, OP=[1, 0, 0]),
    dict(N=1, C_in=64, C_out=32, L=[3, 2, 4], K=[2] * 3, P=[0] * 3, OP=[0, 1, 0]),
    dict(N=1, C_in=64, C_out=48, L=[2, 2, 9], K=[2] * 3, P=[1] * 3, OP=[0, 0, 0]),
    dict(N=2, C_in=128, C_out=128, L=[2, 4, 16], K=[4] * 3, P=[1] * 3, OP=[0, 0, 0]),
    dict(N=1, C_in=64, C_out=256, L=[2, 2, 8], K=[4] * 3, P=[1] * 3, OP=[1, 1, 0]),
    dict(N=1, C_in=64, C_out=64, L=[2, 3, 4], K=[6] * 3, P=[2] * 3, OP=[0, 0, 0]),
    dict(N=1, C_in=64, C_out=64, L=[2, 2, 4], K=[8] * 3, P=[3] * 3, OP=[0, 0, 0]),
    dict(N=1, C_in=64, C_out=96, L=[2, 3, 7], K=[4] * 3, P=[0] * 3, OP=[0, 0, 0]),
    dict(N=1, C_in=64, C_out=64, L=[3, 5, 16], K=[4] * 3, P=[1] * 3, OP=[1, 1, 0]),
    dict(N=8, C_in=64, C_out=16, L=[16, 16, 16], K=[2] * 3, P=[0] * 3, OP=[0, 0, 0]),
    dict(N=10, C_in=64, C_out=32, L=[4, 16, 16], K=[4] * 3, P=[1] * 3, OP=[0, 0, 0]),
]


@pytest.mark.parametrize("k", range(len(UMMA)))
def test_bf16_tensor_core_shapes(k):
    c = dict(nd=3, G=1, S=[2, 2, 2], DL=[1, 1, 1], bias=bool(k % 2 == 0), add=False,
             dtype="bf16", **UMMA[k])
    assert path_of(c) == "umma_bf16", (c, path_of(c))
    t = cc.make_inputs(c, seed=700 + k)
    y = cc.run_gpu(c, t).cpu().numpy()
    cc.assert_close(y, cc.run_oracle(c, t), "bf16", "umma case %d %r" % (k, c))


# Shapes for the FP32 3-D tensor-core path (stride 2, dilation 1, kernel
# extents 2..4 mixed across dimensions, padding even and odd): C_in 32 and 64
# (one and two K blocks), C_out 16 (one chunk) to 128 (a single set of TMEM
# accumulators), odd D and H output extents, and a case with several units
# per persistent CTA; every case runs plain and with the fused add epilogue.
TC3D = [
    dict(N=2, C_in=32, C_out=64, L=[3, 4, 8], K=[3, 3, 3], P=[1, 1, 1], OP=[1, 1, 1]),
    dict(N=1, C_in=64, C_out=32, L=[2, 3, 4], K=[4, 4, 4], P=[1, 1, 1], OP=[0, 0, 0]),
    dict(N=1, C_in=32, C_out=16, L=[3, 2, 8], K=[2, 3, 4], P=[0, 1, 1], OP=[1, 0, 0]),
    dict(N=1, C_in=32, C_out=128, L=[2, 2, 4], K=[3, 3, 3], P=[1, 1, 1], OP=[1, 1, 1]),
    dict(N=1, C_in=32, C_out=48, L=[2, 5, 16], K=[3, 3, 3], P=[0, 2, 1], OP=[0, 1, 1]),
    dict(N=16, C_in=32, C_out=16, L=[8, 16, 16], K=[2, 2, 2], P=[0, 0, 0], OP=[0, 0, 0]),
]


@pytest.mark.parametrize("add", [False, True])
@pytest.mark.parametrize("k", range(len(TC3D)))
def test_fp32_3d_tensor_core_shapes(k, add):
    c = dict(nd=3, G=1, S=[2, 2, 2], DL=[1, 1, 1], bias=bool(k % 2 == 0), add=add, dtype="f32",
             **TC3D[k])
    assert path_of(c) == "tc3d_tf32x3", (c, path_of(c))
    t = cc.make_inputs(c, seed=800 + k + (50 if add else 0))
    y = cc.run_gpu(c, t).cpu().numpy()
    cc.assert_close(y, cc.run_oracle(c, t), "f32", "tc3d case %d add=%s %r" % (k, add, c))


# Shapes for the FP32 3-D tensor-core path of 32 input channels in groups
# (one MMA-issuing warp per group, K steps of the shared 128-byte rows):
# 4 groups of 8 with the asymmetric (3, 5, 7) kernel and ragged qw / qh
# blocks, 2 groups of 16 with even kernels, one group with kernels beyond the
# dense path's range or 8 output channels, a kernel of extent 1 along D (odd
# residues receive no tap: bias only), and a case with several units per
# persistent CTA (both accumulator sets, ring wrap-around).
TC3DG = [
    dict(N=1, C_in=32, C_out=32, G=4, L=[3, 5, 8], K=[3, 5, 7], P=[1, 2, 3], OP=[1, 1, 1]),
    dict(N=2, C_in=32, C_out=32, G=2, L=[2, 4, 8], K=[2, 4, 6], P=[0, 1, 2], OP=[0, 1, 0]),
    dict(N=1, C_in=32, C_out=16, G=1, L=[2, 3, 4], K=[5, 5, 5], P=[2, 2, 2], OP=[1, 1, 1]),
    dict(N=1, C_in=32, C_out=8, G=1, L=[3, 3, 4], K=[3, 3, 3], P=[1, 1, 1], OP=[1, 1, 1]),
    dict(N=1, C_in=32, C_out=32, G=4, L=[3, 4, 6], K=[1, 3, 5], P=[0, 1, 2], OP=[0, 0, 1]),
    dict(N=8, C_in=32, C_out=32, G=4, L=[16, 16, 16], K=[3, 5, 7], P=[1, 2, 3], OP=[1, 1, 1]),
]


@pytest.mark.parametrize("k", range(len(TC3DG)))
def test_fp32_3d_grouped_tensor_core_shapes(k):
    c = dict(nd=3, S=[2, 2, 2], DL=[1, 1, 1], bias=bool(k % 2 == 0), add=False, dtype="f32", **TC3DG[k])
    assert path_of(c) == "tc3dg_tf32x3", (c, path_of(c))
    t = cc.make_inputs(c, seed=900 + k)
    y = cc.run_gpu(c, t).cpu().numpy()
    cc.assert_close(y, cc.run_oracle(c, t), "f32", "tc3dg case %d %r" % (k, c))
    if k < 3:
        # small integers are exact in the tf32 part, so the split and the fp32
        # accumulation reproduce the oracle bit for bit
        ti = cc.make_inputs(c, seed=950 + k, int_range=3)
        yi = cc.run_gpu(c, ti).cpu().numpy()
        assert np.array_equal(yi.astype(np.float64), cc.run_oracle(c, ti)), "tc3dg integer case %d" % k


# ConvTranspose2d: the 3-D operator with a unit D dimension, through the same
# kernels.  FP32 dense shapes for the tensor-core path (plain and fused): C_in
# 32 and 64, C_out 16..128, kernel extents 2..4 mixed across H and W, padding
# even and odd, an odd H output (ragged qh block), W outputs from 8 to 256
# (tiles of 16 qh rows down to one qh row of 128 qw) and a case with several
# units per persistent CTA.
TC2D = [
    dict(N=2, C_in=32, C_out=64, L=[8, 16], K=[4, 4], P=[1, 1], OP=[0, 0]),
    dict(N=1, C_in=64, C_out=32, L=[5, 8], K=[3, 3], P=[1, 1], OP=[1, 1]),
    dict(N=1, C_in=32, C_out=16, L=[3, 4], K=[2, 3], P=[0, 1], OP=[1, 1]),
    dict(N=1, C_in=32, C_out=128, L=[4, 64], K=[4, 4], P=[1, 1], OP=[0, 0]),
    dict(N=3, C_in=32, C_out=48, L=[7, 128], K=[3, 3], P=[1, 1], OP=[1, 1]),
    dict(N=8, C_in=32, C_out=32, L=[32, 32], K=[4, 4], P=[1, 1], OP=[0, 0]),
]


@pytest.mark.parametrize("add", [False, True])
@pytest.mark.parametrize("k", range(len(TC2D)))
def test_fp32_2d_tensor_core_shapes(k, add):
    c = dict(nd=2, G=1, S=[2, 2], DL=[1, 1], bias=bool(k % 2 == 0), add=add, dtype="f32", **TC2D[k])
    assert path_of(c) == "tc3d_tf32x3", (c, path_of(c))
    t = cc.make_inputs(c, seed=1000 + k + (50 if add else 0))
    y = cc.run_gpu(c, t).cpu().numpy()
    cc.assert_close(y, cc.run_oracle(c, t), "f32", "2-D tc case %d add=%s %r" % (k, add, c))
    if k < 2 and not add:
        ti = cc.make_inputs(c, seed=1100 + k, int_range=3)
        yi = cc.run_gpu(c, ti).cpu().numpy()
        assert np.array_equal(yi.astype(np.float64), cc.run_oracle(c, ti)), "2-D tc integer case %d" % k


# Grouped ConvTranspose2d (32 input channels in 4, 2 or 1 groups) on the
# grouped tensor-core path: the unit D dimension planned as a stride-2 D of
# extent 1 (its odd residue has no plane); asymmetric kernels, and a case with
# several units per persistent CTA.
TC2DG = [
    dict(N=2, C_in=32, C_out=32, G=4, L=[16, 16], K=[5, 7], P=[2, 3], OP=[1, 1]),
    dict(N=1, C_in=32, C_out=32, G=2, L=[8, 12], K=[4, 6], P=[1, 2], OP=[0, 0]),
    dict(N=4, C_in=32, C_out=8, G=1, L=[32, 32], K=[3, 3], P=[1, 1], OP=[1, 1]),
]


@pytest.mark.parametrize("k", range(len(TC2DG)))
def test_fp32_2d_grouped_tensor_core_shapes(k):
    c = dict(nd=2, S=[2, 2], DL=[1, 1], bias=bool(k % 2 == 0), add=False, dtype="f32", **TC2DG[k])
    assert path_of(c) == "tc3dg_tf32x3", (c, path_of(c))
    t = cc.make_inputs(c, seed=1700 + k)
    y = cc.run_gpu(c, t).cpu().numpy()
    cc.assert_close(y, cc.run_oracle(c, t), "f32", "2-D grouped case %d %r" % (k, c))
    if k == 0:
        ti = cc.make_inputs(c, seed=1750, int_range=3)
        yi = cc.run_gpu(c, ti).cpu().numpy()
        assert np.array_equal(yi.astype(np.float64), cc.run_oracle(c, ti)), "2-D grouped integer case"


# bf16 ConvTranspose2d on the bf16 tensor-core path: kernel extents 4 and 8
# (the weight repack moves 16-byte pieces, so kH*kW must be a multiple of 8),
# C_out 16..256, odd H output, padding 0..3, several tiles per CTA, and 160
# tile pairs (on 152 SMs the last round's 8 pairs run as 16 single tiles).
UMMA2D = [
    dict(N=1, C_in=64, C_out=64, L=[8, 16], K=[4, 4], P=[1, 1], OP=[0, 0]),
    dict(N=2, C_in=128, C_out=128, L=[5, 12], K=[4, 4], P=[1, 1], OP=[1, 0]),
    dict(N=1, C_in=64, C_out=256, L=[4, 8], K=[4, 4], P=[1, 1], OP=[0, 0]),
    dict(N=1, C_in=64, C_out=32, L=[3, 4], K=[8, 8], P=[3, 3], OP=[0, 0]),
    dict(N=4, C_in=64, C_out=16, L=[32, 32], K=[4, 4], P=[0, 0], OP=[0, 0]),
    dict(N=20, C_in=64, C_out=32, L=[32, 32], K=[4, 4], P=[1, 1], OP=[0, 0]),
]


@pytest.mark.parametrize("k", range(len(UMMA2D)))
def test_bf16_2d_tensor_core_shapes(k):
    c = dict(nd=2, G=1, S=[2, 2], DL=[1, 1], bias=bool(k % 2 == 0), add=False, dtype="bf16",
             **UMMA2D[k])
    assert path_of(c) == "umma_bf16", (c, path_of(c))
    t = cc.make_inputs(c, seed=1200 + k)
    y = cc.run_gpu(c, t).cpu().numpy()
    cc.assert_close(y, cc.run_oracle(c, t), "bf16", "2-D umma case %d %r" % (k, c))
    if k == 0:
        ti = cc.make_inputs(c, seed=1250, int_range=3)
        yi = cc.run_gpu(c, ti).cpu().numpy()
        assert np.array_equal(yi.astype(np.float64), cc.run_oracle(c, ti)), "2-D umma integer case"


# 2-D shapes outside the tuned kernels' range take the generic kernel: groups,
# stride 3 and 1, dilation, a bf16 kernel of extent 2, the fused epilogue on
# a grouped layer.
GEN2D = [
    dict(N=2, C_in=6, C_out=4, G=2, L=[5, 7], K=[3, 2], S=[2, 3], P=[1, 0], OP=[1, 2], DL=[1, 1],
         dtype="f32", add=False),
    dict(N=1, C_in=4, C_out=8, G=1, L=[6, 5], K=[3, 3], S=[1, 2], P=[2, 1], OP=[0, 1], DL=[2, 1],
         dtype="f32", add=False),
    dict(N=1, C_in=64, C_out=32, G=1, L=[4, 8], K=[2, 2], S=[2, 2], P=[0, 0], OP=[0, 0], DL=[1, 1],
         dtype="bf16", add=False),
    dict(N=2, C_in=8, C_out=8, G=4, L=[4, 6], K=[3, 3], S=[2, 2], P=[1, 1], OP=[1, 1], DL=[1, 1],
         dtype="f32", add=True),
]


@pytest.mark.parametrize("k", range(len(GEN2D)))
def test_2d_generic_shapes(k):
    c = dict(nd=2, bias=True, **GEN2D[k])
    assert path_of(c) == "gather_generic", (c, path_of(c))
    t = cc.make_inputs(c, seed=1300 + k)
    y = cc.run_gpu(c, t).cpu().numpy()
    cc.assert_close(y, cc.run_oracle(c, t), c["dtype"], "2-D generic case %d %r" % (k, c))


# Accuracy of the splits of the FP32 tensor-core kernels, measured against
# S = sum |x| |w| of each output (the oracle run on |x|, |w| without bias):
#  * tf32x3 (CT_F32, the default): every product is x_t w_t + x_t w_l + x_l w_t
#    with the dropped terms below 3 x 2^-22 |x||w|; with the fp32 accumulation
#    an output must stay within 2^-19 S -- and within a small factor of the
#    error the FP32 FFMA kernel (plain fp32 multiply-adds) makes on the same
#    inputs, i.e. as accurate as fp32 arithmetic;
#  * bf16x2 (CT_F32_BF16X2, opt-in): every product is (x_hi + x_lo)(w_hi +
#    w_lo) with each part's remainder below 2^-17, so an output stays within a
#    small multiple of 2^-16 S.
SPLIT_CASES = ["convT3d_add_hswish", "convT3d_grouped", "convT2d_f32"]


def _split_ratio(c, t, split2):
    y = cc.run_gpu(dict(c, split2=split2), t).cpu().numpy().astype(np.float64)
    ref = cc.run_oracle(c, t)
    mag = dict(t, x=np.abs(t["x"]), w=np.abs(t["w"]), bias=None)
    S = cc.run_oracle(dict(c, bias=False), mag)
    return float((np.abs(y - ref) / (S + 1e-30)).max())


@pytest.mark.parametrize("k", range(len(SPLIT_CASES)))
def test_fp32_split_error_bound(k):
    import transposed_convolution_convtranspose_gb300 as ct
    name = SPLIT_CASES[k]
    c = cc.case_from_config(name, N=1)
    c["add"] = False                      # the bound concerns the convolution itself
    t = cc.make_inputs(c, seed=1400 + k, bound=workloads.CONFIGS[name]["bound"])
    assert path_of(c) in ("tc3d_tf32x3", "tc3dg_tf32x3"), path_of(c)
    r3 = _split_ratio(c, t, False)
    assert path_of(dict(c, split2=True)) in ("tc3d_bf16x2", "tc3dg_bf16x2"), path_of(dict(c, split2=True))
    r2 = _split_ratio(c, t, True)
    ct.ct_set_path_override(2)            # the FFMA kernels: plain fp32 arithmetic
    try:
        assert path_of(c) in ("phase3d_f32", "gather_generic"), path_of(c)
        rf = _split_ratio(c, t, False)
    finally:
        ct.ct_set_path_override(0)
    print("%s: max |err| / sum|x||w|: tf32x3 2^%.1f, fp32 FFMA 2^%.1f, bf16x2 2^%.1f"
          % (name, np.log2(max(r3, 1e-300)), np.log2(max(rf, 1e-300)), np.log2(max(r2, 1e-300))))
    assert r3 < 2.0 ** -19, (name, r3)
    assert r3 < 4.0 * rf + 2.0 ** -22, (name, r3, rf)
    assert r2 < 2.0 ** -14, (name, r2)


# The opt-in two-term bf16 split (CT_F32_BF16X2) on the dense, grouped and
# 2-D FP32 tensor-core shapes: within the FP32 tolerance of the oracle, and
# exact on small integers (each integer in [-3, 3] is its own bf16 hi part).
SPLIT2_CASES = [
    dict(nd=3, G=1, S=[2, 2, 2], DL=[1, 1, 1], add=True, **TC3D[0]),
    dict(nd=3, G=1, S=[2, 2, 2], DL=[1, 1, 1], add=False, **TC3D[1]),
    dict(nd=3, S=[2, 2, 2], DL=[1, 1, 1], add=False, **TC3DG[0]),
    dict(nd=2, G=1, S=[2, 2], DL=[1, 1], add=False, **TC2D[1]),
    dict(nd=2, S=[2, 2], DL=[1, 1], add=False, **TC2DG[1]),
]


@pytest.mark.parametrize("k", range(len(SPLIT2_CASES)))
def test_fp32_bf16x2_opt_in_shapes(k):
    c = dict(SPLIT2_CASES[k], bias=True, dtype="f32", split2=True)
    want = "tc3dg_bf16x2" if c["G"] > 1 else "tc3d_bf16x2"
    assert path_of(c) == want, (c, path_of(c))
    t = cc.make_inputs(c, seed=1450 + k)
    cc.assert_close(cc.run_gpu(c, t).cpu().numpy(), cc.run_oracle(c, t), "f32", "bf16x2 case %d %r" % (k, c))
    if not c["add"]:
        ti = cc.make_inputs(c, seed=1470 + k, int_range=3)
        yi = cc.run_gpu(c, ti).cpu().numpy()
        assert np.array_equal(yi.astype(np.float64), cc.run_oracle(c, ti)), "bf16x2 integer case %d" % k


# Shapes with s > (k - 1) d: the stride phases do not overlap, every output
# receives at most one tap per dimension (some none), and a scatter
# formulation would write disjoint outputs.  The gather kernels compute each
# output once in any case; integer inputs make every result exact.  Covers the
# FP32 and bf16 3-D tensor-core kernels (s = 2, k = 2) and the generic kernel
# (s = 3, 4; 1-D, 2-D, 3-D, groups).
DISJOINT = [
    dict(nd=1, N=2, C_in=8, C_out=16, G=1, L=[300], K=[2], S=[3], P=[0], OP=[2], DL=[1], dtype="f32"),
    dict(nd=1, N=1, C_in=4, C_out=4, G=2, L=[77], K=[3], S=[4], P=[1], OP=[3], DL=[1], dtype="f32"),
    dict(nd=3, N=1, C_in=32, C_out=32, G=1, L=[4, 6, 8], K=[2, 2, 2], S=[2, 2, 2], P=[0, 0, 0],
         OP=[1, 0, 0], DL=[1, 1, 1], dtype="f32"),
    dict(nd=3, N=1, C_in=64, C_out=32, G=1, L=[3, 4, 8], K=[2, 2, 2], S=[2, 2, 2], P=[0, 0, 0],
         OP=[0, 0, 0], DL=[1, 1, 1], dtype="bf16"),
    dict(nd=3, N=1, C_in=6, C_out=9, G=3, L=[3, 4, 5], K=[3, 2, 3], S=[3, 3, 4], P=[1, 0, 2],
         OP=[2, 1, 0], DL=[1, 1, 1], dtype="f32"),
    dict(nd=2, N=2, C_in=5, C_out=7, G=1, L=[6, 9], K=[2, 3], S=[3, 4], P=[0, 1], OP=[1, 3], DL=[1, 1],
         dtype="f32"),
]


@pytest.mark.parametrize("k", range(len(DISJOINT)))
def test_disjoint_phase_shapes_exact(k):
    c = dict(DISJOINT[k], bias=True, add=False)
    if k in (2, 3):
        assert path_of(c) in ("tc3d_tf32x3", "umma_bf16"), path_of(c)
    t = cc.make_inputs(c, seed=1500 + k, int_range=3)
    y = cc.run_gpu(c, t).cpu().numpy()
    ref = cc.run_oracle(c, t)
    assert y.shape == ref.shape
    assert np.array_equal(y.astype(np.float64), ref), "disjoint case %d (%s) not exact" % (k, path_of(c))


# The FP32 tensor-core path for strides 1 to 4 and any dilation (one residue
# pair per unit, the W phases as accumulators): stride 3 with k = s (every
# output one tap, disjoint phases), stride 3 with overlapping k = 5, stride 4
# with k = 2 (residues without a tap: bias only), mixed strides (1, 3, 2) with
# dilation 2, stride 2 with kernel 5, stride 1, 2-D and long 1-D shapes (W
# split into several unit blocks), and the fused epilogue with several W
# blocks.  Random inputs within the FP32 tolerance; integer inputs exact.
TC3S = [
    dict(nd=3, N=1, C_in=32, C_out=32, L=[3, 4, 4], K=[3, 3, 3], S=[3, 3, 3], P=[0, 0, 0], OP=[0, 0, 0],
         DL=[1, 1, 1], add=False),
    dict(nd=3, N=1, C_in=32, C_out=16, L=[2, 3, 4], K=[5, 5, 5], S=[3, 3, 3], P=[2, 2, 2], OP=[1, 1, 2],
         DL=[1, 1, 1], add=True),
    dict(nd=3, N=2, C_in=32, C_out=32, L=[2, 3, 4], K=[2, 2, 2], S=[4, 4, 4], P=[0, 0, 0], OP=[1, 0, 2],
         DL=[1, 1, 1], add=False),
    dict(nd=3, N=1, C_in=64, C_out=48, L=[3, 4, 6], K=[2, 3, 3], S=[1, 3, 2], P=[0, 1, 1], OP=[0, 2, 1],
         DL=[1, 2, 1], add=False),
    dict(nd=3, N=1, C_in=64, C_out=32, L=[3, 4, 8], K=[5, 5, 5], S=[2, 2, 2], P=[2, 2, 2], OP=[1, 1, 1],
         DL=[1, 1, 1], add=True),
    dict(nd=2, N=2, C_in=32, C_out=64, L=[5, 8], K=[3, 3], S=[3, 3], P=[1, 1], OP=[0, 2], DL=[1, 1], add=False),
    dict(nd=1, N=2, C_in=32, C_out=32, L=[300], K=[3], S=[4], P=[0], OP=[1], DL=[1], add=False),
    dict(nd=2, N=1, C_in=32, C_out=32, L=[6, 12], K=[3, 3], S=[1, 1], P=[1, 1], OP=[0, 0], DL=[1, 1], add=False),
    dict(nd=3, N=1, C_in=32, C_out=16, L=[2, 2, 40], K=[3, 3, 3], S=[3, 3, 3], P=[0, 0, 0], OP=[0, 0, 0],
         DL=[1, 1, 1], add=True),
    dict(nd=3, N=3, C_in=32, C_out=128, L=[4, 4, 4], K=[4, 4, 4], S=[4, 4, 4], P=[0, 0, 0], OP=[0, 0, 0],
         DL=[1, 1, 1], add=False),
    # outputs shorter than the stride: one output row at H stride 3 (H residues 1
    # and 2 have no rows), two output planes at D stride 4 (D residues 2, 3 none)
    dict(nd=3, N=2, C_in=32, C_out=16, L=[1, 1, 8], K=[2, 1, 3], S=[4, 3, 3], P=[0, 0, 1], OP=[0, 0, 2],
         DL=[1, 1, 1], add=True),
]


@pytest.mark.parametrize("k", range(len(TC3S)))
def test_fp32_any_stride_tensor_core_shapes(k):
    c = dict(G=1, bias=bool(k % 2 == 0), dtype="f32", **TC3S[k])
    assert path_of(c) == "tc3s_tf32x3", (c, path_of(c))
    t = cc.make_inputs(c, seed=1800 + k)
    y = cc.run_gpu(c, t).cpu().numpy()
    cc.assert_close(y, cc.run_oracle(c, t), "f32", "tc3s case %d %r" % (k, c))
    if not c["add"]:
        ti = cc.make_inputs(c, seed=1850 + k, int_range=3)
        yi = cc.run_gpu(c, ti).cpu().numpy()
        assert np.array_equal(yi.astype(np.float64), cc.run_oracle(c, ti)), "tc3s integer case %d" % k
    if k in (0, 2):
        c2 = dict(c, split2=True)
        assert path_of(c2) == "tc3s_bf16x2", path_of(c2)
        cc.assert_close(cc.run_gpu(c2, t).cpu().numpy(), cc.run_oracle(c, t), "f32", "tc3s bf16x2 case %d" % k)


# Channels-last layouts (x (N, spatial..., C_in), y and add (N, spatial...,
# C_out)): the inputs are the same draws moved to channels-last on the device,
# the result is moved back and compared with the oracle.  bf16 shapes of the
# bf16 tensor-core kernel (3-D and 2-D: x read in place), dense FP32 shapes of
# the FP32 tensor-core kernel (3-D and 2-D, plain and fused, odd D and H
# outputs), and the generic kernel for groups, 1-D, other strides and the
# bf16 fused epilogue (fused cases also in place).
CL = [
    dict(nd=3, N=1, C_in=64, C_out=16, G=1, L=[2, 3, 8], K=[4] * 3, S=[2] * 3, P=[1] * 3, OP=[1, 0, 0],
         DL=[1] * 3, dtype="bf16", add=False, path="umma_bf16"),
    dict(nd=3, N=2, C_in=128, C_out=128, G=1, L=[2, 4, 16], K=[4] * 3, S=[2] * 3, P=[1] * 3,
         OP=[0] * 3, DL=[1] * 3, dtype="bf16", add=False, path="umma_bf16"),
    dict(nd=3, N=1, C_in=64, C_out=256, G=1, L=[2, 2, 8], K=[4] * 3, S=[2] * 3, P=[1] * 3,
         OP=[1, 1, 0], DL=[1] * 3, dtype="bf16", add=False, path="umma_bf16"),
    dict(nd=3, N=1, C_in=64, C_out=48, G=1, L=[2, 2, 9], K=[2] * 3, S=[2] * 3, P=[1] * 3, OP=[0] * 3,
         DL=[1] * 3, dtype="bf16", add=False, path="umma_bf16"),
    dict(nd=2, N=2, C_in=128, C_out=128, G=1, L=[5, 12], K=[4, 4], S=[2, 2], P=[1, 1], OP=[1, 0],
         DL=[1, 1], dtype="bf16", add=False, path="umma_bf16"),
    dict(nd=3, N=1, C_in=32, C_out=64, G=1, L=[3, 4, 8], K=[3] * 3, S=[2] * 3, P=[1] * 3, OP=[1] * 3,
         DL=[1] * 3, dtype="f32", add=True, path="tc3d_tf32x3"),
    dict(nd=3, N=2, C_in=64, C_out=32, G=1, L=[2, 3, 4], K=[4] * 3, S=[2] * 3, P=[1] * 3, OP=[0] * 3,
         DL=[1] * 3, dtype="f32", add=False, path="tc3d_tf32x3"),
    dict(nd=2, N=2, C_in=32, C_out=48, G=1, L=[7, 64], K=[3, 3], S=[2, 2], P=[1, 1], OP=[1, 1],
         DL=[1, 1], dtype="f32", add=False, path="tc3d_tf32x3"),
    dict(nd=2, N=1, C_in=32, C_out=16, G=1, L=[3, 4], K=[2, 3], S=[2, 2], P=[0, 1], OP=[1, 1],
         DL=[1, 1], dtype="f32", add=True, path="tc3d_tf32x3"),
    dict(nd=3, N=2, C_in=6, C_out=4, G=2, L=[3, 4, 5], K=[2, 3, 4], S=[3, 1, 2], P=[1, 0, 2], OP=[2, 0, 1],
         DL=[1, 2, 1], dtype="f32", add=False, path="gather_generic"),
    dict(nd=2, N=2, C_in=8, C_out=8, G=4, L=[4, 6], K=[3, 3], S=[2, 2], P=[1, 1], OP=[1, 1], DL=[1, 1],
         dtype="f32", add=False, path="gather_generic"),
    dict(nd=1, N=2, C_in=32, C_out=64, G=1, L=[777], K=[3], S=[2], P=[1], OP=[0], DL=[2], dtype="f32",
         add=False, path="gather_generic"),
    dict(nd=3, N=1, C_in=64, C_out=32, G=1, L=[3, 3, 4], K=[3] * 3, S=[2] * 3, P=[1] * 3, OP=[1] * 3,
         DL=[1] * 3, dtype="bf16", add=True, path="gather_generic"),
]


def _path_cl(c):
    import transposed_convolution_convtranspose_gb300 as ct
    dt = ct.CT_BF16 if c["dtype"] == "bf16" else ct.CT_F32
    return ct.ct_path_cl(c["nd"], c["N"], c["C_in"], c["C_out"], c["L"], c["K"], c["G"], c["S"], c["P"],
                         c["OP"], c["DL"], dt, c["add"])


def _run_cl(c, t, inplace=False):
    import transposed_convolution_convtranspose_gb300 as ct
    x, w, b, a = cc.to_device(t, c, "cuda:0")
    xcl = x.movedim(1, -1).contiguous()
    acl = a.movedim(1, -1).contiguous() if a is not None else None
    kw = cc.kwargs(c)
    if c["nd"] == 1:
        kw = {k: (v if k == "groups" else (v,)) for k, v in kw.items()}
    y = ct.conv_transpose_cl(xcl, w, b, acl, out=acl if inplace else None, **kw)
    return y.movedim(-1, 1).contiguous().cpu().numpy()


@pytest.mark.parametrize("k", range(len(CL)))
def test_channels_last_shapes(k):
    c = dict(CL[k], bias=bool(k % 2 == 0))
    want = c.pop("path")
    assert _path_cl(c) == want, (c, _path_cl(c))
    t = cc.make_inputs(c, seed=1600 + k)
    ref = cc.run_oracle(c, t)
    cc.assert_close(_run_cl(c, t), ref, c["dtype"], "channels-last case %d %r" % (k, c))
    if c["add"]:
        cc.assert_close(_run_cl(c, t, inplace=True), ref, c["dtype"], "channels-last in place %d" % k)
    if k in (1, 6, 9):
        ti = cc.make_inputs(c, seed=1650 + k, int_range=3)
        assert np.array_equal(_run_cl(c, ti).astype(np.float64), cc.run_oracle(c, ti)), "cl integer %d" % k


def test_fp32_3d_without_workspace_takes_ffma():
    """A call given no workspace runs the FFMA kernel, with the same result."""
    import torch
    import transposed_convolution_convtranspose_gb300 as ct
    c = dict(nd=3, G=1, S=[2, 2, 2], DL=[1, 1, 1], bias=True, add=True, dtype="f32", **TC3D[0])
    t = cc.make_inputs(c, seed=870)
    x, w, b, a = cc.to_device(t, c, "cuda:0")
    y = torch.empty(cc.out_shape(c), device="cuda:0")
    ct.ct_forward_3d_add_hswish(x, w, b, a, y, c["N"], c["C_in"], c["C_out"], c["L"], c["K"], 1,
                                c["S"], c["P"], c["OP"], c["DL"], ct.CT_F32, None, 0,
                                torch.cuda.current_stream())
    ref = cc.run_oracle(c, t)
    cc.assert_close(y.cpu().numpy(), ref, "f32", "fused without workspace")
    ct.ct_set_path_override(2)
    try:
        assert path_of(c) == "phase3d_f32"
        y2 = cc.run_gpu(c, t).cpu().numpy()
    finally:
        ct.ct_set_path_override(0)
    cc.assert_close(y2, ref, "f32", "fused, FFMA kernel forced")


EDGE = [
    # 1-D: single input, unit kernel, stride larger than kernel (empty phases),
    # large dilation, maximal output_padding, depthwise groups, ragged lengths
    dict(nd=1, N=1, C_in=1, C_out=1, G=1, L=[1], K=[1], S=[1], P=[0], OP=[0], DL=[1]),
    dict(nd=1, N=3, C_in=2, C_out=4, G=1, L=[7], K=[2], S=[5], P=[0], OP=[4], DL=[1]),
    dict(nd=1, N=2, C_in=6, C_out=6, G=6, L=[33], K=[3], S=[2], P=[1], OP=[1], DL=[1]),
    dict(nd=1, N=1, C_in=4, C_out=8, G=2, L=[50], K=[4], S=[3], P=[2], OP=[3], DL=[4]),
    dict(nd=1, N=2, C_in=32, C_out=64, G=1, L=[4999], K=[3], S=[2], P=[1], OP=[0], DL=[2]),
    dict(nd=1, N=1, C_in=32, C_out=64, G=1, L=[1], K=[3], S=[2], P=[1], OP=[0], DL=[2]),
    dict(nd=1, N=1, C_in=32, C_out=64, G=1, L=[2], K=[3], S=[2], P=[1], OP=[1], DL=[2]),
    # 3-D: unit spatial dims, asymmetric everything, kernel 1, ragged W
    dict(nd=3, N=1, C_in=2, C_out=3, G=1, L=[1, 1, 1], K=[1, 1, 1], S=[1, 1, 1], P=[0, 0, 0],
         OP=[0, 0, 0], DL=[1, 1, 1]),
    dict(nd=3, N=2, C_in=4, C_out=6, G=2, L=[3, 4, 5], K=[2, 3, 4], S=[3, 1, 2], P=[1, 0, 2],
         OP=[2, 0, 1], DL=[1, 2, 1]),
    dict(nd=3, N=1, C_in=32, C_out=32, G=4, L=[5, 7, 9], K=[3, 5, 7], S=[2, 2, 2], P=[1, 2, 3],
         OP=[1, 1, 1], DL=[1, 1, 1]),
    dict(nd=3, N=1, C_in=32, C_out=64, G=1, L=[3, 5, 7], K=[3, 3, 3], S=[2, 2, 2], P=[1, 1, 1],
         OP=[1, 1, 1], DL=[1, 1, 1]),
    dict(nd=3, N=1, C_in=32, C_out=64, G=1, L=[1, 1, 1], K=[3, 3, 3], S=[2, 2, 2], P=[1, 1, 1],
         OP=[1, 1, 1], DL=[1, 1, 1]),
]


@pytest.mark.parametrize("k", range(len(EDGE)))
@pytest.mark.parametrize("bias", [False, True])
def test_edge_cases(k, bias):
    c = dict(EDGE[k], bias=bias, add=False, dtype="f32")
    t = cc.make_inputs(c, seed=500 + k)
    y = cc.run_gpu(c, t).cpu().numpy()
    cc.assert_close(y, cc.run_oracle(c, t), "f32", "edge %d (%s)" % (k, path_of(c)))


def test_fused_in_place_and_edges():
    for k, shape in enumerate([[2, 3, 4], [1, 1, 1], [5, 3, 16]]):
        c = dict(nd=3, N=2, C_in=32, C_out=64, G=1, L=shape, K=[3, 3, 3], S=[2, 2, 2],
                 P=[1, 1, 1], OP=[1, 1, 1], DL=[1, 1, 1], bias=True, add=True, dtype="f32")
        t = cc.make_inputs(c, seed=600 + k)
        ref = cc.run_oracle(c, t)
        y = cc.run_gpu(c, t, inplace_add=True).cpu().numpy()
        cc.assert_close(y, ref, "f32", "fused in place %r (%s)" % (shape, path_of(c)))


def test_empty_batch_is_a_no_op():
    import torch
    import transposed_convolution_convtranspose_gb300 as ct
    x = torch.zeros((0, 4, 16), device="cuda")
    w = torch.ones((4, 8, 3), device="cuda")
    y = torch.full((0, 8, 33), 5.0, device="cuda")
    ct.ct_forward_1d(x, w, None, y, 0, 4, 8, 16, 3, 1, 2, 1, 0, 2, ct.CT_F32)
    ct.ct_last_device_error(torch.cuda.current_stream())


def test_repeat_is_deterministic():
    name = "convT3d_add_hswish"
    c = cc.case_from_config(name, N=2)
    t = cc.make_inputs(c, seed=700)
    y1 = cc.run_gpu(c, t)
    y2 = cc.run_gpu(c, t)
    import torch
    assert torch.equal(y1, y2)


def test_grouped_reproducible_when_asked():
    """ct_set_deterministic(1): the grouped FP32 tensor-core path issues each
    group's MMAs from one thread, so repeated calls give identical bits (by
    default two threads per group accumulate in no fixed order); both within
    the path's tolerance of the oracle."""
    import torch
    import transposed_convolution_convtranspose_gb300 as ct
    c = cc.case_from_config("convT3d_grouped", N=2)
    assert path_of(c) == "tc3dg_tf32x3"
    t = cc.make_inputs(c, seed=710)
    ref = cc.run_oracle(c, t)
    ct.ct_set_deterministic(1)
    try:
        y1 = cc.run_gpu(c, t)
        y2 = cc.run_gpu(c, t)
    finally:
        ct.ct_set_deterministic(0)
    assert torch.equal(y1, y2)
    cc.assert_close(y1.cpu().numpy(), ref, "f32", "grouped, reproducible order")
    y3 = cc.run_gpu(c, t)
    cc.assert_close(y3.cpu().numpy(), ref, "f32", "grouped, two issuers per group")


TC1D = [
    # (C_in, C_out, L_in, k, s, p, op, d): C_in = 32 and d a multiple of s take
    # the FP32 tensor-core path; ragged lengths end tiles mid-way
    (32, 64, 131072 // 64, 3, 2, 1, 0, 2),
    (32, 64, 1000, 3, 2, 1, 1, 2),
    (32, 16, 516, 3, 2, 0, 0, 2),
    (32, 32, 256, 4, 2, 2, 1, 2),
    (32, 48, 300, 2, 2, 1, 0, 4),
    (32, 64, 128, 3, 1, 1, 0, 1),
    (32, 64, 131, 3, 2, 1, 0, 2),
    (32, 64, 260, 1, 2, 0, 1, 2),
    (32, 32, 4, 3, 2, 1, 0, 2),
    (32, 64, 1, 3, 2, 1, 0, 2),
]


@pytest.mark.parametrize("mode", [0, 2])
@pytest.mark.parametrize("k", range(len(TC1D)))
def test_fp32_1d_tensor_core_and_ffma_paths(k, mode):
    """The FP32 1-D shapes the tensor-core path takes, through that path
    (mode 0) and through the FFMA phase kernel (mode 2), against the oracle."""
    import transposed_convolution_convtranspose_gb300 as ct
    C_in, C_out, L, kk, s, p, op, d = TC1D[k]
    c = dict(nd=1, N=2, C_in=C_in, C_out=C_out, G=1, L=[L], K=[kk], S=[s], P=[p], OP=[op],
             DL=[d], bias=bool(k % 2), add=False, dtype="f32")
    ct.ct_set_path_override(mode)
    try:
        path = path_of(c)
        if mode == 0 and L % 4 == 0:
            assert path == "tc1d_tf32x3", path
        t = cc.make_inputs(c, seed=800 + k)
        y = cc.run_gpu(c, t).cpu().numpy()
        cc.assert_close(y, cc.run_oracle(c, t), "f32", "1-D case %r (%s)" % (TC1D[k], path))
        ti = cc.make_inputs(c, seed=850 + k, int_range=3)
        yi = cc.run_gpu(c, ti).cpu().numpy()
        assert np.array_equal(yi.astype(np.float64), cc.run_oracle(c, ti)), \
            "integer inputs not exact for %r (%s)" % (TC1D[k], path)
    finally:
        ct.ct_set_path_override(0)


# A seeded sweep of the tensor-core planners: per family, random draws within
# the family's range (channel counts, kernel extents, padding, output padding,
# spatial extents with ragged tiles, batch, fused epilogue, channels-last
# layout), kept when the host path query names the family's kernel (with
# split2, the opt-in bf16 pair's).  Inputs stay small enough for the oracle to
# finish each case in well under a second.
def _tc_sweep(family, n, seed, split2=False):
    rng = np.random.default_rng(seed)
    pick = lambda seq: seq[int(rng.integers(0, len(seq)))]
    out = []
    for _ in range(5000):
        if len(out) == n:
            break
        layout, add, G, dtype = "cf", False, 1, "f32"
        if family == "tc3d":
            nd = pick([2, 3])
            C_in, C_out = pick([32, 64]), pick([16, 32, 48, 64, 96, 128])
            K = [int(rng.integers(2, 5)) for _ in range(nd)]
            S, DL = [2] * nd, [1] * nd
            L = ([int(rng.integers(1, 5))] if nd == 3 else []) + [int(rng.integers(1, 8)), pick([2, 4, 8, 16, 32])]
            add, layout = bool(rng.integers(0, 2)), pick(["cf", "cf", "cl"])
            want = "tc3d_tf32x3"
        elif family == "tc3dg":
            nd = pick([2, 3])
            G = pick([1, 2, 4])
            C_in, C_out = 32, G * pick([8, 16])
            K = [int(rng.integers(1, 8)) for _ in range(nd)]
            S, DL = [2] * nd, [1] * nd
            L = ([int(rng.integers(1, 5))] if nd == 3 else []) + [int(rng.integers(1, 17)), int(rng.integers(2, 40))]
            want = "tc3dg_tf32x3"
        elif family == "tc3s":
            nd = pick([1, 2, 3])
            C_in, C_out = pick([32, 64]), pick([16, 32, 64])
            S = [int(rng.integers(1, 5)) for _ in range(nd)]
            DL = [pick([1, 1, 2]) for _ in range(nd)]
            K = [int(rng.integers(1, 6)) for _ in range(nd)]
            L = [int(rng.integers(1, 5)) for _ in range(nd - 1)] + [int(rng.integers(2, 12))]
            if nd == 1:
                L = [int(rng.integers(8, 200))]
            add = nd > 1 and bool(rng.integers(0, 3) == 0)     # no channels-first 1-D fused call
            want = "tc3s_tf32x3"
        elif family == "tc1d":
            nd = 1
            C_in, C_out = 32, pick([16, 32, 48, 64, 96, 128])
            K, S = [int(rng.integers(1, 5))], [int(rng.integers(1, 5))]
            DL = [S[0] * pick([1, 2])]
            L = [4 * int(rng.integers(1, 600))]
            want = "tc1d_tf32x3"
        elif family == "ffma":
            # the FFMA phase kernels (path override 2 keeps the tensor cores out):
            # any 1-D shape; in 3-D the compiled kernel shapes, k 3 (W padding 1)
            # and the grouped k (3, 5, 7) (W padding 3)
            nd = pick([1, 3])
            if nd == 1:
                C_in, C_out = pick([4, 8, 16, 32]), pick([4, 8, 16, 32, 64])
                K, S, DL = [int(rng.integers(1, 5))], [int(rng.integers(1, 4))], [pick([1, 1, 2])]
                L = [int(rng.integers(2, 700))]
            else:
                grouped = bool(rng.integers(0, 2))
                G = pick([1, 2, 4]) if grouped else 1
                K = [3, 5, 7] if grouped else [3, 3, 3]
                C_in, C_out = G * pick([4, 8]), G * (8 if grouped else 16) * pick([1, 2])
                S, DL = [2] * 3, [1] * 3
                L = [int(rng.integers(1, 5)), int(rng.integers(1, 9)), 4 * int(rng.integers(1, 9))]
                add = bool(rng.integers(0, 3) == 0)
            want = "phase1d_f32" if nd == 1 else "phase3d_f32"
        elif family == "cl_generic":
            # channels-last shapes no tensor-core kernel takes: the generic kernel
            # with layout strides (groups, any stride and dilation, fused 1-D too)
            nd = pick([1, 2, 3])
            r = oracle_pins.random_case(rng, nd)
            C_in, C_out, G, K, S, DL, L = r["C_in"], r["C_out"], r["G"], r["K"], r["S"], r["DL"], r["L"]
            add, layout = bool(rng.integers(0, 2)), "cl"
            dtype = pick(["f32", "f32", "bf16"])
            if dtype == "bf16":
                add = False
            want = "gather_generic"
        else:
            nd = pick([2, 3])
            C_in, C_out = pick([64, 128]), pick([16, 32, 48, 64, 96, 128, 256])
            k = pick([2, 4]) if nd == 3 else pick([4, 4, 8])
            K, S, DL = [k] * nd, [2] * nd, [1] * nd
            L = ([int(rng.integers(1, 4))] if nd == 3 else []) + [int(rng.integers(1, 8)), int(rng.integers(2, 20))]
            dtype, layout = "bf16", pick(["cf", "cl"])
            want = "umma_bf16"
        P = [int(rng.integers(0, max(1, DL[d] * (K[d] - 1) // 2 + 1))) for d in range(nd)]
        if family == "ffma" and nd == 3:
            P[2] = (K[2] - 1) // 2                 # the compiled W padding
        OP = [int(rng.integers(0, max(S[d], DL[d]))) for d in range(nd)]
        c = dict(nd=nd, N=pick([1, 1, 2, 4]), C_in=C_in, C_out=C_out, G=G, L=L, K=K, S=S, P=P, OP=OP,
                 DL=DL, bias=bool(rng.integers(0, 2)), add=add, dtype=dtype, layout=layout, split2=split2)
        if split2:
            want = want.replace("tf32x3", "bf16x2")
        if min(cc.out_shape(c)[2:]) < 1:
            continue
        if path_of(c) == want:
            out.append(c)
    assert len(out) == n, "%s: only %d of %d shapes found" % (family, len(out), n)
    return out


@pytest.mark.parametrize("family,n,seed,split2", [
    ("tc3d", 32, 51, False), ("tc3dg", 24, 52, False), ("tc3s", 32, 53, False), ("umma", 24, 54, False),
    ("tc1d", 16, 55, False), ("ffma", 24, 56, False), ("cl_generic", 40, 57, False),
    ("tc3d", 12, 61, True), ("tc3dg", 12, 62, True), ("tc3s", 12, 63, True)])
def test_random_tensor_core_planner_sweep(family, n, seed, split2):
    import transposed_convolution_convtranspose_gb300 as ct
    ct.ct_set_path_override(2 if family == "ffma" else 0)
    try:
        _run_sweep(family, n, seed, split2)
    finally:
        ct.ct_set_path_override(0)


def _run_sweep(family, n, seed, split2):
    import torch
    import transposed_convolution_convtranspose_gb300 as ct
    for k, c in enumerate(_tc_sweep(family, n, seed, split2)):
        t = cc.make_inputs(c, seed=2000 + 100 * seed + k)
        yt = cc.run_gpu(c, t)
        y = yt.cpu().numpy()
        ref = cc.run_oracle(c, t)
        cc.assert_close(y, ref, c["dtype"], "%s sweep case %d %r" % (family, k, c))
        if c["dtype"] == "f32" and not c["add"] and family not in ("ffma", "cl_generic"):
            # the split's bound against sum |x||w| (+ |bias|, added in fp32):
            # tf32x3 at fp32 level, the bf16 pair at about 16-bit operands
            mag = dict(t, x=np.abs(t["x"]), w=np.abs(t["w"]), bias=None)
            den = cc.run_oracle(dict(c, bias=False), mag)
            if t["bias"] is not None:
                den = den + np.abs(np.asarray(t["bias"], np.float64)).reshape([1, -1] + [1] * c["nd"])
            r = float((np.abs(y.astype(np.float64) - ref) / (den + 1e-30)).max())
            assert r < (2.0 ** -14 if split2 else 2.0 ** -19), "%s sweep case %d: error 2^%.1f of sum|x||w| %r" % (
                family, k, np.log2(max(r, 1e-300)), c)
        if family == "tc3dg" and k % 2 == 0:
            # one issuing thread per group: repeated calls agree bit for bit
            ct.ct_set_deterministic(1)
            try:
                assert torch.equal(cc.run_gpu(c, t), cc.run_gpu(c, t)), "%s sweep case %d" % (family, k)
            finally:
                ct.ct_set_deterministic(0)
        if k % 3 == 0:
            # small integers: every product and partial sum is exact (the fused
            # epilogue's division by 6 is compared at fp32 tolerance)
            ti = cc.make_inputs(c, seed=3000 + 100 * seed + k, int_range=3)
            yi = cc.run_gpu(c, ti).cpu().numpy()
            ri = cc.run_oracle(c, ti)
            if c["add"]:
                cc.assert_close(yi, ri, "f32", "%s sweep integer case %d" % (family, k))
            else:
                assert np.array_equal(yi.astype(np.float64), ri), "%s sweep integer case %d %r" % (family, k, c)


def test_bounded_wait_timeout_reports_and_recovers():
    """A kernel whose bounded mbarrier wait runs out records the timeout in the
    device status word; the host reads it once, and the context stays usable."""
    import torch
    import transposed_convolution_convtranspose_gb300 as ct
    s = torch.cuda.current_stream()
    assert ct.ct_last_device_error_code(s) == ct.CT_OK        # clear any earlier state
    ct.ct_selftest_wait_timeout(1_000_000, s)                  # 1 ms limit, nothing arrives
    assert ct.ct_last_device_error_code(s) == ct.CT_ERR_DEVICE_TIMEOUT
    assert ct.ct_last_device_error_code(s) == ct.CT_OK         # read and cleared
    # the context still runs the tensor-core kernels correctly
    c = dict(nd=3, G=1, S=[2, 2, 2], DL=[1, 1, 1], bias=True, add=True, dtype="f32", **TC3D[0])
    t = cc.make_inputs(c, seed=880)
    y = cc.run_gpu(c, t).cpu().numpy()
    cc.assert_close(y, cc.run_oracle(c, t), "f32", "after a reported timeout")
    assert ct.ct_last_device_error_code(s) == ct.CT_OK


def test_timeout_is_reported_by_the_next_forward_call():
    """A timeout recorded by one launch is returned by the next forward call
    (before it launches anything), once; the call after that runs normally."""
    import torch
    import transposed_convolution_convtranspose_gb300 as ct
    s = torch.cuda.current_stream()
    assert ct.ct_last_device_error_code(s) == ct.CT_OK
    c = dict(nd=3, G=1, S=[2, 2, 2], DL=[1, 1, 1], bias=True, add=False, dtype="f32", **TC3D[1])
    t = cc.make_inputs(c, seed=890)
    ct.ct_selftest_wait_timeout(1_000_000, s)                  # 1 ms limit, nothing arrives
    torch.cuda.synchronize()                                   # the kernel has written the word
    with pytest.raises(ct.CTError) as ei:
        cc.run_gpu(c, t)
    assert ei.value.code == ct.CT_ERR_DEVICE_TIMEOUT
    y = cc.run_gpu(c, t).cpu().numpy()                         # reported once: this call runs
    cc.assert_close(y, cc.run_oracle(c, t), "f32", "after a timeout reported by a forward call")
    assert ct.ct_last_device_error_code(s) == ct.CT_OK
