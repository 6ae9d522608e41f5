"""Host-side tests of the C ABI (no GPU): the library loads, exports every
symbol include/ct.h declares, validates arguments before any launch, and its
host logic (output lengths, kernel selection, workspace sizes) is right."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as ora
import transposed_convolution_convtranspose_gb300 as ct
from transposed_convolution_convtranspose_gb300 import build as ctbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ctbuild.build()
    return ct.load()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(ct_\w+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert {"ct_forward_1d", "ct_forward_3d", "ct_forward_3d_add_hswish"} <= syms
    raw = ctypes.CDLL(ct.LIB_PATH)
    for s in sorted(syms):
        assert hasattr(raw, s), "libct.so does not export %s" % s
    assert set(ct.EXPORTED) <= syms


def test_binding_names_match_abi(lib):
    for s in declared_symbols():
        assert hasattr(ct, s), "binding lacks %s" % s


def test_out_len_matches_oracle(lib):
    rng = np.random.default_rng(0)
    for _ in range(2000):
        L, k, s, p, dl = (int(rng.integers(1, 50)), int(rng.integers(1, 8)), int(rng.integers(1, 5)),
                          int(rng.integers(0, 6)), int(rng.integers(1, 4)))
        op = int(rng.integers(0, max(s, dl)))
        want = ora.out_len(L, k, s, p, op, dl)
        got = ct.ct_out_len(L, k, s, p, op, dl)
        assert got == (want if want >= 1 else -1)
    assert ct.ct_out_len(131072, 3, 2, 1, 0, 2) == 262145
    assert ct.ct_out_len(0, 3, 2, 1, 0, 2) == -1
    assert ct.ct_out_len(4, 0, 2, 1, 0, 2) == -1


FAKE = 0x10000000   # never dereferenced: every call below fails validation first


def call1d(lib, **kw):
    a = dict(x=FAKE, w=FAKE + (1 << 24), bias=None, y=FAKE + (1 << 26), N=2, C_in=4, C_out=8,
             L_in=16, k=3, groups=1, stride=2, padding=1, output_padding=0, dilation=2,
             dtype=ct.CT_F32)
    a.update(kw)
    return lib.ct_forward_1d(a["x"], a["w"], a["bias"], a["y"], a["N"], a["C_in"], a["C_out"],
                             a["L_in"], a["k"], a["groups"], a["stride"], a["padding"],
                             a["output_padding"], a["dilation"], a["dtype"], None, 0, None)


def test_argument_errors_before_launch(lib):
    assert call1d(lib, x=None) == 1
    assert call1d(lib, y=None) == 1
    assert call1d(lib, dtype=7) == 1
    assert call1d(lib, C_in=0) == 1
    assert call1d(lib, groups=3) == 2            # 3 does not divide 4
    assert call1d(lib, k=0) == 2
    assert call1d(lib, stride=0) == 2
    assert call1d(lib, padding=-1) == 2
    assert call1d(lib, output_padding=2) == 2    # op >= max(s, dl)
    assert call1d(lib, L_in=1, k=1, padding=1) == 2   # L_out <= 0
    assert call1d(lib, x=FAKE + 2) == 3          # misaligned fp32
    assert call1d(lib, y=FAKE + 16) == 1         # y overlaps x
    assert call1d(lib, N=0) == 0                 # empty batch: valid, nothing launched


def callcl(lib, nd=3, **kw):
    a = dict(x=FAKE, w=FAKE + (1 << 24), bias=None, add=None, y=FAKE + (1 << 26), N=2, C_in=4, C_out=8,
             dtype=ct.CT_F32)
    a.update(kw)
    v = lambda t: (ctypes.c_int * max(1, nd))(*([t] * max(1, nd)))
    return lib.ct_forward_cl(nd, a["x"], a["w"], a["bias"], a["add"], a["y"], a["N"], a["C_in"], a["C_out"],
                             v(5), v(3), 1, v(2), v(1), v(0), v(1), a["dtype"], None, 0, None)


def test_channels_last_argument_errors_before_launch(lib):
    assert callcl(lib, nd=0) == 1                      # 1 to 3 spatial dimensions
    assert callcl(lib, nd=4) == 1
    assert callcl(lib, x=None) == 1
    assert callcl(lib, y=FAKE + 16) == 1               # y overlaps x
    assert callcl(lib, add=FAKE + (1 << 26) + 8) == 1  # add overlaps y without being y
    assert callcl(lib, x=FAKE + 2) == 3                # misaligned fp32
    assert callcl(lib, C_in=0) == 1
    assert callcl(lib, N=0) == 0                       # empty batch: valid, nothing launched
    assert callcl(lib, nd=1, N=0) == 0 and callcl(lib, nd=2, N=0) == 0


def test_fused_requires_add(lib):
    i3 = ct._I3
    st = lib.ct_forward_3d_add_hswish(FAKE, FAKE + (1 << 24), None, None, FAKE + (1 << 26), 1, 4,
                                      4, i3(2, 2, 2), i3(3, 3, 3), 1, i3(2, 2, 2), i3(1, 1, 1),
                                      i3(1, 1, 1), i3(1, 1, 1), ct.CT_F32, None, 0, None)
    assert st == 1


def test_status_strings(lib):
    for code in range(8):
        assert ct.ct_status_str(code).startswith(ct.CT_STATUS[code])


def test_path_selection(lib):
    # the tiny and the long 1-D workloads
    for N, L in ((2, 64), (16, 131072)):
        p = ct.ct_path_1d(N, 32 if N == 16 else 4, 64 if N == 16 else 8, L, 3, 1, 2, 1, 0, 2, ct.CT_F32)
        assert p in ("tc1d_tf32x3", "phase1d_f32", "gather_generic")
    assert ct.ct_path_1d(16, 32, 64, 131072, 3, 1, 2, 1, 0, 2, ct.CT_F32) == "tc1d_tf32x3"
    ct.ct_set_path_override(2)
    try:
        assert ct.ct_path_1d(16, 32, 64, 131072, 3, 1, 2, 1, 0, 2, ct.CT_F32) == "phase1d_f32"
    finally:
        ct.ct_set_path_override(0)
    assert ct.ct_path_1d(1, 4, 8, 0, 3, 1, 2, 1, 0, 2, ct.CT_F32) is None
    # the grouped workload: the grouped FP32 tensor-core path, the FFMA kernel
    # under override 2
    grouped = (8, 32, 32, (16, 32, 32), (3, 5, 7), 4, (2, 2, 2), (1, 2, 3), (1, 1, 1), (1, 1, 1), ct.CT_F32)
    assert ct.ct_path_3d(*grouped) == "tc3dg_tf32x3"
    ct.ct_set_path_override(2)
    try:
        assert ct.ct_path_3d(*grouped) == "phase3d_f32"
    finally:
        ct.ct_set_path_override(0)
    ct.ct_set_path_override(1)
    try:
        assert ct.ct_path_3d(8, 32, 32, (16, 32, 32), (3, 5, 7), 4, (2, 2, 2), (1, 2, 3),
                             (1, 1, 1), (1, 1, 1), ct.CT_F32) == "gather_generic"
    finally:
        ct.ct_set_path_override(0)
    # the fused workload: FP32 tensor-core path, FFMA kernel under override 2
    fused = (128, 32, 64, (16, 16, 16), (3, 3, 3), 1, (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1),
             ct.CT_F32, 1)
    assert ct.ct_path_3d(*fused) == "tc3d_tf32x3"
    ct.ct_set_path_override(2)
    try:
        assert ct.ct_path_3d(*fused) == "phase3d_f32"
    finally:
        ct.ct_set_path_override(0)


def test_path_selection_2d(lib):
    """A 2-D call is the 3-D operator with a unit D dimension: dense stride-2
    layers take the tensor-core kernels, the rest the generic kernel."""
    dense = (32, 64, 64, (128, 128), (4, 4), 1, (2, 2), (1, 1), (0, 0), (1, 1))
    assert ct.ct_path_2d(*dense, ct.CT_F32) == "tc3d_tf32x3"
    assert ct.ct_path_2d(*dense, ct.CT_F32, fused=True) == "tc3d_tf32x3"
    assert ct.ct_path_2d(*dense, ct.CT_BF16) == "umma_bf16"
    # kH * kW = 4: the bf16 weight repack needs multiples of 8 -> generic
    assert ct.ct_path_2d(1, 64, 32, (4, 8), (2, 2), 1, (2, 2), (0, 0), (0, 0), (1, 1),
                         ct.CT_BF16) == "gather_generic"
    assert ct.ct_path_2d(2, 6, 4, (5, 7), (3, 2), 2, (2, 3), (1, 0), (1, 2), (1, 1),
                         ct.CT_F32) == "gather_generic"
    # 32 input channels in groups: the grouped tensor-core path (fused: generic)
    assert ct.ct_path_2d(2, 32, 32, (16, 16), (5, 7), 4, (2, 2), (2, 3), (1, 1), (1, 1),
                         ct.CT_F32) == "tc3dg_tf32x3"
    assert ct.ct_path_2d(2, 32, 32, (16, 16), (5, 7), 4, (2, 2), (2, 3), (1, 1), (1, 1),
                         ct.CT_F32, fused=True) == "gather_generic"
    ct.ct_set_path_override(2)
    try:
        assert ct.ct_path_2d(*dense, ct.CT_F32) == "gather_generic"
    finally:
        ct.ct_set_path_override(0)
    assert ct.ct_path_2d(1, 4, 8, (0, 4), (3, 3), 1, (2, 2), (1, 1), (0, 0), (1, 1), ct.CT_F32) is None
    with pytest.raises(ct.CTError) as e:
        ct.ct_workspace_size_2d(1, 4, 8, (4, 4), (3, 3), 1, (2, 2), (1, 1), (2, 0), (1, 1), ct.CT_F32)
    assert e.value.code == ct.CT_ERR_SHAPE
    # the same layer through the 2-D and the 3-D entry (unit D) needs the same workspace
    n2 = ct.ct_workspace_size_2d(*dense, ct.CT_F32)
    n3 = ct.ct_workspace_size_3d(32, 64, 64, (1, 128, 128), (1, 4, 4), 1, (1, 2, 2), (0, 1, 1),
                                 (0, 0, 0), (1, 1, 1), ct.CT_F32)
    assert n2 == n3 >= 32 * 64 * 128 * 128 * 4
    nb2 = ct.ct_workspace_size_2d(*dense, ct.CT_BF16)
    # channels-last bf16 x plus the weight panels: 4 phases x 2 x 2 taps per phase
    assert nb2 >= 32 * 64 * 128 * 128 * 2 + 4 * 4 * 64 * 64 * 2


def test_path_selection_channels_last(lib):
    """Channels-last calls: bf16 shapes of the bf16 tensor-core kernel take it
    (x read in place: workspace only for the weight panels), dense FP32 shapes
    the FP32 tensor-core kernel, the rest the generic kernel."""
    dense = (16, 256, 128, (16, 16, 16), (4, 4, 4), 1, (2, 2, 2), (1, 1, 1), (0, 0, 0), (1, 1, 1))
    assert ct.ct_path_cl(3, *dense, ct.CT_BF16) == "umma_bf16"
    assert ct.ct_path_cl(3, *dense, ct.CT_BF16, fused=True) == "gather_generic"
    assert ct.ct_path_cl(3, *dense, ct.CT_F32) == "tc3d_tf32x3"
    assert ct.ct_path_cl(3, *dense, ct.CT_F32, fused=True) == "tc3d_tf32x3"
    grouped = (8, 32, 32, (16, 32, 32), (3, 5, 7), 4, (2, 2, 2), (1, 2, 3), (1, 1, 1), (1, 1, 1))
    assert ct.ct_path_cl(3, *grouped, ct.CT_F32) == "gather_generic"
    d2 = (16, 256, 128, (64, 64), (4, 4), 1, (2, 2), (1, 1), (0, 0), (1, 1))
    assert ct.ct_path_cl(2, *d2, ct.CT_BF16) == "umma_bf16"
    assert ct.ct_path_cl(1, 16, 32, 64, (131072,), (3,), 1, (2,), (1,), (0,), (2,), ct.CT_F32) == "gather_generic"
    n_cf = ct.ct_workspace_size_3d(*dense, ct.CT_BF16)
    n_cl = ct.ct_workspace_size_cl(3, *dense, ct.CT_BF16)
    x_bytes = 16 * 256 * 16 ** 3 * 2
    assert n_cl == n_cf - x_bytes and n_cl >= 8 * 128 * 8 * 256 * 2
    # FP32: the bf16 (hi, lo) copy of x and the panels, as channels first
    assert ct.ct_workspace_size_cl(3, *dense, ct.CT_F32) == ct.ct_workspace_size_3d(*dense, ct.CT_F32)
    assert ct.ct_path_cl(4, *dense, ct.CT_BF16) is None
    with pytest.raises(ct.CTError) as e:
        ct.ct_workspace_size_cl(3, 1, 4, 8, (4, 4, 4), (3, 3, 3), 3, (2, 2, 2), (1, 1, 1), (0, 0, 0),
                                (1, 1, 1), ct.CT_F32)
    assert e.value.code == ct.CT_ERR_SHAPE


def test_workspace_sizes(lib):
    assert ct.ct_workspace_size_1d(16, 32, 64, 131072, 3, 1, 2, 1, 0, 2, ct.CT_F32) == 0
    # FP32 3-D tensor-core path: a channels-last copy of x as tf32 (t, l) pairs
    # (8 bytes per value) and the per-tap weight panels (8 bytes per weight);
    # the opt-in bf16 split keeps (hi, lo) bf16 pairs (4 bytes per value)
    fused = (128, 32, 64, (16, 16, 16), (3, 3, 3), 1, (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1))
    nf = ct.ct_workspace_size_3d(*fused, ct.CT_F32)
    assert nf >= 128 * 32 * 16 ** 3 * 8 + 27 * 64 * 32 * 8
    nf2 = ct.ct_workspace_size_3d(*fused, ct.CT_F32_BF16X2)
    assert 128 * 32 * 16 ** 3 * 4 + 2 * 27 * 64 * 32 * 4 <= nf2 < nf
    # the grouped workload: an (N, D, W, H, 64) copy of x (tf32 t and l parts:
    # 8 bytes per value) and one t + l panel per input offset (24 offsets, 1920
    # rows of 128 bytes)
    ng = ct.ct_workspace_size_3d(8, 32, 32, (16, 32, 32), (3, 5, 7), 4, (2, 2, 2), (1, 2, 3),
                                 (1, 1, 1), (1, 1, 1), ct.CT_F32)
    assert ng >= 8 * 32 * 16 * 32 * 32 * 8 + 1920 * 32 * 4
    nb = ct.ct_workspace_size_3d(16, 256, 128, (16, 16, 16), (4, 4, 4), 1, (2, 2, 2), (1, 1, 1),
                                 (0, 0, 0), (1, 1, 1), ct.CT_BF16)
    path = ct.ct_path_3d(16, 256, 128, (16, 16, 16), (4, 4, 4), 1, (2, 2, 2), (1, 1, 1),
                         (0, 0, 0), (1, 1, 1), ct.CT_BF16)
    if path == "umma_bf16":
        # channels-last x copy plus phase-packed weights, both bf16
        assert nb >= 16 * 256 * 16 ** 3 * 2 + 8 * 128 * 8 * 256 * 2
    else:
        assert nb == 0


def test_selftest_rejects_out_of_range_limits(lib):
    # argument checks come before anything touches a device
    for bad in (0, 2_000_000_000):
        with pytest.raises(ct.CTError) as ei:
            ct.ct_selftest_wait_timeout(bad)
        assert ei.value.code == ct.CT_ERR_ARG


def test_opt_in_split_path_names(lib):
    """CT_F32_BF16X2 stores x and w as fp32 and selects the two-term bf16 split
    on the FP32 2-D / 3-D tensor-core paths only; every other path is the
    CT_F32 one."""
    fused = (128, 32, 64, (16, 16, 16), (3, 3, 3), 1, (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1))
    assert ct.ct_path_3d(*fused, ct.CT_F32_BF16X2, 1) == "tc3d_bf16x2"
    grouped = (8, 32, 32, (16, 32, 32), (3, 5, 7), 4, (2, 2, 2), (1, 2, 3), (1, 1, 1), (1, 1, 1))
    assert ct.ct_path_3d(*grouped, ct.CT_F32_BF16X2, 0) == "tc3dg_bf16x2"
    assert ct.ct_path_2d(64, 32, 64, (128, 128), (3, 3), 1, (2, 2), (1, 1), (1, 1), (1, 1),
                         ct.CT_F32_BF16X2, 0) == "tc3d_bf16x2"
    assert ct.ct_path_1d(16, 32, 64, 131072, 3, 1, 2, 1, 0, 2, ct.CT_F32_BF16X2) == "tc1d_tf32x3"
    assert ct.ct_path_3d(1, 6, 4, (3, 4, 5), (2, 3, 4), 2, (3, 1, 2), (1, 0, 2), (2, 0, 1), (1, 2, 1),
                         ct.CT_F32_BF16X2, 0) == "gather_generic"
    assert call1d(lib, dtype=ct.CT_F32_BF16X2, N=0) == 0
    assert call1d(lib, dtype=3) == 1


def _fused_call(lib, ws, ws_bytes):
    i3 = ct._I3
    return lib.ct_forward_3d_add_hswish(FAKE, FAKE + (1 << 24), None, FAKE + (1 << 26), FAKE + (1 << 28), 1, 32,
                                        64, i3(4, 4, 4), i3(3, 3, 3), 1, i3(2, 2, 2), i3(1, 1, 1),
                                        i3(1, 1, 1), i3(1, 1, 1), ct.CT_F32, ws, ws_bytes, None)


def test_workspace_rule(lib):
    """A workspace is absent or at least the reported size: a non-zero one that
    is too small (or misaligned, or a NULL pointer with a size) is rejected
    before any launch instead of silently changing the kernel; ct_path_call
    reports the kernel of a call with a given workspace size."""
    args = (3, 0, 1, 32, 64, (4, 4, 4), (3, 3, 3), 1, (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1))
    need = ct.ct_workspace_size_3d(1, 32, 64, (4, 4, 4), (3, 3, 3), 1, (2, 2, 2), (1, 1, 1), (1, 1, 1),
                                   (1, 1, 1), ct.CT_F32)
    assert need > 0
    WS = FAKE + (1 << 30)
    assert _fused_call(lib, WS, need - 256) == ct.CT_ERR_WORKSPACE
    assert _fused_call(lib, WS + 16, need) == ct.CT_ERR_WORKSPACE     # not 256-byte aligned
    assert _fused_call(lib, None, need) == ct.CT_ERR_WORKSPACE         # a size without a buffer
    assert ct.ct_path_call(*args, ct.CT_F32, 1, need) == "tc3d_tf32x3"
    assert ct.ct_path_call(*args, ct.CT_F32, 1, need + 4096) == "tc3d_tf32x3"
    assert ct.ct_path_call(*args, ct.CT_F32, 1, need - 256) is None
    assert ct.ct_path_call(*args, ct.CT_F32, 1, 0) == "phase3d_f32"   # no workspace: the FFMA kernel
    assert ct.ct_path_call(*args, ct.CT_F32_BF16X2, 1, 0) == "phase3d_f32"
    # bf16 on the tensor cores needs its workspace; channels-last bf16 only the panels
    dense = (3, 0, 16, 256, 128, (16, 16, 16), (4, 4, 4), 1, (2, 2, 2), (1, 1, 1), (0, 0, 0), (1, 1, 1))
    nb = ct.ct_workspace_size_3d(*dense[2:], ct.CT_BF16)
    assert ct.ct_path_call(*dense, ct.CT_BF16, 0, 0) is None
    assert ct.ct_path_call(*dense, ct.CT_BF16, 0, nb) == "umma_bf16"
    dense_cl = (3, 1) + dense[2:]
    ncl = ct.ct_workspace_size_cl(3, *dense[2:], ct.CT_BF16)
    assert ct.ct_path_call(*dense_cl, ct.CT_BF16, 0, ncl) == "umma_bf16"
    # paths without scratch accept any workspace and none
    assert ct.ct_path_call(1, 0, 16, 32, 64, (131072,), (3,), 1, (2,), (1,), (0,), (2,), ct.CT_F32, 0, 0) == \
        "tc1d_tf32x3"
    assert ct.ct_path_call(1, 0, 16, 32, 64, (0,), (3,), 1, (2,), (1,), (0,), (2,), ct.CT_F32, 0, 0) is None


def test_noalloc_scratch_constant_matches_header(lib):
    txt = open(os.path.join(ROOT, "include", "ct.h")).read()
    m = re.search(r"#define\s+CT_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*\*\s*(\d+)u\s*\*\s*(\d+)u\)", txt)
    assert m, "CT_NOALLOC_SCRATCH_BYTES not found in include/ct.h"
    assert int(m.group(1)) * int(m.group(2)) * int(m.group(3)) == ct.CT_NOALLOC_SCRATCH_BYTES


_SCRATCH_FREE = {"gather_generic", "phase1d_f32", "phase3d_f32", "tc1d_tf32x3"}
_SCRATCH = {"umma_bf16", "tc3d_tf32x3", "tc3d_bf16x2", "tc3dg_tf32x3", "tc3dg_bf16x2", "tc3s_tf32x3",
            "tc3s_bf16x2"}


def test_path_and_workspace_queries_agree(lib):
    """For random shapes, small ones and ones in the tensor-core kernels'
    ranges: the kernel a path query names needs scratch exactly when the
    workspace query reports some (a multiple of 256 bytes); a call given that
    much takes that kernel, one given 256 bytes less is rejected, and one given
    none runs a kernel without scratch (fp32) or is rejected (bf16)."""
    rng = np.random.default_rng(77)
    pick = lambda seq: seq[int(rng.integers(0, len(seq)))]
    seen = set()
    for t in range(800):
        nd = 1 + t % 3
        mode = (t // 3) % 4          # 0 any; 1 tensor-core channel counts; 2 stride 2; 3 FFMA 3-D shapes
        G = pick([1, 1, 2, 4])
        C_in, C_out = G * pick([1, 2, 8, 16, 32]), G * pick([1, 4, 8, 16, 32])
        dt = pick([ct.CT_F32, ct.CT_F32, ct.CT_BF16, ct.CT_F32_BF16X2])
        if mode in (1, 2):
            G = pick([1, 1, 1, 2, 4])
            C_in, C_out = pick([32, 64, 128]), pick([16, 32, 64, 128])
        K = [int(rng.integers(1, 6)) for _ in range(nd)]
        S = [pick([1, 2, 2, 3, 4]) for _ in range(nd)]
        DL = [pick([1, 1, 2]) for _ in range(nd)]
        if mode == 2:
            K = [pick([2, 3, 4]) for _ in range(nd)]
            S, DL = [2] * nd, [1] * nd
            if dt == ct.CT_BF16:            # the bf16 kernel: equal even extents, dense channels
                K, G, C_in = [pick([2, 4]) if nd == 3 else 4] * nd, 1, pick([64, 128])
        if mode == 1 and nd == 1 and t % 2:     # the 1-D tensor-core kernel's range
            C_in, G, K, DL = 32, 1, [pick([1, 2, 3, 4])], [S[0] * pick([1, 2])]
        if mode == 3 and nd == 3:
            dt, G = ct.CT_F32, pick([1, 2])
            C_in, C_out = G * pick([4, 8]), G * 16
            K, S, DL = pick([[3, 3, 3], [3, 5, 7]]), [2] * 3, [1] * 3
        P = [int(rng.integers(0, DL[d] * (K[d] - 1) // 2 + 1)) for d in range(nd)]
        if mode == 3 and nd == 3:
            P[2] = (K[2] - 1) // 2
        OP = [int(rng.integers(0, max(S[d], DL[d]))) for d in range(nd)]
        L = [int(rng.integers(1, 9)) for _ in range(nd - 1)] + [pick([2, 4, 8, 16, 32, 5, 12, 60])]
        if nd == 1:
            L = [4 * int(rng.integers(1, 1000))]
        if C_in % G or C_out % G:
            G = 1
        N = pick([1, 2])
        if any(ct.ct_out_len(L[d], K[d], S[d], P[d], OP[d], DL[d]) < 1 for d in range(nd)):
            continue
        if nd == 1:
            a1 = (N, C_in, C_out, L[0], K[0], G, S[0], P[0], OP[0], DL[0], dt)
            path, need = ct.ct_path_1d(*a1), ct.ct_workspace_size_1d(*a1)
        elif nd == 2:
            a2 = (N, C_in, C_out, L, K, G, S, P, OP, DL, dt)
            path, need = ct.ct_path_2d(*a2), ct.ct_workspace_size_2d(*a2)
        else:
            a3 = (N, C_in, C_out, L, K, G, S, P, OP, DL, dt)
            path, need = ct.ct_path_3d(*a3), ct.ct_workspace_size_3d(*a3)
        what = (nd, N, C_in, C_out, G, L, K, S, P, OP, DL, dt, path, need)
        assert path in _SCRATCH_FREE | _SCRATCH, what
        assert (need > 0) == (path in _SCRATCH), what
        assert need % 256 == 0, what
        call = (nd, 0, N, C_in, C_out, L, K, G, S, P, OP, DL, dt, 0)
        assert ct.ct_path_call(*call, need) == path, what
        if need:
            assert ct.ct_path_call(*call, need - 256) is None, what
            bare = ct.ct_path_call(*call, 0)
            assert (bare is None) if dt == ct.CT_BF16 else (bare in _SCRATCH_FREE), (what, bare)
            seen.add(bare)
        seen.add(path)
    assert seen >= _SCRATCH_FREE | _SCRATCH, sorted(x for x in seen if x)
