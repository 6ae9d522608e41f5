"""GPU test of ct_forward_3d_noalloc, the entry point for callers that cannot
allocate device memory (for instance an engine that reserves all device
memory at start-up and forbids allocation afterwards, or a plugin inside a
framework that owns the device memory pool).  It runs the bf16 tensor-core
ConvTranspose3d with the library's own fixed scratch buffer instead of a
caller-supplied workspace.  On two calls in a row with different inputs (so
that leftovers of the first call cannot hide in the second) its output must
be bit for bit the output of the regular ct_forward_3d -- the same kernels on
the same bits, so any difference is a scratch-offset mistake -- and must match
the CPU oracle: within the bf16 tolerance for random inputs, exactly for
small integers.

The file name makes pytest collect it last."""
import numpy as np
import pytest

import ctcase as cc
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transposed_convolution_convtranspose_gb300 import build
    build.build()
    import transposed_convolution_convtranspose_gb300 as ct
    ct.load()
    torch.cuda.set_device(0)
    return ct


def _args(c):
    return (c["N"], c["C_in"], c["C_out"], c["L"], c["K"], c["G"], c["S"], c["P"], c["OP"], c["DL"])


def test_noalloc_matches_workspace_entry_point_twice(lib):
    import torch
    ct = lib
    name = "convT3d_bf16_dense"
    # the bf16 workload's layer on 8^3 inputs, batch 2 (the oracle finishes in seconds)
    c = cc.case_from_config(name, N=2)
    c["L"] = [8, 8, 8]
    N, C_in, C_out, L, K, G, S, P, OP, DL = _args(c)
    assert ct.ct_path_3d(N, C_in, C_out, L, K, G, S, P, OP, DL, ct.CT_BF16) == "umma_bf16"
    out_shape = cc.out_shape(c)
    stream = torch.cuda.current_stream()
    for call, (seed, int_range) in enumerate(((901, None), (902, 3))):
        t = cc.make_inputs(c, seed=seed, bound=workloads.CONFIGS[name]["bound"], int_range=int_range)
        x, w, b, _ = cc.to_device(t, c, "cuda:0")
        # the regular entry point, with a workspace
        nb = ct.ct_workspace_size_3d(N, C_in, C_out, L, K, G, S, P, OP, DL, ct.CT_BF16)
        assert 0 < nb <= ct.CT_NOALLOC_SCRATCH_BYTES
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda:0")
        y_ref = torch.empty(out_shape, dtype=torch.float32, device="cuda:0")
        ct.ct_forward_3d(x, w, b, y_ref, N, C_in, C_out, L, K, G, S, P, OP, DL, ct.CT_BF16, ws, nb,
                         stream)
        # the no-allocation entry point
        y = torch.full(out_shape, float("nan"), dtype=torch.float32, device="cuda:0")
        ct.ct_forward_3d_noalloc(x, w, b, y, N, C_in, C_out, L, K, G, S, P, OP, DL, ct.CT_BF16,
                                 stream)
        torch.cuda.synchronize()
        assert ct.ct_last_device_error_code(stream) == ct.CT_OK
        assert torch.equal(y, y_ref), "no-alloc call %d differs from ct_forward_3d" % (call + 1)
        ref = cc.run_oracle(c, t)
        got = y.cpu().numpy()
        if int_range is None:
            cc.assert_close(got, ref, "bf16", "no-alloc call %d vs oracle" % (call + 1))
        else:
            assert np.array_equal(got.astype(np.float64), ref), "no-alloc integer call %d not exact" % (call + 1)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    ct = lib
    # the full bf16 workload at batch 32 needs about 71 MB of scratch
    c = cc.case_from_config("convT3d_bf16_dense", N=32)
    N, C_in, C_out, L, K, G, S, P, OP, DL = _args(c)
    need = ct.ct_workspace_size_3d(N, C_in, C_out, L, K, G, S, P, OP, DL, ct.CT_BF16)
    assert need > ct.CT_NOALLOC_SCRATCH_BYTES
    FAKE = 1 << 40   # never dereferenced: the call is rejected before any launch
    with pytest.raises(ct.CTError) as ei:
        ct.ct_forward_3d_noalloc(FAKE, FAKE + (1 << 30), None, FAKE + (1 << 32), N, C_in, C_out, L,
                                 K, G, S, P, OP, DL, ct.CT_BF16)
    assert ei.value.name == "CT_ERR_WORKSPACE"
    # fp32 problems take paths without scratch; this entry point does not run them
    with pytest.raises(ct.CTError) as ei:
        ct.ct_forward_3d_noalloc(FAKE, FAKE + (1 << 30), None, FAKE + (1 << 32), 1, 32, 64,
                                 (4, 4, 4), (3, 3, 3), 1, (2, 2, 2), (1, 1, 1), (1, 1, 1),
                                 (1, 1, 1), ct.CT_F32)
    assert ei.value.name == "CT_ERR_UNSUPPORTED"
