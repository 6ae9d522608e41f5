"""Shared helpers of the GPU parity tests: run one case through the C ABI
and through the CPU oracle on the same seeded inputs, and compare."""
import numpy as np

import oracle as ora
import workloads

F32_TOL = 1e-4      # |err| <= 1e-4 * (1 + |ref|)
BF16_TOL = 2e-2     # |err| <= 2e-2 * (|ref| + rms(ref))


def case_from_config(name, N=None):
    c = workloads.CONFIGS[name]
    return dict(nd=c["nd"], N=c["N"] if N is None else N, C_in=c["C_in"], C_out=c["C_out"],
                G=c["groups"], L=list(c["L_in"]), K=list(c["k"]), S=list(c["stride"]),
                P=list(c["padding"]), OP=list(c["output_padding"]), DL=list(c["dilation"]),
                bias=c["bias"], add=c["add"], dtype=c["dtype"], layout=c.get("layout", "cf"))


def out_shape(c):
    Lo = [ora.out_len(c["L"][d], c["K"][d], c["S"][d], c["P"][d], c["OP"][d], c["DL"][d])
          for d in range(c["nd"])]
    return [c["N"], c["C_out"]] + Lo


def make_inputs(c, seed, int_range=None, bound=None):
    x_shape = [c["N"], c["C_in"]] + c["L"]
    w_shape = [c["C_in"], c["C_out"] // c["G"]] + c["K"]
    if bound is None:
        import math
        bound = 1.0 / math.sqrt(max(1, (c["C_out"] // c["G"]) * int(np.prod(c["K"]))))
    add_shape = out_shape(c) if c["add"] else None
    return workloads.make_tensors(seed, x_shape, w_shape, bound,
                                  bias_len=c["C_out"] if c["bias"] else None,
                                  add_shape=add_shape, dtype=c["dtype"], int_range=int_range)


def to_device(t, c, dev):
    import torch
    if c["dtype"] == "bf16":
        x = torch.from_numpy(t["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
        w = torch.from_numpy(t["w_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        x = torch.from_numpy(t["x"]).to(dev)
        w = torch.from_numpy(t["w"]).to(dev)
    b = torch.from_numpy(t["bias"]).to(dev) if t["bias"] is not None else None
    a = torch.from_numpy(t["add"]).to(dev) if t["add"] is not None else None
    return x, w, b, a


def kwargs(c):
    if c["nd"] == 1:
        return dict(stride=c["S"][0], padding=c["P"][0], output_padding=c["OP"][0],
                    dilation=c["DL"][0], groups=c["G"])
    return dict(stride=tuple(c["S"]), padding=tuple(c["P"]), output_padding=tuple(c["OP"]),
                dilation=tuple(c["DL"]), groups=c["G"])


def run_gpu(c, t, dev="cuda:0", inplace_add=False):
    """Run the case through the library (C ABI via the binding); returns a torch tensor."""
    import transposed_convolution_convtranspose_gb300 as ct
    x, w, b, a = to_device(t, c, dev)
    kw = kwargs(c)
    kw["split2"] = bool(c.get("split2", False))
    if c.get("layout", "cf") == "cl":
        # channels-last call on the same values; the result is returned in the
        # oracle's channels-first order
        xcl = x.movedim(1, -1).contiguous()
        acl = a.movedim(1, -1).contiguous() if a is not None else None
        if c["nd"] == 1:
            kw = {k: (v if k in ("groups", "split2") else (v,)) for k, v in kw.items()}
        y = ct.conv_transpose_cl(xcl, w, b, acl, out=acl if inplace_add else None, **kw)
        return y.movedim(-1, 1).contiguous()
    if c["nd"] == 1:
        if c["add"]:
            # no channels-first 1-D fused entry point (the channels-last one has it)
            raise ValueError("fused 1-D case needs layout 'cl': %r" % (c,))
        y = ct.conv_transpose1d(x, w, b, **kw)
    elif c["nd"] == 2:
        if c["add"]:
            y = ct.conv_transpose2d_add_hswish(x, w, b, a, out=a if inplace_add else None, **kw)
        else:
            y = ct.conv_transpose2d(x, w, b, **kw)
    elif c["add"]:
        y = ct.conv_transpose3d_add_hswish(x, w, b, a, out=a if inplace_add else None, **kw)
    else:
        y = ct.conv_transpose3d(x, w, b, **kw)
    return y


def run_oracle(c, t):
    y = ora.conv_transpose(t["x"], t["w"], t["bias"], c["S"], c["P"], c["OP"], c["DL"], c["G"])
    if c["add"]:
        y = ora.add_hswish(y, t["add"])
    return y


def oracle_at(c, t, flat):
    y = ora.conv_transpose_at(t["x"], t["w"], flat, t["bias"], c["S"], c["P"], c["OP"], c["DL"],
                              c["G"])
    if c["add"]:
        y = ora.add_hswish(y, t["add"].reshape(-1)[flat])
    return y


def assert_close(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, "%s: shape %r vs oracle %r" % (what, got.shape, ref.shape)
    if got.size == 0:
        return
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    err = np.abs(got - ref)
    if dtype == "bf16":
        lim = BF16_TOL * (np.abs(ref) + np.sqrt(np.mean(ref * ref)))
    else:
        lim = F32_TOL * (1.0 + np.abs(ref))
    bad = err > lim
    if bad.any():
        i = int(np.argmax(err - lim))
        raise AssertionError("%s: %d/%d outputs out of tolerance; worst flat index %d got %r ref %r"
                             % (what, int(bad.sum()), bad.size, i, got.ravel()[i], ref.ravel()[i]))


def sample_indices(shape, n_random, seed):
    """Random flat indices plus the corners and edges of every spatial dim."""
    rng = np.random.default_rng(seed)
    total = int(np.prod(shape))
    idx = list(rng.integers(0, total, size=n_random))
    N, C = shape[:2]
    sp = shape[2:]
    for n in (0, N - 1):
        for cch in (0, C - 1, C // 2):
            for corner in range(1 << len(sp)):
                pos = []
                for d, L in enumerate(sp):
                    hi = (corner >> d) & 1
                    pos.append(L - 1 - int(rng.integers(0, min(3, L))) if hi
                               else int(rng.integers(0, min(3, L))))
                idx.append(np.ravel_multi_index([n, cch] + pos, shape))
    return np.unique(np.array(idx, dtype=np.int64))
