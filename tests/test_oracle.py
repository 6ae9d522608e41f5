"""The CPU oracle against its pins (no GPU).  See tests/oracle_pins.py."""
import numpy as np
import pytest

import oracle as ora
import oracle_pins as pins


@pytest.fixture(scope="module")
def lib():
    return ora.oracle.load_library(ora.build_oracle())


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_impulse_returns_weight_patch(lib):
    """An impulse at input (n, ic, i) returns w[ic] placed at i*s - p, clipped
    to the output, in the output channels of ic's group only (bias 0)."""
    rng = np.random.default_rng(11)
    for t in range(30):
        nd = 1 + t % 3
        c = pins.random_case(rng, nd)
        x = np.zeros([c["N"], c["C_in"]] + c["L"])
        n = int(rng.integers(c["N"]))
        ic = int(rng.integers(c["C_in"]))
        i = [int(rng.integers(L)) for L in c["L"]]
        x[(n, ic) + tuple(i)] = 1.0
        w = rng.standard_normal([c["C_in"], c["C_out"] // c["G"]] + c["K"])
        y = ora.conv_transpose(x, w, None, c["S"], c["P"], c["OP"], c["DL"], c["G"], lib=lib)
        Cog = c["C_out"] // c["G"]
        g = ic // (c["C_in"] // c["G"])
        want = np.zeros_like(y)
        import itertools
        for kk in itertools.product(*[range(k) for k in c["K"]]):
            o = [i[d] * c["S"][d] - c["P"][d] + kk[d] * c["DL"][d] for d in range(nd)]
            if all(0 <= o[d] < y.shape[2 + d] for d in range(nd)):
                want[(n, slice(g * Cog, (g + 1) * Cog)) + tuple(o)] += w[(ic, slice(None)) + kk]
        assert np.array_equal(y, want), c


def test_group_block_diagonal(lib):
    """A weight change inside group g changes only the outputs of group g."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((2, 6, 4, 5, 3))
    w = rng.standard_normal((6, 2, 3, 2, 3))
    args = dict(stride=(2, 1, 2), padding=(1, 0, 1), output_padding=(1, 0, 0),
                dilation=(1, 2, 1), groups=3)
    y0 = ora.conv_transpose(x, w, None, lib=lib, **args)
    for g in range(3):
        w2 = w.copy()
        w2[2 * g:2 * g + 2] += rng.standard_normal(w2[2 * g:2 * g + 2].shape)
        y1 = ora.conv_transpose(x, w2, None, lib=lib, **args)
        changed = np.any(y1 != y0, axis=(0, 2, 3, 4))
        assert list(np.nonzero(changed)[0]) == [2 * g, 2 * g + 1]


def test_linearity(lib):
    rng = np.random.default_rng(13)
    x1 = rng.standard_normal((2, 4, 7))
    x2 = rng.standard_normal((2, 4, 7))
    w = rng.standard_normal((4, 3, 3))
    kw = dict(stride=2, padding=1, dilation=2)
    y = ora.conv_transpose(2.5 * x1 - 0.5 * x2, w, lib=lib, **kw)
    y12 = 2.5 * ora.conv_transpose(x1, w, lib=lib, **kw) - 0.5 * ora.conv_transpose(x2, w, lib=lib, **kw)
    assert np.allclose(y, y12, rtol=0, atol=1e-12)


def test_empty_phase_is_bias(lib):
    """For (k=3, s=2, p=1, d=2) no tap lands on an even output: those hold
    exactly the bias (odd-only support of the l1_p79 trace)."""
    rng = np.random.default_rng(14)
    x = rng.standard_normal((2, 4, 64))
    w = rng.standard_normal((4, 8, 3))
    b = rng.standard_normal(8)
    y = ora.conv_transpose(x, w, b, stride=2, padding=1, dilation=2, lib=lib)
    assert y.shape == (2, 8, 129)
    assert np.array_equal(y[:, :, 0::2], np.broadcast_to(b[None, :, None], y[:, :, 0::2].shape))
    assert np.all(y[:, :, 1::2] != b[None, :, None])


def test_rejects_invalid(lib):
    with pytest.raises(ValueError):
        ora.conv_transpose(np.ones((1, 3, 4)), np.ones((3, 1, 3)), groups=2, lib=lib)
    with pytest.raises(ValueError):   # L_out <= 0
        ora.conv_transpose(np.ones((1, 1, 1)), np.ones((1, 1, 1)), padding=1, lib=lib)


def test_all_cores_baseline_matches_oracle():
    """The all-cores baseline (ct_oracle_mt.c) computes the same definition as
    the parity oracle, split by output slice: equal up to summation order on
    random small cases of every dimensionality, with groups, on 1, 3 and 8
    threads."""
    rng = np.random.default_rng(23)
    for t in range(24):
        nd = 1 + t % 3
        c = pins.random_case(rng, nd)
        x = rng.standard_normal([c["N"], c["C_in"]] + c["L"])
        w = rng.standard_normal([c["C_in"], c["C_out"] // c["G"]] + c["K"])
        b = rng.standard_normal(c["C_out"]) if t % 2 else None
        kw = dict(stride=c["S"], padding=c["P"], output_padding=c["OP"], dilation=c["DL"], groups=c["G"])
        ref = ora.conv_transpose(x, w, b, **kw)
        got = ora.conv_transpose_mt(x, w, b, threads=(1, 3, 8)[t % 3], **kw)
        assert got.shape == ref.shape
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12), (t, c)
