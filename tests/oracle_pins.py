"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each check takes the loaded oracle library (so the planted-mistake test can
run the same checks against a deliberately broken copy) and raises
AssertionError on failure.  None of them re-types the oracle's scatter loop:
they compare it with the pages' printed values, with library routines
(torch's CPU convolutions), with an independently written direct
convolution through the adjoint identity, and with the zero-insertion plus
flipped-kernel restatement of the operator.
"""
import configparser
import itertools
import os
import re

import numpy as np

import oracle as ora

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- fixtures
def load_out_len():
    rows = []
    with open(os.path.join(GOLDEN, "out_len.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            lhs, src = line.split("|", 1)
            args, res = lhs.split("->")
            rows.append(([int(v) for v in args.split()], int(res), src.strip()))
    return rows


def load_worked_1d():
    cp = configparser.ConfigParser(comment_prefixes=("#",), inline_comment_prefixes=None)
    cp.read(os.path.join(GOLDEN, "worked_1d.txt"))
    out = []
    for sec in cp.sections():
        s = cp[sec]
        out.append(dict(name=sec, source=s["source"], L_in=int(s["L_in"]), k=int(s["k"]),
                        s=int(s["s"]), p=int(s["p"]), op=int(s["op"]), d=int(s["d"]),
                        x=s["x"].split(), w=s["w"].split(),
                        y=[e.strip() for e in s["y"].split(";")]))
    return out


def load_tap_counts():
    rows = []
    with open(os.path.join(GOLDEN, "tap_counts.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            params, head, tail = [t.strip() for t in line.split("|")]
            extra = {}
            for item in tail.split():
                pos, cnt = item.split(":")
                extra[int(pos)] = int(cnt)
            rows.append(([int(v) for v in params.split()], [int(v) for v in head.split()], extra))
    return rows


_TERM = re.compile(r"^[A-Za-z]\w*(\*[A-Za-z]\w*)*$")


def eval_expr(expr, env):
    """Evaluate a sum of products of names ('a*w1 + b*w0') or the literal 0."""
    total = 0
    for term in expr.split("+"):
        term = term.strip().replace(" ", "")
        if term == "0":
            continue
        assert _TERM.match(term), "bad fixture term %r" % term
        val = 1
        for name in term.split("*"):
            val = val * env[name]
        total += val
    return total


# ---------------------------------------------------------------- pins
def pin_out_len(lib):
    for (L, k, s, p, op, d), want, src in load_out_len():
        got = ora.out_len(L, k, s, p, op, d, lib=lib)
        assert got == want, "out_len %s: got %d want %d (%s)" % ((L, k, s, p, op, d), got, want, src)


def pin_worked_examples(lib, seed=0):
    rng = np.random.default_rng(seed)
    for ex in load_worked_1d():
        # distinct integers: every product and sum is exact in double
        names = ex["x"] + ex["w"]
        vals = rng.choice(np.arange(2, 200), size=len(names), replace=False)
        env = dict(zip(names, [int(v) for v in vals]))
        x = np.array([env[n] for n in ex["x"]], dtype=np.float64).reshape(1, 1, -1)
        w = np.array([env[n] for n in ex["w"]], dtype=np.float64).reshape(1, 1, -1)
        y = ora.conv_transpose(x, w, stride=ex["s"], padding=ex["p"], output_padding=ex["op"],
                               dilation=ex["d"], lib=lib)
        want = np.array([eval_expr(e, env) for e in ex["y"]], dtype=np.float64)
        assert y.shape == (1, 1, want.size), "%s: shape %r, want %d outputs (%s)" % (
            ex["name"], y.shape, want.size, ex["source"])
        assert np.array_equal(y[0, 0], want), "%s: %r != %r (%s)" % (
            ex["name"], y[0, 0], want, ex["source"])


def pin_tap_counts(lib):
    for (L, k, s, p, op, d), head, extra in load_tap_counts():
        x = np.ones((1, 1, L))
        w = np.ones((1, 1, k))
        y = ora.conv_transpose(x, w, stride=s, padding=p, output_padding=op, dilation=d, lib=lib)[0, 0]
        assert list(y[:len(head)].astype(int)) == head, "tap counts %s: %r != %r" % (
            (L, k, s, p, op, d), list(y[:len(head)]), head)
        for pos, cnt in extra.items():
            assert int(y[pos]) == cnt, "tap count at %d: %r != %d" % (pos, y[pos], cnt)


def torch_conv_transpose(x, w, bias, stride, padding, output_padding, dilation, groups):
    import torch
    import torch.nn.functional as F
    nd = x.ndim - 2
    fn = {1: F.conv_transpose1d, 2: F.conv_transpose2d, 3: F.conv_transpose3d}[nd]
    b = None if bias is None else torch.from_numpy(np.asarray(bias, np.float64))
    y = fn(torch.from_numpy(np.asarray(x, np.float64)), torch.from_numpy(np.asarray(w, np.float64)),
           b, stride=tuple(stride), padding=tuple(padding), output_padding=tuple(output_padding),
           groups=groups, dilation=tuple(dilation))
    return y.numpy()


def torch_conv(z, w, stride, padding, dilation, groups):
    import torch
    import torch.nn.functional as F
    nd = z.ndim - 2
    fn = {1: F.conv1d, 2: F.conv2d, 3: F.conv3d}[nd]
    return fn(torch.from_numpy(np.asarray(z, np.float64)), torch.from_numpy(np.asarray(w, np.float64)),
              None, stride=tuple(stride), padding=tuple(padding), dilation=tuple(dilation),
              groups=groups).numpy()


def random_case(rng, nd, small=True):
    """A random valid parameter set with 1..3 spatial dims (tiny sizes)."""
    while True:
        G = int(rng.choice([1, 1, 2, 3]))
        C_in = G * int(rng.integers(1, 4))
        C_out = G * int(rng.integers(1, 4))
        N = int(rng.integers(1, 3))
        L = [int(rng.integers(1, 6 if nd == 3 else 9)) for _ in range(nd)]
        K = [int(rng.integers(1, 5)) for _ in range(nd)]
        S = [int(rng.integers(1, 4)) for _ in range(nd)]
        DL = [int(rng.integers(1, 4)) for _ in range(nd)]
        P = [int(rng.integers(0, 3)) for _ in range(nd)]
        OP = [int(rng.integers(0, max(S[d], DL[d]))) for d in range(nd)]
        Lo = [(L[d] - 1) * S[d] - 2 * P[d] + DL[d] * (K[d] - 1) + OP[d] + 1 for d in range(nd)]
        if min(Lo) >= 1:
            return dict(N=N, C_in=C_in, C_out=C_out, G=G, L=L, K=K, S=S, P=P, OP=OP, DL=DL)


def pin_vs_torch(lib, n_cases=40, seed=1):
    """Special case that reduces to a library routine: torch's CPU conv_transpose."""
    rng = np.random.default_rng(seed)
    for t in range(n_cases):
        nd = 1 + t % 3
        c = random_case(rng, nd)
        x = rng.standard_normal([c["N"], c["C_in"]] + c["L"])
        w = rng.standard_normal([c["C_in"], c["C_out"] // c["G"]] + c["K"])
        b = rng.standard_normal(c["C_out"]) if t % 2 else None
        y = ora.conv_transpose(x, w, b, c["S"], c["P"], c["OP"], c["DL"], c["G"], lib=lib)
        yt = torch_conv_transpose(x, w, b, c["S"], c["P"], c["OP"], c["DL"], c["G"])
        assert y.shape == yt.shape, "case %r: shape %r vs torch %r" % (c, y.shape, yt.shape)
        err = np.max(np.abs(y - yt)) if y.size else 0.0
        assert err <= 1e-12 * (1 + np.max(np.abs(yt))), "case %r: max err %g vs torch" % (c, err)


def pin_direct_vs_torch(lib, n_cases=30, seed=2):
    rng = np.random.default_rng(seed)
    for t in range(n_cases):
        nd = 1 + t % 3
        c = random_case(rng, nd)
        Lo = [ora.out_len(c["L"][d], c["K"][d], c["S"][d], c["P"][d], c["OP"][d], c["DL"][d], lib=lib)
              for d in range(nd)]
        z = rng.standard_normal([c["N"], c["C_out"]] + Lo)
        w = rng.standard_normal([c["C_in"], c["C_out"] // c["G"]] + c["K"])
        xa = ora.conv_direct(z, w, [c["N"], c["C_in"]] + c["L"], c["S"], c["P"], c["OP"], c["DL"],
                             c["G"], lib=lib)
        xt = torch_conv(z, w, c["S"], c["P"], c["DL"], c["G"])
        # torch's conv yields L_in + floor(op/s) positions (more than L_in only
        # when output_padding >= stride); compare on the common positions
        sl = tuple(slice(0, min(a, b)) for a, b in zip(xa.shape, xt.shape))
        assert np.allclose(xa[sl], xt[sl], rtol=0, atol=1e-12 * (1 + np.max(np.abs(xt)))), \
            "direct conv differs from torch conv for %r" % (c,)


def pin_adjoint(lib, n_cases=40, seed=3):
    """<convT(x), z> == <x, conv(z)> with the separately written direct conv."""
    rng = np.random.default_rng(seed)
    for t in range(n_cases):
        nd = 1 + t % 3
        c = random_case(rng, nd)
        x = rng.standard_normal([c["N"], c["C_in"]] + c["L"])
        w = rng.standard_normal([c["C_in"], c["C_out"] // c["G"]] + c["K"])
        y = ora.conv_transpose(x, w, None, c["S"], c["P"], c["OP"], c["DL"], c["G"], lib=lib)
        z = rng.standard_normal(y.shape)
        xa = ora.conv_direct(z, w, x.shape, c["S"], c["P"], c["OP"], c["DL"], c["G"], lib=lib)
        lhs, rhs = float(np.sum(y * z)), float(np.sum(x * xa))
        scale = float(np.sum(np.abs(y * z))) + 1e-300
        assert abs(lhs - rhs) <= 1e-12 * scale, "adjoint identity fails for %r: %r vs %r" % (c, lhs, rhs)


def zero_insert_flip(x, w, stride, padding, output_padding, dilation, groups):
    """The zero-insertion view (l2_p26): insert s-1 zeros between inputs, pad
    d*(k-1)-p on the left and d*(k-1)-p+op on the right (negative pads crop),
    then correlate with the spatially flipped kernel whose channel axes are
    swapped, dilated by d.  Written with numpy, independent of the oracle."""
    nd = x.ndim - 2
    N, C_in = x.shape[:2]
    Cog = w.shape[1]
    C_out = Cog * groups
    Cig = C_in // groups
    L = x.shape[2:]
    K = w.shape[2:]
    up_shape = [(L[d] - 1) * stride[d] + 1 for d in range(nd)]
    up = np.zeros((N, C_in) + tuple(up_shape))
    up[(slice(None), slice(None)) + tuple(slice(None, None, stride[d]) for d in range(nd))] = x
    # pad / crop
    for d in range(nd):
        lo = dilation[d] * (K[d] - 1) - padding[d]
        hi = lo + output_padding[d]
        ax = 2 + d
        if lo >= 0:
            pw = [(0, 0)] * up.ndim
            pw[ax] = (lo, 0)
            up = np.pad(up, pw)
        else:
            up = np.take(up, range(-lo, up.shape[ax]), axis=ax)
        if hi >= 0:
            pw = [(0, 0)] * up.ndim
            pw[ax] = (0, hi)
            up = np.pad(up, pw)
        else:
            up = np.take(up, range(0, up.shape[ax] + hi), axis=ax)
    ext = [dilation[d] * (K[d] - 1) + 1 for d in range(nd)]
    Lo = [up.shape[2 + d] - ext[d] + 1 for d in range(nd)]
    y = np.zeros((N, C_out) + tuple(Lo))
    wf = w[(slice(None), slice(None)) + tuple(slice(None, None, -1) for _ in range(nd))]
    for g in range(groups):
        for kk in itertools.product(*[range(k) for k in K]):
            sl = tuple(slice(kk[d] * dilation[d], kk[d] * dilation[d] + Lo[d]) for d in range(nd))
            win = up[(slice(None), slice(g * Cig, (g + 1) * Cig)) + sl]       # N, Cig, Lo...
            wt = wf[(slice(g * Cig, (g + 1) * Cig), slice(None)) + kk]         # Cig, Cog
            y[:, g * Cog:(g + 1) * Cog] += np.einsum("nc...,co->no...", win, wt)
    return y


def pin_zero_insertion(lib, n_cases=30, seed=4):
    rng = np.random.default_rng(seed)
    for t in range(n_cases):
        nd = 1 + t % 3
        c = random_case(rng, nd)
        x = rng.standard_normal([c["N"], c["C_in"]] + c["L"])
        w = rng.standard_normal([c["C_in"], c["C_out"] // c["G"]] + c["K"])
        y = ora.conv_transpose(x, w, None, c["S"], c["P"], c["OP"], c["DL"], c["G"], lib=lib)
        y2 = zero_insert_flip(x, w, c["S"], c["P"], c["OP"], c["DL"], c["G"])
        assert y.shape == y2.shape, "shape %r vs zero-insertion %r for %r" % (y.shape, y2.shape, c)
        assert np.allclose(y, y2, rtol=0, atol=1e-12 * (1 + np.max(np.abs(y2)))), \
            "zero-insertion view differs for %r" % (c,)


def pin_hswish(lib):
    """Closed forms of t*hardswish(t): 0 for t <= -3, t^2 for t >= 3, and
    t^2 (t+3)/6 in between; plus the add."""
    t = np.array([-4.0, -3.0, -1.5, 0.0, 1.0, 3.0, 4.0, 2.5, -0.5])
    want = np.array([0.0, 0.0, 0.5625, 0.0, 4.0 / 6.0, 9.0, 16.0, 2.5 * 2.5 * 5.5 / 6.0,
                     0.25 * 2.5 / 6.0])
    got = ora.add_hswish(t, None, lib=lib)
    assert np.allclose(got, want, rtol=1e-15, atol=0), "hswish %r != %r" % (got, want)
    a = np.array([1.0, -1.0, 0.5, 2.0, -2.0, 0.0, 0.0, 0.5, 0.5])
    got2 = ora.add_hswish(t - a, a, lib=lib)
    assert np.allclose(got2, want, rtol=1e-14, atol=1e-15), "hswish with add %r != %r" % (got2, want)


def pin_at_matches_full(lib, n_cases=20, seed=5):
    rng = np.random.default_rng(seed)
    for t in range(n_cases):
        nd = 1 + t % 3
        c = random_case(rng, nd)
        x = rng.standard_normal([c["N"], c["C_in"]] + c["L"])
        w = rng.standard_normal([c["C_in"], c["C_out"] // c["G"]] + c["K"])
        b = rng.standard_normal(c["C_out"])
        y = ora.conv_transpose(x, w, b, c["S"], c["P"], c["OP"], c["DL"], c["G"], lib=lib)
        idx = np.arange(y.size)
        ya = ora.conv_transpose_at(x, w, idx, b, c["S"], c["P"], c["OP"], c["DL"], c["G"], lib=lib)
        assert np.allclose(ya, y.ravel(), rtol=0, atol=1e-12 * (1 + np.max(np.abs(y)))), \
            "pointwise oracle differs from the scatter oracle for %r" % (c,)


ALL_PINS = [pin_out_len, pin_worked_examples, pin_tap_counts, pin_vs_torch, pin_direct_vs_torch,
            pin_adjoint, pin_zero_insertion, pin_hswish, pin_at_matches_full]
