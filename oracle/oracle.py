"""ctypes marshalling for the C oracle in ``ct_oracle.c`` -- TEST INFRASTRUCTURE ONLY.

Builds ``_build/libct_oracle.so`` with gcc (no fast-math, no threads) on first
use and exposes numpy-level wrappers.  Every wrapper converts its inputs to
contiguous float64 (fp32 and bf16 values widen exactly) and returns float64.
Which page passage each C function follows is stated in ``ct_oracle.c``.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ct_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libct_oracle.so")
_lock = threading.Lock()
_lib = None

_I64P = ctypes.POINTER(ctypes.c_int64)
_DP = ctypes.POINTER(ctypes.c_double)


def oracle_library_path():
    return _LIB_PATH


def build_oracle(src=_SRC, out=_LIB_PATH, force=False):
    """Compile the oracle with gcc -O2 (IEEE semantics kept: no -ffast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
           "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_MT_SRC = os.path.join(_HERE, "ct_oracle_mt.c")
_MT_LIB_PATH = os.path.join(_BUILD_DIR, "libct_oracle_mt.so")
_mt_lib = None


def build_oracle_mt(src=_MT_SRC, out=_MT_LIB_PATH, force=False):
    """Compile the all-cores baseline (pthreads) with the oracle's flags."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def host_cores():
    """Cores this process may run on (the affinity mask; os.cpu_count otherwise)."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def load_library(path):
    lib = ctypes.CDLL(path)
    lib.ora_out_len.restype = ctypes.c_int64
    lib.ora_out_len.argtypes = [ctypes.c_int64] * 6
    common = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
              _I64P, _I64P, _I64P, _I64P, _I64P, _I64P]
    lib.ora_conv_transpose.restype = ctypes.c_int
    lib.ora_conv_transpose.argtypes = common + [_DP, _DP, _DP, _DP]
    lib.ora_conv_transpose_at.restype = ctypes.c_int
    lib.ora_conv_transpose_at.argtypes = common + [_DP, _DP, _DP, ctypes.c_int64, _I64P, _DP]
    lib.ora_conv_direct.restype = ctypes.c_int
    lib.ora_conv_direct.argtypes = common + [_DP, _DP, _DP]
    lib.ora_add_hswish.restype = None
    lib.ora_add_hswish.argtypes = [ctypes.c_int64, _DP, _DP, _DP]
    return lib


def _get():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build_oracle())
    return _lib


def _dp(a):
    return a.ctypes.data_as(_DP) if a is not None else None


def _i64(seq):
    arr = (ctypes.c_int64 * len(seq))(*[int(v) for v in seq])
    return arr


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _spatial(nd, v, name):
    if np.isscalar(v):
        return [int(v)] * nd
    v = [int(t) for t in v]
    if len(v) != nd:
        raise ValueError("%s needs %d entries" % (name, nd))
    return v


def out_len(L_in, k, s=1, p=0, op=0, dl=1, lib=None):
    lib = lib or _get()
    return int(lib.ora_out_len(L_in, k, s, p, op, dl))


def _args(x, w, groups, stride, padding, output_padding, dilation):
    nd = x.ndim - 2
    if nd < 1 or nd > 3:
        raise ValueError("x must be (N, C_in, L...) with 1 to 3 spatial dims")
    N, C_in = x.shape[:2]
    K = list(w.shape[2:])
    if len(K) != nd:
        raise ValueError("w must be (C_in, C_out/groups, k...)")
    C_out = w.shape[1] * groups
    S = _spatial(nd, stride, "stride")
    P = _spatial(nd, padding, "padding")
    OP = _spatial(nd, output_padding, "output_padding")
    DL = _spatial(nd, dilation, "dilation")
    return nd, N, C_in, C_out, list(x.shape[2:]), K, S, P, OP, DL


def conv_transpose(x, w, bias=None, stride=1, padding=0, output_padding=0, dilation=1,
                   groups=1, lib=None):
    """y = ConvTranspose(x) by the scatter definition, float64."""
    lib = lib or _get()
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    nd, N, C_in, C_out, L, K, S, P, OP, DL = _args(x, w, groups, stride, padding,
                                                   output_padding, dilation)
    Lo = [out_len(L[d], K[d], S[d], P[d], OP[d], DL[d], lib=lib) for d in range(nd)]
    if min(Lo) <= 0:
        raise ValueError("non-positive output length %r" % (Lo,))
    y = np.empty([N, C_out] + Lo, dtype=np.float64)
    rc = lib.ora_conv_transpose(nd, N, C_in, C_out, groups, _i64(L), _i64(K), _i64(S), _i64(P),
                                _i64(OP), _i64(DL), _dp(x), _dp(w), _dp(bias), _dp(y))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (rc=%d)" % rc)
    return y


def conv_transpose_at(x, w, flat_idx, bias=None, stride=1, padding=0, output_padding=0,
                      dilation=1, groups=1, lib=None):
    """The definition evaluated at flat output indices only (float64)."""
    lib = lib or _get()
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    nd, N, C_in, C_out, L, K, S, P, OP, DL = _args(x, w, groups, stride, padding,
                                                   output_padding, dilation)
    idx = np.ascontiguousarray(flat_idx, dtype=np.int64)
    out = np.empty(idx.shape[0], dtype=np.float64)
    rc = lib.ora_conv_transpose_at(nd, N, C_in, C_out, groups, _i64(L), _i64(K), _i64(S),
                                   _i64(P), _i64(OP), _i64(DL), _dp(x), _dp(w), _dp(bias),
                                   idx.shape[0], idx.ctypes.data_as(_I64P), _dp(out))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (rc=%d)" % rc)
    return out


def conv_direct(z, w, in_shape, stride=1, padding=0, output_padding=0, dilation=1,
                groups=1, lib=None):
    """Direct strided conv from C_out to C_in channels (adjoint of convT)."""
    lib = lib or _get()
    z, w = _f64(z), _f64(w)
    N, C_in = in_shape[:2]
    nd = len(in_shape) - 2
    L = list(in_shape[2:])
    K = list(w.shape[2:])
    C_out = w.shape[1] * groups
    S = _spatial(nd, stride, "stride")
    P = _spatial(nd, padding, "padding")
    OP = _spatial(nd, output_padding, "output_padding")
    DL = _spatial(nd, dilation, "dilation")
    xa = np.empty(list(in_shape), dtype=np.float64)
    rc = lib.ora_conv_direct(nd, N, C_in, C_out, groups, _i64(L), _i64(K), _i64(S), _i64(P),
                             _i64(OP), _i64(DL), _dp(z), _dp(w), _dp(xa))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (rc=%d)" % rc)
    return xa


def add_hswish(y, add=None, lib=None):
    """out = t * hardswish(t), t = y + add (float64, elementwise)."""
    lib = lib or _get()
    y = _f64(y)
    a = _f64(add)
    if a is not None and a.shape != y.shape:
        raise ValueError("add must have the shape of y")
    out = np.empty_like(y)
    lib.ora_add_hswish(y.size, _dp(y), _dp(a), _dp(out))
    return out


def _get_mt():
    global _mt_lib
    with _lock:
        if _mt_lib is None:
            lib = ctypes.CDLL(build_oracle_mt())
            lib.ora_mt_conv_transpose.restype = ctypes.c_int
            lib.ora_mt_conv_transpose.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.c_int64, _I64P, _I64P, _I64P, _I64P,
                                                  _I64P, _I64P, _DP, _DP, _DP, _DP]
            _mt_lib = lib
    return _mt_lib


def conv_transpose_mt(x, w, bias=None, stride=1, padding=0, output_padding=0, dilation=1,
                      groups=1, threads=None):
    """The scatter definition on `threads` host threads (default: every core
    of the affinity mask), split by output slice (n, oc) -- the CPU baseline
    of the benchmark.  Same result as conv_transpose up to summation order."""
    lib = _get_mt()
    threads = host_cores() if threads is None else int(threads)
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    nd, N, C_in, C_out, L, K, S, P, OP, DL = _args(x, w, groups, stride, padding,
                                                   output_padding, dilation)
    Lo = [out_len(L[d], K[d], S[d], P[d], OP[d], DL[d]) for d in range(nd)]
    if min(Lo) <= 0:
        raise ValueError("non-positive output length %r" % (Lo,))
    y = np.empty([N, C_out] + Lo, dtype=np.float64)
    rc = lib.ora_mt_conv_transpose(threads, nd, N, C_in, C_out, groups, _i64(L), _i64(K), _i64(S),
                                   _i64(P), _i64(OP), _i64(DL), _dp(x), _dp(w), _dp(bias), _dp(y))
    if rc != 0:
        raise ValueError("all-cores oracle rejected the arguments (rc=%d)" % rc)
    return y
