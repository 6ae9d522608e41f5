"""Python binding of libct.so, the GB300 (sm_103a) forward transposed-convolution library.

The functions named ``ct_*`` are the C entry points of ``include/ct.h`` with
the same names and arguments; they only marshal arguments (a device pointer
may be given as an int or as a torch tensor, whose ``data_ptr()`` is used) and
raise :class:`CTError` on a non-zero status.  Every step of the computation
runs in the library's CUDA kernels.  The ``conv_transpose*`` helpers allocate
the fp32 output (and the workspace, if the chosen path needs one) with torch
and call the corresponding entry point on torch's current stream; with
``split2=True`` an fp32 call passes ``CT_F32_BF16X2`` (the opt-in two-term bf16
split of the FP32 tensor-core paths) instead of ``CT_F32``.

There is no fallback: if ``libct.so`` has not been built, every call raises.
Build it with ``python -m transposed_convolution_convtranspose_gb300.build``.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libct.so")

CT_F32 = 0
CT_BF16 = 1
CT_F32_BF16X2 = 2   # fp32 x and w; opt-in two-term bf16 split on the FP32 tensor-core paths

CT_OK, CT_ERR_ARG, CT_ERR_SHAPE, CT_ERR_ALIGN = 0, 1, 2, 3
CT_ERR_WORKSPACE, CT_ERR_UNSUPPORTED, CT_ERR_CUDA, CT_ERR_DEVICE_TIMEOUT = 4, 5, 6, 7
CT_STATUS = {0: "CT_OK", 1: "CT_ERR_ARG", 2: "CT_ERR_SHAPE", 3: "CT_ERR_ALIGN",
             4: "CT_ERR_WORKSPACE", 5: "CT_ERR_UNSUPPORTED", 6: "CT_ERR_CUDA",
             7: "CT_ERR_DEVICE_TIMEOUT"}

EXPORTED = ["ct_out_len", "ct_workspace_size_1d", "ct_workspace_size_2d", "ct_workspace_size_3d",
            "ct_forward_1d", "ct_forward_2d", "ct_forward_2d_add_hswish", "ct_forward_3d",
            "ct_forward_3d_add_hswish", "ct_path_1d", "ct_path_2d", "ct_path_3d",
            "ct_workspace_size_cl", "ct_forward_cl", "ct_path_cl", "ct_path_call",
            "ct_set_path_override", "ct_set_deterministic", "ct_get_deterministic", "ct_status_str",
            "ct_last_device_error",
            "ct_forward_3d_noalloc", "ct_selftest_wait_timeout"]

# bytes of the library-owned scratch buffer used by ct_forward_3d_noalloc
CT_NOALLOC_SCRATCH_BYTES = 48 * 1024 * 1024


class CTError(RuntimeError):
    def __init__(self, code, where=""):
        self.code = int(code)
        self.name = CT_STATUS.get(self.code, "unknown")
        msg = _status_str(self.code)
        super().__init__("%s%s" % (where + ": " if where else "", msg))


_lib = None
_load_error = None

_I = ctypes.c_int
_P = ctypes.c_void_p
_I2 = ctypes.c_int * 2
_I3 = ctypes.c_int * 3


def _setup(lib):
    lib.ct_out_len.restype = ctypes.c_int64
    lib.ct_out_len.argtypes = [ctypes.c_int64, _I, _I, _I, _I, _I]
    lib.ct_workspace_size_1d.restype = _I
    lib.ct_workspace_size_1d.argtypes = [_I] * 10 + [_I, ctypes.POINTER(ctypes.c_size_t)]
    lib.ct_workspace_size_3d.restype = _I
    lib.ct_workspace_size_3d.argtypes = [_I, _I, _I, _I3, _I3, _I, _I3, _I3, _I3, _I3, _I,
                                         ctypes.POINTER(ctypes.c_size_t)]
    lib.ct_workspace_size_2d.restype = _I
    lib.ct_workspace_size_2d.argtypes = [_I, _I, _I, _I2, _I2, _I, _I2, _I2, _I2, _I2, _I,
                                         ctypes.POINTER(ctypes.c_size_t)]
    lib.ct_forward_2d.restype = _I
    lib.ct_forward_2d.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I2, _I2, _I, _I2, _I2, _I2, _I2,
                                  _I, _P, ctypes.c_size_t, _P]
    lib.ct_forward_2d_add_hswish.restype = _I
    lib.ct_forward_2d_add_hswish.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I2, _I2, _I, _I2,
                                             _I2, _I2, _I2, _I, _P, ctypes.c_size_t, _P]
    lib.ct_path_2d.restype = ctypes.c_char_p
    lib.ct_path_2d.argtypes = [_I, _I, _I, _I2, _I2, _I, _I2, _I2, _I2, _I2, _I, _I]
    _IP = ctypes.POINTER(_I)
    lib.ct_workspace_size_cl.restype = _I
    lib.ct_workspace_size_cl.argtypes = [_I, _I, _I, _I, _IP, _IP, _I, _IP, _IP, _IP, _IP, _I,
                                         ctypes.POINTER(ctypes.c_size_t)]
    lib.ct_forward_cl.restype = _I
    lib.ct_forward_cl.argtypes = [_I, _P, _P, _P, _P, _P, _I, _I, _I, _IP, _IP, _I, _IP, _IP, _IP, _IP,
                                  _I, _P, ctypes.c_size_t, _P]
    lib.ct_path_cl.restype = ctypes.c_char_p
    lib.ct_path_cl.argtypes = [_I, _I, _I, _I, _IP, _IP, _I, _IP, _IP, _IP, _IP, _I, _I]
    lib.ct_path_call.restype = ctypes.c_char_p
    lib.ct_path_call.argtypes = [_I, _I, _I, _I, _I, _IP, _IP, _I, _IP, _IP, _IP, _IP, _I, _I, ctypes.c_size_t]
    lib.ct_forward_1d.restype = _I
    lib.ct_forward_1d.argtypes = [_P, _P, _P, _P] + [_I] * 10 + [_I, _P, ctypes.c_size_t, _P]
    lib.ct_forward_3d.restype = _I
    lib.ct_forward_3d.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I3, _I3, _I, _I3, _I3, _I3, _I3,
                                  _I, _P, ctypes.c_size_t, _P]
    lib.ct_forward_3d_add_hswish.restype = _I
    lib.ct_forward_3d_add_hswish.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I3, _I3, _I, _I3,
                                             _I3, _I3, _I3, _I, _P, ctypes.c_size_t, _P]
    lib.ct_forward_3d_noalloc.restype = _I
    lib.ct_forward_3d_noalloc.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I3, _I3, _I, _I3, _I3, _I3,
                                          _I3, _I, _P]
    lib.ct_path_1d.restype = ctypes.c_char_p
    lib.ct_path_1d.argtypes = [_I] * 10 + [_I]
    lib.ct_path_3d.restype = ctypes.c_char_p
    lib.ct_path_3d.argtypes = [_I, _I, _I, _I3, _I3, _I, _I3, _I3, _I3, _I3, _I, _I]
    lib.ct_set_path_override.restype = None
    lib.ct_set_path_override.argtypes = [_I]
    lib.ct_set_deterministic.restype = None
    lib.ct_set_deterministic.argtypes = [_I]
    lib.ct_get_deterministic.restype = _I
    lib.ct_get_deterministic.argtypes = []
    lib.ct_status_str.restype = ctypes.c_char_p
    lib.ct_status_str.argtypes = [_I]
    lib.ct_last_device_error.restype = _I
    lib.ct_last_device_error.argtypes = [_P]
    lib.ct_selftest_wait_timeout.restype = _I
    lib.ct_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _P]
    return lib


def load(path=LIB_PATH):
    """Load (or return the already loaded) libct.so; raises if it is missing."""
    global _lib, _load_error
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libct.so is not built (%s); run `python -m "
                           "transposed_convolution_convtranspose_gb300.build`" % path)
    _lib = _setup(ctypes.CDLL(path))
    return _lib


def _status_str(code):
    try:
        return load().ct_status_str(int(code)).decode()
    except Exception:
        return CT_STATUS.get(int(code), "status %d" % int(code))


def _ptr(v):
    if v is None:
        return None
    if isinstance(v, int):
        return v or None
    return v.data_ptr() or None   # torch tensor


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None  # torch.cuda.Stream


def _i2(v):
    v = tuple(int(t) for t in v)
    if len(v) != 2:
        raise ValueError("expected 2 values (H, W)")
    return _I2(*v)


def _ivec(v):
    v = tuple(int(t) for t in v)
    if not 1 <= len(v) <= 3:
        raise ValueError("expected 1 to 3 values")
    return (_I * len(v))(*v)


def _i3(v):
    v = tuple(int(t) for t in v)
    if len(v) != 3:
        raise ValueError("expected 3 values (D, H, W)")
    return _I3(*v)


def _check(code, where):
    if code != 0:
        raise CTError(code, where)


# ------------------------------------------------------------------ raw ABI
def ct_out_len(L_in, k, s, p, op, dl):
    return int(load().ct_out_len(int(L_in), int(k), int(s), int(p), int(op), int(dl)))


def ct_workspace_size_1d(N, C_in, C_out, L_in, k, groups, stride, padding, output_padding,
                         dilation, dtype):
    out = ctypes.c_size_t(0)
    _check(load().ct_workspace_size_1d(N, C_in, C_out, L_in, k, groups, stride, padding,
                                       output_padding, dilation, dtype, ctypes.byref(out)),
           "ct_workspace_size_1d")
    return int(out.value)


def ct_workspace_size_3d(N, C_in, C_out, in_dhw, k_dhw, groups, stride, padding,
                         output_padding, dilation, dtype):
    out = ctypes.c_size_t(0)
    _check(load().ct_workspace_size_3d(N, C_in, C_out, _i3(in_dhw), _i3(k_dhw), groups,
                                       _i3(stride), _i3(padding), _i3(output_padding),
                                       _i3(dilation), dtype, ctypes.byref(out)),
           "ct_workspace_size_3d")
    return int(out.value)


def ct_forward_1d(x, w, bias, y, N, C_in, C_out, L_in, k, groups, stride, padding,
                  output_padding, dilation, dtype, workspace=None, ws_bytes=0, stream=None):
    _check(load().ct_forward_1d(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), N, C_in, C_out, L_in, k,
                                groups, stride, padding, output_padding, dilation, dtype,
                                _ptr(workspace), int(ws_bytes), _stream(stream)),
           "ct_forward_1d")


def ct_workspace_size_2d(N, C_in, C_out, in_hw, k_hw, groups, stride, padding, output_padding,
                         dilation, dtype):
    n = ctypes.c_size_t(0)
    _check(load().ct_workspace_size_2d(N, C_in, C_out, _i2(in_hw), _i2(k_hw), groups, _i2(stride),
                                       _i2(padding), _i2(output_padding), _i2(dilation), dtype,
                                       ctypes.byref(n)),
           "ct_workspace_size_2d")
    return int(n.value)


def ct_forward_2d(x, w, bias, y, N, C_in, C_out, in_hw, k_hw, groups, stride, padding,
                  output_padding, dilation, dtype, workspace=None, ws_bytes=0, stream=None):
    _check(load().ct_forward_2d(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), N, C_in, C_out,
                                _i2(in_hw), _i2(k_hw), groups, _i2(stride), _i2(padding),
                                _i2(output_padding), _i2(dilation), dtype, _ptr(workspace),
                                ws_bytes, _stream(stream)),
           "ct_forward_2d")


def ct_forward_2d_add_hswish(x, w, bias, add, y, N, C_in, C_out, in_hw, k_hw, groups, stride,
                             padding, output_padding, dilation, dtype, workspace=None, ws_bytes=0,
                             stream=None):
    _check(load().ct_forward_2d_add_hswish(_ptr(x), _ptr(w), _ptr(bias), _ptr(add), _ptr(y), N,
                                           C_in, C_out, _i2(in_hw), _i2(k_hw), groups, _i2(stride),
                                           _i2(padding), _i2(output_padding), _i2(dilation), dtype,
                                           _ptr(workspace), ws_bytes, _stream(stream)),
           "ct_forward_2d_add_hswish")


def ct_forward_3d(x, w, bias, y, N, C_in, C_out, in_dhw, k_dhw, groups, stride, padding,
                  output_padding, dilation, dtype, workspace=None, ws_bytes=0, stream=None):
    _check(load().ct_forward_3d(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), N, C_in, C_out,
                                _i3(in_dhw), _i3(k_dhw), groups, _i3(stride), _i3(padding),
                                _i3(output_padding), _i3(dilation), dtype, _ptr(workspace),
                                int(ws_bytes), _stream(stream)),
           "ct_forward_3d")


def ct_forward_3d_add_hswish(x, w, bias, add, y, N, C_in, C_out, in_dhw, k_dhw, groups, stride,
                             padding, output_padding, dilation, dtype, workspace=None,
                             ws_bytes=0, stream=None):
    _check(load().ct_forward_3d_add_hswish(_ptr(x), _ptr(w), _ptr(bias), _ptr(add), _ptr(y), N,
                                           C_in, C_out, _i3(in_dhw), _i3(k_dhw), groups,
                                           _i3(stride), _i3(padding), _i3(output_padding),
                                           _i3(dilation), dtype, _ptr(workspace), int(ws_bytes),
                                           _stream(stream)),
           "ct_forward_3d_add_hswish")


def ct_forward_3d_noalloc(x, w, bias, y, N, C_in, C_out, in_dhw, k_dhw, groups, stride, padding,
                          output_padding, dilation, dtype, stream=None):
    """ct_forward_3d for callers that cannot allocate: the bf16 tensor-core
    path with the library's own fixed scratch buffer instead of a workspace."""
    _check(load().ct_forward_3d_noalloc(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), N, C_in, C_out,
                                        _i3(in_dhw), _i3(k_dhw), groups, _i3(stride), _i3(padding),
                                        _i3(output_padding), _i3(dilation), dtype, _stream(stream)),
           "ct_forward_3d_noalloc")


def ct_path_1d(N, C_in, C_out, L_in, k, groups, stride, padding, output_padding, dilation, dtype):
    r = load().ct_path_1d(N, C_in, C_out, L_in, k, groups, stride, padding, output_padding,
                          dilation, dtype)
    return None if r is None else r.decode()


def ct_workspace_size_cl(nd, N, C_in, C_out, in_size, k, groups, stride, padding, output_padding,
                         dilation, dtype):
    n = ctypes.c_size_t(0)
    _check(load().ct_workspace_size_cl(nd, N, C_in, C_out, _ivec(in_size), _ivec(k), groups,
                                       _ivec(stride), _ivec(padding), _ivec(output_padding),
                                       _ivec(dilation), dtype, ctypes.byref(n)),
           "ct_workspace_size_cl")
    return int(n.value)


def ct_forward_cl(nd, x, w, bias, add, y, N, C_in, C_out, in_size, k, groups, stride, padding,
                  output_padding, dilation, dtype, workspace=None, ws_bytes=0, stream=None):
    _check(load().ct_forward_cl(nd, _ptr(x), _ptr(w), _ptr(bias), _ptr(add), _ptr(y), N, C_in, C_out,
                                _ivec(in_size), _ivec(k), groups, _ivec(stride), _ivec(padding),
                                _ivec(output_padding), _ivec(dilation), dtype, _ptr(workspace),
                                ws_bytes, _stream(stream)),
           "ct_forward_cl")


def ct_path_cl(nd, N, C_in, C_out, in_size, k, groups, stride, padding, output_padding, dilation,
               dtype, fused=False):
    r = load().ct_path_cl(nd, N, C_in, C_out, _ivec(in_size), _ivec(k), groups, _ivec(stride),
                          _ivec(padding), _ivec(output_padding), _ivec(dilation), dtype,
                          int(bool(fused)))
    return None if r is None else r.decode()


def ct_path_call(nd, channels_last, N, C_in, C_out, in_size, k, groups, stride, padding, output_padding,
                 dilation, dtype, fused, ws_bytes):
    """Kernel family a forward call with exactly ws_bytes of workspace launches
    (None if the arguments are invalid or the call would fail with
    CT_ERR_WORKSPACE)."""
    r = load().ct_path_call(nd, int(bool(channels_last)), N, C_in, C_out, _ivec(in_size), _ivec(k), groups,
                            _ivec(stride), _ivec(padding), _ivec(output_padding), _ivec(dilation), dtype,
                            int(bool(fused)), int(ws_bytes))
    return r.decode() if r is not None else None


def ct_path_2d(N, C_in, C_out, in_hw, k_hw, groups, stride, padding, output_padding, dilation,
               dtype, fused=False):
    r = load().ct_path_2d(N, C_in, C_out, _i2(in_hw), _i2(k_hw), groups, _i2(stride),
                          _i2(padding), _i2(output_padding), _i2(dilation), dtype, int(bool(fused)))
    return None if r is None else r.decode()


def ct_path_3d(N, C_in, C_out, in_dhw, k_dhw, groups, stride, padding, output_padding, dilation,
               dtype, fused=False):
    r = load().ct_path_3d(N, C_in, C_out, _i3(in_dhw), _i3(k_dhw), groups, _i3(stride),
                          _i3(padding), _i3(output_padding), _i3(dilation), dtype, int(bool(fused)))
    return None if r is None else r.decode()


def ct_set_path_override(mode):
    load().ct_set_path_override(int(mode))


def ct_set_deterministic(on):
    """Bitwise-reproducible results on every path (process-wide); see include/ct.h."""
    load().ct_set_deterministic(int(bool(on)))


def ct_get_deterministic():
    return bool(load().ct_get_deterministic())


def ct_status_str(code):
    return load().ct_status_str(int(code)).decode()


def ct_last_device_error(stream=None):
    code = load().ct_last_device_error(_stream(stream))
    _check(code, "ct_last_device_error")


def ct_last_device_error_code(stream=None):
    """The status code of ct_last_device_error (synchronises, reads and clears)."""
    return int(load().ct_last_device_error(_stream(stream)))


def ct_selftest_wait_timeout(limit_ns, stream=None):
    _check(load().ct_selftest_wait_timeout(int(limit_ns), _stream(stream)), "ct_selftest_wait_timeout")


# ------------------------------------------------------------------ helpers (torch allocation)
def _triple(v):
    if isinstance(v, int):
        return (v, v, v)
    v = tuple(int(t) for t in v)
    if len(v) != 3:
        raise ValueError("expected an int or 3 values")
    return v


def _need(t, name):
    if t is None:
        return
    if not t.is_cuda or not t.is_contiguous():
        raise CTError(1, "%s must be a contiguous CUDA tensor" % name)


def _dtype_code(t, split2=False):
    import torch
    if t.dtype == torch.float32:
        return CT_F32_BF16X2 if split2 else CT_F32
    if t.dtype == torch.bfloat16:
        return CT_BF16
    raise TypeError("x and w must be float32 or bfloat16, got %s" % t.dtype)


def _workspace(nbytes, device):
    import torch
    if nbytes == 0:
        return None
    # 256-byte aligned: torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def conv_transpose1d(x, w, bias=None, stride=1, padding=0, output_padding=0, dilation=1,
                     groups=1, out=None, split2=False):
    import torch
    for t, nm in ((x, "x"), (w, "w"), (bias, "bias"), (out, "out")):
        _need(t, nm)
    N, C_in, L_in = x.shape
    k = w.shape[2]
    C_out = w.shape[1] * groups
    dt = _dtype_code(x, split2)
    L_out = ct_out_len(L_in, k, stride, padding, output_padding, dilation)
    if L_out < 1:
        raise CTError(2, "conv_transpose1d")
    y = out if out is not None else torch.empty((N, C_out, L_out), dtype=torch.float32,
                                                device=x.device)
    nb = ct_workspace_size_1d(N, C_in, C_out, L_in, k, groups, stride, padding, output_padding,
                              dilation, dt)
    ws = _workspace(nb, x.device)
    ct_forward_1d(x, w, bias, y, N, C_in, C_out, L_in, k, groups, stride, padding,
                  output_padding, dilation, dt, ws, nb, torch.cuda.current_stream(x.device))
    return y


def _out3(x, w, groups, stride, padding, output_padding, dilation):
    S, P, OP, D = _triple(stride), _triple(padding), _triple(output_padding), _triple(dilation)
    K = tuple(w.shape[2:])
    L = tuple(x.shape[2:])
    Lo = tuple(ct_out_len(L[i], K[i], S[i], P[i], OP[i], D[i]) for i in range(3))
    if min(Lo) < 1:
        raise CTError(2, "conv_transpose3d")
    return S, P, OP, D, K, L, Lo


def conv_transpose3d(x, w, bias=None, stride=1, padding=0, output_padding=0, dilation=1,
                     groups=1, out=None, split2=False):
    import torch
    for t, nm in ((x, "x"), (w, "w"), (bias, "bias"), (out, "out")):
        _need(t, nm)
    N, C_in = x.shape[:2]
    C_out = w.shape[1] * groups
    dt = _dtype_code(x, split2)
    S, P, OP, D, K, L, Lo = _out3(x, w, groups, stride, padding, output_padding, dilation)
    y = out if out is not None else torch.empty((N, C_out) + Lo, dtype=torch.float32,
                                                device=x.device)
    nb = ct_workspace_size_3d(N, C_in, C_out, L, K, groups, S, P, OP, D, dt)
    ws = _workspace(nb, x.device)
    ct_forward_3d(x, w, bias, y, N, C_in, C_out, L, K, groups, S, P, OP, D, dt, ws, nb,
                  torch.cuda.current_stream(x.device))
    return y


def conv_transpose3d_add_hswish(x, w, bias, add, stride=1, padding=0, output_padding=0,
                                dilation=1, groups=1, out=None, split2=False):
    import torch
    for t, nm in ((x, "x"), (w, "w"), (bias, "bias"), (add, "add"), (out, "out")):
        _need(t, nm)
    N, C_in = x.shape[:2]
    C_out = w.shape[1] * groups
    dt = _dtype_code(x, split2)
    S, P, OP, D, K, L, Lo = _out3(x, w, groups, stride, padding, output_padding, dilation)
    if tuple(add.shape) != (N, C_out) + Lo or add.dtype != torch.float32:
        raise CTError(1, "conv_transpose3d_add_hswish: add must be fp32 with the output's shape")
    y = out if out is not None else torch.empty_like(add)
    nb = ct_workspace_size_3d(N, C_in, C_out, L, K, groups, S, P, OP, D, dt)
    ws = _workspace(nb, x.device)
    ct_forward_3d_add_hswish(x, w, bias, add, y, N, C_in, C_out, L, K, groups, S, P, OP, D, dt,
                             ws, nb, torch.cuda.current_stream(x.device))
    return y


def _pair(v):
    if isinstance(v, int):
        return (v, v)
    v = tuple(int(t) for t in v)
    if len(v) != 2:
        raise ValueError("expected an int or 2 values")
    return v


def _out2(x, w, stride, padding, output_padding, dilation):
    S, P, OP, D = _pair(stride), _pair(padding), _pair(output_padding), _pair(dilation)
    K = tuple(w.shape[2:])
    L = tuple(x.shape[2:])
    Lo = tuple(ct_out_len(L[i], K[i], S[i], P[i], OP[i], D[i]) for i in range(2))
    if min(Lo) < 1:
        raise CTError(2, "conv_transpose2d")
    return S, P, OP, D, K, L, Lo


def conv_transpose2d(x, w, bias=None, stride=1, padding=0, output_padding=0, dilation=1,
                     groups=1, out=None, split2=False):
    import torch
    for t, nm in ((x, "x"), (w, "w"), (bias, "bias"), (out, "out")):
        _need(t, nm)
    N, C_in = x.shape[:2]
    C_out = w.shape[1] * groups
    dt = _dtype_code(x, split2)
    S, P, OP, D, K, L, Lo = _out2(x, w, stride, padding, output_padding, dilation)
    y = out if out is not None else torch.empty((N, C_out) + Lo, dtype=torch.float32,
                                                device=x.device)
    nb = ct_workspace_size_2d(N, C_in, C_out, L, K, groups, S, P, OP, D, dt)
    ws = _workspace(nb, x.device)
    ct_forward_2d(x, w, bias, y, N, C_in, C_out, L, K, groups, S, P, OP, D, dt, ws, nb,
                  torch.cuda.current_stream(x.device))
    return y


def conv_transpose2d_add_hswish(x, w, bias, add, stride=1, padding=0, output_padding=0,
                                dilation=1, groups=1, out=None, split2=False):
    import torch
    for t, nm in ((x, "x"), (w, "w"), (bias, "bias"), (add, "add"), (out, "out")):
        _need(t, nm)
    N, C_in = x.shape[:2]
    C_out = w.shape[1] * groups
    dt = _dtype_code(x, split2)
    S, P, OP, D, K, L, Lo = _out2(x, w, stride, padding, output_padding, dilation)
    if tuple(add.shape) != (N, C_out) + Lo or add.dtype != torch.float32:
        raise CTError(1, "conv_transpose2d_add_hswish: add must be fp32 with the output's shape")
    y = out if out is not None else torch.empty_like(add)
    nb = ct_workspace_size_2d(N, C_in, C_out, L, K, groups, S, P, OP, D, dt)
    ws = _workspace(nb, x.device)
    ct_forward_2d_add_hswish(x, w, bias, add, y, N, C_in, C_out, L, K, groups, S, P, OP, D, dt,
                             ws, nb, torch.cuda.current_stream(x.device))
    return y


def conv_transpose_cl(x, w, bias=None, add=None, stride=1, padding=0, output_padding=0, dilation=1,
                      groups=1, out=None, split2=False):
    """Transposed convolution of a channels-last x (N, spatial..., C_in), 1 to 3
    spatial dimensions; returns y (N, spatial out..., C_out) fp32.  With add
    (channels-last, y's shape) the fused add + t*hardswish(t) epilogue."""
    import torch
    for t, nm in ((x, "x"), (w, "w"), (bias, "bias"), (add, "add"), (out, "out")):
        _need(t, nm)
    nd = x.dim() - 2
    if not 1 <= nd <= 3 or w.dim() != nd + 2:
        raise CTError(1, "conv_transpose_cl: x must be (N, spatial..., C_in), 1 to 3 spatial dims")

    def vec(v):
        v = (v,) * nd if isinstance(v, int) else tuple(int(t) for t in v)
        if len(v) != nd:
            raise ValueError("expected an int or %d values" % nd)
        return v
    S, P, OP, D = vec(stride), vec(padding), vec(output_padding), vec(dilation)
    N, C_in = x.shape[0], x.shape[-1]
    L = tuple(x.shape[1:-1])
    K = tuple(w.shape[2:])
    C_out = w.shape[1] * groups
    dt = _dtype_code(x, split2)
    Lo = tuple(ct_out_len(L[i], K[i], S[i], P[i], OP[i], D[i]) for i in range(nd))
    if min(Lo) < 1:
        raise CTError(2, "conv_transpose_cl")
    shape = (N,) + Lo + (C_out,)
    if add is not None and (tuple(add.shape) != shape or add.dtype != torch.float32):
        raise CTError(1, "conv_transpose_cl: add must be fp32 with the output's shape")
    y = out if out is not None else torch.empty(shape, dtype=torch.float32, device=x.device)
    nb = ct_workspace_size_cl(nd, N, C_in, C_out, L, K, groups, S, P, OP, D, dt)
    ws = _workspace(nb, x.device)
    ct_forward_cl(nd, x, w, bias, add, y, N, C_in, C_out, L, K, groups, S, P, OP, D, dt, ws, nb,
                  torch.cuda.current_stream(x.device))
    return y
