"""Python binding of libtm (include/tm.h): argument marshalling only.

Every step of the update runs in libtm's CUDA kernels; this module converts
torch tensors to device pointers and the current CUDA stream to a handle, and
raises ``TmError`` on a non-OK status. torch is used for device memory and
streams only. There is no fallback: without the built library or without a
GPU every call raises.

The function names mirror the C ABI: tm_create, tm_forward, tm_forward_ex, tm_forward_host,
tm_forward_noalloc, tm_pair_update, tm_backward, tm_attn_create, tm_attn_forward,
tm_project, tm_project_ex, tm_x_exponent, tm_contract, tm_contract_ex, tm_finish, tm_finish_ex,
tm_project_block, tm_contract_block, tm_sync_status, tm_watchdog_selftest, tm_probe_ex2_rate, tm_set_timing,
tm_get_timing, tm_launch_count, tm_workspace_bytes, tm_ctx_info, tm_status_string, tm_last_error,
tm_destroy.

The C calls see raw pointers only, not the sizes of the buffers behind them, so every wrapper
checks the tensors it is given (shape, dtype, element count) against the ctx's shape
(tm_ctx_info) before any pointer is handed over. ``TriMul`` (the update, with ``backward``) and
``TriangleAttention`` wrap a context for convenience.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "libtm.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "tm.h")

TM_OK, TM_ERR_INVALID, TM_ERR_UNSUPPORTED, TM_ERR_OOM, TM_ERR_CUDA, TM_ERR_TIMEOUT = range(6)
TM_OUTGOING, TM_INCOMING = 0, 1
TM_F32, TM_BF16 = 0, 1
DIRECTIONS = {"outgoing": TM_OUTGOING, "incoming": TM_INCOMING}

WEIGHT_FIELDS = ("ln_in_gamma", "ln_in_beta", "w_a", "w_ga", "w_b", "w_gb", "w_g",
                 "ln_out_gamma", "ln_out_beta", "w_o")


class TmWeights(C.Structure):
    _fields_ = [(n, C.POINTER(C.c_float)) for n in WEIGHT_FIELDS]


TM_X_FP16, TM_X_FP32 = 0, 1
X_STORAGE = {"fp16": TM_X_FP16, "fp32": TM_X_FP32}


class TmOptions(C.Structure):
    _fields_ = [("block", C.c_int), ("timeout_ms", C.c_int), ("workspace_limit", C.c_size_t),
                ("x_storage", C.c_int), ("residual", C.c_int), ("reserved", C.c_int * 6)]


class TmTiming(C.Structure):
    _fields_ = [("launches", C.c_int * 12), ("ms", C.c_double * 12), ("units", C.c_longlong * 12)]


ATTN_WEIGHT_FIELDS = ("ln_gamma", "ln_beta", "w_q", "w_k", "w_v", "w_g", "w_b", "w_o")
ATTN_NODES = {"starting": 0, "ending": 1}


class TmAttnWeights(C.Structure):
    _fields_ = [(n, C.POINTER(C.c_float)) for n in ATTN_WEIGHT_FIELDS]


class TmGrads(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in WEIGHT_FIELDS]


class TmError(RuntimeError):
    def __init__(self, status, detail=""):
        self.status = status
        super().__init__(f"libtm: {tm_status_string(status)} ({status}){': ' + detail if detail else ''}")


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libtm.so and declare its prototypes. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libtm.so not found at {path}; build it with "
                           "`python -m pair_representation_boltz_b300.build`")
    lib = C.CDLL(path)
    vp, i, st = C.c_void_p, C.c_int, C.c_int
    sigs = {
        "tm_create": (st, [i, i, C.POINTER(TmWeights), C.POINTER(vp)]),
        "tm_forward": (st, [vp, vp, vp, i, i, i, vp, vp]),
        "tm_forward_ex": (st, [vp, vp, vp, i, i, i, vp, vp, C.POINTER(TmOptions)]),
        "tm_forward_host": (st, [vp, vp, vp, i, i, i, vp, vp]),
        "tm_pair_update": (st, [vp, vp, vp, i, i, vp, C.POINTER(TmOptions)]),
        "tm_forward_noalloc": (st, [vp, vp, vp, i, i, vp, vp]),
        "tm_project": (st, [vp, vp, vp, i, i, vp, vp, i, vp]),
        "tm_project_ex": (st, [vp, vp, vp, i, i, vp, vp, i, vp, vp]),
        "tm_x_exponent": (i, [vp, i]),
        "tm_contract": (st, [vp, vp, vp, i, i, i, i, i, i, i, i, vp, i, vp]),
        "tm_contract_ex": (st, [vp, vp, vp, i, i, i, i, i, i, i, i, vp, i, i, vp]),
        "tm_finish": (st, [vp, vp, i, vp, i, i, i, i, i, i, vp, vp]),
        "tm_finish_ex": (st, [vp, vp, i, i, vp, vp, i, i, i, i, i, i, vp, vp]),
        "tm_ctx_info": (st, [vp, C.POINTER(i), C.POINTER(i), C.POINTER(i)]),
        "tm_project_block": (st, [vp, vp, vp, vp, i, vp, vp, i, vp, vp]),
        "tm_contract_block": (st, [vp, vp, vp, i, i, i, vp, i, i, vp]),
        "tm_backward": (st, [vp, vp, vp, i, i, i, vp, vp, C.POINTER(TmGrads), vp, C.POINTER(TmOptions)]),
        "tm_attn_create": (st, [i, i, i, C.POINTER(TmAttnWeights), C.POINTER(vp)]),
        "tm_attn_forward": (st, [vp, vp, vp, i, i, i, vp, vp, C.POINTER(TmOptions)]),
        "tm_sync_status": (st, [vp, vp]),
        "tm_watchdog_selftest": (st, [vp, i, vp]),
        "tm_probe_ex2_rate": (st, [vp, C.POINTER(C.c_double), vp]),
        "tm_set_timing": (st, [vp, i]),
        "tm_get_timing": (st, [vp, C.POINTER(TmTiming)]),
        "tm_launch_count": (C.c_longlong, [vp]),
        "tm_workspace_bytes": (C.c_size_t, [vp]),
        "tm_status_string": (C.c_char_p, [st]),
        "tm_last_error": (C.c_char_p, [vp]),
        "tm_destroy": (None, [vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_functions(path: str = HEADER) -> list[str]:
    """Names of the functions include/tm.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tm_[a-z_]+)\s*\(", text)))


# ------------------------------------------------------------------ marshalling helpers

def _ptr(t):
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return TM_BF16
    if t.dtype == torch.float32:
        return TM_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use torch.bfloat16 or torch.float32")


def _check(ctx, status):
    if status != TM_OK:
        detail = load_library().tm_last_error(ctx).decode() if ctx else ""
        raise TmError(status, detail)


def _direction(d):
    if isinstance(d, str):
        if d not in DIRECTIONS:
            raise ValueError(f"direction must be one of {tuple(DIRECTIONS)}")
        return DIRECTIONS[d]
    return int(d)


# ------------------------------------------------------------------ argument checks
# libtm's calls receive raw pointers and cannot see how large the buffers behind them are, so the
# wrappers check every tensor against the sizes the call will touch before handing it over.

def _ctx_dims(ctx):
    """(c_z, c_hidden, layer) of a ctx (tm_ctx_info)."""
    if not ctx:
        raise TmError(TM_ERR_INVALID, "no ctx")
    cz, ch, layer = C.c_int(), C.c_int(), C.c_int()
    _check(ctx, load_library().tm_ctx_info(ctx, C.byref(cz), C.byref(ch), C.byref(layer)))
    return cz.value, ch.value, layer.value


def check_pair_tensor(name, t, c, N=None):
    """t must be a [N][N][c] tensor (N = t.shape[0] unless given); returns N."""
    if t.dim() != 3 or t.shape[0] != t.shape[1] or t.shape[2] != c or (N is not None and t.shape[0] != N):
        want = f"[{N if N is not None else 'N'}][{N if N is not None else 'N'}][{c}]"
        raise ValueError(f"{name} must have shape {want}, got {tuple(t.shape)}")
    return int(t.shape[0])


def check_like(name, t, ref, ref_name="z"):
    """t must have ref's shape and dtype."""
    if tuple(t.shape) != tuple(ref.shape) or t.dtype != ref.dtype:
        raise ValueError(f"{name} must match {ref_name} ({tuple(ref.shape)}, {ref.dtype}), "
                         f"got {tuple(t.shape)}, {t.dtype}")


def check_mask(mask, N):
    """mask: None, or a float32 vector of N token-mask values."""
    if mask is None:
        return
    if mask.dim() != 1 or mask.shape[0] != N or str(mask.dtype) != "torch.float32":
        raise ValueError(f"mask must be a float32 vector of N={N} values, got {tuple(mask.shape)}, {mask.dtype}")


def check_min_numel(name, t, n, dtype=None):
    """t must hold at least n elements (of dtype, when given)."""
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.numel() < n:
        raise ValueError(f"{name} holds {t.numel()} elements; the call touches {n}")


def grad_shapes(c_z, c_h):
    """Shape of every parameter (and of its gradient), keyed by the tm_weights member name."""
    return {"ln_in_gamma": (c_z,), "ln_in_beta": (c_z,), "w_a": (c_h, c_z), "w_ga": (c_h, c_z),
            "w_b": (c_h, c_z), "w_gb": (c_h, c_z), "w_g": (c_z, c_z), "ln_out_gamma": (c_h,),
            "ln_out_beta": (c_h,), "w_o": (c_z, c_h)}


def check_grads(grads, c_z, c_h):
    """grads: dict of float32 tensors keyed by parameter name, each in its parameter's shape."""
    shapes = grad_shapes(c_z, c_h)
    for n, t in grads.items():
        if n not in shapes:
            raise KeyError(f"unknown parameter {n!r}")
        if str(t.dtype) != "torch.float32":
            raise TypeError(f"gradient {n} must be float32")
        if tuple(t.shape) != shapes[n]:
            raise ValueError(f"gradient {n} must have shape {shapes[n]}, got {tuple(t.shape)}")


# ------------------------------------------------------------------ C-ABI mirrors

def tm_status_string(status: int) -> str:
    return load_library().tm_status_string(status).decode()


def tm_last_error(ctx) -> str:
    return load_library().tm_last_error(ctx).decode()


def tm_create(c_z: int, c_hidden: int, weights: dict):
    """Create a context from host float32 weights (dict of numpy arrays, Linear layout [out][in])."""
    lib = load_library()
    arrays = {k: np.ascontiguousarray(weights[k], dtype=np.float32) for k in WEIGHT_FIELDS}
    w = TmWeights(*[a.ctypes.data_as(C.POINTER(C.c_float)) for a in (arrays[k] for k in WEIGHT_FIELDS)])
    ctx = C.c_void_p()
    _check(None, lib.tm_create(c_z, c_hidden, C.byref(w), C.byref(ctx)))
    return ctx


def tm_destroy(ctx) -> None:
    if ctx:
        load_library().tm_destroy(ctx)


def _check_forward(ctx, z, mask, out):
    c_z, _, _ = _ctx_dims(ctx)
    N = check_pair_tensor("z", z, c_z)
    check_like("out", out, z)
    check_mask(mask, N)
    return N


def tm_forward_ex(ctx, z, mask, direction, out, stream=None, block=0, timeout_ms=0, workspace_limit=0,
                  x_storage="fp16", residual=False):
    N = _check_forward(ctx, z, mask, out)
    opt = TmOptions(block, timeout_ms, workspace_limit, X_STORAGE[x_storage], 1 if residual else 0)
    _check(ctx, load_library().tm_forward_ex(ctx, _ptr(z), _ptr(mask), N, _dtype_code(z), _direction(direction),
                                             _ptr(out), _stream(stream), C.byref(opt)))
    return out


def tm_pair_update(ctx, z, mask=None, stream=None, block=0, timeout_ms=0, workspace_limit=0, x_storage="fp16"):
    """z <- z + outgoing(z); z <- z + incoming(z), in place (z: contiguous CUDA tensor [N][N][c_z])."""
    N = _check_forward(ctx, z, mask, z)
    opt = TmOptions(block, timeout_ms, workspace_limit, X_STORAGE[x_storage], 1)
    _check(ctx, load_library().tm_pair_update(ctx, _ptr(z), _ptr(mask), N, _dtype_code(z), _stream(stream),
                                              C.byref(opt)))
    return z


def tm_forward(ctx, z, mask, direction, out, stream=None):
    N = _check_forward(ctx, z, mask, out)
    _check(ctx, load_library().tm_forward(ctx, _ptr(z), _ptr(mask), N, _dtype_code(z), _direction(direction),
                                          _ptr(out), _stream(stream)))
    return out


def tm_forward_host(ctx, z, mask, direction, out, stream=None):
    """z, mask, out: CPU tensors (pin_memory() for asynchronous copies); the stream must be synchronised
    before out is read."""
    import torch
    for t in (z, out) + ((mask,) if mask is not None else ()):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("tm_forward_host takes contiguous host tensors")
    code = TM_BF16 if z.dtype == torch.bfloat16 else TM_F32
    N = _check_forward(ctx, z, mask, out)
    _check(ctx, load_library().tm_forward_host(ctx, C.c_void_p(z.data_ptr()),
                                               C.c_void_p(mask.data_ptr()) if mask is not None else None, N, code,
                                               _direction(direction), C.c_void_p(out.data_ptr()), _stream(stream)))
    return out


def tm_forward_noalloc(ctx, z, mask, direction, out, stream=None):
    """tm_forward for bf16 z with N <= 128 whose scratch is a static array inside libtm: the call
    allocates no device memory (for callers that may not allocate; see include/tm.h)."""
    if _dtype_code(z) != TM_BF16:
        raise TypeError("tm_forward_noalloc takes bf16 z")
    N = _check_forward(ctx, z, mask, out)
    _check(ctx, load_library().tm_forward_noalloc(ctx, _ptr(z), _ptr(mask), N, _direction(direction), _ptr(out),
                                                  _stream(stream)))
    return out


def _check_project(ctx, z, mask, a, b, ld):
    c_z, c_h, _ = _ctx_dims(ctx)
    N = check_pair_tensor("z", z, c_z)
    check_mask(mask, N)
    for name, t in (("a", a), ("b", b)):
        check_min_numel(name, t, c_h * N * ld, z.dtype)
    return N


def tm_project(ctx, z, mask, a, b, ld, stream=None):
    N = _check_project(ctx, z, mask, a, b, ld)
    _check(ctx, load_library().tm_project(ctx, _ptr(z), _ptr(mask), N, _dtype_code(z), _ptr(a), _ptr(b), ld,
                                          _stream(stream)))


def tm_project_ex(ctx, z, mask, a, b, ld, zstat=None, stream=None):
    """tm_project that also writes the per-pair LayerNorm_in statistics zstat (float32 [N][N][2]) that
    the fp16-x finish step reads."""
    N = _check_project(ctx, z, mask, a, b, ld)
    if zstat is not None:
        import torch
        check_min_numel("zstat", zstat, 2 * N * N, torch.float32)
    _check(ctx, load_library().tm_project_ex(ctx, _ptr(z), _ptr(mask), N, _dtype_code(z), _ptr(a), _ptr(b), ld,
                                             _ptr(zstat), _stream(stream)))


def tm_x_exponent(ctx, N: int) -> int:
    """e of the fp16 storage of x (every value stored times 2^e) for a grid of N tokens."""
    return load_library().tm_x_exponent(ctx, N)


def _check_contract(ctx, a, b, N, ld, bi, ldx, x, x_dtype):
    _, c_h, _ = _ctx_dims(ctx)
    for name, t in (("a", a), ("b", b)):
        check_min_numel(name, t, c_h * N * ld, a.dtype)
    check_min_numel("x", x, c_h * bi * ldx, x_dtype)


def tm_contract(ctx, a, b, N, ld, direction, i0, j0, bi, bj, x, ldx, stream=None):
    import torch
    _check_contract(ctx, a, b, N, ld, bi, ldx, x, torch.float32)
    _check(ctx, load_library().tm_contract(ctx, _ptr(a), _ptr(b), N, ld, _dtype_code(a), _direction(direction),
                                           i0, j0, bi, bj, _ptr(x), ldx, _stream(stream)))


def tm_contract_ex(ctx, a, b, N, ld, direction, i0, j0, bi, bj, x, ldx, x_storage="fp16", stream=None):
    """tm_contract with x stored as fp16 times 2^tm_x_exponent(N) ("fp16", x: torch.float16) or float32."""
    import torch
    _check_contract(ctx, a, b, N, ld, bi, ldx, x, torch.float16 if x_storage == "fp16" else torch.float32)
    _check(ctx, load_library().tm_contract_ex(ctx, _ptr(a), _ptr(b), N, ld, _dtype_code(a), _direction(direction),
                                              i0, j0, bi, bj, _ptr(x), ldx, X_STORAGE[x_storage], _stream(stream)))


def _check_finish(ctx, x, ldx, z, bi, out, x_dtype):
    c_z, c_h, _ = _ctx_dims(ctx)
    N = check_pair_tensor("z", z, c_z)
    check_like("out", out, z)
    check_min_numel("x", x, c_h * bi * ldx, x_dtype)
    return N


def tm_finish(ctx, x, ldx, z, i0, j0, bi, bj, out, stream=None):
    import torch
    N = _check_finish(ctx, x, ldx, z, bi, out, torch.float32)
    _check(ctx, load_library().tm_finish(ctx, _ptr(x), ldx, _ptr(z), N, _dtype_code(z), i0, j0, bi, bj, _ptr(out),
                                         _stream(stream)))


def tm_finish_ex(ctx, x, ldx, z, i0, j0, bi, bj, out, x_storage="fp16", zstat=None, stream=None):
    """tm_finish of an x block stored as tm_contract_ex wrote it; fp16 x needs tm_project_ex's zstat."""
    import torch
    N = _check_finish(ctx, x, ldx, z, bi, out, torch.float16 if x_storage == "fp16" else torch.float32)
    if zstat is not None:
        check_min_numel("zstat", zstat, 2 * N * N, torch.float32)
    _check(ctx, load_library().tm_finish_ex(ctx, _ptr(x), ldx, X_STORAGE[x_storage], _ptr(zstat), _ptr(z), N,
                                            _dtype_code(z), i0, j0, bi, bj, _ptr(out), _stream(stream)))


def tm_project_block(ctx, z, mask_rows, mask_cols, a, b, ld, zstat=None, stream=None):
    """a, b of one B x B block of a pair representation split into blocks (row and column token masks
    of the block; None = ones)."""
    import torch
    c_z, c_h, _ = _ctx_dims(ctx)
    B = check_pair_tensor("z", z, c_z)
    check_mask(mask_rows, B)
    check_mask(mask_cols, B)
    for name, t in (("a", a), ("b", b)):
        check_min_numel(name, t, c_h * B * ld, z.dtype)
    if zstat is not None:
        check_min_numel("zstat", zstat, 2 * B * B, torch.float32)
    _check(ctx, load_library().tm_project_block(ctx, _ptr(z), _ptr(mask_rows), _ptr(mask_cols), B, _ptr(a),
                                                _ptr(b), ld, _ptr(zstat), _stream(stream)))


def tm_contract_block(ctx, a, b, B, ld, direction, x, ldx, accumulate=False, stream=None):
    """x (+)= the contraction of one pair of B x B operand blocks (float32 x [c_h][B][ldx])."""
    import torch
    _, c_h, _ = _ctx_dims(ctx)
    for name, t in (("a", a), ("b", b)):
        check_min_numel(name, t, c_h * B * ld, a.dtype)
    check_min_numel("x", x, c_h * B * ldx, torch.float32)
    _check(ctx, load_library().tm_contract_block(ctx, _ptr(a), _ptr(b), B, ld, _direction(direction), _ptr(x),
                                                 ldx, 1 if accumulate else 0, _stream(stream)))


def tm_ctx_info(ctx) -> dict:
    """{"c_z", "c_hidden", "layer"} of a ctx (layer 0: update, 1: triangle attention)."""
    c_z, c_h, layer = _ctx_dims(ctx)
    return {"c_z": c_z, "c_hidden": c_h, "layer": layer}


def tm_backward(ctx, z, mask, direction, dout, dz, grads=None, stream=None, timeout_ms=0, workspace_limit=0,
                block=0):
    """dz = dL/dz and grads[name] = dL/dW for the cotangent dout of out = update(z).

    grads: dict of contiguous float32 CUDA tensors keyed by parameter name (a missing key is not
    written), or None. dz may be dout itself. block: edge of the square blocks of the block-streamed
    schedule (bf16; 0 = automatic)."""
    g = None
    c_z, c_h, _ = _ctx_dims(ctx)
    if grads is not None:
        check_grads(grads, c_z, c_h)
    N = check_pair_tensor("z", z, c_z)
    check_like("dout", dout, z)
    check_like("dz", dz, z)
    check_mask(mask, N)
    if grads is not None:
        g = TmGrads(*[_ptr(grads[n]) if n in grads else None for n in WEIGHT_FIELDS])
    if not isinstance(block, int) or block < 0:
        raise ValueError(f"block must be a non-negative int, got {block!r}")
    opt = TmOptions(block, timeout_ms, workspace_limit, 0, 0)
    _check(ctx, load_library().tm_backward(ctx, _ptr(z), _ptr(mask), N, _dtype_code(z), _direction(direction),
                                           _ptr(dout), _ptr(dz), C.byref(g) if g is not None else None,
                                           _stream(stream), C.byref(opt)))
    return dz


def tm_attn_create(c_z: int, heads: int, c_head: int, weights: dict):
    """A triangle attention context from host float32 weights (dict of numpy arrays, [out][in])."""
    lib = load_library()
    arrays = {k: np.ascontiguousarray(weights[k], dtype=np.float32) for k in ATTN_WEIGHT_FIELDS}
    w = TmAttnWeights(*[arrays[k].ctypes.data_as(C.POINTER(C.c_float)) for k in ATTN_WEIGHT_FIELDS])
    ctx = C.c_void_p()
    _check(None, lib.tm_attn_create(c_z, heads, c_head, C.byref(w), C.byref(ctx)))
    return ctx


def tm_attn_forward(ctx, z, mask, node, out, stream=None, timeout_ms=0, workspace_limit=0):
    """out = triangle attention ("starting" or "ending" node) of bf16 z [N][N][128]."""
    N = _check_forward(ctx, z, mask, out)
    opt = TmOptions(0, timeout_ms, workspace_limit, 0, 0)
    _check(ctx, load_library().tm_attn_forward(ctx, _ptr(z), _ptr(mask), N, _dtype_code(z),
                                               ATTN_NODES[node] if isinstance(node, str) else int(node),
                                               _ptr(out), _stream(stream), C.byref(opt)))
    return out


def tm_sync_status(ctx, stream=None) -> int:
    return load_library().tm_sync_status(ctx, _stream(stream))


def tm_watchdog_selftest(ctx, timeout_ms: int, stream=None) -> None:
    _check(ctx, load_library().tm_watchdog_selftest(ctx, timeout_ms, _stream(stream)))


def tm_probe_ex2_rate(ctx, stream=None) -> float:
    """Exponentials (ex2.approx.ftz.f32) per second this device sustains (a roofline peak)."""
    r = C.c_double()
    _check(ctx, load_library().tm_probe_ex2_rate(ctx, C.byref(r), _stream(stream)))
    return r.value


def tm_set_timing(ctx, enable: bool) -> None:
    _check(ctx, load_library().tm_set_timing(ctx, 1 if enable else 0))


def tm_get_timing(ctx) -> dict:
    t = TmTiming()
    _check(ctx, load_library().tm_get_timing(ctx, C.byref(t)))
    names = ("project", "contract", "finish", "f32", "out_backward", "proj_backward", "aux_backward", "unused7",
             "attn_project", "attn_attend", "attn_out", "unused11")
    return {n: {"launches": t.launches[k], "ms": t.ms[k], "units": t.units[k]} for k, n in enumerate(names)}


def tm_launch_count(ctx) -> int:
    return load_library().tm_launch_count(ctx)


def tm_workspace_bytes(ctx) -> int:
    return load_library().tm_workspace_bytes(ctx)


# ------------------------------------------------------------------ convenience wrappers

class TriangleAttention:
    """A libtm triangle attention layer: ``TriangleAttention(weights)(z, mask, "starting")``."""

    def __init__(self, weights: dict, c_z: int = 128, heads: int = 4, c_head: int = 32):
        self.ctx = tm_attn_create(c_z, heads, c_head, weights)

    def __call__(self, z, mask=None, node="starting", out=None, stream=None, **opts):
        import torch
        if out is None:
            out = torch.empty_like(z)
        return tm_attn_forward(self.ctx, z, mask, node, out, stream, **opts)

    def close(self):
        if self.ctx:
            tm_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class TriMul:
    """A libtm context: ``TriMul(c_z, c_hidden, weights)(z, mask, "outgoing")``."""

    def __init__(self, c_z: int, c_hidden: int, weights: dict):
        self.c_z, self.c_hidden = c_z, c_hidden
        self.ctx = tm_create(c_z, c_hidden, weights)

    def __call__(self, z, mask=None, direction="outgoing", out=None, stream=None, **opts):
        import torch
        if out is None:
            out = torch.empty_like(z)
        if opts:
            return tm_forward_ex(self.ctx, z, mask, direction, out, stream, **opts)
        return tm_forward(self.ctx, z, mask, direction, out, stream)

    def backward(self, z, dout, mask=None, direction="outgoing", dz=None, stream=None, **opts):
        """(dz, grads): the gradient of sum(dout * self(z, mask, direction)) with respect to z and to
        every parameter (a dict of float32 CUDA tensors in the parameters' shapes)."""
        import torch
        if dz is None:
            dz = torch.empty_like(z)
        shapes = grad_shapes(self.c_z, self.c_hidden)
        grads = {n: torch.empty(shp, dtype=torch.float32, device=z.device) for n, shp in shapes.items()}
        tm_backward(self.ctx, z, mask, direction, dout, dz, grads, stream, **opts)
        return dz, grads

    def close(self):
        if self.ctx:
            tm_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
