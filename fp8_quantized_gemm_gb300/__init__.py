"""Thin Python binding of libfp8gemm.so (the C ABI in include/fp8gemm.h).

Argument marshalling only: each function takes torch CUDA tensors, passes
their device pointers, sizes and the current CUDA stream to the C entry point
of the same name, and raises ``Fp8Error`` on a non-zero status.  Every step of
the computation runs in the library's CUDA kernels; there is no CPU path.

The library must have been built (``python -c "import __graft_entry__ as g;
g.build()"`` or ``python fp8_quantized_gemm_gb300/build.py``); importing this
package without it raises ImportError.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8gemm.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libfp8gemm.so is not built (%s); run fp8_quantized_gemm_gb300/build.py" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

# enums (include/fp8gemm.h)
FP8_OK, FP8_ERR_INVALID_ARG, FP8_ERR_MISALIGNED = 0, -1, -2
FP8_ERR_UNSUPPORTED, FP8_ERR_CUDA, FP8_ERR_TIMEOUT, FP8_ERR_NO_DEVICE = -3, -4, -5, -6
FP8_ERR_SCRATCH_LIMIT = -7
IN_BF16, IN_F32 = 0, 1
E4M3, E5M2 = 0, 1
SCALE_F32, SCALE_UE8M0 = 0, 1
OUT_F32, OUT_BF16 = 0, 1
K_MAJOR, MN_MAJOR = 0, 1

_vp, _i64, _int, _d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
_SIGS = {
    "fp8_amax": [_vp, _int, _i64, _vp, _vp],
    "fp8_quantize_tensor": [_vp, _int, _i64, _i64, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "fp8_quantize_token_group": [_vp, _int, _i64, _i64, _int, _int, _vp, _vp, _vp],
    "fp8_quantize_block": [_vp, _int, _i64, _i64, _int, _int, _vp, _vp, _vp],
    "fp8_quantize_mx": [_vp, _int, _i64, _i64, _int, _vp, _vp, _vp, _vp, _vp],
    "fp8_quantize_mx1": [_vp, _int, _i64, _i64, _int, _vp, _vp, _vp, _vp],
    "fp8_quantize_block32": [_vp, _int, _i64, _i64, _int, _vp, _vp, _vp, _vp],
    "fp8_dequantize_block": [_vp, _int, _vp, _int, _i64, _i64, _vp, _vp],
    "fp8_gemm_tensor": [_vp, _int, _vp, _int, _vp, _vp, _i64, _i64, _i64, _int, _vp, _i64, _int, _vp],
    "fp8_gemm_group": [_vp, _vp, _vp, _vp, _int, _i64, _i64, _i64, _vp, _i64, _vp],
    "fp8_gemm_tensor_grouped": [_vp, _int, _vp],
    "fp8_quantize_tensors": [_vp, _int, _vp, _vp],
    "fp8_gemm_group_experts": [_vp, _vp, _vp, _vp, _int, _vp, _int, _i64, _i64, _i64, _vp, _i64, _vp],
    "fp8_gemm_group_bias": [_vp, _vp, _vp, _vp, _int, _i64, _i64, _i64, _vp, _vp, _i64, _vp],
    "fp8_amax_rows": [_vp, _int, _i64, _i64, _vp, _vp],
    "fp8_quantize_mx_rows": [_vp, _int, _i64, _i64, _int, _vp, _vp, _vp, _vp, _vp],
    "fp8_gemm_mx_rows": [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _i64, _vp],
    "fp8_gemm_mx": [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _i64, _vp],
    "fp8_gemm_group_noalloc": [_vp, _vp, _vp, _vp, _int, _i64, _i64, _i64, _vp, _i64, _vp],
    "fp8_delayed_state_update": [_vp, _vp, _vp, _i64, _int, _vp],
    "fp8_delayed_state_update_multi": [_vp, _int, _vp],
    "fp8_auto_weight_scale": [_vp, _i64, _d, _int, _vp, _vp],
    "fp8_swiglu_forward": [_vp, _vp, _vp, _i64, _vp],
    "fp8_swiglu_backward": [_vp, _vp, _vp, _vp, _vp, _i64, _vp],
    "fp8_adamw_step": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _d, _d, _d, _d, _d, _vp],
    "fp8_swiglu_forward_quantize": [_vp, _vp, _i64, _int, _vp, _vp, _vp, _vp],
    "fp8_swiglu_backward_quantize": [_vp, _vp, _vp, _i64, _int, _vp, _vp, _vp, _vp, _vp, _vp,
                                     _vp],
    "fp8_adamw_multi": [_vp, _int, _vp, _int, _d, _d, _d, _d, _d, _vp],
    "fp8_quantize_token_group32": [_vp, _int, _i64, _i64, _int, _int, _vp, _vp, _vp],
    "fp8_quantize_block32_f32": [_vp, _int, _i64, _i64, _int, _vp, _vp, _vp],
    "fp8_gemm_group32": [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp],
    "fp8_get_last_device_error": [ctypes.POINTER(ctypes.c_int), _vp],
    "fp8_set_option": [_int, _int],
}
for _name, _args in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = ctypes.c_int
_lib.fp8_status_string.argtypes = [_int]
_lib.fp8_status_string.restype = ctypes.c_char_p
_lib.fp8_version.argtypes = []
_lib.fp8_version.restype = ctypes.c_char_p

EXPORTED = tuple(_SIGS) + ("fp8_status_string", "fp8_version")


class Fp8Error(RuntimeError):
    def __init__(self, name: str, status: int):
        super().__init__("%s failed: %s (%d)" % (name, status_string(status), status))
        self.status = status


def status_string(status: int) -> str:
    return _lib.fp8_status_string(int(status)).decode()


def version() -> str:
    return _lib.fp8_version().decode()


def _p(t):
    """Device pointer of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _call(name, *args):
    rc = getattr(_lib, name)(*args)
    if rc != FP8_OK:
        raise Fp8Error(name, rc)


def _in_dt(t) -> int:
    if t.dtype == torch.bfloat16:
        return IN_BF16
    if t.dtype == torch.float32:
        return IN_F32
    raise ValueError("input must be bf16 or fp32")


# ----------------------------------------------------------------- calls --

def fp8_amax(x, amax_out, stream=None):
    _call("fp8_amax", _p(x), _in_dt(x), x.numel(), _p(amax_out), _stream(stream))


def fp8_quantize_tensor(x, fmt, q, *, amax_in=None, scale=None, scale_out=None, q_t=None,
                        amax_out=None, stream=None):
    rows, cols = x.shape
    _call("fp8_quantize_tensor", _p(x), _in_dt(x), rows, cols, fmt, _p(amax_in), _p(scale),
          _p(scale_out), _p(q), _p(q_t), _p(amax_out), _stream(stream))


def fp8_quantize_token_group(x, fmt, sfmt, q, scales, stream=None):
    m, k = x.shape
    _call("fp8_quantize_token_group", _p(x), _in_dt(x), m, k, fmt, sfmt, _p(q), _p(scales),
          _stream(stream))


def fp8_quantize_block(w, fmt, sfmt, q, scales, stream=None):
    n, k = w.shape
    _call("fp8_quantize_block", _p(w), _in_dt(w), n, k, fmt, sfmt, _p(q), _p(scales),
          _stream(stream))


def fp8_quantize_mx(x, fmt, amax, global_out, q, local, stream=None):
    r, k = x.shape
    _call("fp8_quantize_mx", _p(x), _in_dt(x), r, k, fmt, _p(amax), _p(global_out), _p(q),
          _p(local), _stream(stream))


def fp8_quantize_mx1(x, fmt, global_out, q, local, stream=None):
    r, k = x.shape
    _call("fp8_quantize_mx1", _p(x), _in_dt(x), r, k, fmt, _p(global_out), _p(q), _p(local),
          _stream(stream))


def fp8_quantize_block32(w, fmt, q, scales, local, stream=None):
    n, k = w.shape
    _call("fp8_quantize_block32", _p(w), _in_dt(w), n, k, fmt, _p(q), _p(scales), _p(local),
          _stream(stream))


def fp8_quantize_token_group32(x, fmt, sfmt, q, scales, stream=None):
    """1x32 token groups; scales group-major [ceil(K/32), M]."""
    m, k = x.shape
    _call("fp8_quantize_token_group32", _p(x), _in_dt(x), m, k, fmt, sfmt, _p(q), _p(scales),
          _stream(stream))


def fp8_quantize_block32_f32(w, fmt, q, scales, stream=None):
    """32x32 weight blocks with fp32 scales [ceil(N/32), K/32]."""
    n, k = w.shape
    _call("fp8_quantize_block32_f32", _p(w), _in_dt(w), n, k, fmt, _p(q), _p(scales),
          _stream(stream))


def fp8_gemm_group32(a, sa, b, sb, out, stream=None):
    """Per-K-group GEMM with fp32 scales of 1x32 groups and 32x32 blocks."""
    m, k = a.shape
    n = b.shape[0]
    _call("fp8_gemm_group32", _p(a), _p(sa), _p(b), _p(sb), m, n, k, _p(out), out.stride(0),
          _stream(stream))


def fp8_dequantize_block(q, fmt, scales, sfmt, out, stream=None):
    n, k = q.shape
    _call("fp8_dequantize_block", _p(q), fmt, _p(scales), sfmt, n, k, _p(out), _stream(stream))


def fp8_gemm_tensor(a, fa, b, fb, sa, sb, out, *, out_dt=None, accumulate=False, stream=None):
    m, k = a.shape
    n = b.shape[0]
    if out_dt is None:
        out_dt = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    _call("fp8_gemm_tensor", _p(a), fa, _p(b), fb, _p(sa), _p(sb), m, n, k, out_dt, _p(out),
          out.stride(0), int(bool(accumulate)), _stream(stream))


class AdamwEpilogue(ctypes.Structure):
    """fp8_adamw_epilogue_t (include/fp8gemm.h)."""
    _fields_ = [("p", _vp), ("m", _vp), ("v", _vp), ("p_bf16", _vp), ("step", _vp),
                ("lr", _d), ("beta1", _d), ("beta2", _d), ("eps", _d), ("weight_decay", _d)]


class SwigluEpilogue(ctypes.Structure):
    """fp8_swiglu_epilogue_t (include/fp8gemm.h)."""
    _fields_ = [("b_up", _vp), ("sb_up", _vp), ("u", _vp), ("q", _vp), ("fmt", _int),
                ("scale", _vp), ("amax", _vp)]


class GemmProblem(ctypes.Structure):
    """fp8_gemm_problem_t (include/fp8gemm.h)."""
    _fields_ = [("a", _vp), ("b", _vp), ("sa", _vp), ("sb", _vp), ("M", _i64), ("N", _i64),
                ("K", _i64), ("fa", _int), ("fb", _int), ("out_dt", _int), ("accumulate", _int),
                ("c", _vp), ("ldc", _i64), ("a_layout", _int), ("b_layout", _int),
                ("bias", _vp), ("adamw", ctypes.POINTER(AdamwEpilogue)),
                ("swiglu", ctypes.POINTER(SwigluEpilogue))]


def adamw_epilogue(p, m, v, p_bf16, step, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8,
                   weight_decay=0.01):
    """AdamW epilogue of a weight-gradient GEMM: the GEMM result (shape of p)
    updates p, m, v and the bf16 copy in place at t = step[0] (device int64,
    read only)."""
    assert step.dtype == torch.int64 and step.numel() == 1
    return AdamwEpilogue(_p(p), _p(m), _p(v), _p(p_bf16), _p(step), lr, beta1, beta2, eps,
                         weight_decay)


def swiglu_epilogue(b_up, sb_up, u, q, fmt, scale, amax):
    """Gated SwiGLU epilogue: the problem's b (W1) and b_up (W3) give h (the
    problem's output) and u; q receives the codes of silu(h) u under `scale`."""
    return SwigluEpilogue(_p(b_up), _p(sb_up), _p(u), _p(q), fmt, _p(scale), _p(amax))


def gemm_problem(a, fa, b, fb, sa, sb, out, *, accumulate=False, a_layout=K_MAJOR,
                 b_layout=K_MAJOR, bias=None, adamw=None, swiglu=None, n=None, ldc=None):
    """Descriptor of one per-tensor GEMM for fp8_gemm_tensor_grouped.  With
    K_MAJOR a is [M, K] and b [N, K]; with MN_MAJOR a is [K, M] and b [K, N];
    bias: optional device fp32 [N] added to every row.  adamw / swiglu:
    epilogue descriptors (adamw_epilogue / swiglu_epilogue); with adamw, `out`
    may be None (the result updates the parameters instead)."""
    m, k = a.shape if a_layout == K_MAJOR else a.shape[::-1]
    if n is None:
        n = b.shape[0] if b_layout == K_MAJOR else b.shape[1]
    if out is None:
        out_dt, c, pitch = OUT_F32, None, ldc if ldc is not None else n
    else:
        out_dt = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
        c, pitch = _p(out), out.stride(0)
    prob = GemmProblem(_p(a), _p(b), _p(sa), _p(sb), m, n, k, fa, fb, out_dt,
                       int(bool(accumulate)), c, pitch, a_layout, b_layout,
                       _p(bias) if bias is not None else None,
                       ctypes.pointer(adamw) if adamw is not None else None,
                       ctypes.pointer(swiglu) if swiglu is not None else None)
    prob._keep = (adamw, swiglu)  # the descriptors live as long as the problem
    return prob


class QuantItem(ctypes.Structure):
    """fp8_quant_item_t (include/fp8gemm.h)."""
    _fields_ = [("x", _vp), ("in_dt", _int), ("n", _i64), ("fmt", _int), ("q", _vp),
                ("amax_out", _vp), ("scale_out", _vp)]


def quant_item(x, fmt, q, scale_out, amax_out=None):
    """Descriptor of one tensor for fp8_quantize_tensors (current scaling)."""
    assert q.numel() == x.numel()
    return QuantItem(_p(x), _in_dt(x), x.numel(), fmt, _p(q),
                     _p(amax_out) if amax_out is not None else None, _p(scale_out))


QUANT_SYNC_WORDS = 8


def fp8_quantize_tensors(items, sync, stream=None):
    """Current scaling of up to four tensors in one launch (pipelined in
    order); `sync` is a device int32 tensor of QUANT_SYNC_WORDS words."""
    assert sync.numel() * sync.element_size() >= 4 * QUANT_SYNC_WORDS
    arr = (QuantItem * len(items))(*items)
    _call("fp8_quantize_tensors", ctypes.cast(arr, _vp), len(items), _p(sync), _stream(stream))


def fp8_gemm_tensor_grouped(problems, stream=None):
    arr = (GemmProblem * len(problems))(*problems)
    _call("fp8_gemm_tensor_grouped", ctypes.cast(arr, _vp), len(problems), _stream(stream))


def fp8_gemm_group(a, sa, b, sb, sfmt, out, stream=None, *, bias=None):
    m, k = a.shape
    n = b.shape[0]
    if bias is not None:
        _call("fp8_gemm_group_bias", _p(a), _p(sa), _p(b), _p(sb), sfmt, m, n, k, _p(bias),
              _p(out), out.stride(0), _stream(stream))
        return
    _call("fp8_gemm_group", _p(a), _p(sa), _p(b), _p(sb), sfmt, m, n, k, _p(out), out.stride(0),
          _stream(stream))


def fp8_gemm_group_experts(a, sa, b, sb, sfmt, offsets, out, stream=None):
    """Per-K-group GEMM of a MoE layer: a [M, K] rows grouped by expert
    (offsets: device int32 [E + 1]), b [E, N, K], sb [E, ceil(N/128), K/128]."""
    m, k = a.shape
    e, n, kb = b.shape
    assert kb == k and offsets.dtype == torch.int32 and offsets.numel() == e + 1
    _call("fp8_gemm_group_experts", _p(a), _p(sa), _p(b), _p(sb), sfmt, _p(offsets), e, m, n, k,
          _p(out), out.stride(0), _stream(stream))


def fp8_gemm_group_noalloc(a, sa, b, sb, sfmt, out, stream=None):
    """fp8_gemm_group without any device allocation (fixed in-library scratch)."""
    m, k = a.shape
    n = b.shape[0]
    _call("fp8_gemm_group_noalloc", _p(a), _p(sa), _p(b), _p(sb), sfmt, m, n, k, _p(out),
          out.stride(0), _stream(stream))


def fp8_gemm_mx(a, la, ga, b, lb, gb, out, *, out_dt=None, stream=None):
    m, k = a.shape
    n = b.shape[0]
    if out_dt is None:
        out_dt = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    _call("fp8_gemm_mx", _p(a), _p(la), _p(ga), _p(b), _p(lb), _p(gb), m, n, k, out_dt, _p(out),
          out.stride(0), _stream(stream))


def fp8_amax_rows(x, amax_out, stream=None):
    r, k = x.shape
    _call("fp8_amax_rows", _p(x), _in_dt(x), r, k, _p(amax_out), _stream(stream))


def fp8_quantize_mx_rows(x, fmt, amax_rows, global_out, q, local, stream=None):
    r, k = x.shape
    _call("fp8_quantize_mx_rows", _p(x), _in_dt(x), r, k, fmt, _p(amax_rows), _p(global_out),
          _p(q), _p(local), _stream(stream))


def fp8_gemm_mx_rows(a, la, ga, b, lb, gb, out, *, out_dt=None, stream=None):
    m, k = a.shape
    n = b.shape[0]
    if out_dt is None:
        out_dt = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    _call("fp8_gemm_mx_rows", _p(a), _p(la), _p(ga), _p(b), _p(lb), _p(gb), m, n, k, out_dt,
          _p(out), out.stride(0), _stream(stream))


def fp8_delayed_state_update(hist, scale, amax_cur, fmt, stream=None):
    _call("fp8_delayed_state_update", _p(hist), _p(scale), _p(amax_cur), hist.numel(), fmt,
          _stream(stream))


class DelayedItem(ctypes.Structure):
    """fp8_delayed_item_t (include/fp8gemm.h)."""
    _fields_ = [("hist", _vp), ("scale", _vp), ("amax_cur", _vp), ("L", ctypes.c_int64),
                ("fmt", _int)]


def delayed_item(hist, scale, amax_cur, fmt):
    return DelayedItem(_p(hist), _p(scale), _p(amax_cur), hist.numel(), fmt)


def fp8_delayed_state_update_multi(items, stream=None):
    """Several amax-history steps in one launch (items from delayed_item)."""
    arr = (DelayedItem * len(items))(*items)
    _call("fp8_delayed_state_update_multi", ctypes.cast(arr, ctypes.c_void_p), len(items),
          _stream(stream))


def fp8_auto_weight_scale(amax0, t, lr, fmt, scale_out, stream=None):
    _call("fp8_auto_weight_scale", _p(amax0), int(t), float(lr), fmt, _p(scale_out),
          _stream(stream))


def fp8_swiglu_forward(h, u, a, stream=None):
    _call("fp8_swiglu_forward", _p(h), _p(u), _p(a), h.numel(), _stream(stream))


def fp8_swiglu_backward(da, h, u, dh, du, stream=None):
    _call("fp8_swiglu_backward", _p(da), _p(h), _p(u), _p(dh), _p(du), h.numel(), _stream(stream))


def fp8_adamw_step(p, g, m, v, p_bf16, step, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8,
                   weight_decay=0.01, stream=None):
    _call("fp8_adamw_step", _p(p), _p(g), _p(m), _p(v), _p(p_bf16), p.numel(), int(step), lr,
          beta1, beta2, eps, weight_decay, _stream(stream))


def fp8_swiglu_forward_quantize(h, u, fmt, scale, q, amax_out=None, stream=None):
    """a = bf16(silu(h) * u) quantized with the given (delayed) scale into q;
    amax_out receives max |a|.  The bf16 a is not written."""
    assert q.numel() == h.numel() == u.numel()
    _call("fp8_swiglu_forward_quantize", _p(h), _p(u), h.numel(), fmt, _p(scale), _p(q),
          _p(amax_out), _stream(stream))


def fp8_swiglu_backward_quantize(da, h, u, fmt, scale_dh, scale_du, q_dh, q_du, amax_dh=None,
                                 amax_du=None, stream=None):
    """dh, du of a = silu(h) * u, each quantized with its own scale."""
    assert q_dh.numel() == q_du.numel() == h.numel() == u.numel() == da.numel()
    _call("fp8_swiglu_backward_quantize", _p(da), _p(h), _p(u), h.numel(), fmt, _p(scale_dh),
          _p(scale_du), _p(q_dh), _p(q_du), _p(amax_dh), _p(amax_du), _stream(stream))


class AdamwItem(ctypes.Structure):
    """fp8_adamw_item_t (include/fp8gemm.h)."""
    _fields_ = [("p", _vp), ("g", _vp), ("m", _vp), ("v", _vp), ("p_bf16", _vp), ("n", _i64),
                ("q", _vp), ("q_scale", _vp), ("q_amax", _vp), ("q_fmt", _int)]


def adamw_item(p, g, m, v, p_bf16=None, *, q=None, q_scale=None, q_amax=None, q_fmt=E4M3):
    """One tensor of fp8_adamw_multi; with q, also the codes of the updated
    weights (as bf16) under q_scale and their amax (q_amax, nullable)."""
    assert p.numel() == g.numel() == m.numel() == v.numel()
    assert q is None or q.numel() == p.numel()
    return AdamwItem(_p(p), _p(g), _p(m), _p(v), _p(p_bf16), p.numel(), _p(q), _p(q_scale),
                     _p(q_amax), q_fmt)


def fp8_adamw_multi(items, step, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
                    stream=None, advance=True):
    """One AdamW step over several tensors; `step` is a device int64 tensor of
    one element, incremented by the call first (the update uses the new
    value) unless advance=False (the update uses it as it stands).  No items:
    only the increment."""
    assert step.dtype == torch.int64 and step.numel() == 1
    arr = (AdamwItem * len(items))(*items) if items else None
    _call("fp8_adamw_multi", ctypes.cast(arr, _vp) if arr is not None else None, len(items),
          _p(step), int(bool(advance)), lr, beta1, beta2, eps, weight_decay, _stream(stream))


def fp8_get_last_device_error(stream=None):
    """(status, where): status 0 or FP8_ERR_TIMEOUT; clears the word."""
    where = ctypes.c_int(0)
    rc = _lib.fp8_get_last_device_error(ctypes.byref(where), _stream(stream))
    return rc, where.value


(OPT_GEMM_CTA_PAIRS, OPT_WAIT_LIMIT_US, OPT_GEMM_MULTICAST, OPT_GEMM_TMA_STORE,
 OPT_GEMM_FEW_ROWS, OPT_GEMM_BAND_ROWS, OPT_GEMM_SKINNY) = 1, 2, 3, 4, 5, 6, 7


def fp8_set_option(option, value):
    _call("fp8_set_option", int(option), int(value))


# ------------------------------------------------------------ allocation --

def mx_local_words(rows: int, k: int, device="cuda"):
    """Buffer for fp8_quantize_mx's packed local factors: uint32 [K/128, R_pad]."""
    rpad = (rows + 127) // 128 * 128
    return torch.empty((k // 128, rpad), dtype=torch.int32, device=device)
