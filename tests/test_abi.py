"""The C-ABI library: it loads, exports every entry point include/fp8gemm.h
declares, and rejects bad arguments on the host (no GPU needed: validation
runs before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8gemm.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return ctypes.CDLL(path)


def declared_symbols():
    text = open(HEADER, encoding="utf-8").read()
    return sorted(set(re.findall(r"^FP8_API[^;(]*?\b(fp8_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("fp8_amax", "fp8_quantize_tensor", "fp8_quantize_token_group", "fp8_quantize_block",
              "fp8_quantize_mx", "fp8_gemm_tensor", "fp8_gemm_group", "fp8_gemm_mx",
              "fp8_delayed_state_update"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    import fp8_quantized_gemm_gb300 as F
    assert set(F.EXPORTED) == set(declared_symbols())


def test_options(lib):
    f = lib.fp8_set_option
    f.argtypes = [ctypes.c_int, ctypes.c_int]
    for opt in (1, 3, 4, 5, 7):  # CTA pairs, multicast, TMA-store epilogue, few rows, skinny
        assert f(opt, 0) == 0 and f(opt, 1) == 0
    assert f(6, 0) == -1 and f(6, 16) == 0 and f(6, 8) == 0  # band rows (1..4096)
    assert f(2, -1) == -1                           # negative wait bound
    assert f(2, 2_000_000) == 0
    assert f(99, 1) == -1                           # unknown option


def test_status_strings(lib):
    lib.fp8_status_string.restype = ctypes.c_char_p
    assert lib.fp8_status_string(0) == b"ok"
    assert b"misaligned" in lib.fp8_status_string(-2)
    lib.fp8_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.fp8_version()


def _gemm(lib, a=16, b=16, sa=16, sb=16, M=128, N=128, K=128, out_dt=1, c=256, ldc=128, acc=0,
          fa=0, fb=0):
    f = lib.fp8_gemm_tensor
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    return f(a, fa, b, fb, sa, sb, M, N, K, out_dt, c, ldc, acc, None)


def test_gemm_argument_validation(lib):
    assert _gemm(lib, a=None) == -1                 # null operand
    assert _gemm(lib, M=0) == -1                    # empty
    assert _gemm(lib, K=17) == -2                   # K % 16
    assert _gemm(lib, a=24) == -2                   # misaligned operand
    assert _gemm(lib, ldc=100) == -1                # ldc < N
    assert _gemm(lib, c=257) == -2                  # output not aligned to its element
    assert _gemm(lib, acc=1, out_dt=1) == -3        # accumulate needs f32 output
    assert _gemm(lib, fa=2) == -1                   # bad format enum
    # a well-formed call reaches the device check: no GPU here
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if not has_gpu:
        assert _gemm(lib) == -6


def test_group_and_mx_need_k_multiple_of_128(lib):
    g = lib.fp8_gemm_group
    g.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] + [ctypes.c_int64] * 3 + [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    assert g(16, 16, 16, 16, 0, 128, 128, 144, 256, 128, None) == -2
    assert g(16, 16, 16, 16, 7, 128, 128, 128, 256, 128, None) == -1
    q = lib.fp8_quantize_mx
    q.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert q(16, 0, 4, 96, 0, 16, 16, 16, 16, None) == -2


def test_quantize_validation(lib):
    f = lib.fp8_quantize_tensor
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int] + \
        [ctypes.c_void_p] * 7
    assert f(16, 0, 4, 12, 0, 16, None, None, 16, None, None, None) == -2   # cols % 8
    assert f(16, 0, 4, 16, 0, None, None, None, 16, None, None, None) == -1  # no scale source
    assert f(16, 3, 4, 16, 0, 16, None, None, 16, None, None, None) == -1    # bad input dtype
    d = lib.fp8_delayed_state_update
    d.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    assert d(16, 16, 16, 0, 0, None) == -1
    assert d(16, 16, 16, 1 << 20, 0, None) == -1


def test_quantize_block32_validation(lib):
    f = lib.fp8_quantize_block32
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int] + \
        [ctypes.c_void_p] * 4
    assert f(None, 0, 64, 128, 0, 16, None, 16, None) == -1   # no input
    assert f(16, 0, 64, 128, 0, 16, None, None, None) == -1   # no MX words
    assert f(16, 2, 64, 128, 0, 16, None, 16, None) == -1     # bad input dtype
    assert f(16, 0, 64, 128, 3, 16, None, 16, None) == -1     # bad format
    assert f(16, 0, 0, 128, 0, 16, None, 16, None) == -1      # empty
    assert f(16, 0, 64, 96, 0, 16, None, 16, None) == -2      # K % 128
    assert f(24, 0, 64, 128, 0, 16, None, 16, None) == -2     # misaligned weights
    assert f(16, 0, 64, 128, 0, 16, None, 20, None) == -2     # misaligned words


def _grouped(lib, **kw):
    import fp8_quantized_gemm_gb300 as F
    p = dict(a=16, b=16, sa=16, sb=16, M=128, N=128, K=128, fa=0, fb=0, out_dt=1, accumulate=0,
             c=256, ldc=128, a_layout=0, b_layout=0)
    p.update(kw)
    arr = (F.GemmProblem * 1)(F.GemmProblem(**p))
    f = lib.fp8_gemm_tensor_grouped
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    return f(ctypes.cast(arr, ctypes.c_void_p), 1, None)


def test_grouped_layout_validation(lib):
    """MN-major operands: the pitch (M or N bytes) must be a multiple of 16;
    K % 16 is required only while an operand is K-major."""
    import torch
    no_gpu = not torch.cuda.is_available()
    assert _grouped(lib, a_layout=2) == -1                        # bad layout enum
    assert _grouped(lib, a_layout=1, M=120) == -2                 # MN-major A, M % 16
    assert _grouped(lib, b_layout=1, N=200) == -2                 # MN-major B, N % 16
    assert _grouped(lib, a_layout=1, K=17) == -2                  # B still K-major
    assert _grouped(lib, K=17) == -2
    if no_gpu:
        assert _grouped(lib, a_layout=1, b_layout=1, K=17) == -6  # valid: reaches the device
        assert _grouped(lib, a_layout=1, b_layout=1, M=16, N=32, K=1) == -6
        assert _grouped(lib) == -6


def _qtensors(lib, count=1, sync=16, **kw):
    import fp8_quantized_gemm_gb300 as F
    p = dict(x=16, in_dt=0, n=1024, fmt=0, q=32, amax_out=None, scale_out=48)
    p.update(kw)
    items = [F.QuantItem(**p) for _ in range(max(count, 1))]
    arr = (F.QuantItem * len(items))(*items)
    f = lib.fp8_quantize_tensors
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return f(ctypes.cast(arr, ctypes.c_void_p), count, sync, None)


def test_quantize_tensors_validation(lib):
    import fp8_quantized_gemm_gb300 as F
    import torch
    assert _qtensors(lib, count=0) == -1                 # empty list
    assert _qtensors(lib, count=5) == -1                 # more than four tensors
    assert _qtensors(lib, sync=None) == -1               # no scratch
    assert _qtensors(lib, sync=20) == -2                 # misaligned scratch
    assert _qtensors(lib, scale_out=None) == -1          # scale is an output
    assert _qtensors(lib, amax_out=48) == -1             # amax and scale alias
    assert _qtensors(lib, x=24) == -2                    # misaligned input
    assert _qtensors(lib, fmt=3) == -1
    assert _qtensors(lib, x=None) == -1                  # a non-empty item needs data
    assert _qtensors(lib, q=None) == -1
    assert _qtensors(lib, n=-1) == -1
    items = [F.QuantItem(x=16, in_dt=0, n=64, fmt=0, q=32, amax_out=None, scale_out=48),
             F.QuantItem(x=64, in_dt=1, n=64, fmt=0, q=96, amax_out=None, scale_out=52)]
    arr = (F.QuantItem * 2)(*items)
    f = lib.fp8_quantize_tensors
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    assert f(ctypes.cast(arr, ctypes.c_void_p), 2, 16, None) == -3   # mixed input dtypes
    if not torch.cuda.is_available():
        assert _qtensors(lib) == -6
        assert _qtensors(lib, x=None, q=None, n=0) == -6   # empty item: valid
        assert _qtensors(lib, x=24, q=40, n=0) == -6       # ... read nowhere


def test_gemm_group_experts_validation(lib):
    import torch
    f = lib.fp8_gemm_group_experts
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_int] + \
        [ctypes.c_int64] * 3 + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    ok = dict(a=16, sa=16, b=16, sb=16, sfmt=1, off=16, e=8, m=1024, n=256, k=1024, c=256, ldc=256)

    def call(**kw):
        p = dict(ok)
        p.update(kw)
        return f(p["a"], p["sa"], p["b"], p["sb"], p["sfmt"], p["off"], p["e"], p["m"], p["n"],
                 p["k"], p["c"], p["ldc"], None)
    assert call(e=0) == -1                  # no experts
    assert call(e=257) == -1                # more than 256 experts
    assert call(off=None) == -1             # offsets are required
    assert call(k=1000) == -2               # K % 128
    assert call(sfmt=2) == -1
    assert call(ldc=100) == -1
    if not torch.cuda.is_available():
        assert call() == -6


def test_delayed_state_update_multi_validation(lib):
    """Batched amax-history steps: item count 1..16, the single call's checks
    per item, and no two items writing the same memory."""
    import torch
    import fp8_quantized_gemm_gb300 as F
    f = lib.fp8_delayed_state_update_multi
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]

    def call(items):
        arr = (F.DelayedItem * max(len(items), 1))(*items)
        return f(ctypes.cast(arr, ctypes.c_void_p), len(items), None)

    ok = lambda h, s, L=1024, fmt=0: F.DelayedItem(h, s, 64, L, fmt)
    assert call([]) == -1                                   # no items
    assert call([ok(4096 * (i + 1), 16 + 16 * i) for i in range(17)]) == -1  # more than 16
    assert call([F.DelayedItem(None, 16, 64, 1024, 0)]) == -1
    assert call([F.DelayedItem(4096, 16, None, 1024, 0)]) == -1
    assert call([ok(4096, 16, L=0)]) == -1
    assert call([ok(4096, 16, L=32769)]) == -1
    assert call([ok(4096, 16, fmt=2)]) == -1
    assert call([ok(4096, 16), ok(4096 + 4 * 1000, 20)]) == -1  # histories overlap
    assert call([ok(4096, 16), ok(16384, 16)]) == -1              # one scale word twice
    assert call([ok(4096, 4096 + 8)]) == -1                       # scale inside a history
    assert call([ok(4096, 16), ok(16384, 4096 + 8)]) == -1        # ... of another item
    if not torch.cuda.is_available():
        # disjoint items, one amax shared: valid (reaches the device check)
        assert call([ok(4096, 16), ok(16384, 20)]) == -6


def test_adamw_multi_codes_validation(lib):
    """The fused weight quantization of fp8_adamw_multi: a scale is required
    with codes, a valid format, 4-byte aligned codes, an amax that is neither
    the scale nor another item's amax."""
    import torch
    import fp8_quantized_gemm_gb300 as F
    f = lib.fp8_adamw_multi
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int] + \
        [ctypes.c_double] * 5 + [ctypes.c_void_p]

    def item(base, q=None, sc=None, am=None, fmt=0):
        return F.AdamwItem(base, base + 4096, base + 8192, base + 12288, None, 1024, q, sc, am,
                           fmt)

    def call(items):
        arr = (F.AdamwItem * len(items))(*items)
        return f(ctypes.cast(arr, ctypes.c_void_p), len(items), 64, 1, 1e-4, 0.9, 0.999, 1e-8,
                 0.01, None)

    assert call([item(1 << 20, q=1 << 24)]) == -1                       # no scale
    assert call([item(1 << 20, q=1 << 24, sc=16, fmt=2)]) == -1         # bad format
    assert call([item(1 << 20, q=(1 << 24) + 2, sc=16)]) == -2          # misaligned codes
    assert call([item(1 << 20, q=1 << 24, sc=16, am=16)]) == -1         # amax is the scale
    assert call([item(1 << 20, q=1 << 24, sc=16, am=32),
                 item(1 << 21, q=1 << 25, sc=20, am=32)]) == -1          # one amax twice
    if not torch.cuda.is_available():
        assert call([item(1 << 20, q=1 << 24, sc=16, am=32),
                     item(1 << 21, q=1 << 25, sc=16, am=48)]) == -6      # valid (one scale shared)
