"""ctypes binding of the C ABI in ``include/snip.h`` (library ``_build/libsnip.so``).

The ``snip_*`` functions below take the same arguments as their C
counterparts (device pointers as ints, sizes, enums, the CUDA stream handle)
and raise :class:`SnipError` on a non-OK status.  The lower-case helpers
(``quantize_nvfp4`` ...) only allocate the output tensors with PyTorch and
marshal pointers: every step of the computation runs in the library's CUDA
kernels.  There is no fallback: if the library is missing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsnip.so")

SNIP_OK, SNIP_ERR_INVALID_ARG, SNIP_ERR_SHAPE, SNIP_ERR_ALIGN, SNIP_ERR_NONFINITE, SNIP_ERR_TIMEOUT, \
    SNIP_ERR_CUDA, SNIP_ERR_UNSUPPORTED_DEVICE, SNIP_ERR_WORKSPACE = range(9)
FP8, NVFP4, MXFP4, FP8_E5M2, FP8_E5M2_GRAD = 0, 1, 2, 3, 4
NVFP4_B32, NVFP4_B64, NVFP4_B128 = 5, 6, 7     # NVFP4 with 32 / 64 / 128 elements per scale
NVFP4_BLOCK = {NVFP4: 16, NVFP4_B32: 32, NVFP4_B64: 64, NVFP4_B128: 128}
RTN, SR = 0, 1
ALONG_COLS, ALONG_ROWS = 0, 1
ROWMAJOR, MMA = 0, 1
TAG_X_FWD, TAG_W_FWD, TAG_DY_DGRAD, TAG_WT_DGRAD, TAG_DYT_WGRAD, TAG_XT_WGRAD = range(6)
WS_HEADER_BYTES = 256
STATS_NVALS = 8

# every symbol include/snip.h declares
EXPORTS = (
    "snip_status_string", "snip_version", "snip_device_check", "snip_workspace_init", "snip_workspace_status",
    "snip_quantize_workspace_size", "snip_amax", "snip_tensor_scales", "snip_tensor_scales_multi",
    "snip_tensor_scales_noalloc",
    "snip_wait_check", "snip_quantize_part", "snip_quantize_nvfp4", "snip_quantize_nvfp4_block", "snip_quantize_fp8", "snip_quantize_mxfp4",
    "snip_quantize_e5m2",
    "snip_quantized_bytes", "snip_gemm", "snip_plan_create", "snip_plan_set_rounding", "snip_plan_get",
    "snip_plan_destroy", "snip_qlinear_workspace_size", "snip_qlinear_fwd", "snip_qlinear_bwd",
    "snip_qlinear_fwd_multi_workspace_size", "snip_qlinear_fwd_multi", "snip_qlinear_bwd_chain",
    "snip_qlinear_bwd_q",
    "snip_quant_stats", "snip_quantize_stats", "snip_stats_finalize", "snip_plan_costs", "snip_plan_select",
    "snip_dw_noise_workspace_size", "snip_dw_noise", "snip_dw_noise_finalize", "snip_gemm_requant",
)


class SnipError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else status_string(status))


class SnipRequant(ctypes.Structure):
    _fields_ = [("g_in", ctypes.c_void_p), ("rnd", ctypes.c_int), ("seed", ctypes.c_uint64),
                ("stream_id", ctypes.c_uint64), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("amax_out", ctypes.c_void_p), ("rnd_t", ctypes.c_int), ("stream_id_t", ctypes.c_uint64),
                ("codes_t", ctypes.c_void_p), ("scales_t", ctypes.c_void_p)]


class SnipStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in
                ("sum_x2", "nvfp4_err2", "fp8_err2", "nvfp4_sr_var", "fp8_sr_var", "amax", "count",
                 "ratio_nvfp4", "ratio_fp8")] + [("below_sqrt3_nvfp4", ctypes.c_int), ("below_sqrt3_fp8", ctypes.c_int)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libsnip not built ({path} missing): run sub_byte_mixed_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i64, u64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_size_t
    szp = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "snip_status_string": (ctypes.c_char_p, [i32]),
        "snip_version": (i32, []),
        "snip_device_check": (i32, []),
        "snip_workspace_init": (i32, [vp, sz, vp]),
        "snip_workspace_status": (i32, [vp, vp, ctypes.POINTER(ctypes.c_int)]),
        "snip_quantize_workspace_size": (sz, [i64, i64]),
        "snip_amax": (i32, [vp, i64, vp, vp, sz, vp]),
        "snip_tensor_scales": (i32, [vp, i64, vp, vp, sz, vp]),
        "snip_tensor_scales_noalloc": (i32, [vp, i64, vp, vp]),
        "snip_tensor_scales_multi": (i32, [i32, vp, vp, vp, vp, sz, vp]),
        "snip_wait_check": (i32, [u64, vp, vp, sz, vp]),
        "snip_quantize_part": (i32, [i32, vp, i64, i64, i32, i32, u64, u64, u64, vp, i32, vp, vp, vp, vp, sz, vp]),
        "snip_quantize_nvfp4": (i32, [vp, i64, i64, i32, i32, u64, u64, vp, i32, vp, vp, vp, vp, vp, sz, vp]),
        "snip_quantize_nvfp4_block": (i32, [vp, i64, i64, i32, i32, u64, u64, vp, i32, i32, vp, vp, vp, vp, sz,
                                            vp]),
        "snip_quantize_fp8": (i32, [vp, i64, i64, i32, i32, u64, u64, vp, i32, vp, vp, vp, sz, vp]),
        "snip_quantize_mxfp4": (i32, [vp, i64, i64, i32, i32, u64, u64, i32, vp, vp, vp, sz, vp]),
        "snip_quantize_e5m2": (i32, [vp, i64, i64, i32, i32, u64, u64, vp, i32, vp, vp, vp, sz, vp]),
        "snip_quantized_bytes": (i32, [i32, i32, i64, i64, szp, szp]),
        "snip_gemm": (i32, [i32, vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp, sz, vp]),
        "snip_plan_create": (i32, [i32, ctypes.POINTER(ctypes.c_int), u64, ctypes.POINTER(vp)]),
        "snip_plan_set_rounding": (i32, [vp, i32, i32, i32]),
        "snip_plan_get": (i32, [vp, i32, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_uint64)]),
        "snip_plan_destroy": (None, [vp]),
        "snip_qlinear_workspace_size": (sz, [vp, i32, i64, i64, i64]),
        "snip_qlinear_fwd": (i32, [vp, i32, vp, vp, i64, i64, i64, vp, vp, vp, sz, vp]),
        "snip_qlinear_bwd": (i32, [vp, i32, vp, vp, vp, i64, i64, i64, vp, vp, vp, vp, sz, vp]),
        "snip_qlinear_fwd_multi_workspace_size": (sz, [vp, i32, vp, i64, i64, vp]),
        "snip_qlinear_fwd_multi": (i32, [vp, i32, vp, vp, vp, i64, i64, vp, vp, vp, vp, vp, sz, vp]),
        "snip_qlinear_bwd_chain": (i32, [vp, i32, i32, vp, vp, vp, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                         vp, vp, sz, vp]),
        "snip_qlinear_bwd_q": (i32, [vp, i32, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, vp, vp, sz, vp]),
        "snip_quantize_stats": (i32, [i32, vp, i64, i64, i32, u64, u64, vp, i32, vp, vp, vp, vp, sz, vp]),
        "snip_quant_stats": (i32, [vp, i64, i64, i32, u64, u64, vp, vp, vp, vp, vp, sz, vp]),
        "snip_stats_finalize": (i32, [vp, ctypes.POINTER(SnipStats)]),
        "snip_plan_costs": (i32, [i32, vp, vp, vp]),
        "snip_dw_noise_workspace_size": (sz, [i64, i64]),
        "snip_gemm_requant": (i32, [i32, vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, i64,
                                    ctypes.POINTER(SnipRequant), vp, sz, vp]),
        "snip_dw_noise": (i32, [vp, vp, i64, i64, i64, vp, vp, vp, sz, vp]),
        "snip_dw_noise_finalize": (i32, [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
        "snip_plan_select": (i32, [i32, vp, vp, vp, ctypes.c_double, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().snip_status_string(int(status)).decode()


def check(status: int, what: str = "") -> None:
    if status != SNIP_OK:
        raise SnipError(status, what)


# ----------------------------------------------------------------------------- raw ABI (same names)

def _call(name, *args):
    st = getattr(load(), name)(*args)
    check(st, name)


def snip_device_check():
    _call("snip_device_check")


def snip_workspace_init(ws, ws_bytes, stream):
    _call("snip_workspace_init", ws, ws_bytes, stream)


def snip_workspace_status(ws, stream) -> int:
    out = ctypes.c_int(0)
    _call("snip_workspace_status", ws, stream, ctypes.byref(out))
    return out.value


def snip_quantize_workspace_size(rows, cols) -> int:
    return load().snip_quantize_workspace_size(rows, cols)


def snip_amax(x, n, amax_out, ws, ws_bytes, stream):
    _call("snip_amax", x, n, amax_out, ws, ws_bytes, stream)


def snip_tensor_scales(x, n, scales_out, ws, ws_bytes, stream):
    _call("snip_tensor_scales", x, n, scales_out, ws, ws_bytes, stream)


def snip_tensor_scales_noalloc(x, n, scales_out, stream):
    _call("snip_tensor_scales_noalloc", x, n, scales_out, stream)


def snip_quantize_nvfp4(x, rows, cols, orient, rnd, seed, stream_id, g_in, layout, codes, scales, g_out,
                        block_sqerr, ws, ws_bytes, stream):
    _call("snip_quantize_nvfp4", x, rows, cols, orient, rnd, seed, stream_id, g_in, layout, codes, scales, g_out,
          block_sqerr, ws, ws_bytes, stream)


def snip_quantize_part(fmt, x, rows, cols, orient, rnd, seed, stream_id, index_base, scales_in, layout, codes,
                       scales, raw_out, ws, ws_bytes, stream):
    _call("snip_quantize_part", fmt, x, rows, cols, orient, rnd, seed, stream_id, index_base, scales_in, layout,
          codes, scales, raw_out, ws, ws_bytes, stream)


def quantize_part(fmt, x, index_base, scales_in, orient=ALONG_COLS, rnd=RTN, seed=0, stream_id=0, layout=ROWMAJOR,
                  stats=False, ws: Workspace | None = None):
    """Quantize x, a part of a larger tensor starting at its element index_base, with the whole
    tensor's scales (device {amax, g, s}) -> (codes, scales or None, raw statistics or None)."""
    torch = _torch()
    ws = ws or small_workspace()
    rows, cols = x.shape
    orows, ocols = (rows, cols) if orient == ALONG_COLS else (cols, rows)
    cb, sb = snip_quantized_bytes(fmt, layout, orows, ocols)
    codes = torch.empty(max(cb, 16), dtype=torch.uint8, device=x.device)
    fp4 = fmt in NVFP4_BLOCK or fmt == MXFP4
    sc = torch.empty(max(sb, 16), dtype=torch.uint8, device=x.device) if fp4 else None
    raw = torch.empty(STATS_NVALS, dtype=torch.float64, device=x.device) if stats else None
    snip_quantize_part(fmt, x.data_ptr(), rows, cols, orient, rnd, seed, stream_id, index_base, scales_in.data_ptr(),
                       layout, codes.data_ptr(), _ptr(sc), _ptr(raw), ws.ptr, ws.nbytes, _stream())
    return codes[:cb], (sc[:sb] if fp4 else None), raw


def snip_wait_check(limit_ns, out, ws, ws_bytes, stream):
    _call("snip_wait_check", limit_ns, out, ws, ws_bytes, stream)


def wait_check(limit_ns: int, ws: Workspace):
    """Run the bounded-wait self-check on `ws` -> device uint32 tensor {completed 0, completed 1, ns}."""
    torch = _torch()
    out = torch.full((3,), 0xFFFF, dtype=torch.int32, device=ws.buf.device)
    snip_wait_check(limit_ns, out.data_ptr(), ws.ptr, ws.nbytes, _stream())
    return out


def snip_quantize_nvfp4_block(x, rows, cols, orient, rnd, seed, stream_id, g_in, block, layout, codes, scales,
                              g_out, ws, ws_bytes, stream):
    _call("snip_quantize_nvfp4_block", x, rows, cols, orient, rnd, seed, stream_id, g_in, block, layout, codes,
          scales, g_out, ws, ws_bytes, stream)


def snip_quantize_mxfp4(x, rows, cols, orient, rnd, seed, stream_id, layout, codes, scales, ws, ws_bytes, stream):
    _call("snip_quantize_mxfp4", x, rows, cols, orient, rnd, seed, stream_id, layout, codes, scales, ws, ws_bytes,
          stream)


def snip_quantize_e5m2(x, rows, cols, orient, rnd, seed, stream_id, amax_in, layout, codes, s_out, ws, ws_bytes,
                       stream):
    _call("snip_quantize_e5m2", x, rows, cols, orient, rnd, seed, stream_id, amax_in, layout, codes, s_out, ws,
          ws_bytes, stream)


def snip_quantize_fp8(x, rows, cols, orient, rnd, seed, stream_id, s_in, layout, codes, s_out, ws, ws_bytes, stream):
    _call("snip_quantize_fp8", x, rows, cols, orient, rnd, seed, stream_id, s_in, layout, codes, s_out, ws,
          ws_bytes, stream)


def snip_quantized_bytes(fmt, layout, out_rows, out_cols) -> tuple[int, int]:
    c, s = ctypes.c_size_t(), ctypes.c_size_t()
    _call("snip_quantized_bytes", fmt, layout, out_rows, out_cols, ctypes.byref(c), ctypes.byref(s))
    return c.value, s.value


def snip_gemm(fmt, a_codes, a_scales, ga, b_codes, b_scales, gb, M, N, K, D, ldd, ws, ws_bytes, stream):
    _call("snip_gemm", fmt, a_codes, a_scales, ga, b_codes, b_scales, gb, M, N, K, D, ldd, ws, ws_bytes, stream)


def snip_qlinear_workspace_size(plan, layer, T, K, N) -> int:
    return load().snip_qlinear_workspace_size(plan, layer, T, K, N)


def snip_qlinear_fwd(plan, layer, X, W, T, K, N, Y, stats_out, ws, ws_bytes, stream):
    _call("snip_qlinear_fwd", plan, layer, X, W, T, K, N, Y, stats_out, ws, ws_bytes, stream)


def snip_qlinear_bwd(plan, layer, X, W, dY, T, K, N, dX, dW, stats_out, ws, ws_bytes, stream):
    _call("snip_qlinear_bwd", plan, layer, X, W, dY, T, K, N, dX, dW, stats_out, ws, ws_bytes, stream)


def snip_quantize_stats(fmt, x, rows, cols, rnd, seed, stream_id, scales_in, layout, codes, scales, raw_out, ws,
                        ws_bytes, stream):
    _call("snip_quantize_stats", fmt, x, rows, cols, rnd, seed, stream_id, scales_in, layout, codes, scales, raw_out,
          ws, ws_bytes, stream)


def snip_quant_stats(a, rows, cols, rnd, seed, stream_id, scales_in, raw_out, block_err_nvfp4, block_err_fp8, ws,
                     ws_bytes, stream):
    _call("snip_quant_stats", a, rows, cols, rnd, seed, stream_id, scales_in, raw_out, block_err_nvfp4,
          block_err_fp8, ws, ws_bytes, stream)


def snip_stats_finalize(raw_host) -> SnipStats:
    arr = (ctypes.c_double * STATS_NVALS)(*[float(v) for v in raw_host])
    out = SnipStats()
    _call("snip_stats_finalize", arr, ctypes.byref(out))
    return out


def snip_dw_noise_workspace_size(K, N) -> int:
    return load().snip_dw_noise_workspace_size(K, N)


def snip_dw_noise(X, dY, T, K, N, dW_q, out2, ws, ws_bytes, stream):
    _call("snip_dw_noise", X, dY, T, K, N, dW_q, out2, ws, ws_bytes, stream)


def snip_dw_noise_finalize(out2_host):
    """-> (ratio ||dW|| / ||dW_q - dW||, below sqrt(3))."""
    arr = (ctypes.c_double * 2)(*[float(v) for v in out2_host])
    ratio, flag = ctypes.c_double(), ctypes.c_int()
    _call("snip_dw_noise_finalize", arr, ctypes.byref(ratio), ctypes.byref(flag))
    return ratio.value, bool(flag.value)


def snip_plan_costs(raw_host):
    """raw_host: n_layers x 3 x STATS_NVALS (X, W, dY statistics of each layer)
    -> (cost_fp8, cost_nvfp4) lists."""
    import numpy as np
    raw = np.ascontiguousarray(raw_host, dtype=np.float64).reshape(-1, 3, STATS_NVALS)
    n = raw.shape[0]
    c8 = np.zeros(n, dtype=np.float64)
    c4 = np.zeros(n, dtype=np.float64)
    _call("snip_plan_costs", n, raw.ctypes.data, c8.ctypes.data, c4.ctypes.data)
    return c8, c4


def snip_plan_select(flops, cost_fp8, cost_nvfp4, fp4_fraction):
    """-> (formats per layer, achieved FP4 FLOP share, total cost)."""
    import numpy as np
    f = np.ascontiguousarray(flops, dtype=np.float64)
    c8 = np.ascontiguousarray(cost_fp8, dtype=np.float64)
    c4 = np.ascontiguousarray(cost_nvfp4, dtype=np.float64)
    n = f.shape[0]
    if c8.shape != (n,) or c4.shape != (n,):
        raise ValueError("flops, cost_fp8 and cost_nvfp4 need one entry per layer")
    fmt = np.zeros(max(n, 1), dtype=np.int32)
    frac = ctypes.c_double()
    cost = ctypes.c_double()
    _call("snip_plan_select", n, f.ctypes.data, c8.ctypes.data, c4.ctypes.data, float(fp4_fraction),
          fmt.ctypes.data, ctypes.byref(frac), ctypes.byref(cost))
    return [int(v) for v in fmt[:n]], frac.value, cost.value


# ----------------------------------------------------------------------------- torch conveniences

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    torch = _torch()
    return (stream or torch.cuda.current_stream()).cuda_stream


class Plan:
    """Owns a snip_plan (per-layer formats, rounding per quantization, seed)."""

    def __init__(self, formats, seed: int = 0):
        self.formats = list(formats)
        arr = (ctypes.c_int * len(self.formats))(*self.formats)
        h = ctypes.c_void_p()
        check(load().snip_plan_create(len(self.formats), arr, seed, ctypes.byref(h)), "snip_plan_create")
        self.handle = h
        self.seed = seed

    def set_rounding(self, layer: int, tag: int, rnd: int):
        check(load().snip_plan_set_rounding(self.handle, layer, tag, rnd), "snip_plan_set_rounding")

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.snip_plan_destroy(self.handle)
            self.handle = None


class Workspace:
    """A caller-owned device workspace with an initialised status word."""

    def __init__(self, nbytes: int, device="cuda"):
        torch = _torch()
        self.nbytes = max(int(nbytes), WS_HEADER_BYTES)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        snip_workspace_init(self.buf.data_ptr(), self.nbytes, _stream())

    @property
    def ptr(self):
        return self.buf.data_ptr()

    def status(self) -> int:
        return snip_workspace_status(self.ptr, _stream())

    def reset(self):
        snip_workspace_init(self.ptr, self.nbytes, _stream())


_small_ws = {}


def small_workspace(device=None) -> Workspace:
    """A shared small workspace per device for the standalone quantize/stats/GEMM calls."""
    torch = _torch()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    key = str(dev)
    if key not in _small_ws:
        _small_ws[key] = Workspace(snip_quantize_workspace_size(0, 0), dev)
    return _small_ws[key]


@dataclass
class QuantNVFP4:
    codes: object
    scales: object
    g: object            # device float tensor (1,)
    out_rows: int
    out_cols: int
    layout: int
    block_err: object = None


@dataclass
class QuantMXFP4:
    codes: object
    scales: object
    out_rows: int
    out_cols: int
    layout: int


@dataclass
class QuantFP8:
    codes: object
    s: object
    out_rows: int
    out_cols: int
    layout: int


def tensor_scales_multi(xs, outs, ws: Workspace | None = None):
    """{amax, g, s} of each bf16 tensor in xs into the device float (3,) tensors outs, one launch."""
    ws = ws or small_workspace()
    n = len(xs)
    ptrs = (ctypes.c_void_p * n)(*[x.data_ptr() for x in xs])
    ns = (ctypes.c_int64 * n)(*[x.numel() for x in xs])
    op = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    _call("snip_tensor_scales_multi", n, ptrs, ns, op, ws.ptr, ws.nbytes, _stream())
    return outs


def tensor_scales(x, ws: Workspace | None = None, out=None):
    """Device float tensor (3,) = {amax, NVFP4 g, FP8 s} of a bf16 tensor."""
    torch = _torch()
    ws = ws or small_workspace()
    out = out if out is not None else torch.empty(3, dtype=torch.float32, device=x.device)
    snip_tensor_scales(x.data_ptr(), x.numel(), out.data_ptr(), ws.ptr, ws.nbytes, _stream())
    return out


def amax(x, ws: Workspace | None = None):
    torch = _torch()
    ws = ws or small_workspace()
    out = torch.empty(1, dtype=torch.float32, device=x.device)
    snip_amax(x.data_ptr(), x.numel(), out.data_ptr(), ws.ptr, ws.nbytes, _stream())
    return out


def quantize_nvfp4(x, orient=ALONG_COLS, rnd=RTN, seed=0, stream_id=0, g_in=None, layout=ROWMAJOR,
                   want_block_err=False, ws: Workspace | None = None) -> QuantNVFP4:
    torch = _torch()
    ws = ws or small_workspace()
    rows, cols = x.shape
    orows, ocols = (rows, cols) if orient == ALONG_COLS else (cols, rows)
    cb, sb = snip_quantized_bytes(NVFP4, layout, orows, ocols)
    codes = torch.empty(max(cb, 16), dtype=torch.uint8, device=x.device)
    scales = torch.empty(max(sb, 16), dtype=torch.uint8, device=x.device)
    g = torch.empty(1, dtype=torch.float32, device=x.device)
    berr = torch.empty((orows, ocols // 16), dtype=torch.float32, device=x.device) if want_block_err else None
    snip_quantize_nvfp4(x.data_ptr(), rows, cols, orient, rnd, seed, stream_id, _ptr(g_in), layout,
                        codes.data_ptr(), scales.data_ptr(), g.data_ptr(), _ptr(berr), ws.ptr, ws.nbytes, _stream())
    return QuantNVFP4(codes[:cb], scales[:sb], g, orows, ocols, layout, berr)


def quantize_nvfp4_block(x, block, orient=ALONG_COLS, rnd=RTN, seed=0, stream_id=0, g_in=None, layout=ROWMAJOR,
                         ws: Workspace | None = None) -> QuantNVFP4:
    """NVFP4 with `block` (16, 32, 64, 128) elements per E4M3 scale, in NVFP4's layouts (each scale
    repeated for every 16 elements it covers): an NVFP4 operand for gemm()."""
    torch = _torch()
    ws = ws or small_workspace()
    rows, cols = x.shape
    orows, ocols = (rows, cols) if orient == ALONG_COLS else (cols, rows)
    cb, sb = snip_quantized_bytes(NVFP4, layout, orows, ocols)
    codes = torch.empty(max(cb, 16), dtype=torch.uint8, device=x.device)
    scales = torch.empty(max(sb, 16), dtype=torch.uint8, device=x.device)
    g = torch.empty(1, dtype=torch.float32, device=x.device)
    snip_quantize_nvfp4_block(x.data_ptr(), rows, cols, orient, rnd, seed, stream_id, _ptr(g_in), block, layout,
                              codes.data_ptr(), scales.data_ptr(), g.data_ptr(), ws.ptr, ws.nbytes, _stream())
    return QuantNVFP4(codes[:cb], scales[:sb], g, orows, ocols, layout)


def quantize_fp8(x, orient=ALONG_COLS, rnd=RTN, seed=0, stream_id=0, s_in=None, layout=ROWMAJOR,
                 ws: Workspace | None = None) -> QuantFP8:
    torch = _torch()
    ws = ws or small_workspace()
    rows, cols = x.shape
    orows, ocols = (rows, cols) if orient == ALONG_COLS else (cols, rows)
    cb, _ = snip_quantized_bytes(FP8, layout, orows, ocols)
    codes = torch.empty(max(cb, 16), dtype=torch.uint8, device=x.device)
    s = torch.empty(1, dtype=torch.float32, device=x.device)
    snip_quantize_fp8(x.data_ptr(), rows, cols, orient, rnd, seed, stream_id, _ptr(s_in), layout,
                      codes.data_ptr(), s.data_ptr(), ws.ptr, ws.nbytes, _stream())
    return QuantFP8(codes[:cb], s, orows, ocols, layout)


def quantize_mxfp4(x, orient=ALONG_COLS, rnd=RTN, seed=0, stream_id=0, layout=ROWMAJOR,
                   ws: Workspace | None = None) -> QuantMXFP4:
    torch = _torch()
    ws = ws or small_workspace()
    rows, cols = x.shape
    orows, ocols = (rows, cols) if orient == ALONG_COLS else (cols, rows)
    cb, sb = snip_quantized_bytes(MXFP4, layout, orows, ocols)
    codes = torch.empty(max(cb, 16), dtype=torch.uint8, device=x.device)
    scales = torch.empty(max(sb, 16), dtype=torch.uint8, device=x.device)
    snip_quantize_mxfp4(x.data_ptr(), rows, cols, orient, rnd, seed, stream_id, layout, codes.data_ptr(),
                        scales.data_ptr(), ws.ptr, ws.nbytes, _stream())
    return QuantMXFP4(codes[:cb], scales[:sb], orows, ocols, layout)


def quantize_e5m2(x, orient=ALONG_COLS, rnd=RTN, seed=0, stream_id=0, amax_in=None, layout=ROWMAJOR,
                  ws: Workspace | None = None) -> QuantFP8:
    """FP8 E5M2 quantization (tensor scale amax / 57344), returned like QuantFP8."""
    torch = _torch()
    ws = ws or small_workspace()
    rows, cols = x.shape
    orows, ocols = (rows, cols) if orient == ALONG_COLS else (cols, rows)
    cb, _ = snip_quantized_bytes(FP8_E5M2, layout, orows, ocols)
    codes = torch.empty(max(cb, 16), dtype=torch.uint8, device=x.device)
    s = torch.empty(1, dtype=torch.float32, device=x.device)
    snip_quantize_e5m2(x.data_ptr(), rows, cols, orient, rnd, seed, stream_id, _ptr(amax_in), layout,
                       codes.data_ptr(), s.data_ptr(), ws.ptr, ws.nbytes, _stream())
    return QuantFP8(codes[:cb], s, orows, ocols, layout)


def gemm(fmt, a, b, M, N, K, out=None, ws: Workspace | None = None):
    """D = A B^T on two MMA-layout quantized operands (QuantNVFP4 / QuantFP8)."""
    torch = _torch()
    ws = ws or small_workspace()
    D = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=a.codes.device)
    if fmt in NVFP4_BLOCK:   # NVFP4 and its longer-block variants: the same operands and GEMM
        snip_gemm(NVFP4, a.codes.data_ptr(), a.scales.data_ptr(), a.g.data_ptr(), b.codes.data_ptr(),
                  b.scales.data_ptr(), b.g.data_ptr(), M, N, K, D.data_ptr(), D.stride(0), ws.ptr, ws.nbytes,
                  _stream())
    elif fmt == MXFP4:
        snip_gemm(MXFP4, a.codes.data_ptr(), a.scales.data_ptr(), None, b.codes.data_ptr(), b.scales.data_ptr(),
                  None, M, N, K, D.data_ptr(), D.stride(0), ws.ptr, ws.nbytes, _stream())
    else:   # FP8: fmt FP8 (both E4M3) or FP8_E5M2 (A in E5M2, B in E4M3)
        snip_gemm(fmt, a.codes.data_ptr(), None, a.s.data_ptr(), b.codes.data_ptr(), None, b.s.data_ptr(),
                  M, N, K, D.data_ptr(), D.stride(0), ws.ptr, ws.nbytes, _stream())
    return D


def qlinear_workspace(plan: Plan, layer: int, T: int, K: int, N: int, device="cuda") -> Workspace:
    return Workspace(snip_qlinear_workspace_size(plan.handle, layer, T, K, N), device)


def qlinear_fwd(plan: Plan, layer: int, X, W, ws: Workspace, Y=None, stats=None):
    """Y = Q(X) Q(W)^T; `stats` (device float64 (2, STATS_NVALS) or None) receives
    the statistics of X and W from the same quantization passes."""
    torch = _torch()
    T, K = X.shape
    N = W.shape[0]
    Y = Y if Y is not None else torch.empty((T, N), dtype=torch.float32, device=X.device)
    snip_qlinear_fwd(plan.handle, layer, X.data_ptr(), W.data_ptr(), T, K, N, Y.data_ptr(), _ptr(stats), ws.ptr,
                     ws.nbytes, _stream())
    return Y


def _multi_arrays(layers, Ns):
    n = len(layers)
    return (ctypes.c_int * n)(*layers), (ctypes.c_int64 * n)(*Ns)


def qlinear_fwd_multi_workspace(plan: Plan, layers, T: int, K: int, Ns, device="cuda") -> Workspace:
    la, na = _multi_arrays(layers, Ns)
    return Workspace(load().snip_qlinear_fwd_multi_workspace_size(plan.handle, len(layers), la, T, K, na), device)


def qlinear_fwd_multi(plan: Plan, layers, X, Ws, ws: Workspace, Ys=None, stats_x=None, stats_w=None):
    """Forward of the layers `layers` reading one X (Q/K/V, Gate/Up): Ys[i] = Q(X) Q(Ws[i])^T, X's
    scales, statistics (stats_x) and quantization computed once; stats_w: a list of device float64
    (STATS_NVALS,) tensors or None for the weights' statistics."""
    torch = _torch()
    T, K = X.shape
    Ns = [w.shape[0] for w in Ws]
    Ys = Ys if Ys is not None else [torch.empty((T, n), dtype=torch.float32, device=X.device) for n in Ns]
    la, na = _multi_arrays(layers, Ns)
    n = len(layers)
    wa = (ctypes.c_void_p * n)(*[w.data_ptr() for w in Ws])
    ya = (ctypes.c_void_p * n)(*[y.data_ptr() for y in Ys])
    sa = (ctypes.c_void_p * n)(*[_ptr(t) for t in stats_w]) if stats_w is not None else None
    _call("snip_qlinear_fwd_multi", plan.handle, n, la, X.data_ptr(), wa, T, K, na, ya, _ptr(stats_x), sa, ws.ptr,
          ws.nbytes, _stream())
    return Ys


def qlinear_bwd_chain(plan: Plan, layer: int, prev_layer: int, X, W, dY, g_prev, ws: Workspace, want_dx=False,
                      stats=None):
    """The backward of `layer` whose dgrad product is written as prev_layer's NVFP4 gradient operands
    (row blocks, column blocks; tensor scale g_prev, a device float (1,)) -> (dX fp32 or None, dW,
    rows QuantNVFP4, columns QuantNVFP4, amax device float (1,))."""
    torch = _torch()
    T, K = X.shape
    N = W.shape[0]
    dev = X.device
    dX = torch.empty((T, K), dtype=torch.float32, device=dev) if want_dx else None
    dW = torch.empty((N, K), dtype=torch.float32, device=dev)
    cb, sb = snip_quantized_bytes(NVFP4, MMA, T, K)
    cbt, sbt = snip_quantized_bytes(NVFP4, MMA, K, T)
    rc, rs = torch.empty(cb, dtype=torch.uint8, device=dev), torch.empty(sb, dtype=torch.uint8, device=dev)
    tc, ts = torch.empty(cbt, dtype=torch.uint8, device=dev), torch.empty(sbt, dtype=torch.uint8, device=dev)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    _call("snip_qlinear_bwd_chain", plan.handle, layer, prev_layer, X.data_ptr(), W.data_ptr(), dY.data_ptr(), T,
          K, N, _ptr(dX), dW.data_ptr(), _ptr(stats), g_prev.data_ptr(), rc.data_ptr(), rs.data_ptr(),
          tc.data_ptr(), ts.data_ptr(), amax.data_ptr(), ws.ptr, ws.nbytes, _stream())
    return dX, dW, QuantNVFP4(rc, rs, g_prev, T, K, MMA), QuantNVFP4(tc, ts, g_prev, K, T, MMA), amax


def qlinear_bwd_q(plan: Plan, layer: int, X, W, dy_rows, dy_cols, ws: Workspace, dX=None, dW=None):
    """The backward of an NVFP4 layer from its quantized gradient operands (QuantNVFP4 row and
    column blocks sharing one tensor scale) -> (dX, dW)."""
    torch = _torch()
    T, K = X.shape
    N = W.shape[0]
    dX = dX if dX is not None else torch.empty((T, K), dtype=torch.float32, device=X.device)
    dW = dW if dW is not None else torch.empty((N, K), dtype=torch.float32, device=X.device)
    _call("snip_qlinear_bwd_q", plan.handle, layer, X.data_ptr(), W.data_ptr(), dy_rows.codes.data_ptr(),
          dy_rows.scales.data_ptr(), dy_cols.codes.data_ptr(), dy_cols.scales.data_ptr(), dy_rows.g.data_ptr(), T,
          K, N, dX.data_ptr(), dW.data_ptr(), ws.ptr, ws.nbytes, _stream())
    return dX, dW


def qlinear_bwd(plan: Plan, layer: int, X, W, dY, ws: Workspace, dX=None, dW=None, stats=None):
    """dX = Q(dY) Q(W^T)^T and dW = Q(dY^T) Q(X^T)^T; `stats` (device float64
    (STATS_NVALS,) or None) receives the statistics of dY under the dgrad rounding."""
    torch = _torch()
    T, K = X.shape
    N = W.shape[0]
    dX = dX if dX is not None else torch.empty((T, K), dtype=torch.float32, device=X.device)
    dW = dW if dW is not None else torch.empty((N, K), dtype=torch.float32, device=X.device)
    snip_qlinear_bwd(plan.handle, layer, X.data_ptr(), W.data_ptr(), dY.data_ptr(), T, K, N, dX.data_ptr(),
                     dW.data_ptr(), _ptr(stats), ws.ptr, ws.nbytes, _stream())
    return dX, dW


def quantize_stats(fmt, x, rnd=RTN, seed=0, stream_id=0, layout=MMA, scales=None, ws: Workspace | None = None):
    """One pass: quantize x (blocks along cols) and compute its statistics.
    Returns (QuantNVFP4 or QuantFP8 without a g/s tensor, raw statistics)."""
    torch = _torch()
    ws = ws or small_workspace()
    rows, cols = x.shape
    cb, sb = snip_quantized_bytes(fmt, layout, rows, cols)
    codes = torch.empty(max(cb, 16), dtype=torch.uint8, device=x.device)
    sc = torch.empty(max(sb, 16), dtype=torch.uint8, device=x.device)
    raw = torch.empty(STATS_NVALS, dtype=torch.float64, device=x.device)
    snip_quantize_stats(fmt, x.data_ptr(), rows, cols, rnd, seed, stream_id, _ptr(scales), layout, codes.data_ptr(),
                        sc.data_ptr() if fmt in NVFP4_BLOCK or fmt == MXFP4 else None, raw.data_ptr(), ws.ptr,
                        ws.nbytes, _stream())
    return codes[:cb], sc[:sb], raw


def dw_noise(X, dY, dW_q, ws: Workspace | None = None):
    """{||dW||^2, ||dW_q - dW||^2} (device float64 (2,)) with dW = dY^T X from the bf16 tensors."""
    torch = _torch()
    T, K = X.shape
    N = dY.shape[1]
    ws = ws or Workspace(snip_dw_noise_workspace_size(K, N), X.device)
    out = torch.empty(2, dtype=torch.float64, device=X.device)
    snip_dw_noise(X.data_ptr(), dY.data_ptr(), T, K, N, dW_q.data_ptr(), out.data_ptr(), ws.ptr, ws.nbytes,
                  _stream())
    return out


def gemm_requant(fmt, a, b, M, N, K, g_in, rnd=SR, seed=0, stream_id=0, want_d=True, rows=True, cols=False,
                 rnd_t=SR, stream_id_t=0, ws: Workspace | None = None):
    """D = A B^T (fp32, or None) plus D rounded to bf16 and quantized to NVFP4 with the device tensor
    scale g_in (1-element float tensor): row blocks (the M x N operand; rnd, stream_id) and/or column
    blocks (the N x M operand D^T; rnd_t, stream_id_t), both in the MMA layout
    -> (D, rows QuantNVFP4 or None, amax tensor, columns QuantNVFP4 or None)."""
    torch = _torch()
    ws = ws or small_workspace()
    dev = a.codes.device
    D = torch.empty((M, N), dtype=torch.float32, device=dev) if want_d else None

    def buffers(orows, ocols):
        cb, sb = snip_quantized_bytes(NVFP4, MMA, orows, ocols)
        return (torch.empty(max(cb, 16), dtype=torch.uint8, device=dev),
                torch.empty(max(sb, 16), dtype=torch.uint8, device=dev), cb, sb)

    r = buffers(M, N) if rows else None
    c = buffers(N, M) if cols else None
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    rq = SnipRequant(g_in.data_ptr(), rnd, seed, stream_id, r[0].data_ptr() if r else None,
                     r[1].data_ptr() if r else None, amax.data_ptr(), rnd_t, stream_id_t,
                     c[0].data_ptr() if c else None, c[1].data_ptr() if c else None)
    sa = a.scales.data_ptr() if fmt in (NVFP4, MXFP4) else None
    sb_ = b.scales.data_ptr() if fmt in (NVFP4, MXFP4) else None
    ga = (a.g if fmt == NVFP4 else a.s).data_ptr() if fmt != MXFP4 else None
    gb = (b.g if fmt == NVFP4 else b.s).data_ptr() if fmt != MXFP4 else None
    _call("snip_gemm_requant", fmt, a.codes.data_ptr(), sa, ga, b.codes.data_ptr(), sb_, gb, M, N, K,
          D.data_ptr() if D is not None else None, N, ctypes.byref(rq), ws.ptr, ws.nbytes, _stream())
    qr = QuantNVFP4(r[0][:r[2]], r[1][:r[3]], g_in, M, N, MMA) if r else None
    qc = QuantNVFP4(c[0][:c[2]], c[1][:c[3]], g_in, N, M, MMA) if c else None
    return D, qr, amax, qc


def quant_stats(a, rnd=RTN, seed=0, stream_id=0, want_block_err=False, ws: Workspace | None = None, raw=None,
                scales=None):
    """Launch the statistics pass; returns (raw device tensor, block errors or None)."""
    torch = _torch()
    ws = ws or small_workspace()
    rows, cols = a.shape
    raw = raw if raw is not None else torch.empty(STATS_NVALS, dtype=torch.float64, device=a.device)
    b4 = b8 = None
    if want_block_err:
        b4 = torch.empty((rows, cols // 16), dtype=torch.float32, device=a.device)
        b8 = torch.empty((rows, cols // 16), dtype=torch.float32, device=a.device)
    snip_quant_stats(a.data_ptr(), rows, cols, rnd, seed, stream_id, _ptr(scales), raw.data_ptr(), _ptr(b4), _ptr(b8),
                     ws.ptr, ws.nbytes, _stream())
    return raw, (b4, b8)
