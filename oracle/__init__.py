"""CPU oracle for the quantized linear layer (SNIP + NVFP4/FP8).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``sub_byte_mixed_gb300``) never imports it and shares no code with it.

The encoding steps live in ``snip_oracle.c`` (plain C, one IEEE fp32 operation
per step, fp64 accumulation), built with gcc by :func:`build`.  This module
marshals numpy arrays into it and adds the GEMM step: the product of the two
dequantized operands in fp64 via ``numpy.matmul`` (a library primitive, no
blocking or reordering of our own).

Sources (page title, section):
  * "FP4 all the way" (Chmiel et al.), summary page, Outline -- the NVFP4 format
    (16 E2M1 values + one E4M3 scale), round-to-nearest forward, stochastic
    rounding in backpropagation and update, the sqrt(3)-times-noise threshold.
  * "SNIP: An Adaptive Mixed Precision Framework for Subbyte LLM Training",
    Figure 5 -- forward Y = X W^T, dgrad dX = dY W, wgrad dW = dY^T X, each GEMM
    in the layer's chosen precision; Abstract/Figure 2 -- statistics on
    activations, weights and gradients.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "snip_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

ROWS_BLOCKS_ALONG_COLS = 0   # blocks of 16 along the last dim
ROWS_BLOCKS_ALONG_ROWS = 1   # blocks of 16 along the first dim; output transposed
RTN, SR = 0, 1

# raw statistics slots (same order as the C enum)
ST_SUM_X2, ST_NVFP4_ERR2, ST_FP8_ERR2, ST_NVFP4_SRVAR, ST_FP8_SRVAR, ST_AMAX, ST_COUNT = range(7)
ST_N = 8


def build(force: bool = False) -> str:
    """Compile snip_oracle.c into _build/liboracle.so (gcc, -O2, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        c_u8p = ctypes.POINTER(ctypes.c_uint8)
        c_u16p = ctypes.POINTER(ctypes.c_uint16)
        c_u32p = ctypes.POINTER(ctypes.c_uint32)
        c_fp = ctypes.POINTER(ctypes.c_float)
        c_dp = ctypes.POINTER(ctypes.c_double)
        i64, u64, i32, u32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_uint32
        L.oracle_e2m1_value.argtypes = [i32]; L.oracle_e2m1_value.restype = ctypes.c_double
        L.oracle_e4m3_value.argtypes = [i32]; L.oracle_e4m3_value.restype = ctypes.c_double
        L.oracle_e2m1_rtn.argtypes = [ctypes.c_float]; L.oracle_e2m1_rtn.restype = i32
        L.oracle_e4m3_rtn.argtypes = [ctypes.c_float]; L.oracle_e4m3_rtn.restype = i32
        L.oracle_e2m1_sr.argtypes = [ctypes.c_float, u32]; L.oracle_e2m1_sr.restype = i32
        L.oracle_e4m3_sr.argtypes = [ctypes.c_float, u32]; L.oracle_e4m3_sr.restype = i32
        L.oracle_philox4x32_10.argtypes = [c_u32p, c_u32p, c_u32p]; L.oracle_philox4x32_10.restype = None
        L.oracle_sr_bits.argtypes = [u64, u64, u64]; L.oracle_sr_bits.restype = u32
        L.oracle_amax_bf16.argtypes = [c_u16p, i64, c_fp]; L.oracle_amax_bf16.restype = i32
        L.oracle_nvfp4_global_scale.argtypes = [ctypes.c_float]; L.oracle_nvfp4_global_scale.restype = ctypes.c_float
        L.oracle_fp8_tensor_scale.argtypes = [ctypes.c_float]; L.oracle_fp8_tensor_scale.restype = ctypes.c_float
        L.oracle_quantize_nvfp4.argtypes = [c_u16p, i64, i64, i32, i32, u64, u64, c_fp,
                                            c_u8p, c_u8p, c_fp, c_dp, ctypes.POINTER(ctypes.c_int64), i64]
        L.oracle_quantize_nvfp4.restype = i32
        L.oracle_quantize_nvfp4_at.argtypes = [c_u16p, i64, i64, i32, i32, u64, u64, c_fp, u64,
                                               c_u8p, c_u8p, c_fp, c_dp, ctypes.POINTER(ctypes.c_int64), i64]
        L.oracle_quantize_nvfp4_at.restype = i32
        L.oracle_quantize_fp8_at.argtypes = [c_u16p, i64, i64, i32, i32, u64, u64, c_fp, u64, c_u8p, c_fp,
                                             ctypes.POINTER(ctypes.c_int64), i64]
        L.oracle_quantize_fp8_at.restype = i32
        L.oracle_quant_stats_at.argtypes = [c_u16p, i64, i64, i32, u64, u64, c_fp, c_fp, u64, c_dp, c_dp, c_dp]
        L.oracle_quant_stats_at.restype = i32
        L.oracle_dequant_nvfp4.argtypes = [c_u8p, c_u8p, ctypes.c_float, i64, i64, c_dp]
        L.oracle_dequant_nvfp4.restype = None
        L.oracle_quantize_nvfp4_block.argtypes = [c_u16p, i64, i64, i32, i32, u64, u64, c_fp, i32,
                                                  c_u8p, c_u8p, c_fp, ctypes.POINTER(ctypes.c_int64), i64]
        L.oracle_quantize_nvfp4_block.restype = i32
        L.oracle_dequant_nvfp4_block.argtypes = [c_u8p, c_u8p, ctypes.c_float, i32, i64, i64, c_dp]
        L.oracle_dequant_nvfp4_block.restype = None
        L.oracle_e8m0_value.argtypes = [i32]; L.oracle_e8m0_value.restype = ctypes.c_double
        L.oracle_mxfp4_shared_exp.argtypes = [ctypes.c_float]; L.oracle_mxfp4_shared_exp.restype = i32
        c_i64p = ctypes.POINTER(ctypes.c_int64)
        L.oracle_e5m2_value.argtypes = [i32]; L.oracle_e5m2_value.restype = ctypes.c_double
        L.oracle_e5m2_rtn.argtypes = [ctypes.c_float]; L.oracle_e5m2_rtn.restype = i32
        L.oracle_e5m2_sr.argtypes = [ctypes.c_float, u32]; L.oracle_e5m2_sr.restype = i32
        L.oracle_e5m2_tensor_scale.argtypes = [ctypes.c_float]; L.oracle_e5m2_tensor_scale.restype = ctypes.c_float
        L.oracle_quantize_e5m2.argtypes = [c_u16p, i64, i64, i32, i32, u64, u64, c_fp, c_u8p, c_fp, c_i64p, i64]
        L.oracle_quantize_e5m2.restype = i32
        L.oracle_dequant_e5m2.argtypes = [c_u8p, ctypes.c_float, i64, c_dp]
        L.oracle_dequant_e5m2.restype = None
        L.oracle_quantize_mxfp4.argtypes = [c_u16p, i64, i64, i32, i32, u64, u64, c_u8p, c_u8p, c_i64p, i64]
        L.oracle_quantize_mxfp4.restype = i32
        L.oracle_dequant_mxfp4.argtypes = [c_u8p, c_u8p, i64, i64, c_dp]
        L.oracle_dequant_mxfp4.restype = None
        L.oracle_quantize_fp8.argtypes = [c_u16p, i64, i64, i32, i32, u64, u64, c_fp, c_u8p, c_fp, c_i64p, i64]
        L.oracle_quantize_fp8.restype = i32
        L.oracle_dequant_fp8.argtypes = [c_u8p, ctypes.c_float, i64, c_dp]
        L.oracle_dequant_fp8.restype = None
        L.oracle_quant_stats.argtypes = [c_u16p, i64, i64, i32, u64, u64, c_dp, c_dp, c_dp]
        L.oracle_quant_stats.restype = i32
        _lib = L
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class NonFiniteInput(ValueError):
    """The tensor holds an infinity or a NaN: the encodings reject it."""


def _bits_to_f64(x) -> np.ndarray:
    """bf16 tensor -> float64 values (exact: bf16 is the top half of binary32)."""
    b = _bits(x).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _bits(x) -> np.ndarray:
    """bf16 tensor (torch, or uint16 numpy bit patterns) -> contiguous uint16 numpy."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------- scalar format helpers

def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(int(code))


def e2m1_rtn(y: float) -> int:
    return lib().oracle_e2m1_rtn(float(y))


def e4m3_rtn(t: float) -> int:
    return lib().oracle_e4m3_rtn(float(t))


def e2m1_sr(y: float, u16: int) -> int:
    return lib().oracle_e2m1_sr(float(y), int(u16))


def e4m3_sr(y: float, u16: int) -> int:
    return lib().oracle_e4m3_sr(float(y), int(u16))


def e5m2_value(code: int) -> float:
    return lib().oracle_e5m2_value(int(code))


def e5m2_rtn(t: float) -> int:
    return lib().oracle_e5m2_rtn(float(t))


def e5m2_sr(y: float, u16: int) -> int:
    return lib().oracle_e5m2_sr(float(y), int(u16))


def philox4x32_10(ctr, key):
    c = np.array(ctr, dtype=np.uint32)
    k = np.array(key, dtype=np.uint32)
    o = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c, ctypes.c_uint32), _ptr(k, ctypes.c_uint32), _ptr(o, ctypes.c_uint32))
    return [int(v) for v in o]


def sr_bits(seed: int, stream_id: int, e: int) -> int:
    return lib().oracle_sr_bits(seed, stream_id, e)


def nvfp4_global_scale(amax: float) -> float:
    return lib().oracle_nvfp4_global_scale(float(amax))


def fp8_tensor_scale(amax: float) -> float:
    return lib().oracle_fp8_tensor_scale(float(amax))


# ----------------------------------------------------------------------------- tensors

def amax(x) -> float:
    b = _bits(x)
    m = ctypes.c_float()
    if lib().oracle_amax_bf16(_ptr(b.reshape(-1), ctypes.c_uint16), b.size, ctypes.byref(m)):
        raise NonFiniteInput("non-finite input")
    return m.value


class NVFP4:
    """An NVFP4 tensor of shape (rows, cols): codes rows x cols/2 (low nibble =
    even column), E4M3 scales rows x cols/16, fp32 tensor scale g."""

    def __init__(self, codes, scales, g, rows, cols, block_sqerr=None):
        self.codes, self.scales, self.g = codes, scales, g
        self.rows, self.cols = rows, cols
        self.block_sqerr = block_sqerr

    def dequant(self) -> np.ndarray:
        out = np.empty((self.rows, self.cols), dtype=np.float64)
        lib().oracle_dequant_nvfp4(_ptr(self.codes, ctypes.c_uint8), _ptr(self.scales, ctypes.c_uint8),
                                   self.g, self.rows, self.cols, _ptr(out, ctypes.c_double))
        return out


class NVFP4Block:
    """E2M1 codes with one E4M3 scale per `block` elements (B = 16 is NVFP4): codes
    rows x cols/2 (low nibble = even column), scales rows x cols/block, tensor scale g."""

    def __init__(self, codes, scales, g, rows, cols, block):
        self.codes, self.scales, self.g = codes, scales, g
        self.rows, self.cols, self.block = rows, cols, block

    def dequant(self) -> np.ndarray:
        out = np.empty((self.rows, self.cols), dtype=np.float64)
        lib().oracle_dequant_nvfp4_block(_ptr(self.codes, ctypes.c_uint8), _ptr(self.scales, ctypes.c_uint8),
                                         self.g, self.block, self.rows, self.cols, _ptr(out, ctypes.c_double))
        return out


class MXFP4:
    """An MXFP4 tensor of shape (rows, cols): codes rows x cols/2 (low nibble =
    even column), E8M0 scales rows x cols/32; no tensor scale."""

    def __init__(self, codes, scales, rows, cols):
        self.codes, self.scales = codes, scales
        self.rows, self.cols = rows, cols
        self.g = 1.0

    def dequant(self) -> np.ndarray:
        out = np.empty((self.rows, self.cols), dtype=np.float64)
        lib().oracle_dequant_mxfp4(_ptr(self.codes, ctypes.c_uint8), _ptr(self.scales, ctypes.c_uint8),
                                   self.rows, self.cols, _ptr(out, ctypes.c_double))
        return out


class FP8:
    """An FP8 E4M3 tensor of shape (rows, cols) with one fp32 scale s."""

    def __init__(self, codes, s, rows, cols):
        self.codes, self.s, self.rows, self.cols = codes, s, rows, cols

    def dequant(self) -> np.ndarray:
        out = np.empty((self.rows, self.cols), dtype=np.float64)
        lib().oracle_dequant_fp8(_ptr(self.codes, ctypes.c_uint8), self.s, self.rows * self.cols,
                                 _ptr(out, ctypes.c_double))
        return out


def _selection(rows):
    """Output-row selection (None = all) -> (int64 array or None, pointer, count)."""
    if rows is None:
        return None, None, 0
    sel = np.ascontiguousarray(rows, dtype=np.int64)
    return sel, _ptr(sel, ctypes.c_int64), sel.shape[0]


def quantize_nvfp4(x, orient: int = 0, rnd: int = RTN, seed: int = 0, stream_id: int = 0,
                   g_in: float | None = None, want_block_err: bool = False, rows=None,
                   index_base: int = 0) -> NVFP4:
    """NVFP4 quantization of a bf16 (rows, cols) tensor; orient=1 quantizes the
    transpose with blocks along the original rows (random bits still indexed
    by the source element).  rows (optional): compute only these output rows
    (tensor scale and random bits as for the whole tensor).  index_base: x is
    the part of a larger row-major tensor that starts at that element (random
    bits as for the larger tensor; pass its tensor scale as g_in)."""
    b = _bits(x)
    sel, psel, nsel = _selection(rows)
    rows, cols = b.shape
    OR, OC = (rows, cols) if orient == 0 else (cols, rows)
    if sel is not None:
        assert np.all((sel >= 0) & (sel < OR))
        OR = nsel
    codes = np.zeros((OR, OC // 2), dtype=np.uint8)
    scales = np.zeros((OR, OC // 16), dtype=np.uint8)
    berr = np.zeros((OR, OC // 16), dtype=np.float64) if want_block_err else None
    g = ctypes.c_float()
    gin = ctypes.byref(ctypes.c_float(g_in)) if g_in is not None else None
    st = lib().oracle_quantize_nvfp4_at(_ptr(b, ctypes.c_uint16), rows, cols, orient, rnd, seed, stream_id,
                                     gin, index_base, _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                     ctypes.byref(g),
                                     _ptr(berr, ctypes.c_double) if berr is not None else None, psel, nsel)
    if st == 1:
        raise NonFiniteInput("non-finite input")
    if st != 0:
        raise ValueError(f"shape error: blocks of 16 need the blocked dim % 16 == 0 (got {OR}x{OC})")
    return NVFP4(codes, scales, g.value, OR, OC, berr)


def quantize_nvfp4_block(x, block: int, orient: int = 0, rnd: int = RTN, seed: int = 0, stream_id: int = 0,
                         g_in: float | None = None, rows=None) -> NVFP4Block:
    """E2M1 + E4M3 quantization with one scale per `block` (16, 32, 64, 128) elements
    along the blocked dim; otherwise as quantize_nvfp4."""
    b = _bits(x)
    sel, psel, nsel = _selection(rows)
    rows, cols = b.shape
    OR, OC = (rows, cols) if orient == 0 else (cols, rows)
    if sel is not None:
        assert np.all((sel >= 0) & (sel < OR))
        OR = nsel
    if OC % block != 0:
        raise ValueError(f"shape error: blocks of {block} need the blocked dim % {block} == 0 (got {OR}x{OC})")
    codes = np.zeros((OR, OC // 2), dtype=np.uint8)
    scales = np.zeros((OR, OC // block), dtype=np.uint8)
    g = ctypes.c_float()
    gin = ctypes.byref(ctypes.c_float(g_in)) if g_in is not None else None
    st = lib().oracle_quantize_nvfp4_block(_ptr(b, ctypes.c_uint16), rows, cols, orient, rnd, seed, stream_id,
                                           gin, block, _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                           ctypes.byref(g), psel, nsel)
    if st == 1:
        raise NonFiniteInput("non-finite input")
    if st != 0:
        raise ValueError(f"bad block size {block} or shape {OR}x{OC}")
    return NVFP4Block(codes, scales, g.value, OR, OC, block)


def quantize_fp8(x, orient: int = 0, rnd: int = RTN, seed: int = 0, stream_id: int = 0,
                 s_in: float | None = None, rows=None, index_base: int = 0) -> FP8:
    """E4M3 with one tensor scale; orientation, rows and index_base as for quantize_nvfp4."""
    b = _bits(x)
    sel, psel, nsel = _selection(rows)
    rows, cols = b.shape
    OR, OC = (rows, cols) if orient == 0 else (cols, rows)
    if sel is not None:
        assert np.all((sel >= 0) & (sel < OR))
        OR = nsel
    codes = np.zeros((OR, OC), dtype=np.uint8)
    s = ctypes.c_float()
    sin = ctypes.byref(ctypes.c_float(s_in)) if s_in is not None else None
    st = lib().oracle_quantize_fp8_at(_ptr(b, ctypes.c_uint16), rows, cols, orient, rnd, seed, stream_id,
                                      sin, index_base, _ptr(codes, ctypes.c_uint8), ctypes.byref(s), psel, nsel)
    if st == 1:
        raise NonFiniteInput("non-finite input")
    return FP8(codes, s.value, OR, OC)


class E5M2:
    """An FP8 E5M2 tensor of shape (rows, cols) with one fp32 scale s."""

    def __init__(self, codes, s, rows, cols):
        self.codes, self.s, self.rows, self.cols = codes, s, rows, cols

    def dequant(self) -> np.ndarray:
        out = np.empty((self.rows, self.cols), dtype=np.float64)
        lib().oracle_dequant_e5m2(_ptr(self.codes, ctypes.c_uint8), self.s, self.rows * self.cols,
                                  _ptr(out, ctypes.c_double))
        return out


def quantize_e5m2(x, orient: int = 0, rnd: int = RTN, seed: int = 0, stream_id: int = 0,
                  s_in: float | None = None, rows=None) -> E5M2:
    """FP8 E5M2 quantization with one tensor scale amax / 57344; orientation,
    random bits and row selection as for the other formats."""
    b = _bits(x)
    sel, psel, nsel = _selection(rows)
    rows, cols = b.shape
    OR, OC = (rows, cols) if orient == 0 else (cols, rows)
    if sel is not None:
        assert np.all((sel >= 0) & (sel < OR))
        OR = nsel
    codes = np.zeros((OR, OC), dtype=np.uint8)
    s = ctypes.c_float()
    sin = ctypes.byref(ctypes.c_float(s_in)) if s_in is not None else None
    st = lib().oracle_quantize_e5m2(_ptr(b, ctypes.c_uint16), rows, cols, orient, rnd, seed, stream_id,
                                    sin, _ptr(codes, ctypes.c_uint8), ctypes.byref(s), psel, nsel)
    if st == 1:
        raise NonFiniteInput("non-finite input")
    return E5M2(codes, s.value, OR, OC)


def quantize_mxfp4(x, orient: int = 0, rnd: int = RTN, seed: int = 0, stream_id: int = 0, rows=None) -> MXFP4:
    """MXFP4 quantization (OCP Microscaling v1.0: 32 E2M1 values per E8M0
    power-of-two scale) of a bf16 (rows, cols) tensor; orientation, random
    bits and the output-row selection as for NVFP4."""
    b = _bits(x)
    sel, psel, nsel = _selection(rows)
    rows, cols = b.shape
    OR, OC = (rows, cols) if orient == 0 else (cols, rows)
    if sel is not None:
        assert np.all((sel >= 0) & (sel < OR))
        OR = nsel
    codes = np.zeros((OR, OC // 2), dtype=np.uint8)
    scales = np.zeros((OR, OC // 32), dtype=np.uint8)
    st = lib().oracle_quantize_mxfp4(_ptr(b, ctypes.c_uint16), rows, cols, orient, rnd, seed, stream_id,
                                     _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8), psel, nsel)
    if st == 1:
        raise NonFiniteInput("non-finite input")
    if st != 0:
        raise ValueError(f"shape error: blocks of 32 need the blocked dim % 32 == 0 (got {OR}x{OC})")
    return MXFP4(codes, scales, OR, OC)


def quantize(fmt: str, x, orient=0, rnd=RTN, seed=0, stream_id=0, rows=None):
    if fmt == "e5m2":
        return quantize_e5m2(x, orient, rnd, seed, stream_id, rows=rows)
    if fmt == "mxfp4":
        return quantize_mxfp4(x, orient, rnd, seed, stream_id, rows=rows)
    if fmt == "nvfp4":
        return quantize_nvfp4(x, orient, rnd, seed, stream_id, rows=rows)
    if fmt.startswith("nvfp4-b"):   # nvfp4-b32 / -b64 / -b128: longer scale blocks
        return quantize_nvfp4_block(x, int(fmt[7:]), orient, rnd, seed, stream_id, rows=rows)
    if fmt == "fp8":
        return quantize_fp8(x, orient, rnd, seed, stream_id, rows=rows)
    raise ValueError(fmt)


# ----------------------------------------------------------------------------- GEMMs (SNIP Figure 5)

def gemm_tn(a_hat: np.ndarray, b_hat: np.ndarray, rows: np.ndarray | None = None) -> np.ndarray:
    """D = A_hat @ B_hat^T in fp64 on dequantized operands (both stored with the
    contraction dim last).  ``rows`` restricts the result to selected rows of A."""
    if rows is not None:
        a_hat = a_hat[rows]
    return np.matmul(a_hat, b_hat.T)


# stream ids of the six quantizations of one linear layer
TAG_X_FWD, TAG_W_FWD, TAG_DY_DGRAD, TAG_WT_DGRAD, TAG_DYT_WGRAD, TAG_XT_WGRAD = range(6)


def stream_id(layer: int, tag: int) -> int:
    return layer * 8 + tag


def qlinear_fwd(fmt, X, W, layer=0, seed=0, rnd_x=RTN, rnd_w=RTN, rows=None):
    """Y = Q(X) Q(W)^T, both quantized along K (forward: round to nearest)."""
    xq = quantize(fmt, X, 0, rnd_x, seed, stream_id(layer, TAG_X_FWD))
    wq = quantize(fmt, W, 0, rnd_w, seed, stream_id(layer, TAG_W_FWD))
    return gemm_tn(xq.dequant(), wq.dequant(), rows)


def qlinear_dgrad(fmt, dY, W, layer=0, seed=0, rnd_dy=SR, rnd_wt=SR, rows=None):
    """dX = Q(dY) Q(W^T)^T: dY quantized along N (its rows), W along N (its
    columns, i.e. W^T along its rows); stochastic rounding by default."""
    dyq = quantize(fmt, dY, 0, rnd_dy, seed, stream_id(layer, TAG_DY_DGRAD))
    wtq = quantize(fmt, W, 1, rnd_wt, seed, stream_id(layer, TAG_WT_DGRAD))
    return gemm_tn(dyq.dequant(), wtq.dequant(), rows)


def qlinear_wgrad(fmt, dY, X, layer=0, seed=0, rnd_dyt=SR, rnd_xt=SR, rows=None):
    """dW = Q(dY^T) Q(X^T)^T: both quantized along T (the token dim)."""
    dytq = quantize(fmt, dY, 1, rnd_dyt, seed, stream_id(layer, TAG_DYT_WGRAD))
    xtq = quantize(fmt, X, 1, rnd_xt, seed, stream_id(layer, TAG_XT_WGRAD))
    return gemm_tn(dytq.dequant(), xtq.dequant(), rows)


def dw_noise(X, dY, dW_q):
    """The weight-gradient form of the sqrt(3) check ("FP4 all the way",
    Outline): with dW = dY^T X of the unquantized bf16 tensors (fp64 product),
    returns (||dW||^2, ||dW_q - dW||^2)."""
    x = _bits_to_f64(X)
    dy = _bits_to_f64(dY)
    dw = dy.T @ x
    d = np.asarray(dW_q, dtype=np.float64) - dw
    return float(np.sum(dw * dw)), float(np.sum(d * d))


# ----------------------------------------------------------------------------- statistics

def quant_stats(x, rnd=RTN, seed=0, stream_id=0, want_block_err=False, g_in=None, s_in=None, index_base=0):
    """SNIP statistics of one tensor: raw sums (ST_* slots) plus derived ratios.
    ratio_f = ||A|| / ||Q_f(A) - A||, below_sqrt3_f = ratio_f < sqrt(3) ("FP4 all
    the way", Outline: quantized learning loses efficiency when the gradient
    norm falls below ~sqrt(3) x the quantization noise).  For a part of a larger
    tensor: g_in / s_in its tensor scales and index_base the part's first
    element (the raw sums of the parts add up to the tensor's)."""
    b = _bits(x)
    rows, cols = b.shape
    raw = np.zeros(ST_N, dtype=np.float64)
    be4 = np.zeros((rows, cols // 16), dtype=np.float64) if want_block_err else None
    be8 = np.zeros((rows, cols // 16), dtype=np.float64) if want_block_err else None
    gin = ctypes.byref(ctypes.c_float(g_in)) if g_in is not None else None
    sin = ctypes.byref(ctypes.c_float(s_in)) if s_in is not None else None
    st = lib().oracle_quant_stats_at(_ptr(b, ctypes.c_uint16), rows, cols, rnd, seed, stream_id, gin, sin,
                                     index_base, _ptr(raw, ctypes.c_double),
                                  _ptr(be4, ctypes.c_double) if be4 is not None else None,
                                  _ptr(be8, ctypes.c_double) if be8 is not None else None)
    if st == 1:
        raise NonFiniteInput("non-finite input")
    if st != 0:
        raise ValueError("shape error")
    return derive_stats(raw) | {"raw": raw, "block_err_nvfp4": be4, "block_err_fp8": be8}


def derive_stats(raw) -> dict:
    def ratio(num, den):
        if den == 0.0:
            return math.inf
        return math.sqrt(num / den)
    r4 = ratio(raw[ST_SUM_X2], raw[ST_NVFP4_ERR2])
    r8 = ratio(raw[ST_SUM_X2], raw[ST_FP8_ERR2])
    return {
        "sum_x2": raw[ST_SUM_X2], "nvfp4_err2": raw[ST_NVFP4_ERR2], "fp8_err2": raw[ST_FP8_ERR2],
        "nvfp4_sr_var": raw[ST_NVFP4_SRVAR], "fp8_sr_var": raw[ST_FP8_SRVAR],
        "amax": raw[ST_AMAX], "count": raw[ST_COUNT],
        "ratio_nvfp4": r4, "ratio_fp8": r8,
        "below_sqrt3_nvfp4": r4 < math.sqrt(3.0), "below_sqrt3_fp8": r8 < math.sqrt(3.0),
    }
