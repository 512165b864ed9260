"""Helpers shared by the GPU parity tests: unpacking the MMA operand layout,
and the GEMM tolerance (relative Frobenius error <= 1e-5 and max |diff| <=
1e-3 * rms of the fp64 reference)."""
import numpy as np
import torch

GEMM_REL_FRO = 1e-5
GEMM_MAX_ABS_OF_RMS = 1e-3
STATS_REL = 1e-4


def need_gpu():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sub_byte_mixed_gb300 import build, snip
    build.build()
    snip.load()
    snip.snip_device_check()
    return snip


def mma_codes_to_rowmajor(codes, out_rows, out_cols, fmt_nvfp4=True):
    """Slice the padded MMA-layout code matrix back to out_rows x (bytes per row)."""
    c = codes.cpu().numpy()
    ocp = ((out_cols + 255) // 256 * 256) if fmt_nvfp4 else ((out_cols + 127) // 128 * 128)
    orp = (out_rows + 255) // 256 * 256
    width = ocp // 2 if fmt_nvfp4 else ocp
    m = c.reshape(orp, width)
    return m, m[:out_rows, : (out_cols // 2 if fmt_nvfp4 else out_cols)]


def mma_scales_to_rowmajor(scales, out_rows, out_cols):
    """Gather the chunked MMA-layout E4M3 scales into a padded rows x blocks matrix."""
    s = scales.cpu().numpy()
    ocp = (out_cols + 255) // 256 * 256
    orp = (out_rows + 255) // 256 * 256
    r = np.arange(orp)[:, None]
    kb = np.arange(ocp // 16)[None, :]
    chunk = (r // 128) * (ocp // 64) + kb // 4
    off = chunk * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    full = s[off]
    return full, full[:out_rows, : out_cols // 16]


def gemm_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what
    nrm = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nrm if nrm > 0 else np.linalg.norm(got)
    rms = np.sqrt(np.mean(ref ** 2))
    mx = np.max(np.abs(got - ref)) if ref.size else 0.0
    assert rel <= GEMM_REL_FRO, f"{what}: rel Frobenius {rel:.3e}"
    assert mx <= GEMM_MAX_ABS_OF_RMS * rms + 1e-30, f"{what}: max abs {mx:.3e} vs rms {rms:.3e}"
    return rel, mx / rms if rms > 0 else 0.0


def mma_mx_scales_to_rowmajor(scales, out_rows, out_cols):
    """Gather the chunked MMA-layout E8M0 scales of MXFP4 (chunks of four
    32-element blocks) into a padded rows x blocks matrix."""
    s = scales.cpu().numpy()
    ocp = (out_cols + 255) // 256 * 256
    orp = (out_rows + 255) // 256 * 256
    r = np.arange(orp)[:, None]
    kb = np.arange(ocp // 32)[None, :]
    chunk = (r // 128) * (ocp // 128) + kb // 4
    off = chunk * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    full = s[off]
    return full, full[:out_rows, : out_cols // 32]
