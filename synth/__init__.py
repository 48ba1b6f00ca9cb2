"""Seeded synthetic inputs shared by the oracle harness, the tests and the benchmark.

Every tensor is a pure function of (seed, stream id, logical element id); the host
library and the device library compute the same bits (see ``synth.h``).  Nothing
here performs any step of the attention method.
"""
import ctypes
import os

import numpy as np
import torch

from . import build as _build

_HOST = None
_CUDA = None

# Stream ids: one per logical tensor.
KV, SCORE, PLANE, INDEX_K, RING, Q, IQ, W, SINK, LENGTHS, CAND, SWA_LINEAR = range(1, 13)
LAYER_STRIDE = 64  # per-layer tensors use stream + LAYER_STRIDE * layer

_i64, _u64, _vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p


def _host():
    global _HOST
    if _HOST is None:
        if not os.path.exists(_build.HOST_LIB):
            _build.build(cuda=False)
        lib = ctypes.CDLL(_build.HOST_LIB)
        lib.synth_fill_normal_bf16.argtypes = [_vp, _i64, _u64, _u64, _u64]
        lib.synth_fill_normal_f32.argtypes = [_vp, _i64, _u64, _u64, _u64]
        lib.synth_fill_u64.argtypes = [_vp, _i64, _u64, _u64, _u64]
        lib.synth_fill_rows_bf16.argtypes = [_vp, _u64, _i64, _i64, _i64, _u64, _u64]
        lib.synth_fill_rows_f32.argtypes = [_vp, _u64, _i64, _i64, _i64, _u64, _u64]
        lib.synth_fill_rowlist_bf16.argtypes = [_vp, _u64, _vp, _i64, _i64, _u64, _u64]
        lib.synth_fill_rows_fp8s128.argtypes = [_vp, _u64, _i64, _i64, _u64, _u64]
        for f in ("synth_fill_normal_bf16", "synth_fill_normal_f32", "synth_fill_u64",
                  "synth_fill_rows_bf16", "synth_fill_rows_f32", "synth_fill_rowlist_bf16",
                  "synth_fill_rows_fp8s128"):
            getattr(lib, f).restype = None
        _HOST = lib
    return _HOST


def _cuda():
    global _CUDA
    if _CUDA is None:
        if not os.path.exists(_build.CUDA_LIB):
            raise RuntimeError("device input generator not built (run __graft_entry__.build())")
        lib = ctypes.CDLL(_build.CUDA_LIB)
        lib.synth_fill_normal_bf16_cuda.argtypes = [_vp, _i64, _u64, _u64, _u64, _vp]
        lib.synth_fill_normal_f32_cuda.argtypes = [_vp, _i64, _u64, _u64, _u64, _vp]
        lib.synth_fill_rows_bf16_cuda.argtypes = [_vp, _u64, _i64, _i64, _i64, _u64, _u64, _vp]
        lib.synth_fill_rows_fp8s128_cuda.argtypes = [_vp, _u64, _i64, _i64, _u64, _u64, _vp]
        for f in ("synth_fill_normal_bf16_cuda", "synth_fill_normal_f32_cuda",
                  "synth_fill_rows_bf16_cuda", "synth_fill_rows_fp8s128_cuda"):
            getattr(lib, f).restype = ctypes.c_int
        _CUDA = lib
    return _CUDA


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"device input generator failed: cudaError {rc}")


def u64(n, seed, stream, offset=0):
    out = np.empty(n, dtype=np.uint64)
    _host().synth_fill_u64(out.ctypes.data, n, seed, stream, offset)
    return out


def normal_f32(n, seed, stream, offset=0, device="cpu"):
    out = torch.empty(n, dtype=torch.float32, device=device)
    if out.is_cuda:
        _check(_cuda().synth_fill_normal_f32_cuda(out.data_ptr(), n, seed, stream, offset, _stream()))
    else:
        _host().synth_fill_normal_f32(out.data_ptr(), n, seed, stream, offset)
    return out


def rows_bf16(b, j0, nrows, D, seed, stream, device="cpu", out=None):
    """Rows j0..j0+nrows-1 (width D) of sequence b, bf16 ~N(0,1)."""
    if out is None:
        out = torch.empty((nrows, D), dtype=torch.bfloat16, device=device)
    assert out.is_contiguous() and out.numel() == nrows * D and out.dtype == torch.bfloat16
    if nrows == 0:
        return out
    if out.is_cuda:
        _check(_cuda().synth_fill_rows_bf16_cuda(out.data_ptr(), b, j0, nrows, D, seed, stream,
                                                  _stream()))
    else:
        _host().synth_fill_rows_bf16(out.data_ptr(), b, j0, nrows, D, seed, stream)
    return out


def rows_f32(b, j0, nrows, D, seed, stream):
    """Same elements as rows_bf16 before the bf16 rounding (host only)."""
    out = torch.empty((nrows, D), dtype=torch.float32)
    if nrows:
        _host().synth_fill_rows_f32(out.data_ptr(), b, j0, nrows, D, seed, stream)
    return out


def rowlist_bf16(b, rows, D, seed, stream):
    """Host rows listed in `rows` (int64 array) of sequence b."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = torch.empty((len(rows), D), dtype=torch.bfloat16)
    if len(rows):
        _host().synth_fill_rowlist_bf16(out.data_ptr(), b, rows.ctypes.data, len(rows), D, seed,
                                        stream)
    return out


def rows_fp8s128(b, j0, nrows, seed, stream, device="cpu", out=None):
    """FP8 E4M3 rows with four fp32 scales each: uint8 [nrows, 528]."""
    if out is None:
        out = torch.empty((nrows, 528), dtype=torch.uint8, device=device)
    assert out.is_contiguous() and out.numel() == nrows * 528
    if nrows == 0:
        return out
    if out.is_cuda:
        _check(_cuda().synth_fill_rows_fp8s128_cuda(out.data_ptr(), b, j0, nrows, seed, stream,
                                                     _stream()))
    else:
        _host().synth_fill_rows_fp8s128(out.data_ptr(), b, j0, nrows, seed, stream)
    return out
