"""Python binding of the CSA2 C-ABI library (libcsa2.so, sm_103a).

Argument marshalling only: every function here forwards torch CUDA tensors as raw
device pointers to the entry point of the same name in ``include/csa2.h`` and raises
:class:`Csa2Error` on a non-zero status.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and importing this
module fails loudly when the library has not been built.
"""
import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "Csa2Error", "Swa", "lib", "csa2_version", "csa2_last_error", "csa2_device_status",
    "csa2_compress",
    "csa2_compress_index",
    "csa2_index_topk_workspace_size", "csa2_index_topk", "csa2_compress_index_topk",
    "csa2_index_topk_noalloc",
    "csa2_index_topk_pool_workspace_size", "csa2_index_topk_pool", "csa2_topk_workspace_size",
    "csa2_index_plane_fp8_bytes", "csa2_index_plane_fp8", "csa2_index_topk_fp8_workspace_size",
    "csa2_index_topk_fp8", "csa2_index_plane_fp4_bytes", "csa2_index_plane_fp4",
    "csa2_index_topk_fp4_workspace_size", "csa2_index_topk_fp4",
    "csa2_topk_scores", "csa2_attn_workspace_size", "csa2_sparse_attn", "csa2_reuse_attn",
    "csa2_sparse_attn_rope", "csa2_reuse_attn_rope", "csa2_plane_fp4_bytes", "csa2_plane_fp4",
    "csa2_sparse_attn_fp4", "csa2_selftest_wait_timeout",
]

STATUS = {0: "CSA2_OK", 1: "CSA2_EINVAL", 2: "CSA2_ECUDA", 3: "CSA2_ETIMEOUT", 4: "CSA2_EBOUNDS",
          5: "CSA2_ENOSPACE"}
SWA_RING, SWA_LINEAR = 0, 1
SWA_BF16, SWA_FP8_S128, SWA_FP8_E8M0 = 0, 1, 2


class Csa2Error(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class _SwaC(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("dtype", ctypes.c_int32), ("data", ctypes.c_void_p),
                ("n_rows", ctypes.c_int64), ("lin_base", ctypes.c_void_p),
                ("lin_pos0", ctypes.c_void_p)]


_vp, _i32, _i64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_size_t)
_SIGS = {
    "csa2_last_error": ([], ctypes.c_char_p),
    "csa2_version": ([], ctypes.c_char_p),
    "csa2_device_status": ([_vp], _i32),
    "csa2_selftest_wait_timeout": ([_i64, _vp], _i32),
    "csa2_compress": ([_vp, _vp, _i32, _vp, _i32, _vp, _i32, _vp, _vp, _vp, _i64, _vp, _vp, _f32,
                       _vp, _vp], _i32),
    "csa2_compress_index": ([_vp, _vp, _i32, _vp, _i32, _vp, _i32, _vp, _vp, _vp, _i64, _vp,
                             _vp, _f32, _vp, _vp, _vp, _vp, _vp], _i32),
    "csa2_index_topk_workspace_size": ([_i32, _i32, _i64, _i32], _sz),
    "csa2_index_topk": ([_vp, _vp, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _i32,
                         _i32, _i64, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "csa2_compress_index_topk": ([_vp, _vp, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _f32,
                                  _vp, _vp, _vp, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _i32,
                                  _vp, _i32, _i32, _i32, _i64, _vp, _vp, _vp, _vp, _sz, _vp],
                                 _i32),
    "csa2_index_topk_noalloc": ([_vp, _vp, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _i32, _vp,
                                 _i32, _i32, _i32, _i64, _vp, _vp, _vp, _vp], _i32),
    "csa2_index_topk_pool_workspace_size": ([_i32, _i32, _i64, _i32, _i32], _sz),
    "csa2_index_topk_pool": ([_vp, _vp, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32,
                              _i64, _vp, _vp, _vp, _i32, _vp, _vp, _sz, _vp], _i32),
    "csa2_index_plane_fp8_bytes": ([_i64], _sz),
    "csa2_index_plane_fp8": ([_vp, _i64, _vp, _vp], _i32),
    "csa2_index_topk_fp8_workspace_size": ([_i32, _i32, _i64, _i32], _sz),
    "csa2_index_topk_fp8": ([_vp, _vp, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _i32, _vp, _i32,
                             _i32, _i32, _i64, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "csa2_index_plane_fp4_bytes": ([_i64], _sz),
    "csa2_index_plane_fp4": ([_vp, _i64, _vp, _vp], _i32),
    "csa2_index_topk_fp4_workspace_size": ([_i32, _i32, _i64, _i32], _sz),
    "csa2_index_topk_fp4": ([_vp, _vp, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _i32, _vp, _i32,
                             _i32, _i32, _i64, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "csa2_topk_workspace_size": ([_i32, _i64, _i32], _sz),
    "csa2_topk_scores": ([_vp, _vp, _i32, _i64, _i32, _vp, _vp, _vp, _sz, _vp], _i32),
    "csa2_attn_workspace_size": ([_i32, _i32], _sz),
    "csa2_sparse_attn": ([_vp, _i32, _vp, _vp, ctypes.POINTER(_SwaC), _vp, _i64, _vp, _vp, _i32,
                          _vp, _f32, _vp, _vp, _vp, _sz, _vp], _i32),
    "csa2_reuse_attn": ([_vp, _i32, _vp, _vp, ctypes.POINTER(_SwaC), _vp, _i64, _vp, _vp, _i32,
                         _vp, _f32, _vp, _vp, _vp, _sz, _vp], _i32),
    "csa2_sparse_attn_rope": ([_vp, _i32, _vp, _vp, ctypes.POINTER(_SwaC), _vp, _i64, _vp, _vp,
                               _i32, _vp, _f32, _vp, _vp, _vp, _sz, _vp, _vp], _i32),
    "csa2_plane_fp4_bytes": ([_i64], _sz),
    "csa2_plane_fp4": ([_vp, _i64, _vp, _vp], _i32),
    "csa2_sparse_attn_fp4": ([_vp, _i32, _vp, _vp, ctypes.POINTER(_SwaC), _vp, _i64, _vp, _vp,
                              _i32, _vp, _f32, _vp, _vp, _vp, _sz, _vp, _vp], _i32),
    "csa2_reuse_attn_rope": ([_vp, _i32, _vp, _vp, ctypes.POINTER(_SwaC), _vp, _i64, _vp, _vp,
                              _i32, _vp, _f32, _vp, _vp, _vp, _sz, _vp, _vp], _i32),
}

_LIB = None


def lib():
    """The loaded libcsa2.so (raises if it was not built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libcsa2.so not found at {_build.LIB}: run __graft_entry__.build()")
        L = ctypes.CDLL(_build.LIB)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _LIB = L
    return _LIB


def _check(st):
    if st != 0:
        raise Csa2Error(st, lib().csa2_last_error().decode())


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("csa2: tensors must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("csa2: tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def csa2_version():
    return lib().csa2_version().decode()


def csa2_last_error():
    """Text of the last failure on the calling thread ('' if none)."""
    return (lib().csa2_last_error() or b"").decode()


def csa2_device_status(stream=None):
    _check(lib().csa2_device_status(_stream(stream)))


def csa2_selftest_wait_timeout(limit_ns, stream=None):
    _check(lib().csa2_selftest_wait_timeout(int(limit_ns), _stream(stream)))


@dataclass
class Swa:
    """Window source of csa2_sparse_attn: RING [B,128,row] or LINEAR rows."""
    data: torch.Tensor
    mode: int = SWA_RING
    lin_base: Optional[torch.Tensor] = None
    lin_pos0: Optional[torch.Tensor] = None
    fp8_dtype: int = SWA_FP8_S128  # the layout of uint8 rows: SWA_FP8_S128 or SWA_FP8_E8M0

    def c(self):
        dtype = self.fp8_dtype if self.data.dtype == torch.uint8 else SWA_BF16
        row = 512 if dtype == SWA_BF16 else 528
        n_rows = self.data.numel() // row
        return _SwaC(self.mode, dtype, _p(self.data), n_rows, _p(self.lin_base), _p(self.lin_pos0))


def csa2_compress(kv, score, cu_seqlens, start_pos, ratio, kv_state, score_state, plane, row_base,
                  inv_freq, norm_w=None, eps=1e-6, stream=None):
    T = kv.shape[0]
    B = cu_seqlens.numel() - 1
    _check(lib().csa2_compress(_p(kv), _p(score), T, _p(cu_seqlens), B, _p(start_pos), ratio,
                               _p(kv_state), _p(score_state), _p(plane), plane.shape[0],
                               _p(row_base), _p(norm_w), float(eps), _p(inv_freq),
                               _stream(stream)))


def csa2_compress_index(kv, score, cu_seqlens, start_pos, ratio, kv_state, score_state, plane,
                        row_base, inv_freq, wk, index_plane, knorm_w=None, norm_w=None, eps=1e-6,
                        stream=None):
    """csa2_compress plus each written row's index K (wk [128, 512] bf16) in index_plane."""
    T = kv.shape[0]
    B = cu_seqlens.numel() - 1
    _check(lib().csa2_compress_index(_p(kv), _p(score), T, _p(cu_seqlens), B, _p(start_pos),
                                     ratio, _p(kv_state), _p(score_state), _p(plane),
                                     plane.shape[0], _p(row_base), _p(norm_w), float(eps),
                                     _p(inv_freq), _p(wk), _p(knorm_w), _p(index_plane),
                                     _stream(stream)))


def csa2_index_topk_workspace_size(Q, H, max_scored, k):
    return int(lib().csa2_index_topk_workspace_size(Q, H, max_scored, k))


def csa2_index_topk(iq, w, index_k, row_base, q_seq, q_pos, ratio, k, max_scored, sel,
                    ws, sel_scores=None, cand=None, relu=True, scores_out=None, stream=None):
    Q, H = iq.shape[0], iq.shape[1]
    ncb = 0 if cand is None else cand.shape[1]
    _check(lib().csa2_index_topk(_p(iq), _p(w), Q, H, _p(index_k), index_k.shape[0],
                                 _p(row_base), _p(q_seq), _p(q_pos), ratio, _p(cand), ncb, k,
                                 1 if relu else 0, max_scored, _p(sel), _p(sel_scores),
                                 _p(scores_out), _p(ws), ws.numel() * ws.element_size(),
                                 _stream(stream)))


def csa2_compress_index_topk(kv, score, cu_seqlens, start_pos, kv_state, score_state, plane,
                             inv_freq, iq, w, index_k, row_base, q_seq, q_pos, ratio, k,
                             max_scored, sel, ws, sel_scores=None, cand=None, relu=True,
                             scores_out=None, norm_w=None, eps=1e-6, stream=None):
    """csa2_compress followed by csa2_index_topk in one call (the compressor's tokens run on
    extra CTAs of the top-k launch)."""
    T = kv.shape[0]
    B = cu_seqlens.numel() - 1
    Q, H = iq.shape[0], iq.shape[1]
    ncb = 0 if cand is None else cand.shape[1]
    _check(lib().csa2_compress_index_topk(
        _p(kv), _p(score), T, _p(cu_seqlens), B, _p(start_pos), _p(kv_state), _p(score_state),
        _p(plane), plane.shape[0], _p(norm_w), float(eps), _p(inv_freq), _p(iq), _p(w), Q, H,
        _p(index_k), index_k.shape[0], _p(row_base), _p(q_seq), _p(q_pos), ratio, _p(cand), ncb,
        k, 1 if relu else 0, max_scored, _p(sel), _p(sel_scores), _p(scores_out), _p(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def csa2_index_topk_noalloc(iq, w, index_k, row_base, q_seq, q_pos, ratio, k, max_scored, sel,
                            sel_scores=None, cand=None, relu=True, scores_out=None, stream=None):
    """csa2_index_topk without a workspace: for callers that cannot allocate device
    memory; its scratch is a fixed 64 MiB device array inside the library."""
    Q, H = iq.shape[0], iq.shape[1]
    ncb = 0 if cand is None else cand.shape[1]
    _check(lib().csa2_index_topk_noalloc(_p(iq), _p(w), Q, H, _p(index_k), index_k.shape[0],
                                         _p(row_base), _p(q_seq), _p(q_pos), ratio, _p(cand),
                                         ncb, k, 1 if relu else 0, max_scored, _p(sel),
                                         _p(sel_scores), _p(scores_out), _stream(stream)))


def csa2_index_topk_pool_workspace_size(Q, H, max_scored, k, nbk):
    return int(lib().csa2_index_topk_pool_workspace_size(Q, H, max_scored, k, nbk))


def csa2_index_topk_pool(iq, w, index_k, row_base, q_seq, q_pos, ratio, k, max_scored, sel,
                         pool, ws, sel_scores=None, relu=True, scores_out=None, stream=None):
    """FULL-mode csa2_index_topk plus the candidate pool [Q][nbk] (nbk = pool.shape[1])."""
    Q, H = iq.shape[0], iq.shape[1]
    _check(lib().csa2_index_topk_pool(_p(iq), _p(w), Q, H, _p(index_k), index_k.shape[0],
                                      _p(row_base), _p(q_seq), _p(q_pos), ratio, k,
                                      1 if relu else 0, max_scored, _p(sel), _p(sel_scores),
                                      _p(scores_out), pool.shape[1], _p(pool), _p(ws),
                                      ws.numel() * ws.element_size(), _stream(stream)))


def csa2_index_plane_fp8_bytes(rows):
    return int(lib().csa2_index_plane_fp8_bytes(rows))


def csa2_index_plane_fp8(index_k, plane, stream=None):
    """bf16 index rows [rows, 128] -> FP8 plane bytes (blocks of 8 rows, 1056 B each)."""
    _check(lib().csa2_index_plane_fp8(_p(index_k), index_k.shape[0], _p(plane), _stream(stream)))


def csa2_index_topk_fp8_workspace_size(Q, H, max_scored, k):
    return int(lib().csa2_index_topk_fp8_workspace_size(Q, H, max_scored, k))


def csa2_index_topk_fp8(iq, w, plane, index_rows, row_base, q_seq, q_pos, ratio, k, max_scored,
                        sel, ws, sel_scores=None, cand=None, relu=True, scores_out=None,
                        stream=None):
    """csa2_index_topk on an FP8 index plane of index_rows rows."""
    Q, H = iq.shape[0], iq.shape[1]
    ncb = 0 if cand is None else cand.shape[1]
    _check(lib().csa2_index_topk_fp8(_p(iq), _p(w), Q, H, _p(plane), index_rows, _p(row_base),
                                     _p(q_seq), _p(q_pos), ratio, _p(cand), ncb, k,
                                     1 if relu else 0, max_scored, _p(sel), _p(sel_scores),
                                     _p(scores_out), _p(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)))


def csa2_index_plane_fp4_bytes(rows):
    return int(lib().csa2_index_plane_fp4_bytes(rows))


def csa2_index_plane_fp4(index_k, plane, stream=None):
    """bf16 index rows [rows, 128] -> MXFP4 plane bytes (blocks of 8 rows, 544 B each)."""
    _check(lib().csa2_index_plane_fp4(_p(index_k), index_k.shape[0], _p(plane), _stream(stream)))


def csa2_index_topk_fp4_workspace_size(Q, H, max_scored, k):
    return int(lib().csa2_index_topk_fp4_workspace_size(Q, H, max_scored, k))


def csa2_index_topk_fp4(iq, w, plane, index_rows, row_base, q_seq, q_pos, ratio, k, max_scored,
                        sel, ws, sel_scores=None, cand=None, relu=True, scores_out=None,
                        stream=None):
    """csa2_index_topk on an MXFP4 index plane of index_rows rows."""
    Q, H = iq.shape[0], iq.shape[1]
    ncb = 0 if cand is None else cand.shape[1]
    _check(lib().csa2_index_topk_fp4(_p(iq), _p(w), Q, H, _p(plane), index_rows, _p(row_base),
                                     _p(q_seq), _p(q_pos), ratio, _p(cand), ncb, k,
                                     1 if relu else 0, max_scored, _p(sel), _p(sel_scores),
                                     _p(scores_out), _p(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)))


def csa2_topk_workspace_size(Q, ld, k):
    return int(lib().csa2_topk_workspace_size(Q, ld, k))


def csa2_topk_scores(scores, n, k, sel, sel_scores=None, ws=None, stream=None):
    Q, ld = scores.shape
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().csa2_topk_scores(_p(scores), _p(n), Q, ld, k, _p(sel), _p(sel_scores), _p(ws),
                                  nbytes, _stream(stream)))


def csa2_attn_workspace_size(Q, nsel):
    return int(lib().csa2_attn_workspace_size(Q, nsel))


def _attn(fn, q, q_seq, q_pos, swa, plane, row_base, sel, sink, out, lse, scale, ws, stream,
          *extra):
    sw = swa.c()
    nsel = 0 if sel is None else sel.shape[1]
    plane_rows = 0 if plane is None else plane.shape[0]
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(fn(_p(q), q.shape[0], _p(q_seq), _p(q_pos), ctypes.byref(sw), _p(plane), plane_rows,
              _p(row_base), _p(sel), nsel, _p(sink), float(scale), _p(out), _p(lse), _p(ws),
              nbytes, *[_p(x) for x in extra], _stream(stream)))


def csa2_sparse_attn(q, q_seq, q_pos, swa: Swa, plane, row_base, sel, sink, out, lse=None,
                     scale=512 ** -0.5, ws=None, stream=None):
    _attn(lib().csa2_sparse_attn, q, q_seq, q_pos, swa, plane, row_base, sel, sink, out, lse,
          scale, ws, stream)


def csa2_reuse_attn(q, q_seq, q_pos, swa: Swa, plane, row_base, sel, sink, out, lse=None,
                    scale=512 ** -0.5, ws=None, stream=None):
    _attn(lib().csa2_reuse_attn, q, q_seq, q_pos, swa, plane, row_base, sel, sink, out, lse,
          scale, ws, stream)


def csa2_sparse_attn_rope(q, q_seq, q_pos, swa: Swa, plane, row_base, sel, sink, out, inv_freq,
                          lse=None, scale=512 ** -0.5, ws=None, stream=None):
    """csa2_sparse_attn with the output's dims 448..511 rotated back by q_pos."""
    _attn(lib().csa2_sparse_attn_rope, q, q_seq, q_pos, swa, plane, row_base, sel, sink, out,
          lse, scale, ws, stream, inv_freq)


def csa2_reuse_attn_rope(q, q_seq, q_pos, swa: Swa, plane, row_base, sel, sink, out, inv_freq,
                         lse=None, scale=512 ** -0.5, ws=None, stream=None):
    """csa2_reuse_attn with the output's dims 448..511 rotated back by q_pos."""
    _attn(lib().csa2_reuse_attn_rope, q, q_seq, q_pos, swa, plane, row_base, sel, sink, out,
          lse, scale, ws, stream, inv_freq)


def csa2_plane_fp4_bytes(rows):
    return int(lib().csa2_plane_fp4_bytes(rows))


def csa2_plane_fp4(plane, out, stream=None):
    """bf16 plane rows [rows, 512] -> FP4 rows (288 bytes each) in out."""
    _check(lib().csa2_plane_fp4(_p(plane), plane.shape[0], _p(out), _stream(stream)))


def csa2_sparse_attn_fp4(q, q_seq, q_pos, swa, plane4, plane_rows, row_base, sel, sink, out,
                         inv_freq=None, lse=None, scale=512 ** -0.5, ws=None, stream=None):
    """csa2_sparse_attn with the selected rows read from an FP4 plane of plane_rows rows."""
    Q = q.shape[0]
    nsel = 0 if sel is None else sel.shape[1]
    sw = swa.c()
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().csa2_sparse_attn_fp4(_p(q), Q, _p(q_seq), _p(q_pos), ctypes.byref(sw),
                                      _p(plane4), plane_rows, _p(row_base), _p(sel), nsel,
                                      _p(sink), float(scale), _p(out), _p(lse), _p(ws), nbytes,
                                      _p(inv_freq), _stream(stream)))
