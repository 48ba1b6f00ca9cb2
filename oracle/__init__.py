"""CPU oracle of the CSA2 attention step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline`` /
reference leg may import this package.  The product path never calls it and has
no CPU fallback.  The arithmetic lives in ``oracle.c`` (plain C, IEEE double);
this module only marshals numpy / torch CPU arrays.

Every function is pinned by ``tests/test_oracle_pins.py`` against brute force,
closed forms, invariants and the counts the pages print.
"""
import ctypes
import os

import numpy as np
import torch

from . import build as _build

_LIB = None
_vp, _i32, _i64, _dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double


def lib():
    global _LIB
    if _LIB is None:
        _build.build()
        L = ctypes.CDLL(_build.LIB)
        L.orc_f64_to_bf16.argtypes = [_dbl]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_e4m3_val.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_val.restype = _dbl
        L.orc_n_visible.argtypes = [_i64, _i32]
        L.orc_n_visible.restype = _i64
        L.orc_compress.argtypes = [_vp, _vp, _vp, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
                                   _dbl, _vp]
        L.orc_compress.restype = _i64
        L.orc_compress_index.argtypes = [_vp, _vp, _vp, _i32, _vp, _i32, _vp, _vp, _vp, _vp,
                                         _vp, _vp, _dbl, _vp, _vp, _vp, _vp, _vp]
        L.orc_compress_index.restype = _i64
        L.orc_index_scores.argtypes = [_vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _i32,
                                       _i32, _vp, _vp, _i64]
        L.orc_index_scores.restype = None
        L.orc_e4m3_code.argtypes = [_dbl]
        L.orc_e4m3_code.restype = ctypes.c_uint8
        L.orc_ue8m0_scale.argtypes = [_dbl]
        L.orc_ue8m0_scale.restype = _dbl
        L.orc_index_plane_fp8.argtypes = [_vp, _i64, _vp]
        L.orc_index_plane_fp8.restype = None
        L.orc_index_scores_fp8.argtypes = [_vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp,
                                           _i32, _i32, _vp, _vp, _i64]
        L.orc_index_scores_fp8.restype = None
        L.orc_topk.argtypes = [_vp, _vp, _i64, _i32, _vp]
        L.orc_topk.restype = _i32
        L.orc_sparse_attn.argtypes = [_vp, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _vp,
                                      _vp, _vp, _i32, _vp, _dbl, _vp, _vp]
        L.orc_e2m1_val.argtypes = [ctypes.c_uint8]
        L.orc_e2m1_val.restype = _dbl
        L.orc_e2m1_code.argtypes = [_dbl]
        L.orc_e2m1_code.restype = ctypes.c_uint8
        L.orc_index_plane_fp4.argtypes = [_vp, _i64, _vp]
        L.orc_index_plane_fp4.restype = None
        L.orc_index_scores_fp4.argtypes = [_vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp,
                                           _i32, _i32, _vp, _vp, _i64]
        L.orc_index_scores_fp4.restype = None
        L.orc_plane_fp4.argtypes = [_vp, _i64, _vp]
        L.orc_plane_fp4.restype = None
        L.orc_sparse_attn.restype = None
        L.orc_inverse_rope.argtypes = [_vp, _i32, _vp, _vp]
        L.orc_inverse_rope.restype = None
        L.orc_candidate_pool.argtypes = [_vp, _vp, _i64, _i32, _vp]
        L.orc_candidate_pool.restype = _i32
        _LIB = L
    return _LIB


def _p(a):
    """Address of a C-contiguous numpy array or CPU tensor (None -> NULL)."""
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        assert a.device.type == "cpu" and a.is_contiguous()
        return a.data_ptr()
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def bf16_bits(t):
    """bf16 tensor -> contiguous uint16 numpy view of its bits."""
    t = t.detach().to("cpu").contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_from_bits(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)


def f64_to_bf16(x):
    return lib().orc_f64_to_bf16(float(x))


def e4m3_value(code):
    return lib().orc_e4m3_val(int(code))


def n_visible(p, m):
    return int(lib().orc_n_visible(int(p), int(m)))


def compress(kv, score, cu_seqlens, start_pos, ratio, kv_state, score_state, plane, row_base,
             inv_freq, norm_w=None, eps=1e-6):
    """In place on plane (uint16 bits [rows,512]) and the double states [B,m,512].
    Returns (rows emitted, plane_f64 [rows,512])."""
    kv = bf16_bits(kv) if isinstance(kv, torch.Tensor) else kv
    score = None if score is None else (bf16_bits(score) if isinstance(score, torch.Tensor)
                                        else score)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    sp = np.ascontiguousarray(start_pos, dtype=np.int64)
    rb = np.ascontiguousarray(row_base, dtype=np.int64)
    invf = np.ascontiguousarray(inv_freq, dtype=np.float32)
    nw = None if norm_w is None else np.ascontiguousarray(norm_w, dtype=np.float32)
    assert kv_state.dtype == np.float64 and score_state.dtype == np.float64
    assert plane.dtype == np.uint16
    pf = np.zeros(plane.shape, dtype=np.float64)
    n = lib().orc_compress(_p(kv), _p(score), _p(cu), len(cu) - 1, _p(sp), ratio, _p(kv_state),
                           _p(score_state), _p(plane), _p(pf), _p(rb), _p(nw), eps, _p(invf))
    return n, pf


def compress_index(kv, score, cu_seqlens, start_pos, ratio, kv_state, score_state, plane,
                   index_plane, row_base, inv_freq, wk, knorm_w=None, norm_w=None, eps=1e-6):
    """compress() plus the index K of every emitted row (index_plane uint16 [rows,128], in
    place).  Returns (rows emitted, plane_f64 [rows,512], index_f64 [rows,128])."""
    kv = bf16_bits(kv) if isinstance(kv, torch.Tensor) else kv
    score = None if score is None else (bf16_bits(score) if isinstance(score, torch.Tensor)
                                        else score)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    sp = np.ascontiguousarray(start_pos, dtype=np.int64)
    rb = np.ascontiguousarray(row_base, dtype=np.int64)
    invf = np.ascontiguousarray(inv_freq, dtype=np.float32)
    nw = None if norm_w is None else np.ascontiguousarray(norm_w, dtype=np.float32)
    kw = None if knorm_w is None else np.ascontiguousarray(knorm_w, dtype=np.float32)
    wkb = bf16_bits(wk) if isinstance(wk, torch.Tensor) else np.ascontiguousarray(wk, np.uint16)
    assert wkb.shape == (128, 512)
    assert index_plane.dtype == np.uint16 and index_plane.shape[1] == 128
    pf = np.zeros(plane.shape, dtype=np.float64)
    kf = np.zeros(index_plane.shape, dtype=np.float64)
    n = lib().orc_compress_index(_p(kv), _p(score), _p(cu), len(cu) - 1, _p(sp), ratio,
                                 _p(kv_state), _p(score_state), _p(plane), _p(pf), _p(rb),
                                 _p(nw), eps, _p(invf), _p(wkb), _p(kw), _p(index_plane), _p(kf))
    return n, pf, kf


def index_scores(iq, w, index_k, row_base, q_seq, q_pos, ratio, cand=None, relu=True, ld=None):
    """Returns (scores [Q,ld] float64, rows [Q,ld] int64; -1 = not scored)."""
    iqb = bf16_bits(iq)
    Q, H = iqb.shape[0], iqb.shape[1]
    wf = np.ascontiguousarray(w.detach().cpu().numpy() if isinstance(w, torch.Tensor) else w,
                              dtype=np.float32)
    kb = bf16_bits(index_k)
    rb = np.ascontiguousarray(row_base, dtype=np.int64)
    qs = np.ascontiguousarray(q_seq, dtype=np.int32)
    qp = np.ascontiguousarray(q_pos, dtype=np.int64)
    cd = None if cand is None else np.ascontiguousarray(cand, dtype=np.int32)
    ncb = 0 if cand is None else cd.shape[1]
    if ld is None:
        ld = ncb * 8 if cand is not None else int(max(n_visible(p, ratio) for p in qp))
    ld = max(int(ld), 1)
    sc = np.zeros((Q, ld), dtype=np.float64)
    rows = np.zeros((Q, ld), dtype=np.int64)
    lib().orc_index_scores(_p(iqb), _p(wf), Q, H, _p(kb), _p(rb), _p(qs), _p(qp), ratio, _p(cd),
                           ncb, 1 if relu else 0, _p(sc), _p(rows), ld)
    return sc, rows


def e2m1_value(code):
    return float(lib().orc_e2m1_val(int(code)))


def e2m1_code(x):
    """E2M1 code of a double: nearest, ties to the even code, saturating at 6."""
    return int(lib().orc_e2m1_code(float(x)))


FP4_ROW_BYTES = 288  # 256 bytes of codes (two per byte, low nibble first), 32 E4M3 scales


def plane_fp4(rows):
    """bf16 [n, 512] plane rows -> FP4 rows [n, 288] uint8."""
    rb = bf16_bits(rows)
    out = np.zeros((rb.shape[0], FP4_ROW_BYTES), dtype=np.uint8)
    lib().orc_plane_fp4(_p(rb), rb.shape[0], _p(out))
    return out


def e4m3_code(x):
    """E4M3 code of a double: nearest, ties to even, saturating at 448."""
    return int(lib().orc_e4m3_code(float(x)))


def ue8m0_scale(amax):
    """Smallest power of two s with amax / s <= 448 (1 for amax == 0)."""
    return float(lib().orc_ue8m0_scale(float(amax)))


FP8_BLOCK_BYTES = 1056  # 8 rows x (128 E4M3 codes) then 8 fp32 scales


def index_plane_fp8(index_k):
    """bf16 [n, 128] index rows -> FP8 plane bytes [ceil(n / 8) * 1056] (uint8)."""
    kb = bf16_bits(index_k)
    n = kb.shape[0]
    out = np.zeros(((n + 7) // 8) * FP8_BLOCK_BYTES, dtype=np.uint8)
    lib().orc_index_plane_fp8(_p(kb), n, _p(out))
    return out


def index_scores_fp8(iq, w, plane, row_base, q_seq, q_pos, ratio, cand=None, relu=True, ld=None):
    """index_scores on an FP8 plane (row_base multiples of 8); the query is quantised
    per (token, head) inside, as the FP8 indexer does."""
    iqb = bf16_bits(iq)
    Q, H = iqb.shape[0], iqb.shape[1]
    wf = np.ascontiguousarray(w.detach().cpu().numpy() if isinstance(w, torch.Tensor) else w,
                              dtype=np.float32)
    pl = np.ascontiguousarray(plane, dtype=np.uint8)
    rb = np.ascontiguousarray(row_base, dtype=np.int64)
    assert np.all(rb % 8 == 0)
    qs = np.ascontiguousarray(q_seq, dtype=np.int32)
    qp = np.ascontiguousarray(q_pos, dtype=np.int64)
    cd = None if cand is None else np.ascontiguousarray(cand, dtype=np.int32)
    ncb = 0 if cand is None else cd.shape[1]
    if ld is None:
        ld = ncb * 8 if cand is not None else int(max(n_visible(p, ratio) for p in qp))
    ld = max(int(ld), 1)
    sc = np.zeros((Q, ld), dtype=np.float64)
    rows = np.zeros((Q, ld), dtype=np.int64)
    lib().orc_index_scores_fp8(_p(iqb), _p(wf), Q, H, _p(pl), _p(rb), _p(qs), _p(qp), ratio,
                               _p(cd), ncb, 1 if relu else 0, _p(sc), _p(rows), ld)
    return sc, rows


FP4_INDEX_BLOCK_BYTES = 544  # 8 rows x 64 code bytes, then 8 x 4 E8M0 scales


def index_plane_fp4(index_k):
    """bf16 [n, 128] index rows -> MXFP4 plane bytes [ceil(n / 8) * 544] (uint8)."""
    kb = bf16_bits(index_k)
    n = kb.shape[0]
    out = np.zeros(((n + 7) // 8) * FP4_INDEX_BLOCK_BYTES, dtype=np.uint8)
    lib().orc_index_plane_fp4(_p(kb), n, _p(out))
    return out


def index_scores_fp4(iq, w, plane, row_base, q_seq, q_pos, ratio, cand=None, relu=True, ld=None):
    """index_scores on an MXFP4 plane (row_base multiples of 8), bf16 queries."""
    iqb = bf16_bits(iq)
    Q, H = iqb.shape[0], iqb.shape[1]
    wf = np.ascontiguousarray(w.detach().cpu().numpy() if isinstance(w, torch.Tensor) else w,
                              dtype=np.float32)
    pl = np.ascontiguousarray(plane, dtype=np.uint8)
    rb = np.ascontiguousarray(row_base, dtype=np.int64)
    assert np.all(rb % 8 == 0)
    qs = np.ascontiguousarray(q_seq, dtype=np.int32)
    qp = np.ascontiguousarray(q_pos, dtype=np.int64)
    cd = None if cand is None else np.ascontiguousarray(cand, dtype=np.int32)
    ncb = 0 if cand is None else cd.shape[1]
    if ld is None:
        ld = ncb * 8 if cand is not None else int(max(n_visible(p, ratio) for p in qp))
    ld = max(int(ld), 1)
    sc = np.zeros((Q, ld), dtype=np.float64)
    rows = np.zeros((Q, ld), dtype=np.int64)
    lib().orc_index_scores_fp4(_p(iqb), _p(wf), Q, H, _p(pl), _p(rb), _p(qs), _p(qp), ratio,
                               _p(cd), ncb, 1 if relu else 0, _p(sc), _p(rows), ld)
    return sc, rows


def topk(scores, rows, k):
    """scores/rows: [n] (or [Q,n]); returns int32 sel [k] (or [Q,k])."""
    scores = np.asarray(scores, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    if scores.ndim == 2:
        return np.stack([topk(scores[i], rows[i], k) for i in range(scores.shape[0])])
    s = np.ascontiguousarray(scores)
    r = np.ascontiguousarray(rows)
    out = np.zeros(k, dtype=np.int32)
    lib().orc_topk(_p(s), _p(r), len(s), k, _p(out))
    return out


def sparse_attn(q, q_seq, q_pos, swa, plane, row_base, sel, sink, scale=512 ** -0.5,
                swa_mode="ring", lin_base=None, lin_pos0=None, inv_freq=None, swa_e8m0=False):
    """q [Q,64,512] bf16, swa ring [B,128,512] bf16 / [B,128,528] uint8 or linear rows,
    plane [rows,512] bf16, sel [Q,nsel] int32.  Returns (out [Q,64,512], lse [Q,64])
    in float64."""
    qb = bf16_bits(q)
    Q = qb.shape[0]
    if swa.dtype == torch.uint8:
        swa_arr, dt = np.ascontiguousarray(swa.cpu().numpy()), 2 if swa_e8m0 else 1
    else:
        swa_arr, dt = bf16_bits(swa), 0
    if isinstance(plane, np.ndarray) and plane.dtype == np.uint8:
        pb, pdt = np.ascontiguousarray(plane), 1  # FP4 rows of 288 bytes
    elif isinstance(plane, torch.Tensor) and plane.dtype == torch.uint8:
        pb, pdt = np.ascontiguousarray(plane.cpu().numpy()), 1
    else:
        pb, pdt = bf16_bits(plane), 0
    sl = np.ascontiguousarray(sel, dtype=np.int32)
    if sl.ndim == 1:
        sl = sl.reshape(Q, -1)
    nsel = sl.shape[1] if sl.size else 0
    sk = None if sink is None else np.ascontiguousarray(
        sink.cpu().numpy() if isinstance(sink, torch.Tensor) else sink, dtype=np.float32)
    qs = np.ascontiguousarray(q_seq, dtype=np.int32)
    qp = np.ascontiguousarray(q_pos, dtype=np.int64)
    rb = np.ascontiguousarray(row_base, dtype=np.int64)
    mode = 0 if swa_mode == "ring" else 1
    lb = None if lin_base is None else np.ascontiguousarray(lin_base, dtype=np.int64)
    lp = None if lin_pos0 is None else np.ascontiguousarray(lin_pos0, dtype=np.int64)
    out = np.zeros((Q, 64, 512), dtype=np.float64)
    lse = np.zeros((Q, 64), dtype=np.float64)
    lib().orc_sparse_attn(_p(qb), Q, _p(qs), _p(qp), mode, dt, _p(swa_arr), _p(lb), _p(lp),
                          pdt, _p(pb), _p(rb), _p(sl), nsel, _p(sk), scale, _p(out), _p(lse))
    if inv_freq is not None:
        inverse_rope(out, qp, inv_freq)
    return out, lse


def inverse_rope(out, q_pos, inv_freq):
    """Rotate dims 448..511 of out [Q,64,512] (float64, in place) back by each query's
    position: pair i times e^{-i p inv_freq[i]}."""
    assert out.dtype == np.float64 and out.flags["C_CONTIGUOUS"]
    qp = np.ascontiguousarray(q_pos, dtype=np.int64)
    f = np.ascontiguousarray(inv_freq, dtype=np.float32)
    lib().orc_inverse_rope(_p(out), out.shape[0], _p(qp), _p(f))
    return out


def candidate_pool(scores, rows, nbk=2048):
    """One query's FULL logits (float64 [ld]) and row ids ([ld], -1 = not scored) ->
    candidate block ids [nbk] int32: block maxima, newest block pinned, top nbk blocks,
    ascending, -1 padded."""
    sc = np.ascontiguousarray(scores, dtype=np.float64)
    rw = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty(nbk, dtype=np.int32)
    lib().orc_candidate_pool(_p(sc), _p(rw), len(sc), nbk, _p(out))
    return out
