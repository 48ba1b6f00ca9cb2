"""Oracle-side evaluation of one query of a synthetic workload -- TEST INFRASTRUCTURE.

Regenerates, on the host and from the seeded generator only, the inputs the oracle
needs for one query (the sequence's new tokens through the oracle compressor, the
index plane, the query's iq / w / q, its window rows and the selected plane rows),
so that full-size workloads can be checked on sampled queries without copying any
GPU output into the oracle.
"""
from functools import lru_cache

import numpy as np
import torch

import synth

from . import bf16_bits, bf16_from_bits, compress, index_scores, plane_fp4, sparse_attn, topk

# ---- host regeneration of one sequence's inputs ------------------------------------------

class HostSeq:
    """Oracle-side inputs of sequence b, regenerated on the host."""

    def __init__(self, wl, b):
        self.wl, self.b = wl, b
        s = wl.seed
        m = wl.ratio
        start = int(wl.start_pos[b])
        ctx = int(wl.ctx[b])
        self.n_hist, self.n_rows = int(wl.n_hist[b]), int(wl.n_rows[b])
        # oracle compressor over the step's tokens, starting from the synthetic tail
        kv = synth.rows_bf16(b, start, ctx - start, 512, s, synth.KV)
        sc = synth.rows_bf16(b, start, ctx - start, 512, s, synth.SCORE)
        ks = np.zeros((1, m, 512))
        ss = np.zeros((1, m, 512))
        for pp in wl.pending(b):
            ks[0, pp % m] = synth.rows_f32(b, pp, 1, 512, s, synth.KV)[0].bfloat16().double().numpy()
            ss[0, pp % m] = synth.rows_f32(b, pp, 1, 512, s, synth.SCORE)[0].bfloat16().double().numpy()
        new = self.n_rows - self.n_hist
        plane = np.zeros((max(self.n_rows, 1), 512), dtype=np.uint16)
        n, pf = compress(kv, sc, [0, ctx - start], [start], m, ks, ss, plane, [0],
                                wl.inv_freq)
        assert n == new
        self.new_rows = plane[self.n_hist:self.n_rows].copy()
        self.new_rows_f64 = pf[self.n_hist:self.n_rows].copy()
        self.kv_state, self.score_state = ks, ss

    def plane_rows(self, rows):
        """uint16 [len(rows), 512] plane rows (history from the generator, new rows
        from the oracle's compressor)."""
        rows = np.asarray(rows, dtype=np.int64)
        out = np.zeros((len(rows), 512), dtype=np.uint16)
        hist = rows < self.n_hist
        if hist.any():
            out[hist] = bf16_bits(synth.rowlist_bf16(self.b, rows[hist], 512,
                                                            self.wl.seed, synth.PLANE))
        if (~hist).any():
            out[~hist] = self.new_rows[rows[~hist] - self.n_hist]
        return out

    def index_k(self):
        return synth.rows_bf16(self.b, 0, self.n_rows, 128, self.wl.seed, synth.INDEX_K)


@lru_cache(maxsize=8)
def host_seq(wl_key, b):
    return HostSeq(_WL[wl_key], b)


_WL = {}


def register(wl):
    key = (wl.name, wl.seed, int(wl.B), int(wl.ctx.sum()), int(wl.chunk.sum()))
    _WL[key] = wl
    return key


def query_inputs(wl, q):
    b, j = int(wl.q_seq[q]), int(wl.q_local[q])
    iq = synth.rows_bf16(b, j, 1, wl.H * 128, wl.seed, synth.IQ).view(1, wl.H, 128)
    w = synth.rows_f32(b, j, 1, wl.H, wl.seed, synth.W)
    return iq, w


def oracle_index(wl, key, q, relu=True):
    """Oracle scores/rows/sel for query q."""
    b = int(wl.q_seq[q])
    hs = host_seq(key, b)
    iq, w = query_inputs(wl, q)
    cand = None if wl.cand is None else wl.cand[q:q + 1]
    sc, rows = index_scores(iq, w, hs.index_k(), [0], [0], [int(wl.q_pos[q])], wl.ratio,
                                   cand=cand, relu=relu)
    sel = topk(sc[0], rows[0], wl.k)
    return sc[0], rows[0], sel


def window_rows(wl, q, layer):
    """The query's window entries as a compact SWA source for the oracle."""
    b, p = int(wl.q_seq[q]), int(wl.q_pos[q])
    if wl.swa == "ring":
        st = synth.RING + synth.LAYER_STRIDE * layer
        if wl.swa_dtype == "fp8":
            ring = synth.rows_fp8s128(b, 0, 128, wl.seed, st).view(1, 128, 528)
        else:
            ring = synth.rows_bf16(b, 0, 128, 512, wl.seed, st).view(1, 128, 512)
        return dict(swa=ring, swa_mode="ring", lin_base=None, lin_pos0=None)
    st = synth.SWA_LINEAR + synth.LAYER_STRIDE * layer
    lo = max(0, p - 127)
    r0 = lo - int(wl.lin_pos0[b])
    lin = synth.rows_bf16(b, r0, p - lo + 1, 512, wl.seed, st)
    return dict(swa=lin, swa_mode="linear", lin_base=[0], lin_pos0=[lo])


def oracle_attn(wl, key, q, sel, layer=0, head_scale=None, inv_freq=None, fp4_plane=False):
    """Oracle output and lse of query q over its window and `sel`.  `head_scale`
    (optional, 64 powers of two) multiplies the query of each head, exactly in bf16.
    fp4_plane: the selected rows are read through the FP4 plane format."""
    b = int(wl.q_seq[q])
    hs = host_seq(key, b)
    sel = np.asarray(sel, dtype=np.int32)
    valid = sel >= 0
    plane = hs.plane_rows(sel[valid]) if valid.any() else np.zeros((1, 512), np.uint16)
    sel_c = np.full(len(sel), -1, dtype=np.int32)
    sel_c[valid] = np.arange(int(valid.sum()), dtype=np.int32)
    qh = wl.host_q(q, layer).view(1, 64, 512)
    if head_scale is not None:
        hsc = torch.as_tensor(np.asarray(head_scale, dtype=np.float64)).view(1, 64, 1)
        qh = (qh.double() * hsc).to(torch.bfloat16)  # exact for powers of two
    win = window_rows(wl, q, layer)
    sink = synth.normal_f32(64, wl.seed, synth.SINK)
    plane_in = plane_fp4(bf16_from_bits(plane)) if fp4_plane else bf16_from_bits(plane)
    out, lse = sparse_attn(qh, [0], [int(wl.q_pos[q])], win["swa"],
                                  plane_in, [0], sel_c.reshape(1, -1), sink,
                                  swa_mode=win["swa_mode"], lin_base=win["lin_base"],
                                  lin_pos0=win["lin_pos0"], inv_freq=inv_freq)
    return out[0], lse[0]


