"""Seeded synthetic workloads with the shapes of the five CSA2 configurations.

A workload is host metadata (sequence lengths, positions, layout offsets and the
candidate pool) plus a recipe that fills every tensor from the generator in
``synth``.  ``materialize(device)`` builds all tensors on one device; the oracle
harness instead regenerates, on the host, only the rows it needs for a query.

Recipe (all values ~N(0,1) unless noted):
  * kv, score: the step's new tokens, one 512-wide row per absolute position.
  * kv_state/score_state: fp32 copies of the tokens of an incomplete group that
    precede the step (the per-request compressor tail).
  * plane: rows of complete groups that precede the step are synthetic; the rows
    the step completes are left zero for the compressor to write.
  * index_k: every visible row is synthetic (index-K production is not part of
    the step).
  * q, iq, ring / linear SWA rows: synthetic, taken as already rotated (a RoPE
    rotation of an isotropic Gaussian pair is again isotropic Gaussian).
  * w: indexer head weights; sink: per-head attention sink logits.
  * candidates (REINDEX): 2048 distinct 8-row blocks drawn without replacement
    from the full visible blocks, the newest block always included, ascending.
  * RoPE table: theta = 160000, inv_freq[i] = theta^(-2i/64), i < 32.
"""
from dataclasses import dataclass, field

import numpy as np
import torch

from . import (CAND, INDEX_K, IQ, KV, LAYER_STRIDE, LENGTHS, PLANE, Q, RING, SCORE, SINK,
               SWA_LINEAR, W, normal_f32, rows_bf16, rows_f32, rows_fp8s128, u64)

D_LATENT = 512
D_INDEX = 128
N_HEADS = 64
RING_SLOTS = 128
ROPE_THETA = 160000.0


def rope_inv_freq(theta=ROPE_THETA):
    return (theta ** (-np.arange(0, 64, 2, dtype=np.float64) / 64.0)).astype(np.float32)


@dataclass
class Workload:
    name: str
    seed: int
    ratio: int
    ctx: np.ndarray            # [B] tokens processed after the step
    chunk: np.ndarray          # [B] new tokens in the step
    nq: np.ndarray             # [B] queries per sequence (the last nq positions)
    H: int = 64
    k: int = 512
    swa: str = "ring"          # "ring" | "linear"
    swa_dtype: str = "bf16"    # "bf16" | "fp8"
    reindex: bool = False
    ncb: int = 2048
    layers: int = 1
    description: str = ""
    extra: dict = field(default_factory=dict)

    def __post_init__(self):
        self.ctx = np.asarray(self.ctx, dtype=np.int64)
        self.chunk = np.asarray(self.chunk, dtype=np.int64)
        self.nq = np.asarray(self.nq, dtype=np.int64)
        self.B = len(self.ctx)
        m = self.ratio
        self.start_pos = self.ctx - self.chunk
        self.cu_seqlens = np.concatenate([[0], np.cumsum(self.chunk)]).astype(np.int32)
        self.T = int(self.cu_seqlens[-1])
        self.n_rows = self.ctx // m                 # plane / index rows after the step
        self.n_hist = self.start_pos // m           # rows that precede the step
        self.row_base = np.concatenate([[0], np.cumsum(self.n_rows)[:-1]]).astype(np.int64)
        self.total_rows = int(self.n_rows.sum())
        qs, qp, qj = [], [], []
        for b in range(self.B):
            for j in range(int(self.nq[b])):
                qs.append(b)
                qp.append(int(self.ctx[b] - self.nq[b] + j))
                qj.append(j)
        self.q_seq = np.asarray(qs, dtype=np.int32)
        self.q_pos = np.asarray(qp, dtype=np.int64)
        self.q_local = np.asarray(qj, dtype=np.int64)
        self.Q = len(qs)
        if self.swa == "linear":
            # One row per position from RING_SLOTS positions before the chunk to the end.
            self.lin_pos0 = np.maximum(self.start_pos - RING_SLOTS, 0)
            self.lin_len = self.ctx - self.lin_pos0
            self.lin_base = np.concatenate([[0], np.cumsum(self.lin_len)[:-1]]).astype(np.int64)
        self.cand = self._candidates() if self.reindex else None
        self.inv_freq = rope_inv_freq()

    # ---- candidate pool (REINDEX) -------------------------------------------------
    def _candidates(self):
        out = np.full((self.Q, self.ncb), -1, dtype=np.int32)
        for q in range(self.Q):
            nvis = int((self.q_pos[q] + 1) // self.ratio)
            nb = nvis // 8
            take = min(self.ncb, nb)
            if take <= 0:
                continue
            keys = u64(nb - 1, self.seed, CAND, offset=q << 32)
            order = np.argsort(keys, kind="stable")[: take - 1]
            blocks = np.sort(np.concatenate([order, [nb - 1]]))
            out[q, :take] = blocks
        return out

    # ---- pending compressor tail before the step ----------------------------------
    def pending(self, b):
        """Positions of the incomplete group that precedes the step in sequence b."""
        m = self.ratio
        s = int(self.start_pos[b])
        g0 = (s // m) * m
        return list(range(g0, s))

    # ---- tensors -----------------------------------------------------------------
    def materialize(self, device):
        dev = torch.device(device)
        s = self.seed
        t = {}
        kv = torch.empty((self.T, D_LATENT), dtype=torch.bfloat16, device=dev)
        sc = torch.empty((self.T, D_LATENT), dtype=torch.bfloat16, device=dev)
        for b in range(self.B):
            a, e = int(self.cu_seqlens[b]), int(self.cu_seqlens[b + 1])
            rows_bf16(b, int(self.start_pos[b]), e - a, D_LATENT, s, KV, out=kv[a:e])
            rows_bf16(b, int(self.start_pos[b]), e - a, D_LATENT, s, SCORE, out=sc[a:e])
        t["kv"], t["score"] = kv, sc
        ks = torch.zeros((self.B, 2, D_LATENT), dtype=torch.float32)
        ss = torch.zeros((self.B, 2, D_LATENT), dtype=torch.float32)
        for b in range(self.B):
            for p in self.pending(b):
                slot = p % self.ratio
                ks[b, slot] = rows_f32(b, p, 1, D_LATENT, s, KV)[0].bfloat16().float()
                ss[b, slot] = rows_f32(b, p, 1, D_LATENT, s, SCORE)[0].bfloat16().float()
        t["kv_state"], t["score_state"] = ks.to(dev), ss.to(dev)
        t["cu_seqlens"] = torch.from_numpy(self.cu_seqlens).to(dev)
        t["start_pos"] = torch.from_numpy(self.start_pos).to(dev)
        t["row_base"] = torch.from_numpy(self.row_base).to(dev)
        plane = torch.zeros((max(self.total_rows, 1), D_LATENT), dtype=torch.bfloat16, device=dev)
        ik = torch.empty((max(self.total_rows, 1), D_INDEX), dtype=torch.bfloat16, device=dev)
        for b in range(self.B):
            r0, nh, nr = int(self.row_base[b]), int(self.n_hist[b]), int(self.n_rows[b])
            rows_bf16(b, 0, nh, D_LATENT, s, PLANE, out=plane[r0:r0 + nh])
            rows_bf16(b, 0, nr, D_INDEX, s, INDEX_K, out=ik[r0:r0 + nr])
        t["plane"], t["index_k"] = plane, ik
        iq = torch.empty((self.Q, self.H, D_INDEX), dtype=torch.bfloat16, device=dev)
        w = torch.empty((self.Q, self.H), dtype=torch.float32, device=dev)
        for q in range(self.Q):
            b, j = int(self.q_seq[q]), int(self.q_local[q])
            rows_bf16(b, j, 1, self.H * D_INDEX, s, IQ, out=iq[q].view(1, -1))
        # w is small: generate on the host and copy.
        wh = torch.empty((self.Q, self.H), dtype=torch.float32)
        for q in range(self.Q):
            b, j = int(self.q_seq[q]), int(self.q_local[q])
            wh[q] = rows_f32(b, j, 1, self.H, s, W)[0]
        w.copy_(wh)
        t["iq"], t["w"] = iq, w
        t["q_seq"] = torch.from_numpy(self.q_seq).to(dev)
        t["q_pos"] = torch.from_numpy(self.q_pos).to(dev)
        qs = []
        for layer in range(self.layers):
            ql = torch.empty((self.Q, N_HEADS, D_LATENT), dtype=torch.bfloat16, device=dev)
            self._fill_q(ql, layer)
            qs.append(ql)
        t["q"] = qs
        swa = []
        for layer in range(self.layers):
            swa.append(self._make_swa(layer, dev))
        t["swa"] = swa
        if self.swa == "linear":
            t["lin_base"] = torch.from_numpy(self.lin_base).to(dev)
            t["lin_pos0"] = torch.from_numpy(self.lin_pos0).to(dev)
        t["sink"] = normal_f32(N_HEADS, s, SINK).to(dev)
        t["inv_freq"] = torch.from_numpy(self.inv_freq).to(dev)
        if self.reindex:
            t["cand"] = torch.from_numpy(self.cand).to(dev)
        return t

    def _fill_q(self, out, layer):
        st = Q + LAYER_STRIDE * layer
        for b in range(self.B):
            q0 = int(np.searchsorted(self.q_seq, b))
            n = int(self.nq[b])
            if n:
                rows_bf16(b, 0, n, N_HEADS * D_LATENT, self.seed, st,
                          out=out[q0:q0 + n].view(n, -1))

    def _make_swa(self, layer, dev):
        if self.swa == "ring":
            st = RING + LAYER_STRIDE * layer
            if self.swa_dtype == "fp8":
                r = torch.empty((self.B, RING_SLOTS, 528), dtype=torch.uint8, device=dev)
                for b in range(self.B):
                    rows_fp8s128(b, 0, RING_SLOTS, self.seed, st, out=r[b])
            else:
                r = torch.empty((self.B, RING_SLOTS, D_LATENT), dtype=torch.bfloat16, device=dev)
                for b in range(self.B):
                    rows_bf16(b, 0, RING_SLOTS, D_LATENT, self.seed, st, out=r[b])
            return r
        st = SWA_LINEAR + LAYER_STRIDE * layer
        total = int(self.lin_len.sum())
        r = torch.empty((total, D_LATENT), dtype=torch.bfloat16, device=dev)
        for b in range(self.B):
            a, n = int(self.lin_base[b]), int(self.lin_len[b])
            rows_bf16(b, 0, n, D_LATENT, self.seed, st, out=r[a:a + n])
        return r

    def host_q(self, q, layer=0):
        b, j = int(self.q_seq[q]), int(self.q_local[q])
        return rows_bf16(b, j, 1, N_HEADS * D_LATENT, self.seed,
                         Q + LAYER_STRIDE * layer).view(N_HEADS, D_LATENT)


# ---- the five configurations --------------------------------------------------------

def tiny_decode(B=4, S=4096, ratio=2, seed=0):
    """B sequences of S tokens compressed from position 0, one decode query each at S-1."""
    return Workload("tiny_full_decode", seed, ratio, ctx=[S] * B, chunk=[S] * B, nq=[1] * B,
                    description=f"FULL decode, B={B}, S={S}, m={ratio}, compressor over S tokens")


def decode_batch(B=64, lo=16384, hi=65536, ratio=2, seed=1):
    """B decode queries; context lengths uniform in [lo, hi]; one new token each."""
    L = lo + (u64(B, seed, LENGTHS) % np.uint64(hi - lo + 1)).astype(np.int64)
    return Workload("full_decode_batch", seed, ratio, ctx=L, chunk=[1] * B, nq=[1] * B,
                    description=f"FULL decode, B={B}, ctx~U[{lo},{hi}], m={ratio}")


def reindex_decode(B=32, ctx=262144, ncb=2048, seed=2):
    return Workload("reindex_decode", seed, 1, ctx=[ctx] * B, chunk=[1] * B, nq=[1] * B,
                    reindex=True, ncb=ncb,
                    description=f"REINDEX decode, B={B}, ctx={ctx}, m=1, {ncb}x8 candidates")


def prefill_reuse(n_new=4096, ctx=131072, ratio=2, layers=6, seed=3):
    return Workload("prefill_reuse", seed, ratio, ctx=[ctx], chunk=[n_new], nq=[n_new],
                    swa="linear", layers=layers,
                    description=f"prefill chunk of {n_new} at {ctx - n_new}, m={ratio}, "
                                f"top-512 once + {layers} attention layers")


def long_decode(B=8, ctx=1048576, seed=4):
    return Workload("long_decode_fp8ring", seed, 1, ctx=[ctx] * B, chunk=[1] * B, nq=[1] * B,
                    swa_dtype="fp8",
                    description=f"FULL decode, B={B}, ctx={ctx}, m=1, FP8 E4M3 ring")


CONFIGS = {
    "tiny": tiny_decode,
    "decode": decode_batch,
    "reindex": reindex_decode,
    "prefill": prefill_reuse,
    "long": long_decode,
}
