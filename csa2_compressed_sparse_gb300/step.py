"""One CSA2 attention step over resident device tensors, through the C ABI.

A step is: compress the new tokens -> index + top-k (FULL or REINDEX) -> sparse
attention for the scoring layer -> REUSE attention for the following layers of the
index group (same selection, each layer with its own q and window).  By default the
first two parts are one call (csa2_compress_index_topk).
"""
from dataclasses import dataclass, field
from typing import List, Optional

import torch

from . import (Swa, SWA_LINEAR, SWA_RING, csa2_attn_workspace_size, csa2_compress,
               csa2_compress_index_topk, csa2_index_topk, csa2_index_topk_workspace_size,
               csa2_reuse_attn, csa2_sparse_attn)


@dataclass
class StepSpec:
    ratio: int
    H: int = 64
    k: int = 512
    max_scored: int = 0          # FULL: >= max visible rows; REINDEX: ncb * 8
    swa_mode: int = SWA_RING
    scale: float = 512 ** -0.5
    eps: float = 1e-6
    relu: bool = True


@dataclass
class StepBuffers:
    sel: torch.Tensor
    sel_scores: Optional[torch.Tensor]
    out: List[torch.Tensor]
    lse: List[Optional[torch.Tensor]]
    ws: torch.Tensor
    attn_ws: Optional[torch.Tensor] = None
    scores_out: Optional[torch.Tensor] = None
    launches: int = 0


def allocate(spec: StepSpec, t, want_scores=False, want_lse=False) -> StepBuffers:
    dev = t["iq"].device
    Q = t["iq"].shape[0]
    layers = len(t["q"])
    ws_bytes = csa2_index_topk_workspace_size(Q, spec.H, spec.max_scored, spec.k)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    aws_bytes = csa2_attn_workspace_size(Q, spec.k)
    attn_ws = torch.empty(aws_bytes, dtype=torch.uint8, device=dev) if aws_bytes else None
    return StepBuffers(
        sel=torch.empty((Q, spec.k), dtype=torch.int32, device=dev),
        sel_scores=torch.empty((Q, spec.k), dtype=torch.float32, device=dev),
        out=[torch.empty((Q, 64, 512), dtype=torch.bfloat16, device=dev) for _ in range(layers)],
        lse=[torch.empty((Q, 64), dtype=torch.float32, device=dev) if want_lse else None
             for _ in range(layers)],
        ws=ws,
        attn_ws=attn_ws,
        scores_out=(torch.full((Q, spec.max_scored), float("nan"), dtype=torch.float32,
                               device=dev) if want_scores else None),
    )


def swa_of(spec: StepSpec, t, layer):
    if spec.swa_mode == SWA_LINEAR:
        return Swa(t["swa"][layer], SWA_LINEAR, t["lin_base"], t["lin_pos0"])
    return Swa(t["swa"][layer], SWA_RING)


def topk_chunks(ld: int) -> int:
    """Chunk CTAs per row of the top-k (the library's rule: whole rows up to 32768
    positions, else chunks of 32768)."""
    return (ld + 32767) // 32768


def kernel_launches(spec: StepSpec, t, fused=True) -> int:
    """Kernels one step launches: the index prep, the score kernel and the top-k (it
    merges in its last CTA; fused, its launch also runs the compressor's tokens), a
    separate compressor when not fused, and the attention layers."""
    from . import lib  # noqa: F401  (library must be loaded)
    n = 0
    Q = t["iq"].shape[0]
    if t["kv"].shape[0] and (not fused or Q == 0):
        n += 1
    if Q:
        n += 3
        split = csa2_attn_workspace_size(Q, spec.k) > 0
        n += len(t["q"]) * (2 if split else 1)
    return n


def run_step(spec: StepSpec, t, buf: StepBuffers, stream=None, compress=True, side=None,
             fused=True):
    """One step on `stream` (default: the current stream).  With `fused` the compressor
    runs inside the indexer's call (csa2_compress_index_topk: its tokens on extra CTAs of
    the top-k launch), so the step is one chain of kernels on one stream.  Otherwise csa2_compress is a call of its own; it writes only
    the main plane, which the indexer does not read, so with a `side` stream it runs there,
    concurrently with index + top-k, and the attention waits for both."""
    main = stream if stream is not None else torch.cuda.current_stream()
    comp = compress and t["kv"].shape[0] > 0
    if fused and comp:
        csa2_compress_index_topk(t["kv"], t["score"], t["cu_seqlens"], t["start_pos"],
                                 t["kv_state"], t["score_state"], t["plane"], t["inv_freq"],
                                 t["iq"], t["w"], t["index_k"], t["row_base"], t["q_seq"],
                                 t["q_pos"], spec.ratio, spec.k, spec.max_scored, buf.sel, buf.ws,
                                 sel_scores=buf.sel_scores, cand=t.get("cand"), relu=spec.relu,
                                 scores_out=buf.scores_out, eps=spec.eps, stream=main)
    else:
        fork = side is not None and comp
        if fork:
            side.wait_stream(main)
            with torch.cuda.stream(side):
                csa2_compress(t["kv"], t["score"], t["cu_seqlens"], t["start_pos"], spec.ratio,
                              t["kv_state"], t["score_state"], t["plane"], t["row_base"],
                              t["inv_freq"], eps=spec.eps, stream=side)
        elif comp:
            csa2_compress(t["kv"], t["score"], t["cu_seqlens"], t["start_pos"], spec.ratio,
                          t["kv_state"], t["score_state"], t["plane"], t["row_base"],
                          t["inv_freq"], eps=spec.eps, stream=main)
        csa2_index_topk(t["iq"], t["w"], t["index_k"], t["row_base"], t["q_seq"], t["q_pos"],
                        spec.ratio, spec.k, spec.max_scored, buf.sel, buf.ws,
                        sel_scores=buf.sel_scores, cand=t.get("cand"), relu=spec.relu,
                        scores_out=buf.scores_out, stream=main)
        if fork:
            main.wait_stream(side)
    for layer in range(len(t["q"])):
        fn = csa2_sparse_attn if layer == 0 else csa2_reuse_attn
        fn(t["q"][layer], t["q_seq"], t["q_pos"], swa_of(spec, t, layer), t["plane"],
           t["row_base"], buf.sel, t["sink"], buf.out[layer], lse=buf.lse[layer],
           scale=spec.scale, ws=buf.attn_ws, stream=main)


def block_index_plane(index_k, row_base, n_rows, fmt="fp8"):
    """The FP8 ("fp8") or MXFP4 ("fp4") index plane of bf16 index rows held per sequence
    at row_base[b] (host int sequences n_rows / row_base): every sequence is re-laid to
    start on an 8-row block, then quantised on the device.  Returns (plane, block-aligned
    row_base on the device, rows in the plane)."""
    import numpy as np
    import torch
    from . import (csa2_index_plane_fp4, csa2_index_plane_fp4_bytes, csa2_index_plane_fp8,
                   csa2_index_plane_fp8_bytes)
    quant, nbytes = {"fp8": (csa2_index_plane_fp8, csa2_index_plane_fp8_bytes),
                     "fp4": (csa2_index_plane_fp4, csa2_index_plane_fp4_bytes)}[fmt]
    n = np.asarray(n_rows, dtype=np.int64)
    padded = (n + 7) // 8 * 8
    rb8 = np.concatenate([[0], np.cumsum(padded)[:-1]]).astype(np.int64)
    total = max(int(padded.sum()), 8)
    kpad = torch.zeros((total, index_k.shape[1]), dtype=index_k.dtype, device=index_k.device)
    for b in range(len(n)):
        r0 = int(row_base[b])
        kpad[int(rb8[b]):int(rb8[b]) + int(n[b])] = index_k[r0:r0 + int(n[b])]
    plane = torch.empty(nbytes(total), dtype=torch.uint8, device=index_k.device)
    quant(kpad, plane)
    return plane, torch.from_numpy(rb8).to(index_k.device), total


def fp8_index_plane(index_k, row_base, n_rows):
    """block_index_plane in the FP8 format."""
    return block_index_plane(index_k, row_base, n_rows, "fp8")
