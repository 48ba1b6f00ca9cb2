"""The FP8 index plane through the C ABI: the quantiser is bit-exact against the oracle's,
and the FP8 indexer (queries quantised per (token, head), E4M3 x E4M3 tensor-core dot
products) matches the oracle's FP8 scores within the score tolerance and its selection up
to near ties.  Oracle inputs are regenerated on the host; the oracle builds its own plane.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import workloads as W

from _harness import check_scores, check_sel, host_seq, query_inputs, register, spec_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def fp8_plane_of(wl, t):
    """The workload's index rows re-laid so that every sequence starts on an 8-row block,
    quantised on the device.  Returns (plane, row_base, rows)."""
    from csa2_compressed_sparse_gb300 import csa2_device_status
    from csa2_compressed_sparse_gb300.step import fp8_index_plane
    out = fp8_index_plane(t["index_k"], wl.row_base, wl.n_rows)
    csa2_device_status()
    return out


def run_fp8(wl, t, plane, rb8, rows, cand=None):
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_index_topk_fp8,
                                              csa2_index_topk_fp8_workspace_size)
    spec = spec_of(wl)
    Q = wl.Q
    ws = torch.empty(csa2_index_topk_fp8_workspace_size(Q, spec.H, spec.max_scored, spec.k),
                     dtype=torch.uint8, device="cuda")
    sel = torch.empty((Q, spec.k), dtype=torch.int32, device="cuda")
    ss = torch.empty((Q, spec.k), dtype=torch.float32, device="cuda")
    sc = torch.full((Q, spec.max_scored), float("nan"), device="cuda")
    csa2_index_topk_fp8(t["iq"], t["w"], plane, rows, rb8, t["q_seq"], t["q_pos"], wl.ratio,
                        spec.k, spec.max_scored, sel, ws, sel_scores=ss, cand=cand, scores_out=sc)
    csa2_device_status()
    return sel.cpu().numpy(), ss.cpu().numpy(), sc.cpu().numpy()


def oracle_fp8(wl, key, q, cand_row=None):
    hs = host_seq(key, int(wl.q_seq[q]))
    plane = oracle.index_plane_fp8(hs.index_k())
    iq, w = query_inputs(wl, q)
    cand = None if cand_row is None else cand_row[None, :]
    sc, rows = oracle.index_scores_fp8(iq, w, plane, [0], [0], [int(wl.q_pos[q])], wl.ratio,
                                       cand=cand)
    return sc[0], rows[0], oracle.topk(sc[0], rows[0], wl.k)


def test_plane_quantiser_is_bit_exact():
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_index_plane_fp8,
                                              csa2_index_plane_fp8_bytes)
    g = np.random.default_rng(5)
    n = 1003  # a partial last block
    x = g.standard_normal((n, 128)) * np.exp2(g.integers(-20, 20, (n, 1)))
    x[3] = 0.0                                   # all-zero row: scale 1
    x[4] = 448.0 * 2.0 ** -3                     # exactly at a scale boundary
    x[5, :] = 2.0 ** -130                        # bf16 subnormals
    x[6, ::2] *= 1e-6                            # values flushed to E4M3 subnormals / zero
    x[7] = g.integers(-8, 8, 128) * 0.0625       # ties between E4M3 neighbours
    k = torch.from_numpy(x.astype(np.float32)).bfloat16()
    plane = torch.empty(csa2_index_plane_fp8_bytes(n), dtype=torch.uint8, device="cuda")
    plane.fill_(0xA5)
    csa2_index_plane_fp8(k.cuda(), plane)
    csa2_device_status()
    ref = oracle.index_plane_fp8(k)
    got = plane.cpu().numpy()
    assert got.size == ref.size
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at block {bad[0] // 1056}"


@pytest.mark.parametrize("ratio,ctx,nq", [
    (2, [600, 4097, 9001, 20000], 1),    # FULL decode, ragged tails, m = 2
    (1, [3000, 12345], 4),               # query groups (4 per sequence), m = 1
    (1, [300, 40000, 7], 1),             # short histories (< k rows) and a long one
])
def test_fp8_indexer_matches_the_oracle(ratio, ctx, nq):
    wl = W.Workload("fp8_index", 71, ratio, ctx=ctx, chunk=[nq] * len(ctx), nq=[nq] * len(ctx))
    key = register(wl)
    t = wl.materialize("cuda")
    plane, rb8, rows = fp8_plane_of(wl, t)
    sel, ss, sc = run_fp8(wl, t, plane, rb8, rows)
    diffs = []
    for q in range(wl.Q):
        osc, orows, osel = oracle_fp8(wl, key, q)
        n = len(orows)
        check_scores(sc[q, :n], osc, orows)
        diffs.append(check_sel(sel[q], osel, osc, orows, wl.k))
        nv = int((sel[q] >= 0).sum())
        assert np.array_equal(ss[q, :nv], sc[q, sel[q, :nv]])
    print(f"\nfp8 {ctx}: near-tie differences {diffs}")


def test_fp8_reindex_matches_the_oracle():
    wl = W.reindex_decode(B=3, ctx=24576, ncb=256, seed=72)
    key = register(wl)
    t = wl.materialize("cuda")
    plane, rb8, rows = fp8_plane_of(wl, t)
    sel, _, sc = run_fp8(wl, t, plane, rb8, rows, cand=t["cand"])
    for q in range(wl.Q):
        osc, orows, osel = oracle_fp8(wl, key, q, cand_row=wl.cand[q])
        check_scores(sc[q, :len(orows)], osc, orows)
        check_sel(sel[q], osel, osc, orows, wl.k)


def test_fp8_indexer_full_decode_batch_sampled():
    wl = W.decode_batch()
    key = register(wl)
    t = wl.materialize("cuda")
    plane, rb8, rows = fp8_plane_of(wl, t)
    sel, _, sc = run_fp8(wl, t, plane, rb8, rows)
    for q in (0, 17, 63):
        osc, orows, osel = oracle_fp8(wl, key, q)
        check_scores(sc[q, :len(orows)], osc, orows)
        check_sel(sel[q], osel, osc, orows, wl.k)
