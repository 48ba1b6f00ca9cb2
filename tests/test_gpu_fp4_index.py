"""The MXFP4 index plane through the C ABI: the quantiser is bit-exact against the oracle's,
the tile conversion decodes every (code, scale) pair exactly, and the FP4 indexer (bf16
queries against decoded E2M1 x 2^k rows on the tensor cores) matches the oracle's FP4
scores within the score tolerance and its selection up to near ties.  Oracle inputs are
regenerated on the host; the oracle builds its own plane from the bf16 rows.
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


def fp4_plane_of(wl, t):
    """The workload's index rows re-laid so that every sequence starts on an 8-row block,
    quantised on the device.  Returns (plane, row_base, rows)."""
    from csa2_compressed_sparse_gb300 import csa2_device_status
    from csa2_compressed_sparse_gb300.step import block_index_plane
    out = block_index_plane(t["index_k"], wl.row_base, wl.n_rows, "fp4")
    csa2_device_status()
    return out


def run_fp4(iq, w, plane, rows, rb, q_seq, q_pos, ratio, k, max_scored, cand=None, relu=True):
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_index_topk_fp4,
                                              csa2_index_topk_fp4_workspace_size)
    Q, H = iq.shape[0], iq.shape[1]
    ws = torch.empty(csa2_index_topk_fp4_workspace_size(Q, H, max_scored, k),
                     dtype=torch.uint8, device="cuda")
    sel = torch.empty((Q, k), dtype=torch.int32, device="cuda")
    ss = torch.empty((Q, k), dtype=torch.float32, device="cuda")
    sc = torch.full((Q, max_scored), float("nan"), device="cuda")
    csa2_index_topk_fp4(iq, w, plane, rows, rb, q_seq, q_pos, ratio, k, max_scored, sel, ws,
                        sel_scores=ss, cand=cand, relu=relu, scores_out=sc)
    csa2_device_status()
    return sel.cpu().numpy(), ss.cpu().numpy(), sc.cpu().numpy()


def run_wl(wl, t, plane, rb8, rows, cand=None):
    spec = spec_of(wl)
    return run_fp4(t["iq"], t["w"], plane, rows, rb8, t["q_seq"], t["q_pos"], wl.ratio, spec.k,
                   spec.max_scored, cand=cand)


def oracle_fp4(wl, key, q, cand_row=None):
    hs = host_seq(key, int(wl.q_seq[q]))
    plane = oracle.index_plane_fp4(hs.index_k())
    iq, w = query_inputs(wl, q)
    cand = None if cand_row is None else cand_row[None, :]
    sc, rows = oracle.index_scores_fp4(iq, w, plane, [0], [0], [int(wl.q_pos[q])], wl.ratio,
                                       cand=cand)
    return sc[0], rows[0], oracle.topk(sc[0], rows[0], wl.k)


def test_index_plane_quantiser_is_bit_exact():
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_index_plane_fp4,
                                              csa2_index_plane_fp4_bytes)
    g = np.random.default_rng(6)
    n = 1005  # a partial last block
    x = g.standard_normal((n, 128)) * np.exp2(g.integers(-30, 30, (n, 1)))
    x[3] = 0.0                                   # all-zero row: codes 0, scale code 127
    x[4] = 6.0 * 2.0 ** -3                       # amax exactly 6 * 2^k
    x[5, :] = 2.0 ** -130                        # bf16 subnormals: scale code 0
    x[6, ::2] *= 1e-3                            # values rounded to zero codes
    x[7] = g.choice([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0], 128)
    x[7, ::32] = 6.0                             # ties between E2M1 neighbours at scale 1
    x[8] = 1.5 * 2.0 ** 20                       # M = 1.5 exactly
    x[9] = 1.5078125 * 2.0 ** 20                 # M just above 1.5
    x[10] = 2.0 ** 100 * g.standard_normal(128)  # large scales
    k = torch.from_numpy(x.astype(np.float32)).bfloat16()
    plane = torch.empty(csa2_index_plane_fp4_bytes(n), dtype=torch.uint8, device="cuda")
    plane.fill_(0xA5)
    csa2_index_plane_fp4(k.cuda(), plane)
    csa2_device_status()
    ref = oracle.index_plane_fp4(k)
    got = plane.cpu().numpy()
    assert got.size == ref.size == ((n + 7) // 8) * 544
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at byte {bad[0]} (block {bad[0] // 544})"


def _decode_plane():
    """64 rows whose 256 groups take scale codes 0 .. 252 (every value stays finite in
    fp32) and whose dims cycle through all 16 codes."""
    nrow = 64
    plane = np.zeros(nrow // 8 * 544, dtype=np.uint8)
    codes = np.zeros((nrow, 128), dtype=np.uint8)
    for r in range(nrow):
        blk = plane[(r // 8) * 544:(r // 8 + 1) * 544]
        for d in range(128):
            c = (d + 3 * r) % 16
            codes[r, d] = c
            blk[(r % 8) * 64 + d // 2] |= c << (4 * (d & 1))
        for j in range(4):
            blk[512 + (r % 8) * 4 + j] = (4 * r + j) % 253
    return plane, codes


def test_fp4_tile_conversion_is_exact_for_every_code_and_scale():
    # One-hot queries read single plane values: with H = 32, w = (1, 0, ...) and no ReLU,
    # the score of row r for the query hot at dim d is alpha * 2^s * K[r][d] -- one exact
    # product on the tensor cores, then the scaling by alpha (about 1/64, rounded on each
    # side), so wherever the value is a normal float the GPU's equals the oracle's to a few
    # fp32 ulps, while a wrong code or scale would be off by a third or more.  Three query
    # scales 2^s bring every scale code into range.
    plane, codes = _decode_plane()
    nrow = codes.shape[0]
    H, scales = 32, (-100, 0, 100)
    Q = 128 * len(scales)
    iq = torch.zeros((Q, H, 128), dtype=torch.float32)
    for i, s in enumerate(scales):
        for d in range(128):
            iq[i * 128 + d, 0, d] = 2.0 ** s
    iq = iq.bfloat16()
    w = torch.zeros((Q, H), dtype=torch.float32)
    w[:, 0] = 1.0
    q_seq = np.zeros(Q, dtype=np.int32)
    q_pos = np.full(Q, nrow - 1, dtype=np.int64)
    _, _, sc = run_fp4(iq.cuda(), w.cuda(), torch.from_numpy(plane).cuda(), nrow,
                       torch.zeros(1, dtype=torch.int64, device="cuda"),
                       torch.from_numpy(q_seq).cuda(), torch.from_numpy(q_pos).cuda(), 1, 8,
                       nrow, relu=False)
    ref, rows = oracle.index_scores_fp4(iq, w, plane, [0], q_seq, q_pos, 1, relu=False, ld=nrow)
    assert np.all(rows == np.arange(nrow)[None, :])
    # keys below 2^-126 are bf16 subnormals: whether the tensor cores keep them is not
    # asserted (reported only)
    kval = np.array([[oracle.e2m1_value(codes[r, d]) *
                      2.0 ** (int(plane[(r // 8) * 544 + 512 + (r % 8) * 4 + d // 32]) - 127)
                      for d in range(128)] for r in range(nrow)])
    sub = np.tile(((np.abs(kval) > 0) & (np.abs(kval) < 2.0 ** -126)).T, (len(scales), 1))
    a = np.abs(ref)
    inrange = (a >= 2.0 ** -110) & (a <= 2.0 ** 110)
    check = inrange & ~sub
    def close(g, r):
        return np.abs(g.astype(np.float64) - r) <= 2.0 ** -20 * np.abs(r)
    assert np.all(close(sc[check], ref[check]))
    ks = inrange & sub
    print(f"\nsubnormal keys kept: {int(close(sc[ks], ref[ks]).sum())} of {int(ks.sum())}")
    zero = (codes & 7) == 0  # [row][dim]
    for i in range(len(scales)):
        assert np.all(sc[i * 128:(i + 1) * 128].T[zero] == 0.0)
    seen = np.zeros((nrow, 128), dtype=bool)
    for i in range(len(scales)):
        seen |= check[i * 128:(i + 1) * 128].T
    normal = np.abs(kval) >= 2.0 ** -126
    assert np.all(seen | zero | ~normal), "some (code, scale) pairs were never compared"


@pytest.mark.parametrize("ratio,ctx,nq", [
    (2, [600, 4097, 9001, 20000], 1),    # FULL decode, ragged tails, m = 2
    (1, [3000, 12345], 4),               # query groups (4 per sequence), m = 1
    (1, [300, 40000, 7], 1),             # short histories (< k rows) and a long one
])
def test_fp4_indexer_matches_the_oracle(ratio, ctx, nq):
    wl = W.Workload("fp4_index", 73, ratio, ctx=ctx, chunk=[nq] * len(ctx), nq=[nq] * len(ctx))
    key = register(wl)
    t = wl.materialize("cuda")
    plane, rb8, rows = fp4_plane_of(wl, t)
    sel, ss, sc = run_wl(wl, t, plane, rb8, rows)
    diffs = []
    for q in range(wl.Q):
        osc, orows, osel = oracle_fp4(wl, key, q)
        n = len(orows)
        check_scores(sc[q, :n], osc, orows)
        diffs.append(check_sel(sel[q], osel, osc, orows, wl.k))
        nv = int((sel[q] >= 0).sum())
        assert np.array_equal(ss[q, :nv], sc[q, sel[q, :nv]])
    print(f"\nfp4 {ctx}: near-tie differences {diffs}")


def test_fp4_reindex_matches_the_oracle():
    wl = W.reindex_decode(B=3, ctx=24576, ncb=256, seed=74)
    key = register(wl)
    t = wl.materialize("cuda")
    plane, rb8, rows = fp4_plane_of(wl, t)
    sel, _, sc = run_wl(wl, t, plane, rb8, rows, cand=t["cand"])
    for q in range(wl.Q):
        osc, orows, osel = oracle_fp4(wl, key, q, cand_row=wl.cand[q])
        check_scores(sc[q, :len(orows)], osc, orows)
        check_sel(sel[q], osel, osc, orows, wl.k)


def test_fp4_indexer_full_decode_batch_sampled():
    wl = W.decode_batch()
    key = register(wl)
    t = wl.materialize("cuda")
    plane, rb8, rows = fp4_plane_of(wl, t)
    sel, _, sc = run_wl(wl, t, plane, rb8, rows)
    for q in (0, 29, 63):
        osc, orows, osel = oracle_fp4(wl, key, q)
        check_scores(sc[q, :len(orows)], osc, orows)
        check_sel(sel[q], osel, osc, orows, wl.k)
