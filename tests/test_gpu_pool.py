"""The candidate pool of a FULL layer (block maxima, newest block pinned, top-nbk blocks)
through the C ABI, and a REINDEX call that takes the pool straight from the device.

Three checks:
  * the pool is exactly the top-nbk blocks of the block maxima of the scores the kernel
    itself reports (scores_out), with the newest block pinned and ties to the lower
    block id: a property of the output, recomputed here with numpy;
  * against the oracle (host-regenerated inputs, fp64 scores): equal, except blocks
    whose oracle block maximum lies within the score tie tolerance of the nbk-th one;
  * the REINDEX call that consumes the device pool equals the oracle's REINDEX on the
    oracle's own pool (queries whose two pools agree).
The selection of k = 2048 itself is also checked bit-exactly on given scores.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import workloads as W

from _harness import (TIE_RTOL, check_scores, check_sel, host_seq, oracle_index, query_inputs,
                      register, spec_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _pool_workload(ctx, ratio, nq=1, seed=61):
    B = len(ctx)
    return W.Workload("pool_decode", seed, ratio, ctx=ctx, chunk=[nq] * B, nq=[nq] * B,
                      description="FULL decode with the candidate pool")


def _run_pool(t, spec, nbk):
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_index_topk,
                                              csa2_index_topk_pool,
                                              csa2_index_topk_pool_workspace_size,
                                              csa2_index_topk_workspace_size)
    Q = t["iq"].shape[0]
    ws = torch.empty(csa2_index_topk_pool_workspace_size(Q, spec.H, spec.max_scored, spec.k, nbk),
                     dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)  # the call must not depend on the workspace's contents
    sel = torch.empty((Q, spec.k), dtype=torch.int32, device="cuda")
    pool = torch.full((Q, nbk), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((Q, spec.max_scored), float("nan"), device="cuda")
    csa2_index_topk_pool(t["iq"], t["w"], t["index_k"], t["row_base"], t["q_seq"], t["q_pos"],
                         spec.ratio, spec.k, spec.max_scored, sel, pool, ws, scores_out=sc)
    csa2_device_status()
    # the same FULL call without the pool selects the same rows
    ws2 = torch.empty(csa2_index_topk_workspace_size(Q, spec.H, spec.max_scored, spec.k),
                      dtype=torch.uint8, device="cuda")
    sel2 = torch.empty_like(sel)
    csa2_index_topk(t["iq"], t["w"], t["index_k"], t["row_base"], t["q_seq"], t["q_pos"],
                    spec.ratio, spec.k, spec.max_scored, sel2, ws2)
    csa2_device_status()
    assert torch.equal(sel, sel2)
    return sel, pool, sc


def _expected_from_scores(scores, nvis, nbk):
    """Top-nbk blocks of the block maxima of `scores[0:nvis]` (newest block pinned)."""
    nb = (nvis + 7) // 8
    if nb == 0:
        return np.full(nbk, -1, dtype=np.int32)
    s = np.full(nb * 8, -np.inf)
    s[:nvis] = scores[:nvis]
    bm = s.reshape(nb, 8).max(axis=1)
    bm[nb - 1] = np.inf
    order = np.lexsort((np.arange(nb), -bm))[:min(nbk, nb)]
    out = np.full(nbk, -1, dtype=np.int32)
    out[:len(order)] = np.sort(order)
    return out


def check_pool(pool_gpu, pool_ref, sc, rows, nbk):
    """Equal up to near ties of the nbk-th oracle block maximum; ascending, -1 padded."""
    ng, nr = int((pool_gpu >= 0).sum()), int((pool_ref >= 0).sum())
    assert ng == nr, f"blocks selected: gpu {ng}, oracle {nr}"
    assert np.all(pool_gpu[ng:] == -1) and np.all(np.diff(pool_gpu[:ng]) > 0)
    if np.array_equal(pool_gpu, pool_ref):
        return 0
    valid = rows >= 0
    nb = (int(rows[valid].max()) + 8) // 8
    bm = np.full(nb, -np.inf)
    np.maximum.at(bm, rows[valid] // 8, sc[valid])
    newest = nb - 1
    assert newest in set(pool_gpu[:ng].tolist()), "newest block missing"
    kth = min(bm[b] for b in pool_ref[:nr] if b != newest)
    diff = set(pool_gpu[:ng].tolist()) ^ set(pool_ref[:nr].tolist())
    for b in diff:
        assert abs(bm[b] - kth) <= TIE_RTOL * abs(kth) + 1e-12, (
            f"block {b} differs with maximum {bm[b]} vs nbk-th {kth}")
    return len(diff)


@pytest.mark.parametrize("k", [2048, 512])
def test_topk_scores_large_k_bit_exact(k):
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_topk_scores,
                                              csa2_topk_workspace_size)
    for ld in (1500, 2048, 5000, 32768, 100000):
        g = np.random.default_rng(ld)
        Q = 5
        s = g.standard_normal((Q, ld)).astype(np.float32)
        s[1] = (g.integers(-30, 30, ld) / 4.0).astype(np.float32)  # heavy ties
        s[2, ::3] = np.nan
        # all keys within one quarter octave: the sampled threshold bin is refined
        s[4] = (1.0 + 1e-3 * g.standard_normal(ld)).astype(np.float32)
        n = np.array([ld, ld, ld - 1, ld // 3, ld], dtype=np.int32)
        sel = torch.empty((Q, k), dtype=torch.int32, device="cuda")
        ws = torch.empty(max(csa2_topk_workspace_size(Q, ld, k), 256), dtype=torch.uint8,
                         device="cuda")
        csa2_topk_scores(torch.from_numpy(s).cuda(), torch.from_numpy(n).cuda(), k, sel, ws=ws)
        csa2_device_status()
        sel = sel.cpu().numpy()
        for q in range(Q):
            ref = oracle.topk(s[q, :n[q]].astype(np.float64), np.arange(n[q]), k)
            assert np.array_equal(sel[q], ref), f"ld {ld} row {q}"


@pytest.mark.parametrize("ratio,ctx,nq", [
    (1, [5, 300, 2057, 16391, 16384, 40003], 1),   # fewer blocks than nbk, ragged newest block
    (2, [90000, 33333, 70001], 3),                 # groups of 3 queries, m = 2
    (1, [300001, 262151], 1),                      # > 32768 blocks: chunked block selection
])
def test_pool_matches_its_own_scores_and_the_oracle(ratio, ctx, nq):
    nbk = 2048
    wl = _pool_workload(ctx, ratio, nq=nq)
    key = register(wl)
    t = wl.materialize("cuda")
    spec = spec_of(wl)
    sel, pool, sc = _run_pool(t, spec, nbk)
    pool = pool.cpu().numpy()
    sc = sc.cpu().numpy()
    ndiff = []
    for q in range(wl.Q):
        nvis = int((wl.q_pos[q] + 1) // ratio)
        exp = _expected_from_scores(sc[q].astype(np.float64), nvis, nbk)
        assert np.array_equal(pool[q], exp), f"query {q}: pool is not the top blocks of its scores"
    for q in sorted({0, wl.Q - 1}):
        osc, rows, _ = oracle_index(wl, key, q)
        ref = oracle.candidate_pool(osc, rows, nbk)
        ndiff.append(check_pool(pool[q], ref, osc, rows, nbk))
    print(f"\npool {ctx}: blocks differing at near ties {ndiff}")


def test_reindex_takes_the_pool_from_the_device():
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_index_topk,
                                              csa2_index_topk_workspace_size)
    nbk = 2048
    wl = _pool_workload([40003, 77777, 24001], 1, seed=62)
    key = register(wl)
    t = wl.materialize("cuda")
    spec = spec_of(wl)
    _, pool_d, _ = _run_pool(t, spec, nbk)
    Q, ms = wl.Q, nbk * 8
    ws = torch.empty(csa2_index_topk_workspace_size(Q, spec.H, ms, spec.k), dtype=torch.uint8,
                     device="cuda")
    sel = torch.empty((Q, spec.k), dtype=torch.int32, device="cuda")
    sc = torch.full((Q, ms), float("nan"), device="cuda")
    csa2_index_topk(t["iq"], t["w"], t["index_k"], t["row_base"], t["q_seq"], t["q_pos"],
                    wl.ratio, spec.k, ms, sel, ws, cand=pool_d, scores_out=sc)
    csa2_device_status()
    pool = pool_d.cpu().numpy()
    sel = sel.cpu().numpy()
    sc = sc.cpu().numpy()
    checked = 0
    for q in range(Q):
        osc, rows, _ = oracle_index(wl, key, q)
        ref_pool = oracle.candidate_pool(osc, rows, nbk)
        check_pool(pool[q], ref_pool, osc, rows, nbk)
        if not np.array_equal(pool[q], ref_pool):
            continue
        iq, w = query_inputs(wl, q)
        hs = host_seq(key, int(wl.q_seq[q]))
        rsc, rrows = oracle.index_scores(iq, w, hs.index_k(), [0], [0], [int(wl.q_pos[q])],
                                         wl.ratio, cand=ref_pool[None, :])
        ref_sel = oracle.topk(rsc[0], rrows[0], spec.k)
        check_scores(sc[q, :len(rrows[0])], rsc[0], rrows[0])
        check_sel(sel[q], ref_sel, rsc[0], rrows[0], spec.k)
        checked += 1
    assert checked >= 2
