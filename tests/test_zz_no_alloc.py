"""csa2_index_topk_noalloc: the indexer + top-k for callers that cannot allocate device
memory (a plugin interface that only passes inputs and outputs, an engine that owns all
of HBM through its own pool, or a path that cannot pay for cudaMalloc's device-wide
synchronisation).  Its scratch is a fixed device array inside the library, shared by
all calls.  This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.

Checked through the C ABI against csa2_index_topk with a caller workspace, on two calls
in a row (the second call finds the first call's leftovers in the shared array), with
the tolerances the other parity tests use.
"""
import ctypes

import numpy as np
import pytest
import torch

from synth import workloads as W

from _harness import check_scores, spec_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _with_workspace(t, spec, cand):
    from csa2_compressed_sparse_gb300 import csa2_index_topk, csa2_index_topk_workspace_size
    Q = t["iq"].shape[0]
    ws = torch.empty(max(csa2_index_topk_workspace_size(Q, spec.H, spec.max_scored, spec.k), 256),
                     dtype=torch.uint8, device="cuda")
    sel = torch.empty((Q, spec.k), dtype=torch.int32, device="cuda")
    ss = torch.empty((Q, spec.k), dtype=torch.float32, device="cuda")
    sc = torch.full((Q, spec.max_scored), float("nan"), device="cuda")
    csa2_index_topk(t["iq"], t["w"], t["index_k"], t["row_base"], t["q_seq"], t["q_pos"],
                    spec.ratio, spec.k, spec.max_scored, sel, ws, sel_scores=ss, cand=cand,
                    scores_out=sc)
    return sel, ss, sc


def _without_workspace(t, spec, cand):
    from csa2_compressed_sparse_gb300 import csa2_index_topk_noalloc
    Q = t["iq"].shape[0]
    sel = torch.full((Q, spec.k), -7, dtype=torch.int32, device="cuda")
    ss = torch.empty((Q, spec.k), dtype=torch.float32, device="cuda")
    sc = torch.full((Q, spec.max_scored), float("nan"), device="cuda")
    csa2_index_topk_noalloc(t["iq"], t["w"], t["index_k"], t["row_base"], t["q_seq"],
                            t["q_pos"], spec.ratio, spec.k, spec.max_scored, sel,
                            sel_scores=ss, cand=cand, scores_out=sc)
    return sel, ss, sc


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    from csa2_compressed_sparse_gb300 import csa2_device_status
    cases = [W.decode_batch(B=12, lo=300, hi=9000, seed=41),          # FULL, ragged
             W.reindex_decode(B=3, ctx=24576, ncb=256, seed=42)]      # REINDEX
    for wl in cases:
        t = wl.materialize("cuda")
        spec = spec_of(wl)
        cand = t.get("cand")
        ref_sel, ref_ss, ref_sc = _with_workspace(t, spec, cand)
        csa2_device_status()
        got_sel, got_ss, got_sc = _without_workspace(t, spec, cand)
        csa2_device_status()
        assert torch.equal(got_sel, ref_sel), wl.name
        nv = (ref_sel >= 0)
        assert torch.equal(got_ss[nv], ref_ss[nv]), wl.name
        r = ref_sc.cpu().numpy()
        g = got_sc.cpu().numpy()
        for q in range(r.shape[0]):
            rows = np.where(np.isnan(r[q]), -1, 0)
            check_scores(g[q], np.nan_to_num(r[q]).astype(np.float64), rows)


def test_noalloc_refuses_sizes_beyond_its_array():
    from csa2_compressed_sparse_gb300 import Csa2Error, csa2_index_topk_noalloc
    from csa2_compressed_sparse_gb300 import lib
    dummy = torch.zeros(256, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    # 4096 queries x 65536 positions of 4-byte keys is 1 GiB of scratch: refused
    st = lib().csa2_index_topk_noalloc(p, p, 4096, 64, p, 70000, p, p, p, 2, None, 0, 512, 1,
                                       65536, p, None, None, None)
    assert st == 5
    assert b"scratch" in lib().csa2_last_error()
