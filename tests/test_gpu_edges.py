"""Parity with the CPU oracle at the edges of the window and of the visible history.

[A] Fig. 2a: a query at position p sees the window positions max(0, p - 127) .. p, so a
query below 127 has a window of p + 1 < 128 rows and its first window chunk
(positions p - 127 .. p - 64) is partly or wholly empty.  [A] "visible 是每行自己的前缀
长度": a query with n_vis < 512 visible compressed rows selects all of them and pads
with -1; a ratio-2 query at p = 0 has none (k_eff = 0) and attends to its window alone.
These cases run through both ways the attention lays out a query (one CTA, or a
two-CTA cluster that merges in distributed shared memory).  The LINEAR window's lower bound and the
bounded waits' timeout path are checked too.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads as W

from _harness import check_attn, oracle_attn, register, spec_of
from test_gpu_parity import check_queries, run_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import csa2_compressed_sparse_gb300 as csa2
    csa2.lib()


def test_cold_prefill_from_position_zero():
    """300 new tokens compressed from position 0 (ratio 2, LINEAR windows, two layers):
    windows of 1 .. 128 rows, n_vis from 0 to 150; more queries than SMs, so one CTA per
    SM walks its queries (ragged windows and empty selections inside that layout)."""
    wl = W.Workload("cold_prefill", 41, 2, ctx=[300], chunk=[300], nq=[300], swa="linear",
                    layers=2, description="prefill of 300 tokens from position 0")
    t, spec, buf = run_workload(wl)
    sel = buf.sel.cpu().numpy()
    assert np.all(sel[0] == -1) and np.all(sel[1, 1:] == -1) and sel[1, 0] == 0
    qs = [0, 1, 2, 3, 62, 63, 64, 65, 126, 127, 128, 129, 200, 299]
    check_queries(wl, t, buf, qs)


def _short_history(ratio):
    ctx = [1, 2, 64, 65, 127, 128, 129]
    return W.Workload(f"short_decode_m{ratio}", 42 + ratio, ratio, ctx=ctx, chunk=ctx,
                      nq=[1] * len(ctx), description="decode at p = 0, 1, 63, 64, 126, 127, 128")


@pytest.mark.parametrize("ratio", [1, 2])
def test_short_history_decode_through_every_merge_path(ratio):
    """Decode queries at p in {0, 1, 63, 64, 126, 127, 128} on a RING window: the step
    itself (two CTAs per query, the cluster merge; several of the CTAs have no rows),
    then the same selection once more on its own and through one CTA per query (the
    seven queries repeated twelve times)."""
    from csa2_compressed_sparse_gb300 import csa2_device_status, csa2_sparse_attn
    from csa2_compressed_sparse_gb300.step import swa_of
    wl = _short_history(ratio)
    t, spec, buf = run_workload(wl)
    assert buf.attn_ws is None  # the attention needs no workspace
    check_queries(wl, t, buf, list(range(wl.Q)))
    key = register(wl)
    sel = buf.sel
    refs = [oracle_attn(wl, key, q, sel[q].cpu().numpy())[0] for q in range(wl.Q)]
    # the same selection on its own (two CTAs per query, merged in distributed shared
    # memory)
    out = torch.empty_like(buf.out[0])
    csa2_sparse_attn(t["q"][0], t["q_seq"], t["q_pos"], swa_of(spec, t, 0), t["plane"],
                     t["row_base"], sel, t["sink"], out)
    csa2_device_status()
    for q in range(wl.Q):
        check_attn(out[q].float().cpu().numpy(), refs[q])
    # one CTA per query: 84 queries fill the GPU
    idx = torch.arange(wl.Q, device="cuda").repeat(12)
    out = torch.empty((len(idx), 64, 512), dtype=torch.bfloat16, device="cuda")
    csa2_sparse_attn(t["q"][0][idx].contiguous(), t["q_seq"][idx].contiguous(),
                     t["q_pos"][idx].contiguous(), swa_of(spec, t, 0), t["plane"], t["row_base"],
                     sel[idx].contiguous(), t["sink"], out)
    csa2_device_status()
    for i in range(len(idx)):
        check_attn(out[i].float().cpu().numpy(), refs[i % wl.Q])


def test_linear_window_below_its_first_row_is_flagged_and_skipped():
    """A LINEAR window whose first stored position (50) lies above the query's window
    start (p - 127 < 0): the positions below it raise CSA2_EBOUNDS and are skipped, so
    the result is the attention over the stored positions 50 .. p plus the selection.
    Attention does not depend on positions beyond which rows take part, so the oracle's
    query at p' = 50 over the same 51 rows (its whole window) gives the expected value."""
    from csa2_compressed_sparse_gb300 import (Csa2Error, Swa, SWA_LINEAR, csa2_device_status,
                                              csa2_sparse_attn)
    seed = 47
    p, p0 = 100, 50
    nrow = p - p0 + 1
    q = synth.rows_bf16(0, 0, 1, 64 * 512, seed, synth.Q).view(1, 64, 512)
    lin = synth.rows_bf16(0, 0, nrow, 512, seed, synth.SWA_LINEAR)
    plane = synth.rows_bf16(0, 0, 40, 512, seed, synth.PLANE)
    sink = synth.normal_f32(64, seed, synth.SINK)
    sel = np.full((1, 512), -1, dtype=np.int32)
    sel[0, :40] = np.arange(40)
    # the previous "sequence" occupies rows 0..9 of the buffer: an unguarded kernel
    # would read them for positions 40..49
    buf_rows = torch.cat([torch.full((10, 512), 7.0, dtype=torch.bfloat16), lin])
    out = torch.empty((1, 64, 512), dtype=torch.bfloat16, device="cuda")
    csa2_sparse_attn(q.cuda(), torch.zeros(1, dtype=torch.int32, device="cuda"),
                     torch.tensor([p], dtype=torch.int64, device="cuda"),
                     Swa(buf_rows.cuda(), SWA_LINEAR, torch.tensor([10], device="cuda"),
                         torch.tensor([p0], device="cuda")),
                     plane.cuda(), torch.zeros(1, dtype=torch.int64, device="cuda"),
                     torch.from_numpy(sel).cuda(), sink.cuda(), out)
    with pytest.raises(Csa2Error) as e:
        csa2_device_status()
    assert e.value.status == 4
    csa2_device_status()  # cleared by the read
    ref, _ = oracle.sparse_attn(q, [0], [p0], lin, plane, [0], sel, sink, swa_mode="linear",
                                lin_base=[0], lin_pos0=[0])
    check_attn(out[0].float().cpu().numpy(), ref[0])


def test_bounded_wait_runs_out_and_reports_a_timeout():
    """A kernel waits for an mbarrier phase that nothing completes, with a 1 ms limit:
    the wait runs out, the kernel returns, csa2_device_status reports CSA2_ETIMEOUT once,
    and the context stays usable (a following call computes and reports clean)."""
    from csa2_compressed_sparse_gb300 import (Csa2Error, csa2_device_status,
                                              csa2_selftest_wait_timeout, csa2_topk_scores)
    csa2_device_status()
    csa2_selftest_wait_timeout(1_000_000)
    with pytest.raises(Csa2Error) as e:
        csa2_device_status()
    assert e.value.status == 3
    csa2_device_status()  # clean on the next read
    s = torch.arange(100, dtype=torch.float32, device="cuda").view(1, 100)
    n = torch.tensor([100], dtype=torch.int32, device="cuda")
    sel = torch.empty((1, 5), dtype=torch.int32, device="cuda")
    csa2_topk_scores(s, n, 5, sel)
    csa2_device_status()
    assert sel.cpu().tolist() == [[95, 96, 97, 98, 99]]
