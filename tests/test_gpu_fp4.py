"""The FP4 main plane through the C ABI: the quantiser is bit-exact against the oracle's,
and the attention reading FP4 plane rows matches the oracle's (which decodes the same
format by definition) within the attention tolerance, on ring, FP8 ring and linear
windows, one, two (cluster) and several CTAs per query, with and without the inverse
RoPE.  The selected rows are history rows (bit-identical on host and device), drawn
without replacement per query with some -1 entries."""
import numpy as np
import pytest
import torch

import oracle
from synth import workloads as W

from _harness import check_attn, oracle_attn, register, spec_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def test_plane_fp4_quantiser_is_bit_exact():
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_plane_fp4,
                                              csa2_plane_fp4_bytes)
    g = np.random.default_rng(9)
    n = 333
    x = g.standard_normal((n, 512)) * np.exp2(g.integers(-12, 12, (n, 32)).repeat(16, axis=1))
    x[4, :16] = 0.0                                   # an all-zero group
    e4 = np.array([oracle.e4m3_value(c) for c in range(1, 0x7F)])
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])
    for r in range(8, 40):                            # E2M1 ties at exact E4M3 scales
        s = e4[g.integers(20, 110)]
        x[r, :16] = g.choice(mids, 16) * s * g.choice([-1.0, 1.0], 16)
        x[r, 0] = 6.0 * s                             # pins the scale to s
    x[41, :16] = 1e-30                                # tiny: the smallest scales
    k = torch.from_numpy(x.astype(np.float32)).bfloat16()
    out = torch.full((csa2_plane_fp4_bytes(n),), 0xA5, dtype=torch.uint8, device="cuda")
    csa2_plane_fp4(k.cuda(), out)
    csa2_device_status()
    ref = oracle.plane_fp4(k).reshape(-1)
    got = out.cpu().numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first row {bad[0] // 288} byte {bad[0] % 288}"


def _sel_history(wl, nsel, seed):
    g = np.random.default_rng(seed)
    sel = np.full((wl.Q, nsel), -1, dtype=np.int32)
    for q in range(wl.Q):
        nh = int(wl.n_hist[wl.q_seq[q]])
        take = min(nsel - nsel // 8, nh)
        sel[q, :take] = np.sort(g.choice(nh, take, replace=False))
    return sel


@pytest.mark.parametrize("name", ["ring", "fp8ring", "linear", "many"])
def test_attention_on_an_fp4_plane_matches_the_oracle(name):
    from csa2_compressed_sparse_gb300 import (csa2_attn_workspace_size, csa2_device_status,
                                              csa2_plane_fp4, csa2_plane_fp4_bytes,
                                              csa2_sparse_attn_fp4)
    from csa2_compressed_sparse_gb300.step import swa_of
    if name == "ring":
        wl = W.decode_batch(B=6, lo=3000, hi=9000, seed=81)
    elif name == "fp8ring":
        wl = W.Workload("fp4_fp8ring", 82, 1, ctx=[20000, 5001], chunk=[1, 1], nq=[1, 1],
                        swa_dtype="fp8")
    elif name == "linear":
        wl = W.prefill_reuse(n_new=96, ctx=8192, layers=1, seed=83)
    else:  # many queries: one CTA per query
        wl = W.decode_batch(B=160, lo=2000, hi=4000, seed=84)
    key = register(wl)
    t = wl.materialize("cuda")
    spec = spec_of(wl)
    sel = _sel_history(wl, 512, seed=85)
    rows = t["plane"].shape[0]
    p4 = torch.empty(csa2_plane_fp4_bytes(rows), dtype=torch.uint8, device="cuda")
    csa2_plane_fp4(t["plane"], p4)
    out = torch.empty((wl.Q, 64, 512), dtype=torch.bfloat16, device="cuda")
    # a workspace is accepted and unused (its size is 0): the runs with and without one
    # take the same path (two CTAs per query for few queries, merged in distributed
    # shared memory)
    ws = torch.empty(max(csa2_attn_workspace_size(wl.Q, 512), 256), dtype=torch.uint8,
                     device="cuda")
    runs = [(False, ws), (True, ws)] + ([(False, None), (True, None)] if wl.Q <= 76 else [])
    for rope, ws in runs:
        invf = t["inv_freq"] if rope else None
        csa2_sparse_attn_fp4(t["q"][0], t["q_seq"], t["q_pos"], swa_of(spec, t, 0), p4, rows,
                             t["row_base"], torch.from_numpy(sel).cuda(), t["sink"], out,
                             inv_freq=invf, ws=ws)
        csa2_device_status()
        got = out.float().cpu().numpy()
        for q in sorted({0, wl.Q // 2, wl.Q - 1}):
            ref, _ = oracle_attn(wl, key, q, sel[q], inv_freq=wl.inv_freq if rope else None,
                                 fp4_plane=True)
            check_attn(got[q], ref)


def test_attention_on_an_e8m0_fp8_window_matches_the_oracle():
    # the pool switch's 528-byte window rows (512 E4M3, 16 E8M0 scales) in a ring
    from csa2_compressed_sparse_gb300 import (SWA_FP8_E8M0, SWA_RING, Swa, csa2_device_status,
                                              csa2_sparse_attn)
    g = np.random.default_rng(77)
    B, Q = 3, 5
    ring = np.zeros((B, 128, 528), dtype=np.uint8)
    ring[..., :512] = (g.integers(0, 0x7F, (B, 128, 512)) |
                       (g.integers(0, 2, (B, 128, 512)) << 7)).astype(np.uint8)
    ring[..., 512:] = g.integers(121, 133, (B, 128, 16)).astype(np.uint8)
    plane = torch.from_numpy(g.standard_normal((300, 512)).astype(np.float32)).bfloat16()
    q = torch.from_numpy(g.standard_normal((Q, 64, 512)).astype(np.float32)).bfloat16()
    q_seq = np.array([0, 1, 2, 2, 0], dtype=np.int32)
    q_pos = np.array([700, 33, 1000, 999, 128], dtype=np.int64)
    row_base = np.array([0, 100, 200], dtype=np.int64)
    sel = g.integers(0, 100, (Q, 256)).astype(np.int32)
    sel[:, 200:] = -1
    sink = g.standard_normal(64).astype(np.float32)
    out = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device="cuda")
    swa = Swa(torch.from_numpy(ring).cuda(), SWA_RING, fp8_dtype=SWA_FP8_E8M0)
    csa2_sparse_attn(q.cuda(), torch.from_numpy(q_seq).cuda(), torch.from_numpy(q_pos).cuda(),
                     swa, plane.cuda(), torch.from_numpy(row_base).cuda(),
                     torch.from_numpy(sel).cuda(), torch.from_numpy(sink).cuda(), out)
    csa2_device_status()
    ref, _ = oracle.sparse_attn(q, q_seq, q_pos, torch.from_numpy(ring), plane, row_base, sel,
                                sink, swa_e8m0=True)
    got = out.float().cpu().numpy()
    for i in range(Q):
        check_attn(got[i], ref[i])


def test_attention_without_a_sink_through_every_path():
    """sink = NULL (no sink term): the running max starts at the first chunk's own
    largest score.  Heads 0..15 carry queries scaled by 2^8, so their later chunks also
    overtake the running max.  Two CTAs per query (the cluster merge), with and without
    the (unused) workspace argument, and one CTA per query (the queries repeated to fill
    the GPU)."""
    from csa2_compressed_sparse_gb300 import (SWA_RING, Swa, csa2_attn_workspace_size,
                                              csa2_device_status, csa2_sparse_attn)
    g = np.random.default_rng(91)
    B, Q = 3, 6
    ring = torch.from_numpy(g.standard_normal((B, 128, 512)).astype(np.float32)).bfloat16()
    plane = torch.from_numpy(g.standard_normal((900, 512)).astype(np.float32)).bfloat16()
    qf = g.standard_normal((Q, 64, 512))
    qf[:, :16] *= 256.0
    q = torch.from_numpy(qf.astype(np.float32)).bfloat16()
    q_seq = np.array([0, 1, 2, 2, 0, 1], dtype=np.int32)
    q_pos = np.array([700, 5, 1000, 999, 128, 64], dtype=np.int64)
    row_base = np.array([0, 300, 600], dtype=np.int64)
    sel = g.integers(0, 300, (Q, 512)).astype(np.int32)
    sel[1, 100:] = -1
    sel[5, :] = -1
    ref, ref_lse = oracle.sparse_attn(q, q_seq, q_pos, ring, plane, row_base, sel, None)
    dev = dict(q_seq=torch.from_numpy(q_seq).cuda(), q_pos=torch.from_numpy(q_pos).cuda(),
               row_base=torch.from_numpy(row_base).cuda(), sel=torch.from_numpy(sel).cuda())
    swa = Swa(ring.cuda(), SWA_RING)
    ws = torch.empty(csa2_attn_workspace_size(Q, 512), dtype=torch.uint8, device="cuda")
    for w in (None, ws):
        out = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((Q, 64), dtype=torch.float32, device="cuda")
        csa2_sparse_attn(q.cuda(), dev["q_seq"], dev["q_pos"], swa, plane.cuda(),
                         dev["row_base"], dev["sel"], None, out, lse=lse, ws=w)
        csa2_device_status()
        got = out.float().cpu().numpy()
        for i in range(Q):
            check_attn(got[i], ref[i])
            assert np.abs(lse[i].cpu().numpy() - ref_lse[i]).max() < 2e-2
    idx = torch.arange(Q, device="cuda").repeat(14)
    out = torch.empty((len(idx), 64, 512), dtype=torch.bfloat16, device="cuda")
    csa2_sparse_attn(q.cuda()[idx].contiguous(), dev["q_seq"][idx].contiguous(),
                     dev["q_pos"][idx].contiguous(), swa, plane.cuda(), dev["row_base"],
                     dev["sel"][idx].contiguous(), None, out)
    csa2_device_status()
    got = out.float().cpu().numpy()
    for i in range(len(idx)):
        check_attn(got[i], ref[i % Q])
