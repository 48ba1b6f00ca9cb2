"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small workloads span several tiles, ragged tails, short histories (< 512 rows), both
ratios, FULL and REINDEX, ring / linear / FP8 windows and query groups; the five
configurations are also run at full size and checked on sampled queries.  Oracle
inputs are always regenerated on the host from the seeded generator.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads as W

from _harness import (check_attn, check_scores, check_sel, host_seq, oracle_attn, oracle_index,
                      register, spec_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import csa2_compressed_sparse_gb300 as csa2
    csa2.lib()


def run_workload(wl):
    from csa2_compressed_sparse_gb300 import csa2_device_status
    from csa2_compressed_sparse_gb300.step import allocate, run_step
    t = wl.materialize("cuda")
    spec = spec_of(wl)
    buf = allocate(spec, t, want_scores=True, want_lse=True)
    run_step(spec, t, buf)
    csa2_device_status()
    return t, spec, buf


def check_queries(wl, t, buf, queries, layers=None):
    from csa2_compressed_sparse_gb300 import csa2_device_status, csa2_sparse_attn
    from csa2_compressed_sparse_gb300.step import swa_of
    key = register(wl)
    spec = spec_of(wl)
    layers = range(len(t["q"])) if layers is None else layers
    sel_gpu = buf.sel.cpu().numpy()
    scores_gpu = buf.scores_out.cpu().numpy()
    outs = [buf.out[l].float().cpu().numpy() for l in range(len(t["q"]))]
    stats = []
    for q in queries:
        sc, rows, sel_ref = oracle_index(wl, key, q)
        n = len(rows)
        rel = check_scores(scores_gpu[q, :n], sc, rows)
        ndiff = check_sel(sel_gpu[q], sel_ref, sc, rows, wl.k)
        sel_scores = buf.sel_scores[q].cpu().numpy()
        nv = int((sel_gpu[q] >= 0).sum())
        assert np.array_equal(sel_scores[:nv], scores_gpu[q, _positions(wl, q, sel_gpu[q][:nv])])
        for layer in layers:
            if ndiff == 0:
                ref, _ = oracle_attn(wl, key, q, sel_ref, layer)
                err = check_attn(outs[layer][q], ref)
            else:
                # near-tie rows differ: the step's own output is checked against the oracle's
                # attention over the GPU's selection (a valid top-k up to those ties) ...
                ref_g, _ = oracle_attn(wl, key, q, sel_gpu[q], layer)
                err = check_attn(outs[layer][q], ref_g)
                # ... and the attention kernel once more on the oracle's own selection
                one = torch.from_numpy(sel_ref.reshape(1, -1)).cuda()
                o1 = torch.empty((1, 64, 512), dtype=torch.bfloat16, device="cuda")
                csa2_sparse_attn(t["q"][layer][q:q + 1].contiguous(), t["q_seq"][q:q + 1],
                                 t["q_pos"][q:q + 1], swa_of(spec, t, layer), t["plane"],
                                 t["row_base"], one, t["sink"], o1)
                csa2_device_status()
                ref, _ = oracle_attn(wl, key, q, sel_ref, layer)
                err = max(err, check_attn(o1[0].float().cpu().numpy(), ref))
            stats.append((q, layer, rel, ndiff, err))
    print(f"\n{wl.name}: q/layer/score-rel/sel-diff/attn-rel", stats[:8])
    return stats


def _positions(wl, q, rows):
    if wl.cand is None:
        return rows
    pos = {}
    for i, blk in enumerate(wl.cand[q]):
        if blk >= 0:
            for r in range(8):
                pos[int(blk) * 8 + r] = i * 8 + r
    return np.array([pos[int(r)] for r in rows], dtype=np.int64)


# ---- the generator itself -------------------------------------------------------------------

def test_device_generator_matches_host():
    a = synth.rows_bf16(3, 100, 77, 512, 9, synth.PLANE)
    b = synth.rows_bf16(3, 100, 77, 512, 9, synth.PLANE, device="cuda").cpu()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    a = synth.rows_fp8s128(1, 5, 33, 9, synth.RING)
    b = synth.rows_fp8s128(1, 5, 33, 9, synth.RING, device="cuda").cpu()
    assert torch.equal(a, b)
    a = synth.normal_f32(1000, 4, synth.SINK)
    b = synth.normal_f32(1000, 4, synth.SINK, device="cuda").cpu()
    assert torch.equal(a, b)


# ---- top-k on given scores: bit-exact -------------------------------------------------------

@pytest.mark.parametrize("ld,k", [(1, 1), (700, 17), (16384, 512), (16385, 512), (40000, 512),
                                  (300000, 512), (5000, 1)])
def test_topk_scores_bit_exact(ld, k):
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_topk_scores,
                                              csa2_topk_workspace_size)
    g = np.random.default_rng(ld + k)
    Q = 7
    s = (g.integers(-40, 40, (Q, ld)) / 8.0).astype(np.float32)  # heavy ties
    s[1] = g.standard_normal(ld).astype(np.float32)
    s[2, ::7] = np.nan
    s[3, ::5] = -0.0
    s[4, ::3] = -np.inf
    # one value everywhere: past 8192 positions a chunk keeps more pairs than its buffer
    # holds and selects over the whole chunk instead; below, ties decide every place
    s[6] = 1.5
    n = np.array([ld, ld, max(ld - 3, 0), ld // 2, min(ld, 511), 0, ld], dtype=np.int32)
    st = torch.from_numpy(s).cuda()
    nt = torch.from_numpy(n).cuda()
    sel = torch.empty((Q, k), dtype=torch.int32, device="cuda")
    ss = torch.empty((Q, k), dtype=torch.float32, device="cuda")
    wsb = csa2_topk_workspace_size(Q, ld, k)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    csa2_topk_scores(st, nt, k, sel, ss, ws)
    csa2_device_status()
    sel = sel.cpu().numpy()
    ss = ss.cpu().numpy()
    for q in range(Q):
        ref = oracle.topk(s[q, :n[q]].astype(np.float64), np.arange(n[q]), k)
        assert np.array_equal(sel[q], ref), f"row {q}"
        m = ref >= 0
        exp = s[q, ref[m]].copy()
        exp[np.isnan(exp)] = -np.inf
        exp[exp == 0] = 0.0
        assert np.array_equal(ss[q, m], exp)


@pytest.mark.parametrize("ld", [16384, 40000])
def test_topk_scores_far_above_the_threshold(ld):
    """Rows whose best keys lie many octaves above the sampled threshold, so that the
    k-th key falls in the kept keys' shared top bin (and the exact recount path runs): a
    block of huge distinct scores, a block of +inf, and huge scores with ties among them."""
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_topk_scores,
                                              csa2_topk_workspace_size)
    g = np.random.default_rng(ld)
    Q, k = 3, 512
    s = g.standard_normal((Q, ld)).astype(np.float32)
    big = g.choice(ld, 700, replace=False)
    s[0, big] = (1e30 * (1.0 + np.arange(700) * 2.0 ** -20)).astype(np.float32)
    s[1, big[:600]] = np.inf
    s[2, big] = (1e25 * (1.0 + (np.arange(700) % 50) * 2.0 ** -16)).astype(np.float32)
    n = np.full(Q, ld, dtype=np.int32)
    st, nt = torch.from_numpy(s).cuda(), torch.from_numpy(n).cuda()
    sel = torch.empty((Q, k), dtype=torch.int32, device="cuda")
    ss = torch.empty((Q, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(csa2_topk_workspace_size(Q, ld, k), 256), dtype=torch.uint8,
                     device="cuda")
    csa2_topk_scores(st, nt, k, sel, ss, ws)
    csa2_device_status()
    sel = sel.cpu().numpy()
    for q in range(Q):
        ref = oracle.topk(s[q].astype(np.float64), np.arange(ld), k)
        assert np.array_equal(sel[q], ref), f"row {q}"


# ---- compressor ---------------------------------------------------------------------------

def _compress_case(ratio, lens_a, lens_b, seed=11):
    """Two chunked calls vs one oracle pass per sequence."""
    from csa2_compressed_sparse_gb300 import csa2_compress, csa2_device_status
    B = len(lens_a)
    tot = [a + b for a, b in zip(lens_a, lens_b)]
    nrows = [t // ratio for t in tot]
    rb = np.concatenate([[0], np.cumsum(nrows)[:-1]]).astype(np.int64)
    plane = torch.zeros((max(sum(nrows), 1), 512), dtype=torch.bfloat16, device="cuda")
    ks = torch.zeros((B, 2, 512), dtype=torch.float32, device="cuda")
    ss = torch.zeros((B, 2, 512), dtype=torch.float32, device="cuda")
    invf = torch.from_numpy(W.rope_inv_freq()).cuda()
    for start_of, lens in ((lambda b: 0, lens_a), (lambda b: lens_a[b], lens_b)):
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        kv = torch.cat([synth.rows_bf16(b, start_of(b), lens[b], 512, seed, synth.KV)
                        for b in range(B)]).cuda()
        sc = torch.cat([synth.rows_bf16(b, start_of(b), lens[b], 512, seed, synth.SCORE)
                        for b in range(B)]).cuda()
        sp = torch.tensor([start_of(b) for b in range(B)], dtype=torch.int64, device="cuda")
        csa2_compress(kv, sc, torch.from_numpy(cu).cuda(), sp, ratio, ks, ss, plane,
                      torch.from_numpy(rb).cuda(), invf)
    csa2_device_status()
    got = oracle.bf16_bits(plane)
    for b in range(B):
        kv = synth.rows_bf16(b, 0, tot[b], 512, seed, synth.KV)
        sc = synth.rows_bf16(b, 0, tot[b], 512, seed, synth.SCORE)
        ref = np.zeros((max(nrows[b], 1), 512), dtype=np.uint16)
        oks, oss = np.zeros((1, ratio, 512)), np.zeros((1, ratio, 512))
        n, pf = oracle.compress(kv, sc, [0, tot[b]], [0], ratio, oks, oss, ref, [0], W.rope_inv_freq())
        g = got[rb[b]:rb[b] + nrows[b]]
        gv = oracle.bf16_from_bits(g).double().numpy()
        err = np.abs(gv - pf[:nrows[b]])
        # one bf16 ulp of the oracle value, plus fp32 rounding at the row's scale (the
        # rotation of dims 448..511 can cancel down to values far below the row's size)
        exact = pf[:nrows[b]]
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
        tol = ulp + 2.0 ** -21 * np.abs(exact).max(axis=1, keepdims=True)
        if not np.all(err <= tol):
            i = np.unravel_index(np.argmax(err / tol), err.shape)
            raise AssertionError(f"seq {b}: row {i[0]} dim {i[1]}: gpu {gv[i]!r} oracle "
                                 f"{exact[i]!r} err {err[i]:.3g} tol {tol[i]:.3g}")
        assert np.mean(g == ref[:nrows[b]]) > 0.99
        if ratio == 2 and tot[b] % 2 == 1:  # pending tail token in slot 0
            last = synth.rows_f32(b, tot[b] - 1, 1, 512, seed, synth.KV)[0].bfloat16().float()
            assert torch.equal(ks[b, 0].cpu(), last)


@pytest.mark.parametrize("ratio", [1, 2])
def test_compress_chunked_parity(ratio):
    _compress_case(ratio, [37, 50, 1, 0, 129], [63, 1, 1, 8, 0])


def test_compress_decode_tail_roundtrip():
    _compress_case(2, [4095, 4096, 3], [1, 1, 2])


# ---- the step on small workloads -------------------------------------------------------------

SMALL = {
    "tiny": lambda: W.tiny_decode(),
    "decode_small": lambda: W.decode_batch(B=12, lo=300, hi=9000, seed=21),
    "reindex_small": lambda: W.reindex_decode(B=3, ctx=24576, ncb=256, seed=22),
    # 100 blocks: the candidate list ends inside a 16-block work tile
    "reindex_ragged": lambda: W.reindex_decode(B=3, ctx=9000, ncb=100, seed=26),
    "prefill_small": lambda: W.prefill_reuse(n_new=128, ctx=4224, layers=3, seed=23),
    "long_small": lambda: W.long_decode(B=2, ctx=40000, seed=24),
    # three prefilling sequences, 2100 queries: query runs cross the 1024-query blocks of
    # the grouping pass (groups of four queries restart at every sequence)
    "prefill_multi": lambda: W.Workload(
        "prefill_multi", 27, 2, ctx=[2000, 1601, 2300], chunk=[700, 501, 900],
        nq=[700, 501, 900], swa="linear", layers=1,
        description="three prefill chunks, 2101 queries"),
}

# queries checked per small workload (all of them when there are few)
SMALL_QUERIES = {"prefill_multi": [0, 3, 699, 700, 701, 1020, 1023, 1024, 1027, 1200, 1201,
                                   1202, 2047, 2048, 2100]}


@pytest.mark.parametrize("name", list(SMALL))
def test_step_small(name):
    wl = SMALL[name]()
    t, spec, buf = run_workload(wl)
    qs = SMALL_QUERIES.get(name, list(range(wl.Q)) if wl.Q <= 12 else [0, 1, 31, 64, 65, wl.Q - 1])
    check_queries(wl, t, buf, qs)


def test_step_h32_and_no_relu():
    from csa2_compressed_sparse_gb300 import csa2_device_status
    from csa2_compressed_sparse_gb300.step import allocate, run_step
    wl = W.decode_batch(B=5, lo=2000, hi=5000, seed=25)
    wl.H = 32
    t = wl.materialize("cuda")
    spec = spec_of(wl)
    for relu in (True, False):
        spec.relu = relu
        buf = allocate(spec, t, want_scores=True)
        run_step(spec, t, buf, compress=relu)
        csa2_device_status()
        key = register(wl)
        for q in range(wl.Q):
            sc, rows, sel_ref = oracle_index(wl, key, q, relu=relu)
            check_scores(buf.scores_out[q, :len(rows)].cpu().numpy(), sc, rows)
            check_sel(buf.sel[q].cpu().numpy(), sel_ref, sc, rows, wl.k)


@pytest.mark.parametrize("make", [
    lambda: W.decode_batch(B=12, lo=300, hi=9000, seed=29),            # one compressor CTA
    lambda: W.prefill_reuse(n_new=300, ctx=8192, layers=2, seed=31),   # 300 tokens: 10 CTAs
    lambda: W.reindex_decode(B=3, ctx=40000, ncb=96, seed=33),         # ratio 1
])
def test_fused_compress_index_topk_equals_the_separate_calls(make):
    """csa2_compress_index_topk (the compressor's tokens on extra CTAs of the top-k launch,
    one stream) against csa2_compress on a second stream next to csa2_index_topk, from the same
    starting plane and tail state: the plane, the states, the selection, the scores and the
    attention output are the same bits."""
    from csa2_compressed_sparse_gb300 import csa2_device_status
    from csa2_compressed_sparse_gb300.step import allocate, run_step
    wl = make()
    t = wl.materialize("cuda")
    spec = spec_of(wl)
    start = {k: t[k].clone() for k in ("plane", "kv_state", "score_state")}
    runs = []
    for fused in (True, False):
        for k, v in start.items():
            t[k].copy_(v)
        buf = allocate(spec, t, want_scores=True, want_lse=True)
        side = torch.cuda.Stream()
        run_step(spec, t, buf, side=side, fused=fused)
        torch.cuda.synchronize()
        csa2_device_status()
        runs.append([t["plane"].clone(), t["kv_state"].clone(), t["score_state"].clone(),
                     buf.sel.clone(), buf.scores_out.clone(), buf.out[-1].clone(),
                     buf.lse[-1].clone()])
    assert not torch.equal(runs[0][0], start["plane"]) or wl.T == 0  # the step wrote rows
    for x, y in zip(*runs):
        assert torch.equal(x.view(torch.uint8) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.uint8) if y.dtype == torch.bfloat16 else y) or \
            torch.equal(torch.nan_to_num(x.float(), nan=7.0), torch.nan_to_num(y.float(), nan=7.0))


def many_queries(q):
    """Repeats of q queries that exceed the SM count: one CTA per SM then carries on from
    query to query (the persistent layout)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return -(-(sms + 1) // q) + 1


def test_attention_split_and_unsplit_agree_with_the_oracle():
    """The same queries through two CTAs per query (a cluster: nine queries), through one
    CTA per query (the nine repeated nine times fill the GPU) and through one CTA per SM
    carrying on from query to query (more repeats than SMs); the workspace argument is
    accepted and unused."""
    from csa2_compressed_sparse_gb300 import (csa2_attn_workspace_size, csa2_device_status,
                                              csa2_sparse_attn)
    from csa2_compressed_sparse_gb300.step import swa_of
    wl = W.decode_batch(B=9, lo=300, hi=7000, seed=26)
    t, spec, buf = run_workload(wl)
    key = register(wl)
    assert csa2_attn_workspace_size(wl.Q, spec.k) == 0
    refs = [oracle_attn(wl, key, q, buf.sel[q].cpu().numpy()) for q in range(wl.Q)]
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    for rep, w in ((1, None), (1, ws), (9, None), (many_queries(wl.Q), None)):
        idx = torch.arange(wl.Q, device="cuda").repeat(rep)
        out = torch.empty((len(idx), 64, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((len(idx), 64), dtype=torch.float32, device="cuda")
        csa2_sparse_attn(t["q"][0][idx].contiguous(), t["q_seq"][idx].contiguous(),
                         t["q_pos"][idx].contiguous(), swa_of(spec, t, 0), t["plane"],
                         t["row_base"], buf.sel[idx].contiguous(), t["sink"], out, lse=lse,
                         ws=w)
        csa2_device_status()
        for i in range(len(idx)):
            ref, ref_lse = refs[i % wl.Q]
            check_attn(out[i].float().cpu().numpy(), ref)
            assert np.abs(lse[i].cpu().numpy() - ref_lse).max() < 1e-2


@pytest.mark.parametrize("rep", [1, 9, 0])
def test_attention_with_the_inverse_rope_epilogue(rep):
    """csa2_sparse_attn_rope: the output's dims 448..511 rotated back by the query position
    ([A] "出来之后"), through the two-CTA cluster merge (nine queries), through one CTA
    per query (the nine repeated nine times) and through one CTA per SM carrying on from
    query to query (rep 0: more repeats than SMs).  The other dims are the plain call's."""
    from csa2_compressed_sparse_gb300 import (csa2_device_status, csa2_sparse_attn,
                                              csa2_sparse_attn_rope)
    from csa2_compressed_sparse_gb300.step import swa_of
    wl = W.decode_batch(B=9, lo=300, hi=700000, seed=31)
    t, spec, buf = run_workload(wl)
    key = register(wl)
    idx = torch.arange(wl.Q, device="cuda").repeat(rep or many_queries(wl.Q))
    args = (t["q"][0][idx].contiguous(), t["q_seq"][idx].contiguous(),
            t["q_pos"][idx].contiguous(), swa_of(spec, t, 0), t["plane"], t["row_base"],
            buf.sel[idx].contiguous(), t["sink"])
    plain = torch.empty((len(idx), 64, 512), dtype=torch.bfloat16, device="cuda")
    rot = torch.empty_like(plain)
    csa2_sparse_attn(*args, plain)
    csa2_sparse_attn_rope(*args, rot, t["inv_freq"])
    csa2_device_status()
    assert torch.equal(plain[:, :, :448], rot[:, :, :448])
    invf = t["inv_freq"].cpu().numpy()
    for q in range(wl.Q):
        ref, _ = oracle_attn(wl, key, q, buf.sel[q].cpu().numpy(), inv_freq=invf)
        for i in range(q, len(idx), wl.Q):
            check_attn(rot[i].float().cpu().numpy(), ref)


def test_reuse_attention_with_the_inverse_rope_epilogue_one_cta_per_query():
    """csa2_reuse_attn_rope on a prefill chunk (128 queries: one CTA each), LINEAR window."""
    from csa2_compressed_sparse_gb300 import csa2_device_status, csa2_reuse_attn_rope
    from csa2_compressed_sparse_gb300.step import swa_of
    wl = SMALL["prefill_small"]()
    t, spec, buf = run_workload(wl)
    key = register(wl)
    layer = 2
    rot = torch.empty_like(buf.out[layer])
    csa2_reuse_attn_rope(t["q"][layer], t["q_seq"], t["q_pos"], swa_of(spec, t, layer), t["plane"],
                         t["row_base"], buf.sel, t["sink"], rot, t["inv_freq"])
    csa2_device_status()
    invf = t["inv_freq"].cpu().numpy()
    for q in (0, 1, 63, 127):
        ref, _ = oracle_attn(wl, key, q, buf.sel[q].cpu().numpy(), layer, inv_freq=invf)
        check_attn(rot[q].float().cpu().numpy(), ref)


def test_attention_running_max_rescale_paths():
    """Queries of heads 0..31 scaled by 2^8 (exact in bf16): their scores spread over
    hundreds of nats, so later chunks overtake the running max by far more than the
    lazy threshold and the O^T rescale runs; heads 32..63 keep the plain path."""
    from csa2_compressed_sparse_gb300 import (csa2_attn_workspace_size, csa2_device_status,
                                              csa2_sparse_attn)
    from csa2_compressed_sparse_gb300.step import swa_of
    wl = W.decode_batch(B=5, lo=300, hi=7000, seed=28)
    t, spec, buf = run_workload(wl)
    key = register(wl)
    hs = np.ones(64)
    hs[:32] = 256.0
    qs = (t["q"][0].double() * torch.tensor(hs, device="cuda").view(1, 64, 1)).to(torch.bfloat16)
    nb = csa2_attn_workspace_size(wl.Q, spec.k)
    refs = [oracle_attn(wl, key, q, buf.sel[q].cpu().numpy(), head_scale=hs) for q in range(wl.Q)]
    # two CTAs per query, and (more repeats than SMs) one CTA per SM walking its queries
    for rep, ws in ((1, None), (1, torch.empty(nb, dtype=torch.uint8, device="cuda")),
                    (many_queries(wl.Q), None)):
        idx = torch.arange(wl.Q, device="cuda").repeat(rep)
        out = torch.empty((len(idx), 64, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((len(idx), 64), dtype=torch.float32, device="cuda")
        csa2_sparse_attn(qs[idx].contiguous(), t["q_seq"][idx].contiguous(),
                         t["q_pos"][idx].contiguous(), swa_of(spec, t, 0), t["plane"],
                         t["row_base"], buf.sel[idx].contiguous(), t["sink"], out, lse=lse, ws=ws)
        csa2_device_status()
        for i in range(len(idx)):
            ref, ref_lse = refs[i % wl.Q]
            check_attn(out[i].float().cpu().numpy(), ref)
            assert np.abs(lse[i].cpu().numpy() - ref_lse).max() < 2e-2


def test_bounds_fault_is_reported_and_recoverable():
    from csa2_compressed_sparse_gb300 import (Csa2Error, Swa, csa2_device_status,
                                              csa2_sparse_attn)
    q = torch.zeros((1, 64, 512), dtype=torch.bfloat16, device="cuda")
    ring = torch.zeros((1, 128, 512), dtype=torch.bfloat16, device="cuda")
    plane = torch.zeros((10, 512), dtype=torch.bfloat16, device="cuda")
    sel = torch.full((1, 512), -1, dtype=torch.int32, device="cuda")
    sel[0, 0] = 10  # one past the plane: skipped by the kernel and flagged
    out = torch.empty((1, 64, 512), dtype=torch.bfloat16, device="cuda")
    z32 = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.tensor([500], dtype=torch.int64, device="cuda")
    rb = torch.zeros(1, dtype=torch.int64, device="cuda")
    csa2_sparse_attn(q, z32, pos, Swa(ring), plane, rb, sel, None, out)
    with pytest.raises(Csa2Error) as e:
        csa2_device_status()
    assert e.value.status == 4
    sel[0, 0] = 9
    csa2_sparse_attn(q, z32, pos, Swa(ring), plane, rb, sel, None, out)
    csa2_device_status()  # clean again
    assert torch.all(out == 0)


# ---- the five configurations at full size, sampled queries -------------------------------------

FULL = {
    "tiny": (W.tiny_decode, [0, 1, 2, 3]),
    # every query of the decode batch (the benchmarked configuration)
    "decode": (W.decode_batch, list(range(64))),
    "reindex": (W.reindex_decode, [0, 5, 11, 16, 22, 27, 31]),
    # 34 queries spread over the chunk, both ends included
    "prefill": (W.prefill_reuse, sorted(set([0, 1, 2, 3] + list(range(127, 4096, 131)) + [4094, 4095]))),
    "long": (W.long_decode, [0, 3, 7]),
}


@pytest.mark.parametrize("name", list(FULL))
def test_step_full_size(name):
    make, qs = FULL[name]
    wl = make()
    t, spec, buf = run_workload(wl)
    layers = [0, len(t["q"]) - 1] if len(t["q"]) > 1 else [0]
    check_queries(wl, t, buf, qs, layers=layers)
    del t, buf
    torch.cuda.empty_cache()
