"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each pin is an independent route to the same number: a library routine (numpy
matmul, scipy expit, torch's bf16 / float8 conversions), a closed form, an
invariant, brute force on tiny inputs, or a count printed on the pages
(tests/golden).  A plausible slip in the oracle -- a dropped term, a wrong sign,
a transposed operand, an off-by-one in visibility -- fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from synth import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden", "tail_and_visibility.json")
RNG = np.random.default_rng(1234)


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).bfloat16()


def bf16_np(t):
    return t.float().numpy().astype(np.float64)


# ---- number formats ---------------------------------------------------------------

def test_bf16_rounding_matches_torch_on_floats():
    x = (RNG.standard_normal(20000) * np.exp(RNG.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).bfloat16().view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f64_to_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_single_rounding_from_double():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties to even -> 1.0
    assert oracle.f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # just above the tie rounds up; a detour through float would round to the tie
    # and then to even, giving 0x3F80.
    assert oracle.f64_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.f64_to_bf16(-2.0) == 0xC000


def test_e4m3_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = np.array([oracle.e4m3_value(c) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


# ---- visibility ---------------------------------------------------------------------

def test_visibility_closed_form():
    for m in (1, 2, 3, 4):
        for p in list(range(0, 40)) + [1023, 1024, 1025, 4095, 262143, 1048575]:
            assert oracle.n_visible(p, m) == (p + 1) // m


def test_golden_selected_and_window_widths():
    g = json.load(open(GOLD))
    for e in g["selected_width"]:
        assert min(oracle.n_visible(e["pos"], e["ratio"]), 512) == e["width"]
    for e in g["window_width"]:
        assert min(e["pos"] + 1, 128) == e["width"]
    c = g["candidate_rows"]
    assert c["blocks"] * c["block_rows"] == c["rows"] and c["rows"] >= c["topk"]
    assert 128 + 512 == g["max_entries"]


# ---- compressor ---------------------------------------------------------------------

INV_FREQ = workloads.rope_inv_freq()


def run_compress(kv, score, ratio, chunks, start=0, norm_w=None, eps=1e-6):
    """Compress one sequence given as [S,512] float arrays, fed in the given chunk sizes."""
    S = kv.shape[0]
    assert sum(chunks) == S
    nrows = (start + S) // ratio
    plane = np.zeros((max(nrows, 1), 512), dtype=np.uint16)
    pf = np.zeros((max(nrows, 1), 512))
    ks = np.zeros((1, ratio, 512))
    ss = np.zeros((1, ratio, 512))
    total = 0
    off = 0
    for c in chunks:
        kvb = oracle.bf16_bits(bf16(kv[off:off + c]))
        scb = oracle.bf16_bits(bf16(score[off:off + c]))
        n, f = oracle.compress(kvb, scb, [0, c], [start + off], ratio, ks, ss, plane, [0],
                               INV_FREQ, norm_w=norm_w, eps=eps)
        rows_now = (start + off + c) // ratio
        first = (start + off) // ratio
        pf[first:rows_now] = f[first:rows_now]
        total += n
        off += c
    return total, plane, pf, ks, ss


def rope_angles(pos):
    return pos * INV_FREQ.astype(np.float64)


def test_golden_tail_counts():
    g = json.load(open(GOLD))
    for ratio, key in ((2, "tail_ratio2"), (1, "tail_ratio1")):
        for e in g[key]:
            S = e["processed"]
            kv = RNG.standard_normal((S, 512))
            n, *_ = run_compress(kv, kv, ratio, [S - 2, 1, 1] if S > 2 else [S])
            assert n == e["complete_rows"]
            assert S - n * ratio == e["pending_tokens"]


def test_ratio1_norm_and_rotation_invariants():
    S = 40
    kv = bf16_np(bf16(RNG.standard_normal((S, 512)) * 3.0))
    n, plane, pf, *_ = run_compress(kv, kv, 1, [S], eps=1e-6)
    assert n == S
    for t in range(S):
        x = kv[t]
        ms = np.mean(x * x)
        rstd = 1.0 / math.sqrt(ms + 1e-6)
        y = pf[t]
        # NoPE dims are the input scaled by one factor (normalised over all 512 dims)
        np.testing.assert_allclose(y[:448], x[:448] * rstd, rtol=1e-12, atol=1e-12)
        # the rotation preserves each pair's norm
        n_in = x[448::2] ** 2 + x[449::2] ** 2
        n_out = y[448::2] ** 2 + y[449::2] ** 2
        np.testing.assert_allclose(n_out, n_in * rstd * rstd, rtol=1e-12)
        # rotating back by the conjugate phase e^{-i t theta_i} recovers the input
        z = (y[448::2] + 1j * y[449::2]) * np.exp(-1j * rope_angles(t))
        np.testing.assert_allclose(z.real, x[448::2] * rstd, atol=1e-12)
        np.testing.assert_allclose(z.imag, x[449::2] * rstd, atol=1e-12)
        # stored row is the double value rounded to bf16 once
        assert all(plane[t, d] == oracle.f64_to_bf16(y[d]) for d in range(0, 512, 37))


def test_rope_unit_vector_phase_and_sign():
    # (1, 0) at pair i maps to (cos, sin) and (0, 1) to (-sin, cos): multiplication of
    # x_{2i} + i x_{2i+1} by e^{i p theta_i}.
    S = 12
    kv = np.zeros((S, 512))
    kv[:, :448] = 1.0
    kv[::2, 448] = 5.0   # even tokens: unit vector in the first dim of pair 0
    kv[1::2, 449] = 5.0  # odd tokens: second dim of pair 0
    n, _, pf, *_ = run_compress(kv, kv, 1, [S])
    for t in range(S):
        y = pf[t]
        ms = np.mean(kv[t] ** 2)
        r = 5.0 / math.sqrt(ms + 1e-6)
        a = t * float(INV_FREQ[0])
        if t % 2 == 0:
            np.testing.assert_allclose(y[448:450], [r * math.cos(a), r * math.sin(a)], atol=1e-12)
        else:
            np.testing.assert_allclose(y[448:450], [-r * math.sin(a), r * math.cos(a)], atol=1e-12)


def test_inverse_rope_undoes_the_compressor_rotation_at_the_same_position():
    # [A] "出来之后" / [B] §6.1: the attention output's last 64 dims are rotated back at the
    # query's own position.  A row the compressor rotated at position t (ratio 1), read
    # back by a query at position t, must come out as the unrotated RMSNorm row; rows read
    # at another position keep the difference of the two phases.
    S = 9
    kv = RNG.standard_normal((S, 512))
    n, _, pf, *_ = run_compress(kv, kv, 1, [S])
    kvr = bf16(kv).double().numpy()  # the compressor sees bf16 inputs
    plain = kvr / np.sqrt(np.mean(kvr ** 2, axis=1, keepdims=True) + 1e-6)
    out = np.repeat(pf[:, None, :], 64, axis=1).copy()  # every head sees its row
    oracle.inverse_rope(out, np.arange(S), INV_FREQ)
    for t in range(S):
        np.testing.assert_allclose(out[t], np.broadcast_to(plain[t], (64, 512)), atol=1e-12)
    out = np.repeat(pf[:, None, :], 64, axis=1).copy()
    oracle.inverse_rope(out, np.arange(S) + 3, INV_FREQ)  # three positions later
    for t in range(S):
        for i in (0, 5, 31):
            a = -3.0 * float(INV_FREQ[i])
            c, s_ = math.cos(a), math.sin(a)
            x0, x1 = plain[t, 448 + 2 * i], plain[t, 449 + 2 * i]
            np.testing.assert_allclose(out[t, 7, 448 + 2 * i:450 + 2 * i],
                                       [x0 * c - x1 * s_, x0 * s_ + x1 * c], atol=1e-12)


def test_inverse_rope_unit_vector_and_invariants():
    # (1, 0) in pair i at position p maps to (cos p theta_i, -sin p theta_i) (the
    # conjugate phase); the 448 content dims and every pair's norm are unchanged.
    out = np.zeros((3, 64, 512))
    out[:, :, 448::2] = 1.0
    out[:, :, :448] = RNG.standard_normal((3, 64, 448))
    before = out.copy()
    pos = np.array([0, 7, 1048575])
    oracle.inverse_rope(out, pos, INV_FREQ)
    for qi, p in enumerate(pos):
        ang = p * INV_FREQ.astype(np.float64)
        np.testing.assert_allclose(out[qi, 11, 448::2], np.cos(ang), atol=1e-12)
        np.testing.assert_allclose(out[qi, 11, 449::2], -np.sin(ang), atol=1e-12)
    assert np.array_equal(out[:, :, :448], before[:, :, :448])
    norms = out[:, :, 448::2] ** 2 + out[:, :, 449::2] ** 2
    np.testing.assert_allclose(norms, 1.0, atol=1e-12)


def test_ratio2_group_head_position_and_equal_scores_mean():
    # Two identical tokens with equal gates pool to that token; the row must then equal
    # the ratio-1 row at the group's FIRST position j*m (not j*m+1).
    S = 16
    base = RNG.standard_normal((S // 2, 512))
    kv = np.repeat(base, 2, axis=0)
    sc = np.zeros((S, 512))
    _, _, pf2, *_ = run_compress(kv, sc, 2, [S])
    _, _, pf1, *_ = run_compress(kv, sc, 1, [S])
    for j in range(S // 2):
        np.testing.assert_allclose(pf2[j], pf1[2 * j], atol=1e-12)
        assert np.max(np.abs(pf2[j] - pf1[2 * j + 1])) > 1e-3
    # equal gates with different tokens: the mean of the pair, before RMSNorm
    kv = bf16_np(bf16(RNG.standard_normal((S, 512))))
    _, _, pf, *_ = run_compress(kv, np.full((S, 512), 0.25), 2, [S])
    for j in range(S // 2):
        r = 0.5 * (kv[2 * j] + kv[2 * j + 1])
        rstd = 1.0 / math.sqrt(np.mean(r * r) + 1e-6)
        np.testing.assert_allclose(pf[j][:448], r[:448] * rstd, rtol=1e-11, atol=1e-12)


def test_ratio2_gate_is_per_channel_sigmoid():
    # softmax over two slots = logistic function of the difference, channel by channel.
    S = 8
    kv = bf16_np(bf16(RNG.standard_normal((S, 512))))
    sc = bf16_np(bf16(RNG.standard_normal((S, 512)) * 2.0))
    _, _, pf, *_ = run_compress(kv, sc, 2, [S])
    for j in range(S // 2):
        g = expit(sc[2 * j] - sc[2 * j + 1])
        r = kv[2 * j + 1] + g * (kv[2 * j] - kv[2 * j + 1])
        rstd = 1.0 / math.sqrt(np.mean(r * r) + 1e-6)
        np.testing.assert_allclose(pf[j][:448], r[:448] * rstd, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("ratio", [1, 2])
def test_chunked_equals_one_shot(ratio):
    S = 37
    kv = RNG.standard_normal((S, 512))
    sc = RNG.standard_normal((S, 512))
    for start in (0, 5):
        n1, p1, *_ = run_compress(kv, sc, ratio, [S], start=start)
        for chunks in ([1] * S, [3, 4, 1, 29], [2, 2, 33], [36, 1]):
            n2, p2, *_ = run_compress(kv, sc, ratio, chunks, start=start)
            assert n2 == n1
            first = start // ratio
            assert np.array_equal(p1[first:], p2[first:])


def test_norm_weight_applies_per_channel():
    S = 4
    kv = RNG.standard_normal((S, 512))
    nw = RNG.uniform(0.5, 1.5, 512).astype(np.float32)
    _, _, pa, *_ = run_compress(kv, kv, 1, [S])
    _, _, pb, *_ = run_compress(kv, kv, 1, [S], norm_w=nw)
    np.testing.assert_allclose(pb[:, :448], pa[:, :448] * nw[:448].astype(np.float64), rtol=1e-12)


# ---- indexer ------------------------------------------------------------------------

def make_index_case(Q=3, H=64, rows=300, seq=2):
    iq = bf16(RNG.standard_normal((Q, H, 128)))
    K = bf16(RNG.standard_normal((rows * seq, 128)))
    w = RNG.standard_normal((Q, H)).astype(np.float32)
    row_base = np.array([0, rows][:seq], dtype=np.int64)
    return iq, K, w, row_base


def test_index_single_head_is_relu_gemv():
    iq, K, w, rb = make_index_case(Q=2, H=1, rows=200, seq=1)
    w = np.ones((2, 1), dtype=np.float32)
    pos = np.array([399, 250])  # ratio 2 -> 200, 125 visible
    sc, rows = oracle.index_scores(iq, w, K, rb, [0, 0], pos, 2)
    Kd, qd = bf16_np(K), bf16_np(iq)
    for q in range(2):
        nv = (pos[q] + 1) // 2
        ref = np.maximum(Kd[:nv] @ qd[q, 0], 0.0) / math.sqrt(128)
        np.testing.assert_allclose(sc[q, :nv], ref, rtol=1e-12, atol=1e-12)
        assert np.all(rows[q, :nv] == np.arange(nv)) and np.all(rows[q, nv:] == -1)


@pytest.mark.parametrize("H", [32, 64])
def test_index_one_hot_weights_and_linearity(H):
    iq, K, w, rb = make_index_case(Q=1, H=H, rows=150, seq=2)
    Kd, qd = bf16_np(K), bf16_np(iq)
    pos = [299]
    alpha = 1.0 / math.sqrt(128 * H)
    for h in (0, 7, H - 1):
        oh = np.zeros((1, H), dtype=np.float32)
        oh[0, h] = 1.0
        sc, _ = oracle.index_scores(iq, oh, K, rb, [1], pos, 2)
        ref = alpha * np.maximum(Kd[150:300] @ qd[0, h], 0.0)
        np.testing.assert_allclose(sc[0, :150], ref, rtol=1e-12, atol=1e-13)
    # dyadic weights: w1 + w2 is exact in fp32, so the score is exactly linear in w
    w1 = (RNG.integers(-64, 64, (1, H)) / 8.0).astype(np.float32)
    w2 = (RNG.integers(-64, 64, (1, H)) / 8.0).astype(np.float32)
    s1, _ = oracle.index_scores(iq, w1, K, rb, [1], pos, 2)
    s2, _ = oracle.index_scores(iq, w2, K, rb, [1], pos, 2)
    s12, _ = oracle.index_scores(iq, w1 + w2, K, rb, [1], pos, 2)
    np.testing.assert_allclose(s12, s1 + s2, rtol=1e-9, atol=1e-12)


def test_index_without_relu_is_one_gemv():
    iq, K, w, rb = make_index_case(Q=1, H=64, rows=120, seq=1)
    Kd, qd = bf16_np(K), bf16_np(iq)
    sc, _ = oracle.index_scores(iq, w, K, rb, [0], [119], 1, relu=False)
    qc = (w[0].astype(np.float64)[:, None] * qd[0]).sum(0)
    ref = (Kd @ qc) / math.sqrt(128 * 64)
    np.testing.assert_allclose(sc[0, :120], ref, rtol=1e-9, atol=1e-12)


def test_index_reindex_rows_and_masks():
    iq, K, w, rb = make_index_case(Q=1, H=64, rows=200, seq=1)
    cand = np.array([[0, 3, 24, -1]], dtype=np.int32)  # block 24 -> rows 192..199
    pos = [196]  # ratio 1 -> 197 visible: rows 192..196 visible, 197..199 not
    sc, rows = oracle.index_scores(iq, w, K, rb, [0], pos, 1, cand=cand)
    full, frows = oracle.index_scores(iq, w, K, rb, [0], pos, 1)
    expect_rows = list(range(0, 8)) + list(range(24, 32)) + list(range(192, 197)) + [-1] * 11
    assert rows[0].tolist() == expect_rows
    for i, r in enumerate(expect_rows):
        if r >= 0:
            assert sc[0, i] == full[0, r]


# ---- index K production in the compressor ---------------------------------------------------

def run_compress_index(kv, ratio, wk, knorm_w=None, start=0, eps=1e-6):
    """One sequence [S,512] (kv used as score too) in one call: plane, index rows, f64s."""
    S = kv.shape[0]
    nrows = max((start + S) // ratio, 1)
    plane = np.zeros((nrows, 512), dtype=np.uint16)
    ip = np.zeros((nrows, 128), dtype=np.uint16)
    ks = np.zeros((1, ratio, 512))
    ss = np.zeros((1, ratio, 512))
    kvb = oracle.bf16_bits(bf16(kv))
    n, pf, kf = oracle.compress_index(kvb, kvb, [0, S], [start], ratio, ks, ss, plane, ip, [0],
                                      INV_FREQ, wk, knorm_w=knorm_w, eps=eps)
    return n, plane, pf, ip, kf


def _onehot_wk(pairs):
    wk = np.zeros((128, 512), dtype=np.float32)
    for o, d, v in pairs:
        wk[o, d] = v
    return oracle.bf16_bits(bf16(wk))


def test_index_k_single_weight_closed_form():
    # one nonzero weight wk[o][d] = v: k = v x[d] at output o only; the RMSNorm over the
    # 128 outputs turns it into sign(v x[d]) * sqrt(128) (eps negligible), rotated by the
    # row's RoPE phase when o is in the last 64 dims
    S = 12
    kv = bf16_np(bf16(RNG.standard_normal((S, 512)) * 2.0))
    for o, d, v in ((5, 77, 0.75), (64, 300, -1.5), (97, 449, 2.0), (127, 0, 1.0)):
        n, plane, pf, ip, kf = run_compress_index(kv, 1, _onehot_wk([(o, d, v)]), eps=0.0)
        assert n == S
        for t in range(S):
            xd = bf16_np(bf16(pf[t]))  # the latent before RoPE equals pf on NoPE dims
            # the pre-RoPE latent of dim d: undo the main rotation where d is a RoPE dim
            if d >= 448:
                i = (d - 448) // 2
                z = (pf[t, 448 + 2 * i] + 1j * pf[t, 449 + 2 * i]) * np.exp(-1j * rope_angles(t)[i])
                pre = z.real if d % 2 == 0 else z.imag
            else:
                pre = pf[t, d]
            sgn = math.copysign(1.0, v * float(bf16_np(bf16(np.array([pre])))[0]))
            expect = np.zeros(128)
            expect[o] = sgn * math.sqrt(128)
            if o >= 64:
                i = (o - 64) // 2
                ang = rope_angles(t)[i]
                a0, a1 = expect[64 + 2 * i], expect[65 + 2 * i]
                expect[64 + 2 * i] = a0 * math.cos(ang) - a1 * math.sin(ang)
                expect[65 + 2 * i] = a0 * math.sin(ang) + a1 * math.cos(ang)
            np.testing.assert_allclose(kf[t], expect, atol=1e-9)
            assert all(ip[t, c] == oracle.f64_to_bf16(kf[t, c]) for c in range(128))


def test_index_k_projects_the_bf16_latent_before_rope():
    # two outputs below 64 (no rotation): their ratio is the ratio of the two dot products
    # of wk rows with the bf16-rounded latent before RoPE, the main plane is unchanged
    S = 9
    kv = bf16_np(bf16(RNG.standard_normal((S, 512))))
    wrow = RNG.standard_normal((2, 512)).astype(np.float32)
    wk = np.zeros((128, 512), dtype=np.float32)
    wk[3], wk[40] = wrow[0], wrow[1]
    wkb = oracle.bf16_bits(bf16(wk))
    wkd = bf16_np(bf16(wk))
    n, plane, pf, ip, kf = run_compress_index(kv, 1, wkb)
    n0, plane0, pf0, *_ = run_compress(kv, kv, 1, [S])
    assert np.array_equal(plane, plane0)
    for t in range(S):
        pre = pf[t].copy()
        z = (pf[t, 448::2] + 1j * pf[t, 449::2]) * np.exp(-1j * rope_angles(t))
        pre[448::2], pre[449::2] = z.real, z.imag
        x = bf16_np(bf16(pre))
        d3, d40 = wkd[3] @ x, wkd[40] @ x
        np.testing.assert_allclose(kf[t, 3] / kf[t, 40], d3 / d40, rtol=1e-9)
        # and the RMSNorm over the 128 outputs (weight 1, eps 1e-6) sets their sum of
        # squares to 128 ms / (ms + eps)
        ms = (d3 * d3 + d40 * d40) / 128.0
        np.testing.assert_allclose(np.sum(kf[t] ** 2), 128.0 * ms / (ms + 1e-6), rtol=1e-9)


def test_index_k_norm_weight_rope_phase_and_group_position():
    # ratio 2: row j rotates at its group-head position 2j; k_norm's weight scales each
    # output; the rotation keeps each pair's norm and is undone by the conjugate phase
    S = 20
    kv = bf16_np(bf16(RNG.standard_normal((S, 512))))
    wk = oracle.bf16_bits(bf16(RNG.standard_normal((128, 512)) * 0.05))
    kw = (1.0 + RNG.integers(0, 4, 128) * 0.25).astype(np.float32)
    n1, _, _, _, k1 = run_compress_index(kv, 2, wk)
    n2, _, _, _, k2 = run_compress_index(kv, 2, wk, knorm_w=kw)
    assert n1 == n2 == S // 2
    for j in range(S // 2):
        ang = rope_angles(2 * j)
        u1 = (k1[j, 64::2] + 1j * k1[j, 65::2]) * np.exp(-1j * ang)
        u2 = (k2[j, 64::2] + 1j * k2[j, 65::2]) * np.exp(-1j * ang)
        np.testing.assert_allclose(k2[j, :64], k1[j, :64] * kw[:64], rtol=1e-12)
        np.testing.assert_allclose(u2.real, u1.real * kw[64::2], rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(u2.imag, u1.imag * kw[65::2], rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(np.abs(u1) ** 2, k1[j, 64::2] ** 2 + k1[j, 65::2] ** 2,
                                   rtol=1e-12)


# ---- FP4 main plane ----------------------------------------------------------

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_nearest_even(x):
    """Brute force over the 8 magnitudes; ties go to the code with mantissa bit 0."""
    a = min(abs(x), 6.0)
    d = [abs(v - a) for v in E2M1]
    best = min(range(8), key=lambda c: (d[c], c & 1))
    return best | (8 if math.copysign(1.0, x) < 0 else 0)


def test_e2m1_codes_by_brute_force_and_ties():
    vals = E2M1 + [(E2M1[i] + E2M1[i + 1]) / 2 for i in range(7)] + list(RNG.uniform(-7, 7, 3000))
    for x in vals + [-v for v in vals]:
        assert oracle.e2m1_code(x) == _e2m1_nearest_even(x), x
    assert [oracle.e2m1_value(c) for c in range(8)] == E2M1
    assert oracle.e2m1_code(0.25) == 0 and oracle.e2m1_code(0.75) == 2 and oracle.e2m1_code(5.0) == 6
    assert oracle.e2m1_code(100.0) == 7 and oracle.e2m1_code(-100.0) == 15


def test_fp4_plane_layout_scales_and_error():
    n = 6
    x = RNG.standard_normal((n, 512)) * np.exp2(RNG.integers(-4, 4, (n, 32)).repeat(16, axis=1))
    x[2, 16:32] = 0.0  # an all-zero group: scale 0, codes 0
    rows = bf16(x)
    xd = bf16_np(rows)
    out = oracle.plane_fp4(rows)
    assert out.shape == (n, 288)
    e4 = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    for r in range(n):
        codes = np.empty(512, dtype=np.int64)
        codes[0::2] = out[r, :256] & 15
        codes[1::2] = out[r, :256] >> 4
        for g in range(32):
            amax = np.abs(xd[r, 16 * g:16 * g + 16]).max()
            sc = int(out[r, 256 + g])
            if amax == 0:
                assert sc == 0 and np.all(codes[16 * g:16 * g + 16] == 0)
                continue
            s = e4[sc]
            assert 6 * s >= amax and (sc == 0 or 6 * e4[sc - 1] < amax)  # the smallest that fits
            for i in range(16):
                d = 16 * g + i
                assert codes[d] == _e2m1_nearest_even(xd[r, d] / s)
    # row 2, group 1 decodes to zeros; the rest within half a code step of the input
    deq = np.array([[oracle.e2m1_value((out[r, d // 2] >> (4 * (d & 1))) & 15) *
                     e4[out[r, 256 + d // 16]] for d in range(512)] for r in range(n)])
    assert np.all(deq[2, 16:32] == 0)
    rel = np.abs(deq - xd) / np.repeat(np.abs(xd).reshape(n, 32, 16).max(2), 16, axis=1).clip(1e-30)
    # half the widest E2M1 step (2, between 4 and 6) times the scale, and the scale is at
    # most 9/8 of amax / 6 (the smallest E4M3 value above it)
    assert rel.max() <= 1.0 * (9 / 8) / 6 + 1e-12


def test_attention_on_an_fp4_plane_equals_the_dequantised_bf16_plane():
    # E2M1 times E4M3 has at most six significant bits, so the dequantised plane is exact
    # in bf16: the FP4 path must give the bf16 path's result on that plane, bit for bit
    rows = bf16(RNG.standard_normal((40, 512)))
    p4 = oracle.plane_fp4(rows)
    e4 = np.array([oracle.e4m3_value(c) for c in range(256)])
    deq = np.array([[oracle.e2m1_value((p4[r, d // 2] >> (4 * (d & 1))) & 15) *
                     e4[p4[r, 256 + d // 16]] for d in range(512)] for r in range(40)])
    plane_bf = bf16(deq)
    assert np.array_equal(bf16_np(plane_bf), deq)
    q = bf16(RNG.standard_normal((2, 64, 512)))
    ring = bf16(RNG.standard_normal((1, 128, 512)))
    sel = np.array([[3, 0, 39, -1, 17, 8], [5, 5, -1, 22, 1, 30]], dtype=np.int32)
    sink = RNG.standard_normal(64).astype(np.float32)
    a, la = oracle.sparse_attn(q, [0, 0], [300, 77], ring, plane_bf, [0], sel, sink)
    b, lb = oracle.sparse_attn(q, [0, 0], [300, 77], ring, p4, [0], sel, sink)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def _e8m0_ring(g, B):
    """[B,128,528] uint8 rows: random finite E4M3 codes, then 16 E8M0 scales in 2^-6..2^5."""
    ring = np.zeros((B, 128, 528), dtype=np.uint8)
    codes = g.integers(0, 0x7F, (B, 128, 512)) | (g.integers(0, 2, (B, 128, 512)) << 7)
    ring[..., :512] = codes.astype(np.uint8)
    ring[..., 512:] = g.integers(121, 133, (B, 128, 16)).astype(np.uint8)
    return ring


def test_attention_on_an_e8m0_window_equals_the_dequantised_bf16_window():
    # E4M3 times a power of two is exact in bf16: the E8M0 window path must give the
    # bf16 path's result on the dequantised window, bit for bit
    g = np.random.default_rng(31)
    ring = _e8m0_ring(g, 1)
    e4 = np.array([oracle.e4m3_value(c) for c in range(256)])
    deq = e4[ring[..., :512]] * np.exp2(ring[..., 512:].astype(np.float64) - 127).repeat(32, axis=-1)
    ring_bf = bf16(deq)
    assert np.array_equal(bf16_np(ring_bf), deq)
    plane = bf16(RNG.standard_normal((20, 512)))
    q = bf16(RNG.standard_normal((2, 64, 512)))
    sel = np.array([[3, 0, 19, -1], [5, -1, 11, 2]], dtype=np.int32)
    sink = RNG.standard_normal(64).astype(np.float32)
    a, la = oracle.sparse_attn(q, [0, 0], [300, 40], ring_bf, plane, [0], sel, sink)
    b, lb = oracle.sparse_attn(q, [0, 0], [300, 40], torch.from_numpy(ring), plane, [0], sel,
                               sink, swa_e8m0=True)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_mxfp4_index_plane_layout_scales_and_codes():
    n = 13  # a partial second block
    x = RNG.standard_normal((n, 128)) * np.exp2(RNG.integers(-10, 10, (n, 4)).repeat(32, axis=1))
    x[5, 32:64] = 0.0
    K = bf16(x)
    Kd = bf16_np(K)
    pl = oracle.index_plane_fp4(K)
    assert pl.size == 2 * oracle.FP4_INDEX_BLOCK_BYTES
    blocks = pl.reshape(2, 544)
    for r in range(16):
        codes_b = blocks[r // 8, (r % 8) * 64:(r % 8) * 64 + 64]
        sc = blocks[r // 8, 512 + (r % 8) * 4:512 + (r % 8) * 4 + 4]
        if r >= n:
            assert np.all(codes_b == 0) and np.all(sc == 127)
            continue
        codes = np.empty(128, dtype=np.int64)
        codes[0::2], codes[1::2] = codes_b & 15, codes_b >> 4
        for j in range(4):
            amax = np.abs(Kd[r, 32 * j:32 * j + 32]).max()
            e = int(sc[j])
            if amax == 0:
                assert e == 127 and np.all(codes[32 * j:32 * j + 32] == 0)
                continue
            s = 2.0 ** (e - 127)
            assert amax <= 6 * s and amax > 3 * s  # the smallest power of two that fits
            for i in range(32):
                d = 32 * j + i
                assert codes[d] == _e2m1_nearest_even(Kd[r, d] / s)


def test_mxfp4_scores_equal_bf16_scores_when_lossless():
    # rows whose every group holds E2M1 values times one power of two, with 6 * 2^k in
    # the group (which fixes the scale), are quantised losslessly: FULL and REINDEX over
    # two sequences must give the bf16 scorer's scores
    g = np.random.default_rng(41)
    mags = np.array(E2M1[1:])
    v = g.choice(mags, (64, 128)) * g.choice([-1.0, 1.0], (64, 128))
    v[:, ::32] = 6.0
    K = bf16(v * np.exp2(g.integers(-6, 6, (64, 4))).repeat(32, axis=1))
    iq = bf16(g.standard_normal((3, 64, 128)))
    w = g.standard_normal((3, 64)).astype(np.float32)
    rb = np.array([0, 32], dtype=np.int64)
    plane = oracle.index_plane_fp4(K)
    pos, seqs = [60, 31, 17], [0, 1, 1]
    a, ra = oracle.index_scores(iq, w, K, rb, seqs, pos, 1)
    b, rb4 = oracle.index_scores_fp4(iq, w, plane, rb, seqs, pos, 1)
    assert np.array_equal(ra, rb4)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-12)
    cand = np.array([[0, 3, 7, -1], [1, 2, -1, -1], [0, 2, 3, 1]], dtype=np.int32)
    a, ra = oracle.index_scores(iq, w, K, rb, seqs, pos, 1, cand=cand)
    b, rb4 = oracle.index_scores_fp4(iq, w, plane, rb, seqs, pos, 1, cand=cand)
    assert np.array_equal(ra, rb4)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-12)


# ---- FP8 index plane --------------------------------------------------------

def _e4m3_values():
    return np.array([oracle.e4m3_value(c) for c in range(0x7F)])  # +0 .. 448


def test_e4m3_encode_matches_torch_float8_and_ties_to_even():
    vals = _e4m3_values()
    mids = (vals[:-1] + vals[1:]) / 2  # exact in fp32: at most 5 significant bits
    rnd = RNG.uniform(-448, 448, 20000) * np.exp2(RNG.integers(-12, 1, 20000))
    x = np.concatenate([vals, -vals, mids, -mids, rnd]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_code(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # every finite code round-trips; beyond 448 saturates (no infinity in the format)
    assert all(oracle.e4m3_code(oracle.e4m3_value(c)) == c for c in range(0x7F))
    assert oracle.e4m3_code(470.0) == 0x7E and oracle.e4m3_code(-1e6) == 0xFE
    # a tie between 1.0 (mantissa 0) and 1.125 (mantissa 1) goes to the even mantissa
    assert oracle.e4m3_code(1.0625) == 0x38 and oracle.e4m3_code(1.1875) == 0x3A


def test_ue8m0_scale_is_the_smallest_power_of_two_that_fits():
    for amax in np.concatenate([RNG.uniform(0, 1, 200) * np.exp2(RNG.integers(-40, 40, 200)),
                                [448.0, 449.0, 1.0, 2.0 ** -30, 448 * 2.0 ** -5]]):
        s = oracle.ue8m0_scale(amax)
        m, e = math.frexp(s)
        assert m == 0.5  # a power of two
        assert amax / s <= 448.0 < amax / (s / 2)
    assert oracle.ue8m0_scale(448.0) == 1.0 and oracle.ue8m0_scale(448.0 * 2 ** -7) == 2 ** -7
    assert oracle.ue8m0_scale(0.0) == 1.0


def test_fp8_plane_layout_and_quantisation_error():
    n = 21  # two full blocks and a partial third
    x = RNG.standard_normal((n, 128)) * np.exp2(RNG.integers(-6, 6, (n, 1)))
    K = bf16(x)
    Kd = bf16_np(K)
    plane = oracle.index_plane_fp8(K)
    assert plane.size == 3 * oracle.FP8_BLOCK_BYTES
    blocks = plane.reshape(3, oracle.FP8_BLOCK_BYTES)
    codes = blocks[:, :1024].reshape(24, 128)
    scales = blocks[:, 1024:].copy().view(np.float32).reshape(24).astype(np.float64)
    # rows past n: zero codes, scale 1
    assert np.all(codes[n:] == 0) and np.all(scales[n:] == 1.0)
    vals = _e4m3_values()
    for r in range(n):
        amax = np.abs(Kd[r]).max()
        assert 224.0 < amax / scales[r] <= 448.0  # the row's largest value uses the top octave
        deq = np.array([oracle.e4m3_value(c) for c in codes[r]]) * scales[r]
        # nearest E4M3 value: relative error <= 2^-4 in the normal range, absolute
        # <= 2^-10 * scale in the subnormal one
        err = np.abs(deq - Kd[r])
        bound = np.maximum(np.abs(Kd[r]) * 2.0 ** -4, 2.0 ** -10 * scales[r])
        assert np.all(err <= bound * (1 + 1e-12))
        # and it is the nearest one: no other code is closer
        cand = np.abs(vals[None, :] * scales[r] - np.abs(Kd[r])[:, None]).min(1)
        np.testing.assert_allclose(err, cand, rtol=0, atol=1e-300)


def _lossless_fp8_rows(rows, H=None):
    """bf16 rows that the FP8 quantiser represents exactly: every value is an E4M3
    normal value times 2^k, and each row holds 448 * 2^k, which fixes its scale."""
    vals = _e4m3_values()
    normal = vals[(vals >= 2.0 ** -6)]
    shape = (rows, 128) if H is None else (rows, H, 128)
    v = RNG.choice(normal, size=shape) * RNG.choice([-1.0, 1.0], size=shape)
    k = RNG.integers(-8, 4, size=shape[:-1] + (1,))
    v[..., 5] = 448.0
    return bf16(v * np.exp2(k))


def test_fp8_scores_equal_bf16_scores_when_quantisation_is_lossless():
    # two sequences (row_base 0 and 64), FULL and REINDEX: the FP8 path (its own loops,
    # codes and scales) must give the bf16 path's scores when nothing is lost
    K = _lossless_fp8_rows(128)
    iq = _lossless_fp8_rows(3, H=64)
    w = RNG.standard_normal((3, 64)).astype(np.float32)
    rb = np.array([0, 64], dtype=np.int64)
    plane = oracle.index_plane_fp8(K)
    pos = [120, 63, 37]
    seqs = [0, 1, 1]
    for ratio in (1, 2):
        a, ra = oracle.index_scores(iq, w, K, rb, seqs, pos, ratio)
        b, rb8 = oracle.index_scores_fp8(iq, w, plane, rb, seqs, pos, ratio)
        assert np.array_equal(ra, rb8)
        np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-12)
    cand = np.array([[0, 5, 14, -1], [7, 2, -1, -1], [1, 3, 4, 0]], dtype=np.int32)
    a, ra = oracle.index_scores(iq, w, K, rb, seqs, pos, 1, cand=cand)
    b, rb8 = oracle.index_scores_fp8(iq, w, plane, rb, seqs, pos, 1, cand=cand)
    assert np.array_equal(ra, rb8)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-12)


def test_fp8_scores_stay_within_the_quantisation_error_of_bf16():
    iq, K, w, rb = make_index_case(Q=2, H=64, rows=160, seq=1)
    plane = oracle.index_plane_fp8(K)
    a, _ = oracle.index_scores(iq, w, K, rb, [0, 0], [159, 100], 1, relu=False)
    b, _ = oracle.index_scores_fp8(iq, w, plane, rb, [0, 0], [159, 100], 1, relu=False)
    # each factor is within 2^-4 relative (plus subnormal flushes): the sum of |terms|
    # bounds the error
    Kd, qd = bf16_np(K), bf16_np(iq)
    alpha = 1.0 / math.sqrt(128 * 64)
    for q, nv in ((0, 160), (1, 101)):
        mag = alpha * (np.abs(w[q]).astype(np.float64)[:, None, None]
                       * np.abs(qd[q])[:, None, :] * np.abs(Kd[:nv])[None, :, :]).sum((0, 2))
        assert np.all(np.abs(b[q, :nv] - a[q, :nv]) <= 0.14 * mag + 1e-9)
        assert np.corrcoef(a[q, :nv], b[q, :nv])[0, 1] > 0.99


# ---- top-k --------------------------------------------------------------------------

def brute_topk(scores, rows, k):
    valid = [(s if not math.isnan(s) else -math.inf, r) for s, r in zip(scores, rows) if r >= 0]
    best = []
    for _ in range(min(k, len(valid))):  # O(n k): repeatedly take the best remaining
        i = max(range(len(valid)), key=lambda t: (valid[t][0], -valid[t][1]))
        best.append(valid.pop(i)[1])
    best.sort()
    return best + [-1] * (k - len(best))


def test_topk_brute_force_with_ties_and_nan():
    for trial in range(300):
        n = int(RNG.integers(1, 64))
        k = int(RNG.integers(1, 70))
        scores = RNG.integers(-3, 4, n).astype(np.float64)  # many ties
        if trial % 3 == 0:
            scores[RNG.integers(0, n, 3)] = np.nan
        if trial % 5 == 0:
            scores[RNG.integers(0, n, 2)] = -np.inf
        rows = RNG.permutation(1000)[:n].astype(np.int64)
        rows[RNG.random(n) < 0.1] = -1
        got = oracle.topk(scores, rows, k)
        assert got.tolist() == brute_topk(scores, rows, k)


def test_topk_float32_ties_exact_and_negative_zero():
    s = np.array([0.0, -0.0, 1.5, 1.5, -1.0, 1.5], dtype=np.float32).astype(np.float64)
    got = oracle.topk(s, np.arange(6), 4)
    assert got.tolist() == [0, 2, 3, 5]  # -0.0 == 0.0, lower row wins the tie


# ---- sparse attention ---------------------------------------------------------------

def dense_attention(qd, X, scale, sink=None):
    """Textbook softmax attention for one query: qd [64,512], X [n,512]."""
    S = (qd @ X.T) * scale
    if sink is None:
        P = np.exp(S - S.max(1, keepdims=True))
        return (P / P.sum(1, keepdims=True)) @ X
    mx = np.maximum(S.max(1), sink)
    P = np.exp(S - mx[:, None])
    Z = P.sum(1) + np.exp(sink - mx)
    return (P @ X) / Z[:, None]


def attn_case(p, nsel_valid, B=1, nrows=700, seed=0):
    g = np.random.default_rng(seed)
    q = bf16(g.standard_normal((1, 64, 512)))
    ring = bf16(g.standard_normal((B, 128, 512)))
    plane = bf16(g.standard_normal((nrows, 512)))
    sel = np.full((1, 512), -1, dtype=np.int32)
    sel[0, :nsel_valid] = np.sort(g.permutation(nrows)[:nsel_valid])
    sink = g.standard_normal(64).astype(np.float32)
    return q, ring, plane, sel, sink


def window_rows(ring, p, b=0):
    lo = max(0, p - 127)
    return np.stack([bf16_np(ring[b, pos % 128]) for pos in range(lo, p + 1)])


def test_attention_no_sink_all_rows_is_dense_softmax():
    for p, ns in ((4095, 512), (5, 40), (130, 0)):
        q, ring, plane, sel, _ = attn_case(p, ns)
        out, _ = oracle.sparse_attn(q, [0], [p], ring, plane, [0], sel, None)
        X = window_rows(ring, p)
        if ns:
            X = np.concatenate([X, bf16_np(plane)[sel[0, :ns]]])
        ref = dense_attention(bf16_np(q)[0], X, 512 ** -0.5)
        np.testing.assert_allclose(out[0], ref, rtol=1e-10, atol=1e-12)


def test_attention_sink_closed_form_and_lse():
    p, ns = 1000, 300
    q, ring, plane, sel, sink = attn_case(p, ns, seed=3)
    out0, lse0 = oracle.sparse_attn(q, [0], [p], ring, plane, [0], sel, None)
    out1, lse1 = oracle.sparse_attn(q, [0], [p], ring, plane, [0], sel, sink)
    Z = np.exp(lse0[0])  # sum_j e^{s_j}
    factor = Z / (Z + np.exp(sink.astype(np.float64)))
    np.testing.assert_allclose(out1[0], out0[0] * factor[:, None], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(np.exp(lse1[0]), Z + np.exp(sink.astype(np.float64)), rtol=1e-10)
    # a very negative sink is the no-sink case
    out2, _ = oracle.sparse_attn(q, [0], [p], ring, plane, [0], sel, np.full(64, -1e4, np.float32))
    np.testing.assert_allclose(out2, out0, rtol=1e-12, atol=1e-14)


def test_attention_duplicate_entry_counts_twice():
    # A plane row equal to a window row is a second entry, not merged: the pair acts
    # as one entry whose logit is larger by ln 2.
    p = 300
    q, ring, plane, sel, sink = attn_case(p, 10, seed=5)
    plane = plane.clone()
    plane[sel[0, 0]] = ring[0, p % 128]  # duplicate of the current position's window row
    out, _ = oracle.sparse_attn(q, [0], [p], ring, plane, [0], sel, sink)
    X = window_rows(ring, p)
    Y = bf16_np(plane)[sel[0, 1:10]]
    qd = bf16_np(q)[0]
    S = np.concatenate([X, Y]) @ qd.T * 512 ** -0.5  # [n, 64]
    dup = X.shape[0] - 1  # the window row of position p is the last window entry
    S[dup] += math.log(2.0)
    mx = np.maximum(S.max(0), sink)
    P = np.exp(S - mx)
    Z = P.sum(0) + np.exp(sink - mx)
    ref = (P.T @ np.concatenate([X, Y])) / Z[:, None]
    np.testing.assert_allclose(out[0], ref, rtol=1e-10, atol=1e-13)


def test_attention_entry_cap_and_ragged_window():
    # 128 window + 512 selected = 640 entries at most; an early position sees p+1 slots.
    q, ring, plane, sel, _ = attn_case(4095, 512, seed=7)
    X = np.concatenate([window_rows(ring, 4095), bf16_np(plane)[sel[0]]])
    assert X.shape[0] == 640
    q, ring, plane, sel, _ = attn_case(9, 3, seed=8)
    # slots beyond position 9 hold junk that must not be read
    ring2 = ring.clone()
    ring2[0, 10:] = bf16(np.full((118, 512), 1e3))
    a, _ = oracle.sparse_attn(q, [0], [9], ring, plane, [0], sel, None)
    b, _ = oracle.sparse_attn(q, [0], [9], ring2, plane, [0], sel, None)
    assert np.array_equal(a, b)


def test_attention_linear_window_equals_ring():
    p = 500
    q, ring, plane, sel, sink = attn_case(p, 64, seed=9)
    lo = p - 127
    lin = torch.stack([ring[0, pos % 128] for pos in range(lo, p + 1)])
    a, la = oracle.sparse_attn(q, [0], [p], ring, plane, [0], sel, sink)
    b, lb = oracle.sparse_attn(q, [0], [p], lin, plane, [0], sel, sink, swa_mode="linear",
                               lin_base=[0], lin_pos0=[lo])
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_attention_fp8_ring_dequant_matches_torch_float8():
    p = 200
    g = np.random.default_rng(11)
    q = bf16(g.standard_normal((1, 64, 512)))
    codes = g.integers(0, 256, (1, 128, 512)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    scales = g.uniform(0.01, 0.02, (1, 128, 4)).astype(np.float32)
    ring8 = np.concatenate([codes, scales.view(np.uint8).reshape(1, 128, 16)], axis=2)
    plane = bf16(g.standard_normal((10, 512)))
    sel = np.full((1, 512), -1, dtype=np.int32)
    sel[0, :4] = [1, 3, 5, 7]
    out, _ = oracle.sparse_attn(q, [0], [p], torch.from_numpy(ring8), plane, [0], sel, None)
    deq = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    deq = deq * np.repeat(scales.astype(np.float64), 128, axis=2)
    X = np.stack([deq[0, pos % 128] for pos in range(p - 127, p + 1)])
    X = np.concatenate([X, bf16_np(plane)[[1, 3, 5, 7]]])
    ref = dense_attention(bf16_np(q)[0], X, 512 ** -0.5)
    np.testing.assert_allclose(out[0], ref, rtol=1e-10, atol=1e-13)


# ---- generator ----------------------------------------------------------------------

def test_synth_normal_moments_and_determinism():
    import synth
    x = synth.normal_f32(1 << 20, 7, 3).numpy().astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    y = synth.normal_f32(1 << 20, 7, 3).numpy().astype(np.float64)
    assert np.array_equal(x, y)
    z = synth.normal_f32(16, 7, 3, offset=100).numpy()
    assert np.array_equal(z, x[100:116].astype(np.float32))


def test_synth_e4m3_encode_matches_torch():
    import synth
    r = synth.rows_fp8s128(0, 0, 64, 5, 9)
    codes = r[:, :512].contiguous()
    vals = synth.rows_f32(0, 0, 64, 512, 5, 9) * 64.0
    ref = vals.to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(codes, ref)
    sc = r[:, 512:].contiguous().view(torch.float32)
    assert float(sc.min()) >= 0.75 / 64 and float(sc.max()) < 1.25 / 64


# ---- candidate pool (second stage of the FULL layer) ---------------------------------------

def _pool_brute(scores, nvis, nbk):
    """Every block's score by a scan, then all blocks ranked by sorting tuples."""
    nb = (nvis + 7) // 8
    best = []
    for b in range(nb):
        m = -math.inf
        for r in range(8 * b, min(8 * b + 8, nvis)):
            v = scores[r]
            v = -math.inf if math.isnan(v) else (np.finfo(np.float64).max if v == math.inf else v)
            m = max(m, v)
        best.append(math.inf if b == nb - 1 else m)
    order = sorted(range(nb), key=lambda b: (-best[b], b))[:nbk]
    return sorted(order) + [-1] * (nbk - min(nbk, nb))


def test_candidate_pool_brute_force_with_partial_block_ties_nan_and_inf():
    g = np.random.default_rng(7)
    for trial in range(60):
        nvis = int(g.integers(1, 90))
        nbk = int(g.integers(1, 14))
        sc = g.integers(-3, 4, nvis).astype(np.float64)  # heavy ties
        sc[g.random(nvis) < 0.1] = np.nan
        sc[g.random(nvis) < 0.05] = np.inf
        sc[g.random(nvis) < 0.05] = -np.inf
        ld = nvis + int(g.integers(0, 9))  # unscored tail
        scores = np.zeros(ld)
        scores[:nvis] = sc
        rows = np.full(ld, -1, dtype=np.int64)
        rows[:nvis] = np.arange(nvis)
        got = oracle.candidate_pool(scores, rows, nbk)
        assert list(got) == _pool_brute(list(sc), nvis, nbk), trial


def test_candidate_pool_keeps_the_newest_block_and_covers_the_row_top_k():
    g = np.random.default_rng(8)
    nvis, k, nbk = 3001, 64, 72  # the newest block holds 1 row
    sc = g.standard_normal(nvis)
    sc[-1] = -np.inf  # the newest row scores lowest: its block is kept all the same
    rows = np.arange(nvis, dtype=np.int64)
    pool = oracle.candidate_pool(sc, rows, nbk)
    assert (nvis - 1) // 8 in pool
    # every row of the FULL layer's own top-k lies in a selected block
    top = oracle.topk(sc, rows, k)
    assert set(int(r) // 8 for r in top if r >= 0) <= set(int(b) for b in pool if b >= 0)
    # the order of rows inside a block does not matter
    perm = np.arange(nvis)
    for b in range(0, nvis // 8):
        perm[8 * b:8 * b + 8] = g.permutation(perm[8 * b:8 * b + 8])
    assert np.array_equal(oracle.candidate_pool(sc[perm], rows, nbk), pool)
    # fewer blocks than places: every block, then -1
    small = oracle.candidate_pool(sc[:40], rows[:40], nbk)
    assert list(small[:5]) == [0, 1, 2, 3, 4] and (small[5:] == -1).all()
