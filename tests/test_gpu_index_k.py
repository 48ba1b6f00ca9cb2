"""Index K production in the compressor (csa2_compress_index) through the C ABI: the main
plane is bit-identical to csa2_compress's, and every index row matches the oracle's
(latent before RoPE as bf16 -> wk -> RMSNorm over 128 -> RoPE on the last 64 dims).

Tolerance of an index value: one bf16 ulp of the oracle's double value plus 2^-10 of the
row's largest magnitude.  The GPU computes the latent in fp32 and the oracle in double, so
a latent value near a bf16 rounding boundary can round to the neighbouring bf16 value on
one side (about one element in 10^4); one such element moves each output by at most
|wk[o][d]| * 2^-8 |x[d]|, which against outputs that sum 512 such terms stays below
2^-10 of the row's largest value, and the final bf16 rounding adds the ulp.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _weights(seed):
    g = np.random.default_rng(seed)
    wk = torch.from_numpy((g.standard_normal((128, 512)) / np.sqrt(512)).astype(np.float32))
    kw = (1.0 + 0.25 * g.standard_normal(128)).astype(np.float32)
    return wk.bfloat16(), kw


def _case(ratio, lens_a, lens_b, seed=21):
    from csa2_compressed_sparse_gb300 import (csa2_compress, csa2_compress_index,
                                              csa2_device_status)
    B = len(lens_a)
    tot = [a + b for a, b in zip(lens_a, lens_b)]
    nrows = [t // ratio for t in tot]
    rb = np.concatenate([[0], np.cumsum(nrows)[:-1]]).astype(np.int64)
    R = max(sum(nrows), 1)
    wk, kw = _weights(seed)
    wk_d, kw_d = wk.cuda(), torch.from_numpy(kw).cuda()
    invf = torch.from_numpy(W.rope_inv_freq()).cuda()
    planes, index = [], torch.full((R, 128), -1.0, dtype=torch.bfloat16, device="cuda")
    for with_index in (True, False):
        plane = torch.zeros((R, 512), dtype=torch.bfloat16, device="cuda")
        ks = torch.zeros((B, 2, 512), dtype=torch.float32, device="cuda")
        ss = torch.zeros((B, 2, 512), dtype=torch.float32, device="cuda")
        for start_of, lens in ((lambda b: 0, lens_a), (lambda b: lens_a[b], lens_b)):
            cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
            kv = torch.cat([synth.rows_bf16(b, start_of(b), lens[b], 512, seed, synth.KV)
                            for b in range(B)]).cuda()
            sc = torch.cat([synth.rows_bf16(b, start_of(b), lens[b], 512, seed, synth.SCORE)
                            for b in range(B)]).cuda()
            sp = torch.tensor([start_of(b) for b in range(B)], dtype=torch.int64, device="cuda")
            rbd = torch.from_numpy(rb).cuda()
            if with_index:
                csa2_compress_index(kv, sc, cu, sp, ratio, ks, ss, plane, rbd, invf, wk_d, index,
                                    knorm_w=kw_d)
            else:
                csa2_compress(kv, sc, cu, sp, ratio, ks, ss, plane, rbd, invf)
        csa2_device_status()
        planes.append(plane)
    assert torch.equal(planes[0].view(torch.int16), planes[1].view(torch.int16))
    got = index.double().cpu().numpy()
    worst = 0.0
    for b in range(B):
        if nrows[b] == 0:
            continue
        kv = synth.rows_bf16(b, 0, tot[b], 512, seed, synth.KV)
        sc = synth.rows_bf16(b, 0, tot[b], 512, seed, synth.SCORE)
        ref = np.zeros((nrows[b], 512), dtype=np.uint16)
        ip = np.zeros((nrows[b], 128), dtype=np.uint16)
        oks, oss = np.zeros((1, ratio, 512)), np.zeros((1, ratio, 512))
        n, _, kf = oracle.compress_index(kv, sc, [0, tot[b]], [0], ratio, oks, oss, ref, ip, [0],
                                         W.rope_inv_freq(), wk, knorm_w=kw)
        assert n == nrows[b]
        g = got[rb[b]:rb[b] + nrows[b]]
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(kf), 1e-30))) - 7)
        tol = ulp + 2.0 ** -10 * np.abs(kf).max(axis=1, keepdims=True)
        err = np.abs(g - kf)
        assert np.all(err <= tol), f"seq {b}: worst {float((err / tol).max()):.3g} x tol"
        worst = max(worst, float((err / tol).max()))
        # most values are the oracle's own bf16 rounding
        assert np.mean(oracle.bf16_bits(torch.from_numpy(g).bfloat16()) == ip) > 0.98
    return worst


@pytest.mark.parametrize("ratio", [1, 2])
def test_index_k_in_the_compressor_matches_the_oracle(ratio):
    w = _case(ratio, [37, 50, 1, 0, 129], [63, 1, 1, 8, 0])
    print(f"\nratio {ratio}: worst index-K error {w:.3g} x tolerance")


def test_index_k_decode_batch_one_token_each():
    # one new token per sequence after histories of odd and even lengths (m = 2): rows
    # close only where the new token ends a group
    _case(2, [4095, 1000, 17, 2], [1, 1, 1, 1], seed=22)
