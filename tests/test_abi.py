"""The C-ABI library loads, exports every symbol include/csa2.h declares, and rejects
invalid arguments on the host before touching the GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import csa2_compressed_sparse_gb300 as csa2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z_]+)\s*\(", text)))


def test_header_declares_the_step():
    names = declared_functions()
    for n in ("csa2_compress", "csa2_index_topk", "csa2_sparse_attn", "csa2_reuse_attn",
              "csa2_topk_scores", "csa2_device_status", "csa2_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = csa2.lib()
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in csa2.h but not exported"


def test_version_string():
    assert "sm_103a" in csa2.csa2_version()


def _raw():
    return csa2.lib()


def test_compress_rejects_bad_ratio_and_batch():
    L = _raw()
    one = ctypes.c_void_p(16)
    st = L.csa2_compress(one, one, 4, one, 1, one, 3, one, one, one, 10, one, None, 1e-6, one, None)
    assert st == 1 and b"ratio" in L.csa2_last_error()
    st = L.csa2_compress(one, one, 4, one, 0, one, 2, one, one, one, 10, one, None, 1e-6, one, None)
    assert st == 1 and b"B must" in L.csa2_last_error()
    st = L.csa2_compress(one, None, 4, one, 1, one, 2, one, one, one, 10, one, None, 1e-6, one, None)
    assert st == 1 and b"ratio 2" in L.csa2_last_error()
    st = L.csa2_compress(ctypes.c_void_p(18), one, 4, one, 1, one, 1, one, one, one, 10, one, None,
                         1e-6, one, None)
    assert st == 1 and b"aligned" in L.csa2_last_error()
    # nothing to do is not an error
    assert L.csa2_compress(None, None, 0, None, 1, None, 2, None, None, None, 0, None, None,
                           1e-6, None, None) == 0


def test_index_topk_rejects_bad_arguments():
    L = _raw()
    p = ctypes.c_void_p(256)
    args = dict(iq=p, w=p, Q=4, H=64, index_k=p, index_rows=1000, row_base=p, q_seq=p, q_pos=p,
                ratio=2, cand=None, ncb=0, k=512, relu=1, max_scored=2048, sel=p, sel_scores=None,
                scores_out=None, ws=p, ws_bytes=1 << 30, stream=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.csa2_index_topk(*a.values()), L.csa2_last_error()

    st, msg = call(H=48)
    assert st == 1 and b"H must" in msg
    st, msg = call(k=513)
    assert st == 1 and b"k must" in msg
    st, msg = call(ratio=4)
    assert st == 1 and b"ratio" in msg
    # a candidate pool that cannot hold the top-k is refused (2048 x 8 >= 512 rule)
    st, msg = call(cand=p, ncb=63, max_scored=63 * 8)
    assert st == 1 and b"cannot hold" in msg
    st, msg = call(cand=p, ncb=64, max_scored=1000)
    assert st == 1 and b"max_scored" in msg
    st, msg = call(ws_bytes=16)
    assert st == 5 and b"workspace" in msg
    st, msg = call(ws=ctypes.c_void_p(300))
    assert st == 1 and b"256-byte" in msg
    st, msg = call(max_scored=1 << 26)
    assert st == 1 and b"exceeds" in msg


def test_workspace_sizes_are_monotone():
    a = csa2.csa2_index_topk_workspace_size(64, 64, 32768, 512)
    b = csa2.csa2_index_topk_workspace_size(64, 64, 65536, 512)
    assert 0 < a < b
    assert a >= 64 * 32768 * 4
    assert csa2.csa2_topk_workspace_size(8, 32768, 512) == 0  # one chunk: no scratch
    assert csa2.csa2_topk_workspace_size(8, 1 << 20, 512) >= 8 * 32 * 512 * 8


def test_row_selection_chunking():
    """Rows of up to 65536 positions are selected by one CTA each (no merge scratch); longer
    rows are cut into chunks of 32768 whose k-best lists the last chunk CTA merges."""
    assert csa2.csa2_topk_workspace_size(8, 40000, 512) == 0
    assert csa2.csa2_topk_workspace_size(8, 65536, 2048) == 0
    nb = csa2.csa2_topk_workspace_size(8, 65537, 512)
    assert nb >= 8 * 3 * 512 * 8  # three chunks of partial (key, position) lists
    # the merge holds chunks x k <= 32768 pairs, and rows hold at most 48 chunks
    assert csa2.csa2_topk_workspace_size(8, 48 * 32768, 682) > 0  # 32736 pairs
    assert csa2.csa2_topk_workspace_size(8, 48 * 32768, 683) == 0  # 32784 pairs
    assert csa2.csa2_topk_workspace_size(8, 48 * 32768 + 1, 1) == 0
    # the indexer's workspace holds the keys; a one-CTA row adds no partial lists
    a = csa2.csa2_index_topk_workspace_size(64, 64, 65536, 512)
    b = csa2.csa2_index_topk_workspace_size(64, 64, 65537, 512)
    assert b - a >= 64 * 3 * 512 * 8


def test_attn_rejects_bad_arguments():
    L = _raw()
    p = ctypes.c_void_p(256)
    sw = csa2._SwaC(0, 0, 256, 512, None, None)
    st = L.csa2_sparse_attn(p, 2, p, p, ctypes.byref(sw), p, 100, p, p, 513, None, 0.04, p, None,
                            None, 0, None)
    assert st == 1 and b"nsel" in L.csa2_last_error()
    bad = csa2._SwaC(1, 0, 256, 512, None, None)  # LINEAR without lin_base/lin_pos0
    st = L.csa2_reuse_attn(p, 2, p, p, ctypes.byref(bad), p, 100, p, p, 512, None, 0.04, p, None,
                           None, 0, None)
    assert st == 1 and b"LINEAR" in L.csa2_last_error()
    st = L.csa2_sparse_attn(p, 2, p, p, ctypes.byref(sw), p, 100, p, p, 512, None,
                            float("nan"), p, None, None, 0, None)
    assert st == 1 and b"scale" in L.csa2_last_error()


def test_index_topk_pool_rejects_bad_arguments():
    L = _raw()
    p = ctypes.c_void_p(256)
    args = dict(iq=p, w=p, Q=4, H=64, index_k=p, index_rows=1000, row_base=p, q_seq=p, q_pos=p,
                ratio=2, k=512, relu=1, max_scored=20000, sel=p, sel_scores=None,
                scores_out=None, nbk=2048, pool=p, ws=p, ws_bytes=1 << 30, stream=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.csa2_index_topk_pool(*a.values()), L.csa2_last_error()

    for nbk in (0, 2049):
        st, msg = call(nbk=nbk)
        assert st == 1 and b"nbk" in msg
    st, msg = call(pool=None)
    assert st == 1 and b"pool" in msg
    st, msg = call(k=513)
    assert st == 1 and b"k must" in msg
    need = csa2.csa2_index_topk_pool_workspace_size(4, 64, 20000, 512, 2048)
    st, msg = call(ws_bytes=need - 1)
    assert st == 5 and b"workspace" in msg


def test_pool_workspace_holds_the_block_merge():
    base = csa2.csa2_index_topk_workspace_size(64, 64, 16384, 512)
    pool = csa2.csa2_index_topk_pool_workspace_size(64, 64, 16384, 512, 2048)
    assert pool >= base + 64 * 4  # the block selection's arrival counters
    # 2^20 rows: 131072 blocks in 4 chunks, whose 2048-block lists are merged
    big = csa2.csa2_index_topk_pool_workspace_size(8, 64, 1 << 20, 512, 2048)
    assert big >= csa2.csa2_index_topk_workspace_size(8, 64, 1 << 20, 512) + 8 * 4 * 2048 * 8
    assert csa2.csa2_index_topk_pool_workspace_size(8, 64, 1 << 20, 512, 2049) == 0


def test_topk_scores_k_limits():
    L = _raw()
    p = ctypes.c_void_p(256)
    st = L.csa2_topk_scores(p, p, 4, 1000, 2049, p, None, None, 0, None)
    assert st == 1 and b"k must" in L.csa2_last_error()
    # 32 chunks x 2048 pairs do not fit the merge
    st = L.csa2_topk_scores(p, p, 4, 1 << 20, 2048, p, None, p, 1 << 30, None)
    assert st == 1 and b"merge" in L.csa2_last_error()
    assert csa2.csa2_topk_workspace_size(4, 1 << 20, 2048) == 0
    assert csa2.csa2_topk_workspace_size(4, 1 << 17, 2048) >= 4 * 4 * 2048 * 8


def test_block_plane_entry_points_reject_bad_arguments():
    L = _raw()
    p = ctypes.c_void_p(256)
    for name in ("csa2_index_topk_fp8", "csa2_index_topk_fp4"):
        fn = getattr(L, name)
        args = dict(iq=p, w=p, Q=4, H=64, plane=p, index_rows=1000, row_base=p, q_seq=p, q_pos=p,
                    ratio=2, cand=None, ncb=0, k=512, relu=1, max_scored=2048, sel=p,
                    sel_scores=None, scores_out=None, ws=p, ws_bytes=1 << 30, stream=None)

        def call(**kw):
            a = dict(args)
            a.update(kw)
            return fn(*a.values()), L.csa2_last_error()

        st, msg = call(plane=None)
        assert st == 1 and b"plane is required" in msg, name
        st, msg = call(plane=ctypes.c_void_p(264))
        assert st == 1 and b"aligned" in msg, name
        st, msg = call(H=16)
        assert st == 1 and b"H must" in msg, name
        st, msg = call(ws_bytes=64)
        assert st == 5 and b"workspace" in msg, name
        # nothing to do is not an error
        assert call(Q=0, plane=None)[0] == 0, name
    for name in ("csa2_index_plane_fp8", "csa2_index_plane_fp4"):
        fn = getattr(L, name)
        assert fn(p, 0, p, None) == 0, name  # no rows
        assert fn(None, 10, p, None) == 1, name
        assert fn(ctypes.c_void_p(258), 10, p, None) == 1 and b"aligned" in L.csa2_last_error()
        assert fn(p, -1, p, None) == 1, name


def test_block_plane_sizes():
    assert csa2.csa2_index_plane_fp8_bytes(0) == 0
    assert csa2.csa2_index_plane_fp8_bytes(1) == 1056
    assert csa2.csa2_index_plane_fp8_bytes(17) == 3 * 1056
    assert csa2.csa2_index_plane_fp4_bytes(0) == 0
    assert csa2.csa2_index_plane_fp4_bytes(8) == 544
    assert csa2.csa2_index_plane_fp4_bytes(9) == 2 * 544
    # the FP4 indexer needs no query codes: its workspace is the bf16 indexer's
    assert (csa2.csa2_index_topk_fp4_workspace_size(64, 64, 32768, 512) ==
            csa2.csa2_index_topk_workspace_size(64, 64, 32768, 512))
    assert (csa2.csa2_index_topk_fp8_workspace_size(64, 64, 32768, 512) >
            csa2.csa2_index_topk_workspace_size(64, 64, 32768, 512))
    for f in (csa2.csa2_index_topk_fp4_workspace_size, csa2.csa2_index_topk_fp8_workspace_size):
        assert f(4, 48, 1024, 512) == 0 and f(4, 64, 1024, 513) == 0


def test_binding_has_every_declared_function():
    # the Python binding mirrors the C ABI name for name
    missing = [n for n in declared_functions() if not hasattr(csa2, n)]
    assert not missing, f"declared in csa2.h without a binding: {missing}"
    assert all(n in csa2.__all__ for n in declared_functions())


def test_last_error_text_after_a_rejected_call():
    L = _raw()
    one = ctypes.c_void_p(16)
    assert L.csa2_compress(one, one, 4, one, 1, one, 3, one, one, one, 10, one, None, 1e-6,
                           one, None) == 1
    assert "ratio" in csa2.csa2_last_error()
