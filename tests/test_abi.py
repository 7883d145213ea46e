"""The C-ABI library loads and exports every function include/*.h declares;
host-side argument checks return their status codes without touching a
device (no compute calls here)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from serving_sparse_mla_gb300 import binding, build
    build.build()
    return binding.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b((?:sparse_mla|dsa)_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "sparse_mla_fwd" in names and "sparse_mla_decode" in names and "sparse_mla_fwd_varlen" in names
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_header():
    from serving_sparse_mla_gb300 import binding
    assert set(declared_functions()) <= set(binding.SIGNATURES)


def test_status_strings(lib):
    for code in range(7):
        s = lib.sparse_mla_status_string(code).decode()
        assert s.startswith("SPARSE_MLA_")
    assert lib.sparse_mla_status_string(99).decode() == "SPARSE_MLA_UNKNOWN_STATUS"


def _fwd(lib, **kw):
    a = dict(q=16, kv=16, idx=16, scale=0.1, out=16, lse=16, s_q=4, s_kv=8, h_q=8, d_qk=576, d_v=512,
             topk=128, stream=None)
    a.update(kw)
    return lib.sparse_mla_fwd(a["q"], a["kv"], a["idx"], a["scale"], a["out"], a["lse"], a["s_q"], a["s_kv"],
                              a["h_q"], a["d_qk"], a["d_v"], a["topk"], a["stream"])


def test_host_validation_codes(lib):
    assert _fwd(lib, d_qk=512) == 2
    assert _fwd(lib, d_v=576) == 2
    assert _fwd(lib, h_q=0) == 1
    assert _fwd(lib, topk=0) == 1
    assert _fwd(lib, s_q=-1) == 1
    assert _fwd(lib, q=None) == 1
    assert _fwd(lib, out=None) == 1
    assert _fwd(lib, lse=None) == 1
    assert _fwd(lib, q=24) == 1      # not 16-byte aligned
    assert _fwd(lib, idx=18) == 1    # not 4-byte aligned


def test_causal_validation(lib):
    def causal(**kw):
        a = dict(q=16, kv=16, scale=0.1, out=16, lse=16, s_q=4, s_kv=8, h_q=8, d_qk=576, d_v=512, stream=None)
        a.update(kw)
        return lib.sparse_mla_fwd_causal(a["q"], a["kv"], a["scale"], a["out"], a["lse"], a["s_q"], a["s_kv"],
                                         a["h_q"], a["d_qk"], a["d_v"], a["stream"])
    assert causal(d_qk=512) == 2
    assert causal(d_v=256) == 2
    assert causal(h_q=0) == 1
    assert causal(s_q=-1) == 1
    assert causal(s_kv=-1) == 1
    assert causal(q=None) == 1
    assert causal(out=None) == 1
    assert causal(q=24) == 1      # not 16-byte aligned


def test_varlen_and_decode_validation(lib):
    st = lib.sparse_mla_fwd_varlen(16, 16, 16, None, None, 1, 0.1, 16, 16, 4, 4, 8, 576, 512, 64, None)
    assert st == 1
    st = lib.sparse_mla_fwd_varlen(16, 16, 16, 16, 16, 1, 0.1, 16, 16, 4, 4, 8, 576, 256, 64, None)
    assert st == 2
    st = lib.sparse_mla_decode(16, 16, 16, 16, 16, 0.1, 16, 16, 2, 3, 8, 576, 512, 64, 0, 4, 4, None, 0, None)
    assert st == 1   # page_size 0
    st = lib.sparse_mla_decode(16, 16, None, 16, 16, 0.1, 16, 16, 2, 3, 8, 576, 512, 64, 64, 4, 4, None, 0, None)
    assert st == 1   # missing block table
    st = lib.sparse_mla_decode(16, 16, 16, 16, 16, 0.1, 16, 16, 2, 3, 8, 576, 512, 64, 64, 4, 1 << 30, None, 0,
                               None)
    assert st == 1   # num_blocks * page_size overflows int32


def test_workspace_size_rejects_bad_shapes(lib):
    assert lib.sparse_mla_decode_workspace_size(0, 6, 8, 512, 2048) == 0
    assert lib.sparse_mla_decode_workspace_size(4, 6, 8, 256, 2048) == 0


def test_indexer_validation(lib):
    def scores(**kw):
        a = dict(q=16, k=16, w=16, cq=None, ck=None, batch=1, tq=8, tk=40, h=64, d=128, row0=0, n=8, skip=0,
                 out=16, stride=40, stream=None)
        a.update(kw)
        return lib.dsa_indexer_scores(a["q"], a["k"], a["w"], a["cq"], a["ck"], a["batch"], a["tq"], a["tk"],
                                      a["h"], a["d"], a["row0"], a["n"], a["skip"], a["out"], a["stride"],
                                      a["stream"])
    assert scores(d=64) == 2
    assert scores(h=48) == 2
    assert scores(cq=16) == 1            # one offset array without the other
    assert scores(cq=16, ck=16, batch=4096) == 2
    assert scores(q=24) == 1             # not 16-byte aligned
    assert scores(w=8) == 1
    assert scores(row0=4, n=5) == 1      # past the last row
    assert scores(skip=-1) == 1
    assert scores(stride=0) == 1
    assert scores(tq=-1) == 1

    def topk(**kw):
        a = dict(sc=16, stride=40, cq=None, ck=None, batch=1, tq=8, tk=40, row0=0, n=8, topk=16, idx=16,
                 stream=None)
        a.update(kw)
        return lib.dsa_topk(a["sc"], a["stride"], a["cq"], a["ck"], a["batch"], a["tq"], a["tk"], a["row0"],
                            a["n"], a["topk"], a["idx"], a["stream"])
    assert topk(topk=0) == 1
    assert topk(ck=16) == 1
    assert topk(n=9) == 1
    assert topk(idx=None) == 1
    assert topk(idx=18) == 1
    assert topk(sc=None) == 1            # rows longer than topk need scores

    def fused(**kw):
        a = dict(q=16, k=16, w=16, cq=None, ck=None, batch=1, tq=8, tk=40, ms=40, h=64, d=128, topk=16, idx=16,
                 ws=16, wsb=4096, stream=None)
        a.update(kw)
        return lib.dsa_indexer_topk(a["q"], a["k"], a["w"], a["cq"], a["ck"], a["batch"], a["tq"], a["tk"],
                                    a["ms"], a["h"], a["d"], a["topk"], a["idx"], a["ws"], a["wsb"], a["stream"])
    assert fused(ms=41) == 1             # longer than the keys
    assert fused(ms=20) == 1             # one dense sequence: its length is total_kv
    assert fused(topk=0) == 1
    assert fused(h=8) == 2
    assert fused(idx=None) == 1


def test_indexer_workspace_size(lib):
    assert lib.dsa_indexer_workspace_size(10, 4097, 2048) == 10 * 4100 * 4
    assert lib.dsa_indexer_workspace_size(10, 4096, 2048) == 10 * 4096 * 4
    assert lib.dsa_indexer_workspace_size(10, 2048, 2048) == 0      # no row is scored
    assert lib.dsa_indexer_workspace_size(0, 4096, 2048) == 0


def test_paged_indexer_validation(lib):
    def paged(**kw):
        a = dict(q=16, k=16, w=16, bt=16, sl=16, batch=2, s_next=6, h=64, d=128, page=64, mb=8, nb=16, ms=500,
                 topk=64, idx=16, ws=16, wsb=4096, stream=None)
        a.update(kw)
        return lib.dsa_indexer_topk_paged(a["q"], a["k"], a["w"], a["bt"], a["sl"], a["batch"], a["s_next"],
                                          a["h"], a["d"], a["page"], a["mb"], a["nb"], a["ms"], a["topk"], a["idx"],
                                          a["ws"], a["wsb"], a["stream"])
    assert paged(page=32) == 2
    assert paged(h=8) == 2
    assert paged(batch=4096) == 2
    assert paged(s_next=0) == 1
    assert paged(bt=None) == 1
    assert paged(sl=None) == 1
    assert paged(k=24) == 1          # not 16-byte aligned
    assert paged(topk=0) == 1
    assert paged(idx=None) == 1
    st = lib.dsa_indexer_scores_paged(16, 16, 16, 16, 16, 2, 6, 64, 128, 64, 8, 16, 10, 5, 0, 16, 500, None)
    assert st == 1                   # rows past batch * s_next


def test_fp8_decode_and_debug_count_validation(lib):
    """Argument errors of the FP8 decode and of the debug count exports come
    back before any device work."""
    def fp8(**kw):
        a = dict(q=16, kv=16, bt=16, sl=16, idx=16, scale=0.1, out=16, lse=16, batch=2, s_next=3, h_q=8,
                 d_qk=576, d_v=512, topk=64, page=64, max_blocks=4, num_blocks=8, ws=None, ws_bytes=0,
                 stream=None)
        a.update(kw)
        return lib.sparse_mla_decode_fp8(a["q"], a["kv"], a["bt"], a["sl"], a["idx"], a["scale"], a["out"],
                                         a["lse"], a["batch"], a["s_next"], a["h_q"], a["d_qk"], a["d_v"],
                                         a["topk"], a["page"], a["max_blocks"], a["num_blocks"], a["ws"],
                                         a["ws_bytes"], a["stream"])
    assert fp8(d_qk=512) == 2
    assert fp8(batch=-1) == 1
    assert fp8(page=0) == 1
    assert fp8(bt=None) == 1
    assert fp8(q=24) == 1
    assert lib.sparse_mla_debug_valid_count(None, 4, 10, 64, 16, None) == 1
    assert lib.sparse_mla_debug_valid_count(16, 4, 10, 0, 16, None) == 1
    assert lib.sparse_mla_debug_valid_count(16, 4, -1, 64, 16, None) == 1
    assert lib.sparse_mla_debug_valid_count_varlen(16, None, 16, 2, 4, 10, 64, 16, None) == 1
    assert lib.sparse_mla_debug_valid_count_paged(16, 16, 16, 2, 3, 64, 0, 4, 8, 16, None) == 1
    assert lib.sparse_mla_debug_valid_count_paged(16, None, 16, 2, 3, 64, 64, 4, 8, 16, None) == 1
