"""C-ABI checks that need no GPU: the library loads, exports every function
include/smla.h declares, and rejects bad host arguments with the documented
status codes before touching any device memory."""
import ctypes
import os
import re

import pytest

import sparse_mla_attention_fp8_gb300 as smla

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "smla.h")


@pytest.fixture(scope="module")
def L():
    smla.build()
    return smla.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_path_entry_points():
    names = declared_functions()
    for n in ["sparse_mla_decode_fp8", "sparse_mla_prefill_bf16", "mla_cache_store_fp8",
              "sparse_mla_translate_indices", "sparse_mla_decode_workspace_bytes", "smla_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_version(L):
    assert L.smla_version() == 100


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


def _decode(L, **kw):
    a = dict(q=FAKE, cache=FAKE, idx=FAKE, bt=FAKE, req=FAKE, scale=0.1, ns=0, out=FAKE, lse=FAKE,
             T=4, H=16, K=64, R=4, MB=4, NB=16, ws=None, wsb=0, stream=None)
    a.update(kw)
    return L.sparse_mla_decode_fp8(a["q"], a["cache"], a["idx"], a["bt"], a["req"], a["scale"], a["ns"], a["out"],
                                   a["lse"], a["T"], a["H"], a["K"], a["R"], a["MB"], a["NB"], a["ws"], a["wsb"],
                                   a["stream"])


@pytest.mark.parametrize("H", [0, 8, 17, 144, 256])
def test_decode_rejects_unsupported_heads(L, H):
    assert _decode(L, H=H) == -2
    assert b"H=" in L.smla_last_error()


@pytest.mark.parametrize("kw", [dict(T=-1), dict(K=-3), dict(R=0), dict(MB=0), dict(NB=0), dict(ns=-1)])
def test_decode_rejects_bad_sizes(L, kw):
    assert _decode(L, **kw) == -1


def test_decode_rejects_null_and_misaligned(L):
    assert _decode(L, q=None) == -1
    assert _decode(L, out=None) == -1
    assert _decode(L, q=ctypes.c_void_p(0x10008)) == -1
    assert b"aligned" in L.smla_last_error()


def test_decode_empty_batch_is_a_noop(L):
    assert _decode(L, T=0, q=None, out=None) == 0


def test_prefill_rejects_bad_arguments(L):
    f = L.sparse_mla_prefill_bf16
    assert f(FAKE, FAKE, FAKE, 0.1, 0, FAKE, FAKE, 4, 20, 8, 8, None, 0, None) == -2
    assert f(FAKE, FAKE, FAKE, 0.1, 0, FAKE, FAKE, 4, 16, 0, 8, None, 0, None) == -1
    assert f(None, FAKE, FAKE, 0.1, 0, FAKE, FAKE, 4, 16, 8, 8, None, 0, None) == -1


def test_store_and_translate_reject_bad_arguments(L):
    assert L.mla_cache_store_fp8(FAKE, FAKE, FAKE, -1, 4, None) == -1
    assert L.mla_cache_store_fp8(None, FAKE, FAKE, 3, 4, None) == -1
    assert L.mla_cache_store_fp8(ctypes.c_void_p(0x10004), FAKE, FAKE, 3, 4, None) == -1
    assert L.mla_cache_store_fp8(FAKE, FAKE, FAKE, 0, 4, None) == 0
    assert L.sparse_mla_translate_indices(FAKE, FAKE, FAKE, FAKE, 2, 3, 0, 1, 1, None) == -1
    assert L.sparse_mla_translate_indices(None, FAKE, FAKE, FAKE, 2, 3, 1, 1, 1, None) == -1


def test_python_binding_has_no_cpu_path():
    import torch
    q = torch.zeros((1, 16, 576), dtype=torch.bfloat16)
    with pytest.raises(smla.SmlaError):
        smla.sparse_mla_prefill_bf16(q, torch.zeros((4, 576), dtype=torch.bfloat16),
                                     torch.zeros((1, 4), dtype=torch.int32), 0.1)


def test_prefill_chunks_docstring_example(L):
    # flashmla_sparse.py, FlashMLASparseMetadataBuilder: seq_lens [10, 15, 20, 5] in chunks [[0, 2], [2, 4]]
    # have workspace starts [0, 10, 0, 20] after the per-chunk adjustment (any workspace of 25..44 rows)
    for rows in (25, 30, 44):
        bounds, starts = smla.sparse_mla_prefill_chunks([10, 15, 20, 5], rows)
        assert bounds == [(0, 2), (2, 4)] and starts == [0, 10, 0, 20]
    assert smla.sparse_mla_prefill_chunks([10, 15, 20, 5], 45) == ([(0, 3), (3, 4)], [0, 10, 25, 0])
    assert smla.sparse_mla_prefill_chunks([10, 15, 20, 5], 50) == ([(0, 4)], [0, 10, 25, 45])
    assert smla.sparse_mla_prefill_chunks([], 8) == ([], [])
    with pytest.raises(smla.SmlaError, match="status -4"):
        smla.sparse_mla_prefill_chunks([10, 60, 5], 50)


def test_prefill_fp8_rejects_bad_arguments(L):
    args = dict(q=FAKE, cache=FAKE, idx=FAKE, bt=FAKE, req=FAKE, sl=FAKE, st=FAKE, scale=0.1, ns=0, out=FAKE,
                lse=FAKE, T=4, H=16, K=64, R=2, MB=4, NB=16, kvw=FAKE, N=128, ws=None, wsb=0, stream=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.sparse_mla_prefill_fp8(a["q"], a["cache"], a["idx"], a["bt"], a["req"], a["sl"], a["st"],
                                        a["scale"], a["ns"], a["out"], a["lse"], a["T"], a["H"], a["K"], a["R"],
                                        a["MB"], a["NB"], a["kvw"], a["N"], a["ws"], a["wsb"], a["stream"])
    assert call(H=24) == -2
    assert call(N=0) == -1
    assert call(kvw=None) == -1
    assert call(q=ctypes.c_void_p(0x10008)) == -1  # misaligned
    assert call(T=0) == 0
