"""Float64 CPU oracle for sparse MLA attention over the 656-byte FP8 cache.

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product path
(``sparse_mla_attention_fp8_gb300``) never imports this package, and this
package never imports the product.  They share no code; they meet only
through the seeded input generators in ``smla_inputs``.

The arithmetic lives in ``smla_oracle.c`` (plain C, double precision, OpenMP
over tokens); this module builds it with gcc and marshals numpy arrays.
The MLA weight absorption steps around the attention (``absorb_q``,
``v_up_proj``) are float64 numpy matrix products written in this module.
Every function cites the passage of the pages it follows (for the C
functions, in the C source):
vLLM ``flashmla_sparse.py`` (module docstring on the "FP8 with scale" layout,
``triton_convert_req_index_to_global_index`` and its docstring formula,
``FlashMLASparseImpl.forward``), vLLM PR #59342 (the 352-byte
``nvfp4_ds_mla`` row), the OCP 8-bit floating point specification for E4M3
and the OCP Microscaling specification for FP4 E2M1.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libsmla_oracle.so")
_lock = threading.Lock()
_lib = None

ROW_BYTES = 656
NVFP4_ROW_BYTES = 352
D_QK = 576
D_V = 512


def build(force: bool = False) -> str:
    """Compile the oracle shared library in place (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = f64
            lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_dequant_row.argtypes = [P, P]
            lib.oracle_dequant_row.restype = None
            lib.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_to_double.restype = f64
            lib.oracle_e2m1_from_float.argtypes = [ctypes.c_float]
            lib.oracle_e2m1_from_float.restype = ctypes.c_uint8
            lib.oracle_nvfp4_dequant_row.argtypes = [P, P]
            lib.oracle_nvfp4_dequant_row.restype = None
            lib.oracle_nvfp4_quantize_store.argtypes = [P, P, P, i32, i64]
            lib.oracle_nvfp4_quantize_store.restype = None
            lib.oracle_sparse_mla_decode_nvfp4.argtypes = [P, P, P, P, P, f64, i32, i32, i32, i32, i32, i64, P, i32,
                                                           P, P, i32, P, P]
            lib.oracle_sparse_mla_decode_nvfp4.restype = None
            lib.oracle_translate.argtypes = [P, P, P, i32, i32, i32, i32, i64, P]
            lib.oracle_translate.restype = None
            lib.oracle_quantize_store.argtypes = [P, P, P, i32, i64]
            lib.oracle_quantize_store.restype = None
            lib.oracle_sparse_mla_decode.argtypes = [P, P, P, P, P, f64, i32, i32, i32, i32, i32, i64, P, i32,
                                                     P, P, i32, P, P]
            lib.oracle_sparse_mla_decode.restype = None
            lib.oracle_sparse_mla_prefill.argtypes = [P, P, P, f64, i32, i32, i64, i32, P, i32, P, P, i32, P, P]
            lib.oracle_sparse_mla_prefill.restype = None
            lib.oracle_upconvert_row.argtypes = [P, P]
            lib.oracle_upconvert_row.restype = None
            lib.oracle_gather_upconvert.argtypes = [P, i64, P, i32, i32, P, P, P, i64]
            lib.oracle_gather_upconvert.restype = None
            lib.oracle_translate_workspace.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, i32, P]
            lib.oracle_translate_workspace.restype = None
            _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------- formats

def e4m3_to_double(code: int) -> float:
    return _load().oracle_e4m3_to_double(int(code) & 0xFF)


def e4m3_from_float(y: float) -> int:
    return int(_load().oracle_e4m3_from_float(float(y)))


def dequant_row(row: np.ndarray) -> np.ndarray:
    """One 656-byte cache row -> float64[576] (NoPE dequantized, RoPE exact)."""
    row = _c(row, np.uint8).reshape(-1)
    assert row.size == ROW_BYTES
    out = np.empty(D_QK, np.float64)
    _load().oracle_dequant_row(_p(row), _p(out))
    return out


def e2m1_to_double(code: int) -> float:
    """OCP MX FP4 E2M1 code (4 bits) -> value."""
    return _load().oracle_e2m1_to_double(int(code) & 0xF)


def e2m1_from_float(y: float) -> int:
    """Nearest E2M1 code (ties to even, saturating to 6)."""
    return int(_load().oracle_e2m1_from_float(float(y)))


def nvfp4_dequant_row(row: np.ndarray) -> np.ndarray:
    """One 352-byte NVFP4 cache row -> float64[576] (the layout of reading
    R13 in smla_oracle.c: E2M1 NoPE codes with an E4M3 scale per 16 values,
    E4M3 RoPE)."""
    row = _c(row, np.uint8).reshape(-1)
    assert row.size == NVFP4_ROW_BYTES
    out = np.empty(D_QK, np.float64)
    _load().oracle_nvfp4_dequant_row(_p(row), _p(out))
    return out


# ---------------------------------------------------------------- steps

def translate(indices, block_table, req_id_per_token, num_blocks: int) -> np.ndarray:
    """Logical top-k index -> physical cache slot (int32, -1 = invalid)."""
    idx = _c(indices, np.int32)
    bt = _c(block_table, np.int32)
    req = _c(req_id_per_token, np.int32)
    T, K = idx.shape
    R, MB = bt.shape
    out = np.empty((T, K), np.int32)
    _load().oracle_translate(_p(idx), _p(bt), _p(req), T, K, R, MB, int(num_blocks), _p(out))
    return out


def quantize_store(kv_new_bits, slot_mapping, cache: np.ndarray) -> None:
    """Quantize bf16 rows (uint16 bits [T, 576]) into ``cache`` (uint8
    [NB, 64, 656], modified in place) at ``slot_mapping`` (int64 [T])."""
    kv = _c(kv_new_bits, np.uint16)
    sm = _c(slot_mapping, np.int64)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and cache.shape[-1] == ROW_BYTES
    NB = cache.shape[0]
    T = kv.shape[0]
    assert kv.shape == (T, D_QK) and sm.shape == (T,)
    _load().oracle_quantize_store(_p(kv), _p(sm), _p(cache), T, NB)


def nvfp4_quantize_store(kv_new_bits, slot_mapping, cache: np.ndarray) -> None:
    """Quantize bf16 rows (uint16 bits [T, 576]) into the NVFP4 ``cache``
    (uint8 [NB, 64, 352], modified in place) at ``slot_mapping`` (int64 [T])."""
    kv = _c(kv_new_bits, np.uint16)
    sm = _c(slot_mapping, np.int64)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and cache.shape[-1] == NVFP4_ROW_BYTES
    NB = cache.shape[0]
    T = kv.shape[0]
    assert kv.shape == (T, D_QK) and sm.shape == (T,)
    _load().oracle_nvfp4_quantize_store(_p(kv), _p(sm), _p(cache), T, NB)


def sparse_mla_decode(q_bits, cache, indices, block_table, req_id_per_token, sm_scale: float,
                      tokens=None, nthreads: int | None = None):
    """FP8 sparse decode; returns (out float64 [n, H, 512], lse float64 [n, H])
    for the listed tokens (all tokens when ``tokens`` is None)."""
    return _decode(_load().oracle_sparse_mla_decode, ROW_BYTES, q_bits, cache, indices, block_table,
                   req_id_per_token, sm_scale, tokens, nthreads)


def sparse_mla_decode_nvfp4(q_bits, cache, indices, block_table, req_id_per_token, sm_scale: float,
                            tokens=None, nthreads: int | None = None):
    """The same decode over the NVFP4 cache (uint8 [NB, 64, 352])."""
    return _decode(_load().oracle_sparse_mla_decode_nvfp4, NVFP4_ROW_BYTES, q_bits, cache, indices, block_table,
                   req_id_per_token, sm_scale, tokens, nthreads)


def _decode(fn, row_bytes, q_bits, cache, indices, block_table, req_id_per_token, sm_scale, tokens, nthreads):
    q = _c(q_bits, np.uint16)
    T, H, D = q.shape
    assert D == D_QK
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and cache.shape[-1] == row_bytes
    NB = cache.shape[0]
    idx = _c(indices, np.int32)
    K = idx.shape[1]
    bt = _c(block_table, np.int32)
    R, MB = bt.shape
    req = _c(req_id_per_token, np.int32)
    tok = None if tokens is None else _c(tokens, np.int32)
    n = T if tok is None else tok.size
    nth = nthreads or default_threads()
    ws_rows = np.empty((nth, max(K, 1), D_QK), np.float64)
    ws_s = np.empty((nth, max(K, 1)), np.float64)
    out = np.empty((n, H, D_V), np.float64)
    lse = np.empty((n, H), np.float64)
    fn(_p(q), _p(cache), _p(idx), _p(bt), _p(req), float(sm_scale), T, H, K, R, MB, NB, _p(tok), n, _p(ws_rows),
       _p(ws_s), nth, _p(out), _p(lse))
    return out, lse


def sparse_mla_prefill(q_bits, kv_bits, indices, sm_scale: float, tokens=None, nthreads: int | None = None):
    """BF16 sparse prefill over a dense latent buffer (uint16 bits [N, 576])."""
    q = _c(q_bits, np.uint16)
    T, H, D = q.shape
    assert D == D_QK
    kv = _c(kv_bits, np.uint16)
    N = kv.shape[0]
    idx = _c(indices, np.int32)
    K = idx.shape[1]
    tok = None if tokens is None else _c(tokens, np.int32)
    n = T if tok is None else tok.size
    nth = nthreads or default_threads()
    ws_rows = np.empty((nth, max(K, 1), D_QK), np.float64)
    ws_s = np.empty((nth, max(K, 1)), np.float64)
    out = np.empty((n, H, D_V), np.float64)
    lse = np.empty((n, H), np.float64)
    _load().oracle_sparse_mla_prefill(_p(q), _p(kv), _p(idx), float(sm_scale), T, H, N, K, _p(tok), n,
                                      _p(ws_rows), _p(ws_s), nth, _p(out), _p(lse))
    return out, lse


# ---------------------------------------------------------------- separate-mode FP8 prefill

def upconvert_row(row: np.ndarray) -> np.ndarray:
    """One 656-byte cache row -> bf16 bits uint16[576]: NoPE code * scale in
    float32 rounded to bf16 (ties to even), RoPE as stored."""
    row = _c(row, np.uint8).reshape(-1)
    assert row.size == ROW_BYTES
    out = np.empty(D_QK, np.uint16)
    _load().oracle_upconvert_row(_p(row), _p(out))
    return out


def gather_upconvert(cache, block_table, seq_lens, workspace_starts, n_rows: int) -> np.ndarray:
    """Positions 0 .. seq_lens[r] - 1 of each request r up-converted into a
    bf16 workspace (uint16 bits [n_rows, 576]) at rows workspace_starts[r] + p;
    rows nothing is written to are zero."""
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    NB = cache.shape[0]
    bt = _c(block_table, np.int32)
    R, MB = bt.shape
    sl = _c(seq_lens, np.int32)
    st = _c(workspace_starts, np.int32)
    assert sl.shape == (R,) and st.shape == (R,)
    ws = np.zeros((int(n_rows), D_QK), np.uint16)
    _load().oracle_gather_upconvert(_p(cache), NB, _p(bt), R, MB, _p(sl), _p(st), _p(ws), int(n_rows))
    return ws


def translate_workspace(indices, block_table, req_id_per_token, prefill_request_id, workspace_starts,
                        num_blocks: int) -> np.ndarray:
    """Logical top-k index -> cache slot (decode tokens, prefill_request_id < 0)
    or prefill-workspace row (prefill tokens); int32, -1 = invalid."""
    idx = _c(indices, np.int32)
    bt = _c(block_table, np.int32)
    req = _c(req_id_per_token, np.int32)
    pr = _c(prefill_request_id, np.int32)
    st = _c(workspace_starts, np.int32)
    T, K = idx.shape
    R, MB = bt.shape
    out = np.empty((T, K), np.int32)
    _load().oracle_translate_workspace(_p(idx), _p(bt), _p(req), _p(pr), _p(st), T, K, R, MB, int(num_blocks),
                                       st.size, _p(out))
    return out


def sparse_mla_prefill_fp8(q_bits, cache, indices, block_table, req_id_per_token, seq_lens, workspace_starts,
                           n_rows: int, sm_scale: float, tokens=None, nthreads: int | None = None):
    """Separate-mode FP8 prefill of one chunk of prefill requests, step by
    step as the pages do it: the requests' rows up-converted into a bf16
    workspace, the tokens' indices mapped to workspace rows, then the bf16
    prefill over the workspace.  Returns (out, lse) as sparse_mla_prefill."""
    ws = gather_upconvert(cache, block_table, seq_lens, workspace_starts, n_rows)
    req = _c(req_id_per_token, np.int32)
    rows = translate_workspace(indices, block_table, req, req, workspace_starts, cache.shape[0])
    return sparse_mla_prefill(q_bits, ws, rows, sm_scale, tokens=tokens, nthreads=nthreads)


# ---------------------------------------------------------------- MLA weight absorption

def _bf16_to_f64(bits):
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def absorb_q(q_bits, w_uk_t_bits) -> np.ndarray:
    """FlashMLASparseImpl.forward before the attention, in float64: q (bf16
    bits [T, H, P + 64]) is split into q_nope [T, H, P] and q_pe [T, H, 64];
    ql_nope[t, h, :] = q_nope[t, h, :] @ W_UK_T[h] (bf16 bits [H, P, 512]);
    the attention input is ql_nope ++ q_pe, float64 [T, H, 576]."""
    q = _bf16_to_f64(q_bits)
    w = _bf16_to_f64(w_uk_t_bits)
    T, H, D = q.shape
    P = D - 64
    assert w.shape == (H, P, D_V)
    q_nope, q_pe = q[..., :P], q[..., P:]
    ql_nope = np.matmul(q_nope.transpose(1, 0, 2), w).transpose(1, 0, 2)  # (H, T, P) x (H, P, L) -> (T, H, L)
    return np.concatenate([ql_nope, q_pe], axis=-1)


def v_up_proj(attn_out_bits, w_uv_bits) -> np.ndarray:
    """FlashMLASparseImpl._v_up_proj in float64: out[t, h, :] =
    attn_out[t, h, :] @ W_UV[h] for attn_out bf16 bits [T, H, 512] and W_UV
    bf16 bits [H, 512, V]; float64 [T, H, V]."""
    a = _bf16_to_f64(attn_out_bits)
    w = _bf16_to_f64(w_uv_bits)
    T, H, L = a.shape
    assert L == D_V and w.shape[:2] == (H, D_V)
    return np.matmul(a.transpose(1, 0, 2), w).transpose(1, 0, 2)
