"""Sparse MLA attention over the 656-byte FP8 cache, for GB300 (sm_103a).

Thin Python binding of the C-ABI library ``libsmla.so`` (declared in
``include/smla.h``).  Every function here only marshals torch tensors into
pointers and sizes and calls the same-named C entry point; all the work runs
in the library's CUDA kernels.  There is no CPU fallback: if the library has
not been built, or a tensor is not on a CUDA device, the call raises.

Entry points (see include/smla.h for layouts and semantics):
  sparse_mla_decode_fp8, sparse_mla_prefill_bf16, mla_cache_store_fp8,
  sparse_mla_translate_indices, the separate-mode FP8 prefill
  (sparse_mla_prefill_fp8 with its steps sparse_mla_gather_upconvert_fp8 and
  sparse_mla_translate_indices_workspace, and the host-side
  sparse_mla_prefill_chunks), plus workspace-size and status helpers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_CSRC = os.path.join(_PKG, "csrc")
_BUILD = os.path.join(_PKG, "_build")
LIB_PATH = os.path.join(_PKG, "libsmla.so")
HEADER = os.path.join(_ROOT, "include", "smla.h")

SOURCES = ["smla_decode.cu", "smla_attn.cu", "smla_wide.cu", "smla_wide8.cu", "smla_store.cu", "smla_nvfp4.cu", "smla_absorb.cu", "smla_api.cu"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]

SMLA_OK = 0
_lock = threading.Lock()
_lib = None


class SmlaError(RuntimeError):
    pass


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(_CSRC, f) for f in os.listdir(_CSRC) if f.endswith((".cuh", ".h"))] + [HEADER]
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA sources for sm_103a (in parallel) and link libsmla.so
    in place.  Works without a GPU (nvcc cross-compiles)."""
    os.makedirs(_BUILD, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for s in SOURCES:
        src = os.path.join(_CSRC, s)
        obj = os.path.join(_BUILD, s.replace(".cu", ".o"))
        if force or _stale(obj, src):
            jobs.append([nvcc, *NVCC_FLAGS, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise SmlaError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)

    if jobs:
        with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            list(ex.map(run, jobs))
    objs = [os.path.join(_BUILD, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or not os.path.exists(LIB_PATH):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        run([nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise SmlaError(f"{LIB_PATH} is missing: run sparse_mla_attention_fp8_gb300.build() first")
            L = ctypes.CDLL(LIB_PATH)
            P, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
            L.sparse_mla_decode_fp8.argtypes = [P, P, P, P, P, f32, i32, P, P, i32, i32, i32, i32, i32, i32, P, sz, P]
            L.sparse_mla_decode_fp8.restype = i32
            L.sparse_mla_decode_fp8_qfp8.argtypes = L.sparse_mla_decode_fp8.argtypes
            L.sparse_mla_decode_fp8_qfp8.restype = i32
            L.sparse_mla_decode_nvfp4.argtypes = L.sparse_mla_decode_fp8.argtypes
            L.sparse_mla_decode_nvfp4.restype = i32
            L.sparse_mla_decode_nvfp4_workspace_bytes.argtypes = [i32, i32, i32, i32]
            L.sparse_mla_decode_nvfp4_workspace_bytes.restype = sz
            L.mla_cache_store_nvfp4.argtypes = [P, P, P, i32, i32, P]
            L.mla_cache_store_nvfp4.restype = i32
            L.sparse_mla_decode_fp8_noalloc.argtypes = [P, P, P, P, P, f32, i32, P, P, i32, i32, i32, i32, i32, i32, P]
            L.sparse_mla_decode_fp8_noalloc.restype = i32
            L.sparse_mla_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
            L.sparse_mla_decode_workspace_bytes.restype = sz
            L.sparse_mla_prefill_bf16.argtypes = [P, P, P, f32, i32, P, P, i32, i32, i32, i32, P, sz, P]
            L.sparse_mla_prefill_bf16.restype = i32
            L.sparse_mla_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32]
            L.sparse_mla_prefill_workspace_bytes.restype = sz
            L.sparse_mla_attention_plan.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            L.sparse_mla_attention_plan.restype = i32
            L.mla_cache_store_fp8.argtypes = [P, P, P, i32, i32, P]
            L.mla_cache_store_fp8.restype = i32
            L.sparse_mla_translate_indices.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P]
            L.sparse_mla_translate_indices.restype = i32
            L.smla_read_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int), P]
            L.smla_read_device_status.restype = i32
            L.sparse_mla_prefill_fp8.argtypes = [P, P, P, P, P, P, P, f32, i32, P, P, i32, i32, i32, i32, i32, i32,
                                                 P, i32, P, sz, P]
            L.sparse_mla_prefill_fp8.restype = i32
            L.sparse_mla_prefill_fp8_workspace_bytes.argtypes = [i32, i32, i32, i32]
            L.sparse_mla_prefill_fp8_workspace_bytes.restype = sz
            L.sparse_mla_gather_upconvert_fp8.argtypes = [P, P, P, P, i32, i32, i32, P, i32, P]
            L.sparse_mla_gather_upconvert_fp8.restype = i32
            L.sparse_mla_translate_indices_workspace.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, P]
            L.sparse_mla_translate_indices_workspace.restype = i32
            L.sparse_mla_prefill_chunks.argtypes = [P, i32, ctypes.c_int64, P, P, ctypes.POINTER(i32)]
            L.sparse_mla_prefill_chunks.restype = i32
            L.mla_absorb_q.argtypes = [P, P, P, i32, i32, i32, P, sz, P]
            L.mla_absorb_q.restype = i32
            L.mla_v_up_proj.argtypes = [P, P, P, i32, i32, i32, P, sz, P]
            L.mla_v_up_proj.restype = i32
            L.smla_read_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int), P]
            L.smla_read_noalloc_status.restype = i32
            L.smla_last_error.argtypes = []
            L.smla_last_error.restype = ctypes.c_char_p
            L.smla_version.argtypes = []
            L.smla_version.restype = i32
            _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != SMLA_OK:
        msg = lib().smla_last_error().decode(errors="replace")
        raise SmlaError(f"{what} failed with status {rc}: {msg}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(*tensors):
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise SmlaError("all tensors must be CUDA tensors (there is no CPU path)")
        if not t.is_contiguous():
            raise SmlaError("all tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise SmlaError("all tensors must be on the same device")
    return dev


def _expect(t, dtype, shape, name):
    if t.dtype != dtype:
        raise SmlaError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise SmlaError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def decode_workspace_bytes(T: int, H: int, K: int, num_splits: int = 0) -> int:
    return int(lib().sparse_mla_decode_workspace_bytes(T, H, K, num_splits))


def decode_nvfp4_workspace_bytes(T: int, H: int, K: int, num_splits: int = 0) -> int:
    return int(lib().sparse_mla_decode_nvfp4_workspace_bytes(T, H, K, num_splits))


def prefill_workspace_bytes(T: int, H: int, K: int, num_splits: int = 0) -> int:
    return int(lib().sparse_mla_prefill_workspace_bytes(T, H, K, num_splits))


def attention_plan(fp8: bool, T: int, H: int, K: int, num_splits: int = 0) -> tuple:
    """(kernel launches, attention-kernel CTAs) of one decode (fp8=True) or
    prefill call with these sizes on the current device."""
    launches, ctas = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().sparse_mla_attention_plan(int(bool(fp8)), T, H, K, num_splits, ctypes.byref(launches),
                                           ctypes.byref(ctas)), "sparse_mla_attention_plan")
    return int(launches.value), int(ctas.value)


def sparse_mla_decode_fp8(q, kv_cache, indices, block_table, req_id_per_token, sm_scale: float,
                          num_splits: int = 0, out=None, lse=None, workspace=None, stream=None):
    """FP8 sparse decode.  q bf16 [T,H,576]; kv_cache uint8 [NB,64,656];
    indices int32 [T,K] (logical, <0 = none); block_table int32 [R,MB];
    req_id_per_token int32 [T].  Returns (out bf16 [T,H,512], lse fp32 [T,H])."""
    return _decode("sparse_mla_decode_fp8", q, kv_cache, indices, block_table, req_id_per_token, sm_scale,
                   num_splits, out, lse, workspace, stream)


def sparse_mla_decode_fp8_qfp8(q, kv_cache, indices, block_table, req_id_per_token, sm_scale: float,
                               num_splits: int = 0, out=None, lse=None, workspace=None, stream=None):
    """sparse_mla_decode_fp8 with the query quantized to FP8 (two e4m3 terms)
    and both products on the FP8 tensor path; at H = 128 a kernel of its own
    (slower than sparse_mla_decode_fp8's on GB300).  Same arguments and results."""
    return _decode("sparse_mla_decode_fp8_qfp8", q, kv_cache, indices, block_table, req_id_per_token, sm_scale,
                   num_splits, out, lse, workspace, stream)


def sparse_mla_decode_nvfp4(q, kv_cache, indices, block_table, req_id_per_token, sm_scale: float,
                            num_splits: int = 0, out=None, lse=None, workspace=None, stream=None):
    """Sparse decode over the NVFP4 cache (kv_cache uint8 [NB,64,352]); the
    other arguments and the results as for sparse_mla_decode_fp8."""
    return _decode("sparse_mla_decode_nvfp4", q, kv_cache, indices, block_table, req_id_per_token, sm_scale,
                   num_splits, out, lse, workspace, stream, row_bytes=352)


def _decode(name, q, kv_cache, indices, block_table, req_id_per_token, sm_scale, num_splits, out, lse, workspace,
            stream, row_bytes=656):
    import torch
    dev = _dev(q, kv_cache, indices, block_table, req_id_per_token, out, lse, workspace)
    T, H, D = q.shape
    NB = kv_cache.shape[0]
    K = indices.shape[1]
    R, MB = block_table.shape
    _expect(q, torch.bfloat16, (T, H, 576), "q")
    _expect(kv_cache, torch.uint8, (NB, 64, row_bytes), "kv_cache")
    _expect(indices, torch.int32, (T, K), "indices")
    _expect(req_id_per_token, torch.int32, (T,), "req_id_per_token")
    if block_table.dtype != torch.int32:
        raise SmlaError("block_table must be int32")
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    _expect(out, torch.bfloat16, (T, H, 512), "out")
    _expect(lse, torch.float32, (T, H), "lse")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = getattr(lib(), name)(_ptr(q), _ptr(kv_cache), _ptr(indices), _ptr(block_table), _ptr(req_id_per_token),
                              float(sm_scale), int(num_splits), _ptr(out), _ptr(lse), T, H, K, R, MB, NB,
                              _ptr(workspace), ws_bytes, _stream_ptr(stream, dev))
    _check(rc, name)
    return out, lse


def sparse_mla_decode_fp8_noalloc(q, kv_cache, indices, block_table, req_id_per_token, sm_scale: float,
                                  num_splits: int = 0, out=None, lse=None, stream=None):
    """sparse_mla_decode_fp8 for callers that cannot allocate device memory
    at call time (code under CUDA graph capture, allocation-free serving
    loops): the library's fixed 32 MiB per-device scratch replaces the
    workspace.  Pass preallocated `out` and `lse` to keep the call free of
    allocations on the Python side too.  The first call on a device should
    come before any stream capture; calls that overlap on the GPU race on the
    shared scratch.  Raises SmlaError if the work split needs more scratch."""
    import torch
    dev = _dev(q, kv_cache, indices, block_table, req_id_per_token, out, lse)
    T, H, D = q.shape
    NB = kv_cache.shape[0]
    K = indices.shape[1]
    R, MB = block_table.shape
    _expect(q, torch.bfloat16, (T, H, 576), "q")
    _expect(kv_cache, torch.uint8, (NB, 64, 656), "kv_cache")
    _expect(indices, torch.int32, (T, K), "indices")
    _expect(req_id_per_token, torch.int32, (T,), "req_id_per_token")
    if block_table.dtype != torch.int32:
        raise SmlaError("block_table must be int32")
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    _expect(out, torch.bfloat16, (T, H, 512), "out")
    _expect(lse, torch.float32, (T, H), "lse")
    rc = lib().sparse_mla_decode_fp8_noalloc(_ptr(q), _ptr(kv_cache), _ptr(indices), _ptr(block_table),
                                             _ptr(req_id_per_token), float(sm_scale), int(num_splits), _ptr(out),
                                             _ptr(lse), T, H, K, R, MB, NB, _stream_ptr(stream, dev))
    _check(rc, "sparse_mla_decode_fp8_noalloc")
    return out, lse


def sparse_mla_prefill_bf16(q, kv, indices, sm_scale: float, num_splits: int = 0, out=None, lse=None,
                            workspace=None, stream=None):
    """BF16 sparse prefill.  q bf16 [T,H,576]; kv bf16 [N,576]; indices int32
    [T,K] rows of kv (<0 or >=N = none).  Returns (out, lse)."""
    import torch
    dev = _dev(q, kv, indices, out, lse, workspace)
    T, H, D = q.shape
    N = kv.shape[0]
    K = indices.shape[1]
    _expect(q, torch.bfloat16, (T, H, 576), "q")
    _expect(kv, torch.bfloat16, (N, 576), "kv")
    _expect(indices, torch.int32, (T, K), "indices")
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    _expect(out, torch.bfloat16, (T, H, 512), "out")
    _expect(lse, torch.float32, (T, H), "lse")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().sparse_mla_prefill_bf16(_ptr(q), _ptr(kv), _ptr(indices), float(sm_scale), int(num_splits),
                                       _ptr(out), _ptr(lse), T, H, N, K, _ptr(workspace), ws_bytes,
                                       _stream_ptr(stream, dev))
    _check(rc, "sparse_mla_prefill_bf16")
    return out, lse


def prefill_fp8_workspace_bytes(T: int, H: int, K: int, num_splits: int = 0) -> int:
    return int(lib().sparse_mla_prefill_fp8_workspace_bytes(T, H, K, num_splits))


def sparse_mla_prefill_fp8(q, kv_cache, indices, block_table, req_id_per_token, seq_lens, workspace_starts,
                           kv_workspace, sm_scale: float, num_splits: int = 0, out=None, lse=None, workspace=None,
                           stream=None):
    """Separate-mode FP8 prefill of one chunk of prefill requests: the
    requests' cache rows up-converted into kv_workspace (bf16 [N, 576]), the
    logical indices mapped to its rows, then the bf16 prefill.  q bf16
    [T,H,576]; kv_cache uint8 [NB,64,656]; indices int32 [T,K]; block_table
    int32 [R,MB]; req_id_per_token int32 [T]; seq_lens, workspace_starts int32
    [R].  Returns (out bf16 [T,H,512], lse fp32 [T,H])."""
    import torch
    dev = _dev(q, kv_cache, indices, block_table, req_id_per_token, seq_lens, workspace_starts, kv_workspace, out,
               lse, workspace)
    T, H, _ = q.shape
    NB = kv_cache.shape[0]
    K = indices.shape[1]
    R, MB = block_table.shape
    N = kv_workspace.shape[0]
    _expect(q, torch.bfloat16, (T, H, 576), "q")
    _expect(kv_cache, torch.uint8, (NB, 64, 656), "kv_cache")
    _expect(indices, torch.int32, (T, K), "indices")
    _expect(req_id_per_token, torch.int32, (T,), "req_id_per_token")
    _expect(seq_lens, torch.int32, (R,), "seq_lens")
    _expect(workspace_starts, torch.int32, (R,), "workspace_starts")
    _expect(kv_workspace, torch.bfloat16, (N, 576), "kv_workspace")
    if block_table.dtype != torch.int32:
        raise SmlaError("block_table must be int32")
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    _expect(out, torch.bfloat16, (T, H, 512), "out")
    _expect(lse, torch.float32, (T, H), "lse")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().sparse_mla_prefill_fp8(_ptr(q), _ptr(kv_cache), _ptr(indices), _ptr(block_table),
                                      _ptr(req_id_per_token), _ptr(seq_lens), _ptr(workspace_starts),
                                      float(sm_scale), int(num_splits), _ptr(out), _ptr(lse), T, H, K, R, MB, NB,
                                      _ptr(kv_workspace), N, _ptr(workspace), ws_bytes, _stream_ptr(stream, dev))
    _check(rc, "sparse_mla_prefill_fp8")
    return out, lse


def sparse_mla_gather_upconvert_fp8(kv_cache, block_table, seq_lens, workspace_starts, kv_workspace, stream=None):
    """Up-convert positions 0 .. seq_lens[r] - 1 of each request into
    kv_workspace (bf16 [N, 576]) rows workspace_starts[r] + p."""
    import torch
    dev = _dev(kv_cache, block_table, seq_lens, workspace_starts, kv_workspace)
    R, MB = block_table.shape
    _expect(kv_workspace, torch.bfloat16, (kv_workspace.shape[0], 576), "kv_workspace")
    rc = lib().sparse_mla_gather_upconvert_fp8(_ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
                                               _ptr(workspace_starts), R, MB, kv_cache.shape[0], _ptr(kv_workspace),
                                               kv_workspace.shape[0], _stream_ptr(stream, dev))
    _check(rc, "sparse_mla_gather_upconvert_fp8")
    return kv_workspace


def sparse_mla_translate_indices_workspace(indices, block_table, req_id_per_token, prefill_request_id,
                                           workspace_starts, num_blocks: int, out=None, stream=None):
    """Logical top-k indices -> cache slots (decode tokens) or prefill
    workspace rows (prefill tokens), int32 [T, K], -1 = none."""
    import torch
    dev = _dev(indices, block_table, req_id_per_token, prefill_request_id, workspace_starts, out)
    T, K = indices.shape
    R, MB = block_table.shape
    if out is None:
        out = torch.empty((T, K), dtype=torch.int32, device=dev)
    rc = lib().sparse_mla_translate_indices_workspace(_ptr(indices), _ptr(block_table), _ptr(req_id_per_token),
                                                      _ptr(prefill_request_id), _ptr(workspace_starts),
                                                      workspace_starts.numel(), _ptr(out), T, K, R, MB,
                                                      int(num_blocks), _stream_ptr(stream, dev))
    _check(rc, "sparse_mla_translate_indices_workspace")
    return out


def sparse_mla_prefill_chunks(seq_lens, workspace_rows: int):
    """Host-side chunking of prefill requests (a sequence of ints) into
    workspaces of ``workspace_rows`` rows: returns (list of (start, end)
    request ranges, list of chunk-local workspace starts)."""
    R = len(seq_lens)
    sl = (ctypes.c_int32 * max(R, 1))(*[int(v) for v in seq_lens])
    ends = (ctypes.c_int32 * max(R, 1))()
    starts = (ctypes.c_int32 * max(R, 1))()
    n = ctypes.c_int32(0)
    _check(lib().sparse_mla_prefill_chunks(ctypes.cast(sl, ctypes.c_void_p), R, int(workspace_rows),
                                           ctypes.cast(ends, ctypes.c_void_p), ctypes.cast(starts, ctypes.c_void_p),
                                           ctypes.byref(n)), "sparse_mla_prefill_chunks")
    bounds, b = [], 0
    for i in range(n.value):
        bounds.append((b, int(ends[i])))
        b = int(ends[i])
    return bounds, [int(starts[i]) for i in range(R)]


def mla_absorb_q(q, w_uk_t, out=None, workspace=None, stream=None):
    """Attention-ready query from q bf16 [T,H,P+64] and W_UK_T bf16 [H,P,512]:
    bf16 [T,H,576] = (q_nope x W_UK_T per head) ++ q_pe."""
    import torch
    dev = _dev(q, w_uk_t, out, workspace)
    T, H, D = q.shape
    P = D - 64
    _expect(w_uk_t, torch.bfloat16, (H, P, 512), "w_uk_t")
    if q.dtype != torch.bfloat16:
        raise SmlaError("q must be bf16")
    if out is None:
        out = torch.empty((T, H, 576), dtype=torch.bfloat16, device=dev)
    _expect(out, torch.bfloat16, (T, H, 576), "out")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().mla_absorb_q(_ptr(q), _ptr(w_uk_t), _ptr(out), T, H, P, _ptr(workspace), ws_bytes,
                              _stream_ptr(stream, dev)), "mla_absorb_q")
    return out


def mla_v_up_proj(attn_out, w_uv, out=None, workspace=None, stream=None):
    """Per-head value up-projection: attn_out bf16 [T,H,512] x W_UV bf16
    [H,512,V] -> bf16 [T,H,V]."""
    import torch
    dev = _dev(attn_out, w_uv, out, workspace)
    T, H, _ = attn_out.shape
    V = w_uv.shape[2]
    _expect(attn_out, torch.bfloat16, (T, H, 512), "attn_out")
    _expect(w_uv, torch.bfloat16, (H, 512, V), "w_uv")
    if out is None:
        out = torch.empty((T, H, V), dtype=torch.bfloat16, device=dev)
    _expect(out, torch.bfloat16, (T, H, V), "out")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().mla_v_up_proj(_ptr(attn_out), _ptr(w_uv), _ptr(out), T, H, V, _ptr(workspace), ws_bytes,
                               _stream_ptr(stream, dev)), "mla_v_up_proj")
    return out


def mla_cache_store_fp8(kv_new, slot_mapping, kv_cache, stream=None):
    """Quantize bf16 [T,576] rows into kv_cache uint8 [NB,64,656] at
    slot_mapping int64 [T] (<0 skips).  Modifies kv_cache in place."""
    import torch
    dev = _dev(kv_new, slot_mapping, kv_cache)
    T = kv_new.shape[0]
    NB = kv_cache.shape[0]
    _expect(kv_new, torch.bfloat16, (T, 576), "kv_new")
    _expect(slot_mapping, torch.int64, (T,), "slot_mapping")
    _expect(kv_cache, torch.uint8, (NB, 64, 656), "kv_cache")
    rc = lib().mla_cache_store_fp8(_ptr(kv_new), _ptr(slot_mapping), _ptr(kv_cache), T, NB, _stream_ptr(stream, dev))
    _check(rc, "mla_cache_store_fp8")
    return kv_cache


def mla_cache_store_nvfp4(kv_new, slot_mapping, kv_cache, stream=None):
    """Quantize bf16 [T,576] rows into the NVFP4 kv_cache uint8 [NB,64,352] at
    slot_mapping int64 [T] (<0 skips).  Modifies kv_cache in place."""
    import torch
    dev = _dev(kv_new, slot_mapping, kv_cache)
    T = kv_new.shape[0]
    NB = kv_cache.shape[0]
    _expect(kv_new, torch.bfloat16, (T, 576), "kv_new")
    _expect(slot_mapping, torch.int64, (T,), "slot_mapping")
    _expect(kv_cache, torch.uint8, (NB, 64, 352), "kv_cache")
    rc = lib().mla_cache_store_nvfp4(_ptr(kv_new), _ptr(slot_mapping), _ptr(kv_cache), T, NB, _stream_ptr(stream, dev))
    _check(rc, "mla_cache_store_nvfp4")
    return kv_cache


def sparse_mla_translate_indices(indices, block_table, req_id_per_token, num_blocks: int, out=None, stream=None):
    """Logical top-k indices -> physical cache slots (int32 [T,K], -1 = none)."""
    import torch
    dev = _dev(indices, block_table, req_id_per_token, out)
    T, K = indices.shape
    R, MB = block_table.shape
    if out is None:
        out = torch.empty((T, K), dtype=torch.int32, device=dev)
    rc = lib().sparse_mla_translate_indices(_ptr(indices), _ptr(block_table), _ptr(req_id_per_token), _ptr(out),
                                            T, K, R, MB, int(num_blocks), _stream_ptr(stream, dev))
    _check(rc, "sparse_mla_translate_indices")
    return out


def read_noalloc_status(stream=None) -> int:
    """Synchronize and read/clear the status word of the allocation-free
    decode's fixed scratch on the current device (0 = ok)."""
    import torch
    st = ctypes.c_int(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    _check(lib().smla_read_noalloc_status(ctypes.byref(st), _stream_ptr(stream, dev)), "smla_read_noalloc_status")
    return int(st.value)


def read_device_status(workspace=None, stream=None) -> int:
    """Synchronize and read/clear the kernels' device status word (0 = ok)."""
    import torch
    st = ctypes.c_int(0)
    dev = workspace.device if workspace is not None else torch.device("cuda", torch.cuda.current_device())
    rc = lib().smla_read_device_status(_ptr(workspace), ctypes.byref(st), _stream_ptr(stream, dev))
    _check(rc, "smla_read_device_status")
    return int(st.value)
