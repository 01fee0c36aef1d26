"""Per-tile timelines of the FP8 decode kernels, for performance work.

Builds a separate traced copy of the library (all sources compiled with
SMLA_TRACE, in ``_build_trace/``), runs the memory-bound decode workload
(64 requests x 1 token, H = 16, top-k 2048) a few times, then once with the
trace buffer attached, and prints per-tile timings taken from %globaltimer at
the kernel roles' hand-off points (median over CTAs, microseconds from the
CTA's first index translation); with --wide, the same for the 128-head
CTA-pair kernel on its tensor-bound workload (clock64 cycles within a CTA):

    python -m sparse_mla_attention_fp8_gb300.trace
    python -m sparse_mla_attention_fp8_gb300.trace --wide   # the 128-head FP8 decode
    python -m sparse_mla_attention_fp8_gb300.trace --wide-prefill  # the 128-head bf16 prefill
    python -m sparse_mla_attention_fp8_gb300.trace --wide8  # its FP8-query variant
    python -m sparse_mla_attention_fp8_gb300.trace --nvfp4  # the NVFP4 decode (16-head groups)

The normal library (``libsmla.so``) carries none of this: the hooks compile
to nothing without SMLA_TRACE.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

from . import NVCC_FLAGS, SOURCES, _CSRC, _PKG, _nvcc

EVENTS = ["idx", "buf_free", "issued", "landed", "op_full", "qk", "soft_start", "soft_bar", "p_written", "pv",
          "epilogue", "q_ready", "epi_start", "merge_wait", "merge_go", "enter", "exit", "epi_lse", "epi_signal",
          "epi_ready", "epi_sent", "epi_written", "setup"]
# per-tile links: (name, from event, to event, tile offset of the end event)
LINKS = [("copy issue (loader 0)", "buf_free", "issued", 0), ("copy landing (loader 0)", "issued", "landed", 0),
         ("other loaders after loader 0", "landed", "op_full", 0), ("QK^T issue", "op_full", "qk", 0),
         ("S ready after issue", "qk", "soft_start", 0), ("softmax to tile-max barrier", "soft_start", "soft_bar", 0),
         ("softmax barrier to P' (warp 0)", "soft_bar", "p_written", 0), ("P' (warp 0) to P.V issued", "p_written", "pv", 0),
         ("P.V issued to code panel 0 free (tile + 2)", "pv", "buf_free", 2), ("Q ready to tile full", "q_ready", "op_full", 0),
         ("last P.V issued to epilogue start", "pv", "epi_start", 0),
         ("epilogue start to merge wait", "epi_start", "merge_wait", 0),
         ("merge wait (other CTA)", "merge_wait", "merge_go", 0), ("merge to epilogue end", "merge_go", "epilogue", 0)]
TILES = 16


def build_traced(csrc: str = _CSRC, out_dir: str | None = None) -> str:
    """Compile the sources in ``csrc`` with SMLA_TRACE into ``out_dir``."""
    out_dir = out_dir or os.path.join(_PKG, "_build_trace")
    os.makedirs(out_dir, exist_ok=True)
    objs = []
    for s in SOURCES:
        obj = os.path.join(out_dir, s.replace(".cu", ".o"))
        subprocess.run([_nvcc(), *NVCC_FLAGS, "-DSMLA_TRACE", "-c", os.path.join(csrc, s), "-o", obj], check=True)
        objs.append(obj)
    lib = os.path.join(out_dir, "libsmla_trace.so")
    subprocess.run([_nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", lib], check=True)
    return lib


def main(lib_path: str | None = None):
    import torch

    root = os.path.dirname(_PKG)
    if root not in sys.path:
        sys.path.insert(0, root)
    import smla_inputs as inp

    L = ctypes.CDLL(lib_path or build_traced())
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.sparse_mla_decode_fp8.argtypes = [P, P, P, P, P, f32, i32, P, P, i32, i32, i32, i32, i32, i32, P, sz, P]
    L.mla_cache_store_fp8.argtypes = [P, P, P, i32, i32, P]
    L.sparse_mla_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.sparse_mla_decode_workspace_bytes.restype = sz
    L.sparse_mla_attention_plan.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.smla_trace_set_fp8.argtypes = [P]
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    dev = torch.device("cuda", 0)
    case = inp.rotating_decode(seed=1)
    T, H, K, NB = case.q.shape[0], case.H, case.K, case.num_blocks
    cache = torch.zeros((NB, 64, 656), dtype=torch.uint8, device=dev)
    lat = inp.device_latent(len(case.ctx_slots), case.latent_seed, case.outlier_channels, dev)
    slots = torch.from_numpy(case.ctx_slots).to(dev)
    assert L.mla_cache_store_fp8(ptr(lat), ptr(slots), ptr(cache), lat.shape[0], NB, None) == 0
    q = torch.from_numpy(case.q.view(np.int16)).to(dev)
    idx = [torch.from_numpy(s).to(dev) for s in case.index_sets]
    bt = torch.from_numpy(case.block_table).to(dev)
    req = torch.from_numpy(case.req_id_per_token).to(dev)
    ws_bytes = L.sparse_mla_decode_workspace_bytes(T, H, K, 0)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    launches, ctas = ctypes.c_int(0), ctypes.c_int(0)
    L.sparse_mla_attention_plan(1, T, H, K, 0, ctypes.byref(launches), ctypes.byref(ctas))
    G = ctas.value
    buf = torch.zeros((G, TILES, len(EVENTS)), dtype=torch.int64, device=dev)

    def call(i):
        rc = L.sparse_mla_decode_fp8(ptr(q), ptr(cache), ptr(idx[i % len(idx)]), ptr(bt), ptr(req),
                                     f32(case.sm_scale), 0, ptr(out), ptr(lse), T, H, K, bt.shape[0], bt.shape[1],
                                     NB, ptr(ws), ws_bytes, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0

    for i in range(5):
        call(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(40):
        call(i)
    e1.record()
    torch.cuda.synchronize()
    print(f"decode call (attention + combine), eager, rotating index sets: {e0.elapsed_time(e1) / 40 * 1e3:.1f} us")
    assert L.smla_trace_set_fp8(ptr(buf)) == 0
    call(5)
    torch.cuda.synchronize()
    assert L.smla_trace_set_fp8(None) == 0
    ev = buf.cpu().numpy().astype(np.float64)
    t0 = np.where(ev[:, 0, 0] > 0, ev[:, 0, 0], np.nan)
    start = np.nanmin(t0[np.isfinite(t0)])
    rel = np.where(ev > 0, (ev - start) / 1e3, np.nan)  # microseconds from the first CTA's first translation
    print(f"CTAs {G}; first index translation spread over CTAs: {np.nanmax(t0 - start) / 1e3:.2f} us")
    print("median over CTAs, us from the earliest CTA start; columns = tiles")
    print("event        " + " ".join(f"{t:6d}" for t in range(TILES)))
    for e, name in enumerate(EVENTS):
        med = np.nanmedian(rel[:, :, e], axis=0)
        print(f"{name:12s} " + " ".join("   -  " if np.isnan(x) else f"{x:6.2f}" for x in med))
    print("per-tile links, median over CTAs and tiles (us):")
    for name, a, b, off in LINKS:
        ea, eb = rel[:, :, EVENTS.index(a)], rel[:, :, EVENTS.index(b)]
        d = eb[:, off:] - ea[:, :TILES - off]
        if np.isfinite(d).any():
            print(f"  {name:38s} {np.nanmedian(d):6.2f}  (p90 {np.nanpercentile(d, 90):5.2f}, n {np.isfinite(d).sum()})")
    pv = rel[:, :, EVENTS.index("pv")]
    last = np.nanmax(pv, axis=1)
    print(f"last P.V issued: min {np.nanmin(last):.2f} median {np.nanmedian(last):.2f} max {np.nanmax(last):.2f} us")
    d = np.diff(pv, axis=1)
    print(f"P.V cadence: median {np.nanmedian(d):.2f} us (p10 {np.nanpercentile(d, 10):.2f}, "
          f"p90 {np.nanpercentile(d, 90):.2f})")
    enter, ex = rel[:, 0, EVENTS.index("enter")], rel[:, 0, EVENTS.index("exit")]
    if G == 2 * T:  # clusters of two (ranks 0 and 1 alternate)
        for name, sel in (("rank 0", slice(0, G, 2)), ("rank 1", slice(1, G, 2))):
            lastpv = np.nanmax(pv[sel], axis=1)
            cols = [("last P.V", lastpv)] + [(e, np.nanmax(rel[sel, :, EVENTS.index(e)], axis=1))
                                            for e in ("epi_start", "epi_lse", "epi_signal", "epi_ready", "epi_sent",
                                                      "merge_go", "merge_wait", "epi_written", "epilogue", "exit")]
            print(f"{name:8s} " + "  ".join(f"{n} {np.nanmedian(v):6.2f}" for n, v in cols))
    print(f"CTA entry: first {np.nanmin(enter):.2f} last {np.nanmax(enter):.2f} us; exit: first {np.nanmin(ex):.2f} "
          f"median {np.nanmedian(ex):.2f} last {np.nanmax(ex):.2f} us; first entry to last exit "
          f"{np.nanmax(ex) - np.nanmin(enter):.2f} us")
    setup = rel[:, 0, EVENTS.index("setup")]
    print(f"start-up (median over CTAs, us from the CTA's entry): set-up done {np.nanmedian(setup - enter):.2f}, "
          f"tile 0 translated {np.nanmedian(rel[:, 0, 0] - enter):.2f}, its copies issued "
          f"{np.nanmedian(rel[:, 0, EVENTS.index('issued')] - enter):.2f}, landed "
          f"{np.nanmedian(rel[:, 0, EVENTS.index('landed')] - enter):.2f}, first P.V {np.nanmedian(pv[:, 0] - enter):.2f}")
    # the same call timed alone and in CUDA graphs of 1 and 8 calls (no trace buffer)
    for n in (1, 8):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                call(i)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(40):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        print(f"decode call in CUDA graphs of {n}: {e0.elapsed_time(e1) / (40 * n) * 1e3:.1f} us per call")


WIDE_EVENTS = ["s_full", "s_loaded", "x_free", "sent", "x_full", "p_ready", "p_full", "qk", "pv", "issue", "qk_seen",
               "k_empty", "converted", "raw_full", "x_top", "x_k_full", "enter", "epi_start", "epi_end", "exit"]
WIDE_TILES = 64


def main_wide(lib_path: str | None = None):
    """Per-tile timeline of the 128-head FP8 decode (128 requests x 1 token,
    H = 128, top-k 2048, context 65536) from the CTA-pair kernel's clock64()
    marks: cycles within each CTA (SM clocks are not comparable across SMs)."""
    import torch

    root = os.path.dirname(_PKG)
    if root not in sys.path:
        sys.path.insert(0, root)
    import smla_inputs as inp

    L = ctypes.CDLL(lib_path or build_traced())
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.sparse_mla_decode_fp8.argtypes = [P, P, P, P, P, f32, i32, P, P, i32, i32, i32, i32, i32, i32, P, sz, P]
    L.mla_cache_store_fp8.argtypes = [P, P, P, i32, i32, P]
    L.sparse_mla_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.sparse_mla_decode_workspace_bytes.restype = sz
    L.sparse_mla_attention_plan.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.smla_trace_set_wide.argtypes = [P]
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    dev = torch.device("cuda", 0)
    case = inp.rotating_decode(seed=2, R=128, ctx_lo=65536, ctx_hi=65536, K=2048, H=128, outliers=True)
    T, H, K, NB = case.q.shape[0], case.H, case.K, case.num_blocks
    cache = torch.zeros((NB, 64, 656), dtype=torch.uint8, device=dev)
    lat = inp.device_latent(len(case.ctx_slots), case.latent_seed, case.outlier_channels, dev)
    slots = torch.from_numpy(case.ctx_slots).to(dev)
    assert L.mla_cache_store_fp8(ptr(lat), ptr(slots), ptr(cache), lat.shape[0], NB, None) == 0
    del lat
    q = torch.from_numpy(case.q.view(np.int16)).to(dev)
    idx = [torch.from_numpy(s).to(dev) for s in case.index_sets]
    bt = torch.from_numpy(case.block_table).to(dev)
    req = torch.from_numpy(case.req_id_per_token).to(dev)
    ws_bytes = L.sparse_mla_decode_workspace_bytes(T, H, K, 0)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    launches, ctas = ctypes.c_int(0), ctypes.c_int(0)
    L.sparse_mla_attention_plan(1, T, H, K, 0, ctypes.byref(launches), ctypes.byref(ctas))
    G = ctas.value
    buf = torch.zeros((G, WIDE_TILES, len(WIDE_EVENTS)), dtype=torch.int64, device=dev)

    def call(i):
        rc = L.sparse_mla_decode_fp8(ptr(q), ptr(cache), ptr(idx[i % len(idx)]), ptr(bt), ptr(req),
                                     f32(case.sm_scale), 0, ptr(out), ptr(lse), T, H, K, bt.shape[0], bt.shape[1],
                                     NB, ptr(ws), ws_bytes, None)
        assert rc == 0

    for i in range(4):
        call(i)
    torch.cuda.synchronize()
    assert L.smla_trace_set_wide(ptr(buf)) == 0
    call(4)
    torch.cuda.synchronize()
    assert L.smla_trace_set_wide(None) == 0
    _wide_report(buf, G, launches.value)

def _wide_report(buf, G, n_launches):
    """Timeline summary of a traced call of the CTA-pair kernel (main_wide, main_wide_prefill)."""
    launches = ctypes.c_int(n_launches)
    ev = buf.cpu().numpy().astype(np.float64)
    ev[ev == 0] = np.nan
    E = {n: ev[:, :, i] for i, n in enumerate(WIDE_EVENTS)}
    kc = lambda x: f"{np.nanmedian(x) / 1e3:7.2f}"  # noqa: E731
    print(f"CTAs {G} ({G // 2} pairs), {launches.value} launches per call; clock64 cycles within each CTA (K = 1000)")
    print("event position in its tile relative to the tile's QK^T issue (median K cycles):")
    for n in WIDE_EVENTS[:16]:
        d = E[n] - E["qk"]
        if np.isfinite(d).any():
            print(f"  {n:10s} {kc(d)}")
    pv = E["pv"]
    n_t = np.sum(np.isfinite(pv), axis=1)
    seg_first = np.isfinite(E["epi_start"])  # a segment ends at this tile
    d = np.diff(pv, axis=1)
    cross = seg_first[:, :-1]  # the step from a segment's last tile to the next segment's first
    print(f"P.V cadence inside a segment: {kc(d[~cross])} K cycles; across a segment boundary: {kc(d[cross])}")
    print(f"segment epilogue (start -> end): {kc(E['epi_end'] - E['epi_start'])} K cycles; "
          f"segments per CTA: {np.nanmedian(np.sum(seg_first, axis=1)):.1f}, tiles per CTA {np.median(n_t):.0f}")
    # epilogue by segment kind: a CTA's first segment starts mid-token (the
    # token's second part) except in the first pair, its last ends mid-token
    # (first part, merged there) except in the last pair, the others are whole
    kinds = {"second part (publishes)": [], "whole token": [], "first part (merges)": []}
    for i in range(G):
        ends = np.where(np.isfinite(E["epi_start"][i]))[0]
        for j, t in enumerate(ends):
            dd = E["epi_end"][i, t] - E["epi_start"][i, t]
            if j == 0 and i >= 2:
                kinds["second part (publishes)"].append(dd)
            elif j == len(ends) - 1 and i < G - 2:
                kinds["first part (merges)"].append(dd)
            else:
                kinds["whole token"].append(dd)
    print("segment epilogue by kind (median K cycles): " +
          ", ".join(f"{k} {np.median(v) / 1e3:.2f}" for k, v in kinds.items() if v))
    enter, ex = E["enter"][:, 0], E["exit"][:, 0]
    first_pv = pv[:, 0]
    last_pv = np.array([row[np.isfinite(row)][-1] if np.isfinite(row).any() else np.nan for row in pv])
    print(f"entry -> first P.V {kc(first_pv - enter)}; last P.V -> exit {kc(ex - last_pv)}; "
          f"entry -> exit {kc(ex - enter)} K cycles")



def main_wide_prefill(lib_path: str | None = None):
    """Per-tile timeline of the 128-head bf16 prefill (4 requests x 1024 new
    tokens over 3072 cached, H = 128, top-k 2048, latent buffer [16384, 576])
    from the CTA-pair kernel's clock64() marks."""
    import torch

    root = os.path.dirname(_PKG)
    if root not in sys.path:
        sys.path.insert(0, root)
    import smla_inputs as inp

    L = ctypes.CDLL(lib_path or build_traced())
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.sparse_mla_prefill_bf16.argtypes = [P, P, P, f32, i32, P, P, i32, i32, i32, i32, P, sz, P]
    L.sparse_mla_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.sparse_mla_prefill_workspace_bytes.restype = sz
    L.sparse_mla_attention_plan.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.smla_trace_set_wide.argtypes = [P]
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    dev = torch.device("cuda", 0)
    case = inp.prefill(3)
    T, H, K = case.T, case.H, case.K
    N = case.kv.shape[0]
    q = torch.from_numpy(np.ascontiguousarray(case.q).view(np.int16)).to(dev)
    kv = torch.from_numpy(np.ascontiguousarray(case.kv).view(np.int16)).to(dev)
    idx = torch.from_numpy(case.indices).to(dev)
    ws_bytes = L.sparse_mla_prefill_workspace_bytes(T, H, K, 0)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    launches, ctas = ctypes.c_int(0), ctypes.c_int(0)
    L.sparse_mla_attention_plan(0, T, H, K, 0, ctypes.byref(launches), ctypes.byref(ctas))
    G = ctas.value
    buf = torch.zeros((G, WIDE_TILES, len(WIDE_EVENTS)), dtype=torch.int64, device=dev)

    def call():
        assert L.sparse_mla_prefill_bf16(ptr(q), ptr(kv), ptr(idx), f32(case.sm_scale), 0, ptr(out), ptr(lse), T, H,
                                         N, K, ptr(ws), ws_bytes, None) == 0

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert L.smla_trace_set_wide(ptr(buf)) == 0
    call()
    torch.cuda.synchronize()
    assert L.smla_trace_set_wide(None) == 0
    _wide_report(buf, G, launches.value)


WIDE8_EVENTS = ["idx", "kfull", "qk", "s_read", "sent", "received", "l_ready", "l_read", "pv_prev_done", "p_full",
                "pv", "load_issue", "k_empty", "epi_start", "epi_end", "enter", "exit", "q_full"]


def main_wide8(lib_path: str | None = None):
    """Per-tile timeline of the FP8-query 128-head decode (sparse_mla_decode_fp8_qfp8)
    on the tensor-bound workload: clock64 cycles within each CTA."""
    import torch

    root = os.path.dirname(_PKG)
    if root not in sys.path:
        sys.path.insert(0, root)
    import smla_inputs as inp

    L = ctypes.CDLL(lib_path or build_traced())
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.sparse_mla_decode_fp8_qfp8.argtypes = [P, P, P, P, P, f32, i32, P, P, i32, i32, i32, i32, i32, i32, P, sz, P]
    L.mla_cache_store_fp8.argtypes = [P, P, P, i32, i32, P]
    L.sparse_mla_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.sparse_mla_decode_workspace_bytes.restype = sz
    L.smla_trace_set_wide8.argtypes = [P]
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    dev = torch.device("cuda", 0)
    case = inp.rotating_decode(seed=2, R=128, ctx_lo=65536, ctx_hi=65536, K=2048, H=128, outliers=True)
    T, H, K, NB = case.q.shape[0], case.H, case.K, case.num_blocks
    cache = torch.zeros((NB, 64, 656), dtype=torch.uint8, device=dev)
    lat = inp.device_latent(len(case.ctx_slots), case.latent_seed, case.outlier_channels, dev)
    slots = torch.from_numpy(case.ctx_slots).to(dev)
    assert L.mla_cache_store_fp8(ptr(lat), ptr(slots), ptr(cache), lat.shape[0], NB, None) == 0
    del lat
    q = torch.from_numpy(case.q.view(np.int16)).to(dev)
    idx = [torch.from_numpy(s).to(dev) for s in case.index_sets]
    bt = torch.from_numpy(case.block_table).to(dev)
    req = torch.from_numpy(case.req_id_per_token).to(dev)
    ws_bytes = L.sparse_mla_decode_workspace_bytes(T, H, K, 0)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    buf = torch.zeros((n_sms, WIDE_TILES, len(WIDE8_EVENTS)), dtype=torch.int64, device=dev)

    def call(i):
        rc = L.sparse_mla_decode_fp8_qfp8(ptr(q), ptr(cache), ptr(idx[i % len(idx)]), ptr(bt), ptr(req),
                                          f32(case.sm_scale), 0, ptr(out), ptr(lse), T, H, K, bt.shape[0],
                                          bt.shape[1], NB, ptr(ws), ws_bytes, None)
        assert rc == 0

    for i in range(4):
        call(i)
    torch.cuda.synchronize()
    assert L.smla_trace_set_wide8(ptr(buf)) == 0
    call(4)
    torch.cuda.synchronize()
    assert L.smla_trace_set_wide8(None) == 0
    ev = buf.cpu().numpy().astype(np.float64)
    ev[ev == 0] = np.nan
    ev = ev[np.isfinite(ev[:, 0, WIDE8_EVENTS.index("enter")])]  # CTAs of the launch
    E = {n: ev[:, :, i] for i, n in enumerate(WIDE8_EVENTS)}
    kc = lambda x: f"{np.nanmedian(x) / 1e3:7.2f}"  # noqa: E731
    print(f"CTAs {ev.shape[0]}; clock64 cycles within each CTA (K = 1000), medians over CTAs and tiles")
    print("event position in its tile relative to the tile's QK^T issue:")
    for n in ["load_issue", "kfull", "q_full", "qk", "s_read", "sent", "received", "l_ready", "l_read",
              "pv_prev_done", "p_full", "pv"]:
        print(f"  {n:13s} {kc(E[n] - E['qk'])}")
    print(f"cadence (QK^T issue to the next): {kc(np.diff(E['qk'], axis=1))}; "
          f"P.V: {kc(np.diff(E['pv'], axis=1))}")
    print(f"exchange warps, one tile (l_ready to the next): {kc(np.diff(E['l_ready'], axis=1))}; "
          f"softmax, L read to P' written: {kc(E['p_full'] - E['l_read'])}")
    print(f"row gather, issue to full: {kc(E['kfull'] - E['load_issue'])}; "
          f"tile buffer free (P.V of tile t done) to reload (tile t + 4): {kc(E['k_empty'][:, 4:] - E['pv'][:, :-4])}")
    print(f"segment epilogue: {kc(E['epi_end'] - E['epi_start'])}")
    enter, ex = E["enter"][:, 0], E["exit"][:, 0]
    print(f"entry -> first QK^T {kc(E['qk'][:, 0] - enter)}; entry -> exit {kc(ex - enter)}")


ATTN_EVENTS = ["idx", "conv_issue", "conv_full", "qk", "soft_start", "soft_bar", "p_full", "pv", "epi_end", "enter",
               "exit", "pv_wait", "conv_start", "conv_row3", "conv_landed"]


def main_nvfp4(lib_path: str | None = None):
    """Per-tile timeline of the NVFP4 decode (the 16-head-group kernel of
    smla_attn.cu with NVFP4 rows) on the memory-bound decode's workload (64
    requests x 1 token, H = 16, top-k 2048): clock64 cycles within each CTA."""
    import torch

    root = os.path.dirname(_PKG)
    if root not in sys.path:
        sys.path.insert(0, root)
    import smla_inputs as inp

    L = ctypes.CDLL(lib_path or build_traced())
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.sparse_mla_decode_nvfp4.argtypes = [P, P, P, P, P, f32, i32, P, P, i32, i32, i32, i32, i32, i32, P, sz, P]
    L.mla_cache_store_nvfp4.argtypes = [P, P, P, i32, i32, P]
    L.sparse_mla_decode_nvfp4_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.sparse_mla_decode_nvfp4_workspace_bytes.restype = sz
    L.smla_trace_set_attn.argtypes = [P]
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    dev = torch.device("cuda", 0)
    case = inp.rotating_decode(seed=1)
    T, H, K, NB = case.q.shape[0], case.H, case.K, case.num_blocks
    cache = torch.zeros((NB, 64, 352), dtype=torch.uint8, device=dev)
    lat = inp.device_latent(len(case.ctx_slots), case.latent_seed, case.outlier_channels, dev)
    slots = torch.from_numpy(case.ctx_slots).to(dev)
    assert L.mla_cache_store_nvfp4(ptr(lat), ptr(slots), ptr(cache), lat.shape[0], NB, None) == 0
    del lat
    q = torch.from_numpy(case.q.view(np.int16)).to(dev)
    idx = [torch.from_numpy(s).to(dev) for s in case.index_sets]
    bt = torch.from_numpy(case.block_table).to(dev)
    req = torch.from_numpy(case.req_id_per_token).to(dev)
    ws_bytes = L.sparse_mla_decode_nvfp4_workspace_bytes(T, H, K, 0)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    buf = torch.zeros((n_sms, WIDE_TILES, len(ATTN_EVENTS)), dtype=torch.int64, device=dev)

    def call(i):
        rc = L.sparse_mla_decode_nvfp4(ptr(q), ptr(cache), ptr(idx[i % len(idx)]), ptr(bt), ptr(req),
                                       f32(case.sm_scale), 0, ptr(out), ptr(lse), T, H, K, bt.shape[0], bt.shape[1],
                                       NB, ptr(ws), ws_bytes, None)
        assert rc == 0

    for i in range(4):
        call(i)
    torch.cuda.synchronize()
    assert L.smla_trace_set_attn(ptr(buf)) == 0
    call(4)
    torch.cuda.synchronize()
    assert L.smla_trace_set_attn(None) == 0
    ev = buf.cpu().numpy().astype(np.float64)
    ev[ev == 0] = np.nan
    ev = ev[np.isfinite(ev[:, 0, ATTN_EVENTS.index("enter")])]
    E = {n: ev[:, :, i] for i, n in enumerate(ATTN_EVENTS)}
    kc = lambda x: f"{np.nanmedian(x) / 1e3:7.2f}"  # noqa: E731
    print(f"CTAs {ev.shape[0]}; clock64 cycles within each CTA (K = 1000), medians over CTAs and tiles")
    print("event position in its tile relative to the tile's QK^T issue:")
    for n in ["idx", "conv_issue", "conv_landed", "conv_start", "conv_full", "qk", "soft_start", "soft_bar",
              "pv_wait", "p_full", "pv"]:
        print(f"  {n:11s} {kc(E[n] - E['qk'])}")
    print(f"cadence (QK^T to QK^T): {kc(np.diff(E['qk'], axis=1))}; P.V: {kc(np.diff(E['pv'], axis=1))}; "
          f"converter full: {kc(np.diff(E['conv_full'], axis=1))}; softmax P written: {kc(np.diff(E['p_full'], axis=1))}")
    print(f"converter warp 0: tile buffer free after P.V(t - 2) issue {kc(E['conv_start'][:, 2:] - E['pv'][:, :-2])}; "
          f"conversion (buffer free to tile full) {kc(E['conv_full'] - E['conv_start'])}")
    print(f"converter, first issue to full: {kc(E['conv_full'] - E['conv_issue'])}; "
          f"tile t + 2 full after P.V of tile t: {kc(E['conv_full'][:, 2:] - E['pv'][:, :-2])}")
    enter, ex = E["enter"][:, 0], E["exit"][:, 0]
    print(f"entry -> first QK^T {kc(E['qk'][:, 0] - enter)}; entry -> exit {kc(ex - enter)}")


if __name__ == "__main__":
    if "--nvfp4" in sys.argv:
        main_nvfp4()
    elif "--wide8" in sys.argv:
        main_wide8()
    elif "--wide-prefill" in sys.argv:
        main_wide_prefill()
    elif "--wide" in sys.argv:
        main_wide()
    else:
        main()
