#!/usr/bin/env python
"""Benchmark: sparse MLA decode throughput over the 656-byte FP8 cache.

Default workload (one step = the whole decode hot path over one batch):
  64 requests x 1 query token, H = 16 heads, top-k = 2048, per-request
  context uniform in [8192, 32768], block size 64, shuffled block table,
  latent N(0,1) with 1% of the channels x8, quantized into the FP8 cache.
  A step is: quantize-and-store of the 64 new tokens' rows, then the sparse
  decode (index translation, row gather + dequantization, QK^T, online
  softmax, P.V, split combine).  Eight independent top-k index sets rotate
  from step to step, so each step gathers ~86 MB of rows that were not just
  read (8 x 86 MB >> 129 MB of L2).

Prints one JSON line (rank 0).  --impl reference times the float64 CPU
oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import smla_inputs as inp  # noqa: E402

METRIC = "sparse MLA decode query-tokens/s + HBM GB/s (H=16, topk=2048) vs roofline"
UNIT = "query-tokens/s"


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one decode
# launch, from an ncu capture of the kernels built from the sources whose
# hash is the key: the attention kernel plus, where units are split across
# CTAs outside a cluster, the combine.  Once the kernel sources change, the
# figure no longer applies and the roofline reports null.
TRAFFIC_SOURCES = ("smla_decode.cu", "smla_combine.cuh", "smla_common.cuh", "sm103_ptx.cuh")
TRAFFIC_BY_SOURCE = {
    # 128-row tiles refilled panel by panel, two-part clusters merged from raw sums by one bulk copy
    # (writes vary 0.09 - 2.3 MB between launches with the L2's write-back; the middle one)
    "936d956d040f5ef2": 100_892_416 + 253_952,
    "5dc4295d6b49c62c": 100_892_416 + 253_952,  # re-keyed: a comment of the same kernel rewritten
}
# The same for the 128-head CTA-pair kernel, per workload: the bf16 prefill's
# attention kernel plus its combine; the FP8 decode's attention kernel, which
# merges its split tokens itself (the Q preparation, 18.9 MB, is left out).
WIDE_TRAFFIC_SOURCES = ("smla_wide.cu", "smla_combine.cuh", "smla_common.cuh", "sm103_ptx.cuh")
WIDE_TRAFFIC_BY_SOURCE = {
    ("f1d467be26141655", "prefill_h128_k2048"): (672_552_192 + 528_722_432 + 37_843_456 + 123_392,
                                                 "attention kernel + combine"),
    ("f1d467be26141655", "decode_h128_k2048"): (250_082_048 + 20_681_472, "attention kernel (merges its split tokens)"),
    # re-keyed: the shared header gained a helper that only the 16-head decode uses; these kernels are unchanged
    ("ad3021e155c41e5f", "prefill_h128_k2048"): (672_552_192 + 528_722_432 + 37_843_456 + 123_392, "attention kernel + combine"),
    ("ad3021e155c41e5f", "decode_h128_k2048"): (250_082_048 + 20_681_472, "attention kernel (merges its split tokens)"),
}


# The same for the NVFP4 decode (the 16-head-group kernel with NVFP4 rows,
# plus the combine of tokens split between CTAs).
NVFP4_TRAFFIC_SOURCES = ("smla_attn.cu", "smla_combine.cuh", "smla_common.cuh", "sm103_ptx.cuh")
NVFP4_TRAFFIC_BY_SOURCE = {
    "d63690ea74b7e5b2": (59_163_648 + 14_848 + 6_849_024, "attention kernel + combine"),
    # re-keyed: the shared header gained a helper that only the 16-head decode uses; this kernel is unchanged
    "44d0ca0de63d94b5": (59_163_648 + 14_848 + 6_849_024, "attention kernel + combine"),
}


# The same for the separate-mode FP8 prefill (gather + up-convert, workspace
# translation, the 128-head bf16 kernel, the combine: one step) and for the
# two weight-absorption GEMM launches of one step.
PREFILL_FP8_TRAFFIC_SOURCES = ("smla_store.cu", "smla_wide.cu", "smla_combine.cuh", "smla_common.cuh", "sm103_ptx.cuh")
PREFILL_FP8_TRAFFIC_BY_SOURCE = {
    "6884e8a0cd6030d4": (10_755_584 + 33_576_704 + 180_224 + 672_449_536 + 528_017_920 + 37_842_176 + 112_640,
              "gather + up-convert, translation, attention kernel, combine"),
    # re-keyed: the quantize-and-store kernel of the same file changed; this step's kernels did not
    "a6a9548cdc5f94ae": (10_755_584 + 33_576_704 + 180_224 + 672_449_536 + 528_017_920 + 37_842_176 + 112_640,
                         "gather + up-convert, translation, attention kernel, combine"),
}
ABSORB_TRAFFIC_SOURCES = ("smla_absorb.cu", "sm103_ptx.cuh")
ABSORB_TRAFFIC_BY_SOURCE = {
    "34ee1d10223418ff": (218_148_608 + 543_458_048 + 553_696_000 + 111_604_480, "both head_gemm launches"),
}


def _source_key(files):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_mla_attention_fp8_gb300", "csrc")
    try:
        for f in files:
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    return h.hexdigest()[:16]


def captured_traffic():
    return TRAFFIC_BY_SOURCE.get(_source_key(TRAFFIC_SOURCES))


def captured_wide_traffic(workload):
    return WIDE_TRAFFIC_BY_SOURCE.get((_source_key(WIDE_TRAFFIC_SOURCES), workload), (None, None))


# ---------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="smla_clocks_", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[4:8], float(parts[8])))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_under_load": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        busy = [r for r in rows if r[4] >= 50.0]  # samples while the GPU was busy
        use = busy or rows
        return {"sm_mhz": statistics.median(r[0] for r in use), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "reasons": reasons, "samples": len(rows),
                "samples_under_load": len(busy)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def decode_algorithmic_bytes(case: inp.RotatingDecode, index_set: np.ndarray, row_bytes: int = 656) -> int:
    """Bytes one decode launch must move at minimum: every valid gathered row
    once per query token (656 B, or 352 B for the NVFP4 cache), q, out, lse,
    the index row, the request id and the used part of the request's
    block-table row."""
    T, H = case.q.shape[0], case.H
    rows = int((index_set >= 0).sum())
    used_blocks = int(((case.ctx_lens + 63) // 64).sum())  # block-table entries read (one request per token)
    return (rows * row_bytes + T * H * 576 * 2 + T * H * 512 * 2 + T * H * 4 + index_set.size * 4 + T * 4
            + used_blocks * 4)


def decode_flops(case, index_set) -> int:
    return 2 * case.H * int((index_set >= 0).sum()) * (576 + 512)


# ---------------------------------------------------------------- CPU oracle sample

def host_sample_cache(case: inp.RotatingDecode, index_set: np.ndarray, tokens: np.ndarray, seed: int,
                      nvfp4: bool = False):
    """Host cache holding every row the sampled tokens reference, quantized by
    the oracle (FP8 rows, or NVFP4 rows) from host-drawn latent rows of the
    same distribution."""
    import oracle
    slots = oracle.translate(index_set[tokens], case.block_table, case.req_id_per_token[tokens], case.num_blocks)
    need = np.unique(slots[slots >= 0]).astype(np.int64)
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((len(need), 576), dtype=np.float32)
    if len(case.outlier_channels):
        x[:, case.outlier_channels] *= 8.0
    cache = np.zeros((case.num_blocks, 64, 352 if nvfp4 else 656), np.uint8)
    (oracle.nvfp4_quantize_store if nvfp4 else oracle.quantize_store)(inp.bf16_bits(x), need, cache)
    return cache


def time_oracle(case, index_set, tokens, cache, nthreads):
    import oracle
    t0 = time.perf_counter()
    oracle.sparse_mla_decode(case.q, cache, index_set, case.block_table, case.req_id_per_token, case.sm_scale,
                             tokens=tokens, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(case, budget_s: float = 12.0):
    """Oracle throughput on the host cores: whole passes over the 64 tokens of
    index set 0 until about budget_s of CPU work (at least one pass)."""
    import oracle
    nth = oracle.default_threads()
    tokens = np.arange(case.q.shape[0], dtype=np.int32)
    cache = host_sample_cache(case, case.index_sets[0], tokens, seed=12345)
    n_tok, elapsed, passes = 0, 0.0, 0
    while passes == 0 or elapsed < budget_s:
        elapsed += time_oracle(case, case.index_sets[0], tokens, cache, nth)
        n_tok += len(tokens)
        passes += 1
    return {"value": n_tok / elapsed, "unit": UNIT, "cores": nth, "kind": "oracle",
            "sample": f"{passes} pass(es) over all {len(tokens)} query tokens of one index set "
                      f"(float64 C oracle, OpenMP over tokens, {nth} threads), {elapsed:.1f} s"}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, local = dist_setup()
    if rank != 0:
        barrier(world)
        return
    import oracle
    oracle.build()
    case = inp.rotating_decode(seed=1)
    nth = oracle.default_threads()
    S = max(1, min(case.q.shape[0], nth))  # tokens per step: one per host thread
    rng = np.random.default_rng(99)
    toks = [np.sort(rng.choice(case.q.shape[0], S, replace=False)).astype(np.int32)
            for _ in range(args.warmup + args.steps)]
    all_tok = np.unique(np.concatenate(toks)).astype(np.int32)
    cache = host_sample_cache(case, case.index_sets[0], all_tok, seed=12345)
    for i in range(args.warmup):
        time_oracle(case, case.index_sets[0], toks[i], cache, nth)
    t = 0.0
    for i in range(args.steps):
        t += time_oracle(case, case.index_sets[0], toks[args.warmup + i], cache, nth)
    value = args.steps * S / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{case.name}: memory-bound FP8 sparse decode, 64 requests x 1 token, H=16, "
                                   f"top-k 2048, context U[8192,32768], 656-byte FP8 cache",
                       "step": f"float64 CPU oracle on {S} of the 64 query tokens (one per host thread)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nth, "kind": "oracle",
                             "sample": f"{S} query tokens per step, {args.steps} steps"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    barrier(world)


# ---------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import sparse_mla_attention_fp8_gb300 as smla

    rank, world, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the library path (use --impl reference for the oracle)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    smla.build()
    peaks = load_peaks()

    case = inp.rotating_decode(seed=1 + rank)
    T, H, K = case.q.shape[0], case.H, case.K
    NB = case.num_blocks
    stream = torch.cuda.Stream(device)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)

    with torch.cuda.stream(stream):
        cache = torch.zeros((NB, 64, 656), dtype=torch.uint8, device=device)
        lat = inp.device_latent(len(case.ctx_slots), case.latent_seed, case.outlier_channels, device)
        smla.mla_cache_store_fp8(lat, torch.from_numpy(case.ctx_slots).to(device), cache, stream=stream)
        new_rows = inp.device_latent(T, case.latent_seed + 1, case.outlier_channels, device)
        new_slots = torch.from_numpy(case.new_slots).to(device)
        q = bf16(case.q)
        idx_sets = [torch.from_numpy(s).to(device) for s in case.index_sets]
        bt = torch.from_numpy(case.block_table).to(device)
        req = torch.from_numpy(case.req_id_per_token).to(device)
        ws = torch.zeros(smla.decode_workspace_bytes(T, H, K, 0), dtype=torch.uint8, device=device)
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=device)
        lse = torch.empty((T, H), dtype=torch.float32, device=device)
    stream.synchronize()
    del lat

    def store():
        smla.mla_cache_store_fp8(new_rows, new_slots, cache, stream=stream)

    def decode(i):
        smla.sparse_mla_decode_fp8(q, cache, idx_sets[i % len(idx_sets)], bt, req, case.sm_scale, 0, out, lse, ws,
                                   stream=stream)

    # warm-up through the binding (sets kernel attributes)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            store()
            decode(i)
    stream.synchronize()
    if smla.read_device_status(ws, stream) != 0:
        raise SystemExit("device status reports a kernel wait timeout")
    n_rot = len(idx_sets)
    # The timed steps call the C entry points directly, with argument lists
    # built once per rotating index set: the host issues a step in a few
    # microseconds, well ahead of the GPU, and consecutive launches follow each
    # other without a CUDA-graph launch in between.
    import ctypes
    L = smla.lib()
    cs = ctypes.c_void_p(stream.cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    R, MB = case.block_table.shape
    store_args = (ptr(new_rows), ptr(new_slots), ptr(cache), T, NB, cs)
    decode_args = [(ptr(q), ptr(cache), ptr(idx_sets[j]), ptr(bt), ptr(req), ctypes.c_float(case.sm_scale), 0,
                    ptr(out), ptr(lse), T, H, K, R, MB, NB, ptr(ws), ws.numel(), cs) for j in range(n_rot)]
    c_store, c_decode = L.mla_cache_store_fp8, L.sparse_mla_decode_fp8

    def step(i):  # quantize-and-store of the new rows, then the decode
        if c_store(*store_args) | c_decode(*decode_args[i % n_rot]):
            raise SystemExit("C-ABI call failed: " + L.smla_last_error().decode())

    def decode_alone(i):
        if c_decode(*decode_args[i % n_rot]):
            raise SystemExit("C-ABI call failed: " + L.smla_last_error().decode())

    for i in range(args.warmup):
        step(i)
    stream.synchronize()

    launches_per_step = 1 + smla.attention_plan(True, T, H, K, 0)[0]  # store + the decode's launches

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    # ---- clocks: sampled from an untimed burst of >= 1.2 s of steps under load
    # through the timed region
    clocks.start()
    t_burst = time.perf_counter()
    with torch.cuda.stream(stream):
        while time.perf_counter() - t_burst < 1.2:
            for i in range(n_rot * 16):
                step(i)
            stream.synchronize()
    # ---- timed region: exactly K steps
    barrier(world, device)
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(world, device)
    step_ms = e0.elapsed_time(e1) / args.steps
    # ---- the decode launches alone, same rotation (roofline of the dominant kernel)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            decode_alone(i)
        e1.record(stream)
    torch.cuda.synchronize(device)
    clk = clocks.stop()
    decode_ms = e0.elapsed_time(e1) / args.steps
    if smla.read_device_status(ws, stream) != 0:
        raise SystemExit("device status reports a kernel wait timeout")

    step_ms_max = max_over_ranks(step_ms, world, device)
    value = world * T / (step_ms_max * 1e-3)
    alg_bytes = statistics.mean(decode_algorithmic_bytes(case, s) for s in case.index_sets)
    flops = statistics.mean(decode_flops(case, s) for s in case.index_sets)
    achieved_gbs = alg_bytes / (decode_ms * 1e-3) / 1e9

    # ---- end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, smla, case, device, stream, cache, ws)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case)

    # ---- the tensor-bound configurations, each with its own roofline (rank 0, N = 1)
    extra = {}
    if rank == 0 and world == 1 and not args.no_extra:
        del cache
        torch.cuda.empty_cache()
        for name, k in (("decode_h128_k2048", max(20, args.steps // 20)), ("prefill_h128_k2048", max(5, args.steps // 200)),
                        ("prefill_fp8_h128_k2048", max(5, args.steps // 200)), ("mla_absorb_h128", max(20, args.steps // 20)),
                        ("decode_nvfp4_h16_k2048", max(20, args.steps // 20))):
            sub = argparse.Namespace(**vars(args))
            sub.workload, sub.steps = name, k
            sub.no_cpu_baseline = True
            extra[name] = tensor_workload(sub, quiet=True)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {
                "workload": f"{case.name}: memory-bound FP8 sparse decode, {T} requests x 1 token, H={H}, "
                            f"top-k {K}, context U[8192,32768], block 64, 656-byte FP8 cache ({NB} blocks, "
                            f"{NB * 64 * 656 / 1e9:.2f} GB)",
                "step": "quantize-and-store of the 64 new rows + sparse decode (translate, gather/dequant, "
                        "QK^T, softmax, P.V, combine)",
                "l2": f"{n_rot} rotating top-k index sets ({n_rot} x {alg_bytes / 1e6:.0f} MB gathered) > 129 MB L2",
                "parallelism": f"weak: {world} independent replica(s), one per GPU",
                "launch": "C-ABI calls on one stream, argument lists built once; the host stays ahead of the GPU",
            },
            "gb_per_s": achieved_gbs,
            "tflops": flops / (decode_ms * 1e-3) / 1e12,
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": captured_traffic(),
                         "peak_source": peaks["source"],
                         "kernel": "sparse decode launch (attention kernel, plus the combine where units are split "
                                   "outside a cluster)",
                         "algorithmic_bytes_per_launch": int(alg_bytes), "avg_launch_us": decode_ms * 1e3},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
        }
        for name, r in extra.items():
            line[name] = r
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- tensor-bound workloads (not the default line)

def tensor_peak_tflops(peaks, fp8: bool) -> float:
    """Dense tensor peak for the path's MMA type: the measured bf16 burst
    figure, times the nominal fp8 / bf16 ratio (4.5 / 2.25) for FP8 MMAs."""
    return peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)


def time_graphs(graphs, steps, stream):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_tensor_workload(args):
    print(json.dumps(tensor_workload(args)), flush=True)


def tensor_workload(args, quiet=False):
    """The tensor-bound configurations of the hot path, for the record (the
    default line is the memory-bound decode):
      decode_h128_k2048: FP8 decode, 128 requests x 1 token, H = 128, top-k
        2048, context 65536 (5.5 GB cache), 8 rotating index sets;
      prefill_h128_k2048: bf16 prefill, 4 requests x 1024 new tokens over
        3072 cached, H = 128, top-k 2048, dense latent buffer of 16384 rows;
      prefill_fp8_h128_k2048: the same prefill over the FP8 cache (gather +
        up-convert, index mapping, bf16 prefill);
      mla_absorb_h128: the two weight-absorption GEMMs around the attention
        at 4096 tokens, H = 128 (HBM-bound: ~93 FLOP per byte).
    Prints one JSON line: query-tokens/s, TFLOP/s against the dense tensor
    peak of the path's MMA type (HBM GB/s against measured copy bandwidth for
    the absorption), and the oracle on a bounded token sample."""
    import torch
    import oracle
    import sparse_mla_attention_fp8_gb300 as smla
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the library path")
    device = torch.device("cuda", torch.cuda.current_device())
    smla.build()
    oracle.build()
    peaks = load_peaks()
    stream = torch.cuda.Stream(device)
    nth = oracle.default_threads()

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)

    algo_bytes = None  # set for an HBM-bound workload: its roofline is then bytes over measured copy bandwidth
    if args.workload == "decode_h128_k2048":
        ctx = args.context or 65536
        case = inp.rotating_decode(seed=2, R=128, ctx_lo=ctx, ctx_hi=ctx, K=2048, H=128, outliers=True)
        T, H, K, NB = case.q.shape[0], case.H, case.K, case.num_blocks
        with torch.cuda.stream(stream):
            cache = torch.zeros((NB, 64, 656), dtype=torch.uint8, device=device)
            lat = inp.device_latent(len(case.ctx_slots), case.latent_seed, case.outlier_channels, device)
            smla.mla_cache_store_fp8(lat, torch.from_numpy(case.ctx_slots).to(device), cache, stream=stream)
            q = bf16(case.q)
            idx_sets = [torch.from_numpy(x).to(device) for x in case.index_sets]
            bt = torch.from_numpy(case.block_table).to(device)
            req = torch.from_numpy(case.req_id_per_token).to(device)
            ws = torch.zeros(smla.decode_workspace_bytes(T, H, K, 0), dtype=torch.uint8, device=device)
            out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=device)
            lse = torch.empty((T, H), dtype=torch.float32, device=device)
        stream.synchronize()
        del lat

        def launch(i):
            smla.sparse_mla_decode_fp8(q, cache, idx_sets[i % len(idx_sets)], bt, req, case.sm_scale, 0, out, lse,
                                       ws, stream=stream)
        n_graphs = len(idx_sets)
        flops = statistics.mean(decode_flops(case, x) for x in case.index_sets)
        # 128 heads run the CTA-pair kernel: FP8 rows converted to f16 on chip, f16 / bf16 MMAs
        fp8 = H != 128
        mma_dtype = "f16" if H == 128 else "fp8"
        launches = smla.attention_plan(True, T, H, K, 0)[0]
        desc = (f"{case.name}: tensor-bound FP8 sparse decode, {T} requests x 1 token, H={H}, top-k {K}, "
                f"context {ctx}, 656-byte FP8 cache ({NB} blocks, {NB * 64 * 656 / 1e9:.1f} GB), "
                f"{n_graphs} rotating index sets")
        # oracle sample: a few tokens on a host cache holding the rows they reference
        tok = np.arange(min(nth, 8), dtype=np.int32)
        hcache = host_sample_cache(case, case.index_sets[0], tok, seed=777)

        def oracle_run():
            oracle.sparse_mla_decode(case.q, hcache, case.index_sets[0], case.block_table, case.req_id_per_token,
                                     case.sm_scale, tokens=tok, nthreads=nth)
    elif args.workload == "decode_nvfp4_h16_k2048":
        # the memory-bound decode's workload over the NVFP4 cache (352-byte rows, read as stored)
        case = inp.rotating_decode(seed=1)
        T, H, K, NB = case.q.shape[0], case.H, case.K, case.num_blocks
        with torch.cuda.stream(stream):
            cache = torch.zeros((NB, 64, 352), dtype=torch.uint8, device=device)
            lat = inp.device_latent(len(case.ctx_slots), case.latent_seed, case.outlier_channels, device)
            smla.mla_cache_store_nvfp4(lat, torch.from_numpy(case.ctx_slots).to(device), cache, stream=stream)
            q = bf16(case.q)
            idx_sets = [torch.from_numpy(x).to(device) for x in case.index_sets]
            bt = torch.from_numpy(case.block_table).to(device)
            req = torch.from_numpy(case.req_id_per_token).to(device)
            ws = torch.zeros(smla.decode_nvfp4_workspace_bytes(T, H, K, 0), dtype=torch.uint8, device=device)
            out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=device)
            lse = torch.empty((T, H), dtype=torch.float32, device=device)
        stream.synchronize()
        del lat

        def launch(i):
            smla.sparse_mla_decode_nvfp4(q, cache, idx_sets[i % len(idx_sets)], bt, req, case.sm_scale, 0, out, lse,
                                         ws, stream=stream)
        n_graphs = len(idx_sets)
        flops = statistics.mean(decode_flops(case, x) for x in case.index_sets)
        algo_bytes = statistics.mean(decode_algorithmic_bytes(case, x, 352) for x in case.index_sets)
        fp8 = False
        mma_dtype = "bf16"
        launches = smla.attention_plan(False, T, H, K, 0)[0]
        desc = (f"{case.name}: NVFP4 sparse decode, {T} requests x 1 token, H={H}, top-k {K}, context "
                f"U[8192,32768], 352-byte NVFP4 cache ({NB} blocks, {NB * 64 * 352 / 1e9:.2f} GB), "
                f"{n_graphs} rotating index sets")
        tok = np.arange(min(nth, 16), dtype=np.int32)
        hcache = host_sample_cache(case, case.index_sets[0], tok, seed=778, nvfp4=True)

        def oracle_run():
            oracle.sparse_mla_decode_nvfp4(case.q, hcache, case.index_sets[0], case.block_table,
                                           case.req_id_per_token, case.sm_scale, tokens=tok, nthreads=nth)
    elif args.workload == "mla_absorb_h128":
        # the weight absorption around the attention at the prefill workload's shape: 4096 tokens, H = 128,
        # q_nope 128 -> 512 (with q_pe appended) and 512 -> V = 128, synthetic weights
        T, H, P, V = 4096, 128, 128, 128
        K = 0
        rng = np.random.default_rng(8)
        with torch.cuda.stream(stream):
            q = bf16(inp.bf16_bits(rng.standard_normal((T, H, P + 64), dtype=np.float32)))
            w_uk = bf16(inp.bf16_bits((rng.standard_normal((H, P, 512), dtype=np.float32) * 0.08)))
            a_out = bf16(inp.bf16_bits(rng.standard_normal((T, H, 512), dtype=np.float32)))
            w_uv = bf16(inp.bf16_bits((rng.standard_normal((H, 512, V), dtype=np.float32) * 0.05)))
            q_out = torch.empty((T, H, 576), dtype=torch.bfloat16, device=device)
            y = torch.empty((T, H, V), dtype=torch.bfloat16, device=device)
            ws = torch.zeros(256, dtype=torch.uint8, device=device)
        stream.synchronize()

        def launch(i):
            smla.mla_absorb_q(q, w_uk, q_out, ws, stream=stream)
            smla.mla_v_up_proj(a_out, w_uv, y, ws, stream=stream)
        n_graphs = 1
        flops = 2 * T * H * P * 512 + 2 * T * H * 512 * V
        # q_nope read (the RoPE part is copied), W_UK_T, q_out written; attn_out, W_UV, the projection written
        algo_bytes = 2 * (T * H * (P + 64) + H * P * 512 + T * H * 576 + T * H * 512 + H * 512 * V + T * H * V)
        fp8 = False
        mma_dtype = "bf16"
        launches = 2
        desc = (f"mla_absorb_h128: per-head GEMMs around the attention, {T} tokens, H={H}: q_nope ({P}) x W_UK_T "
                f"-> 512 with q_pe appended, and 512 x W_UV -> {V}; synthetic weights")
        tok = np.arange(min(nth, 8), dtype=np.int32)
        qh = inp.bf16_bits(rng.standard_normal((len(tok), H, P + 64), dtype=np.float32))
        wh = inp.bf16_bits(rng.standard_normal((H, P, 512), dtype=np.float32) * 0.08)
        ah = inp.bf16_bits(rng.standard_normal((len(tok), H, 512), dtype=np.float32))
        vh = inp.bf16_bits(rng.standard_normal((H, 512, V), dtype=np.float32) * 0.05)

        def oracle_run():
            oracle.absorb_q(qh, wh)
            oracle.v_up_proj(ah, vh)
    elif args.workload == "prefill_fp8_h128_k2048":
        # the bf16 prefill workload's shape over the FP8 paged cache, separate mode: each call gathers and
        # up-converts the chunk's 4 x 4096 rows into a bf16 workspace, maps the indices, runs the bf16 prefill
        case = inp.fp8_prefill_chunk(seed=5)
        T, H, K, NB = case.T, case.H, case.K, case.num_blocks
        R = case.block_table.shape[0]
        seq_lens = np.zeros(R, np.int32)
        for t in range(T):
            r = case.req_id_per_token[t]
            seq_lens[r] = max(seq_lens[r], case.positions[t] + 1)
        starts = np.concatenate([[0], np.cumsum(seq_lens)[:-1]]).astype(np.int32)
        N = int(seq_lens.sum())
        with torch.cuda.stream(stream):
            cache = torch.zeros((NB, 64, 656), dtype=torch.uint8, device=device)
            smla.mla_cache_store_fp8(bf16(case.cache_rows), torch.from_numpy(case.cache_slots).to(device), cache,
                                     stream=stream)
            smla.mla_cache_store_fp8(bf16(case.new_rows), torch.from_numpy(case.new_slots).to(device), cache,
                                     stream=stream)
            q = bf16(case.q)
            idx = torch.from_numpy(case.indices).to(device)
            bt = torch.from_numpy(case.block_table).to(device)
            req = torch.from_numpy(case.req_id_per_token).to(device)
            d_sl = torch.from_numpy(seq_lens).to(device)
            d_st = torch.from_numpy(starts).to(device)
            kvw = torch.empty((N, 576), dtype=torch.bfloat16, device=device)
            ws = torch.zeros(smla.prefill_fp8_workspace_bytes(T, H, K, 0), dtype=torch.uint8, device=device)
            out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=device)
            lse = torch.empty((T, H), dtype=torch.float32, device=device)
        stream.synchronize()

        def launch(i):
            smla.sparse_mla_prefill_fp8(q, cache, idx, bt, req, d_sl, d_st, kvw, case.sm_scale, 0, out, lse, ws,
                                        stream=stream)
        n_graphs = 1
        flops = 2 * H * int((case.indices >= 0).sum()) * (576 + 512)
        fp8 = False
        mma_dtype = "bf16"
        launches = 2 + smla.attention_plan(False, T, H, K, 0)[0]  # gather + translate + the prefill's launches
        desc = (f"{case.name}: separate-mode FP8 prefill, 4 requests x 1024 new tokens over 3072 cached in the "
                f"656-byte FP8 paged cache, H={H}, top-k {K}: gather + up-convert of {N} rows to bf16, index "
                f"mapping, bf16 prefill")
        tok = np.linspace(0, T - 1, min(nth, 8)).astype(np.int32)
        host_cache = np.zeros((NB, 64, 656), np.uint8)
        oracle.quantize_store(case.cache_rows, case.cache_slots, host_cache)
        oracle.quantize_store(case.new_rows, case.new_slots, host_cache)

        def oracle_run():
            oracle.sparse_mla_prefill_fp8(case.q, host_cache, case.indices, case.block_table, case.req_id_per_token,
                                          seq_lens, starts, N, case.sm_scale, tokens=tok, nthreads=nth)
    else:
        case = inp.prefill(seed=3)
        T, H, K = case.T, case.H, case.K
        N = case.kv.shape[0]
        with torch.cuda.stream(stream):
            q = bf16(case.q)
            kv = bf16(case.kv)
            idx = torch.from_numpy(case.indices).to(device)
            ws = torch.zeros(smla.prefill_workspace_bytes(T, H, K, 0), dtype=torch.uint8, device=device)
            out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=device)
            lse = torch.empty((T, H), dtype=torch.float32, device=device)
        stream.synchronize()

        def launch(i):
            smla.sparse_mla_prefill_bf16(q, kv, idx, case.sm_scale, 0, out, lse, ws, stream=stream)
        n_graphs = 1
        flops = 2 * H * int((case.indices >= 0).sum()) * (576 + 512)
        fp8 = False
        mma_dtype = "bf16"
        launches = smla.attention_plan(False, T, H, K, 0)[0]
        desc = (f"{case.name}: bf16 sparse prefill, 4 requests x 1024 new tokens over 3072 cached, H={H}, "
                f"top-k {K}, dense latent buffer [{N}, 576] (L2-resident)")
        tok = np.linspace(0, T - 1, min(nth, 8)).astype(np.int32)

        def oracle_run():
            oracle.sparse_mla_prefill(case.q, case.kv, case.indices, case.sm_scale, tokens=tok, nthreads=nth)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            launch(i)
    stream.synchronize()
    graphs = []
    for i in range(n_graphs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launch(i)
        graphs.append(g)
    time_graphs(graphs, max(args.warmup, 3), stream)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    if not quiet:  # an untimed burst of >= 1.2 s under load for the clock record
        t_burst = time.perf_counter()
        while time.perf_counter() - t_burst < 1.2:
            time_graphs(graphs, max(3, args.steps // 4), stream)
    ms = time_graphs(graphs, args.steps, stream)
    clk = clocks.stop()
    if smla.read_device_status(ws, stream) != 0:
        raise SystemExit("device status reports a kernel wait timeout")
    tflops = flops / (ms * 1e-3) / 1e12
    peak = tensor_peak_tflops(peaks, fp8)
    wide_traffic, wide_traffic_kernels = captured_wide_traffic(args.workload)
    if args.workload == "prefill_fp8_h128_k2048":
        wide_traffic, wide_traffic_kernels = PREFILL_FP8_TRAFFIC_BY_SOURCE.get(
            _source_key(PREFILL_FP8_TRAFFIC_SOURCES), (None, None))
    cpu = None
    if not args.no_cpu_baseline:
        t0 = time.perf_counter()
        oracle_run()
        el = time.perf_counter() - t0
        cpu = {"value": len(tok) / el, "unit": UNIT, "cores": nth, "kind": "oracle",
               "sample": f"{len(tok)} query tokens of the workload (float64 C oracle, {nth} threads), {el:.1f} s"}
    line = {
        "metric": f"{args.workload} query-tokens/s + TFLOP/s vs tensor roofline", "value": T / (ms * 1e-3),
        "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": mma_dtype,
        "data": "synthetic",
        "config": {"workload": desc, "step": "one attention launch (plus the split combine)",
                   "l2": "8 rotating index sets (decode); the prefill's 18.9 MB buffer is L2-resident by design",
                   "parallelism": "single GPU", "launch": "CUDA graph per step"},
        "tflops": tflops,
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "traffic": wide_traffic, "traffic_kernels": wide_traffic_kernels, "peak_source": peaks["source"] + (" bf16 x 2 (fp8/bf16 nominal)" if fp8 else ""),
                     "kernel": "attention launch (attention kernel + split combine)", "flops_per_launch": flops,
                     "avg_launch_us": ms * 1e3},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": launches * args.steps, "clocks": clk,
    }
    if args.workload == "decode_h128_k2048":
        # the FP8-query variant of the same call (its own CTA-pair kernel at 128 heads: e4m3 MMAs)
        def launch_q8(i):
            smla.sparse_mla_decode_fp8_qfp8(q, cache, idx_sets[i % len(idx_sets)], bt, req, case.sm_scale, 0, out,
                                            lse, ws, stream=stream)
        with torch.cuda.stream(stream):
            for i in range(max(args.warmup, 3)):
                launch_q8(i)
        stream.synchronize()
        graphs_q8 = []
        for i in range(n_graphs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                launch_q8(i)
            graphs_q8.append(g)
        time_graphs(graphs_q8, max(args.warmup, 3), stream)
        ms_q8 = time_graphs(graphs_q8, args.steps, stream)
        if smla.read_device_status(ws, stream) != 0:
            raise SystemExit("device status reports a kernel wait timeout")
        tf_q8 = flops / (ms_q8 * 1e-3) / 1e12
        line["fp8_query_variant"] = {
            "call": "sparse_mla_decode_fp8_qfp8", "ms_per_step": ms_q8, "value": T / (ms_q8 * 1e-3), "unit": UNIT,
            "tflops": tf_q8, "dtype": "e4m3", "frac_of_fp8_peak": tf_q8 / tensor_peak_tflops(peaks, True),
            "frac_of_bf16_peak": tf_q8 / peak, "gpu_launches": launches * args.steps}
    if algo_bytes is not None:
        gbs = algo_bytes / (ms * 1e-3) / 1e9
        line["metric"] = f"{args.workload} query-tokens/s + GB/s vs HBM roofline"
        traffic, traffic_kernels = None, None
        if args.workload == "decode_nvfp4_h16_k2048":
            line["dtype"] = "e2m1"
            line["config"]["step"] = "one sparse decode launch over the NVFP4 cache (rows dequantized in the kernel)"
            line["config"]["l2"] = "8 rotating top-k index sets (8 x 46 MB gathered) > 129 MB L2"
            kernel = "sparse_mla_attn_kernel<16, NVFP4 rows> (plus the combine)"
            traffic, traffic_kernels = NVFP4_TRAFFIC_BY_SOURCE.get(_source_key(NVFP4_TRAFFIC_SOURCES), (None, None))
        else:
            line["config"]["step"] = "the query-side and value-side GEMM launches"
            line["config"]["l2"] = "inputs (1.5 GB per step) larger than L2"
            kernel = "head_gemm_kernel (two launches per step)"
            traffic, traffic_kernels = ABSORB_TRAFFIC_BY_SOURCE.get(_source_key(ABSORB_TRAFFIC_SOURCES), (None, None))
        line["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": gbs / peaks["hbm_gbs"], "traffic": traffic, "traffic_kernels": traffic_kernels,
                            "peak_source": peaks["source"], "kernel": kernel, "bytes_per_step": algo_bytes,
                            "avg_step_us": ms * 1e3}
    return line


def _cudart():
    """The CUDA toolkit's runtime library, for the end-to-end step's copies,
    event records and waits (streams and events are shared with torch through
    the device's primary context), or None when it cannot be loaded."""
    import ctypes
    import ctypes.util
    cands = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcudart.so")]
    found = ctypes.util.find_library("cudart")
    if found:
        cands.append(found)
    for c in cands:
        try:
            rt = ctypes.CDLL(c)
        except OSError:
            continue
        P = ctypes.c_void_p
        rt.cudaMemcpyAsync.argtypes = [P, P, ctypes.c_size_t, ctypes.c_int, P]
        rt.cudaEventRecord.argtypes = [P, P]
        rt.cudaStreamWaitEvent.argtypes = [P, P, ctypes.c_uint]
        rt.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(P), ctypes.c_uint]
        return rt
    return None


def run_e2e(args, smla, case, device, stream, cache, ws):
    """The same step end to end through the C ABI with host buffers: every
    step copies its inputs (q, the step's top-k indices, block table, request
    ids, the new rows and their slots) from one pinned host buffer to the
    device in one copy, runs quantize-and-store + decode through the C entry
    points, and copies out + lse back in one copy.  Inputs and outputs are
    double-buffered on the device, and the copies run on their own streams,
    so step i's copies overlap steps i - 1 and i + 1's kernels."""
    import ctypes

    import torch
    T, H, K = case.q.shape[0], case.H, case.K
    R, MB = case.block_table.shape
    NB = case.num_blocks
    n_rot = len(case.index_sets)
    L = smla.lib()

    def seg(nbytes):
        return (nbytes + 255) // 256 * 256
    rows = inp.device_latent(T, case.latent_seed + 1, case.outlier_channels, device).view(torch.int16).cpu().numpy()
    parts = [("q", case.q.view(np.uint8)), ("idx", None), ("bt", case.block_table.view(np.uint8)),
             ("req", case.req_id_per_token.view(np.uint8)), ("rows", rows.view(np.uint8)),
             ("slots", case.new_slots.view(np.uint8))]
    sizes = {"q": case.q.nbytes, "idx": case.index_sets[0].nbytes, "bt": case.block_table.nbytes,
             "req": case.req_id_per_token.nbytes, "rows": rows.nbytes, "slots": case.new_slots.nbytes}
    offs, off = {}, 0
    for name, _ in parts:
        offs[name] = off
        off += seg(sizes[name])
    in_bytes = off
    h_in = []
    for j in range(n_rot):  # one packed host input buffer per rotating index set
        buf = np.zeros(in_bytes, np.uint8)
        for name, arr in parts:
            src = case.index_sets[j].view(np.uint8) if name == "idx" else arr
            buf[offs[name]:offs[name] + sizes[name]] = src.reshape(-1)
        h_in.append(torch.from_numpy(buf).pin_memory())
    out_bytes = T * H * 512 * 2
    o_lse = seg(out_bytes)
    res_bytes = o_lse + T * H * 4
    d_in = [torch.empty(in_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
    d_res = [torch.empty(res_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
    h_res = [torch.empty(res_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    cstream = ctypes.c_void_p(stream.cuda_stream)
    cache_p = ctypes.c_void_p(cache.data_ptr())
    ws_p, ws_n = ctypes.c_void_p(ws.data_ptr()), ws.numel()
    # per buffer slot: the C-ABI calls' argument lists, built once
    store_args, decode_args = [], []
    for k in range(2):
        base_in, base_res = d_in[k].data_ptr(), d_res[k].data_ptr()
        P = lambda name: ctypes.c_void_p(base_in + offs[name])  # noqa: E731
        store_args.append((P("rows"), P("slots"), cache_p, T, NB, cstream))
        decode_args.append((P("q"), cache_p, P("idx"), P("bt"), P("req"), ctypes.c_float(case.sm_scale), 0,
                            ctypes.c_void_p(base_res), ctypes.c_void_p(base_res + o_lse), T, H, K, R, MB, NB, ws_p,
                            ws_n, cstream))
    store, decode = L.mla_cache_store_fp8, L.sparse_mla_decode_fp8
    rt = _cudart()
    if rt is not None:
        # copies, event records and waits straight through the CUDA runtime:
        # the step's host-side cost stays below its GPU time
        def mkev():
            ev = ctypes.c_void_p()
            if rt.cudaEventCreateWithFlags(ctypes.byref(ev), 2) != 0:  # cudaEventDisableTiming
                raise SystemExit("e2e: cudaEventCreateWithFlags failed")
            return ev
        ev_in, ev_done, ev_out = [mkev(), mkev()], [mkev(), mkev()], [mkev(), mkev()]
        hs, ds = ctypes.c_void_p(s_h2d.cuda_stream), ctypes.c_void_p(s_d2h.cuda_stream)
        h_in_p = [ctypes.c_void_p(t.data_ptr()) for t in h_in]
        d_in_p = [ctypes.c_void_p(t.data_ptr()) for t in d_in]
        d_res_p = [ctypes.c_void_p(t.data_ptr()) for t in d_res]
        h_res_p = [ctypes.c_void_p(t.data_ptr()) for t in h_res]
        in_sz, res_sz = ctypes.c_size_t(in_bytes), ctypes.c_size_t(res_bytes)
        memcpy, record, wait = rt.cudaMemcpyAsync, rt.cudaEventRecord, rt.cudaStreamWaitEvent

        def step(i):
            k = i & 1
            err = 0
            if i >= 2:
                err |= wait(hs, ev_done[k], 0)  # the slot's inputs are free
            err |= memcpy(d_in_p[k], h_in_p[i % n_rot], in_sz, 1, hs)  # host to device
            err |= record(ev_in[k], hs)
            err |= wait(cstream, ev_in[k], 0)
            if i >= 2:
                err |= wait(cstream, ev_out[k], 0)  # the slot's previous results are copied out
            rc = store(*store_args[k]) | decode(*decode_args[k])
            if rc != 0:
                raise SystemExit("e2e: C-ABI call failed: " + L.smla_last_error().decode())
            err |= record(ev_done[k], cstream)
            err |= wait(ds, ev_done[k], 0)
            err |= memcpy(h_res_p[k], d_res_p[k], res_sz, 2, ds)  # device to host
            err |= record(ev_out[k], ds)
            if err != 0:
                raise SystemExit("e2e: a CUDA runtime call failed")
    else:
        ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of the slot copied
        ev_done = [torch.cuda.Event() for _ in range(2)]   # kernels of the slot done (inputs free, results ready)
        ev_out = [torch.cuda.Event() for _ in range(2)]    # results of the slot copied back

        def step(i):
            k = i % 2
            with torch.cuda.stream(s_h2d):
                if i >= 2:
                    s_h2d.wait_event(ev_done[k])
                d_in[k].copy_(h_in[i % n_rot], non_blocking=True)
                ev_in[k].record(s_h2d)
            stream.wait_event(ev_in[k])
            if i >= 2:
                stream.wait_event(ev_out[k])
            rc = store(*store_args[k]) | decode(*decode_args[k])
            if rc != 0:
                raise SystemExit("e2e: C-ABI call failed: " + L.smla_last_error().decode())
            ev_done[k].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[k])
                h_res[k].copy_(d_res[k], non_blocking=True)
                ev_out[k].record(s_d2h)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_h2d)
    for i in range(args.steps):
        step(i)
    e1.record(s_d2h)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / args.steps
    # the last step's results as copied back agree with the device buffers
    last = (args.steps - 1) % 2
    assert torch.equal(h_res[last].to(device), d_res[last])
    return {"value": T / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": int(in_bytes),
            "d2h_bytes_per_step": int(res_bytes), "ms_per_step": ms,
            "path": "C ABI (ctypes) with pinned host buffers: one host-to-device copy of the packed inputs and one "
                    "device-to-host copy of out + lse per step, double-buffered on copy streams"}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="leave the tensor-bound configurations out of the default line")
    ap.add_argument("--workload", choices=["decode_h16_k2048", "decode_h128_k2048", "decode_nvfp4_h16_k2048", "prefill_h128_k2048",
                                           "prefill_fp8_h128_k2048", "mla_absorb_h128"],
                    default="decode_h16_k2048",
                    help="decode_h16_k2048 (default) is the headline; each other workload is reported on its own "
                         "line (and inside the default line, unless --no-extra)")
    ap.add_argument("--context", type=int, default=0,
                    help="decode_h128_k2048 only: per-request context (default 65536, a 5.5 GB cache); a smaller "
                         "one gives the same kernel launch on less device memory, for profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "decode_h16_k2048":
        run_tensor_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
