"""Seeded synthetic inputs for the sparse MLA attention workloads.

This module is shared by the oracle-side tests and the CUDA-side tests and
benchmark.  It holds none of the method's arithmetic: it only draws random
numbers and lays out index structures (block tables, top-k index lists,
request ids, slot mappings).  Quantizing the latent rows into the 656-byte
cache is the job of each side (the oracle's quantizer or the CUDA
quantize-and-store kernel).

Workload shapes follow the pages' decode/prefill setting (vLLM
``flashmla_sparse.py``: block size 64, top-k 2048, MQA 576/512,
``req_id_per_token`` as a repeat of request ids over query lengths, decode
requests before prefill requests in a mixed batch).  Everything is synthetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK = 64
D_QK = 576
D_V = 512


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> bfloat16 bit patterns (uint16), round to nearest even
    (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u >> 16) & 1
    r += 0x7FFF
    r += u
    r >>= 16
    return r.astype(np.uint16)


def bits_to_float(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class DecodeCase:
    """One FP8 sparse-decode step over a paged 656-byte cache.

    ``cache_rows`` (bf16 bits [n, 576]) are latent rows already in the cache
    before the step, to be quantized at ``cache_slots``; ``new_rows`` /
    ``new_slots`` are the step's new tokens (written by quantize-and-store
    before attention, empty for pure decode)."""
    name: str
    H: int
    K: int
    sm_scale: float
    q: np.ndarray                 # uint16 [T, H, 576]
    indices: np.ndarray           # int32 [T, K] logical positions, -1 = none
    block_table: np.ndarray       # int32 [R, MB]
    req_id_per_token: np.ndarray  # int32 [T]
    num_blocks: int               # NB
    cache_rows: np.ndarray        # uint16 [n, 576]
    cache_slots: np.ndarray       # int64 [n]
    new_rows: np.ndarray = field(default_factory=lambda: np.zeros((0, D_QK), np.uint16))
    new_slots: np.ndarray = field(default_factory=lambda: np.zeros((0,), np.int64))
    positions: np.ndarray | None = None  # int64 [T], position of each query token in its request

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def R(self) -> int:
        return int(self.block_table.shape[0])

    @property
    def MB(self) -> int:
        return int(self.block_table.shape[1])


@dataclass
class PrefillCase:
    """One BF16 sparse-prefill step over a dense latent buffer kv [N, 576]."""
    name: str
    H: int
    K: int
    sm_scale: float
    q: np.ndarray        # uint16 [T, H, 576]
    kv: np.ndarray       # uint16 [N, 576]
    indices: np.ndarray  # int32 [T, K] row numbers of kv, -1 = none

    @property
    def T(self) -> int:
        return int(self.q.shape[0])


# ---------------------------------------------------------------- helpers

def _paged_layout(rng: np.random.Generator, ctx_lens: np.ndarray):
    """Shuffled block table: request r owns ceil(ctx_r/64) blocks drawn from a
    random permutation of all NB physical blocks.  Unused entries are 0."""
    nblk = (ctx_lens + BLOCK - 1) // BLOCK
    NB = int(nblk.sum())
    MB = int(nblk.max())
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.zeros((len(ctx_lens), MB), np.int32)
    off = 0
    for r, n in enumerate(nblk):
        bt[r, :n] = perm[off:off + n]
        off += n
    return bt, NB


def _slot_of(bt: np.ndarray, r: int, pos: np.ndarray) -> np.ndarray:
    pos = np.asarray(pos, np.int64)
    return bt[r, pos // BLOCK].astype(np.int64) * BLOCK + pos % BLOCK


def _causal_topk(rng: np.random.Generator, visible: int, K: int) -> np.ndarray:
    """K unique unsorted positions from [0, visible); -1 padding if fewer."""
    out = np.full(K, -1, np.int32)
    n = min(K, visible)
    if n > 0:
        out[:n] = rng.choice(visible, size=n, replace=False).astype(np.int32)
    return out


def _latent(rng: np.random.Generator, n: int, outlier_channels: np.ndarray | None) -> np.ndarray:
    x = rng.standard_normal((n, D_QK), dtype=np.float32)
    if outlier_channels is not None and len(outlier_channels):
        x[:, outlier_channels] *= 8.0
    return bf16_bits(x)


def _decode_case(name, seed, ctx_lens, q_per_req, H, K, outliers=False, prefill_reqs=(), sm_scale=None,
                 all_context_rows=False) -> DecodeCase:
    """Generic decode/mixed step.  Request r has ctx_lens[r] tokens in total,
    the last q_per_req[r] of which are this step's query tokens (new rows
    written by quantize-and-store before attention when r is a prefill request
    or q_per_req[r] > 1; for a pure single-token decode the token's own row is
    treated as already cached).  Each query token at position p attends to K
    unique positions in [0, p]."""
    rng = np.random.default_rng(seed)
    ctx_lens = np.asarray(ctx_lens, np.int64)
    q_per_req = np.asarray(q_per_req, np.int64)
    R = len(ctx_lens)
    bt, NB = _paged_layout(rng, ctx_lens)
    outlier_ch = np.sort(rng.choice(D_QK, size=int(np.ceil(0.01 * D_QK)), replace=False)) if outliers else None
    T = int(q_per_req.sum())
    req = np.repeat(np.arange(R, dtype=np.int32), q_per_req)
    positions = np.concatenate([np.arange(c - n, c) for c, n in zip(ctx_lens, q_per_req)]).astype(np.int64)
    indices = np.stack([_causal_topk(rng, int(p) + 1, K) for p in positions]) if T else np.zeros((0, K), np.int32)
    q = bf16_bits(rng.standard_normal((T, H, D_QK), dtype=np.float32))
    # rows written this step: every query token of a request with >1 query token
    writes_new = np.array([(n > 1) or (r in prefill_reqs) for r, n in enumerate(q_per_req)])
    new_slots = []
    for r in range(R):
        if writes_new[r]:
            new_slots.append(_slot_of(bt, r, np.arange(ctx_lens[r] - q_per_req[r], ctx_lens[r])))
    new_slots = np.concatenate(new_slots) if new_slots else np.zeros(0, np.int64)
    # cached rows: every referenced position that is not written this step
    if all_context_rows:
        ref = [np.arange(ctx_lens[r]) for r in range(R)]
    else:
        ref = [np.unique(np.concatenate([indices[t][indices[t] >= 0] for t in np.nonzero(req == r)[0]]))
               if np.any(req == r) else np.zeros(0, np.int64) for r in range(R)]
    cached = []
    for r in range(R):
        pos = np.asarray(ref[r], np.int64)
        if writes_new[r]:
            pos = pos[pos < ctx_lens[r] - q_per_req[r]]
        cached.append(_slot_of(bt, r, pos))
    cache_slots = np.unique(np.concatenate(cached)) if cached else np.zeros(0, np.int64)
    cache_rows = _latent(rng, len(cache_slots), outlier_ch)
    new_rows = _latent(rng, len(new_slots), outlier_ch)
    return DecodeCase(name=name, H=H, K=K, sm_scale=(D_QK ** -0.5) if sm_scale is None else sm_scale, q=q,
                      indices=indices.astype(np.int32), block_table=bt, req_id_per_token=req, num_blocks=NB,
                      cache_rows=cache_rows, cache_slots=cache_slots.astype(np.int64), new_rows=new_rows,
                      new_slots=new_slots.astype(np.int64), positions=positions)


# ---------------------------------------------------------------- the five workloads

def tiny_decode(seed: int = 0) -> DecodeCase:
    """4 requests x 1 token, H=16, context 256 each (4 blocks, 16 shuffled
    physical blocks), top-k 64 unique indices from [0, 256)."""
    rng = np.random.default_rng(seed)
    R, ctx, H, K = 4, 256, 16, 64
    bt, NB = _paged_layout(rng, np.full(R, ctx))
    q = bf16_bits(rng.standard_normal((R, H, D_QK), dtype=np.float32))
    indices = np.stack([rng.choice(ctx, size=K, replace=False) for _ in range(R)]).astype(np.int32)
    slots = np.concatenate([_slot_of(bt, r, np.arange(ctx)) for r in range(R)])
    rows = _latent(rng, len(slots), None)
    return DecodeCase(name="tiny_decode_h16_k64", H=H, K=K, sm_scale=D_QK ** -0.5, q=q, indices=indices,
                      block_table=bt, req_id_per_token=np.arange(R, dtype=np.int32), num_blocks=NB,
                      cache_rows=rows, cache_slots=slots.astype(np.int64),
                      positions=np.full(R, ctx - 1, np.int64))


def memory_bound_decode(seed: int = 1, R: int = 64, ctx_lo: int = 8192, ctx_hi: int = 32768, K: int = 2048,
                        H: int = 16) -> DecodeCase:
    """R requests x 1 token, H=16, top-k 2048, per-request context uniform in
    [ctx_lo, ctx_hi], latent N(0,1) with 1% of the channels scaled x8."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=R)
    return _decode_case(f"decode_h{H}_k{K}_r{R}", seed + 1000, ctx, np.ones(R, np.int64), H, K, outliers=True)


def tensor_bound_decode(seed: int = 2, R: int = 128, ctx: int = 65536, K: int = 2048, H: int = 128) -> DecodeCase:
    """R requests x 1 token, H=128, top-k 2048, context 65536 each, with the
    memory-bound workload's cache distribution (latent N(0,1) with 1% of the
    channels scaled x8)."""
    return _decode_case(f"decode_h{H}_k{K}_r{R}", seed + 1000, np.full(R, ctx), np.ones(R, np.int64), H, K,
                        outliers=True)


def mixed_batch(seed: int = 4, n_decode: int = 32, decode_qlen: int = 2, n_prefill: int = 2,
                prefill_tokens: int = 2048, ctx_lo: int = 4096, ctx_hi: int = 65536, K: int = 1024,
                H: int = 16) -> DecodeCase:
    """Decode requests (query length 2, speculative) followed by prefill
    chunks, all through the FP8 decode kernel as one batch; the step's new
    tokens are first written into the cache at their (random physical) slots."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=n_decode + n_prefill)
    ctx = np.maximum(ctx, prefill_tokens + 1)
    qlen = np.array([decode_qlen] * n_decode + [prefill_tokens] * n_prefill, np.int64)
    return _decode_case(f"mixed_h{H}_k{K}", seed + 1000, ctx, qlen, H, K,
                        prefill_reqs=tuple(range(n_decode, n_decode + n_prefill)))


def fp8_prefill_chunk(seed: int = 5, R: int = 4, cached: int = 3072, new: int = 1024, K: int = 2048,
                      H: int = 128) -> DecodeCase:
    """One chunk of R prefill requests over the FP8 paged cache: request r
    has ``cached`` positions already in the cache and ``new`` query tokens
    (positions cached .. cached + new - 1, written by quantize-and-store);
    token at position p attends to K unique positions in [0, p] (-1 padding
    when fewer are visible); latent N(0,1); shuffled block table."""
    ctx = np.full(R, cached + new, np.int64)
    return _decode_case(f"fp8_prefill_h{H}_k{K}_t{R * new}", seed + 1000, ctx, np.full(R, new, np.int64), H, K,
                        prefill_reqs=tuple(range(R)), all_context_rows=True)


def prefill(seed: int = 3, R: int = 4, cached: int = 3072, new: int = 1024, K: int = 2048, H: int = 128) -> PrefillCase:
    """R requests x ``new`` tokens appended to ``cached`` tokens each, in a
    dense bf16 latent buffer of R*(cached+new) rows; token i of request r sits
    at position cached+i and attends to K unique rows among positions
    [0, cached+i] of its own request (-1 padding when fewer are visible)."""
    rng = np.random.default_rng(seed)
    per = cached + new
    N = R * per
    kv = bf16_bits(rng.standard_normal((N, D_QK), dtype=np.float32))
    T = R * new
    q = bf16_bits(rng.standard_normal((T, H, D_QK), dtype=np.float32))
    indices = np.full((T, K), -1, np.int32)
    t = 0
    for r in range(R):
        for i in range(new):
            row = _causal_topk(rng, cached + i + 1, K)
            valid = row >= 0
            row[valid] += r * per
            indices[t] = row
            t += 1
    return PrefillCase(name=f"prefill_h{H}_k{K}_t{T}", H=H, K=K, sm_scale=D_QK ** -0.5, q=q, kv=kv, indices=indices)


def make_cache(case: DecodeCase, quantize_store, row_bytes: int = 656) -> np.ndarray:
    """Allocate a zeroed [NB, 64, row_bytes] cache (656: FP8 rows, 352: NVFP4
    rows) and fill the pre-existing rows with the given quantize-and-store
    implementation (rows, slots, cache)."""
    cache = np.zeros((case.num_blocks, BLOCK, row_bytes), np.uint8)
    if len(case.cache_slots):
        quantize_store(case.cache_rows, case.cache_slots, cache)
    return cache


# ---------------------------------------------------------------- benchmark inputs

@dataclass
class RotatingDecode:
    """A decode workload with several independent top-k index sets over one
    cache, so successive steps gather different rows.  Latent rows are drawn
    on the device (``device_latent``) because the cache holds every context
    row of every request: ``ctx_slots`` are positions 0..ctx-2 of each
    request, ``new_slots`` the step's new token (position ctx-1), one per
    decode token."""
    name: str
    H: int
    K: int
    sm_scale: float
    q: np.ndarray
    index_sets: list
    block_table: np.ndarray
    req_id_per_token: np.ndarray
    num_blocks: int
    ctx_lens: np.ndarray
    ctx_slots: np.ndarray
    new_slots: np.ndarray
    outlier_channels: np.ndarray
    latent_seed: int


def rotating_decode(seed: int = 1, R: int = 64, ctx_lo: int = 8192, ctx_hi: int = 32768, K: int = 2048, H: int = 16,
                    n_sets: int = 8, outliers: bool = True) -> RotatingDecode:
    """Benchmark form of the memory-bound decode workload: R requests x 1
    token, context uniform in [ctx_lo, ctx_hi], latent N(0,1) with 1% of the
    channels x8, unique unsorted top-k indices, ``n_sets`` independent index
    sets."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=R).astype(np.int64)
    bt, NB = _paged_layout(rng, ctx)
    outlier_ch = (np.sort(rng.choice(D_QK, size=int(np.ceil(0.01 * D_QK)), replace=False)) if outliers
                  else np.zeros(0, np.int64))
    q = bf16_bits(rng.standard_normal((R, H, D_QK), dtype=np.float32))
    sets = [np.stack([_causal_topk(rng, int(c), K) for c in ctx]).astype(np.int32) for _ in range(n_sets)]
    ctx_slots = np.concatenate([_slot_of(bt, r, np.arange(ctx[r] - 1)) for r in range(R)])
    new_slots = np.array([_slot_of(bt, r, np.array([ctx[r] - 1]))[0] for r in range(R)], np.int64)
    return RotatingDecode(name=f"decode_h{H}_k{K}_r{R}", H=H, K=K, sm_scale=D_QK ** -0.5, q=q, index_sets=sets,
                          block_table=bt, req_id_per_token=np.arange(R, dtype=np.int32), num_blocks=NB,
                          ctx_lens=ctx, ctx_slots=ctx_slots.astype(np.int64), new_slots=new_slots,
                          outlier_channels=outlier_ch, latent_seed=seed + 7919)


def device_latent(n: int, seed: int, outlier_channels, device="cuda"):
    """n latent rows N(0,1) (1% outlier channels x8) as a bf16 torch tensor
    [n, 576] drawn on ``device`` with a seeded torch generator (deterministic
    for a given torch build and device type)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn((n, D_QK), generator=g, device=device, dtype=torch.float32)
    if outlier_channels is not None and len(outlier_channels):
        x[:, torch.as_tensor(np.asarray(outlier_channels), device=device)] *= 8.0
    return x.to(torch.bfloat16)
