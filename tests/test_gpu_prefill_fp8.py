"""GPU parity: the separate-mode FP8 prefill (gather + up-convert of the
prefill requests' cache rows into a bf16 workspace, workspace-mapped index
translation, bf16 prefill) against the float64 oracle: the two data steps
bit-exact, attention within atol 1e-2 + rtol 2e-2 on the output and 1e-3 on
the LSE."""
import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import assert_lse_close, assert_out_close, bf16_dev, dev, oracle_cache, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


def _chunk_inputs(case):
    """seq_lens (each request's length), one chunk's workspace starts, and the
    token -> request map of an fp8_prefill_chunk case."""
    R = case.block_table.shape[0]
    seq_lens = np.zeros(R, np.int32)
    for t in range(case.T):
        r = case.req_id_per_token[t]
        seq_lens[r] = max(seq_lens[r], case.positions[t] + 1)
    starts = np.concatenate([[0], np.cumsum(seq_lens)[:-1]]).astype(np.int32)
    return seq_lens, starts, int(seq_lens.sum())


def test_gather_upconvert_bit_exact():
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.fp8_prefill_chunk(seed=1, R=3, cached=200, new=70, K=64, H=16)
    cache = oracle_cache(case)
    bt = case.block_table.copy()
    bt[1, 2] = case.num_blocks + 3  # an invalid physical block: zero rows
    seq_lens, starts, N = _chunk_inputs(case)
    starts = starts + 5  # rows 0..4 of the workspace are not covered: left as they are
    N += 9
    ref = oracle.gather_upconvert(cache, bt, seq_lens, starts, N)
    ws = torch.full((N, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    smla.sparse_mla_gather_upconvert_fp8(dev(cache), dev(bt), dev(seq_lens), dev(starts), ws)
    got = ws.view(torch.int16).cpu().numpy().view(np.uint16)
    covered = np.zeros(N, bool)
    for r in range(len(seq_lens)):
        covered[starts[r]:starts[r] + seq_lens[r]] = True
    assert np.array_equal(got[covered], ref[covered])
    assert np.all(np.isnan(ws.float().cpu().numpy()[~covered]))  # untouched


def test_translate_indices_workspace_bit_exact():
    import sparse_mla_attention_fp8_gb300 as smla
    rng = np.random.default_rng(3)
    R, MB, NB, T, K = 6, 9, 50, 40, 300
    bt = rng.integers(-2, NB + 3, size=(R, MB)).astype(np.int32)
    req = rng.integers(0, R, size=T).astype(np.int32)
    pr = np.where(rng.random(T) < 0.5, rng.integers(0, 4, size=T), -1).astype(np.int32)
    starts = np.array([0, 300, 700], np.int32)  # prefill request 3 has no start
    idx = rng.integers(-3, MB * 64 + 40, size=(T, K)).astype(np.int32)
    ref = oracle.translate_workspace(idx, bt, req, pr, starts, NB)
    got = smla.sparse_mla_translate_indices_workspace(dev(idx), dev(bt), dev(req), dev(pr), dev(starts), NB)
    assert np.array_equal(got.cpu().numpy(), ref)


def _check_prefill_fp8(case, num_splits=0, tokens=None):
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    cache = oracle_cache(case)
    seq_lens, starts, N = _chunk_inputs(case)
    kvw = torch.empty((N, 576), dtype=torch.bfloat16, device="cuda")
    out, lse = smla.sparse_mla_prefill_fp8(bf16_dev(case.q), dev(cache), dev(case.indices), dev(case.block_table),
                                           dev(case.req_id_per_token), dev(seq_lens), dev(starts), kvw,
                                           case.sm_scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert smla.read_device_status() == 0
    ref_out, ref_lse = oracle.sparse_mla_prefill_fp8(case.q, cache, case.indices, case.block_table,
                                                     case.req_id_per_token, seq_lens, starts, N, case.sm_scale,
                                                     tokens=tokens)
    sel = slice(None) if tokens is None else np.asarray(tokens)
    assert_out_close(out.float().cpu().numpy()[sel], ref_out, case.name)
    assert_lse_close(lse.cpu().numpy()[sel], ref_lse, case.name)


@pytest.mark.parametrize("H", [16, 32, 128])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_prefill_fp8_small(H, num_splits):
    # 3 requests x 40 new tokens over 150 cached, K = 200: three full 64-row tiles and a ragged tail;
    # the first tokens see fewer than K positions (-1 padding)
    case = inp.fp8_prefill_chunk(seed=2, R=3, cached=150, new=40, K=200, H=H)
    _check_prefill_fp8(case, num_splits=num_splits)


def test_prefill_fp8_full_size_h128_k2048():
    # the bf16 prefill workload's shape over the FP8 paged cache: 4 requests x 1024 new tokens over 3072
    # cached, H = 128, top-k 2048; the oracle on a seeded token sample with the first and last token
    case = inp.fp8_prefill_chunk(seed=5)
    _check_prefill_fp8(case, tokens=sample_tokens(case.T, 6, seed=5))
