"""GPU parity: FP8 sparse decode against the float64 oracle on the same
stored bytes (atol 1e-2 + rtol 2e-2 on the output, 1e-3 on the LSE)."""
import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import (assert_lse_close, assert_out_close, bf16_dev, check_decode, dev, oracle_cache,
                     run_gpu_decode, sample_tokens)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


def test_tiny_decode_h16_k64():
    check_decode(inp.tiny_decode(0))


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("num_splits", [0, 1, 2, 3, 5])
def test_ragged_topk_several_tiles(num_splits, H):
    # K = 200: one full 128-row tile and a ragged tail of 72 (H = 16), or three 64-row tiles and a tail of 8
    # (H = 128, the CTA-pair kernel)
    case = inp.memory_bound_decode(seed=5, R=9, ctx_lo=300, ctx_hi=2500, K=200, H=H)
    check_decode(case, num_splits=num_splits)


@pytest.mark.parametrize("H", [32, 48, 64, 128])
def test_head_counts(H):
    case = inp.memory_bound_decode(seed=6, R=5, ctx_lo=200, ctx_hi=900, K=150, H=H)
    check_decode(case)
    check_decode(case, num_splits=1)


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("K", [1, 37, 64, 65, 2048])
def test_topk_widths(K, H):
    case = inp.memory_bound_decode(seed=7, R=6, ctx_lo=2100, ctx_hi=4000, K=K, H=H)
    check_decode(case)


@pytest.mark.parametrize("H", [16, 128])
def test_all_indices_invalid_gives_zero_and_minus_inf(H):
    case = inp.memory_bound_decode(seed=8, R=4, ctx_lo=200, ctx_hi=400, K=130, H=H)
    case.indices[:] = -1
    out, lse = run_gpu_decode(case, oracle_cache(case))
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    case.indices[1, 77] = 5  # one token with a single valid row
    check_decode(case)
    check_decode(case, num_splits=2)


@pytest.mark.parametrize("H", [16, 128])
def test_single_valid_index_returns_its_row(H):
    case = inp.memory_bound_decode(seed=9, R=6, ctx_lo=300, ctx_hi=500, K=96, H=H)
    rng = np.random.default_rng(0)
    keep = rng.integers(0, 96, size=6)
    for t in range(6):
        v = case.indices[t, keep[t]]
        case.indices[t, :] = -1
        case.indices[t, keep[t]] = v
    check_decode(case)


@pytest.mark.parametrize("H", [16, 128])
def test_duplicated_and_out_of_range_indices(H):
    case = inp.memory_bound_decode(seed=10, R=5, ctx_lo=700, ctx_hi=900, K=180, H=H)
    case.indices[:, 100:140] = case.indices[:, 0:40]          # duplicates count once per occurrence
    case.indices[0, 5] = case.block_table.shape[1] * 64 + 3    # block id >= MB
    case.indices[1, 7] = -77
    case.block_table[2, 3] = case.num_blocks + 9               # physical block >= NB
    case.block_table[3, 1] = -4                                # negative physical block
    check_decode(case)


def test_speculative_two_token_requests():
    case = inp.mixed_batch(11, n_decode=6, n_prefill=0, ctx_lo=500, ctx_hi=3000, K=256)
    check_decode(case)


def test_mixed_batch_store_then_decode():
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.mixed_batch(12, n_decode=5, n_prefill=2, prefill_tokens=200, ctx_lo=400, ctx_hi=1500, K=128)
    ref_cache = oracle_cache(case, with_new=True)
    cache = torch.from_numpy(oracle_cache(case, with_new=False)).cuda()
    smla.mla_cache_store_fp8(bf16_dev(case.new_rows), dev(case.new_slots), cache)
    assert np.array_equal(cache.cpu().numpy(), ref_cache)
    out, lse = smla.sparse_mla_decode_fp8(bf16_dev(case.q), cache, dev(case.indices), dev(case.block_table),
                                          dev(case.req_id_per_token), case.sm_scale)
    ref_out, ref_lse = oracle.sparse_mla_decode(case.q, ref_cache, case.indices, case.block_table,
                                                case.req_id_per_token, case.sm_scale)
    assert_out_close(out.float().cpu().numpy(), ref_out, case.name)
    assert_lse_close(lse.cpu().numpy(), ref_lse, case.name)


def test_explicit_workspace_and_too_small_workspace():
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    # 5 parts per token (more than a cluster merges): partial results in the workspace
    case = inp.memory_bound_decode(seed=13, R=4, ctx_lo=800, ctx_hi=1500, K=700)
    cache = oracle_cache(case)
    need = smla.decode_workspace_bytes(case.T, case.H, case.K, 5)
    assert need > 256
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out, lse = run_gpu_decode(case, cache, num_splits=5, workspace=ws)
    ref_out, ref_lse = oracle.sparse_mla_decode(case.q, cache, case.indices, case.block_table,
                                                case.req_id_per_token, case.sm_scale)
    assert_out_close(out, ref_out)
    assert_lse_close(lse, ref_lse)
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(smla.SmlaError, match="status -4"):
        smla.sparse_mla_decode_fp8(bf16_dev(case.q), dev(cache), dev(case.indices), dev(case.block_table),
                                   dev(case.req_id_per_token), case.sm_scale, num_splits=5, workspace=small)


def test_repeated_calls_are_deterministic():
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.memory_bound_decode(seed=14, R=8, ctx_lo=1000, ctx_hi=3000, K=512)
    cache = dev(oracle_cache(case))
    args = (bf16_dev(case.q), cache, dev(case.indices), dev(case.block_table), dev(case.req_id_per_token),
            case.sm_scale)
    o1, l1 = smla.sparse_mla_decode_fp8(*args)
    o2, l2 = smla.sparse_mla_decode_fp8(*args)
    assert (o1 == o2).all() and (l1 == l2).all()


@pytest.mark.parametrize("H", [16, 128])
def test_zero_topk_gives_zero_and_minus_inf(H):
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.memory_bound_decode(seed=14, R=3, ctx_lo=200, ctx_hi=300, K=64, H=H)
    cache = dev(oracle_cache(case))
    idx0 = torch.zeros((case.T, 0), dtype=torch.int32, device="cuda")
    out, lse = smla.sparse_mla_decode_fp8(bf16_dev(case.q), cache, idx0, dev(case.block_table),
                                          dev(case.req_id_per_token), case.sm_scale)
    torch.cuda.synchronize()
    assert smla.read_device_status() == 0
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def _mixed_case_on_device(seed):
    import torch
    case = inp.mixed_batch(seed, n_decode=5, n_prefill=2, prefill_tokens=200, ctx_lo=400, ctx_hi=1500, K=128)
    old = torch.from_numpy(oracle_cache(case, with_new=False)).cuda()
    ref_cache = oracle_cache(case, with_new=True)
    ref_out, ref_lse = oracle.sparse_mla_decode(case.q, ref_cache, case.indices, case.block_table,
                                                case.req_id_per_token, case.sm_scale)
    args = dict(new_rows=bf16_dev(case.new_rows), new_slots=dev(case.new_slots), q=bf16_dev(case.q),
                idx=dev(case.indices), bt=dev(case.block_table), req=dev(case.req_id_per_token))
    return case, old, ref_out, ref_lse, args


def test_store_then_decode_without_host_sync():
    # The decode is launched as a programmatic dependent of the store: its
    # prologue may overlap the store, its reads of the cache may not.
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    case, old, ref_out, ref_lse, a = _mixed_case_on_device(21)
    cache = old.clone()
    torch.cuda.synchronize()
    smla.mla_cache_store_fp8(a["new_rows"], a["new_slots"], cache)
    out, lse = smla.sparse_mla_decode_fp8(a["q"], cache, a["idx"], a["bt"], a["req"], case.sm_scale)
    torch.cuda.synchronize()
    assert_out_close(out.float().cpu().numpy(), ref_out, case.name + " store->decode")
    assert_lse_close(lse.cpu().numpy(), ref_lse, case.name + " store->decode")


def test_store_then_decode_in_a_cuda_graph():
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    case, old, ref_out, ref_lse, a = _mixed_case_on_device(22)
    T, H = case.q.shape[0], case.q.shape[1]
    cache = old.clone()
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = torch.zeros(smla.decode_workspace_bytes(T, H, case.K, 0), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):  # eager once: kernel attributes are set outside the capture
        smla.mla_cache_store_fp8(a["new_rows"], a["new_slots"], cache, stream=stream)
        smla.sparse_mla_decode_fp8(a["q"], cache, a["idx"], a["bt"], a["req"], case.sm_scale, 0, out, lse, ws,
                                   stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        smla.mla_cache_store_fp8(a["new_rows"], a["new_slots"], cache, stream=stream)
        smla.sparse_mla_decode_fp8(a["q"], cache, a["idx"], a["bt"], a["req"], case.sm_scale, 0, out, lse, ws,
                                   stream=stream)
    for _ in range(3):
        cache.copy_(old)  # the rows the store writes are absent again before every replay
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert_out_close(out.float().cpu().numpy(), ref_out, case.name + " graph")
        assert_lse_close(lse.cpu().numpy(), ref_lse, case.name + " graph")
    assert smla.read_device_status(ws) == 0


@pytest.mark.parametrize("H", [16, 128])
def test_back_to_back_decodes_into_the_same_buffers(H):
    # The second call's result must replace the first's, whatever the calls'
    # launches overlap.
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    c1 = inp.memory_bound_decode(seed=31, R=6, ctx_lo=500, ctx_hi=2000, K=256, H=H)
    c2 = inp.memory_bound_decode(seed=32, R=6, ctx_lo=500, ctx_hi=2000, K=256, H=H)
    assert c1.q.shape == c2.q.shape and c1.num_blocks == c2.num_blocks
    T = c1.q.shape[0]
    caches = [dev(oracle_cache(c)) for c in (c1, c2)]
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for c, cache in zip((c1, c2), caches):
        smla.sparse_mla_decode_fp8(bf16_dev(c.q), cache, dev(c.indices), dev(c.block_table),
                                   dev(c.req_id_per_token), c.sm_scale, 0, out, lse)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.sparse_mla_decode(c2.q, oracle_cache(c2), c2.indices, c2.block_table,
                                                c2.req_id_per_token, c2.sm_scale)
    assert_out_close(out.float().cpu().numpy(), ref_out, c2.name + " second call")
    assert_lse_close(lse.cpu().numpy(), ref_lse, c2.name + " second call")


def test_h128_split_tokens_merged_in_the_attention_kernel():
    # 100 tokens of 11 tiles over the resident CTA pairs (14 tiles each): every pair's range holds more
    # than a token, so each split token has two parts, merged in the attention kernel (no combine launch).
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.memory_bound_decode(seed=41, R=100, ctx_lo=800, ctx_hi=3000, K=700, H=128)
    launches, ctas = smla.attention_plan(True, 100, 128, 700, 0)
    assert launches == 2 and ctas >= 2 * 50  # Q preparation + attention, pairs on most SMs
    case.indices[7, 350:] = -1   # parts without valid rows
    case.indices[8, :400] = -1
    case.indices[9, :] = -1      # a token without any
    check_decode(case)
    check_decode(case)  # the merge flags start from zero on the next call too


def test_h128_in_kernel_merge_with_ranges_one_token_long():
    # 77 tokens of 19 tiles (the last one ragged, 48 rows) over 76 CTA pairs: most ranges are exactly one
    # token long, so a pair's first segment is a token's second part and its last the next token's first
    # part, with no whole token in between.
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.memory_bound_decode(seed=42, R=77, ctx_lo=1300, ctx_hi=3000, K=1200, H=128)
    launches, _ = smla.attention_plan(True, 77, 128, 1200, 0)
    assert launches in (2, 3)
    check_decode(case)


@pytest.mark.parametrize("H", [16, 32])
@pytest.mark.parametrize("K", [512, 1000])
@pytest.mark.parametrize("num_splits", [3, 4])
def test_cluster_merge_of_three_and_four_parts(num_splits, K, H):
    # every unit cut into 3 or 4 aligned parts run as one cluster: each CTA writes the value chunks q with
    # q % S == rank and receives the others' values of them (S = 3: ranks own 2, 1, 1 chunks)
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.memory_bound_decode(seed=43, R=5, ctx_lo=1100, ctx_hi=3000, K=K, H=H)
    launches, ctas = smla.attention_plan(True, 5, H, K, num_splits)
    assert launches == 1 and ctas == 5 * (H // 16) * num_splits  # no combine launch: merged in the cluster
    check_decode(case, num_splits=num_splits)


def test_store_launched_after_a_decode_waits_for_it():
    # decode, then a cache store that overwrites 64 rows the decode reads (the store is launched as a
    # programmatic dependent of the decode), then a second decode: the first sees the old rows only,
    # the second the new ones
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.memory_bound_decode(seed=44, R=6, ctx_lo=500, ctx_hi=1500, K=256, H=16)
    cache_old = oracle_cache(case)
    slots = oracle.translate(case.indices, case.block_table, case.req_id_per_token, case.num_blocks)
    tgt = np.unique(slots[slots >= 0])[:64].astype(np.int64)
    rng = np.random.default_rng(45)
    new_rows = inp.bf16_bits((rng.standard_normal((len(tgt), 576)) * 2.0).astype(np.float32))
    cache_new = cache_old.copy()
    oracle.quantize_store(new_rows, tgt, cache_new)
    T = case.q.shape[0]
    d_cache = dev(cache_old)
    q, idx, bt, req = bf16_dev(case.q), dev(case.indices), dev(case.block_table), dev(case.req_id_per_token)
    outs = [torch.empty((T, 16, 512), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    lses = [torch.empty((T, 16), dtype=torch.float32, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    smla.sparse_mla_decode_fp8(q, d_cache, idx, bt, req, case.sm_scale, 0, outs[0], lses[0])
    smla.mla_cache_store_fp8(bf16_dev(new_rows), dev(tgt), d_cache)
    smla.sparse_mla_decode_fp8(q, d_cache, idx, bt, req, case.sm_scale, 0, outs[1], lses[1])
    torch.cuda.synchronize()
    for k, cache in enumerate((cache_old, cache_new)):
        ref_out, ref_lse = oracle.sparse_mla_decode(case.q, cache, case.indices, case.block_table,
                                                    case.req_id_per_token, case.sm_scale)
        assert_out_close(outs[k].float().cpu().numpy(), ref_out, f"decode {k}")
        assert_lse_close(lses[k].cpu().numpy(), ref_lse, f"decode {k}")
    assert np.array_equal(d_cache.cpu().numpy(), cache_new)


@pytest.mark.parametrize("R", [24, 40, 48, 56])
def test_automatic_split_between_token_counts(R):
    # the automatic split for token counts around the SM count's divisors: clusters of 2, 3 or 4 parts where
    # all of them are resident at once, else contiguous ranges with the combine (the choice depends on the
    # GPU's clusters); sampled tokens against the oracle, the first and last included
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.memory_bound_decode(seed=45 + R, R=R, ctx_lo=4096, ctx_hi=9000, K=2048, H=16)
    launches, ctas = smla.attention_plan(True, R, 16, 2048, 0)
    assert launches in (1, 2) and R <= ctas <= 4 * R
    check_decode(case, tokens=sample_tokens(case.T, 6, seed=R))


@pytest.mark.parametrize("R,H,K", [(160, 16, 1024), (24, 48, 2048)])
def test_long_ranges_across_units(R, H, K):
    # more tiles than one ring pass per CTA, ranges that cross unit boundaries (160 tokens x 8 tiles over the
    # SMs), and several 16-head groups per token: the operand buffers' per-panel barriers go through many
    # phases and segments change inside a CTA; sampled tokens against the oracle
    case = inp.memory_bound_decode(seed=46, R=R, ctx_lo=3000, ctx_hi=9000, K=K, H=H)
    check_decode(case, tokens=sample_tokens(case.T, 6, seed=R))
