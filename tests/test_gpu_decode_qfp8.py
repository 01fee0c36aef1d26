"""GPU parity of the FP8-query decode (sparse_mla_decode_fp8_qfp8): the query
in two e4m3 terms, both products on the FP8 tensor path, the row scales folded
into the logits and into P.  At 128 heads it runs a CTA-pair kernel of its own;
it answers to the same float64 oracle and the same tolerance as the decode
(atol 1e-2 + rtol 2e-2 on the output, 1e-3 on the LSE)."""
import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import check_decode, oracle_cache, run_gpu_decode, sample_tokens
from test_gpu_range import BIG, TOKEN_FACTORS, _scale_groups

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


@pytest.mark.parametrize("num_splits", [0, 1, 2, 3, 5])
def test_ragged_topk_several_tiles(num_splits):
    # K = 200: three full tiles of 64 rows and a ragged tail of 8
    case = inp.memory_bound_decode(seed=5, R=9, ctx_lo=300, ctx_hi=2500, K=200, H=128)
    check_decode(case, num_splits=num_splits, qfp8=True)


def test_sixteen_heads_is_the_decode():
    # below 128 heads the decode already computes this way: the same kernel, the same bytes
    case = inp.memory_bound_decode(seed=5, R=9, ctx_lo=300, ctx_hi=2500, K=200, H=16)
    cache = oracle_cache(case)
    o1, l1 = run_gpu_decode(case, cache)
    o2, l2 = run_gpu_decode(case, cache, qfp8=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("K", [1, 37, 64, 65, 2048])
def test_topk_widths(K):
    case = inp.memory_bound_decode(seed=7, R=6, ctx_lo=2100, ctx_hi=4000, K=K, H=128)
    check_decode(case, qfp8=True)


def test_invalid_rows_single_rows_and_duplicates():
    case = inp.memory_bound_decode(seed=8, R=4, ctx_lo=200, ctx_hi=400, K=130, H=128)
    case.indices[:] = -1
    out, lse = run_gpu_decode(case, oracle_cache(case), qfp8=True)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    case.indices[1, 77] = 5  # one token with a single valid row: out is that row's dequantized values
    check_decode(case, qfp8=True)
    check_decode(case, num_splits=2, qfp8=True)
    case = inp.memory_bound_decode(seed=10, R=5, ctx_lo=700, ctx_hi=900, K=180, H=128)
    case.indices[:, 100:140] = case.indices[:, 0:40]          # duplicates count once per occurrence
    case.indices[0, 5] = case.block_table.shape[1] * 64 + 3    # block id >= MB
    case.indices[1, 7] = -77
    case.block_table[2, 3] = case.num_blocks + 9               # physical block >= NB
    case.block_table[3, 1] = -4                                # negative physical block
    check_decode(case, qfp8=True)


def test_zero_topk_gives_zero_and_minus_inf():
    case = inp.memory_bound_decode(seed=14, R=3, ctx_lo=200, ctx_hi=300, K=64, H=128)
    case.indices = case.indices[:, :0].copy()
    out, lse = run_gpu_decode(case, oracle_cache(case), qfp8=True)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_split_tokens_merged_in_the_attention_kernel():
    # every pair's range holds more than a token: split tokens have two parts, merged in the kernel
    case = inp.memory_bound_decode(seed=41, R=100, ctx_lo=800, ctx_hi=3000, K=700, H=128)
    case.indices[7, 350:] = -1   # parts without valid rows
    case.indices[8, :400] = -1
    case.indices[9, :] = -1      # a token without any
    check_decode(case, qfp8=True)
    check_decode(case, qfp8=True)  # the merge flags start from zero on the next call too


def test_ranges_one_token_long():
    case = inp.memory_bound_decode(seed=42, R=77, ctx_lo=1300, ctx_hi=3000, K=1200, H=128)
    check_decode(case, qfp8=True)


@pytest.mark.parametrize("num_splits", [0, 3])
def test_scale_range_per_token(num_splits):
    # scale groups far above f16's range and far below it: R_g, the running power-of-two
    # bound of a group's scales, and P' = p sc / R_g 2^7 must hold over the whole range
    case = inp.memory_bound_decode(seed=41, R=8, ctx_lo=300, ctx_hi=2500, K=200, H=128)
    f = np.repeat(np.asarray(TOKEN_FACTORS, np.float64)[:, None], 4, axis=1)
    case = _scale_groups(case, f, f > BIG)
    cache = inp.make_cache(case, oracle.quantize_store)
    check_decode(case, num_splits=num_splits, cache_np=cache, qfp8=True)


def test_repeated_calls_are_deterministic():
    case = inp.memory_bound_decode(seed=12, R=20, ctx_lo=900, ctx_hi=2000, K=512, H=128)
    cache = oracle_cache(case)
    o1, l1 = run_gpu_decode(case, cache, qfp8=True)
    o2, l2 = run_gpu_decode(case, cache, qfp8=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_full_tensor_bound_decode_h128_k2048():
    # the 128-request, top-k 2048 workload with its outlier channels, sampled tokens against the oracle
    case = inp.tensor_bound_decode(2)
    check_decode(case, tokens=sample_tokens(case.T, 10, seed=2), qfp8=True)
