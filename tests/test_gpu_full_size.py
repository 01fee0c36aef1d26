"""GPU parity at the five workloads' full sizes, in the launch configuration
the benchmark times (automatic work split).  Where the oracle would take too
long, it is evaluated on a seeded sample of tokens that always includes the
first and the last."""
import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import (assert_lse_close, assert_out_close, bf16_dev, check_decode, dev, oracle_cache,
                     sample_tokens)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


def test_full_tiny_decode():
    check_decode(inp.tiny_decode(0))


def test_full_memory_bound_decode_h16_k2048():
    case = inp.memory_bound_decode(1)
    check_decode(case)  # all 64 tokens


def test_full_tensor_bound_decode_h128_k2048():
    case = inp.tensor_bound_decode(2)
    check_decode(case, tokens=sample_tokens(case.T, 10, seed=2))


def test_full_prefill_h128_k2048():
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.prefill(3)
    out, lse = smla.sparse_mla_prefill_bf16(bf16_dev(case.q), bf16_dev(case.kv), dev(case.indices), case.sm_scale)
    torch.cuda.synchronize()
    assert smla.read_device_status() == 0
    tok = sample_tokens(case.T, 6, seed=3)
    ref_out, ref_lse = oracle.sparse_mla_prefill(case.q, case.kv, case.indices, case.sm_scale, tokens=tok)
    assert_out_close(out.float().cpu().numpy()[tok], ref_out, case.name)
    assert_lse_close(lse.cpu().numpy()[tok], ref_lse, case.name)


def test_full_mixed_batch_store_then_decode():
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.mixed_batch(4)
    ref_cache = oracle_cache(case, with_new=True)
    cache = torch.from_numpy(oracle_cache(case, with_new=False)).cuda()
    smla.mla_cache_store_fp8(bf16_dev(case.new_rows), dev(case.new_slots), cache)
    got = cache.cpu().numpy()
    assert np.array_equal(got, ref_cache), "cache bytes differ after quantize-and-store"
    out, lse = smla.sparse_mla_decode_fp8(bf16_dev(case.q), cache, dev(case.indices), dev(case.block_table),
                                          dev(case.req_id_per_token), case.sm_scale)
    torch.cuda.synchronize()
    tok = sample_tokens(case.T, 40, seed=4)
    tok = np.unique(np.concatenate([tok, np.arange(64, dtype=np.int32)]))  # every speculative decode token
    ref_out, ref_lse = oracle.sparse_mla_decode(case.q, ref_cache, case.indices, case.block_table,
                                                case.req_id_per_token, case.sm_scale, tokens=tok)
    assert_out_close(out.float().cpu().numpy()[tok], ref_out, case.name)
    assert_lse_close(lse.cpu().numpy()[tok], ref_lse, case.name)
