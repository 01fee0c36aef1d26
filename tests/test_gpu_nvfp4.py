"""GPU parity of the NVFP4 cache (the 352-byte nvfp4_ds_mla row of vLLM PR
#59342, in the layout read for it): quantize-and-store bit-exact against the
oracle's bytes, and the decode over the stored rows against the float64
oracle at the decode's tolerance (atol 1e-2 + rtol 2e-2 on the output, 1e-3
on the LSE), for 16 and 128 heads and the pages' native top-k widths."""
import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import assert_lse_close, assert_out_close, bf16_dev, dev, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


def _nvfp4_cache(case):
    cache = inp.make_cache(case, oracle.nvfp4_quantize_store, row_bytes=352)
    if len(case.new_slots):
        oracle.nvfp4_quantize_store(case.new_rows, case.new_slots, cache)
    return cache


def _check(case, num_splits=0, tokens=None, cache=None):
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    cache = _nvfp4_cache(case) if cache is None else cache
    out, lse = smla.sparse_mla_decode_nvfp4(bf16_dev(case.q), dev(cache), dev(case.indices), dev(case.block_table),
                                            dev(case.req_id_per_token), case.sm_scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert smla.read_device_status() == 0
    ref_out, ref_lse = oracle.sparse_mla_decode_nvfp4(case.q, cache, case.indices, case.block_table,
                                                      case.req_id_per_token, case.sm_scale, tokens=tokens)
    sel = slice(None) if tokens is None else np.asarray(tokens)
    assert_out_close(out.float().cpu().numpy()[sel], ref_out, case.name + " nvfp4")
    assert_lse_close(lse.cpu().numpy()[sel], ref_lse, case.name + " nvfp4")


def test_store_is_bit_exact():
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    rng = np.random.default_rng(31)
    T = 300
    x = rng.standard_normal((T, 576), dtype=np.float32) * np.exp(rng.uniform(-8, 5, (T, 1))).astype(np.float32)
    x[5, 16:32] = 0.0                         # a zero block
    x[6, :16] = [6, -6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, 0.375, -0.3125, 0, 1, 2, 3, 4]  # ties of the E2M1 grid
    x[7, :16] = -1e-3                         # codes that round to -0
    x[7, 0] = -6.0
    x[8, 512:] = rng.choice([448.0, 500.0, -1e4, 2.0 ** -11, 2.0 ** -9, 0.0], 64)  # RoPE saturation and underflow
    x[9, 32:48] = 1e4                         # block scales that saturate (amax / 6 > 448)
    bits = inp.bf16_bits(x)
    NB = 8
    slots = rng.permutation(NB * 64)[:T].astype(np.int64)
    slots[10] = -1                            # skipped tokens
    slots[11] = NB * 64
    want = np.full((NB, 64, 352), 0x5A, np.uint8)
    oracle.nvfp4_quantize_store(bits, slots, want)
    got = torch.full((NB, 64, 352), 0x5A, dtype=torch.uint8, device="cuda")
    smla.mla_cache_store_nvfp4(bf16_dev(bits), dev(slots), got)
    got = got.cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, [(tuple(b), hex(got[tuple(b)]), hex(want[tuple(b)])) for b in bad[:8]]


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("K", [512, 1024, 2048])
def test_decode_native_topk_widths(K, H):
    case = inp.memory_bound_decode(seed=61, R=6, ctx_lo=2100, ctx_hi=4000, K=K, H=H)
    _check(case)


@pytest.mark.parametrize("H", [32, 48])
def test_decode_several_head_groups(H):
    # below 128 heads the NVFP4 decode runs 16-head groups: H / 16 units per token
    case = inp.memory_bound_decode(seed=65, R=5, ctx_lo=900, ctx_hi=2000, K=700, H=H)
    _check(case)
    _check(case, num_splits=2)


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_ragged_topk_and_splits(num_splits, H):
    # K = 200: three full tiles of 64 rows and a ragged tail of 8 (H = 128 stages the rows)
    case = inp.memory_bound_decode(seed=62, R=9, ctx_lo=300, ctx_hi=2500, K=200, H=H)
    _check(case, num_splits=num_splits)


@pytest.mark.parametrize("H", [16, 128])
def test_decode_invalid_rows_single_rows_and_zero_topk(H):
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.memory_bound_decode(seed=63, R=5, ctx_lo=700, ctx_hi=900, K=180, H=H)
    case.indices[:, 100:140] = case.indices[:, 0:40]          # duplicates count once per occurrence
    case.indices[0, 5] = case.block_table.shape[1] * 64 + 3    # block id >= MB
    case.indices[1, :] = -1                                    # a token without any valid row
    case.indices[2, :] = -1
    case.indices[2, 17] = 40                                   # a token with one row
    case.block_table[3, 1] = -4                                # negative physical block
    _check(case)
    cache = dev(_nvfp4_cache(case))
    idx0 = torch.zeros((case.T, 0), dtype=torch.int32, device="cuda")
    out, lse = smla.sparse_mla_decode_nvfp4(bf16_dev(case.q), cache, idx0, dev(case.block_table),
                                            dev(case.req_id_per_token), case.sm_scale)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_store_then_decode():
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    case = inp.mixed_batch(5, n_decode=5, n_prefill=2, prefill_tokens=200, ctx_lo=400, ctx_hi=1500, K=128)
    ref_cache = _nvfp4_cache(case)
    old = inp.make_cache(case, oracle.nvfp4_quantize_store, row_bytes=352)
    cache = torch.from_numpy(old).cuda()
    smla.mla_cache_store_nvfp4(bf16_dev(case.new_rows), dev(case.new_slots), cache)
    assert np.array_equal(cache.cpu().numpy(), ref_cache)
    _check(case, cache=ref_cache)


def test_full_size_decode_h16_k2048():
    # the memory-bound decode's shape (64 requests x 1 token, top-k 2048), sampled tokens against the oracle
    case = inp.memory_bound_decode(seed=64, R=64, ctx_lo=8192, ctx_hi=8192, K=2048, H=16)
    _check(case, tokens=sample_tokens(case.T, 12, seed=5))
