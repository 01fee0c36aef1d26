"""GPU parity: quantize-and-store and index translation, bit-exact against
the oracle."""
import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import bf16_dev, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


def _rows(seed, n):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 576)).astype(np.float32)
    x[:, rng.choice(576, 6, replace=False)] *= 8.0
    x[1, 0:128] = 0.0                 # zero group -> scale 0, codes 0
    x[2, 256:384] *= 1e-39            # scale underflows to 0 or a float32 denormal
    x[3, 384:512] *= 3e-36            # tiny but normal scale: subnormal e4m3 codes
    x[4, 128:256] = 0.0
    x[4, 200] = -1e-3                 # one non-zero value in a group
    x[5] *= 1e30                      # large magnitudes
    x[6, 130] = -0.0
    return inp.bf16_bits(x)


@pytest.mark.parametrize("seed,n,NB", [(0, 37, 2), (1, 300, 9), (2, 4096, 80)])
def test_store_bit_exact(smla, seed, n, NB):
    import torch
    rows = _rows(seed, n)
    rng = np.random.default_rng(seed + 100)
    slots = rng.permutation(NB * 64)[:n].astype(np.int64)
    slots[rng.choice(n, size=max(1, n // 10), replace=False)] = -1  # skipped tokens
    slots[0] = NB * 64 + 5                                          # out of range -> skipped
    ref = np.full((NB, 64, 656), 0xAB, np.uint8)
    oracle.quantize_store(rows, slots, ref)
    cache = torch.full((NB, 64, 656), 0xAB, dtype=torch.uint8, device="cuda")
    smla.mla_cache_store_fp8(bf16_dev(rows), dev(slots), cache)
    got = cache.cpu().numpy()
    diff = np.nonzero(got.reshape(-1, 656) != ref.reshape(-1, 656))
    assert diff[0].size == 0, f"{diff[0].size} bytes differ, first at row {diff[0][0]} byte {diff[1][0]}"


def test_store_mixed_batch_new_tokens_bit_exact(smla):
    import torch
    case = inp.mixed_batch(4, n_decode=8, n_prefill=1, prefill_tokens=300, ctx_lo=600, ctx_hi=3000, K=128)
    ref = inp.make_cache(case, oracle.quantize_store)
    cache = torch.from_numpy(ref.copy()).cuda()
    oracle.quantize_store(case.new_rows, case.new_slots, ref)
    smla.mla_cache_store_fp8(bf16_dev(case.new_rows), dev(case.new_slots), cache)
    assert np.array_equal(cache.cpu().numpy(), ref)


@pytest.mark.parametrize("seed", [0, 1])
def test_translate_bit_exact_with_invalid_entries(smla, seed):
    rng = np.random.default_rng(seed)
    R, MB, NB = 7, 33, 150
    bt = rng.integers(-2, NB + 4, size=(R, MB)).astype(np.int32)
    T, K = 50, 2048 + 37
    req = rng.integers(-1, R + 1, size=T).astype(np.int32)
    idx = rng.integers(-5, MB * 64 + 200, size=(T, K)).astype(np.int32)
    ref = oracle.translate(idx, bt, req, NB)
    got = smla.sparse_mla_translate_indices(dev(idx), dev(bt), dev(req), NB).cpu().numpy()
    assert np.array_equal(got, ref)


def test_translate_memory_bound_workload(smla):
    case = inp.memory_bound_decode(1)
    ref = oracle.translate(case.indices, case.block_table, case.req_id_per_token, case.num_blocks)
    got = smla.sparse_mla_translate_indices(dev(case.indices), dev(case.block_table), dev(case.req_id_per_token),
                                            case.num_blocks).cpu().numpy()
    assert np.array_equal(got, ref)
    assert (ref >= 0).all()
