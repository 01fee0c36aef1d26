"""GPU parity over the whole range of legal cache rows: scale groups whose
amax is far above f16's largest value (65504) or far below its normal range,
against the float64 oracle at the stated tolerance (output atol 1e-2 + rtol
2e-2, LSE atol 1e-3), on both the 16-head kernel and the 128-head CTA-pair
kernel.

The "FP8 with scale" row of vLLM flashmla_sparse.py (module docstring) keeps
one float32 scale per group of 128 values, so any finite amax is a valid
row; the quantize-and-store step writes such rows for any bf16 input.  The
query is scaled inversely on the same channels so that the logits stay of
order one (otherwise an LSE tolerance of 1e-3 would be below the float32
resolution of the logits themselves).  Scale groups of very large values
hold values of one sign, so that the output elements do not cancel to far
below the magnitude of the terms that make them (an atol of 1e-2 is a
relative bound of 1e-7 at 1e5)."""
import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import check_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


def _scale_groups(case: inp.DecodeCase, factor: np.ndarray, one_signed: np.ndarray) -> inp.DecodeCase:
    """Multiply the NoPE scale group g of every cache row that token t reads by
    factor[t, g] (taking |x| first where one_signed[t, g]), and q[t, :, group g]
    by 1 / factor[t, g].  Needs rows read by one token only (one query token
    per request, requests own disjoint blocks)."""
    slots = oracle.translate(case.indices, case.block_table, case.req_id_per_token, case.num_blocks)
    rows = inp.bits_to_float(case.cache_rows).copy()
    q = inp.bits_to_float(case.q).copy()
    pos = np.searchsorted(case.cache_slots, slots)
    seen = np.zeros(len(case.cache_slots), bool)
    for t in range(case.T):
        ri = np.unique(pos[t][slots[t] >= 0])
        assert not seen[ri].any(), "a cache row is read by two tokens"
        seen[ri] = True
        for g in range(4):
            cols = slice(128 * g, 128 * g + 128)
            blk = rows[np.ix_(ri, np.arange(128 * g, 128 * g + 128))]
            if one_signed[t, g]:
                blk = np.abs(blk)
            rows[np.ix_(ri, np.arange(128 * g, 128 * g + 128))] = blk * np.float32(factor[t, g])
            q[t, :, cols] /= np.float32(factor[t, g])
    case.cache_rows = inp.bf16_bits(rows)
    case.q = inp.bf16_bits(q)
    return case


# per-token factors: amax of about 1e5 .. 1e9 (scales far above f16's range
# for the largest), about 1e-3 (scales below f16's normal range) and 1e-6
# (scales below f16's smallest subnormal)
TOKEN_FACTORS = [1.0, 5e4, 2e-4, 1e7, 1e-7, 3e5, 1e-3, 1.0]
BIG = 1e3


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_scale_range_per_token(H, num_splits):
    # 8 requests x 1 token, K = 200 (3 full tiles and a ragged tail), 1 % outlier channels x8
    case = inp.memory_bound_decode(seed=41, R=8, ctx_lo=300, ctx_hi=2500, K=200, H=H)
    f = np.repeat(np.asarray(TOKEN_FACTORS, np.float64)[:, None], 4, axis=1)
    case = _scale_groups(case, f, f > BIG)
    cache = inp.make_cache(case, oracle.quantize_store)
    scales = cache[..., 512:528].copy().view(np.float32)
    assert scales.max() > 65504 and 0 < scales[scales > 0].min() < 2.0 ** -24  # both ends of f16 are crossed
    check_decode(case, num_splits=num_splits, cache_np=cache)


@pytest.mark.parametrize("H", [16, 128])
def test_scale_range_across_groups_of_a_row(H):
    # every row holds one group of large one-signed values (amax > 1e5) and
    # groups 1, 1e-1 and 1e-2 times the latent; the large group rotates with
    # the token, so it lands in either CTA's half of the 128-head kernel
    case = inp.memory_bound_decode(seed=42, R=8, ctx_lo=300, ctx_hi=2500, K=200, H=H)
    base = np.array([4e4, 1.0, 1e-1, 1e-2])
    f = np.stack([np.roll(base, t) for t in range(case.T)])
    case = _scale_groups(case, f, f > BIG)
    check_decode(case)
    check_decode(case, num_splits=2)
