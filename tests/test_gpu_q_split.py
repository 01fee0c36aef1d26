"""GPU: the e4m3 hi + lo split of the query (the 16-head decode, and the
FP8-query decode at 128 heads), checked against its stated error bound rather
than against the parity tolerance alone.

The split scales each (head, 128-column group) of q by a power of two that
puts the group's largest magnitude in (224, 448], rounds to f16 (exact for
bf16 inputs in range), takes hi = e4m3(x) and lo = e4m3(x - hi).  Per
component |q - (hi + lo)| <= 2^-8 |q| + 2^-17 max_group |q|: hi and lo carry
3 stored mantissa bits each, and e4m3's smallest subnormal (2^-9) sets the
absolute floor.  The logits are exact sums of products otherwise (fp32
accumulation, scales applied in fp32), and the LSE is 1-Lipschitz in the
maximum norm of the logits, so
  |lse_gpu - lse_exact| <= sm_scale * max_j sum_i (2^-8 |q_i| + 2^-17 m_g(i)) |k_ji|
up to fp32 rounding.  The query here spans 15 binary orders of magnitude
inside every group, where a single e4m3 term would be far off.  With 128
heads the CTA pair's 16-bit exchange of partial logits adds its own bound."""
import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import oracle_cache, run_gpu_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


def _bf16_value(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("H, qfp8", [(16, False), (128, True)])
def test_q_split_error_within_its_bound(H, qfp8):
    case = inp.memory_bound_decode(seed=51, R=8, ctx_lo=300, ctx_hi=900, K=256, H=H)
    rng = np.random.default_rng(52)
    T, H = case.q.shape[:2]
    # magnitudes log-uniform over 2^-14 .. 2^0 in every group, random signs; RoPE part as generated
    q = _bf16_value(case.q).reshape(T, H, 576)
    mag = np.exp2(rng.uniform(-14.0, 0.0, size=(T, H, 512)))
    q[..., :512] = np.where(rng.random((T, H, 512)) < 0.5, -mag, mag) * 3.0
    case.q = inp.bf16_bits(q.astype(np.float32))
    qv = _bf16_value(case.q).reshape(T, H, 576)

    cache = oracle_cache(case)
    out, lse = run_gpu_decode(case, cache, qfp8=qfp8)
    ref_out, ref_lse = oracle.sparse_mla_decode(case.q, cache, case.indices, case.block_table,
                                                case.req_id_per_token, case.sm_scale)
    slots = oracle.translate(case.indices, case.block_table, case.req_id_per_token, case.num_blocks)
    rows = cache.reshape(-1, 656)
    worst = 0.0
    for t in range(T):
        valid = slots[t][slots[t] >= 0]
        kfull = np.stack([oracle.dequant_row(rows[s]) for s in valid])  # [n, 576]
        kmat = kfull[:, :512]
        for h in range(H):
            qn = qv[t, h, :512]
            gmax = np.repeat(np.abs(qn).reshape(4, 128).max(axis=1), 128)
            dq = 2.0 ** -8 * np.abs(qn) + 2.0 ** -17 * gmax
            bound = case.sm_scale * float(np.max(np.abs(kmat) @ dq))
            bound += 1e-6 * (1.0 + case.sm_scale * float(np.max(np.abs(kmat) @ np.abs(qn))))  # fp32 rounding
            if H == 128:
                # the CTA pair trades partial logits in 16-bit fixed point: off by at most
                # 2^-16 of the largest partial magnitude, itself <= sm_scale sum_i |q_i| |k_ji|
                bound += 2.0 ** -16 * case.sm_scale * float(np.max(np.abs(kfull) @ np.abs(qv[t, h])))
            err = abs(float(lse[t, h]) - float(ref_lse[t, h]))
            assert err <= bound, (t, h, err, bound)
            worst = max(worst, err / bound)
    # the bound is not vacuous: the outputs stay within the parity tolerance too
    assert np.max(np.abs(out - ref_out) - 2e-2 * np.abs(ref_out)) <= 1e-2
    assert worst <= 1.0
