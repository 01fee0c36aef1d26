"""GPU parity: MLA weight absorption around the attention (the query's NoPE
part times W_UK_T per head with the RoPE part appended; the V up-projection)
against the float64 oracle.  The GPU accumulates bf16 products in fp32 and
rounds the result to bf16 once, so each element is within half a bf16 unit
of the exact value plus the fp32 accumulation error:
|gpu - exact| <= 2^-8 |exact| + 2^-14 sum_k |a_k b_k|.  The appended RoPE
part is bit-exact."""
import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import bf16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


def _bits(rng, shape, scale):
    return inp.bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def _f64(bits):
    return inp.bits_to_float(bits).astype(np.float64)


def _check(got_bits, ref, bound_abs):
    got = _f64(got_bits)
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * bound_abs
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside; worst excess {(err - bound).max():.3e}"


def _to_bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("T,H", [(1, 16), (100, 16), (257, 128)])
def test_absorb_q(T, H):
    rng = np.random.default_rng(T + H)
    P = 128
    q = _bits(rng, (T, H, P + 64), 1.0)
    w = _bits(rng, (H, P, 512), 0.08)
    import sparse_mla_attention_fp8_gb300 as smla
    out = smla.mla_absorb_q(bf16_dev(q), bf16_dev(w))
    got = _to_bits(out)
    ref = oracle.absorb_q(q, w)
    absprod = oracle.absorb_q(inp.bf16_bits(np.abs(_f64(q)).astype(np.float32)),
                              inp.bf16_bits(np.abs(_f64(w)).astype(np.float32)))[..., :512]
    _check(got[..., :512], ref[..., :512], absprod)
    assert np.array_equal(got[..., 512:], q[..., P:])  # the RoPE part, copied


@pytest.mark.parametrize("T,H,V", [(1, 16, 128), (100, 16, 128), (257, 128, 128), (64, 16, 256)])
def test_v_up_proj(T, H, V):
    rng = np.random.default_rng(T + H + V)
    a = _bits(rng, (T, H, 512), 1.0)
    w = _bits(rng, (H, 512, V), 0.05)
    import sparse_mla_attention_fp8_gb300 as smla
    out = smla.mla_v_up_proj(bf16_dev(a), bf16_dev(w))
    ref = oracle.v_up_proj(a, w)
    absprod = oracle.v_up_proj(inp.bf16_bits(np.abs(_f64(a)).astype(np.float32)),
                               inp.bf16_bits(np.abs(_f64(w)).astype(np.float32)))
    _check(_to_bits(out), ref, absprod)


def test_absorb_then_decode_then_v_up_matches_the_oracle_chain():
    # One MLA attention step around the kernel: the absorbed query feeds the FP8 decode, whose output
    # feeds the V up-projection; each stage is compared with the oracle on the GPU's previous stage.
    import torch
    import sparse_mla_attention_fp8_gb300 as smla
    from helpers import assert_lse_close, assert_out_close, dev, oracle_cache
    case = inp.memory_bound_decode(seed=31, R=6, ctx_lo=300, ctx_hi=1500, K=256, H=16)
    rng = np.random.default_rng(31)
    P, V = 128, 128
    q_raw = _bits(rng, (case.T, 16, P + 64), 1.0)
    w_uk = _bits(rng, (16, P, 512), 0.08)
    w_uv = _bits(rng, (16, 512, V), 0.05)
    q = smla.mla_absorb_q(bf16_dev(q_raw), bf16_dev(w_uk))
    cache = oracle_cache(case)
    out, lse = smla.sparse_mla_decode_fp8(q, dev(cache), dev(case.indices), dev(case.block_table),
                                          dev(case.req_id_per_token), case.sm_scale)
    y = smla.mla_v_up_proj(out, bf16_dev(w_uv))
    torch.cuda.synchronize()
    q_bits = _to_bits(q)
    ref_out, ref_lse = oracle.sparse_mla_decode(q_bits, cache, case.indices, case.block_table,
                                                case.req_id_per_token, case.sm_scale)
    assert_out_close(out.float().cpu().numpy(), ref_out, "decode of the absorbed query")
    assert_lse_close(lse.cpu().numpy(), ref_lse, "decode of the absorbed query")
    out_bits = _to_bits(out)
    absprod = oracle.v_up_proj(inp.bf16_bits(np.abs(_f64(out_bits)).astype(np.float32)),
                               inp.bf16_bits(np.abs(_f64(w_uv)).astype(np.float32)))
    _check(_to_bits(y), oracle.v_up_proj(out_bits, w_uv), absprod)
