"""Randomized GPU parity of the FP8 decode (a fixed seed, so the cases are the
same on every run): random token counts, head counts 16..80 (the 16-head-group
kernel with several groups per token), top-k 1..2048, contexts, split modes
and invalid indices, each against the float64 oracle on sampled tokens, and
each re-run for bit-identical results (the merge orders are fixed)."""
import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import assert_lse_close, assert_out_close, oracle_cache, run_gpu_decode, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


def _cases(n, seed=7):
    rng = np.random.default_rng(seed)
    for i in range(n):
        R = int(rng.integers(1, 97))
        H = int(rng.choice([16, 32, 48, 64, 80]))
        K = int(rng.integers(1, 2049))
        ns = int(rng.choice([0, 0, 0, 1, 2, 3, 4, 5]))
        lo = max(K, int(rng.integers(64, 6000)))
        hi = lo + int(rng.integers(0, 4000))
        case = inp.memory_bound_decode(seed=int(rng.integers(1 << 30)), R=R, ctx_lo=lo, ctx_hi=hi, K=K, H=H)
        if rng.random() < 0.3:
            case.indices[rng.random(case.indices.shape) < 0.1] = -1
        yield i, case, ns


def test_random_shapes_and_splits():
    for i, case, ns in _cases(40):
        cache = oracle_cache(case)
        toks = sample_tokens(case.T, 4, seed=i)
        out, lse = run_gpu_decode(case, cache, ns)
        ref_out, ref_lse = oracle.sparse_mla_decode(case.q, cache, case.indices, case.block_table,
                                                    case.req_id_per_token, case.sm_scale, tokens=toks)
        what = f"case {i}: T={case.T} H={case.H} K={case.K} num_splits={ns}"
        assert_out_close(out[toks], ref_out, what)
        assert_lse_close(lse[toks], ref_lse, what)
        out2, lse2 = run_gpu_decode(case, cache, ns)
        assert np.array_equal(out2.view(np.uint32), out.view(np.uint32)), what + ": output differs between runs"
        assert np.array_equal(lse2.view(np.uint32), lse.view(np.uint32)), what + ": lse differs between runs"
