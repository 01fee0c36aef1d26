"""GPU: the allocation-free decode entry point (fixed library scratch instead
of a workspace) against the workspace entry point and against the float64
oracle on the same inputs, two calls in a row with different inputs, through
the C ABI."""
import ctypes

import numpy as np
import pytest

import oracle
import smla_inputs as inp
from helpers import assert_lse_close, assert_out_close, bf16_dev, dev, oracle_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def smla():
    import sparse_mla_attention_fp8_gb300 as m
    m.build()
    return m


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc_call(smla, case, cache, out, lse, num_splits):
    import torch
    q = bf16_dev(case.q)
    idx, bt, req = dev(case.indices), dev(case.block_table), dev(case.req_id_per_token)
    T, H, _ = case.q.shape
    K = case.indices.shape[1]
    R, MB = case.block_table.shape
    NB = cache.shape[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = smla.lib().sparse_mla_decode_fp8_noalloc(_ptr(q), _ptr(cache), _ptr(idx), _ptr(bt), _ptr(req),
                                                 ctypes.c_float(case.sm_scale), num_splits, _ptr(out), _ptr(lse),
                                                 T, H, K, R, MB, NB, stream)
    assert rc == 0, smla.lib().smla_last_error().decode()
    torch.cuda.synchronize()


def _workspace_call(smla, case, cache, num_splits):
    import torch
    out, lse = smla.sparse_mla_decode_fp8(bf16_dev(case.q), cache, dev(case.indices), dev(case.block_table),
                                          dev(case.req_id_per_token), case.sm_scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_noalloc_matches_workspace_entry_point_twice(smla, num_splits, H):
    import torch
    # two different batches (ragged top-k of 200 = 3 full tiles + a tail of 8), same shapes; H = 128 runs
    # the CTA-pair kernel, whose prepared Q also lives in the fixed scratch
    cases = [inp.memory_bound_decode(seed=s, R=9, ctx_lo=300, ctx_hi=2500, K=200, H=H) for s in (5, 15)]
    T, H, _ = cases[0].q.shape
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    for case in cases:
        cache_np = oracle_cache(case)
        cache = dev(cache_np)
        ws_out, ws_lse = _workspace_call(smla, case, cache, num_splits)
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        _noalloc_call(smla, case, cache, out, lse, num_splits)
        got_out, got_lse = out.float().cpu().numpy(), lse.cpu().numpy()
        assert np.all(np.isfinite(got_out))
        assert_out_close(got_out, ws_out, case.name + " noalloc vs workspace entry point")
        assert_lse_close(got_lse, ws_lse, case.name + " noalloc vs workspace entry point")
        ref_out, ref_lse = oracle.sparse_mla_decode(case.q, cache_np, case.indices, case.block_table,
                                                    case.req_id_per_token, case.sm_scale)
        assert_out_close(got_out, ref_out, case.name + " noalloc vs oracle")
        assert_lse_close(got_lse, ref_lse, case.name + " noalloc vs oracle")
    assert smla.read_noalloc_status() == 0


def test_noalloc_rejects_work_beyond_the_fixed_scratch(smla):
    import torch
    # 4096 tokens x 16 heads over all SMs needs > 32 MiB of partial results
    T, H, K, R, MB, NB = 4096, 16, 64, 1, 1, 1
    q = torch.zeros((T, H, 576), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((NB, 64, 656), dtype=torch.uint8, device="cuda")
    idx = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    bt = torch.zeros((R, MB), dtype=torch.int32, device="cuda")
    req = torch.zeros((T,), dtype=torch.int32, device="cuda")
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    need = smla.lib().sparse_mla_decode_workspace_bytes(T, H, K, 0)
    assert need > (32 << 20)
    rc = smla.lib().sparse_mla_decode_fp8_noalloc(_ptr(q), _ptr(cache), _ptr(idx), _ptr(bt), _ptr(req),
                                                 ctypes.c_float(0.1), 0, _ptr(out), _ptr(lse), T, H, K, R, MB, NB,
                                                 None)
    assert rc == -4
    assert "scratch" in smla.lib().smla_last_error().decode()
