"""Shared helpers for the GPU parity tests: moving seeded inputs to the
device, running both sides, and the stated tolerances."""
import numpy as np

import oracle
import smla_inputs as inp

# Parity bar: output within atol 1e-2 + rtol 2e-2 of the float64 oracle on the
# same stored bytes; LSE within 1e-3 absolute; cache bytes and slots bit-exact.
OUT_ATOL = 1e-2
OUT_RTOL = 2e-2
LSE_ATOL = 1e-3


def torch_mod():
    import torch
    return torch


def bf16_dev(bits: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev(a: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_out_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outputs outside atol {OUT_ATOL} + rtol {OUT_RTOL}; "
                           f"worst excess {(err - bound).max():.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    return float(err.max())


def assert_lse_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{what}: -inf pattern differs"
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - ref))
    assert np.all(err <= LSE_ATOL), f"{what}: lse max abs error {err.max():.3e} > {LSE_ATOL}"
    return float(err.max())


def oracle_cache(case: inp.DecodeCase, with_new: bool = True) -> np.ndarray:
    cache = inp.make_cache(case, oracle.quantize_store)
    if with_new and len(case.new_slots):
        oracle.quantize_store(case.new_rows, case.new_slots, cache)
    return cache


def run_gpu_decode(case: inp.DecodeCase, cache_np: np.ndarray, num_splits: int = 0, workspace=None,
                   qfp8: bool = False):
    """The decode through the C-ABI (qfp8: its FP8-query variant)."""
    import sparse_mla_attention_fp8_gb300 as smla
    fn = smla.sparse_mla_decode_fp8_qfp8 if qfp8 else smla.sparse_mla_decode_fp8
    out, lse = fn(bf16_dev(case.q), dev(cache_np), dev(case.indices),
                                          dev(case.block_table), dev(case.req_id_per_token), case.sm_scale,
                                          num_splits=num_splits, workspace=workspace)
    torch = torch_mod()
    torch.cuda.synchronize()
    assert smla.read_device_status(workspace) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check_decode(case: inp.DecodeCase, num_splits: int = 0, tokens=None, cache_np=None, qfp8: bool = False):
    if cache_np is None:
        cache_np = oracle_cache(case)
    out, lse = run_gpu_decode(case, cache_np, num_splits, qfp8=qfp8)
    ref_out, ref_lse = oracle.sparse_mla_decode(case.q, cache_np, case.indices, case.block_table,
                                                case.req_id_per_token, case.sm_scale, tokens=tokens)
    sel = slice(None) if tokens is None else np.asarray(tokens)
    e1 = assert_out_close(out[sel], ref_out, case.name)
    e2 = assert_lse_close(lse[sel], ref_lse, case.name)
    return e1, e2


def sample_tokens(T: int, n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set([0, T - 1])
    pick.update(rng.choice(T, size=min(n, T), replace=False).tolist())
    return np.array(sorted(pick), np.int32)
