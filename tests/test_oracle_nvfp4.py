"""Pins for the oracle's NVFP4 cache (CPU only): the 352-byte row of vLLM PR
#59342 ("Purpose": nvfp4_ds_mla, 352 bytes per token), in the layout and
quantizer read for it in oracle/smla_oracle.c (reading R13).

The oracle is checked against things other than itself: the OCP MX FP4 E2M1
value table (tests/golden/e2m1_values.txt), a brute-force nearest search on
that table, a hand-worked row (tests/golden/nvfp4_row.txt), torch's
float8_e4m3fn for the scale and RoPE bytes, and dense attention through
torch's scaled_dot_product_attention in float64."""
import os

import numpy as np
import torch

import oracle
import smla_inputs as inp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_table():
    vals = {}
    for line in open(os.path.join(GOLDEN, "e2m1_values.txt")):
        if line.startswith("#") or not line.strip():
            continue
        code, v = line.split()
        vals[int(code, 16)] = float(v)
    assert sorted(vals) == list(range(16))
    return np.array([vals[c] for c in range(16)])


def test_e2m1_decode_matches_the_ocp_table():
    table = _e2m1_table()
    mine = np.array([oracle.e2m1_to_double(c) for c in range(16)])
    assert np.array_equal(mine, table)
    assert np.array_equal(np.signbit(mine), np.arange(16) >= 8)  # signed zero kept


def test_e2m1_encode_is_the_nearest_value_ties_to_even():
    table = _e2m1_table()
    mags = table[:8]
    mids = (mags[:-1] + mags[1:]) / 2  # exact ties
    rng = np.random.default_rng(3)
    x = np.concatenate([mids, -mids, rng.uniform(-6, 6, 20000), np.exp(rng.uniform(-12, 1.8, 5000))])
    x = x.astype(np.float32)
    for v in x:
        a = abs(float(v))
        d = np.abs(mags - a)
        best = np.flatnonzero(d == d.min())
        code = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])  # a tie goes to the even code
        if np.signbit(v):
            code |= 8
        assert oracle.e2m1_from_float(float(v)) == code, (float(v), code)


def test_e2m1_encode_roundtrips_and_saturates():
    table = _e2m1_table()
    for c in range(16):
        assert oracle.e2m1_from_float(table[c]) == c
    assert oracle.e2m1_from_float(6.5) == 0x7 and oracle.e2m1_from_float(1e30) == 0x7
    assert oracle.e2m1_from_float(-7.0) == 0xF


def _golden_row():
    x = np.zeros(576, np.float32)
    want_bytes = np.zeros(352, np.uint8)
    want_vals = np.zeros(576)
    for line in open(os.path.join(GOLDEN, "nvfp4_row.txt")):
        if line.startswith("#") or not line.strip():
            continue
        kind, i, v = line.split()
        if kind == "input":
            x[int(i)] = float(v)
        elif kind == "byte":
            want_bytes[int(i)] = int(v, 16)
        else:
            want_vals[int(i)] = float(v)
    return x, want_bytes, want_vals


def test_quantize_and_dequant_golden_row():
    x, want_bytes, want_vals = _golden_row()
    bits = inp.bf16_bits(x[None])
    assert np.array_equal(inp.bits_to_float(bits)[0], x)  # the inputs are bf16 values
    cache = np.full((1, 64, 352), 0xAB, np.uint8)
    oracle.nvfp4_quantize_store(bits, np.array([5], np.int64), cache)
    got = cache[0, 5]
    bad = np.flatnonzero(got != want_bytes)
    assert bad.size == 0, [(int(i), hex(got[i]), hex(want_bytes[i])) for i in bad[:8]]
    assert np.all(cache[0, :5] == 0xAB) and np.all(cache[0, 6:] == 0xAB)  # only the slot's row is written
    np.testing.assert_array_equal(oracle.nvfp4_dequant_row(got), want_vals)


def _dequant_independent(rows):
    """NVFP4 rows [n, 352] -> float64 [n, 576] from the OCP E2M1 table and
    torch's float8_e4m3fn (independent of the oracle's decoders)."""
    table = _e2m1_table()
    rows = np.asarray(rows, np.uint8)
    lo, hi = rows[:, :256] & 0xF, rows[:, :256] >> 4
    codes = np.stack([lo, hi], axis=2).reshape(len(rows), 512)
    sc = torch.from_numpy(rows[:, 256:288].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    rope = torch.from_numpy(rows[:, 288:352].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return np.concatenate([table[codes] * np.repeat(sc, 16, axis=1), rope], axis=1)


def test_dequant_row_matches_independent_decoder():
    rng = np.random.default_rng(5)
    rows = rng.integers(0, 256, size=(64, 352), dtype=np.uint8)
    rows[:, 256:] &= 0x7F  # positive scales, no NaN codes (0x7F excluded below)
    rows[:, 256:][rows[:, 256:] == 0x7F] = 0x7E
    ref = _dequant_independent(rows)
    for i in range(len(rows)):
        np.testing.assert_array_equal(oracle.nvfp4_dequant_row(rows[i]), ref[i])


def test_quantize_error_within_half_an_e2m1_step():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((64, 576), dtype=np.float32) * np.exp(rng.uniform(-6, 4, (64, 1))).astype(np.float32)
    x[3, 32:48] = 0.0  # a zero block
    bits = inp.bf16_bits(x)
    xf = inp.bits_to_float(bits).astype(np.float64)
    cache = np.zeros((1, 64, 352), np.uint8)
    oracle.nvfp4_quantize_store(bits, np.arange(64, dtype=np.int64), cache)
    deq = _dequant_independent(cache[0])
    sc = torch.from_numpy(cache[0, :, 256:288].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for t in range(64):
        for b in range(32):
            xs, ds, s = xf[t, 16 * b:16 * b + 16], deq[t, 16 * b:16 * b + 16], sc[t, b]
            if s == 0.0:
                assert np.all(ds == 0)
                continue
            y = np.abs(xs) / s
            # half the grid step at |y| (0.25 below 2, 0.5 below 4, 1 up to 6); beyond 6 the code saturates
            half = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))
            bound = s * np.maximum(half, y - 6.0) * (1 + 1e-9)
            assert np.all(np.abs(xs - ds) <= bound), (t, b)
            # the block scale is the nearest E4M3 value of amax / 6: within half a step of it (a relative
            # 2^-4 for normal E4M3 values, 2^-10 absolute in the subnormal range below 2^-6)
            a6 = np.max(np.abs(xs)) / 6.0
            assert abs(s - a6) <= max(a6 * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6)
    # RoPE: nearest E4M3 of each value
    ref_rope = torch.from_numpy(xf[:, 512:].astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(deq[:, 512:], ref_rope)


def _small_nvfp4_decode(seed=0, R=3, ctx=150, H=4):
    rng = np.random.default_rng(seed)
    ctx_lens = np.full(R, ctx)
    bt, NB = inp._paged_layout(rng, ctx_lens)
    slots = np.concatenate([inp._slot_of(bt, r, np.arange(ctx)) for r in range(R)])
    rows = inp.bf16_bits(rng.standard_normal((len(slots), 576), dtype=np.float32))
    cache = np.zeros((NB, 64, 352), np.uint8)
    oracle.nvfp4_quantize_store(rows, slots, cache)
    q = inp.bf16_bits(rng.standard_normal((R, H, 576), dtype=np.float32))
    return rng, bt, NB, cache, q


def test_nvfp4_decode_full_coverage_equals_dense_sdpa_float64():
    rng, bt, NB, cache, q = _small_nvfp4_decode(seed=21)
    R, H, ctx = q.shape[0], q.shape[1], 150
    scale = 576 ** -0.5
    idx = np.stack([rng.permutation(ctx) for _ in range(R)]).astype(np.int32)
    out, lse = oracle.sparse_mla_decode_nvfp4(q, cache, idx, bt, np.arange(R, dtype=np.int32), scale)
    flat = cache.reshape(-1, 352)
    for r in range(R):
        kv = torch.from_numpy(_dequant_independent(flat[inp._slot_of(bt, r, np.arange(ctx))]))
        qq = torch.from_numpy(inp.bits_to_float(q[r])).to(torch.float64)
        ref = torch.nn.functional.scaled_dot_product_attention(qq[None], kv[None], kv[None, :, :512], scale=scale)[0]
        ref_lse = torch.logsumexp(qq @ kv.T * scale, dim=-1)
        np.testing.assert_allclose(out[r], ref.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[r], ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_nvfp4_decode_single_index_and_invalid_rows():
    rng, bt, NB, cache, q = _small_nvfp4_decode(seed=22)
    R, H = q.shape[:2]
    idx = np.full((R, 7), -1, np.int32)
    pick = rng.integers(0, 150, size=R)
    idx[np.arange(R), rng.integers(0, 7, size=R)] = pick
    idx[0, :] = -1  # request 0: no valid index
    out, lse = oracle.sparse_mla_decode_nvfp4(q, cache, idx, bt, np.arange(R, dtype=np.int32), 0.3)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    flat = cache.reshape(-1, 352)
    for r in range(1, R):
        kv = _dequant_independent(flat[inp._slot_of(bt, r, np.array([pick[r]]))])[0]
        np.testing.assert_array_equal(out[r], np.broadcast_to(kv[:512], (H, 512)))
        np.testing.assert_allclose(lse[r], inp.bits_to_float(q[r]).astype(np.float64) @ kv * 0.3, rtol=0, atol=1e-12)
