"""Pins for the float64 CPU oracle (CPU only).

The oracle is checked against things other than itself: the OCP E4M3 code
table via torch's float8_e4m3fn dtype, hand-worked fixtures in tests/golden/,
brute-force translation by block-table expansion, dense attention through
torch's scaled_dot_product_attention in float64, and invariants of softmax
attention (single index, permutation / -1 insertion, identical rows, LSE
merge of a partition of the indices).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import smla_inputs as inp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- e4m3 format

def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(mine[~nan], ref[~nan])
    # signed zero kept
    assert np.signbit(mine[0x80]) and not np.signbit(mine[0x00])


def test_e4m3_encode_roundtrips_every_finite_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_from_float(oracle.e4m3_to_double(c)) == c


def test_e4m3_encode_matches_torch_rne_on_grid_and_ties():
    vals = [oracle.e4m3_to_double(c) for c in range(0x7F)]  # non-negative finite, ascending
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]  # exact ties (representable in f32)
    rng = np.random.default_rng(7)
    rand = np.concatenate([rng.uniform(-448, 448, 20000),
                           np.exp(rng.uniform(np.log(1e-5), np.log(448), 20000)) * rng.choice([-1, 1], 20000)])
    x = np.concatenate([np.array(mids), -np.array(mids), rand]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.e4m3_from_float(float(v)) for v in x], dtype=np.uint8)
    bad = np.nonzero(mine != ref)[0]
    assert bad.size == 0, [(float(x[i]), hex(mine[i]), hex(ref[i])) for i in bad[:5]]


def test_e4m3_encode_saturates_to_448():
    assert oracle.e4m3_from_float(448.0) == 0x7E
    assert oracle.e4m3_from_float(460.0) == 0x7E
    assert oracle.e4m3_from_float(1e30) == 0x7E
    assert oracle.e4m3_from_float(-1e30) == 0xFE
    assert oracle.e4m3_from_float(float("inf")) == 0x7E
    assert oracle.e4m3_from_float(2.0 ** -10) == 0x00  # half of the smallest subnormal: tie -> even (0)
    assert oracle.e4m3_from_float(3 * 2.0 ** -10) == 0x02  # 1.5 * 2^-9: tie -> even (2)


# ---------------------------------------------------------------- row format

def _golden_row():
    row = np.zeros(656, np.uint8)
    expect_nope = np.zeros(512)
    expect_rope = np.zeros(64)
    with open(os.path.join(GOLDEN, "fp8_row_dequant.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            if line[0] == "scales":
                sc = np.array([float(v) for v in line[1:]], np.float32)
                row[512:528] = np.frombuffer(sc.astype("<f4").tobytes(), np.uint8)
            elif line[0] == "nope":
                c, code, val = int(line[1]), int(line[2], 16), float(line[3])
                row[c] = code
                expect_nope[c] = val
            elif line[0] == "rope":
                r, bits, val = int(line[1]), int(line[2], 16), float(line[3])
                row[528 + 2 * r:530 + 2 * r] = np.frombuffer(np.array([bits], "<u2").tobytes(), np.uint8)
                expect_rope[r] = val
    return row, np.concatenate([expect_nope, expect_rope])


def test_dequant_row_golden_layout():
    row, expect = _golden_row()
    got = oracle.dequant_row(row)
    assert np.array_equal(got, expect)


# ---------------------------------------------------------------- translate

def test_translate_golden():
    bt_rows = {}
    cases = []
    nb = None
    with open(os.path.join(GOLDEN, "translate_small.txt")) as f:
        for line in f:
            tok = line.split("#")[0].split()
            if not tok:
                continue
            if tok[0] == "block_table":
                bt_rows[int(tok[1])] = [int(v) for v in tok[2:]]
            elif tok[0] == "num_blocks":
                nb = int(tok[1])
            elif tok[0] == "case":
                cases.append((int(tok[1]), int(tok[2]), int(tok[3])))
    bt = np.array([bt_rows[r] for r in sorted(bt_rows)], np.int32)
    idx = np.array([[c[1]] for c in cases], np.int32)
    req = np.array([c[0] for c in cases], np.int32)
    got = oracle.translate(idx, bt, req, nb)[:, 0]
    assert got.tolist() == [c[2] for c in cases]


def _translate_by_expansion(indices, bt, req, nb):
    """Brute force: list every logical position of each request with its
    physical slot, then look indices up in that list."""
    R, MB = bt.shape
    table = []
    for r in range(R):
        pos_to_slot = {}
        for b in range(MB):
            p = int(bt[r, b])
            for o in range(64):
                pos_to_slot[b * 64 + o] = p * 64 + o if 0 <= p < nb else -1
        table.append(pos_to_slot)
    out = np.full(indices.shape, -1, np.int32)
    for t in range(indices.shape[0]):
        r = int(req[t])
        for k in range(indices.shape[1]):
            i = int(indices[t, k])
            if 0 <= r < R and i in table[r]:
                out[t, k] = table[r][i]
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_translate_matches_block_table_expansion(seed):
    rng = np.random.default_rng(seed)
    R, MB, NB = 5, 7, 23
    bt = rng.integers(-2, NB + 3, size=(R, MB)).astype(np.int32)  # includes invalid physical ids
    T, K = 9, 40
    req = rng.integers(-1, R + 1, size=T).astype(np.int32)        # includes invalid request ids
    idx = rng.integers(-3, MB * 64 + 100, size=(T, K)).astype(np.int32)
    assert np.array_equal(oracle.translate(idx, bt, req, NB), _translate_by_expansion(idx, bt, req, NB))


# ---------------------------------------------------------------- quantizer

def _quant_case(seed, n=37, outliers=True, zero_group=True, tiny_group=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 576)).astype(np.float32)
    if outliers:
        x[:, rng.choice(576, 6, replace=False)] *= 8
    if zero_group:
        x[3, 128:256] = 0.0
    if tiny_group:
        x[5, 256:384] *= 1e-38  # denormal-range group: scale underflows
    return inp.bf16_bits(x)


def test_quantize_store_against_ieee_float32_and_torch_cast():
    kv = _quant_case(0)
    T = kv.shape[0]
    NB = 3
    rng = np.random.default_rng(1)
    slots = rng.permutation(NB * 64)[:T].astype(np.int64)
    slots[7] = -1  # skipped token
    cache = np.full((NB, 64, 656), 0xAB, np.uint8)
    oracle.quantize_store(kv, slots, cache)
    flat = cache.reshape(-1, 656)
    x = inp.bits_to_float(kv)
    for t in range(T):
        if slots[t] < 0:
            continue
        row = flat[slots[t]]
        for g in range(4):
            xg = x[t, 128 * g:128 * (g + 1)]
            amax = np.float32(np.max(np.abs(xg)))
            scale = np.float32(amax / np.float32(448.0))  # IEEE float32 division
            got_scale = np.frombuffer(row[512 + 4 * g:516 + 4 * g].tobytes(), "<f4")[0]
            assert got_scale.tobytes() == scale.tobytes()
            if scale == 0:
                assert np.all(row[128 * g:128 * (g + 1)] == 0)
            else:
                y = (xg / scale).astype(np.float32)
                codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                assert np.array_equal(row[128 * g:128 * (g + 1)], codes)
        assert row[528:656].tobytes() == kv[t, 512:576].astype("<u2").tobytes()
    # untouched rows keep their bytes
    used = set(int(s) for s in slots if s >= 0)
    for s in range(NB * 64):
        if s not in used:
            assert np.all(flat[s] == 0xAB)


def test_quantize_dequantize_error_within_half_ulp():
    kv = _quant_case(3, n=64)
    cache = np.zeros((1, 64, 656), np.uint8)
    oracle.quantize_store(kv, np.arange(64, dtype=np.int64), cache)
    x = inp.bits_to_float(kv).astype(np.float64)
    for t in range(64):
        deq = oracle.dequant_row(cache[0, t])
        for g in range(4):
            xs = x[t, 128 * g:128 * (g + 1)]
            scale = float(np.frombuffer(cache[0, t, 512 + 4 * g:516 + 4 * g].tobytes(), "<f4")[0])
            err = np.abs(xs - deq[128 * g:128 * (g + 1)])
            if scale == 0.0:
                assert np.all(deq[128 * g:128 * (g + 1)] == 0)
                assert np.all(np.abs(xs) < 1e-30)
                continue
            y = np.abs(xs) / scale
            # half an e4m3 ulp at |y| (normals: 2^(floor(log2 y) - 3); subnormals: 2^-9), in units of scale
            e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
            half_ulp = 0.5 * 2.0 ** (e - 3)
            assert np.all(err <= scale * half_ulp * (1 + 1e-6) + 1e-300), (t, g, err.max())
        assert np.array_equal(deq[512:], x[t, 512:])


# ---------------------------------------------------------------- attention

def _dequant_torch(cache, slots):
    """Dequantize rows with torch's float8_e4m3fn and float32 scale bytes
    (independent of the oracle's decoder)."""
    rows = torch.from_numpy(cache.reshape(-1, 656)[slots].copy())
    codes = rows[:, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    scales = rows[:, 512:528].contiguous().view(torch.float32).to(torch.float64)
    nope = codes * scales.repeat_interleave(128, dim=1)
    rope = rows[:, 528:656].contiguous().view(torch.bfloat16).to(torch.float64)
    return torch.cat([nope, rope], dim=1)


def _small_decode(seed=0, R=3, ctx=150, K=None, H=4):
    rng = np.random.default_rng(seed)
    ctx_lens = np.full(R, ctx)
    bt, NB = inp._paged_layout(rng, ctx_lens)
    slots = np.concatenate([inp._slot_of(bt, r, np.arange(ctx)) for r in range(R)])
    rows = inp.bf16_bits(rng.standard_normal((len(slots), 576), dtype=np.float32))
    cache = np.zeros((NB, 64, 656), np.uint8)
    oracle.quantize_store(rows, slots, cache)
    q = inp.bf16_bits(rng.standard_normal((R, H, 576), dtype=np.float32))
    return rng, bt, NB, cache, q


def test_full_coverage_equals_dense_sdpa_float64():
    rng, bt, NB, cache, q = _small_decode(seed=11)
    R, H, ctx = q.shape[0], q.shape[1], 150
    scale = 576 ** -0.5
    idx = np.stack([rng.permutation(ctx) for _ in range(R)]).astype(np.int32)
    req = np.arange(R, dtype=np.int32)
    out, lse = oracle.sparse_mla_decode(q, cache, idx, bt, req, scale)
    for r in range(R):
        slots = inp._slot_of(bt, r, np.arange(ctx))
        kv = _dequant_torch(cache, slots)                              # [ctx, 576]
        qq = torch.from_numpy(inp.bits_to_float(q[r])).to(torch.float64)  # [H, 576]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq[None], kv[None], kv[None, :, :512], scale=scale)[0]
        ref_lse = torch.logsumexp(qq @ kv.T * scale, dim=-1)
        np.testing.assert_allclose(out[r], ref.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[r], ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_single_index_returns_that_rows_v_and_logit():
    rng, bt, NB, cache, q = _small_decode(seed=12)
    R, H = q.shape[:2]
    K = 9
    idx = np.full((R, K), -1, np.int32)
    pick = rng.integers(0, 150, size=R)
    idx[np.arange(R), rng.integers(0, K, size=R)] = pick
    out, lse = oracle.sparse_mla_decode(q, cache, idx, bt, np.arange(R, dtype=np.int32), 0.3)
    for r in range(R):
        kv = _dequant_torch(cache, inp._slot_of(bt, r, np.array([pick[r]])))[0].numpy()
        np.testing.assert_array_equal(out[r], np.broadcast_to(kv[:512], (H, 512)))
        s = inp.bits_to_float(q[r]).astype(np.float64) @ kv * 0.3
        np.testing.assert_allclose(lse[r], s, rtol=0, atol=1e-12)


def test_permutation_and_invalid_insertion_invariance():
    rng, bt, NB, cache, q = _small_decode(seed=13)
    R = q.shape[0]
    K = 40
    idx = np.stack([rng.choice(150, K, replace=False) for _ in range(R)]).astype(np.int32)
    req = np.arange(R, dtype=np.int32)
    out0, lse0 = oracle.sparse_mla_decode(q, cache, idx, bt, req, 0.05)
    perm = np.stack([rng.permutation(K) for _ in range(R)])
    idx2 = np.take_along_axis(idx, perm, 1)
    pad = np.full((R, 17), -1, np.int32)
    idx3 = np.concatenate([pad[:, :8], idx2, pad[:, 8:], np.full((R, 3), 10 ** 6, np.int32)], 1)
    out1, lse1 = oracle.sparse_mla_decode(q, cache, idx3, bt, req, 0.05)
    np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse1, lse0, rtol=1e-13, atol=1e-13)


def test_identical_rows_give_uniform_weights():
    rng = np.random.default_rng(14)
    NB, H, n = 2, 3, 7
    row = inp.bf16_bits(rng.standard_normal((1, 576), dtype=np.float32))
    cache = np.zeros((NB, 64, 656), np.uint8)
    oracle.quantize_store(np.repeat(row, n, 0), np.arange(3, 3 + n, dtype=np.int64), cache)
    bt = np.array([[0, 1]], np.int32)
    q = inp.bf16_bits(rng.standard_normal((1, H, 576), dtype=np.float32))
    idx = np.arange(3, 3 + n, dtype=np.int32)[None]
    out, lse = oracle.sparse_mla_decode(q, cache, idx, bt, np.zeros(1, np.int32), 0.1)
    v = _dequant_torch(cache, np.array([3]))[0].numpy()
    np.testing.assert_allclose(out[0], np.broadcast_to(v[:512], (H, 512)), rtol=1e-14, atol=1e-15)
    s = inp.bits_to_float(q[0]).astype(np.float64) @ v * 0.1
    np.testing.assert_allclose(lse[0], s + np.log(n), rtol=0, atol=1e-12)


def test_lse_merge_of_a_partition_equals_whole():
    rng, bt, NB, cache, q = _small_decode(seed=15, H=2)
    R = q.shape[0]
    K = 120
    idx = np.stack([rng.choice(150, K, replace=False) for _ in range(R)]).astype(np.int32)
    req = np.arange(R, dtype=np.int32)
    out, lse = oracle.sparse_mla_decode(q, cache, idx, bt, req, 0.07)
    parts = [(0, 13), (13, 70), (70, 120)]
    outs, lses = [], []
    for a, b in parts:
        sub = np.full_like(idx, -1)
        sub[:, a:b] = idx[:, a:b]
        o, l_ = oracle.sparse_mla_decode(q, cache, sub, bt, req, 0.07)
        outs.append(o)
        lses.append(l_)
    L = np.stack(lses)          # [parts, R, H]
    M = L.max(0)
    w = np.exp(L - M)
    merged = (w[..., None] * np.stack(outs)).sum(0) / w.sum(0)[..., None]
    np.testing.assert_allclose(merged, out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(M + np.log(w.sum(0)), lse, rtol=1e-13, atol=1e-13)


def test_empty_token_gives_zero_and_minus_inf():
    rng, bt, NB, cache, q = _small_decode(seed=16)
    idx = np.full((q.shape[0], 5), -1, np.int32)
    out, lse = oracle.sparse_mla_decode(q, cache, idx, bt, np.arange(q.shape[0], dtype=np.int32), 0.1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_token_subset_matches_full_run():
    rng, bt, NB, cache, q = _small_decode(seed=17)
    idx = np.stack([rng.choice(150, 30, replace=False) for _ in range(3)]).astype(np.int32)
    req = np.arange(3, dtype=np.int32)
    out, lse = oracle.sparse_mla_decode(q, cache, idx, bt, req, 0.1)
    o2, l2 = oracle.sparse_mla_decode(q, cache, idx, bt, req, 0.1, tokens=np.array([2, 0], np.int32))
    np.testing.assert_array_equal(o2, out[[2, 0]])
    np.testing.assert_array_equal(l2, lse[[2, 0]])


def test_prefill_full_coverage_equals_dense_sdpa_float64():
    rng = np.random.default_rng(21)
    N, T, H = 90, 4, 3
    kv = inp.bf16_bits(rng.standard_normal((N, 576), dtype=np.float32))
    q = inp.bf16_bits(rng.standard_normal((T, H, 576), dtype=np.float32))
    idx = np.stack([rng.permutation(N) for _ in range(T)]).astype(np.int32)
    idx = np.concatenate([idx, np.full((T, 6), -1, np.int32), np.full((T, 2), N, np.int32)], 1)
    out, lse = oracle.sparse_mla_prefill(q, kv, idx, 0.04)
    kvt = torch.from_numpy(inp.bits_to_float(kv)).to(torch.float64)
    for t in range(T):
        qq = torch.from_numpy(inp.bits_to_float(q[t])).to(torch.float64)
        ref = torch.nn.functional.scaled_dot_product_attention(qq[None], kvt[None], kvt[None, :, :512], scale=0.04)[0]
        np.testing.assert_allclose(out[t], ref.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[t], torch.logsumexp(qq @ kvt.T * 0.04, -1).numpy(), rtol=1e-12, atol=1e-12)


def test_generators_are_deterministic_and_well_formed():
    a = inp.tiny_decode(0)
    b = inp.tiny_decode(0)
    assert np.array_equal(a.indices, b.indices) and np.array_equal(a.q, b.q)
    assert a.num_blocks == 16 and a.block_table.shape == (4, 4)
    assert sorted(a.block_table.reshape(-1).tolist()) == list(range(16))
    for t in range(4):
        assert len(set(a.indices[t].tolist())) == 64 and a.indices[t].min() >= 0 and a.indices[t].max() < 256
    m = inp.mixed_batch(4, n_decode=3, n_prefill=1, prefill_tokens=40, ctx_lo=100, ctx_hi=300, K=32)
    assert m.T == 3 * 2 + 40
    assert np.all(np.diff(m.req_id_per_token) >= 0)
    for t in range(m.T):
        v = m.indices[t][m.indices[t] >= 0]
        assert len(set(v.tolist())) == len(v) and v.max() <= m.positions[t]
    # bf16 conversion used by the generators is torch's round-to-nearest-even
    x = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    assert np.array_equal(inp.bf16_bits(x), torch.from_numpy(x).to(torch.bfloat16).view(torch.uint16).numpy())


# ---------------------------------------------------------------- separate-mode FP8 prefill

def _bf16_value(bits):
    return inp.bits_to_float(np.asarray(bits, np.uint16)).astype(np.float64)


def _random_rows(rng, n, pow2_scales=False):
    """n 656-byte rows: random codes (no NaN), random or power-of-two scales, random bf16 RoPE."""
    rows = np.zeros((n, 656), np.uint8)
    codes = rng.integers(0, 256, size=(n, 512)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x00
    rows[:, :512] = codes
    if pow2_scales:
        sc = np.ldexp(1.0, rng.integers(-20, 10, size=(n, 4))).astype(np.float32)
    else:
        sc = (np.exp(rng.uniform(np.log(1e-6), np.log(1e4), size=(n, 4)))).astype(np.float32)
    rows[:, 512:528] = sc.astype("<f4").view(np.uint8)
    rows[:, 528:656] = inp.bf16_bits(rng.standard_normal((n, 64)).astype(np.float32)).view(np.uint8)
    return rows


def test_upconvert_row_exact_for_power_of_two_scales():
    # e4m3 values have 4 significant bits, so code * 2^k is a bf16 value: the
    # up-converted row equals the float64 dequantization exactly
    rows = _random_rows(np.random.default_rng(11), 64, pow2_scales=True)
    for row in rows:
        assert np.array_equal(_bf16_value(oracle.upconvert_row(row)), oracle.dequant_row(row))


def test_upconvert_row_matches_torch_float32_product_rounded_to_bf16():
    rows = _random_rows(np.random.default_rng(12), 256)
    codes = torch.from_numpy(rows[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float32)
    scales = torch.from_numpy(rows[:, 512:528].copy().view(np.float32))
    ref = (codes.view(-1, 4, 128) * scales[:, :, None]).view(-1, 512).to(torch.bfloat16)
    ref_bits = ref.view(torch.int16).numpy().view(np.uint16)
    got = np.stack([oracle.upconvert_row(r) for r in rows])
    assert np.array_equal(got[:, :512], ref_bits)
    assert np.array_equal(got[:, 512:], rows[:, 528:656].copy().view(np.uint16))  # RoPE as stored
    # and within half a bf16 unit of the exact dequantization
    deq = np.stack([oracle.dequant_row(r) for r in rows])[:, :512]
    err = np.abs(_bf16_value(got[:, :512]) - deq)
    assert np.all(err <= np.abs(deq) * 2.0 ** -8 * (1 + 2.0 ** -15) + 1e-45)


def test_gather_upconvert_by_block_table_expansion():
    rng = np.random.default_rng(13)
    NB, R, MB = 12, 3, 4
    cache = _random_rows(rng, NB * 64).reshape(NB, 64, 656)
    perm = rng.permutation(NB).astype(np.int32)
    bt = perm[:R * MB].reshape(R, MB).copy()
    bt[2, 3] = NB + 5  # an invalid physical block: its positions give zero rows
    seq_lens = np.array([70, 0, 250], np.int32)
    starts = np.array([3, 73, 80], np.int32)
    N = 340
    ws = oracle.gather_upconvert(cache, bt, seq_lens, starts, N)
    expect = np.zeros((N, 576), np.uint16)
    for r in range(R):
        for pos in range(seq_lens[r]):
            p = int(bt[r, pos // 64])
            if 0 <= p < NB:
                expect[starts[r] + pos] = oracle.upconvert_row(cache[p, pos % 64])
    assert np.array_equal(ws, expect)


def test_translate_workspace_golden():
    bt_rows, cases, nb, starts = {}, [], None, None
    with open(os.path.join(GOLDEN, "translate_workspace_small.txt")) as f:
        for line in f:
            tok = line.split("#")[0].split()
            if not tok:
                continue
            if tok[0] == "block_table":
                bt_rows[int(tok[1])] = [int(v) for v in tok[2:]]
            elif tok[0] == "num_blocks":
                nb = int(tok[1])
            elif tok[0] == "starts":
                starts = np.array([int(v) for v in tok[1:]], np.int32)
            elif tok[0] == "case":
                cases.append(tuple(int(v) for v in tok[1:5]))
    bt = np.array([bt_rows[r] for r in sorted(bt_rows)], np.int32)
    req = np.array([c[0] for c in cases], np.int32)
    pr = np.array([c[1] for c in cases], np.int32)
    idx = np.array([[c[2]] for c in cases], np.int32)
    got = oracle.translate_workspace(idx, bt, req, pr, starts, nb)[:, 0]
    assert got.tolist() == [c[3] for c in cases]


def test_translate_workspace_decode_tokens_as_translate_prefill_tokens_offset():
    rng = np.random.default_rng(14)
    R, MB, NB, T, K = 5, 6, 40, 30, 50
    bt = rng.integers(-2, NB + 3, size=(R, MB)).astype(np.int32)
    req = rng.integers(0, R, size=T).astype(np.int32)
    pr = np.where(rng.random(T) < 0.5, rng.integers(0, 3, size=T), -1).astype(np.int32)
    starts = np.array([0, 200, 450], np.int32)
    idx = rng.integers(-3, MB * 64 + 40, size=(T, K)).astype(np.int32)
    got = oracle.translate_workspace(idx, bt, req, pr, starts, NB)
    dec = pr < 0
    assert np.array_equal(got[dec], oracle.translate(idx[dec], bt, req[dec], NB))
    expect = np.where((idx >= 0) & (idx // 64 < MB), starts[np.maximum(pr, 0)][:, None] + idx, -1)
    assert np.array_equal(got[~dec], expect[~dec])


def test_prefill_fp8_equals_decode_when_upconvert_is_exact():
    # With power-of-two scales the up-converted rows are the dequantized rows,
    # so the separate-mode prefill (workspace + bf16 prefill) must give the
    # decode path's result for the same tokens and logical indices.
    rng = np.random.default_rng(15)
    R, ctx, H, K = 3, 300, 16, 96
    nblk = (ctx + 63) // 64
    NB = R * nblk
    cache = _random_rows(rng, NB * 64, pow2_scales=True).reshape(NB, 64, 656)
    cache[..., :512] = np.where((cache[..., :512] & 0x78) >= 0x58, 0x30, cache[..., :512])  # keep logits moderate
    bt = rng.permutation(NB).astype(np.int32).reshape(R, nblk)
    seq_lens = np.full(R, ctx, np.int32)
    starts = np.array([0, ctx, 2 * ctx], np.int32)
    T = 7
    req = rng.integers(0, R, size=T).astype(np.int32)
    idx = np.stack([rng.choice(ctx, size=K, replace=False) for _ in range(T)]).astype(np.int32)
    idx[0, :10] = -1
    q = inp.bf16_bits(rng.standard_normal((T, H, 576)).astype(np.float32) * 0.05)
    sm = 576 ** -0.5
    o1, l1 = oracle.sparse_mla_prefill_fp8(q, cache, idx, bt, req, seq_lens, starts, R * ctx, sm)
    o2, l2 = oracle.sparse_mla_decode(q, cache, idx, bt, req, sm)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- MLA weight absorption

def _bf16_rand(rng, shape, scale=1.0):
    return inp.bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def test_absorb_q_brute_force_small():
    rng = np.random.default_rng(21)
    T, H, P = 3, 2, 64
    q = _bf16_rand(rng, (T, H, P + 64))
    w = _bf16_rand(rng, (H, P, 512), 0.1)
    got = oracle.absorb_q(q, w)
    qf, wf = _bf16_value(q).reshape(T, H, P + 64), _bf16_value(w).reshape(H, P, 512)
    for t in range(T):
        for h in range(H):
            for l in (0, 17, 300, 511):
                acc = 0.0
                for p in range(P):
                    acc += float(qf[t, h, p]) * float(wf[h, p, l])
                assert abs(got[t, h, l] - acc) <= 1e-12 * (1 + abs(acc))
            assert np.array_equal(got[t, h, 512:], qf[t, h, P:])  # q_pe after the absorbed part


def test_absorb_q_identity_weights_and_head_independence():
    rng = np.random.default_rng(22)
    T, H, P = 5, 3, 128
    q = _bf16_rand(rng, (T, H, P + 64))
    w = np.zeros((H, P, 512), np.float32)
    for h in range(H):
        w[h, :, 128 * h:128 * h + P] = np.eye(P)  # head h copies q_nope into columns 128 h ..
    got = oracle.absorb_q(q, inp.bf16_bits(w))
    qf = _bf16_value(q).reshape(T, H, P + 64)
    for h in range(H):
        expect = np.zeros((T, 512))
        expect[:, 128 * h:128 * h + P] = qf[:, h, :P]
        assert np.array_equal(got[:, h, :512], expect)
    # permuting the heads of q and W permutes the result's heads
    wr = _bf16_rand(rng, (H, P, 512), 0.1)
    perm = np.array([2, 0, 1])
    assert np.allclose(oracle.absorb_q(q[:, perm], wr[perm]), oracle.absorb_q(q, wr)[:, perm], rtol=0, atol=0)


def test_v_up_proj_one_hot_and_brute_force():
    rng = np.random.default_rng(23)
    T, H, V = 4, 2, 128
    a = _bf16_rand(rng, (T, H, 512))
    w = np.zeros((H, 512, V), np.float32)
    w[0, 7, 3] = 1.0
    w[1, 511, 127] = 2.0  # a power of two: exact
    got = oracle.v_up_proj(a, inp.bf16_bits(w))
    af = _bf16_value(a).reshape(T, H, 512)
    expect = np.zeros((T, H, V))
    expect[:, 0, 3] = af[:, 0, 7]
    expect[:, 1, 127] = 2.0 * af[:, 1, 511]
    assert np.array_equal(got, expect)
    wr = _bf16_rand(rng, (H, 512, V), 0.05)
    got = oracle.v_up_proj(a, wr)
    wf = _bf16_value(wr).reshape(H, 512, V)
    t, h, v = 2, 1, 77
    acc = sum(float(af[t, h, k]) * float(wf[h, k, v]) for k in range(512))
    assert abs(got[t, h, v] - acc) <= 1e-12 * (1 + abs(acc))
