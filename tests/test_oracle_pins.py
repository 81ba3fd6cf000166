"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test ties one oracle function to something the oracle does not
compute: the numbers the Prime Inference post prints, hand-worked
encodings, torch's own float8_e4m3fn conversion, exact rational
arithmetic, closed forms of attention, or a dense fp64 softmax(QK^T)V
computed by torch on tiny inputs.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import read_golden
from workloads import bf16_from_f32, f32_from_bf16, make_workload, make_queries, make_rows

ALL_BF16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def torch_e4m3(x_f32: np.ndarray) -> np.ndarray:
    """torch's fp32 -> float8_e4m3fn conversion (round to nearest even, non-saturating)."""
    return torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def finite_bf16():
    v = f32_from_bf16(ALL_BF16)
    return ALL_BF16[np.isfinite(v)], v[np.isfinite(v)]


# ------------------------------------------------------------- row format
def test_row_sizes_match_post():
    g = {k: int(v) for k, v in read_golden("row_format.txt")}
    nv = g["latent_dim"] * g["latent_bits_per_value"] // 8 \
        + g["latent_dim"] // g["latent_values_per_scale"] * g["scale_format_bits"] // 8 \
        + g["rope_dim"] * g["rope_format_bits"] // 8
    assert nv == g["row_bytes_after"] == 352
    assert g["latent_dim"] + g["rope_dim"] == g["row_bytes_before"] == 576
    lat = np.zeros((3, 512), np.uint16)
    rope = np.zeros((3, 64), np.uint16)
    assert oracle.quantize_rows(lat, rope, 0).shape == (3, g["row_bytes_after"])
    assert oracle.quantize_rows(lat, rope, 1).shape == (3, g["row_bytes_before"])


def test_capacity_ratio_is_consistent_with_row_shrink():
    # The post's 1.09M -> 1.63M tokens (other per-token state unchanged) is
    # below the pure row ratio 576/352; the implied other state is ~100 B/token.
    g = {k: int(v) for k, v in read_golden("row_format.txt")}
    before, after = g["tokens_per_decoder_before"], g["tokens_per_decoder_after"]
    assert after / before < g["row_bytes_before"] / g["row_bytes_after"]
    other = (after * g["row_bytes_after"] - before * g["row_bytes_before"]) / (before - after)
    assert 80 < other < 120


# ------------------------------------------------------------------- E4M3
def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_every_bf16():
    bits, v = finite_bf16()
    inside = np.abs(v) < 464  # torch does not saturate; 464 is the tie to the non-finite 480
    got = oracle.e4m3_encode(v[inside].astype(np.float64))
    assert np.array_equal(got, torch_e4m3(v[inside]))
    sat = oracle.e4m3_encode(v[~inside].astype(np.float64))
    assert np.all(sat == np.where(v[~inside] > 0, 0x7E, 0xFE))


def test_e4m3_encode_matches_torch_random_fp32():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    x = x[np.abs(x) < 464]
    assert np.array_equal(oracle.e4m3_encode(x.astype(np.float64)), torch_e4m3(x))


def test_e4m3_hand_worked_values():
    for val, code in read_golden("e4m3_rope_worked.txt"):
        assert oracle.e4m3_encode(np.array([float(val)]))[0] == int(code, 16), val


# ------------------------------------------------------------------- E2M1
def test_e2m1_decode_grid():
    grid = read_golden("e2m1_grid.txt")
    codes = np.array([int(c) for c, _ in grid], np.uint8)
    vals = np.array([float(v) for _, v in grid])
    got = oracle.e2m1_decode(codes)
    assert np.array_equal(got, vals)
    assert np.array_equal(np.signbit(got), np.signbit(vals))


def _exact_nearest_e2m1(v: Fraction) -> int:
    """Nearest grid value by exact rational distance; ties to the even code."""
    grid = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
            Fraction(4), Fraction(6)]
    a = abs(v)
    d = [abs(a - g) for g in grid]
    best = min(d)
    cands = [i for i, x in enumerate(d) if x == best]
    mag = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
    return mag | (8 if v < 0 else 0)


def test_e2m1_encode_exact_rational():
    # Quotients x/S of bf16 x and E4M3 S, checked with exact rational arithmetic.
    rng = np.random.default_rng(11)
    bits, xs = finite_bf16()
    xs = xs[(np.abs(xs) > 2.0 ** -20) & (np.abs(xs) < 1e4)]
    sc = oracle.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8))
    pick_x = rng.choice(xs, 4000)
    pick_s = rng.choice(sc, 4000)
    got = oracle.e2m1_encode(pick_x.astype(np.float64) / pick_s)
    for x, s, g in zip(pick_x, pick_s, got):
        assert g == _exact_nearest_e2m1(Fraction(float(x)) / Fraction(float(s))), (x, s)


def test_e2m1_midpoints_go_to_even_codes():
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert list(oracle.e2m1_encode(mids)) == [0, 2, 2, 4, 4, 6, 6]
    assert list(oracle.e2m1_encode(-mids)) == [8, 10, 10, 12, 12, 14, 14]
    above = np.nextafter(mids, np.inf)
    assert list(oracle.e2m1_encode(above)) == [1, 2, 3, 4, 5, 6, 7]
    below = np.nextafter(mids, -np.inf)
    assert list(oracle.e2m1_encode(below)) == [0, 1, 2, 3, 4, 5, 6]


def test_e2m1_roundtrip_and_monotone():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(oracle.e2m1_encode(oracle.e2m1_decode(codes)), codes)
    v = np.linspace(-8, 8, 100001)
    vals = oracle.e2m1_decode(oracle.e2m1_encode(v))
    assert np.all(np.diff(vals) >= 0)
    assert np.all(np.abs(vals) <= 6)


def test_every_grid_value_times_every_scale_roundtrips():
    # x = g * S (exact) must encode back to g's code under scale S.
    codes = np.arange(16, dtype=np.uint8)
    g = oracle.e2m1_decode(codes)
    S = oracle.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8))
    x = (g[None, :] * S[:, None])
    got = oracle.e2m1_encode(x / S[:, None])
    assert np.array_equal(got, np.broadcast_to(codes, got.shape))


# ----------------------------------------------------------- dequant exactness
def test_dequant_products_exact_in_fp16_and_bf16():
    # Every code x scale product is representable in fp16 and bf16, so FP16
    # MMA operands (the post's "FP16 operands") lose nothing on the KV side.
    g = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    S = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    p = (g[None, :] * S[:, None]).ravel()
    assert np.array_equal(p.astype(np.float16).astype(np.float64), p)
    p32 = p.astype(np.float32)
    assert np.array_equal(f32_from_bf16(bf16_from_f32(p32)).astype(np.float64), p)


# ------------------------------------------------------------ row encoding
def _parse_blocks():
    rows = read_golden("nvfp4_blocks_worked.txt")
    out = []
    for i in range(0, len(rows), 3):
        assert rows[i][0] == "block" and rows[i + 1][0] == "scale" and rows[i + 2][0] == "payload"
        vals = np.array([float(v) for v in rows[i][1:]], np.float32)
        assert vals.size == 16
        out.append((vals, int(rows[i + 1][1], 16), bytes(int(b, 16) for b in rows[i + 2][1:])))
    return out


@pytest.mark.parametrize("block", range(7))
def test_nvfp4_block_hand_worked(block):
    vals, scale, payload = _parse_blocks()[block]
    bits = bf16_from_f32(vals)
    assert np.array_equal(f32_from_bf16(bits), vals), "fixture values must be bf16-exact"
    lat = np.zeros((1, 512), np.uint16)
    lat[0, 16 * 5:16 * 6] = bits  # place the block at block index 5
    rows = oracle.quantize_rows(lat, np.zeros((1, 64), np.uint16))
    assert rows[0, 256 + 5] == scale
    assert bytes(rows[0, 8 * 5:8 * 6]) == payload


def test_rope_hand_worked():
    g = read_golden("e4m3_rope_worked.txt")
    vals = np.array([float(v) for v, _ in g], np.float32)
    codes = np.array([int(c, 16) for _, c in g], np.uint8)
    bits = bf16_from_f32(vals)
    exact = f32_from_bf16(bits) == vals
    assert exact.sum() >= len(vals) - 1  # -100000 is not bf16-exact; it saturates anyway
    rope = np.zeros((1, 64), np.uint16)
    rope[0, :len(vals)] = bits
    rows = oracle.quantize_rows(np.zeros((1, 512), np.uint16), rope)
    assert np.array_equal(rows[0, 288:288 + len(vals)], codes)
    assert not rows[0, 288 + len(vals):].any()


def test_block_scale_is_torch_e4m3_of_amax_over_6():
    wl = make_workload("tiny")
    lat, rope = make_rows(wl, 512)
    rows = oracle.quantize_rows(lat, rope)
    x = f32_from_bf16(lat).reshape(512, 32, 16).astype(np.float64)
    amax = np.abs(x).max(-1)
    want = torch_e4m3((amax / 6.0).astype(np.float32))  # amax/6 is exact enough: see header
    assert np.array_equal(rows[:, 256:288], want)


def test_element_codes_are_nearest_multiples_of_scale():
    wl = make_workload("agent", num_seqs=1, seq_len=4096)  # has x20 outliers
    lat, rope = make_rows(wl, 256)
    rows = oracle.quantize_rows(lat, rope)
    x = f32_from_bf16(lat).astype(np.float64).reshape(256, 512)
    S = oracle.e4m3_decode(rows[:, 256:288]).repeat(16, axis=1)
    codes = np.empty((256, 512), np.uint8)
    codes[:, 0::2] = rows[:, :256] & 15
    codes[:, 1::2] = rows[:, :256] >> 4
    deq = oracle.e2m1_decode(codes) * S
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    cand = np.sign(x)[..., None] * grid * S[..., None]
    dist = np.abs(x[..., None] - cand)
    best = dist.min(-1)
    assert np.all(np.abs(x - deq) == best)          # nearest (exact fp64 arithmetic)
    # sign bit equals the sign bit of x whenever the scale is nonzero
    assert np.array_equal((codes >> 3).astype(bool), np.signbit(x) & (S > 0))


def test_fp8_row_matches_torch():
    wl = make_workload("tiny")
    lat, rope = make_rows(wl, 64)
    for ls, rs in [(1.0, 1.0), (0.75, 2.5)]:
        rows = oracle.quantize_rows(lat, rope, 1, ls, rs)
        ql = (f32_from_bf16(lat) / np.float32(ls)).astype(np.float32)
        qr = (f32_from_bf16(rope) / np.float32(rs)).astype(np.float32)
        assert np.array_equal(rows[:, :512], torch_e4m3(ql))
        assert np.array_equal(rows[:, 512:], torch_e4m3(qr))


def test_quantization_error_bound():
    wl = make_workload("agent", num_seqs=1, seq_len=4096)
    lat, rope = make_rows(wl, 256)
    rows = oracle.quantize_rows(lat, rope)
    x = f32_from_bf16(lat).astype(np.float64).reshape(256, 512)
    d, _ = oracle.dequant_rows(rows)
    S = oracle.e4m3_decode(rows[:, 256:288]).repeat(16, axis=1)
    # half the widest grid gap (1, between 4 and 6) times S, plus the
    # saturation overshoot when amax/6 rounded down (|x| up to 6.375 S)
    assert np.all(np.abs(x - d) <= np.maximum(S * 1.0, np.abs(x) - 6 * S) + 1e-300)
    assert np.all(np.abs(x - d) <= 0.0625 * np.abs(x).reshape(256, 32, 16).max(-1).repeat(16, 1) * 6)


# ---------------------------------------------------------------- append
def test_append_places_rows_through_block_table():
    wl = make_workload("tiny", seq_len=300)  # 5 pages, last one ragged
    rb = 352
    stride = 64 * rb + 128  # padded page stride (multi-layer style)
    cache = np.zeros(wl.num_blocks * stride, np.uint8)
    seq = np.zeros(300, np.int32)
    pos = np.arange(300, dtype=np.int32)
    lat, rope = make_rows(wl, 300)
    bad = oracle.append(lat, rope, seq, pos, wl.block_table, 64, cache, wl.num_blocks, stride)
    assert bad == 0
    rows = oracle.quantize_rows(lat, rope)
    view = cache.reshape(wl.num_blocks, stride)
    for p in range(300):
        blk = wl.block_table[0, p // 64]
        assert np.array_equal(view[blk, (p % 64) * rb:(p % 64 + 1) * rb], rows[p])
    # padding bytes and the unwritten tail of the last page stay untouched
    assert not view[:, 64 * rb:].any()
    last = wl.block_table[0, 4]
    assert not view[last, (300 - 256) * rb:64 * rb].any()


def test_append_skips_and_counts_unresolvable_tokens():
    wl = make_workload("tiny", seq_len=128)
    cache = np.zeros(wl.num_blocks * 64 * 352, np.uint8)
    lat, rope = make_rows(wl, 5)
    seq = np.array([0, 1, -1, 0, 0], np.int32)
    pos = np.array([3, 3, 3, 64 * wl.max_blocks_per_seq, -2], np.int32)
    bad = oracle.append(lat, rope, seq, pos, wl.block_table, 64, cache, wl.num_blocks, 64 * 352)
    assert bad == 4
    blk = wl.block_table[0, 0]
    assert np.array_equal(cache.reshape(-1, 352)[blk * 64 + 3], oracle.quantize_rows(lat, rope)[0])
    assert cache.reshape(-1, 352).any(1).sum() == 1


# ------------------------------------------- row decode, independent of the oracle
def _grid_from_golden() -> np.ndarray:
    """E2M1 value of each of the 16 codes, from the definition in tests/golden."""
    g = np.zeros(16, np.float64)
    for code, val in read_golden("e2m1_grid.txt"):
        g[int(code)] = float(val)
    return g


def indep_dequant(rows: np.ndarray, rope_scale: float = 1.0):
    """Decode 352-byte rows without the oracle: nibble split, the golden E2M1
    grid, torch's float8_e4m3fn view of the scale and rope bytes (row layout:
    codes at 0..255, scales at 256..287, rope at 288..351)."""
    rows = np.ascontiguousarray(rows, np.uint8).reshape(-1, 352)
    grid = _grid_from_golden()
    codes = np.empty((rows.shape[0], 512), np.uint8)
    codes[:, 0::2] = rows[:, :256] & 15
    codes[:, 1::2] = rows[:, :256] >> 4

    def e4m3_view(b):
        return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).double().numpy()

    scales = e4m3_view(rows[:, 256:288])
    lat = grid[codes] * np.repeat(scales, 16, axis=1)
    rope = e4m3_view(rows[:, 288:352]) * float(np.float32(rope_scale))
    return lat, rope


@pytest.mark.parametrize("rs", [0.37, 3.0, 1.0])
def test_nvfp4_rope_dequant_is_e4m3_view_times_rope_scale(rs):
    """The rope part of an NVFP4 row is kept FP8 (the Prime Inference post,
    section "Making room for low-latency decode"), read back as E4M3 times the
    per-tensor rope scale."""
    rng = np.random.default_rng(11)
    # every finite E4M3 code (both signs) appears in the rope bytes of some row
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    n = (finite.size + 63) // 64
    rows = rng.integers(0, 256, (n, 352), dtype=np.uint8)
    rows[:, 256:288] &= 0x7E  # positive, finite scale bytes
    rope_bytes = np.resize(finite, n * 64).reshape(n, 64)
    rows[:, 288:352] = rope_bytes
    lat, rope = oracle.dequant_rows(rows, 0, 1.0, rs)
    want_lat, want_rope = indep_dequant(rows, rs)
    assert np.array_equal(rope, want_rope)
    assert np.array_equal(lat, want_lat)


def test_nvfp4_dense_attention_with_rope_scale_matches_torch():
    """Decode over NVFP4 rows written with rope_scale != 1 equals torch's dense
    fp64 softmax(QK^T)V over rows decoded without the oracle."""
    rs = 1.5
    wl = make_workload("tiny", seq_len=160, num_heads=4)
    lat_bf, rope_bf = make_rows(wl, 160)
    cache = np.zeros(wl.num_blocks * 64 * 352, np.uint8)
    oracle.append(lat_bf, rope_bf, np.zeros(160, np.int32), np.arange(160, dtype=np.int32),
                  wl.block_table, 64, cache, wl.num_blocks, 64 * 352, 0, 1.0, rs)
    ql, qr = make_queries(wl)
    idx = np.arange(160, dtype=np.int32)[None, :]
    out, lse, bad = oracle.sparse_mla_decode(ql, qr, wl.q_seq, idx, wl.block_table, wl.seq_lens,
                                             64, cache, wl.num_blocks, 64 * 352, 0, wl.sm_scale,
                                             1.0, rs)
    assert bad == 0
    rows = np.stack([cache.reshape(-1, 352)[wl.block_table[0, p // 64] * 64 + p % 64]
                     for p in range(160)])
    L, R = indep_dequant(rows, rs)
    Q = torch.from_numpy(f32_from_bf16(ql[0]).astype(np.float64))
    QR = torch.from_numpy(f32_from_bf16(qr[0]).astype(np.float64))
    s = wl.sm_scale * (Q @ torch.from_numpy(L).T + QR @ torch.from_numpy(R).T)
    want = torch.softmax(s, -1) @ torch.from_numpy(L)
    assert np.allclose(out[0], want.numpy(), rtol=1e-12, atol=1e-13)
    assert np.allclose(lse[0], torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)
    # one selected row: out is exactly that row's latent, LSE its score
    one = np.full((1, 8), -1, np.int32)
    one[0, 3] = 97
    o1, l1, _ = oracle.sparse_mla_decode(ql, qr, wl.q_seq, one, wl.block_table, wl.seq_lens, 64,
                                         cache, wl.num_blocks, 64 * 352, 0, wl.sm_scale, 1.0, rs)
    assert np.array_equal(o1[0], np.repeat(L[97][None], 4, 0))
    z = wl.sm_scale * (Q.numpy() @ L[97] + QR.numpy() @ R[97])
    assert np.allclose(l1[0], z, rtol=0, atol=1e-12)


# ------------------------------------------------------------- attention
def _setup(name="tiny", seed=None, **kw):
    wl = make_workload(name, seed=seed, **kw)
    seq, pos = np.repeat(np.arange(wl.num_seqs, dtype=np.int32), wl.seq_lens), \
        np.concatenate([np.arange(n, dtype=np.int32) for n in wl.seq_lens])
    lat, rope = make_rows(wl, seq.size)
    cache = np.zeros(wl.num_blocks * 64 * 352, np.uint8)
    oracle.append(lat, rope, seq, pos, wl.block_table, 64, cache, wl.num_blocks, 64 * 352)
    ql, qr = make_queries(wl)
    return wl, cache, ql, qr


def _decode(wl, cache, ql, qr, idx, **kw):
    return oracle.sparse_mla_decode(ql, qr, wl.q_seq, idx, wl.block_table, wl.seq_lens, 64, cache,
                                    wl.num_blocks, 64 * 352, 0, wl.sm_scale, **kw)


def test_dense_attention_matches_torch_softmax():
    wl, cache, ql, qr = _setup("tiny", seq_len=200, num_heads=4)
    idx = np.arange(200, dtype=np.int32)[None, :]
    out, lse, bad = _decode(wl, cache, ql, qr, idx)
    assert bad == 0
    # independent path: dequantize every row, then torch fp64 dense attention
    rows = np.stack([cache.reshape(-1, 352)[wl.block_table[0, p // 64] * 64 + p % 64]
                     for p in range(200)])
    lat, rope = oracle.dequant_rows(rows)
    L = torch.from_numpy(lat)
    R = torch.from_numpy(rope)
    Q = torch.from_numpy(f32_from_bf16(ql[0]).astype(np.float64))
    QR = torch.from_numpy(f32_from_bf16(qr[0]).astype(np.float64))
    s = wl.sm_scale * (Q @ L.T + QR @ R.T)
    want = torch.softmax(s, -1) @ L
    assert np.allclose(out[0], want.numpy(), rtol=1e-12, atol=1e-13)
    assert np.allclose(lse[0], torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def test_single_index_returns_that_row():
    wl, cache, ql, qr = _setup("tiny", seq_len=256, num_heads=3)
    p = 77
    idx = np.full((1, 8), -1, np.int32)
    idx[0, 5] = p
    out, lse, _ = _decode(wl, cache, ql, qr, idx)
    row = cache.reshape(-1, 352)[wl.block_table[0, p // 64] * 64 + p % 64]
    lat, rope = oracle.dequant_rows(row[None])
    assert np.array_equal(out[0], np.repeat(lat, 3, 0))
    z = wl.sm_scale * (f32_from_bf16(ql[0]).astype(np.float64) @ lat[0]
                       + f32_from_bf16(qr[0]).astype(np.float64) @ rope[0])
    assert np.allclose(lse[0], z, rtol=0, atol=1e-12)


def test_weights_sum_to_one():
    # Every selected row carries the same latent -> out equals that latent.
    wl = make_workload("tiny", seq_len=128, num_heads=4)
    lat, rope = make_rows(wl, 128)
    lat[:] = lat[0]
    cache = np.zeros(wl.num_blocks * 64 * 352, np.uint8)
    oracle.append(lat, rope, np.zeros(128, np.int32), np.arange(128, dtype=np.int32),
                  wl.block_table, 64, cache, wl.num_blocks, 64 * 352)
    ql, qr = make_queries(wl)
    idx = np.arange(0, 128, 3, dtype=np.int32)[None]
    out, _, _ = _decode(wl, cache, ql, qr, idx)
    one, _ = oracle.dequant_rows(oracle.quantize_rows(lat[:1], rope[:1]))
    assert np.allclose(out[0], np.repeat(one, 4, 0), rtol=1e-14, atol=1e-14)


def test_padding_permutation_and_duplicates():
    wl, cache, ql, qr = _setup("tiny", seq_len=500, num_heads=4)
    rng = np.random.default_rng(3)
    base = rng.choice(500, 40, replace=False).astype(np.int32)[None]
    o0, l0, _ = _decode(wl, cache, ql, qr, base)
    padded = np.concatenate([base, np.full((1, 24), -1, np.int32)], 1)
    rng.shuffle(padded[0])
    o1, l1, b1 = _decode(wl, cache, ql, qr, padded)
    assert b1 == 0
    assert np.allclose(o0, o1, rtol=1e-13, atol=1e-14) and np.allclose(l0, l1, rtol=0, atol=1e-13)
    dup = np.concatenate([base, base], 1)
    o2, l2, _ = _decode(wl, cache, ql, qr, dup)
    assert np.allclose(o0, o2, rtol=1e-13, atol=1e-14)
    assert np.allclose(l2, l0 + math.log(2.0), rtol=0, atol=1e-12)


def test_invalid_entries_are_counted_and_ignored():
    wl, cache, ql, qr = _setup("tiny", seq_len=300, num_heads=2)
    good = np.array([[5, 70, 299]], np.int32)
    o0, l0, b0 = _decode(wl, cache, ql, qr, good)
    bad_idx = np.array([[5, 300, 70, -2, 299, 4096, -1]], np.int32)
    o1, l1, b1 = _decode(wl, cache, ql, qr, bad_idx)
    assert b0 == 0 and b1 == 3
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_empty_selection_gives_zero_and_minus_inf():
    wl, cache, ql, qr = _setup("tiny", seq_len=64, num_heads=2)
    out, lse, bad = _decode(wl, cache, ql, qr, np.full((1, 16), -1, np.int32))
    assert bad == 0 and not out.any() and np.all(np.isneginf(lse))
    bad_seq = wl.q_seq.copy()
    bad_seq[0] = 7
    out, lse, bad = oracle.sparse_mla_decode(ql, qr, bad_seq, np.arange(4, dtype=np.int32)[None],
                                             wl.block_table, wl.seq_lens, 64, cache,
                                             wl.num_blocks, 64 * 352, 0, wl.sm_scale)
    assert bad == 4 and not out.any() and np.all(np.isneginf(lse))


def test_fp8_rows_attention_uses_scales():
    wl = make_workload("tiny", seq_len=64, num_heads=2)
    lat, rope = make_rows(wl, 64)
    ls, rs = 0.5, 2.0
    cache = np.zeros(wl.num_blocks * 64 * 576, np.uint8)
    oracle.append(lat, rope, np.zeros(64, np.int32), np.arange(64, dtype=np.int32),
                  wl.block_table, 64, cache, wl.num_blocks, 64 * 576, 1, ls, rs)
    ql, qr = make_queries(wl)
    idx = np.arange(64, dtype=np.int32)[None]
    out, lse, _ = oracle.sparse_mla_decode(ql, qr, wl.q_seq, idx, wl.block_table, wl.seq_lens, 64,
                                           cache, wl.num_blocks, 64 * 576, 1, wl.sm_scale, ls, rs)
    rows = np.stack([cache.reshape(-1, 576)[wl.block_table[0, 0] * 64 + p] for p in range(64)])
    L = oracle.e4m3_decode(rows[:, :512]) * ls
    R = oracle.e4m3_decode(rows[:, 512:]) * rs
    Q = f32_from_bf16(ql[0]).astype(np.float64)
    QR = f32_from_bf16(qr[0]).astype(np.float64)
    s = torch.from_numpy(wl.sm_scale * (Q @ L.T + QR @ R.T))
    want = torch.softmax(s, -1).numpy() @ L
    assert np.allclose(out[0], want, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------ staged FP8 rows
def test_stage_fp8_matches_torch_reencoding_and_placement():
    """Staged rows: torch's float8_e4m3fn of the fp32 quotient dequantised value /
    latent_scale (values kept within +-448 here, where torch does not saturate),
    rope bytes copied, row t * R + j, -1 and unresolvable slots marked -1."""
    wl = make_workload("tiny", num_seqs=2, seq_len=300, num_heads=1, topk=70, q_per_seq=2)
    from workloads import all_tokens
    seq, pos = all_tokens(wl)
    lat, rope = make_rows(wl, int(seq.size))
    stride = 64 * 352
    pool = np.zeros(wl.num_blocks * stride, np.uint8)
    assert oracle.append(lat, rope, seq, pos, wl.block_table, 64, pool, wl.num_blocks,
                         stride) == 0
    idx = wl.topk_idx.copy()
    idx[0, 3] = -1            # empty slot: not counted
    idx[1, 5] = 10 ** 6       # beyond the sequence: counted
    idx[2, 0] = -7            # negative: counted
    ls = 0.375
    staged, sidx, bad = oracle.stage_fp8(wl.q_seq, idx, wl.block_table, wl.seq_lens, 64, pool,
                                         wl.num_blocks, stride, latent_scale=ls)
    assert bad == 2
    R = 128  # 70 rounded up to whole 64-row pages
    assert staged.shape == (wl.num_q * R, 576)
    n_checked = 0
    for t in range(wl.num_q):
        b = wl.q_seq[t]
        for j in range(wl.topk):
            p = idx[t, j]
            ok = 0 <= p < wl.seq_lens[b]
            assert sidx[t, j] == (j if ok else -1)
            row_out = staged[t * R + j]
            if not ok:
                assert not row_out.any()
                continue
            page = wl.block_table[b, p // 64]
            row_in = pool[page * stride + (p % 64) * 352:][:352]
            vals, _ = oracle.dequant_rows(row_in[None], 0)
            q = (vals[0].astype(np.float32) / np.float32(ls)).astype(np.float32)
            assert np.all(np.abs(q) <= 448)
            assert np.array_equal(row_out[:512], torch_e4m3(q))
            assert np.array_equal(row_out[512:], row_in[288:])
            n_checked += 1
    assert n_checked == wl.num_q * wl.topk - 3


# ------------------------------------------------------------ state merge
def test_merge_of_disjoint_parts_equals_decode_of_their_union():
    """Attention over a union of disjoint selections is the LSE-weighted merge of
    the parts' normalised outputs (softmax over a union), to fp64 rounding; an
    empty part contributes nothing; all parts empty gives 0 and -inf."""
    wl = make_workload("tiny", num_seqs=2, seq_len=600, num_heads=4, topk=90, q_per_seq=2)
    from workloads import all_tokens
    seq, pos = all_tokens(wl)
    lat, rope = make_rows(wl, int(seq.size))
    stride = 64 * 352
    pool = np.zeros(wl.num_blocks * stride, np.uint8)
    assert oracle.append(lat, rope, seq, pos, wl.block_table, 64, pool, wl.num_blocks,
                         stride) == 0
    ql, qr = make_queries(wl)

    def dec(idx):
        o, l, _ = oracle.sparse_mla_decode(ql, qr, wl.q_seq, idx, wl.block_table, wl.seq_lens, 64,
                                           pool, wl.num_blocks, stride, 0, wl.sm_scale)
        return o, l
    full, full_lse = dec(wl.topk_idx)
    empty = np.full((wl.num_q, 5), -1, np.int32)
    parts = [wl.topk_idx[:, :17], wl.topk_idx[:, 17:60], empty, wl.topk_idx[:, 60:]]
    outs, lses = zip(*[dec(np.ascontiguousarray(p)) for p in parts])
    out, lse = oracle.merge_states(np.stack(outs), np.stack(lses))
    assert np.max(np.abs(out - full)) < 1e-12 * max(1.0, np.max(np.abs(full)))
    assert np.max(np.abs(lse - full_lse)) < 1e-12 * max(1.0, np.max(np.abs(full_lse)))
    o0, l0 = dec(empty)
    out, lse = oracle.merge_states(np.stack([o0, o0]), np.stack([l0, l0]))
    assert not out.any() and np.all(np.isneginf(lse))
