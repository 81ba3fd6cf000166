"""GPU: quantize-on-append is bit-exact against the oracle (every byte of the pool)."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_cases import build_case, dev_tensor
from workloads import (bf16_from_f32, f32_from_bf16, make_append_batch, make_rows,
                       make_workload)

pytestmark = pytest.mark.gpu


def _gpu_append(wl, lat, rope, seq, pos, row_format=0, stride=None, latent_scale=1.0,
                rope_scale=1.0, pool=None, invalid=None):
    import nvfp4_compressed_mla_gb300 as nm
    rb = 352 if row_format == 0 else 576
    stride = stride or wl.page_size * rb
    if pool is None:
        pool = torch.zeros(wl.num_blocks * stride, dtype=torch.uint8, device="cuda:0")
    nm.nvfp4_mla_append(dev_tensor(lat, torch.bfloat16), dev_tensor(rope, torch.bfloat16),
                        dev_tensor(seq), dev_tensor(pos), dev_tensor(wl.block_table),
                        wl.page_size, pool, wl.num_blocks, stride, row_format, latent_scale,
                        rope_scale, invalid)
    torch.cuda.synchronize()
    return pool


def _direct_rows(lat, rope, row_format=0, latent_scale=1.0, rope_scale=1.0):
    """Encode n tokens into a single contiguous page list (row r at slot r)."""
    n = lat.shape[0]
    pages = (n + 63) // 64
    wl = make_workload("tiny", seq_len=pages * 64)
    wl.block_table[:] = np.arange(wl.block_table.shape[1], dtype=np.int32)
    seq = np.zeros(n, np.int32)
    pos = np.arange(n, dtype=np.int32)
    pool = _gpu_append(wl, lat, rope, seq, pos, row_format, latent_scale=latent_scale,
                       rope_scale=rope_scale)
    rb = 352 if row_format == 0 else 576
    return pool.cpu().numpy().reshape(-1, rb)[:n]


def _all_finite_bf16(seed):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = f32_from_bf16(bits)
    bits = bits[np.isfinite(v)]
    rng = np.random.default_rng(seed)
    return bits, rng


@pytest.mark.parametrize("order", ["shuffled", "sorted"])
def test_every_bf16_latent_value(order):
    bits, rng = _all_finite_bf16(1)
    if order == "shuffled":
        bits = rng.permutation(bits)
    n = (bits.size + 511) // 512
    lat = np.zeros(n * 512, np.uint16)
    lat[:bits.size] = bits
    lat = lat.reshape(n, 512)
    rope = rng.permutation(np.resize(bits, n * 64)).reshape(n, 64).astype(np.uint16)
    got = _direct_rows(lat, rope)
    want = oracle.quantize_rows(lat, rope)
    assert np.array_equal(got, want)


def test_every_scale_code_and_scale_midpoint():
    # blocks whose amax is 6*v (every E4M3 v) or 6 * a midpoint between neighbours
    v = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (v[:-1] + v[1:]) / 2
    amax = np.concatenate([6 * v, 6 * mids]).astype(np.float32)
    assert np.array_equal(f32_from_bf16(bf16_from_f32(amax)), amax)
    rng = np.random.default_rng(2)
    nblk = amax.size
    x = rng.uniform(-1, 1, (nblk, 16)).astype(np.float32) * amax[:, None]
    x[:, 3] = amax
    x[:, 7] = np.where(rng.random(nblk) < 0.5, -amax, x[:, 7])  # sometimes -amax too
    lat_bits = bf16_from_f32(x).reshape(-1)
    n = (lat_bits.size + 511) // 512
    lat = np.zeros(n * 512, np.uint16)
    lat[:lat_bits.size] = lat_bits
    lat = lat.reshape(n, 512)
    rope = np.zeros((n, 64), np.uint16)
    assert np.array_equal(_direct_rows(lat, rope), oracle.quantize_rows(lat, rope))


@pytest.mark.parametrize("rope_scale", [1.0, 0.37, 3.0, 1e-3])
def test_every_bf16_rope_value(rope_scale):
    bits, rng = _all_finite_bf16(3)
    n = (bits.size + 63) // 64
    rope = np.zeros(n * 64, np.uint16)
    rope[:bits.size] = rng.permutation(bits)
    rope = rope.reshape(n, 64)
    lat = np.zeros((n, 512), np.uint16)
    got = _direct_rows(lat, rope, rope_scale=rope_scale)
    want = oracle.quantize_rows(lat, rope, 0, 1.0, rope_scale)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("latent_scale,rope_scale", [(1.0, 1.0), (0.5, 2.0), (2.7, 0.3)])
def test_fp8_rows_every_bf16_value(latent_scale, rope_scale):
    bits, rng = _all_finite_bf16(4)
    n = (bits.size + 511) // 512
    lat = np.zeros(n * 512, np.uint16)
    lat[:bits.size] = rng.permutation(bits)
    lat = lat.reshape(n, 512)
    rope = rng.permutation(np.resize(bits, n * 64)).reshape(n, 64).astype(np.uint16)
    got = _direct_rows(lat, rope, 1, latent_scale, rope_scale)
    want = oracle.quantize_rows(lat, rope, 1, latent_scale, rope_scale)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("row_format", [0, 1])
def test_paged_append_whole_pool(row_format):
    wl = make_workload("agent", num_seqs=3, seq_len=1000)  # ragged last page, outliers
    case = build_case(wl, "all", row_format, stride_pad=48, to_device=False)
    pool = _gpu_append(wl, case.lat, case.rope, case.seq, case.pos, row_format, case.stride)
    assert np.array_equal(pool.cpu().numpy(), case.host_pool)


def test_append_counts_and_skips_unresolvable_tokens():
    wl = make_workload("tiny", seq_len=256)
    lat, rope = make_rows(wl, 6)
    seq = np.array([0, 0, 5, -1, 0, 0], np.int32)
    pos = np.array([1, 64 * wl.max_blocks_per_seq, 1, 1, -3, 200], np.int32)
    inv = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    pool = _gpu_append(wl, lat, rope, seq, pos, invalid=inv)
    host = np.zeros(wl.num_blocks * 64 * 352, np.uint8)
    bad = oracle.append(lat, rope, seq, pos, wl.block_table, 64, host, wl.num_blocks, 64 * 352)
    assert bad == 4 and int(inv.item()) == 4
    assert np.array_equal(pool.cpu().numpy(), host)


def test_append_dense_chunk_full_size():
    # 8 sequences x 4096 appended tokens into pools that already hold a 12288-token prefix
    wl = make_workload("append_dense")
    seq, pos, lat, rope = make_append_batch(wl)
    assert seq.size == 8 * 4096
    pool = _gpu_append(wl, lat, rope, seq, pos)
    host = np.zeros(wl.num_blocks * 64 * 352, np.uint8)
    oracle.append(lat, rope, seq, pos, wl.block_table, 64, host, wl.num_blocks, 64 * 352)
    assert np.array_equal(pool.cpu().numpy(), host)
