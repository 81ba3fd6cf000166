"""GPU: sparse_mla_decode against the fp64 oracle on the same dequantised rows.

Tolerance (from the stated accuracy target): out within 2e-3 relative L2 per
query token over its H x 512 values; natural-log LSE within 1e-3 absolute.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_cases import (TOL_REL_L2, assert_parity, build_case, dev_tensor, gpu_decode,
                             oracle_decode, rel_l2)
from workloads import make_workload

pytestmark = pytest.mark.gpu


# A page stride that is not a whole number of rows (the ABI allows any multiple
# of 16 bytes >= page_size * row_bytes) makes the decode gather each row with
# its own bulk copy instead of the row-indexed tensor copies.
PAD = {0: 48, 1: 16}


@pytest.mark.parametrize("padded", [False, True])
@pytest.mark.parametrize("num_heads,topk,seq_len,splits", [
    (16, 256, 4096, 0),     # the tiny workload's shape
    (16, 37, 600, 1),       # one ragged tile
    (1, 200, 900, 2),       # single head, ragged tail split in two
    (33, 1000, 3000, 3),    # ragged head group, uneven splits
    (128, 300, 2000, 0),    # full head count, ragged
    (64, 64, 64, 1),        # exactly one full tile, every position
])
def test_small_cases(num_heads, topk, seq_len, splits, padded):
    wl = make_workload("tiny", num_seqs=2, seq_len=seq_len, num_heads=num_heads, topk=topk,
                       q_per_seq=2)
    case = build_case(wl, stride_pad=PAD[0] if padded else 0)
    assert (case.stride % case.row_bytes != 0) == padded
    out, lse = gpu_decode(case, num_splits=splits)
    ref, ref_lse, bad = oracle_decode(case)
    assert bad == 0
    e, _ = assert_parity(out, lse, ref, ref_lse)
    assert e < 5e-4  # fp32 output: only FP16 P rounding and fp32 accumulation remain


# More units (query token x split) than the device holds clusters at once:
# each cluster takes several units in turn, its barriers' phases running on
# from one unit to the next. Every token is checked.
@pytest.mark.parametrize("row_format", [0, 1])
@pytest.mark.parametrize("num_heads,topk,splits,out_fp32", [
    (64, 300, 1, False),    # 240 units of three tiles (the last one ragged), bf16 out
    (16, 600, 2, True),     # 480 units: 240 tokens x 2 splits (the second one ragged)
    (128, 64, 1, True),     # 240 one-tile units, full head count
])
def test_more_units_than_resident_clusters(row_format, num_heads, topk, splits, out_fp32):
    wl = make_workload("tiny", num_seqs=4, seq_len=3000, num_heads=num_heads, topk=topk,
                       q_per_seq=60)
    case = build_case(wl, "referenced", row_format)
    ref, ref_lse, bad = oracle_decode(case)
    assert bad == 0
    out, lse = gpu_decode(case, out_fp32=out_fp32, num_splits=splits)
    assert_parity(out, lse, ref, ref_lse)


@pytest.mark.parametrize("padded", [False, True])
@pytest.mark.parametrize("row_format", [0, 1])
def test_bf16_output_and_fp8_rows(row_format, padded):
    wl = make_workload("agent", num_seqs=3, seq_len=5000, topk=700)
    case = build_case(wl, "referenced", row_format, latent_scale=0.75, rope_scale=1.5,
                      stride_pad=PAD[row_format] if padded else 0)
    assert (case.stride % case.row_bytes != 0) == padded
    ref, ref_lse, _ = oracle_decode(case)
    for out_fp32 in (False, True):
        for splits in (0, 3):
            out, lse = gpu_decode(case, out_fp32=out_fp32, num_splits=splits)
            assert_parity(out, lse, ref, ref_lse)


def test_split_counts_agree():
    wl = make_workload("decode_batch", num_seqs=2, seq_len=8192, topk=2048, num_heads=32)
    case = build_case(wl, "referenced")
    ref, ref_lse, _ = oracle_decode(case)
    outs = []
    for s in (1, 2, 3, 4, 8, 13, 32):
        out, lse = gpu_decode(case, num_splits=s)
        assert_parity(out, lse, ref, ref_lse)
        outs.append(out)
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) < 1e-4


def test_empty_slots_invalid_entries_and_empty_tokens():
    wl = make_workload("tiny", num_seqs=3, seq_len=700, num_heads=16, topk=128, q_per_seq=1)
    case = build_case(wl)
    idx = wl.topk_idx.copy()
    idx[0, 100:] = -1                       # short context: -1 tail
    idx[1, ::7] = -1                        # scattered -1
    idx[1, 3] = 700                         # == seq_len -> invalid
    idx[1, 5] = -5                          # negative -> invalid
    idx[1, 9] = 1 << 30                     # far beyond the block table -> invalid
    idx[2, :] = -1                          # nothing selected
    q_seq = wl.q_seq.copy()
    inv = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    out, lse = gpu_decode(case, idx=dev_tensor(idx), num_splits=2, invalid_count=inv)
    ref, ref_lse, bad = oracle_decode(case, idx=idx, q_seq=q_seq)
    assert bad == 3 and int(inv.item()) == 3
    assert_parity(out, lse, ref, ref_lse)
    assert not out[2].any() and np.all(np.isneginf(lse[2]))


def test_bad_block_table_entries_and_sequences():
    wl = make_workload("tiny", num_seqs=2, seq_len=640, num_heads=16, topk=64)
    case = build_case(wl)
    bt = wl.block_table.copy()
    bt[0, 2] = wl.num_blocks + 5            # page outside the pool
    bt[1, 0] = -7
    q_seq = wl.q_seq.copy()
    q_seq[1] = 9                            # no such sequence
    case.wl.block_table = bt
    case.dev["bt"] = dev_tensor(bt)
    inv = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    out, lse = gpu_decode(case, q_seq=dev_tensor(q_seq), invalid_count=inv)
    ref, ref_lse, bad = oracle_decode(case, q_seq=q_seq)
    assert bad > 0 and int(inv.item()) == bad
    assert_parity(out, lse, ref, ref_lse)


def test_duplicates_and_order():
    wl = make_workload("tiny", num_seqs=1, seq_len=900, num_heads=16, topk=96)
    case = build_case(wl)
    idx = wl.topk_idx.copy()
    idx2 = np.concatenate([idx, idx], 1)
    rng = np.random.default_rng(0)
    perm = idx2[:, rng.permutation(idx2.shape[1])]
    out1, lse1 = gpu_decode(case, idx=dev_tensor(idx2))
    out2, lse2 = gpu_decode(case, idx=dev_tensor(np.ascontiguousarray(perm)))
    ref, ref_lse, _ = oracle_decode(case, idx=idx2)
    assert_parity(out1, lse1, ref, ref_lse)
    assert_parity(out2, lse2, ref, ref_lse)
    base, base_lse = gpu_decode(case)
    assert np.allclose(lse1, base_lse + np.log(2.0), atol=1e-4)


# -------------------------------------------------- full-size configurations
def _full(name, row_format=0):
    """Every query token of the workload against the oracle, in the launch the
    benchmark times (automatic splits, bf16 output)."""
    wl = make_workload(name)
    case = build_case(wl, "referenced", row_format)
    out, lse = gpu_decode(case, num_splits=0, out_fp32=False)
    ref, ref_lse, bad = oracle_decode(case)
    assert bad == 0
    assert_parity(out, lse, ref, ref_lse)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("name", ["tiny", "decode_batch", "agent", "multi_token"])
def test_full_size_config(name):
    _full(name)


@pytest.mark.parametrize("row_format", [0, 1])
def test_full_size_append_dense(row_format):
    _full("append_dense", row_format)


# -------------------------------------------------- the largest top-k the ABI accepts
@pytest.mark.parametrize("splits", [0, 1])
def test_maximum_topk(splits):
    """topk = 65536 (512 tiles; automatic splits and one cluster walking all of them),
    128 heads, a -1 tail; every head against the oracle."""
    wl = make_workload("tiny", num_seqs=1, seq_len=70000, num_heads=128, topk=65536,
                       q_per_seq=1)
    case = build_case(wl, "referenced")
    idx = wl.topk_idx.copy()
    idx[:, -1000:] = -1
    out, lse = gpu_decode(case, num_splits=splits, idx=dev_tensor(idx))
    ref, ref_lse, bad = oracle_decode(case, idx=idx)
    assert bad == 0
    assert_parity(out, lse, ref, ref_lse)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
