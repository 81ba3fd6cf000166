"""GPU: sparse_mla_decode_noalloc, the decode entry point that allocates nothing.

It serves callers that cannot allocate device memory themselves (for
example a plugin whose host application owns the device heap and forbids
cudaMalloc): its split-K scratch is a static device buffer inside the
library. Checked through the C ABI against sparse_mla_decode with a
caller-provided workspace, on two calls in a row with different shapes (so
stale scratch from the first call would show up in the second), plus the
size limit. Collected last so a failure here never hides another test.
"""
import numpy as np
import pytest
import torch

from tests.gpu_cases import TOL_LSE_ABS, TOL_REL_L2, build_case, lse_err, rel_l2
from workloads import make_workload

pytestmark = pytest.mark.gpu

ERR_WORKSPACE = 5
SCRATCH_BYTES = 16 * 1024 * 1024


def _noalloc(lib, case, num_splits, out, lse):
    d, wl = case.dev, case.wl
    st = lib.sparse_mla_decode_noalloc(
        d["ql"].data_ptr(), d["qr"].data_ptr(), d["q_seq"].data_ptr(), d["idx"].data_ptr(),
        wl.num_q, wl.num_heads, wl.topk, d["bt"].data_ptr(), wl.num_seqs, wl.max_blocks_per_seq,
        d["seq_lens"].data_ptr(), wl.page_size, d["pool"].data_ptr(), wl.num_blocks, case.stride,
        case.row_format, wl.sm_scale, case.latent_scale, case.rope_scale, out.data_ptr(), 1,
        lse.data_ptr(), num_splits, None, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st


def _with_workspace(lib, case, num_splits):
    d, wl = case.dev, case.wl
    need = lib.sparse_mla_decode_workspace_size(wl.num_q, wl.num_heads, wl.topk, num_splits)
    assert 0 < need <= SCRATCH_BYTES  # the case really uses scratch, and fits the static buffer
    ws = torch.empty(need, dtype=torch.uint8, device="cuda:0")
    out = torch.empty((wl.num_q, wl.num_heads, 512), dtype=torch.float32, device="cuda:0")
    lse = torch.empty((wl.num_q, wl.num_heads), dtype=torch.float32, device="cuda:0")
    st = lib.sparse_mla_decode(
        d["ql"].data_ptr(), d["qr"].data_ptr(), d["q_seq"].data_ptr(), d["idx"].data_ptr(),
        wl.num_q, wl.num_heads, wl.topk, d["bt"].data_ptr(), wl.num_seqs, wl.max_blocks_per_seq,
        d["seq_lens"].data_ptr(), wl.page_size, d["pool"].data_ptr(), wl.num_blocks, case.stride,
        case.row_format, wl.sm_scale, case.latent_scale, case.rope_scale, out.data_ptr(), 1,
        lse.data_ptr(), ws.data_ptr(), need, num_splits, None,
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    from nvfp4_compressed_mla_gb300 import _native
    lib = _native.load()
    cases = [
        (build_case(make_workload("agent", num_seqs=3, seq_len=6000, topk=1000, num_heads=32)), 4),
        (build_case(make_workload("tiny", num_seqs=2, seq_len=900, topk=600, q_per_seq=3),
                    row_format=1, latent_scale=0.5, rope_scale=2.0), 0),
    ]
    for case, splits in cases:  # two calls in a row, different shapes and formats
        wl = case.wl
        out = torch.full((wl.num_q, wl.num_heads, 512), float("nan"), device="cuda:0")
        lse = torch.full((wl.num_q, wl.num_heads), float("nan"), device="cuda:0")
        assert _noalloc(lib, case, splits, out, lse) == 0
        ref_out, ref_lse = _with_workspace(lib, case, splits)
        got_out, got_lse = out.double().cpu().numpy(), lse.double().cpu().numpy()
        assert np.all(rel_l2(got_out, ref_out) <= TOL_REL_L2)
        assert lse_err(got_lse, ref_lse) <= TOL_LSE_ABS


def test_noalloc_rejects_shapes_beyond_the_static_buffer():
    from nvfp4_compressed_mla_gb300 import _native
    lib = _native.load()
    case = build_case(make_workload("tiny", num_seqs=1, seq_len=2048, topk=2048, num_heads=128,
                                    q_per_seq=8))
    # 8 tokens x 32 splits x 128 heads x 513 floats = 67 MB > 16 MiB
    assert lib.sparse_mla_decode_workspace_size(8, 128, 2048, 32) > SCRATCH_BYTES
    out = torch.full((8, 128, 512), 7.0, device="cuda:0")
    lse = torch.full((8, 128), 7.0, device="cuda:0")
    assert _noalloc(lib, case, 32, out, lse) == ERR_WORKSPACE
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())  # nothing was enqueued
