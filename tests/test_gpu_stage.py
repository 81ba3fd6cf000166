"""GPU: the staged-dequant comparison path against the fp64 oracle.

The staged FP8 rows and their indices must match the oracle's staging byte
for byte (the re-encoding is a rounding decision taken in fp32 on both
sides); the FP8 decode over the staged rows is compared with the oracle's
decode of the oracle's staged rows, at the decode tests' tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_cases import assert_parity, build_case, dev_tensor
from workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("topk,latent_scale,num_heads", [
    (200, 1.0, 128),   # ragged pages, full head count
    (64, 0.5, 16),     # exactly one page per token
    (700, 2.0, 33),    # several pages, ragged heads
    (300, 0.75, 64),   # a scale that is not a power of two: the division path
])
def test_staged_rows_and_staged_decode(topk, latent_scale, num_heads):
    import nvfp4_compressed_mla_gb300 as nm
    wl = make_workload("agent", num_seqs=3, seq_len=5000, topk=topk, num_heads=num_heads)
    case = build_case(wl, "referenced")
    idx = wl.topk_idx.copy()
    idx[0, 1] = -1               # empty slot
    idx[1, 2] = 10 ** 7          # beyond the sequence: counted
    idx[2, topk - 1] = -3        # negative: counted
    d = case.dev
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    staged, sidx = nm.nvfp4_mla_stage_fp8(d["q_seq"], dev_tensor(idx), d["bt"], d["seq_lens"],
                                          wl.page_size, d["pool"], wl.num_blocks, case.stride,
                                          latent_scale, invalid_count=cnt)
    torch.cuda.synchronize()
    ref_staged, ref_sidx, bad = oracle.stage_fp8(wl.q_seq, idx, wl.block_table, wl.seq_lens,
                                                 wl.page_size, case.host_pool, wl.num_blocks,
                                                 case.stride, latent_scale)
    assert bad == 2 and int(cnt.item()) == 2
    got_sidx = sidx.cpu().numpy()
    assert np.array_equal(got_sidx, ref_sidx)
    R = nm.nvfp4_mla_staged_rows_per_q(topk, wl.page_size)
    got_rows = staged.cpu().numpy()[: wl.num_q * R * 576].reshape(wl.num_q * R, 576)
    t, j = np.nonzero(ref_sidx >= 0)
    assert np.array_equal(got_rows[t * R + j], ref_staged[t * R + j])

    tb = nm.staged_fp8_tables(wl.num_q, topk, wl.page_size, "cuda:0")
    out, lse = nm.sparse_mla_decode(d["ql"], d["qr"], tb["q_seq"], sidx, tb["block_table"],
                                    tb["seq_lens"], wl.page_size, staged, tb["num_blocks"],
                                    tb["block_stride_bytes"], nm.ROW_FP8_576, wl.sm_scale,
                                    latent_scale, 1.0, out_fp32=True)
    torch.cuda.synchronize()
    P = R // wl.page_size
    ref, ref_lse, rbad = oracle.sparse_mla_decode(
        case.ql, case.qr, np.arange(wl.num_q, dtype=np.int32), ref_sidx,
        np.arange(wl.num_q * P, dtype=np.int32).reshape(wl.num_q, P),
        np.full(wl.num_q, topk, np.int32), wl.page_size, ref_staged.reshape(-1),
        wl.num_q * P, wl.page_size * 576, 1, wl.sm_scale, latent_scale, 1.0)
    assert rbad == 0
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref, ref_lse)


def test_stage_rejects_bad_arguments():
    import nvfp4_compressed_mla_gb300 as nm
    lib = nm._lib()
    assert lib.nvfp4_mla_staged_rows_per_q(0, 64) == 0
    assert lib.nvfp4_mla_staged_rows_per_q(100, 64) == 128
    z = torch.zeros(64, dtype=torch.int32, device="cuda:0")
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda:0")
    p = z.data_ptr()
    # null staged buffer
    assert lib.nvfp4_mla_stage_fp8(p, p, 1, 4, p, 1, 1, p, 64, buf.data_ptr(), 1, 64 * 352, 1.0,
                                   None, p, None, None) == nm_status("NULL")
    # latent_scale not positive
    assert lib.nvfp4_mla_stage_fp8(p, p, 1, 4, p, 1, 1, p, 64, buf.data_ptr(), 1, 64 * 352, 0.0,
                                   buf.data_ptr(), p, None, None) == nm_status("VALUE")
    # misaligned staged buffer
    assert lib.nvfp4_mla_stage_fp8(p, p, 1, 4, p, 1, 1, p, 64, buf.data_ptr(), 1, 64 * 352, 1.0,
                                   buf.data_ptr() + 4, p, None, None) == nm_status("ALIGN")


def nm_status(name):
    return {"NULL": 1, "SHAPE": 2, "ALIGN": 3, "VALUE": 8}[name]
