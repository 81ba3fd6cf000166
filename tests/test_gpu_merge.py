"""GPU: sparse_mla_merge_states against the fp64 oracle merge, and decode
context parallelism emulated in one process (each "rank" decodes its share of
the top-k on the GPU, the parts are merged on the GPU) against the oracle's
decode of the whole selection."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_cases import (TOL_REL_L2, assert_parity, build_case, dev_tensor, oracle_decode,
                             rel_l2)
from workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("parts,out_fp32", [(1, True), (3, True), (8, False)])
def test_merge_matches_oracle(parts, out_fp32):
    import nvfp4_compressed_mla_gb300 as nm
    rng = np.random.default_rng(parts)
    num_q, H = 5, 33
    po = rng.standard_normal((parts, num_q, H, 512)).astype(np.float32)
    pl = (rng.standard_normal((parts, num_q, H)) * 4).astype(np.float32)
    pl[0, 1, :] = -np.inf                 # an empty part
    if parts > 1:
        pl[:, 2, 5] = -np.inf             # a (token, head) with every part empty
    out, lse = nm.sparse_mla_merge_states(dev_tensor(po), dev_tensor(pl), out_fp32=out_fp32)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.merge_states(po.astype(np.float64), pl.astype(np.float64))
    got = out.double().cpu().numpy()
    # bf16 output: round-to-nearest to 8 significant bits alone gives about
    # 2^-8 / sqrt(7) = 1.5e-3 relative L2 on values spread over a binade
    tol = 1e-5 if out_fp32 else TOL_REL_L2
    assert np.all(rel_l2(got, ref) <= tol)
    gl = lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(gl), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    assert np.max(np.abs(gl[fin] - ref_lse[fin])) < 1e-4


@pytest.mark.parametrize("world", [2, 3])
def test_context_parallel_emulated(world):
    import nvfp4_compressed_mla_gb300 as nm
    from nvfp4_compressed_mla_gb300 import dcp
    wl = make_workload("decode_batch", num_seqs=2, seq_len=9000, topk=2048, num_heads=128)
    case = build_case(wl, "referenced")
    d = case.dev
    outs, lses = [], []
    for r in range(world):
        o, l = nm.sparse_mla_decode(d["ql"], d["qr"], d["q_seq"], dcp.shard_topk(d["idx"], r, world),
                                    d["bt"], d["seq_lens"], wl.page_size, d["pool"],
                                    wl.num_blocks, case.stride, 0, wl.sm_scale, out_fp32=True)
        outs.append(o)
        lses.append(l)
    out, lse = nm.sparse_mla_merge_states(torch.stack(outs), torch.stack(lses), out_fp32=True)
    torch.cuda.synchronize()
    ref, ref_lse, _ = oracle_decode(case)
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref, ref_lse)
