"""Decode context parallelism, host side, on CPU: two gloo ranks shard the
top-k, exchange their partial states through dcp.gather_states (host staged)
and merge them; the result equals the single-rank decode of the whole
selection. The oracle stands in for the per-rank attention (no GPU here)."""
import os
import tempfile

import numpy as np
import torch
import torch.multiprocessing as mp


def _case():
    import oracle
    from workloads import all_tokens, make_queries, make_rows, make_workload
    wl = make_workload("tiny", num_seqs=2, seq_len=700, num_heads=8, topk=150, q_per_seq=2)
    seq, pos = all_tokens(wl)
    lat, rope = make_rows(wl, int(seq.size))
    stride = 64 * 352
    pool = np.zeros(wl.num_blocks * stride, np.uint8)
    assert oracle.append(lat, rope, seq, pos, wl.block_table, 64, pool, wl.num_blocks,
                         stride) == 0
    ql, qr = make_queries(wl)
    return wl, pool, stride, ql, qr


def _rank(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import oracle
    from nvfp4_compressed_mla_gb300 import dcp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl, pool, stride, ql, qr = _case()
        local = dcp.shard_topk(torch.from_numpy(wl.topk_idx), rank, world).numpy()
        o, l, _ = oracle.sparse_mla_decode(ql, qr, wl.q_seq, local, wl.block_table, wl.seq_lens,
                                           64, pool, wl.num_blocks, stride, 0, wl.sm_scale)
        all_o, all_l = dcp.gather_states(torch.from_numpy(o), torch.from_numpy(l))
        assert all_o.shape[0] == world
        # rank order is kept: this rank's own state sits at its index
        assert np.array_equal(all_o[rank].numpy(), o)
        out, lse = oracle.merge_states(all_o.numpy(), all_l.numpy())
        np.save(os.path.join(outdir, f"out{rank}.npy"), out)
        np.save(os.path.join(outdir, f"lse{rank}.npy"), lse)
    finally:
        dist.destroy_process_group()


def _run(world):
    import oracle
    with tempfile.TemporaryDirectory() as d:
        port = 29500 + (os.getpid() % 2000)
        mp.start_processes(_rank, args=(world, port, d), nprocs=world, start_method="spawn")
        wl, pool, stride, ql, qr = _case()
        ref, ref_lse, _ = oracle.sparse_mla_decode(ql, qr, wl.q_seq, wl.topk_idx, wl.block_table,
                                                   wl.seq_lens, 64, pool, wl.num_blocks, stride,
                                                   0, wl.sm_scale)
        for r in range(world):
            out = np.load(os.path.join(d, f"out{r}.npy"))
            lse = np.load(os.path.join(d, f"lse{r}.npy"))
            assert np.max(np.abs(out - ref)) < 1e-10
            assert np.max(np.abs(lse - ref_lse)) < 1e-10


def test_two_ranks():
    _run(2)


def test_three_ranks_ragged_shards():
    _run(3)  # 150 columns over 3 ranks


def test_shard_bounds_cover_the_selection():
    from nvfp4_compressed_mla_gb300 import dcp
    for topk in (1, 5, 128, 2048, 2049):
        for world in (1, 2, 3, 4, 8):
            cols = []
            for r in range(world):
                lo, hi = dcp.shard_bounds(topk, r, world)
                cols.extend(range(lo, hi))
            assert cols == list(range(topk))
    idx = torch.arange(5, dtype=torch.int32).view(1, 5)
    assert dcp.shard_topk(idx, 2, 4).tolist() == [[4]]
    assert dcp.shard_topk(idx, 3, 4).tolist() == [[-1]]  # empty range: one empty column
