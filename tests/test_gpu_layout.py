"""GPU: cache layouts the C ABI admits beyond one pool per layer.

- BLHNC-style multi-layer pool: every physical block holds the 64-row pages
  of all layers back to back (layer l at byte l * page_bytes of the block,
  block stride = layers * page_bytes), so one layer is addressed as
  cache = pool + l * page_bytes with that stride.
- Physical-slot indices: a top-k entry names a pool row directly (block *
  64 + row); expressed through the ABI as one sequence spanning the pool
  with the identity block table.
Append bytes are compared with the oracle's appends into the same layout;
decode output with the oracle's decode of the same bytes.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_cases import assert_parity, dev_tensor
from workloads import all_tokens, make_queries, make_rows, make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layers,row_format", [(3, 0), (2, 1)])
def test_interleaved_layers(layers, row_format):
    import nvfp4_compressed_mla_gb300 as nm
    wl = make_workload("decode_batch", num_seqs=3, seq_len=2000, topk=500, num_heads=64)
    rb = 352 if row_format == 0 else 576
    page = wl.page_size * rb
    stride = layers * page
    ls, rs = (1.0, 1.0) if row_format == 0 else (0.5, 2.0)
    seq, pos = all_tokens(wl)
    host = np.zeros(wl.num_blocks * stride + layers * page, np.uint8)  # tail: room for views
    pool = torch.zeros(host.size, dtype=torch.uint8, device="cuda:0")
    bt = dev_tensor(wl.block_table)
    per_layer = []
    for li in range(layers):
        lat, rope = make_rows(make_workload("decode_batch", seed=77 + li, num_seqs=3,
                                            seq_len=2000, topk=500, num_heads=64),
                              int(seq.size))
        view = host[li * page:]
        assert oracle.append(lat, rope, seq, pos, wl.block_table, wl.page_size, view,
                             wl.num_blocks, stride, row_format, ls, rs) == 0
        nm.nvfp4_mla_append(dev_tensor(lat, torch.bfloat16), dev_tensor(rope, torch.bfloat16),
                            dev_tensor(seq), dev_tensor(pos), bt, wl.page_size,
                            pool[li * page:], wl.num_blocks, stride, row_format, ls, rs)
        per_layer.append(li)
    torch.cuda.synchronize()
    assert np.array_equal(pool.cpu().numpy(), host), "interleaved append bytes differ"
    ql, qr = make_queries(wl)
    for li in range(layers):
        out, lse = nm.sparse_mla_decode(
            dev_tensor(ql, torch.bfloat16), dev_tensor(qr, torch.bfloat16), dev_tensor(wl.q_seq),
            dev_tensor(wl.topk_idx), bt, dev_tensor(wl.seq_lens), wl.page_size, pool[li * page:],
            wl.num_blocks, stride, row_format, wl.sm_scale, ls, rs, out_fp32=True)
        torch.cuda.synchronize()
        ref, ref_lse, bad = oracle.sparse_mla_decode(
            ql, qr, wl.q_seq, wl.topk_idx, wl.block_table, wl.seq_lens, wl.page_size,
            host[li * page:], wl.num_blocks, stride, row_format, wl.sm_scale, ls, rs)
        assert bad == 0
        assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref, ref_lse)


def test_physical_slot_indices():
    import nvfp4_compressed_mla_gb300 as nm
    wl = make_workload("tiny", num_seqs=4, seq_len=1500, num_heads=32, topk=300, q_per_seq=1)
    stride = wl.page_size * 352
    seq, pos = all_tokens(wl)
    lat, rope = make_rows(wl, int(seq.size))
    host = np.zeros(wl.num_blocks * stride, np.uint8)
    assert oracle.append(lat, rope, seq, pos, wl.block_table, wl.page_size, host,
                         wl.num_blocks, stride) == 0
    # physical slot of each selected (sequence, position): page id * 64 + row
    phys = np.full_like(wl.topk_idx, -1)
    for t in range(wl.num_q):
        b = wl.q_seq[t]
        for j, p in enumerate(wl.topk_idx[t]):
            if p >= 0:
                phys[t, j] = wl.block_table[b, p // 64] * 64 + p % 64
    ident = np.arange(wl.num_blocks, dtype=np.int32)[None, :]
    q_seq0 = np.zeros(wl.num_q, np.int32)
    lens = np.array([wl.num_blocks * 64], np.int32)
    ql, qr = make_queries(wl)
    out, lse = nm.sparse_mla_decode(
        dev_tensor(ql, torch.bfloat16), dev_tensor(qr, torch.bfloat16), dev_tensor(q_seq0),
        dev_tensor(phys), dev_tensor(ident), dev_tensor(lens), wl.page_size, dev_tensor(host),
        wl.num_blocks, stride, 0, wl.sm_scale, out_fp32=True)
    torch.cuda.synchronize()
    # the same rows through the logical tables
    ref, ref_lse, bad = oracle.sparse_mla_decode(ql, qr, wl.q_seq, wl.topk_idx, wl.block_table,
                                                 wl.seq_lens, wl.page_size, host, wl.num_blocks,
                                                 stride, 0, wl.sm_scale)
    assert bad == 0
    assert_parity(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref, ref_lse)
