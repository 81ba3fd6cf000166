"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol the header declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nvfp4_mla.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_compressed_mla_gb300 import _native
    return _native.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\**\s+\**(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("nvfp4_mla_append", "sparse_mla_decode", "sparse_mla_decode_workspace_size",
                 "sparse_mla_decode_num_splits", "nvfp4_mla_status_string",
                 "nvfp4_mla_row_bytes"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_declares_every_symbol():
    from nvfp4_compressed_mla_gb300 import _native
    assert set(declared_functions()) == set(_native.SIGNATURES)


def test_row_bytes_and_status_strings(lib):
    assert lib.nvfp4_mla_row_bytes(0) == 352
    assert lib.nvfp4_mla_row_bytes(1) == 576
    assert lib.nvfp4_mla_row_bytes(7) == 0
    seen = set()
    for s in range(10):
        msg = lib.nvfp4_mla_status_string(s).decode()
        assert msg and msg != "unknown status"
        seen.add(msg)
    assert len(seen) == 10
    assert lib.nvfp4_mla_status_string(99).decode() == "unknown status"


def test_wait_limit_setting(lib):
    assert lib.nvfp4_mla_set_wait_limit(-1) == 8  # NVFP4_MLA_ERR_VALUE
    assert lib.nvfp4_mla_set_wait_limit(5000) == 0
    assert lib.nvfp4_mla_set_wait_limit(0) == 0   # back to the default


def test_workspace_size_host_logic(lib):
    big = (1 << 64) - 1
    # invalid shapes
    assert lib.sparse_mla_decode_workspace_size(1, 0, 64, 1) == big
    assert lib.sparse_mla_decode_workspace_size(1, 129, 64, 1) == big
    assert lib.sparse_mla_decode_workspace_size(1, 16, 0, 1) == big
    assert lib.sparse_mla_decode_workspace_size(1, 16, 64, 65) == big
    # one split needs nothing; s splits need num_q * s * H * 513 floats
    assert lib.sparse_mla_decode_workspace_size(4, 16, 2048, 1) == 0
    assert lib.sparse_mla_decode_workspace_size(4, 16, 2048, 4) == 4 * 4 * 16 * 513 * 4
    # splits are clamped to the number of 128-slot tiles and never left empty
    assert lib.sparse_mla_decode_workspace_size(2, 8, 200, 8) == 2 * 2 * 8 * 513 * 4
    assert lib.sparse_mla_decode_workspace_size(2, 8, 100, 8) == 0  # one tile: one split
    assert lib.sparse_mla_decode_workspace_size(1, 8, 1280, 4) == 1 * 4 * 8 * 513 * 4  # 3,3,3,1
    assert lib.sparse_mla_decode_workspace_size(1, 8, 1152, 4) == 1 * 3 * 8 * 513 * 4  # 3,3,3


# ------------------------------------------------------------ validation
FAKE = 0x10000  # 16-byte aligned non-null address; never dereferenced on these paths


def _append(lib, **kw):
    a = dict(latent=FAKE, rope=FAKE, seq_ids=FAKE, positions=FAKE, n_tok=4, block_table=FAKE,
             num_seqs=1, max_blocks=4, page_size=64, cache=FAKE, num_blocks=4,
             block_stride=64 * 352, row_format=0, latent_scale=1.0, rope_scale=1.0,
             invalid_count=None, stream=None)
    a.update(kw)
    return lib.nvfp4_mla_append(*a.values())


def _decode(lib, **kw):
    a = dict(q_lat=FAKE, q_rope=FAKE, q_seq=FAKE, topk_idx=FAKE, num_q=2, num_heads=16, topk=64,
             block_table=FAKE, num_seqs=1, max_blocks=4, seq_lens=FAKE, page_size=64, cache=FAKE,
             num_blocks=4, block_stride=64 * 352, row_format=0, sm_scale=0.04, latent_scale=1.0,
             rope_scale=1.0, out=FAKE, out_fp32=0, lse=None, workspace=None, ws_bytes=0,
             num_splits=1, invalid_count=None, stream=None)
    a.update(kw)
    return lib.sparse_mla_decode(*a.values())


ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_FORMAT, ERR_VALUE = 1, 2, 3, 7, 8


@pytest.mark.parametrize("kw,status", [
    (dict(row_format=2), ERR_FORMAT),
    (dict(n_tok=-1), ERR_SHAPE),
    (dict(latent=None), ERR_NULL),
    (dict(cache=None), ERR_NULL),
    (dict(block_table=None), ERR_NULL),
    (dict(page_size=0), ERR_SHAPE),
    (dict(num_blocks=0), ERR_SHAPE),
    (dict(block_stride=64 * 352 - 16), ERR_SHAPE),
    (dict(block_stride=64 * 352 + 8), ERR_ALIGN),
    (dict(latent=FAKE + 8), ERR_ALIGN),
    (dict(cache=FAKE + 4), ERR_ALIGN),
    (dict(rope_scale=0.0), ERR_VALUE),
    (dict(rope_scale=float("nan")), ERR_VALUE),
    (dict(row_format=1, block_stride=64 * 576, latent_scale=-1.0), ERR_VALUE),
    (dict(row_format=1, block_stride=64 * 352), ERR_SHAPE),
])
def test_append_rejects_bad_arguments(lib, kw, status):
    assert _append(lib, **kw) == status


def test_append_zero_tokens_is_a_noop(lib):
    assert _append(lib, n_tok=0, latent=None) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(row_format=5), ERR_FORMAT),
    (dict(num_heads=0), ERR_SHAPE),
    (dict(num_heads=129), ERR_SHAPE),
    (dict(topk=0), ERR_SHAPE),
    (dict(topk=65537), ERR_SHAPE),
    (dict(num_q=-1), ERR_SHAPE),
    (dict(num_splits=65), ERR_SHAPE),
    (dict(q_lat=None), ERR_NULL),
    (dict(out=None), ERR_NULL),
    (dict(seq_lens=None), ERR_NULL),
    (dict(num_seqs=0), ERR_SHAPE),
    (dict(block_stride=100), ERR_SHAPE),
    (dict(q_rope=FAKE + 2), ERR_ALIGN),
    (dict(out=FAKE + 8), ERR_ALIGN),
    (dict(sm_scale=float("inf")), ERR_VALUE),
    (dict(latent_scale=0.0), ERR_VALUE),
])
def test_decode_rejects_bad_arguments(lib, kw, status):
    assert _decode(lib, **kw) == status


def test_decode_zero_queries_is_a_noop(lib):
    assert _decode(lib, num_q=0, q_lat=None) == 0


def test_valid_arguments_without_gpu_report_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _append(lib) in (4, 9)
    assert _decode(lib) in (4, 9)


# ------------------------------------------ staged comparison path and state merge
def _stage(lib, **kw):
    a = dict(q_seq=FAKE, idx=FAKE, num_q=2, topk=100, bt=FAKE, num_seqs=1, max_blocks=4,
             seq_lens=FAKE, page_size=64, cache=FAKE, num_blocks=4, block_stride=64 * 352,
             latent_scale=1.0, staged=FAKE, staged_idx=FAKE, invalid=None, stream=None)
    a.update(kw)
    return lib.nvfp4_mla_stage_fp8(a["q_seq"], a["idx"], a["num_q"], a["topk"], a["bt"],
                                   a["num_seqs"], a["max_blocks"], a["seq_lens"], a["page_size"],
                                   a["cache"], a["num_blocks"], a["block_stride"],
                                   a["latent_scale"], a["staged"], a["staged_idx"], a["invalid"],
                                   a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(topk=0), ERR_SHAPE),
    (dict(topk=65537), ERR_SHAPE),
    (dict(page_size=0), ERR_SHAPE),
    (dict(num_q=-1), ERR_SHAPE),
    (dict(staged=None), ERR_NULL),
    (dict(staged_idx=None), ERR_NULL),
    (dict(cache=None), ERR_NULL),
    (dict(block_stride=64 * 352 - 16), ERR_SHAPE),
    (dict(block_stride=64 * 352 + 8), ERR_ALIGN),
    (dict(staged=FAKE + 4), ERR_ALIGN),
    (dict(latent_scale=-1.0), ERR_VALUE),
    (dict(latent_scale=float("nan")), ERR_VALUE),
])
def test_stage_rejects_bad_arguments(lib, kw, status):
    assert _stage(lib, **kw) == status


def test_stage_zero_queries_and_rows_per_query(lib):
    assert _stage(lib, num_q=0, staged=None) == 0
    assert lib.nvfp4_mla_staged_rows_per_q(100, 64) == 128
    assert lib.nvfp4_mla_staged_rows_per_q(128, 64) == 128
    assert lib.nvfp4_mla_staged_rows_per_q(1, 16) == 16
    assert lib.nvfp4_mla_staged_rows_per_q(0, 64) == 0
    assert lib.nvfp4_mla_staged_rows_per_q(10, 0) == 0


def _merge(lib, **kw):
    a = dict(part_out=FAKE, part_lse=FAKE, parts=2, num_q=3, heads=16, out=FAKE, out_fp32=0,
             lse=None, stream=None)
    a.update(kw)
    return lib.sparse_mla_merge_states(a["part_out"], a["part_lse"], a["parts"], a["num_q"],
                                       a["heads"], a["out"], a["out_fp32"], a["lse"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(parts=0), ERR_SHAPE),
    (dict(parts=1025), ERR_SHAPE),
    (dict(heads=0), ERR_SHAPE),
    (dict(heads=129), ERR_SHAPE),
    (dict(num_q=-2), ERR_SHAPE),
    (dict(part_out=None), ERR_NULL),
    (dict(part_lse=None), ERR_NULL),
    (dict(out=None), ERR_NULL),
    (dict(part_out=FAKE + 4), ERR_ALIGN),
    (dict(out=FAKE + 8), ERR_ALIGN),
])
def test_merge_rejects_bad_arguments(lib, kw, status):
    assert _merge(lib, **kw) == status


def test_new_entry_points_without_gpu_report_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _stage(lib) in (4, 9)
    assert _merge(lib) in (4, 9)
    assert _merge(lib, num_q=0) == 0
