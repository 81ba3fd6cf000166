"""NVFP4-compressed MLA KV cache and sparse decode attention for GB300 (sm_103a).

Thin Python binding over the C ABI declared in ``include/nvfp4_mla.h``:
the functions below carry the C entry points' names and only marshal
arguments (torch tensors -> device pointers, the current CUDA stream).
Every step of the computation runs in the library's CUDA kernels; if the
library is missing or the device is not an sm_103 part the calls raise.

Method: the Prime Inference post ("Prime Inference: Fast, Reliable Serving
for Frontier Open Models"), sections "Making room for low-latency decode"
(352-byte NVFP4 rows) and "Native NVFP4 sparse MLA decode kernel".
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _native

LATENT_DIM = 512
ROPE_DIM = 64
ROW_NVFP4_352 = 0
ROW_FP8_576 = 1
ROW_BYTES = {ROW_NVFP4_352: 352, ROW_FP8_576: 576}

__all__ = [
    "LATENT_DIM", "ROPE_DIM", "ROW_NVFP4_352", "ROW_FP8_576", "ROW_BYTES", "NativeError",
    "nvfp4_mla_row_bytes", "nvfp4_mla_status_string", "nvfp4_mla_append",
    "sparse_mla_decode_num_splits", "sparse_mla_decode_workspace_size", "sparse_mla_decode",
    "nvfp4_mla_set_wait_limit",
    "sparse_mla_merge_states", "nvfp4_mla_staged_rows_per_q", "nvfp4_mla_stage_fp8",
    "staged_fp8_tables", "library_path",
]


class NativeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({nvfp4_mla_status_string(status)})")


def library_path() -> str:
    return _native.library_path()


def _lib():
    return _native.load()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the C ABI must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, where: str) -> None:
    if status != 0:
        raise NativeError(status, where)


def nvfp4_mla_row_bytes(row_format: int) -> int:
    return int(_lib().nvfp4_mla_row_bytes(row_format))


def nvfp4_mla_status_string(status: int) -> str:
    return _lib().nvfp4_mla_status_string(status).decode()


def nvfp4_mla_append(latent: torch.Tensor, rope: torch.Tensor, seq_ids: torch.Tensor,
                     positions: torch.Tensor, block_table: torch.Tensor, page_size: int,
                     cache: torch.Tensor, num_blocks: int, block_stride_bytes: int,
                     row_format: int = ROW_NVFP4_352, latent_scale: float = 1.0,
                     rope_scale: float = 1.0, invalid_count: Optional[torch.Tensor] = None,
                     stream=None) -> None:
    """Quantize ``latent`` [n,512] / ``rope`` [n,64] (bf16) into their paged cache rows."""
    n = latent.shape[0] if latent.dim() else 0
    st = _lib().nvfp4_mla_append(
        _ptr(latent), _ptr(rope), _ptr(seq_ids), _ptr(positions), n, _ptr(block_table),
        block_table.shape[0], block_table.shape[1], page_size, _ptr(cache), num_blocks,
        block_stride_bytes, row_format, latent_scale, rope_scale, _ptr(invalid_count),
        _stream(stream))
    _check(st, "nvfp4_mla_append")


def sparse_mla_decode_num_splits(num_q: int, num_heads: int, topk: int) -> int:
    return int(_lib().sparse_mla_decode_num_splits(num_q, num_heads, topk))


def nvfp4_mla_set_wait_limit(cycles: int) -> None:
    """Bound (SM clock cycles) of the decode kernel's internal waits; 0 = default."""
    _check(_lib().nvfp4_mla_set_wait_limit(int(cycles)), "nvfp4_mla_set_wait_limit")


def sparse_mla_decode_workspace_size(num_q: int, num_heads: int, topk: int,
                                     num_splits: int = 0) -> int:
    n = int(_lib().sparse_mla_decode_workspace_size(num_q, num_heads, topk, num_splits))
    if n == (1 << 64) - 1:
        raise ValueError("invalid decode shape")
    return n


def sparse_mla_decode(q_latent: torch.Tensor, q_rope: torch.Tensor, q_seq: torch.Tensor,
                      topk_idx: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                      page_size: int, cache: torch.Tensor, num_blocks: int,
                      block_stride_bytes: int, row_format: int, sm_scale: float,
                      latent_scale: float = 1.0, rope_scale: float = 1.0,
                      out: Optional[torch.Tensor] = None, out_fp32: bool = False,
                      lse: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, num_splits: int = 0,
                      invalid_count: Optional[torch.Tensor] = None, stream=None):
    """Sparse absorbed-MLA decode; returns (out [num_q,H,512], lse [num_q,H]).

    ``out`` / ``lse`` / ``workspace`` are allocated with torch when not given.
    """
    num_q, H = q_latent.shape[0], q_latent.shape[1]
    topk = topk_idx.shape[1]
    dev = q_latent.device
    if out is None:
        out = torch.empty((num_q, H, LATENT_DIM), device=dev,
                          dtype=torch.float32 if out_fp32 else torch.bfloat16)
    if lse is None:
        lse = torch.empty((num_q, H), device=dev, dtype=torch.float32)
    need = sparse_mla_decode_workspace_size(num_q, H, topk, num_splits) if num_q else 0
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib().sparse_mla_decode(
        _ptr(q_latent), _ptr(q_rope), _ptr(q_seq), _ptr(topk_idx), num_q, H, topk,
        _ptr(block_table), block_table.shape[0], block_table.shape[1], _ptr(seq_lens), page_size,
        _ptr(cache), num_blocks, block_stride_bytes, row_format, sm_scale, latent_scale,
        rope_scale, _ptr(out), 1 if out_fp32 else 0, _ptr(lse), _ptr(workspace), ws_bytes,
        num_splits, _ptr(invalid_count), _stream(stream))
    _check(st, "sparse_mla_decode")
    return out, lse


def sparse_mla_merge_states(part_out: torch.Tensor, part_lse: torch.Tensor,
                            out: Optional[torch.Tensor] = None, out_fp32: bool = False,
                            lse: Optional[torch.Tensor] = None, stream=None):
    """Merge P partial attention states (fp32 [P,num_q,H,512], [P,num_q,H]);
    returns (out [num_q,H,512], lse [num_q,H])."""
    P, num_q, H = part_out.shape[0], part_out.shape[1], part_out.shape[2]
    dev = part_out.device
    if out is None:
        out = torch.empty((num_q, H, LATENT_DIM), device=dev,
                          dtype=torch.float32 if out_fp32 else torch.bfloat16)
    if lse is None:
        lse = torch.empty((num_q, H), device=dev, dtype=torch.float32)
    st = _lib().sparse_mla_merge_states(_ptr(part_out), _ptr(part_lse), P, num_q, H, _ptr(out),
                                        1 if out_fp32 else 0, _ptr(lse), _stream(stream))
    _check(st, "sparse_mla_merge_states")
    return out, lse

# ------------------------------------------------ staged-dequant comparison path
def nvfp4_mla_staged_rows_per_q(topk: int, page_size: int) -> int:
    """Staged FP8 rows per query token (topk rounded up to whole pages)."""
    n = int(_lib().nvfp4_mla_staged_rows_per_q(topk, page_size))
    if n == 0:
        raise ValueError("invalid topk or page_size")
    return n


def nvfp4_mla_stage_fp8(q_seq: torch.Tensor, topk_idx: torch.Tensor, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, page_size: int, cache: torch.Tensor,
                        num_blocks: int, block_stride_bytes: int, latent_scale: float = 1.0,
                        staged: Optional[torch.Tensor] = None,
                        staged_idx: Optional[torch.Tensor] = None,
                        invalid_count: Optional[torch.Tensor] = None, stream=None):
    """Selected NVFP4 rows re-encoded as FP8 rows; returns (staged, staged_idx).

    ``staged`` (uint8, num_q * R * 576 bytes) and ``staged_idx`` (int32
    [num_q, topk]) are allocated with torch when not given.
    """
    num_q, topk = topk_idx.shape[0], topk_idx.shape[1]
    dev = topk_idx.device
    R = nvfp4_mla_staged_rows_per_q(topk, page_size)
    if staged is None:
        staged = torch.empty(max(num_q * R * ROW_BYTES[ROW_FP8_576], 16), dtype=torch.uint8,
                             device=dev)
    if staged_idx is None:
        staged_idx = torch.empty((num_q, topk), dtype=torch.int32, device=dev)
    st = _lib().nvfp4_mla_stage_fp8(
        _ptr(q_seq), _ptr(topk_idx), num_q, topk, _ptr(block_table), block_table.shape[0],
        block_table.shape[1], _ptr(seq_lens), page_size, _ptr(cache), num_blocks,
        block_stride_bytes, latent_scale, _ptr(staged), _ptr(staged_idx), _ptr(invalid_count),
        _stream(stream))
    _check(st, "nvfp4_mla_stage_fp8")
    return staged, staged_idx


def staged_fp8_tables(num_q: int, topk: int, page_size: int, device) -> dict:
    """Index tables for reading the staged rows with sparse_mla_decode (FP8 rows):
    token t is sequence t, its rows fill pages t * P .. t * P + P - 1."""
    R = nvfp4_mla_staged_rows_per_q(topk, page_size)
    P = R // page_size
    return {
        "q_seq": torch.arange(num_q, dtype=torch.int32, device=device),
        "block_table": torch.arange(num_q * P, dtype=torch.int32, device=device).view(num_q, P),
        "seq_lens": torch.full((num_q,), topk, dtype=torch.int32, device=device),
        "num_blocks": num_q * P,
        "block_stride_bytes": page_size * ROW_BYTES[ROW_FP8_576],
    }
