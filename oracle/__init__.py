"""CPU oracle for the NVFP4-compressed MLA decode path (fp64, plain C).

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are its only callers; the library under
``nvfp4_compressed_mla_gb300`` never imports, links or runs it, and it
imports nothing from that library.

The C source (``nvfp4_mla_oracle.c``) states what is computed and which
passage of the Prime Inference post each step follows. This module only
builds it with gcc and marshals numpy arrays.

Parity pins (tests/test_oracle_pins.py) tie every function here to facts
outside the oracle: torch's float8_e4m3fn conversion, exact rational
arithmetic, the row sizes the post prints, closed forms of attention and a
dense fp64 softmax(QK^T)V computed by torch on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

LATENT_DIM = 512
ROPE_DIM = 64
ROW_BYTES = {0: 352, 1: 576}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, OpenMP, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f32, u8 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_uint8
            lib.orc_e4m3_encode.restype = u8
            lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
            lib.orc_e2m1_encode.restype = u8
            lib.orc_e2m1_encode.argtypes = [ctypes.c_double]
            for fn in ("orc_e4m3_encode_n", "orc_e2m1_encode_n", "orc_e4m3_decode_n",
                       "orc_e2m1_decode_n"):
                getattr(lib, fn).argtypes = [P, i64, P]
                getattr(lib, fn).restype = None
            lib.orc_quantize_rows.argtypes = [P, P, i64, i32, f32, f32, P]
            lib.orc_quantize_rows.restype = None
            lib.orc_dequant_rows.argtypes = [P, i64, i32, f32, f32, P, P]
            lib.orc_dequant_rows.restype = None
            lib.orc_append.argtypes = [P, P, P, P, i32, P, i32, i32, i32, P, i64, i64, i32, f32, f32]
            lib.orc_append.restype = i64
            lib.orc_sparse_mla_decode.argtypes = [P, P, P, P, i32, i32, i32, P, i32, i32, P, i32,
                                                  P, i64, i64, i32, f32, f32, f32, P, P,
                                                  ctypes.c_int]
            lib.orc_sparse_mla_decode.restype = i64
            lib.orc_max_threads.restype = ctypes.c_int
            lib.orc_stage_fp8.argtypes = [P, P, i32, i32, P, i32, i32, P, i32, P, i64, i64, f32,
                                          i64, P, P]
            lib.orc_stage_fp8.restype = i64
            lib.orc_merge_states.argtypes = [P, P, i32, i64, P, P]
            lib.orc_merge_states.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().orc_max_threads())


# ------------------------------------------------------------------ codecs
def e4m3_encode(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint8)
    _load().orc_e4m3_encode_n(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_decode(c) -> np.ndarray:
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().orc_e4m3_decode_n(_ptr(c), c.size, _ptr(out))
    return out


def e2m1_encode(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint8)
    _load().orc_e2m1_encode_n(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_decode(c) -> np.ndarray:
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().orc_e2m1_decode_n(_ptr(c), c.size, _ptr(out))
    return out


# --------------------------------------------------------------- row codec
def quantize_rows(latent_bf16, rope_bf16, row_format: int = 0, latent_scale: float = 1.0,
                  rope_scale: float = 1.0) -> np.ndarray:
    """Encode n tokens (bf16 bit patterns [n,512] and [n,64]) into cache rows [n, row_bytes]."""
    lat = _c(latent_bf16, np.uint16).reshape(-1, LATENT_DIM)
    rope = _c(rope_bf16, np.uint16).reshape(-1, ROPE_DIM)
    n = lat.shape[0]
    assert rope.shape[0] == n
    rows = np.empty((n, ROW_BYTES[row_format]), np.uint8)
    _load().orc_quantize_rows(_ptr(lat), _ptr(rope), n, row_format, latent_scale, rope_scale,
                              _ptr(rows))
    return rows


def dequant_rows(rows, row_format: int = 0, latent_scale: float = 1.0, rope_scale: float = 1.0):
    """Decoded fp64 latent [n,512] and rope [n,64] of cache rows."""
    rows = _c(rows, np.uint8).reshape(-1, ROW_BYTES[row_format])
    n = rows.shape[0]
    lat = np.empty((n, LATENT_DIM), np.float64)
    rope = np.empty((n, ROPE_DIM), np.float64)
    _load().orc_dequant_rows(_ptr(rows), n, row_format, latent_scale, rope_scale, _ptr(lat),
                             _ptr(rope))
    return lat, rope


# ------------------------------------------------------------ paged append
def append(latent_bf16, rope_bf16, seq_ids, positions, block_table, page_size: int,
           cache: np.ndarray, num_blocks: int, block_stride: int, row_format: int = 0,
           latent_scale: float = 1.0, rope_scale: float = 1.0) -> int:
    """Quantize tokens into their paged slots of ``cache`` (uint8, modified in place).

    Returns the number of tokens that did not resolve to a slot (skipped).
    """
    lat = _c(latent_bf16, np.uint16)
    rope = _c(rope_bf16, np.uint16)
    seq_ids = _c(seq_ids, np.int32)
    positions = _c(positions, np.int32)
    bt = _c(block_table, np.int32)
    assert cache.flags.c_contiguous and cache.dtype == np.uint8
    assert cache.size >= num_blocks * block_stride
    return int(_load().orc_append(_ptr(lat), _ptr(rope), _ptr(seq_ids), _ptr(positions),
                                  int(seq_ids.shape[0]), _ptr(bt), bt.shape[0], bt.shape[1],
                                  page_size, _ptr(cache), num_blocks, block_stride, row_format,
                                  latent_scale, rope_scale))


# --------------------------------------------------------------- attention
def sparse_mla_decode(q_latent_bf16, q_rope_bf16, q_seq, topk_idx, block_table, seq_lens,
                      page_size: int, cache: np.ndarray, num_blocks: int, block_stride: int,
                      row_format: int, sm_scale: float, latent_scale: float = 1.0,
                      rope_scale: float = 1.0, nthreads: int = 0):
    """fp64 sparse absorbed-MLA decode. Returns (out [num_q,H,512], lse [num_q,H], invalid)."""
    ql = _c(q_latent_bf16, np.uint16)
    qr = _c(q_rope_bf16, np.uint16)
    num_q, H = ql.shape[0], ql.shape[1]
    q_seq = _c(q_seq, np.int32)
    idx = _c(topk_idx, np.int32).reshape(num_q, -1)
    bt = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    assert cache.flags.c_contiguous and cache.dtype == np.uint8
    assert cache.size >= num_blocks * block_stride
    out = np.zeros((num_q, H, LATENT_DIM), np.float64)
    lse = np.zeros((num_q, H), np.float64)
    bad = _load().orc_sparse_mla_decode(
        _ptr(ql), _ptr(qr), _ptr(q_seq), _ptr(idx), num_q, H, idx.shape[1], _ptr(bt),
        bt.shape[0], bt.shape[1], _ptr(seq_lens), page_size, _ptr(cache), num_blocks,
        block_stride, row_format, sm_scale, latent_scale, rope_scale, _ptr(out), _ptr(lse),
        nthreads)
    return out, lse, int(bad)


# ------------------------------------------------------ staged FP8 rows
def stage_fp8(q_seq, topk_idx, block_table, seq_lens, page_size: int, cache: np.ndarray,
              num_blocks: int, block_stride: int, latent_scale: float = 1.0):
    """Selected NVFP4 rows re-encoded as FP8 rows (the staged comparison path).

    Returns (staged [num_q * R, 576] uint8, staged_idx [num_q, topk] int32,
    invalid) with R = topk rounded up to a multiple of page_size; rows of
    slots that do not resolve are zero.
    """
    q_seq = _c(q_seq, np.int32)
    idx = _c(topk_idx, np.int32)
    num_q, topk = idx.shape
    bt = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    R = (topk + page_size - 1) // page_size * page_size
    staged = np.zeros((num_q * R, ROW_BYTES[1]), np.uint8)
    sidx = np.empty((num_q, topk), np.int32)
    bad = _load().orc_stage_fp8(_ptr(q_seq), _ptr(idx), num_q, topk, _ptr(bt), bt.shape[0],
                                bt.shape[1], _ptr(seq_lens), page_size, _ptr(cache), num_blocks,
                                block_stride, latent_scale, R, _ptr(staged), _ptr(sidx))
    return staged, sidx, int(bad)


# ------------------------------------------------------------ state merge
def merge_states(part_out, part_lse):
    """Merge P attention states: part_out [P, num_q, H, 512], part_lse [P, num_q, H]
    (fp64) -> (out [num_q, H, 512], lse [num_q, H])."""
    po = _c(part_out, np.float64)
    pl = _c(part_lse, np.float64)
    P = po.shape[0]
    shape = pl.shape[1:]
    states = int(np.prod(shape))
    out = np.empty(shape + (LATENT_DIM,), np.float64)
    lse = np.empty(shape, np.float64)
    _load().orc_merge_states(_ptr(po), _ptr(pl), P, states, _ptr(out), _ptr(lse))
    return out, lse
