"""Seeded generators for the five decode workloads (and scaled-down copies).

Every array is drawn from ``numpy.random.Generator(PCG64(seed))``; nothing
here quantises, dequantises or attends. Shapes follow the workloads the
Prime Inference post ("Prime Inference: Fast, Reliable Serving for Frontier
Open Models") describes for its decode path:

* 64-token pages scattered over one shared pool (section "Changing the
  layout to reduce fragmentation": 64-token blocks).
* at most 2048 selected positions per query token, unused slots set to -1
  (sections "Decode: NVFP4 KV compression" and "Native NVFP4 sparse MLA
  decode kernel", the empty-slot paragraph).
* agent sessions of about 140K history tokens plus about 6K new tokens per
  turn, 66 sessions (sections "Workload" and "Performance").

Workloads by name:

``tiny``          1 sequence x 4096 tokens, 1 query token, 16 heads, top-k 256.
``decode_batch``  64 sequences x 32768 tokens, 128 heads, 1 query each, top-k 2048.
``agent``         66 sessions of U[142000, 150000] tokens, 128 heads, top-k 2048:
                  1024 from the last 8192 positions + 1024 uniform over the rest;
                  latent values N(0,1) with 1 % of elements scaled by 20.
``multi_token``   32 sequences x 65536 tokens, 15 query tokens per sequence,
                  each with its own causal top-k 2048 set, 128 heads.
``append_dense``  8 sequences: a 12288-token prefix plus an appended 4096-token
                  chunk; decode attends to all 16384 positions, 128 heads.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

CONFIG_NAMES = ("tiny", "decode_batch", "agent", "multi_token", "append_dense")

LATENT_DIM = 512
ROPE_DIM = 64


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def f32_from_bf16(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    num_heads: int
    page_size: int
    topk: int
    seq_lens: np.ndarray        # int32 [num_seqs]
    block_table: np.ndarray     # int32 [num_seqs, max_blocks_per_seq], -1 = unused
    num_blocks: int             # physical pages in the pool
    q_seq: np.ndarray           # int32 [num_q]
    q_pos: np.ndarray           # int32 [num_q] position of the query token's own row
    topk_idx: np.ndarray        # int32 [num_q, topk], -1 = empty slot
    sm_scale: float
    latent_scale: float = 1.0
    rope_scale: float = 1.0
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    prefix_len: int = 0         # append_dense: tokens present before the appended chunk

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_q(self) -> int:
        return int(self.q_seq.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.sum())

    def valid_slots(self) -> int:
        return int((self.topk_idx >= 0).sum())


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def _block_table(rng, seq_lens, page_size):
    pages = [(int(n) + page_size - 1) // page_size for n in seq_lens]
    total = int(sum(pages))
    max_pages = max(pages) if pages else 0
    phys = rng.permutation(total).astype(np.int32)
    bt = np.full((len(seq_lens), max(max_pages, 1)), -1, dtype=np.int32)
    off = 0
    for s, p in enumerate(pages):
        bt[s, :p] = phys[off:off + p]
        off += p
    return bt, total


def _draw(rng, limit: int, k: int, mode: str, recent: int = 8192) -> np.ndarray:
    """k distinct positions in [0, limit), padded with -1 when limit < k."""
    out = np.full(k, -1, dtype=np.int32)
    if limit <= 0:
        return out
    if limit <= k:
        sel = np.arange(limit, dtype=np.int64)
        if mode == "uniform":
            rng.shuffle(sel)
        out[:limit] = sel
        return out
    if mode == "all":
        raise ValueError("mode 'all' needs topk >= context length")
    if mode == "recent_mix" and limit > recent:
        k_recent = k // 2
        lo = limit - recent
        a = rng.choice(recent, size=k_recent, replace=False) + lo
        b = rng.choice(lo, size=k - k_recent, replace=False)
        sel = np.sort(np.concatenate([a, b]))
    else:
        sel = rng.choice(limit, size=k, replace=False)
        if mode != "uniform":
            sel = np.sort(sel)
    out[:] = sel
    return out


def _build(name, seed, seq_lens, q_per_seq, topk, num_heads, mode, page_size=64,
           outlier_frac=0.0, outlier_mult=1.0, prefix_len=0, row_format_scales=(1.0, 1.0)):
    rng = _rng(seed, 0)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    bt, nblk = _block_table(rng, seq_lens, page_size)
    q_seq, q_pos, idx = [], [], []
    for s, L in enumerate(seq_lens):
        for i in range(q_per_seq):
            pos = int(L) - q_per_seq + i           # causal: token i sees positions <= pos
            q_seq.append(s)
            q_pos.append(pos)
            idx.append(_draw(rng, pos + 1, topk, mode))
    return Workload(
        name=name, seed=seed, num_heads=num_heads, page_size=page_size, topk=topk,
        seq_lens=seq_lens, block_table=bt, num_blocks=nblk,
        q_seq=np.asarray(q_seq, dtype=np.int32), q_pos=np.asarray(q_pos, dtype=np.int32),
        topk_idx=np.stack(idx).astype(np.int32) if idx else np.zeros((0, topk), np.int32),
        sm_scale=float(np.float32(1.0 / math.sqrt(LATENT_DIM + ROPE_DIM))),
        latent_scale=row_format_scales[0], rope_scale=row_format_scales[1],
        outlier_frac=outlier_frac, outlier_mult=outlier_mult, prefix_len=prefix_len)


def make_workload(name: str, seed: Optional[int] = None, *, num_seqs: Optional[int] = None,
                  seq_len: Optional[int] = None, num_heads: Optional[int] = None,
                  topk: Optional[int] = None, q_per_seq: Optional[int] = None,
                  page_size: int = 64, mode: Optional[str] = None) -> Workload:
    """Build one of the named workloads; keyword overrides give scaled-down copies.

    The default seed is 1000 + the workload's number (1..5).
    """
    if name not in CONFIG_NAMES:
        raise ValueError(f"unknown workload {name!r}")
    number = CONFIG_NAMES.index(name) + 1
    seed = 1000 + number if seed is None else seed
    if name == "tiny":
        ns, L, H, k, qps, m = 1, 4096, 16, 256, 1, "uniform"
        lens = [seq_len or L] * (num_seqs or ns)
    elif name == "decode_batch":
        ns, L, H, k, qps, m = 64, 32768, 128, 2048, 1, "sorted"
        lens = [seq_len or L] * (num_seqs or ns)
    elif name == "agent":
        ns, H, k, qps, m = 66, 128, 2048, 1, "recent_mix"
        r = _rng(seed, 1)
        n = num_seqs or ns
        lens = (r.integers(142000, 150001, size=n) if seq_len is None
                else np.full(n, seq_len)).tolist()
    elif name == "multi_token":
        ns, L, H, k, qps, m = 32, 65536, 128, 2048, 15, "sorted"
        lens = [seq_len or L] * (num_seqs or ns)
    else:  # append_dense
        ns, L, H, qps, m = 8, 16384, 128, 1, "all"
        n_len = seq_len or L
        lens = [n_len] * (num_seqs or ns)
        k = topk or n_len
        wl = _build(name, seed, lens, q_per_seq or qps, k, num_heads or H, mode or m, page_size,
                    prefix_len=n_len - n_len // 4)
        return wl
    outl = (0.01, 20.0) if name == "agent" else (0.0, 1.0)
    return _build(name, seed, lens, q_per_seq or qps, topk or k, num_heads or H, mode or m,
                  page_size, outlier_frac=outl[0], outlier_mult=outl[1])


def _values(rng, shape, outlier_frac, outlier_mult):
    x = rng.standard_normal(shape, dtype=np.float32)
    if outlier_frac > 0:
        mask = rng.random(shape, dtype=np.float32) < outlier_frac
        x = np.where(mask, x * np.float32(outlier_mult), x)
    return bf16_from_f32(x)


def make_queries(wl: Workload, stream: int = 0):
    """bf16 q_latent [num_q, H, 512] and q_rope [num_q, H, 64] as uint16 bit patterns."""
    r = _rng(wl.seed, 2, stream)
    ql = bf16_from_f32(r.standard_normal((wl.num_q, wl.num_heads, LATENT_DIM), dtype=np.float32))
    qr = bf16_from_f32(r.standard_normal((wl.num_q, wl.num_heads, ROPE_DIM), dtype=np.float32))
    return ql, qr


def make_rows(wl: Workload, n: int, stream: int = 0):
    """bf16 latent [n, 512] and rope [n, 64] values for n cache tokens (uint16 bit patterns)."""
    r = _rng(wl.seed, 3, stream)
    lat = _values(r, (n, LATENT_DIM), wl.outlier_frac, wl.outlier_mult)
    rope = _values(r, (n, ROPE_DIM), 0.0, 1.0)
    return lat, rope


def referenced_tokens(wl: Workload):
    """Unique (seq, pos) pairs that some valid top-k entry selects, sorted."""
    valid = wl.topk_idx >= 0
    seq = np.broadcast_to(wl.q_seq[:, None], wl.topk_idx.shape)[valid].astype(np.int64)
    pos = wl.topk_idx[valid].astype(np.int64)
    key = np.unique(seq * (1 << 32) + pos)
    return (key >> 32).astype(np.int32), (key & 0xFFFFFFFF).astype(np.int32)


def all_tokens(wl: Workload):
    """Every (seq, pos) pair of every sequence, in sequence-major order."""
    seq = np.repeat(np.arange(wl.num_seqs, dtype=np.int32), wl.seq_lens)
    pos = np.concatenate([np.arange(n, dtype=np.int32) for n in wl.seq_lens]) if wl.num_seqs else \
        np.zeros(0, np.int32)
    return seq, pos


def make_append_batch(wl: Workload, stream: int = 0):
    """The tokens appended in one decode step: one per query token at its own position.

    For ``append_dense`` this is the whole 4096-token chunk of every sequence
    (positions prefix_len .. seq_len-1). Returns (seq_ids, positions, latent, rope).
    """
    if wl.prefix_len:
        seq = np.repeat(np.arange(wl.num_seqs, dtype=np.int32), wl.seq_lens - wl.prefix_len)
        pos = np.concatenate([np.arange(wl.prefix_len, n, dtype=np.int32) for n in wl.seq_lens])
    else:
        seq, pos = wl.q_seq.copy(), wl.q_pos.copy()
    lat, rope = make_rows(wl, int(seq.shape[0]), stream=1000 + stream)
    return seq, pos, lat, rope


def redraw_indices(wl: Workload, stream: int) -> np.ndarray:
    """A fresh top-k set per query token for the same sequences (another model layer).

    Same selection rule as the workload's own, drawn from an independent stream.
    """
    mode = {"tiny": "uniform", "decode_batch": "sorted", "agent": "recent_mix",
            "multi_token": "sorted", "append_dense": "all"}[wl.name]
    rng = _rng(wl.seed, 4, stream)
    return np.stack([_draw(rng, int(p) + 1, wl.topk, mode) for p in wl.q_pos]).astype(np.int32)
