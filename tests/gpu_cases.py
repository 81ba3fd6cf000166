"""Helpers for the GPU parity tests: build one workload's cache on both sides.

The oracle quantizes the seeded bf16 rows into a host pool; that pool is
copied to the device for the decode tests, so every oracle input comes from
the generators and the oracle, never from the CUDA path. Append parity is
checked separately (the CUDA append on the same bf16 inputs must reproduce
the oracle's pool byte for byte).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

import oracle
from workloads import (Workload, all_tokens, make_queries, make_rows, referenced_tokens)

TOL_REL_L2 = 2e-3      # attention output, relative L2 per query token (over H x 512)
TOL_LSE_ABS = 1e-3     # natural-log LSE, absolute


def dev_tensor(a: np.ndarray, dtype: Optional[torch.dtype] = None, device="cuda:0"):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


@dataclasses.dataclass
class Case:
    wl: Workload
    row_format: int
    row_bytes: int
    stride: int
    latent_scale: float
    rope_scale: float
    host_pool: np.ndarray
    seq: np.ndarray           # tokens written into the pool
    pos: np.ndarray
    lat: np.ndarray           # their bf16 latent / rope
    rope: np.ndarray
    ql: np.ndarray
    qr: np.ndarray
    dev: dict


def build_case(wl: Workload, fill: str = "all", row_format: int = 0, stride_pad: int = 0,
               latent_scale: float = 1.0, rope_scale: float = 1.0, device="cuda:0",
               to_device: bool = True) -> Case:
    rb = 352 if row_format == 0 else 576
    stride = wl.page_size * rb + stride_pad
    seq, pos = all_tokens(wl) if fill == "all" else referenced_tokens(wl)
    lat, rope = make_rows(wl, int(seq.size))
    host_pool = np.zeros(wl.num_blocks * stride, np.uint8)
    bad = oracle.append(lat, rope, seq, pos, wl.block_table, wl.page_size, host_pool,
                        wl.num_blocks, stride, row_format, latent_scale, rope_scale)
    assert bad == 0
    ql, qr = make_queries(wl)
    dev = {}
    if to_device:
        dev = dict(
            pool=dev_tensor(host_pool, device=device),
            ql=dev_tensor(ql, torch.bfloat16, device), qr=dev_tensor(qr, torch.bfloat16, device),
            q_seq=dev_tensor(wl.q_seq, device=device), idx=dev_tensor(wl.topk_idx, device=device),
            bt=dev_tensor(wl.block_table, device=device),
            seq_lens=dev_tensor(wl.seq_lens, device=device))
    return Case(wl, row_format, rb, stride, latent_scale, rope_scale, host_pool, seq, pos, lat,
                rope, ql, qr, dev)


def gpu_decode(case: Case, num_splits: int = 0, out_fp32: bool = True, idx=None, q_seq=None,
               invalid_count=None, workspace=None):
    import nvfp4_compressed_mla_gb300 as nm
    d = case.dev
    out, lse = nm.sparse_mla_decode(
        d["ql"], d["qr"], d["q_seq"] if q_seq is None else q_seq,
        d["idx"] if idx is None else idx, d["bt"], d["seq_lens"], case.wl.page_size, d["pool"],
        case.wl.num_blocks, case.stride, case.row_format, case.wl.sm_scale, case.latent_scale,
        case.rope_scale, out_fp32=out_fp32, num_splits=num_splits, invalid_count=invalid_count,
        workspace=workspace)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def oracle_decode(case: Case, tokens=None, idx=None, q_seq=None):
    wl = case.wl
    tok = np.arange(wl.num_q) if tokens is None else np.asarray(tokens)
    idx = wl.topk_idx if idx is None else idx
    q_seq = wl.q_seq if q_seq is None else q_seq
    return oracle.sparse_mla_decode(case.ql[tok], case.qr[tok], q_seq[tok], idx[tok],
                                    wl.block_table, wl.seq_lens, wl.page_size, case.host_pool,
                                    wl.num_blocks, case.stride, case.row_format, wl.sm_scale,
                                    case.latent_scale, case.rope_scale)


def rel_l2(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Relative L2 error per query token over its H x 512 outputs (absolute if ref is 0)."""
    g = got.reshape(got.shape[0], -1)
    r = ref.reshape(ref.shape[0], -1)
    num = np.linalg.norm(g - r, axis=1)
    den = np.linalg.norm(r, axis=1)
    return np.where(den > 0, num / np.maximum(den, 1e-300), num)


def lse_err(got: np.ndarray, ref: np.ndarray) -> float:
    both_inf = np.isneginf(got) & np.isneginf(ref)
    if np.any(np.isneginf(got) != np.isneginf(ref)):
        return float("inf")
    d = np.abs(np.where(both_inf, 0.0, got - np.where(both_inf, 0.0, ref)))
    return float(d.max()) if d.size else 0.0


def assert_parity(got_out, got_lse, ref_out, ref_lse, tol=TOL_REL_L2, lse_tol=TOL_LSE_ABS):
    e = rel_l2(got_out, ref_out)
    assert np.all(e <= tol), f"relative L2 per token: max {e.max():.3e} > {tol}"
    le = lse_err(got_lse, ref_lse)
    assert le <= lse_tol, f"lse abs err {le:.3e} > {lse_tol}"
    return float(e.max()), le
