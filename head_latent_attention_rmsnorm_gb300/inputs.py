"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds random-number plumbing only -- none of the attention arithmetic.
Every tensor is a matrix of ``n_rows`` rows drawn from numpy's PCG64 generator,
one stream per block of ``BLOCK`` rows keyed by (seed, tensor id, block index), so
any row range (one simulated sequence-parallel rank, one decode batch) can be
regenerated on its own and matches the same rows of the full tensor bit for bit.

Values are drawn in float32 as N(0, std^2) and rounded once to the run dtype
(bf16 or fp32).  The oracle reads those rounded values widened to float64.
"""
from __future__ import annotations

import numpy as np
import torch

BLOCK = 256

# tensor ids (part of the stream key)
Q_NOPE, Q_PE, C_KV, K_PE, W_KV_B = 1, 2, 3, 4, 5
DEC_Q_NOPE, DEC_Q_PE, DEC_C_CACHE, DEC_KPE_CACHE = 11, 12, 13, 14
NORM_W = 15


def normal_rows(seed: int, tid: int, n_rows: int, row_elems: int, std: float = 1.0,
                r0: int = 0, r1: int | None = None) -> np.ndarray:
    """Rows [r0, r1) of an [n_rows, row_elems] float32 N(0, std^2) matrix."""
    r1 = n_rows if r1 is None else r1
    assert 0 <= r0 <= r1 <= n_rows
    out = np.empty((r1 - r0, row_elems), dtype=np.float32)
    b0, b1 = r0 // BLOCK, (r1 + BLOCK - 1) // BLOCK
    for blk in range(b0, b1):
        lo, hi = blk * BLOCK, min((blk + 1) * BLOCK, n_rows)
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid, blk])))
        vals = rng.standard_normal((hi - lo) * row_elems, dtype=np.float32).reshape(hi - lo, row_elems)
        if std != 1.0:
            vals *= np.float32(std)
        a, b = max(lo, r0), min(hi, r1)
        if a < b:
            out[a - r0:b - r0] = vals[a - lo:b - lo]
    return out


def to_torch(a: np.ndarray, dtype: torch.dtype, shape) -> torch.Tensor:
    """Round a float32 array to ``dtype`` (bf16 or fp32) as a CPU tensor of ``shape``."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(dtype).reshape(shape).contiguous()


def prefill_inputs(cfg, seed: int = 0, q_rows: tuple[int, int] | None = None) -> dict:
    """CPU tensors for one prefill workload.

    q_nope/q_pe cover query positions ``q_rows`` (default: the config's own
    [q_offset, q_offset + s_q)) of a full sequence of ``s_kv`` positions, so that
    slices for different simulated ranks are rows of one and the same tensor.
    """
    dt = cfg.torch_dtype
    B, H, S = cfg.batch, cfg.n_heads, cfg.s_kv
    r0, r1 = q_rows if q_rows is not None else (cfg.q_offset, cfg.q_offset + cfg.s_q)
    n = r1 - r0

    def qgen(tid, d):
        parts = [normal_rows(seed, tid, B * S, H * d, 1.0, b * S + r0, b * S + r1) for b in range(B)]
        return to_torch(np.concatenate(parts, 0), dt, (B, n, H, d))

    q_nope = qgen(Q_NOPE, cfg.d_nope)
    q_pe = qgen(Q_PE, cfg.d_rope)
    c_kv = to_torch(normal_rows(seed, C_KV, B * S, cfg.d_kv), dt, (B, S, cfg.d_kv))
    k_pe = to_torch(normal_rows(seed, K_PE, B * S, cfg.d_rope), dt, (B, S, cfg.d_rope))
    rows = H * (cfg.d_nope + cfg.d_v)
    w = to_torch(normal_rows(seed, W_KV_B, rows, cfg.d_kv, std=cfg.d_kv ** -0.5), dt, (rows, cfg.d_kv))
    rms_w = torch.ones(cfg.d_kv, dtype=dt)
    return dict(q_nope=q_nope, q_pe=q_pe, c_kv=c_kv, k_pe=k_pe, w_kv_b=w, rms_w=rms_w)


def decode_inputs(cfg, seed: int = 0, batches: tuple[int, int] | None = None,
                  with_weights: bool = True) -> dict:
    """CPU tensors for a latent decode workload (cache already normalised/rotated).

    ``batches`` selects a range of sequences; the rows match the full tensors'.
    """
    dt = cfg.torch_dtype
    B, H, L = cfg.batch, cfg.n_heads, cfg.kv_len
    b0, b1 = batches if batches is not None else (0, B)
    nb = b1 - b0
    q_nope = to_torch(normal_rows(seed, DEC_Q_NOPE, B, H * cfg.d_nope, 1.0, b0, b1), dt, (nb, H, cfg.d_nope))
    q_pe = to_torch(normal_rows(seed, DEC_Q_PE, B, H * cfg.d_rope, 1.0, b0, b1), dt, (nb, H, cfg.d_rope))
    c = to_torch(normal_rows(seed, DEC_C_CACHE, B * L, cfg.d_kv, 1.0, b0 * L, b1 * L), dt, (nb, L, cfg.d_kv))
    k = to_torch(normal_rows(seed, DEC_KPE_CACHE, B * L, cfg.d_rope, 1.0, b0 * L, b1 * L), dt, (nb, L, cfg.d_rope))
    d = dict(q_nope=q_nope, q_pe=q_pe, c_cache=c, kpe_cache=k)
    if with_weights:
        rows = H * (cfg.d_nope + cfg.d_v)
        d["w_kv_b"] = to_torch(normal_rows(seed, W_KV_B, rows, cfg.d_kv, std=cfg.d_kv ** -0.5), dt,
                               (rows, cfg.d_kv))
    return d


def norm_weight(d: int, dtype: torch.dtype, seed: int = 0, std: float = 0.1) -> torch.Tensor:
    """A latent-norm weight [d] drawn as 1 + N(0, std^2), rounded to ``dtype`` (the
    prefill workloads use all ones; shard tests want a weight whose slices differ)."""
    return to_torch(1.0 + normal_rows(seed, NORM_W, 1, d, std), dtype, (d,))
