"""Plain CPU oracle for MLA attention from the compressed latent.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``head_latent_attention_rmsnorm_gb300``) never does,
and this package imports nothing from it.

The arithmetic lives in ``mla_oracle.c`` (IEEE double, plain loops; see its header
for the page citations and the readings taken where the pages are silent).  This
module compiles it with gcc and exposes numpy-in / numpy-out wrappers.

Parity status of each function (what pins it: ``tests/test_oracle_pins.py``, repeated over
random small shapes in ``tests/test_oracle_sweep.py``):
  rmsnorm, rope, mla_explicit, mla_absorbed, mla_decode, lse_combine, tpla_decode,
  mla_explicit_bwd, rmsnorm_bwd -- all pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "libmla_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libmla_oracle.so`` (gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        path = os.environ.get("MLA_ORACLE_LIB")   # a variant build (used by the mutation test)
        if not path:
            path = build()
        lib = ctypes.CDLL(path)
        i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.orc_rmsnorm.argtypes = [_dp, _dp, l, i, d, _dp]
        lib.orc_rope.argtypes = [_dp, _dp, l, i, d, _dp]
        fwd = [i, i, i, i, i, i, i, i, i, i, i, i, d, d, d] + [_dp] * 8
        lib.orc_mla_explicit.argtypes = fwd
        lib.orc_mla_absorbed.argtypes = fwd
        lib.orc_mla_decode.argtypes = [i, i, i, i, i, i, i, i, d, d] + [_dp] * 9
        lib.orc_lse_combine.argtypes = [i, l, i, _dp, _dp, _dp, _dp]
        lib.orc_tpla_decode.argtypes = [i, i, i, i, i, i, i, i, d, d, d] + [_dp] * 8
        lib.orc_rmsnorm_bwd.argtypes = [_dp, _dp, l, i, i, d, _dp, _dp, _dp]
        lib.orc_mla_explicit_bwd.argtypes = [i, i, i, i, i, i, i, i, i, i, i, i, d, d, d] + [_dp] * 13
        for f in ("orc_rmsnorm", "orc_rope", "orc_mla_explicit", "orc_mla_absorbed",
                  "orc_mla_decode", "orc_lse_combine", "orc_tpla_decode", "orc_mla_explicit_bwd",
                  "orc_rmsnorm_bwd"):
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    if a is None:
        return ctypes.cast(None, _dp)
    return a.ctypes.data_as(_dp)


def default_scale(d_nope: int, d_rope: int) -> float:
    return 1.0 / float(np.sqrt(d_nope + d_rope))


def rmsnorm(x, w, eps: float) -> np.ndarray:
    x = _f64(x)
    w = _f64(w)
    d = x.shape[-1]
    y = np.empty_like(x)
    _load().orc_rmsnorm(_p(x), _p(w), x.size // d, d, eps, _p(y))
    return y


def rope(x, pos, base: float) -> np.ndarray:
    """Rotate each row of ``x`` (last dim = d_rope) at the per-row position ``pos``."""
    x = _f64(x)
    d = x.shape[-1]
    rows = x.size // d
    pos = _f64(np.broadcast_to(np.asarray(pos, dtype=np.float64), x.shape[:-1])).reshape(rows)
    y = np.empty_like(x)
    _load().orc_rope(_p(x), _p(pos), rows, d, base, _p(y))
    return y


def _fwd(fn, q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, *, n_heads, q_offset=0, causal=True,
         head_begin=0, base=10000.0, eps=1e-6, scale=None):
    q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w = map(_f64, (q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w))
    B, s_q, hc, dn = q_nope.shape
    dr = q_pe.shape[-1]
    s_kv, dk = c_kv.shape[1], c_kv.shape[2]
    dv = w_kv_b.shape[0] // n_heads - dn
    if scale is None:
        scale = default_scale(dn, dr)
    out = np.zeros((B, s_q, hc, dv))
    lse = np.zeros((B, hc, s_q))
    fn(B, s_q, s_kv, q_offset, int(bool(causal)), n_heads, head_begin, hc, dk, dn, dr, dv,
       float(base), float(eps), float(scale), _p(q_nope), _p(q_pe), _p(c_kv), _p(k_pe),
       _p(w_kv_b), _p(rms_w), _p(out), _p(lse))
    return out, lse


def mla_explicit(*args, **kw):
    """Explicit/LAGA MLA forward.  Returns (out [B,s_q,H_loc,Dv], lse [B,H_loc,s_q])."""
    return _fwd(_load().orc_mla_explicit, *args, **kw)


def rmsnorm_bwd(x, w, dy, *, shards=1, eps=1e-6):
    """Gradient of the per-shard RMSNorm over the last dim.  Returns (dx, dw)."""
    x, w, dy = map(_f64, (x, w, dy))
    d = x.shape[-1]
    dx, dw = np.zeros_like(x), np.zeros(d)
    _load().orc_rmsnorm_bwd(_p(x), _p(w), x.size // d, d, shards, float(eps), _p(dy), _p(dx), _p(dw))
    return dx, dw


def mla_explicit_bwd(q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, dout, *, n_heads, q_offset=0, causal=True,
                     head_begin=0, base=10000.0, eps=1e-6, scale=None):
    """Gradients of :func:`mla_explicit`'s output contracted with ``dout``.  Returns a
    dict: q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w (each shaped like its input)."""
    q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, dout = map(_f64, (q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, dout))
    B, s_q, hc, dn = q_nope.shape
    dr = q_pe.shape[-1]
    s_kv, dk = c_kv.shape[1], c_kv.shape[2]
    dv = w_kv_b.shape[0] // n_heads - dn
    if scale is None:
        scale = default_scale(dn, dr)
    g = {k: np.zeros_like(v) for k, v in
         dict(q_nope=q_nope, q_pe=q_pe, c_kv=c_kv, k_pe=k_pe, w_kv_b=w_kv_b, rms_w=rms_w).items()}
    _load().orc_mla_explicit_bwd(B, s_q, s_kv, q_offset, int(bool(causal)), n_heads, head_begin, hc, dk, dn, dr,
                                 dv, float(base), float(eps), float(scale), _p(q_nope), _p(q_pe), _p(c_kv),
                                 _p(k_pe), _p(w_kv_b), _p(rms_w), _p(dout), _p(g["q_nope"]), _p(g["q_pe"]),
                                 _p(g["c_kv"]), _p(g["k_pe"]), _p(g["w_kv_b"]), _p(g["rms_w"]))
    return g


def mla_absorbed(*args, **kw):
    """Absorbed-form MLA forward, same contract as :func:`mla_explicit`."""
    return _fwd(_load().orc_mla_absorbed, *args, **kw)


def mla_decode(q_nope, q_pe, c_cache, kpe_cache, w_kv_b, *, n_splits=1, base=10000.0,
               scale=None, partials=True):
    """Latent decode.  Returns (out [B,H,Dv], lse [B,H], part_out [n,B,H,Dk], part_lse [n,B,H])."""
    q_nope, q_pe, c_cache, kpe_cache, w_kv_b = map(_f64, (q_nope, q_pe, c_cache, kpe_cache, w_kv_b))
    B, H, dn = q_nope.shape
    dr = q_pe.shape[-1]
    L, dk = c_cache.shape[1], c_cache.shape[2]
    dv = w_kv_b.shape[0] // H - dn
    if scale is None:
        scale = default_scale(dn, dr)
    out = np.zeros((B, H, dv))
    lse = np.zeros((B, H))
    po = np.zeros((n_splits, B, H, dk)) if partials else None
    pl = np.zeros((n_splits, B, H)) if partials else None
    _load().orc_mla_decode(B, L, n_splits, H, dk, dn, dr, dv, float(base), float(scale),
                           _p(q_nope), _p(q_pe), _p(c_cache), _p(kpe_cache), _p(w_kv_b),
                           _p(out), _p(lse), _p(po), _p(pl))
    return out, lse, po, pl


def tpla_decode(q_nope, q_pe, c_raw, kpe_cache, w_kv_b, rms_w, *, shards=2, eps=1e-6,
                base=10000.0, scale=None):
    """TPLA latent decode over ``shards`` latent shards (see ``orc_tpla_decode``).

    ``c_raw`` [B,L,Dk] is the latent before normalisation (each shard is RMSNormed on its
    own); with ``rms_w=None`` it is taken as already normalised shard by shard.
    Returns (out [B,H,Dv] summed over shards, shard_lse [shards,B,H])."""
    q_nope, q_pe, c_raw, kpe_cache, w_kv_b = map(_f64, (q_nope, q_pe, c_raw, kpe_cache, w_kv_b))
    rms_w = None if rms_w is None else _f64(rms_w)
    B, H, dn = q_nope.shape
    dr = q_pe.shape[-1]
    L, dk = c_raw.shape[1], c_raw.shape[2]
    if dk % shards:
        raise ValueError("d_kv must divide into the shards")
    dv = w_kv_b.shape[0] // H - dn
    if scale is None:
        scale = default_scale(dn, dr)
    out = np.zeros((B, H, dv))
    slse = np.zeros((shards, B, H))
    _load().orc_tpla_decode(B, L, shards, H, dk, dn, dr, dv, float(base), float(scale), float(eps),
                            _p(q_nope), _p(q_pe), _p(c_raw), _p(kpe_cache), _p(w_kv_b),
                            None if rms_w is None else _p(rms_w),
                            _p(out), _p(slse))
    return out, slse


def lse_combine(part_out, part_lse):
    """Merge split partials [n,rows,D] / [n,rows] into (out [rows,D], lse [rows])."""
    part_out = _f64(part_out)
    part_lse = _f64(part_lse)
    n, rows, D = part_out.shape
    out = np.zeros((rows, D))
    lse = np.zeros(rows)
    _load().orc_lse_combine(n, rows, D, _p(part_out), _p(part_lse), _p(out), _p(lse))
    return out, lse
