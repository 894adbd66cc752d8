"""Thin ctypes binding of ``libmla.so`` (declared in ``include/mla.h``).

Two layers, argument marshalling only:

* ``mla_latent_attn_fwd`` ... ``mla_lse_combine``, the ``*_workspace`` queries,
  ``mla_status_string``, ``mla_check_device_error``: the C entry points under their
  own names, taking integers for pointers and sizes.
* ``latent_attn_fwd``, ``absorbed_attn_fwd``, ``decode_splitkv``, ``lse_combine``,
  ``tpla_decode``, ``rmsnorm``, ``rmsnorm_bwd``:
  the same calls taking torch tensors; they allocate any output or workspace the
  caller did not pass (through torch's allocator, so the CUDA caching allocator sees
  every byte) and raise :class:`MlaError` on a non-OK status.

Every step of the computation runs in the library's CUDA kernels.  If the library
is missing this module raises on first use; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")

MLA_F32, MLA_BF16 = 0, 1
STATUS = {0: "MLA_OK", -1: "MLA_ERR_NULL", -2: "MLA_ERR_SHAPE", -3: "MLA_ERR_DTYPE", -4: "MLA_ERR_ALIGN",
          -5: "MLA_ERR_WORKSPACE", -6: "MLA_ERR_UNSUPPORTED", -7: "MLA_ERR_CUDA",
          -8: "MLA_ERR_DEVICE_TIMEOUT", -9: "MLA_ERR_ALIAS"}
PATH_NONE, PATH_SIMT, PATH_TC, PATH_TC_FUSED = 0, 1, 2, 3


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__("%s: %s" % (where, mla_status_string(status)))
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int), ("d_kv", ctypes.c_int), ("d_nope", ctypes.c_int),
                ("d_rope", ctypes.c_int), ("d_v", ctypes.c_int), ("rope_base", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("softmax_scale", ctypes.c_float)]


def dims(n_heads, d_kv, d_nope, d_rope, d_v, rope_base=10000.0, rms_eps=1e-6, softmax_scale=0.0) -> Dims:
    return Dims(n_heads, d_kv, d_nope, d_rope, d_v, rope_base, rms_eps, softmax_scale)


def dims_of(cfg) -> Dims:
    """Dims of a workload from :mod:`.configs`."""
    eps = getattr(cfg, "rms_eps", 1e-6)
    return dims(cfg.n_heads, cfg.d_kv, cfg.d_nope, cfg.d_rope, cfg.d_v, cfg.rope_base, eps)


_lib = None
_vp, _i, _sz, _fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmla.so is not built (run: python -m head_latent_attention_rmsnorm_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        D = ctypes.POINTER(Dims)
        fwd = [D, _i, _i, _i, _i, _i, _i, _i, _i, _i] + [_vp] * 8 + [_vp, _sz, _vp]
        for f in ("mla_latent_attn_fwd", "mla_absorbed_attn_fwd"):
            getattr(L, f).argtypes = fwd
            getattr(L, f).restype = _i
        L.mla_latent_attn_fused_fwd.argtypes = [D, _i, _i, _i, _i, _i, _i, _i, _i] + [_vp] * 8 + [_vp, _sz, _vp]
        L.mla_latent_attn_fused_fwd.restype = _i
        L.mla_latent_attn_fused_workspace.argtypes = [D, _i, _i, _i, _i, _i, _i, _i]
        L.mla_latent_attn_fused_workspace.restype = _sz
        L.mla_set_fused_cluster.argtypes = [_i]
        L.mla_set_fused_cluster.restype = None
        L.mla_latent_attn_bwd.argtypes = [D, _i, _i, _i, _i, _i, _i, _i, _i, _i] + [_vp] * 15 + [_vp, _sz, _vp]
        L.mla_latent_attn_bwd.restype = _i
        L.mla_latent_attn_bwd_workspace.argtypes = [D, _i, _i, _i, _i, _i, _i, _i, _i]
        L.mla_latent_attn_bwd_workspace.restype = _sz
        L.mla_decode_splitkv.argtypes = [D, _i, _i, _i, _i] + [_vp] * 9 + [_vp, _sz, _vp]
        L.mla_decode_splitkv.restype = _i
        L.mla_decode_splitkv_noalloc.argtypes = [D, _i, _i, _i, _i] + [_vp] * 7 + [_vp]
        L.mla_decode_splitkv_noalloc.restype = _i
        L.mla_lse_combine.argtypes = [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]
        L.mla_lse_combine.restype = _i
        for f in ("mla_latent_attn_workspace", "mla_absorbed_attn_workspace"):
            getattr(L, f).argtypes = [D, _i, _i, _i, _i, _i, _i, _i, _i]
            getattr(L, f).restype = _sz
        L.mla_decode_workspace.argtypes = [D, _i, _i, _i, _i]
        L.mla_decode_workspace.restype = _sz
        L.mla_tpla_decode.argtypes = [D, _i, _i, _i, _i, _i] + [_vp] * 7 + [_vp, _sz, _vp]
        L.mla_tpla_decode.restype = _i
        L.mla_tpla_decode_workspace.argtypes = [D, _i, _i, _i, _i, _i]
        L.mla_tpla_decode_workspace.restype = _sz
        L.mla_rmsnorm.argtypes = [_i, ctypes.c_long, _i, _i, ctypes.c_float, _vp, _vp, _vp, _vp]
        L.mla_rmsnorm.restype = _i
        L.mla_rmsnorm_bwd.argtypes = [_i, ctypes.c_long, _i, _i, ctypes.c_float] + [_vp] * 6 + [_sz, _vp]
        L.mla_rmsnorm_bwd.restype = _i
        L.mla_rmsnorm_bwd_workspace.argtypes = [_i, ctypes.c_long, _i, _i]
        L.mla_rmsnorm_bwd_workspace.restype = _sz
        L.mla_status_string.argtypes = [_i]
        L.mla_status_string.restype = ctypes.c_char_p
        L.mla_check_device_error.argtypes = [_vp]
        L.mla_check_device_error.restype = _i
        L.mla_selftest_bounded_wait.argtypes = [ctypes.c_uint, _vp]
        L.mla_selftest_bounded_wait.restype = _i
        L.mla_last_path.argtypes = []
        L.mla_last_path.restype = _i
        L.mla_set_path_override.argtypes = [_i]
        L.mla_set_path_override.restype = None
        L.mla_launch_count.argtypes = []
        L.mla_launch_count.restype = ctypes.c_ulonglong
        L.mla_profile_enable.argtypes = [_i]
        L.mla_profile_enable.restype = None
        L.mla_profile_reset.argtypes = []
        L.mla_profile_reset.restype = None
        L.mla_profile_kernel.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_longlong),
                                         ctypes.POINTER(ctypes.c_double)]
        L.mla_profile_kernel.restype = _i
        _lib = L
    return _lib


# ------------------------------------------------------------ raw C entry points ----
def mla_latent_attn_fwd(*args) -> int:
    return lib().mla_latent_attn_fwd(*args)


def mla_absorbed_attn_fwd(*args) -> int:
    return lib().mla_absorbed_attn_fwd(*args)


def mla_latent_attn_fused_fwd(*args) -> int:
    return lib().mla_latent_attn_fused_fwd(*args)


def mla_latent_attn_fused_workspace(*args) -> int:
    return lib().mla_latent_attn_fused_workspace(*args)


def mla_latent_attn_bwd(*args) -> int:
    return lib().mla_latent_attn_bwd(*args)


def mla_latent_attn_bwd_workspace(*args) -> int:
    return lib().mla_latent_attn_bwd_workspace(*args)


def mla_decode_splitkv(*args) -> int:
    return lib().mla_decode_splitkv(*args)


def mla_decode_splitkv_noalloc(*args) -> int:
    return lib().mla_decode_splitkv_noalloc(*args)


NOALLOC_SCRATCH_BYTES = 64 << 20   # MLA_NOALLOC_SCRATCH_BYTES in include/mla.h


def mla_lse_combine(*args) -> int:
    return lib().mla_lse_combine(*args)


def mla_latent_attn_workspace(*args) -> int:
    return lib().mla_latent_attn_workspace(*args)


def mla_absorbed_attn_workspace(*args) -> int:
    return lib().mla_absorbed_attn_workspace(*args)


def mla_decode_workspace(*args) -> int:
    return lib().mla_decode_workspace(*args)


def mla_tpla_decode(*args) -> int:
    return lib().mla_tpla_decode(*args)


def mla_tpla_decode_workspace(*args) -> int:
    return lib().mla_tpla_decode_workspace(*args)


def mla_rmsnorm(*args) -> int:
    return lib().mla_rmsnorm(*args)


def mla_rmsnorm_bwd(*args) -> int:
    return lib().mla_rmsnorm_bwd(*args)


def mla_rmsnorm_bwd_workspace(*args) -> int:
    return lib().mla_rmsnorm_bwd_workspace(*args)


def mla_status_string(status: int) -> str:
    return lib().mla_status_string(status).decode()


def mla_check_device_error(stream: int | None = None) -> int:
    return lib().mla_check_device_error(stream)


def mla_selftest_bounded_wait(limit_us: int, stream: int | None = None) -> int:
    return lib().mla_selftest_bounded_wait(limit_us, stream)


def last_path() -> int:
    return lib().mla_last_path()


def set_path_override(mode: int) -> None:
    lib().mla_set_path_override(mode)


KERNELS = ("prep", "latent_prep", "rope_table", "rope_rows", "convert", "gemm_simt", "attn_simt", "lse_combine",
           "tc_gemm", "tc_attn", "tc_latent_attn", "tc_decode_attn", "transpose", "rmsnorm", "rmsnorm_bwd", "tpla_expand",
           "tpla_combine", "wait_probe", "tc_fused_attn", "bwd_rowdot", "attn_bwd_simt", "bwd_rows",
           "bwd_prep", "tc_bwd_dkv", "tc_bwd_dq")


def launch_count() -> int:
    return lib().mla_launch_count()


def profile_enable(on: bool) -> None:
    lib().mla_profile_enable(int(on))


def profile_reset() -> None:
    lib().mla_profile_reset()


def profile_kernel(name: str) -> tuple[int, float]:
    """(launches, summed device ms) recorded for kernel ``name`` while profiling was on."""
    n, ms = ctypes.c_longlong(0), ctypes.c_double(0.0)
    if lib().mla_profile_kernel(name.encode(), ctypes.byref(n), ctypes.byref(ms)) != 0:
        raise RuntimeError("mla_profile_kernel failed for " + name)
    return n.value, ms.value


def profile_all() -> dict:
    out = {}
    for k in KERNELS:
        n, ms = profile_kernel(k)
        if n:
            out[k] = (n, ms)
    return out


# ------------------------------------------------------------- tensor wrappers ----
def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MLA_F32
    if t.dtype == torch.bfloat16:
        return MLA_BF16
    raise TypeError("unsupported dtype %s" % t.dtype)


def _device(t: torch.Tensor) -> torch.device:
    """The call's device: that of its first tensor, which must be a CUDA device (the
    library's kernels dereference every pointer on the GPU)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor, got %s" % type(t).__name__)
    if t.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device, got %s" % t.device)
    return t.device


def _expect(name: str, t, numel: int, dtype: torch.dtype, device: torch.device) -> None:
    """Check one tensor argument before the call: the library reads or writes exactly
    ``numel`` elements of ``dtype`` behind its pointer on ``device``, so a tensor on
    another device, of another dtype or of another size would be misread or accessed
    out of bounds.  None passes (optional arguments)."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s: expected a torch.Tensor, got %s" % (name, type(t).__name__))
    if t.device != device:
        raise ValueError("%s: on %s, the call's tensors are on %s" % (name, t.device, device))
    if t.dtype != dtype:
        raise TypeError("%s: dtype %s, expected %s" % (name, t.dtype, dtype))
    if t.numel() != numel:
        raise ValueError("%s: %d elements, expected %d" % (name, t.numel(), numel))
    if not t.is_contiguous():
        raise ValueError("%s: tensors must be contiguous" % name)


def _prefill_checks(d, q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse):
    dev = _device(q_nope)
    _dt(q_nope)
    tdt = q_nope.dtype
    if q_nope.dim() != 4 or c_kv.dim() != 3:
        raise ValueError("q_nope must be [B, s_q, heads, d_nope] and c_kv [B, s_kv, d_kv]")
    B, s_q, hc, _ = q_nope.shape
    s_kv = c_kv.shape[1]
    _expect("q_nope", q_nope, B * s_q * hc * d.d_nope, tdt, dev)
    _expect("q_pe", q_pe, B * s_q * hc * d.d_rope, tdt, dev)
    _expect("c_kv", c_kv, B * s_kv * d.d_kv, tdt, dev)
    _expect("k_pe", k_pe, B * s_kv * d.d_rope, tdt, dev)
    _expect("w_kv_b", w_kv_b, d.n_heads * (d.d_nope + d.d_v) * d.d_kv, tdt, dev)
    _expect("rms_w", rms_w, d.d_kv, tdt, dev)
    _expect("out", out, B * s_q * hc * d.d_v, tdt, dev)
    _expect("lse", lse, B * hc * s_q, torch.float32, dev)
    return dev, B, s_q, hc, s_kv


def _decode_checks(d, q_nope, q_pe, c_cache, kpe_cache, w_kv_b, out):
    dev = _device(q_nope)
    _dt(q_nope)
    tdt = q_nope.dtype
    if q_nope.dim() != 3 or c_cache.dim() != 3:
        raise ValueError("q_nope must be [B, n_heads, d_nope] and c_cache [B, kv_len, d_kv]")
    B = q_nope.shape[0]
    L = c_cache.shape[1]
    H = d.n_heads
    _expect("q_nope", q_nope, B * H * d.d_nope, tdt, dev)
    _expect("q_pe", q_pe, B * H * d.d_rope, tdt, dev)
    _expect("c_cache", c_cache, B * L * d.d_kv, tdt, dev)
    _expect("kpe_cache", kpe_cache, B * L * d.d_rope, tdt, dev)
    _expect("w_kv_b", w_kv_b, H * (d.d_nope + d.d_v) * d.d_kv, tdt, dev)
    _expect("out", out, B * H * d.d_v, tdt, dev)
    return dev, B, L, H


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MlaError(status, where)


def _workspace(nbytes: int, device, workspace):
    if workspace is not None:
        if not isinstance(workspace, torch.Tensor) or workspace.device != device:
            raise ValueError("workspace: must be a tensor on %s" % device)
        return workspace
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def latent_attn_fwd(d: Dims, q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, *, q_offset=0, causal=True,
                    head_begin=0, head_shard=0, out=None, lse=None, workspace=None, stream=None,
                    absorbed=False):
    """Explicit (or, with ``absorbed=True``, absorbed) MLA prefill.  Returns (out, lse)."""
    _, B, s_q, hc, s_kv = _prefill_checks(d, q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse)
    dt = _dt(q_nope)
    if out is None:
        out = torch.empty(B, s_q, hc, d.d_v, dtype=q_nope.dtype, device=q_nope.device)
    if lse is None:
        lse = torch.empty(B, hc, s_q, dtype=torch.float32, device=q_nope.device)
    wsq = mla_absorbed_attn_workspace if absorbed else mla_latent_attn_workspace
    nbytes = wsq(ctypes.byref(d), dt, B, s_q, s_kv, q_offset, int(causal), hc, head_shard)
    ws = _workspace(nbytes, q_nope.device, workspace)
    fn = mla_absorbed_attn_fwd if absorbed else mla_latent_attn_fwd
    st = fn(ctypes.byref(d), dt, B, s_q, s_kv, q_offset, int(causal), head_begin, hc, head_shard,
            _ptr(q_nope), _ptr(q_pe), _ptr(c_kv), _ptr(k_pe), _ptr(w_kv_b), _ptr(rms_w), _ptr(out),
            _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, fn.__name__)
    return out, lse


def absorbed_attn_fwd(d: Dims, *args, **kw):
    return latent_attn_fwd(d, *args, absorbed=True, **kw)


def latent_attn_fused_fwd(d: Dims, q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, *, q_offset=0, causal=True,
                          head_begin=0, out=None, lse=None, workspace=None, stream=None):
    """Explicit MLA prefill with the K/V up-projection inside the attention kernel (no
    K/V workspace).  Returns (out, lse)."""
    _, B, s_q, hc, s_kv = _prefill_checks(d, q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse)
    dt = _dt(q_nope)
    if out is None:
        out = torch.empty(B, s_q, hc, d.d_v, dtype=q_nope.dtype, device=q_nope.device)
    if lse is None:
        lse = torch.empty(B, hc, s_q, dtype=torch.float32, device=q_nope.device)
    nbytes = mla_latent_attn_fused_workspace(ctypes.byref(d), dt, B, s_q, s_kv, q_offset, int(causal), hc)
    ws = _workspace(nbytes, q_nope.device, workspace)
    st = mla_latent_attn_fused_fwd(ctypes.byref(d), dt, B, s_q, s_kv, q_offset, int(causal), head_begin, hc,
                                   _ptr(q_nope), _ptr(q_pe), _ptr(c_kv), _ptr(k_pe), _ptr(w_kv_b), _ptr(rms_w),
                                   _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "mla_latent_attn_fused_fwd")
    return out, lse


def latent_attn_bwd(d: Dims, q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse, dout, *, q_offset=0, causal=True,
                    head_begin=0, head_shard=0, grads=None, workspace=None, stream=None):
    """Backward of :func:`latent_attn_fwd` for an upstream gradient ``dout`` of its output.
    Returns a dict of gradients: q_nope, q_pe, c_kv, k_pe (input dtype), w_kv_b, rms_w
    (fp32; w_kv_b rows outside the call's heads are zero when this call allocates it)."""
    dev, B, s_q, hc, s_kv = _prefill_checks(d, q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse)
    if out is None or lse is None:
        raise ValueError("the forward's out and lse are required")
    _expect("dout", dout, out.numel(), out.dtype, dev)
    dt = _dt(q_nope)
    g = grads or {}
    for k, like in (("q_nope", q_nope), ("q_pe", q_pe), ("c_kv", c_kv), ("k_pe", k_pe)):
        _expect("grads[%s]" % k, g.get(k), like.numel(), like.dtype, dev)
    _expect("grads[w_kv_b]", g.get("w_kv_b"), w_kv_b.numel(), torch.float32, dev)
    _expect("grads[rms_w]", g.get("rms_w"), rms_w.numel(), torch.float32, dev)
    g.setdefault("q_nope", torch.empty_like(q_nope))
    g.setdefault("q_pe", torch.empty_like(q_pe))
    g.setdefault("c_kv", torch.empty_like(c_kv))
    g.setdefault("k_pe", torch.empty_like(k_pe))
    g.setdefault("w_kv_b", torch.zeros(w_kv_b.shape, dtype=torch.float32, device=dev))
    g.setdefault("rms_w", torch.empty(rms_w.shape, dtype=torch.float32, device=dev))
    nbytes = mla_latent_attn_bwd_workspace(ctypes.byref(d), dt, B, s_q, s_kv, q_offset, int(causal), hc, head_shard)
    ws = _workspace(nbytes, dev, workspace)
    st = mla_latent_attn_bwd(ctypes.byref(d), dt, B, s_q, s_kv, q_offset, int(causal), head_begin, hc, head_shard,
                             _ptr(q_nope), _ptr(q_pe), _ptr(c_kv), _ptr(k_pe), _ptr(w_kv_b), _ptr(rms_w), _ptr(out),
                             _ptr(lse), _ptr(dout), _ptr(g["q_nope"]), _ptr(g["q_pe"]), _ptr(g["c_kv"]),
                             _ptr(g["k_pe"]), _ptr(g["w_kv_b"]), _ptr(g["rms_w"]), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "mla_latent_attn_bwd")
    return g


def set_fused_cluster(size: int) -> None:
    lib().mla_set_fused_cluster(size)


def decode_splitkv(d: Dims, q_nope, q_pe, c_cache, kpe_cache, w_kv_b, *, n_splits=1, out=None, lse=None,
                   part_out=None, part_lse=None, workspace=None, stream=None):
    """Split-KV latent decode.  Returns (out, lse)."""
    dev, B, L, H = _decode_checks(d, q_nope, q_pe, c_cache, kpe_cache, w_kv_b, out)
    _expect("lse", lse, B * H, torch.float32, dev)
    if (part_out is None) != (part_lse is None):
        raise ValueError("part_out and part_lse go together")
    _expect("part_out", part_out, n_splits * B * H * d.d_kv, torch.float32, dev)
    _expect("part_lse", part_lse, n_splits * B * H, torch.float32, dev)
    dt = _dt(q_nope)
    if out is None:
        out = torch.empty(B, H, d.d_v, dtype=q_nope.dtype, device=q_nope.device)
    if lse is None:
        lse = torch.empty(B, H, dtype=torch.float32, device=q_nope.device)
    nbytes = mla_decode_workspace(ctypes.byref(d), dt, B, L, n_splits)
    ws = _workspace(nbytes, q_nope.device, workspace)
    st = mla_decode_splitkv(ctypes.byref(d), dt, B, L, n_splits, _ptr(q_nope), _ptr(q_pe), _ptr(c_cache),
                            _ptr(kpe_cache), _ptr(w_kv_b), _ptr(out), _ptr(lse), _ptr(part_out),
                            _ptr(part_lse), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "mla_decode_splitkv")
    return out, lse


def tpla_decode(d: Dims, q_nope, q_pe, c_cache, kpe_cache, w_kv_b, *, n_shards=2, n_splits=1, out=None,
                shard_lse=None, workspace=None, stream=None):
    """TPLA decode over ``n_shards`` latent shards (``c_cache`` normalised per shard, as
    :func:`rmsnorm` with the same ``n_shards`` writes it).  Returns (out, shard_lse)."""
    dev, B, L, H = _decode_checks(d, q_nope, q_pe, c_cache, kpe_cache, w_kv_b, out)
    _expect("shard_lse", shard_lse, n_shards * B * H, torch.float32, dev)
    dt = _dt(q_nope)
    if out is None:
        out = torch.empty(B, H, d.d_v, dtype=q_nope.dtype, device=q_nope.device)
    if shard_lse is None:
        shard_lse = torch.empty(n_shards, B, H, dtype=torch.float32, device=q_nope.device)
    nbytes = mla_tpla_decode_workspace(ctypes.byref(d), dt, B, L, n_splits, n_shards)
    ws = _workspace(nbytes, q_nope.device, workspace)
    st = mla_tpla_decode(ctypes.byref(d), dt, B, L, n_splits, n_shards, _ptr(q_nope), _ptr(q_pe), _ptr(c_cache),
                         _ptr(kpe_cache), _ptr(w_kv_b), _ptr(out), _ptr(shard_lse), _ptr(ws),
                         ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "mla_tpla_decode")
    return out, shard_lse


def rmsnorm(x, w, *, n_shards=1, eps=1e-6, out=None, stream=None):
    """RMSNorm over the last dim of ``x``, cut into ``n_shards`` shards normalised on
    their own.  Returns ``out``."""
    dev = _device(x)
    _dt(x)
    d = x.shape[-1]
    _expect("x", x, x.numel(), x.dtype, dev)
    _expect("w", w, d, x.dtype, dev)
    _expect("out", out, x.numel(), x.dtype, dev)
    if out is None:
        out = torch.empty_like(x)
    st = mla_rmsnorm(_dt(x), x.numel() // d if d else 0, d, n_shards, float(eps), _ptr(x), _ptr(w), _ptr(out),
                     _stream(stream))
    _check(st, "mla_rmsnorm")
    return out


def rmsnorm_bwd(x, w, dy, *, n_shards=1, eps=1e-6, dx=None, dw=None, workspace=None, stream=None):
    """Backward of :func:`rmsnorm`.  Returns (dx like x, dw fp32 [d])."""
    dev = _device(x)
    _dt(x)
    d = x.shape[-1]
    _expect("x", x, x.numel(), x.dtype, dev)
    _expect("w", w, d, x.dtype, dev)
    _expect("dy", dy, x.numel(), x.dtype, dev)
    _expect("dx", dx, x.numel(), x.dtype, dev)
    _expect("dw", dw, d, torch.float32, dev)
    rows = x.numel() // d if d else 0
    dt = _dt(x)
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty(d, dtype=torch.float32, device=x.device)
    ws = _workspace(mla_rmsnorm_bwd_workspace(dt, rows, d, n_shards), x.device, workspace)
    st = mla_rmsnorm_bwd(dt, rows, d, n_shards, float(eps), _ptr(x), _ptr(w), _ptr(dy), _ptr(dx), _ptr(dw),
                         _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "mla_rmsnorm_bwd")
    return dx, dw


def lse_combine(part_out, part_lse, *, out_dtype=torch.float32, out=None, lse=None, stream=None):
    """Merge fp32 split partials [n, rows, D] / [n, rows].  Returns (out, lse)."""
    dev = _device(part_out)
    if part_out.dim() != 3:
        raise ValueError("part_out must be [n_splits, rows, D]")
    n, rows, D = part_out.shape
    _expect("part_out", part_out, n * rows * D, torch.float32, dev)
    _expect("part_lse", part_lse, n * rows, torch.float32, dev)
    if out is not None:
        _dt(out)
        _expect("out", out, rows * D, out.dtype, dev)
    _expect("lse", lse, rows, torch.float32, dev)
    if out is None:
        out = torch.empty(rows, D, dtype=out_dtype, device=part_out.device)
    if lse is None:
        lse = torch.empty(rows, dtype=torch.float32, device=part_out.device)
    st = mla_lse_combine(_dt(out), n, rows, D, _ptr(part_out), _ptr(part_lse), _ptr(out), _ptr(lse),
                         _stream(stream))
    _check(st, "mla_lse_combine")
    return out, lse
