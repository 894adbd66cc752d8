"""The allocation-free decode entry point (mla_decode_splitkv_noalloc).

Some callers cannot allocate device memory: code running while a stream is being
captured into a CUDA graph, where cudaMalloc is refused, or a plugin inside a host
runtime that owns all device memory through its own pool.  For them the library
keeps one fixed scratch array in device memory and offers a decode call that takes
no workspace.  This test calls it through the C ABI and checks it against the
ordinary mla_decode_splitkv (caller-provided workspace) within the parity
tolerances, on two calls in a row, so that a second call over the scratch the first
one left behind is covered too.  It also checks that a call too large for the fixed
scratch is refused.  The file name sorts last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes
import dataclasses

import pytest
import torch

from head_latent_attention_rmsnorm_gb300 import build as mla_build
from head_latent_attention_rmsnorm_gb300 import configs, inputs, mla

from parity import check_lse, check_out

pytestmark = pytest.mark.gpu


def _noalloc(d, dt, B, L, n, t, out, lse):
    return mla.mla_decode_splitkv_noalloc(ctypes.byref(d), dt, B, L, n, t["q_nope"].data_ptr(),
                                          t["q_pe"].data_ptr(), t["c_cache"].data_ptr(), t["kpe_cache"].data_ptr(),
                                          t["w_kv_b"].data_ptr(), out.data_ptr(), lse.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_decode_matches_workspace_decode(dtype):
    mla_build.build()
    if dtype == "bf16":
        cfg = dataclasses.replace(configs.DECODE, batch=4, kv_len=3000, n_splits=5)
    else:
        cfg = configs.Decode("dec_f32_small", "f32", batch=3, kv_len=777, n_splits=4, n_heads=8, d_kv=64,
                             d_nope=32, d_rope=16, d_v=32)
    d = mla.dims(cfg.n_heads, cfg.d_kv, cfg.d_nope, cfg.d_rope, cfg.d_v, cfg.rope_base)
    dt = mla.MLA_BF16 if dtype == "bf16" else mla.MLA_F32
    assert mla.mla_decode_workspace(ctypes.byref(d), dt, cfg.batch, cfg.kv_len, cfg.n_splits) <= \
        mla.NOALLOC_SCRATCH_BYTES
    t = {k: v.cuda() for k, v in inputs.decode_inputs(cfg).items()}
    ref_o, ref_l = mla.decode_splitkv(d, t["q_nope"], t["q_pe"], t["c_cache"], t["kpe_cache"], t["w_kv_b"],
                                      n_splits=cfg.n_splits)
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        st = _noalloc(d, dt, cfg.batch, cfg.kv_len, cfg.n_splits, t, out, lse)
        assert st == 0, mla.mla_status_string(st)
        torch.cuda.synchronize()
        check_out(out, ref_o.float(), cfg.torch_dtype, "noalloc out")
        check_lse(lse, ref_l, "noalloc lse")
    assert mla.mla_check_device_error(None) == 0


def test_noalloc_rejects_calls_beyond_the_fixed_scratch():
    mla_build.build()
    cfg = configs.DECODE       # 64 x 128 heads x 8 splits of fp32 partials: far above the fixed scratch
    d = mla.dims(cfg.n_heads, cfg.d_kv, cfg.d_nope, cfg.d_rope, cfg.d_v, cfg.rope_base)
    need = mla.mla_decode_workspace(ctypes.byref(d), mla.MLA_BF16, cfg.batch, cfg.kv_len, cfg.n_splits)
    assert need > mla.NOALLOC_SCRATCH_BYTES
    small = dataclasses.replace(cfg, batch=1, kv_len=16)
    t = {k: v.cuda() for k, v in inputs.decode_inputs(small).items()}
    out = torch.empty(cfg.batch, cfg.n_heads, cfg.d_v, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(cfg.batch, cfg.n_heads, device="cuda")
    # the size check comes before any pointer is used, so the small tensors never get read
    st = _noalloc(d, mla.MLA_BF16, cfg.batch, cfg.kv_len, cfg.n_splits, t, out, lse)
    assert st == -5, mla.mla_status_string(st)
