"""GPU parity of the backward pass (mla_latent_attn_bwd) against the oracle's gradients
(orc_mla_explicit_bwd, itself pinned to central finite differences of the pinned
forward).  The GPU backward takes the GPU forward's own out and lse, as a training step
would.  Bars: fp32 storage -> max |err| <= 1e-4 of each gradient; bf16 storage -> the
bf16 bars (max |err| <= 3e-2, relative L2 <= 1e-2) applied to each gradient scaled by
its largest magnitude, since weight and latent gradients are sums over many keys."""
import dataclasses

import numpy as np
import pytest
import torch

from head_latent_attention_rmsnorm_gb300 import build as mla_build
from head_latent_attention_rmsnorm_gb300 import configs, inputs, mla

from parity import np_inputs, to64

pytestmark = pytest.mark.gpu

DOUT_ID = 21   # stream id of the upstream gradient


@pytest.fixture(scope="module", autouse=True)
def built():
    mla_build.build()
    mla.lib()
    yield
    torch.cuda.synchronize()
    assert mla.mla_check_device_error(None) == 0


def dout_for(cfg, n_rows, hc, seed=7):
    a = inputs.normal_rows(seed, DOUT_ID, cfg.batch * n_rows, hc * cfg.d_v)
    return inputs.to_torch(a, cfg.torch_dtype, (cfg.batch, n_rows, hc, cfg.d_v))


def gpu_fwd_bwd(cfg, inp, dout, *, q_offset, causal, head_begin=0, head_shard=None):
    d = mla.dims_of(cfg)
    t = {k: v.cuda() for k, v in inp.items()}
    hs = cfg.head_shard if head_shard is None else head_shard
    out, lse = mla.latent_attn_fwd(d, t["q_nope"], t["q_pe"], t["c_kv"], t["k_pe"], t["w_kv_b"], t["rms_w"],
                                   q_offset=q_offset, causal=causal, head_begin=head_begin, head_shard=hs)
    g = mla.latent_attn_bwd(d, t["q_nope"], t["q_pe"], t["c_kv"], t["k_pe"], t["w_kv_b"], t["rms_w"], out, lse,
                            dout.cuda(), q_offset=q_offset, causal=causal, head_begin=head_begin, head_shard=hs)
    torch.cuda.synchronize()
    return {k: to64(v) for k, v in g.items()}


def oracle_bwd(oracle, cfg, inp, dout, *, q_offset, causal, head_begin=0):
    n = np_inputs(inp)
    return oracle.mla_explicit_bwd(n["q_nope"], n["q_pe"], n["c_kv"], n["k_pe"], n["w_kv_b"], n["rms_w"], to64(dout),
                                   n_heads=cfg.n_heads, q_offset=q_offset, causal=causal, head_begin=head_begin,
                                   base=cfg.rope_base, eps=cfg.rms_eps)


def check_grads(g, r, dtype, rows_w=None, what=""):
    for k in ("q_nope", "q_pe", "c_kv", "k_pe", "w_kv_b", "rms_w"):
        a, b = g[k], r[k]
        if k == "w_kv_b" and rows_w is not None:
            a, b = a[rows_w], b[rows_w]
        assert np.all(np.isfinite(a)), what + k
        err = np.abs(a - b).max()
        if dtype == torch.float32:
            assert err <= 1e-4, "%s%s: max abs err %.3e" % (what, k, err)
        else:
            scale = max(1.0, np.abs(b).max())
            rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
            assert err <= 3e-2 * scale, "%s%s: max abs err %.3e (scale %.2f)" % (what, k, err, scale)
            assert rel <= 1e-2, "%s%s: rel L2 %.3e" % (what, k, rel)


@pytest.mark.parametrize("q_offset,causal", [(0, True), (40, True), (40, False)])
def test_tiny_fp32_backward(oracle, q_offset, causal):
    cfg = configs.TINY
    s_q = cfg.s_kv - q_offset
    inp = inputs.prefill_inputs(cfg, q_rows=(q_offset, cfg.s_kv))
    dout = dout_for(cfg, s_q, cfg.n_heads)
    g = gpu_fwd_bwd(cfg, inp, dout, q_offset=q_offset, causal=causal)
    r = oracle_bwd(oracle, cfg, inp, dout, q_offset=q_offset, causal=causal)
    check_grads(g, r, torch.float32, what="tiny fp32 off %d causal %d: " % (q_offset, causal))


def test_tiny_fp32_backward_head_range(oracle):
    cfg = configs.TINY
    inp = inputs.prefill_inputs(cfg)
    sub = dict(inp, q_nope=inp["q_nope"][:, :, 1:3].contiguous(), q_pe=inp["q_pe"][:, :, 1:3].contiguous())
    dout = dout_for(cfg, cfg.s_q, 2)
    g = gpu_fwd_bwd(cfg, sub, dout, q_offset=0, causal=True, head_begin=1, head_shard=1)
    r = oracle_bwd(oracle, cfg, sub, dout, q_offset=0, causal=True, head_begin=1)
    rows = slice(1 * (cfg.d_nope + cfg.d_v), 3 * (cfg.d_nope + cfg.d_v))
    check_grads(g, r, torch.float32, rows_w=rows, what="head range: ")
    assert np.all(g["w_kv_b"][:rows.start] == 0) and np.all(g["w_kv_b"][rows.stop:] == 0)


def test_tiny_fp32_query_shards_sum_to_one_call():
    """Two query shards of one sequence: their parameter and latent gradients add up to
    those of the single call (LAGA page, "If this is right": the same gradients at any
    number of sequence-parallel ranks), and each shard's query gradients are the single
    call's rows."""
    cfg = configs.TINY
    S = cfg.s_kv
    full = inputs.prefill_inputs(cfg, q_rows=(0, S))
    dfull = dout_for(cfg, S, cfg.n_heads)
    g1 = gpu_fwd_bwd(cfg, full, dfull, q_offset=0, causal=True)
    parts = []
    for lo, hi in ((0, 64), (64, S)):
        sub = dict(full, q_nope=full["q_nope"][:, lo:hi].contiguous(), q_pe=full["q_pe"][:, lo:hi].contiguous())
        parts.append(gpu_fwd_bwd(cfg, sub, dfull[:, lo:hi].contiguous(), q_offset=lo, causal=True))
    for k in ("c_kv", "k_pe", "w_kv_b", "rms_w"):
        np.testing.assert_allclose(parts[0][k] + parts[1][k], g1[k], rtol=0, atol=1e-5 * max(1, np.abs(g1[k]).max()))
    for k in ("q_nope", "q_pe"):
        assert np.array_equal(np.concatenate([parts[0][k], parts[1][k]], 1), g1[k]), k


RAGGED = configs.Prefill("ragged_bf16", "bf16", batch=2, s_kv=300, s_q=200, q_offset=77, n_heads=8,
                         d_kv=512, d_nope=128, d_rope=64, d_v=128, head_shard=3)


@pytest.mark.parametrize("causal", [True, False])
def test_ragged_bf16_backward(oracle, causal):
    cfg = RAGGED
    inp = inputs.prefill_inputs(cfg)
    sub = dict(inp, q_nope=inp["q_nope"][:, :, 2:7].contiguous(), q_pe=inp["q_pe"][:, :, 2:7].contiguous())
    dout = dout_for(cfg, cfg.s_q, 5)
    g = gpu_fwd_bwd(cfg, sub, dout, q_offset=cfg.q_offset, causal=causal, head_begin=2)
    r = oracle_bwd(oracle, cfg, sub, dout, q_offset=cfg.q_offset, causal=causal, head_begin=2)
    rows = slice(2 * 256, 7 * 256)
    check_grads(g, r, torch.bfloat16, rows_w=rows, what="ragged bf16 causal %d: " % causal)
    if causal:   # keys past q_offset + s_q are seen by no query
        assert np.all(g["c_kv"][:, cfg.q_offset + cfg.s_q:] == 0) and np.all(g["k_pe"][:, cfg.q_offset + cfg.s_q:] == 0)


def test_bf16_backward_tensor_core_path_matches_simt_path():
    """The same bf16 backward through the tcgen05 kernels and through the CUDA-core
    kernels (forced): both within the bf16 bars of each other."""
    cfg = dataclasses.replace(RAGGED, s_kv=700, s_q=500, q_offset=200, batch=1, n_heads=4, head_shard=4)
    inp = inputs.prefill_inputs(cfg)
    dout = dout_for(cfg, cfg.s_q, cfg.n_heads)
    g_tc = gpu_fwd_bwd(cfg, inp, dout, q_offset=cfg.q_offset, causal=True)
    assert mla.last_path() == mla.PATH_TC
    mla.set_path_override(1)
    try:
        g_s = gpu_fwd_bwd(cfg, inp, dout, q_offset=cfg.q_offset, causal=True)
        assert mla.last_path() == mla.PATH_SIMT
    finally:
        mla.set_path_override(0)
    check_grads(g_tc, g_s, torch.bfloat16, what="tc vs simt: ")


def test_bf16_backward_query_shards_sum_to_one_call():
    """Two query shards of one bf16 sequence on the tensor-core path: the latent, band and
    parameter gradients of the shards add up to the single call's (within fp32 rounding of
    the different summation order), the shards' query gradients are its rows."""
    cfg = dataclasses.replace(RAGGED, s_kv=512, s_q=512, q_offset=0, batch=1, n_heads=2, head_shard=2)
    S = cfg.s_kv
    full = inputs.prefill_inputs(cfg, q_rows=(0, S))
    dfull = dout_for(cfg, S, cfg.n_heads)
    g1 = gpu_fwd_bwd(cfg, full, dfull, q_offset=0, causal=True)
    parts = []
    for lo, hi in ((0, 256), (256, S)):
        sub = dict(full, q_nope=full["q_nope"][:, lo:hi].contiguous(), q_pe=full["q_pe"][:, lo:hi].contiguous())
        parts.append(gpu_fwd_bwd(cfg, sub, dfull[:, lo:hi].contiguous(), q_offset=lo, causal=True))
    for k in ("w_kv_b", "rms_w"):
        np.testing.assert_allclose(parts[0][k] + parts[1][k], g1[k], rtol=0, atol=2e-3 * max(1, np.abs(g1[k]).max()))
    for k in ("c_kv", "k_pe"):   # bf16 outputs: each side rounded once
        np.testing.assert_allclose(parts[0][k] + parts[1][k], g1[k], rtol=0, atol=2e-2 * max(1, np.abs(g1[k]).max()))
    for k in ("q_nope", "q_pe"):
        assert np.array_equal(np.concatenate([parts[0][k], parts[1][k]], 1), g1[k]), k


def test_v2lite_backward_sampled_against_simt():
    """The bench's backward workload size (V2-Lite prefill, 4096 tokens, 16 heads) on the
    tensor cores against the CUDA-core backward on two heads."""
    cfg = configs.V2LITE
    inp = inputs.prefill_inputs(cfg)
    sub = dict(inp, q_nope=inp["q_nope"][:, :, 5:7].contiguous(), q_pe=inp["q_pe"][:, :, 5:7].contiguous())
    dout = dout_for(cfg, cfg.s_q, 2)
    g_tc = gpu_fwd_bwd(cfg, sub, dout, q_offset=0, causal=True, head_begin=5, head_shard=2)
    assert mla.last_path() == mla.PATH_TC
    mla.set_path_override(1)
    try:
        g_s = gpu_fwd_bwd(cfg, sub, dout, q_offset=0, causal=True, head_begin=5, head_shard=2)
    finally:
        mla.set_path_override(0)
    rows = slice(5 * 256, 7 * 256)
    check_grads(g_tc, g_s, torch.bfloat16, rows_w=rows, what="v2lite tc vs simt: ")
