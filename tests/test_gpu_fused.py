"""GPU parity of the fused prefill (mla_latent_attn_fused_fwd): the K_nope / V
up-projection runs inside the attention kernel, rebuilt 64 keys at a time and shared
by a cluster of query tiles, with no K/V workspace.  Same contract and bars as the
two-kernel explicit path; checked against the oracle on ragged, non-causal, full-size
and simulated sequence-parallel cases, at both cluster sizes."""
import dataclasses

import pytest
import torch

from head_latent_attention_rmsnorm_gb300 import build as mla_build
from head_latent_attention_rmsnorm_gb300 import configs, inputs, mla

from parity import check_lse, check_out, np_inputs

pytestmark = pytest.mark.gpu

RAGGED = configs.Prefill("ragged_bf16", "bf16", batch=2, s_kv=300, s_q=200, q_offset=77, n_heads=8,
                         d_kv=512, d_nope=128, d_rope=64, d_v=128, head_shard=3)


@pytest.fixture(scope="module", autouse=True)
def built():
    mla_build.build()
    mla.lib()
    yield
    mla.set_fused_cluster(0)
    torch.cuda.synchronize()
    assert mla.mla_check_device_error(None) == 0


def dev(inp):
    return {k: v.cuda() for k, v in inp.items()}


def run_fused(cfg, inp, *, q_offset=None, head_begin=0, causal=None, cluster=0):
    mla.set_fused_cluster(cluster)
    try:
        out, lse = mla.latent_attn_fused_fwd(mla.dims_of(cfg), inp["q_nope"], inp["q_pe"], inp["c_kv"], inp["k_pe"],
                                             inp["w_kv_b"], inp["rms_w"],
                                             q_offset=cfg.q_offset if q_offset is None else q_offset,
                                             causal=cfg.causal if causal is None else causal, head_begin=head_begin)
        torch.cuda.synchronize()
        assert mla.last_path() == mla.PATH_TC_FUSED
    finally:
        mla.set_fused_cluster(0)
    return out, lse


def oracle_prefill(oracle, cfg, inp, *, q_offset=None, head_begin=0, causal=None):
    return oracle.mla_explicit(**np_inputs(inp), n_heads=cfg.n_heads,
                               q_offset=cfg.q_offset if q_offset is None else q_offset,
                               causal=cfg.causal if causal is None else causal, head_begin=head_begin,
                               base=cfg.rope_base, eps=cfg.rms_eps)


@pytest.mark.parametrize("cluster", [4, 8])
def test_fused_ragged(oracle, cluster):
    cfg = RAGGED
    inp = inputs.prefill_inputs(cfg)
    sub = dict(inp, q_nope=inp["q_nope"][:, :, 2:7].contiguous(), q_pe=inp["q_pe"][:, :, 2:7].contiguous())
    o, l = run_fused(cfg, dev(sub), head_begin=2, cluster=cluster)
    ro, rl = oracle_prefill(oracle, cfg, sub, head_begin=2)
    check_out(o, ro, torch.bfloat16, "fused ragged")
    check_lse(l, rl, "fused ragged lse")


@pytest.mark.parametrize("cluster", [4, 8])
def test_fused_noncausal(oracle, cluster):
    cfg = dataclasses.replace(RAGGED, s_kv=333, s_q=150, q_offset=3, causal=False, batch=1)
    inp = inputs.prefill_inputs(cfg)
    o, l = run_fused(cfg, dev(inp), cluster=cluster)
    ro, rl = oracle_prefill(oracle, cfg, inp)
    check_out(o, ro, torch.bfloat16)
    check_lse(l, rl)


def test_fused_noncausal_queries_past_keys(oracle):
    big = dataclasses.replace(RAGGED, s_kv=160, s_q=30, q_offset=120, causal=False, batch=2)
    inp = inputs.prefill_inputs(big)
    inp = dict(inp, c_kv=inp["c_kv"][:, :100].contiguous(), k_pe=inp["k_pe"][:, :100].contiguous())
    cfg = dataclasses.replace(big, s_kv=100)
    o, l = run_fused(cfg, dev(inp))
    ro, rl = oracle_prefill(oracle, cfg, inp)
    check_out(o, ro, torch.bfloat16)
    check_lse(l, rl)


def test_fused_matches_two_kernel_path():
    """Same call through the fused kernel and the two-kernel path (reconstruction GEMM +
    attention): the rebuilt K/V tiles and the online softmax agree to the bf16 bars."""
    cfg = dataclasses.replace(RAGGED, s_kv=1000, s_q=700, q_offset=300, batch=1, n_heads=4, head_shard=4)
    d_in = dev(inputs.prefill_inputs(cfg))
    of, lf = run_fused(cfg, d_in)
    o2, l2 = mla.latent_attn_fwd(mla.dims_of(cfg), d_in["q_nope"], d_in["q_pe"], d_in["c_kv"], d_in["k_pe"],
                                 d_in["w_kv_b"], d_in["rms_w"], q_offset=cfg.q_offset, head_shard=4)
    torch.cuda.synchronize()
    assert mla.last_path() == mla.PATH_TC
    check_out(of, o2.float(), torch.bfloat16, "fused vs two-kernel")
    check_lse(lf, l2)


def test_fused_v2lite_full(oracle):
    cfg = configs.V2LITE
    inp = inputs.prefill_inputs(cfg)
    o, l = run_fused(cfg, dev(inp))
    ro, rl = oracle_prefill(oracle, cfg, inp)
    check_out(o, ro, torch.bfloat16, "fused v2lite")
    check_lse(l, rl, "fused v2lite lse")


def test_fused_v3_sampled_heads(oracle):
    cfg = configs.V3
    inp = inputs.prefill_inputs(cfg)
    o, l = run_fused(cfg, dev(inp))
    for h0, hc in ((0, 1), (63, 2), (127, 1)):
        sub = dict(inp, q_nope=inp["q_nope"][:, :, h0:h0 + hc], q_pe=inp["q_pe"][:, :, h0:h0 + hc])
        ro, rl = oracle_prefill(oracle, cfg, sub, head_begin=h0)
        check_out(o[:, :, h0:h0 + hc], ro, torch.bfloat16, "fused v3 heads %d+%d" % (h0, hc))
        check_lse(l[:, h0:h0 + hc], rl)


def test_fused_sp8_ranks_concatenate_and_match_oracle(oracle):
    """All eight simulated ranks of the 16384-token sequence: each rank's call concatenates
    bit for bit to the single full call, and every rank's rows near a query-tile boundary
    match the oracle on sampled heads."""
    cfg = configs.SP8_RANK7
    S = cfg.s_kv
    full_in = dev(inputs.prefill_inputs(cfg, q_rows=(0, S)))
    full_o, full_l = run_fused(cfg, full_in, q_offset=0)
    outs, lses = [], []
    for off in cfg.sweep_offsets:
        sl = slice(off, off + cfg.s_q)
        rank_in = dict(full_in, q_nope=full_in["q_nope"][:, sl].contiguous(), q_pe=full_in["q_pe"][:, sl].contiguous())
        o, l = run_fused(cfg, rank_in, q_offset=off)
        outs.append(o)
        lses.append(l)
    assert torch.equal(torch.cat(outs, 1), full_o), "fused rank outputs do not concatenate to SP=1"
    assert torch.equal(torch.cat(lses, 2), full_l)
    for r, off in enumerate(cfg.sweep_offsets):
        k = 1 + (7 * r) % 15
        q0, n = off + 128 * k - 24, 48
        inp = inputs.prefill_inputs(cfg, q_rows=(q0, q0 + n))
        for h0 in sorted({(29 * r + dh) % cfg.n_heads for dh in (0, 64)}):
            sub = dict(inp, q_nope=inp["q_nope"][:, :, h0:h0 + 1], q_pe=inp["q_pe"][:, :, h0:h0 + 1])
            ro, rl = oracle_prefill(oracle, cfg, sub, q_offset=q0, head_begin=h0)
            i0 = q0 - off
            check_out(outs[r][:, i0:i0 + n, h0:h0 + 1], ro, torch.bfloat16, "fused rank %d head %d" % (r, h0))
            check_lse(lses[r][:, h0:h0 + 1, i0:i0 + n], rl, "fused rank %d lse" % r)


def test_fused_workspace_is_smaller_than_two_kernel():
    import ctypes
    for cfg in (configs.V2LITE, configs.V3, configs.SP8_RANK7):
        d = mla.dims_of(cfg)
        fused = mla.mla_latent_attn_fused_workspace(ctypes.byref(d), mla.MLA_BF16, cfg.batch, cfg.s_q, cfg.s_kv,
                                                    cfg.q_offset, 1, cfg.n_heads)
        two = mla.mla_latent_attn_workspace(ctypes.byref(d), mla.MLA_BF16, cfg.batch, cfg.s_q, cfg.s_kv,
                                            cfg.q_offset, 1, cfg.n_heads, cfg.head_shard)
        kv = cfg.batch * cfg.head_shard * ((cfg.kv_needed() + 127) // 128 * 128) * (cfg.d_nope + cfg.d_v) * 2
        assert 0 < fused and two - fused >= kv, (cfg.name, fused, two, kv)


def test_fused_unsupported_shapes_launch_nothing():
    cfg = configs.TINY   # fp32: no fused kernel
    inp = dev(inputs.prefill_inputs(cfg))
    with pytest.raises(mla.MlaError) as e:
        mla.latent_attn_fused_fwd(mla.dims_of(cfg), inp["q_nope"], inp["q_pe"], inp["c_kv"], inp["k_pe"],
                                  inp["w_kv_b"], inp["rms_w"])
    assert e.value.status == -6
