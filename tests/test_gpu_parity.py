"""GPU parity: the CUDA path through the C ABI against the oracle on the same
seeded inputs, element by element, plus GPU-side invariants (query-shard and
head-range concatenation, split counts, explicit vs absorbed)."""
import dataclasses

import numpy as np
import pytest
import torch

from head_latent_attention_rmsnorm_gb300 import build as mla_build
from head_latent_attention_rmsnorm_gb300 import configs, inputs, mla

from parity import check_lse, check_out, np_inputs, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    mla_build.build()
    mla.lib()
    yield
    torch.cuda.synchronize()
    assert mla.mla_check_device_error(None) == 0


def dev(inp):
    return {k: v.cuda() for k, v in inp.items()}


def run_prefill(cfg, inp, *, absorbed=False, q_offset=None, head_begin=0, head_shard=None, causal=None):
    d = mla.dims_of(cfg)
    q_offset = cfg.q_offset if q_offset is None else q_offset
    causal = cfg.causal if causal is None else causal
    hs = cfg.head_shard if head_shard is None else head_shard
    out, lse = mla.latent_attn_fwd(d, inp["q_nope"], inp["q_pe"], inp["c_kv"], inp["k_pe"], inp["w_kv_b"],
                                   inp["rms_w"], q_offset=q_offset, causal=causal, head_begin=head_begin,
                                   head_shard=hs, absorbed=absorbed)
    torch.cuda.synchronize()
    return out, lse


def oracle_prefill(oracle, cfg, inp, *, absorbed=False, q_offset=None, head_begin=0, causal=None):
    fn = oracle.mla_absorbed if absorbed else oracle.mla_explicit
    n = np_inputs(inp)
    return fn(**n, n_heads=cfg.n_heads, q_offset=cfg.q_offset if q_offset is None else q_offset,
              causal=cfg.causal if causal is None else causal, head_begin=head_begin, base=cfg.rope_base,
              eps=cfg.rms_eps)


# ------------------------------------------------------------------- tiny fp32 ----
@pytest.mark.parametrize("absorbed", [False, True])
def test_tiny_fp32_full(oracle, absorbed):
    cfg = configs.TINY
    inp = inputs.prefill_inputs(cfg)
    out, lse = run_prefill(cfg, dev(inp), absorbed=absorbed)
    ro, rl = oracle_prefill(oracle, cfg, inp, absorbed=absorbed)
    check_out(out, ro, torch.float32)
    check_lse(lse, rl)


def test_tiny_fp32_matches_golden_rows():
    import os
    cfg = configs.TINY
    out, lse = run_prefill(cfg, dev(inputs.prefill_inputs(cfg)))
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_fp32_oracle_rows.txt")
    for line in open(path):
        if line.startswith("#"):
            continue
        f = line.split()
        i, h = int(f[0]), int(f[1])
        assert abs(lse[0, h, i].item() - float(f[2])) <= 1e-3
        np.testing.assert_allclose(to64(out[0, i, h, :8]), [float(x) for x in f[3:]], rtol=0, atol=1e-4)


@pytest.mark.parametrize("absorbed", [False, True])
def test_tiny_fp32_sp_shards(oracle, absorbed):
    cfg = configs.TINY
    full_in = inputs.prefill_inputs(cfg, q_rows=(0, cfg.s_kv))
    full_o, full_l = run_prefill(cfg, dev(full_in), absorbed=absorbed, q_offset=0)
    parts_o, parts_l = [], []
    for off in cfg.sweep_offsets:
        rows = (off, off + cfg.s_kv // len(cfg.sweep_offsets))
        inp = inputs.prefill_inputs(cfg, q_rows=rows)
        o, l = run_prefill(cfg, dev(inp), absorbed=absorbed, q_offset=off)
        ro, rl = oracle_prefill(oracle, cfg, inp, absorbed=absorbed, q_offset=off)
        check_out(o, ro, torch.float32, "shard@%d" % off)
        check_lse(l, rl, "shard lse@%d" % off)
        parts_o.append(o)
        parts_l.append(l)
    assert torch.equal(torch.cat(parts_o, 1), full_o)
    assert torch.equal(torch.cat(parts_l, 2), full_l)


def test_tiny_fp32_head_range_noncausal(oracle):
    cfg = configs.TINY
    inp = inputs.prefill_inputs(cfg)
    sub = dict(inp, q_nope=inp["q_nope"][:, :, 1:3].contiguous(), q_pe=inp["q_pe"][:, :, 1:3].contiguous())
    for causal in (True, False):
        o, l = run_prefill(cfg, dev(sub), head_begin=1, head_shard=1, causal=causal)
        ro, rl = oracle_prefill(oracle, cfg, sub, head_begin=1, causal=causal)
        check_out(o, ro, torch.float32)
        check_lse(l, rl)


# --------------------------------------------------------------- ragged bf16 ----
RAGGED = configs.Prefill("ragged_bf16", "bf16", batch=2, s_kv=300, s_q=200, q_offset=77, n_heads=8,
                         d_kv=512, d_nope=128, d_rope=64, d_v=128, head_shard=3)


@pytest.mark.parametrize("absorbed", [False, True])
def test_ragged_bf16(oracle, absorbed):
    cfg = RAGGED
    inp = inputs.prefill_inputs(cfg)
    sub = dict(inp, q_nope=inp["q_nope"][:, :, 2:7].contiguous(), q_pe=inp["q_pe"][:, :, 2:7].contiguous())
    o, l = run_prefill(cfg, dev(sub), absorbed=absorbed, head_begin=2)
    assert mla.last_path() == mla.PATH_TC
    ro, rl = oracle_prefill(oracle, cfg, sub, absorbed=absorbed, head_begin=2)
    check_out(o, ro, torch.bfloat16)
    check_lse(l, rl)


def test_ragged_bf16_noncausal_small_kv(oracle):
    cfg = dataclasses.replace(RAGGED, s_kv=37, s_q=30, q_offset=3, causal=False, batch=1)
    inp = inputs.prefill_inputs(cfg)
    o, l = run_prefill(cfg, dev(inp))
    ro, rl = oracle_prefill(oracle, cfg, inp)
    check_out(o, ro, torch.bfloat16)
    check_lse(l, rl)


@pytest.mark.parametrize("absorbed", [False, True])
def test_ragged_bf16_noncausal_queries_past_keys(oracle, absorbed):
    """Non-causal: 100 keys, queries at positions 120..149, i.e. past the keys and past
    the 128-row key padding (their RoPE angles come from positions no key has)."""
    big = dataclasses.replace(RAGGED, s_kv=160, s_q=30, q_offset=120, causal=False, batch=2)
    inp = inputs.prefill_inputs(big)
    inp = dict(inp, c_kv=inp["c_kv"][:, :100].contiguous(), k_pe=inp["k_pe"][:, :100].contiguous())
    cfg = dataclasses.replace(big, s_kv=100)
    o, l = run_prefill(cfg, dev(inp), absorbed=absorbed)
    ro, rl = oracle_prefill(oracle, cfg, inp, absorbed=absorbed)
    check_out(o, ro, torch.bfloat16)
    check_lse(l, rl)


# --------------------------------------------------------- full-size prefill ----
def test_v2lite_full(oracle):
    cfg = configs.V2LITE
    inp = inputs.prefill_inputs(cfg)
    o, l = run_prefill(cfg, dev(inp))
    ro, rl = oracle_prefill(oracle, cfg, inp)
    check_out(o, ro, torch.bfloat16)
    check_lse(l, rl)


def test_v3_sampled_heads_and_absorbed(oracle):
    cfg = configs.V3
    inp = inputs.prefill_inputs(cfg)
    d_in = dev(inp)
    o, l = run_prefill(cfg, d_in)
    assert mla.last_path() == mla.PATH_TC
    oa, la = run_prefill(cfg, d_in, absorbed=True)
    assert mla.last_path() == mla.PATH_TC
    # the sampled heads of both forms against the oracle (its explicit and absorbed forms
    # agree to 1e-10 in fp64: tests/test_oracle_pins.py), plus the whole of both outputs
    # against each other
    for h0, hc in ((0, 2), (77, 1), (127, 1)):
        sub = dict(inp, q_nope=inp["q_nope"][:, :, h0:h0 + hc], q_pe=inp["q_pe"][:, :, h0:h0 + hc])
        ro, rl = oracle_prefill(oracle, cfg, sub, head_begin=h0)
        check_out(o[:, :, h0:h0 + hc], ro, torch.bfloat16, "v3 heads %d+%d" % (h0, hc))
        check_lse(l[:, h0:h0 + hc], rl)
        check_out(oa[:, :, h0:h0 + hc], ro, torch.bfloat16, "v3 absorbed heads %d+%d" % (h0, hc))
        check_lse(la[:, h0:h0 + hc], rl, "v3 absorbed lse")
    check_out(oa, o.float(), torch.bfloat16, "absorbed vs explicit")
    check_lse(la, l)


def test_v3_absorbed_sampled_rows_against_absorbed_oracle(oracle):
    """The absorbed V3 call's rows near the causal diagonal and at the end of the
    sequence, two heads, against the oracle's own absorbed form."""
    cfg = configs.V3
    d_in = dev(inputs.prefill_inputs(cfg))
    oa, la = run_prefill(cfg, d_in, absorbed=True)
    assert mla.last_path() == mla.PATH_TC
    for q0, n, h0 in ((100, 56, 5), (cfg.s_kv - 40, 40, 126)):
        inp = inputs.prefill_inputs(cfg, q_rows=(q0, q0 + n))
        sub = dict(inp, q_nope=inp["q_nope"][:, :, h0:h0 + 1], q_pe=inp["q_pe"][:, :, h0:h0 + 1])
        ro, rl = oracle_prefill(oracle, cfg, sub, absorbed=True, q_offset=q0, head_begin=h0)
        check_out(oa[:, q0:q0 + n, h0:h0 + 1], ro, torch.bfloat16, "absorbed rows %d head %d" % (q0, h0))
        check_lse(la[:, h0:h0 + 1, q0:q0 + n], rl, "absorbed lse rows %d head %d" % (q0, h0))


def test_v3_activation_memory_explicit_below_absorbed():
    """LAGA, "What carries the argument": the explicit form's per-token intermediates
    (n_h x (d_nope + d_v)) are smaller than the absorbed form's (n_h x d_kv)."""
    cfg = configs.V3
    d_in = dev(inputs.prefill_inputs(cfg))
    peaks = {}
    for absorbed in (False, True):
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        run_prefill(cfg, d_in, absorbed=absorbed, head_shard=cfg.n_heads)
        peaks[absorbed] = torch.cuda.max_memory_allocated() - base
    assert peaks[False] < peaks[True]


def test_sp8_rank_sweep_concatenates_and_matches_oracle(oracle):
    cfg = configs.SP8_RANK7
    S = cfg.s_kv
    full_in = dev(inputs.prefill_inputs(cfg, q_rows=(0, S)))
    full_o, full_l = run_prefill(cfg, full_in, q_offset=0)
    outs, lses = [], []
    for off in cfg.sweep_offsets:
        sl = slice(off, off + cfg.s_q)
        rank_in = dict(full_in, q_nope=full_in["q_nope"][:, sl].contiguous(),
                       q_pe=full_in["q_pe"][:, sl].contiguous())
        o, l = run_prefill(cfg, rank_in, q_offset=off)
        outs.append(o)
        lses.append(l)
    assert torch.equal(torch.cat(outs, 1), full_o), "rank outputs do not concatenate to SP=1"
    assert torch.equal(torch.cat(lses, 2), full_l)
    # every rank against the oracle: 64 rows straddling the boundary between two of the
    # rank's 128-row query tiles (so both tiles' diagonal key tiles are in play), four
    # heads spread over the head shards
    for r, off in enumerate(cfg.sweep_offsets):
        k = 1 + (5 * r) % 15
        q0, n = off + 128 * k - 32, 64
        heads = sorted({(37 * r + dh) % cfg.n_heads for dh in (0, 41, 83, 127)})
        inp = inputs.prefill_inputs(cfg, q_rows=(q0, q0 + n))
        for h0 in heads:
            sub = dict(inp, q_nope=inp["q_nope"][:, :, h0:h0 + 1], q_pe=inp["q_pe"][:, :, h0:h0 + 1])
            ro, rl = oracle_prefill(oracle, cfg, sub, q_offset=q0, head_begin=h0)
            i0 = q0 - off
            check_out(outs[r][:, i0:i0 + n, h0:h0 + 1], ro, torch.bfloat16, "rank %d rows %d head %d" % (r, q0, h0))
            check_lse(lses[r][:, h0:h0 + 1, i0:i0 + n], rl, "rank %d lse rows %d head %d" % (r, q0, h0))
    # and sampled rows/heads of the last rank (query offset 14336), its end included
    rank7 = outs[-1]
    for q0, h0 in ((cfg.q_offset, 0), (cfg.q_offset + 1000, 64), (S - 48, 127)):
        n = 48
        inp = inputs.prefill_inputs(cfg, q_rows=(q0, q0 + n))
        sub = dict(inp, q_nope=inp["q_nope"][:, :, h0:h0 + 1], q_pe=inp["q_pe"][:, :, h0:h0 + 1])
        ro, rl = oracle_prefill(oracle, cfg, sub, q_offset=q0, head_begin=h0)
        i0 = q0 - cfg.q_offset
        check_out(rank7[:, i0:i0 + n, h0:h0 + 1], ro, torch.bfloat16, "rank7 rows %d head %d" % (q0, h0))
        check_lse(lses[-1][:, h0:h0 + 1, i0:i0 + n], rl)


@pytest.mark.parametrize("causal", [True, False])
def test_long_keys_rows_and_tail_tile(oracle, causal):
    """30000 keys (235 key tiles per (query tile, head) unit, a ragged last tile): sampled
    rows against the oracle, causal at the end of the sequence and non-causal, and the last
    query tile computed alone comes out bit-identical to the same tile of a longer call."""
    s_kv, s_q = 30000, 384
    q_off = s_kv - s_q if causal else 0
    cfg = dataclasses.replace(configs.V2LITE, name="cut3", s_kv=s_kv, s_q=s_q, q_offset=q_off, causal=causal)
    full_in = dev(inputs.prefill_inputs(cfg))
    out, lse = run_prefill(cfg, full_in)
    tail = dict(full_in, q_nope=full_in["q_nope"][:, 256:].contiguous(), q_pe=full_in["q_pe"][:, 256:].contiguous())
    o2, l2 = run_prefill(dataclasses.replace(cfg, s_q=128), tail, q_offset=q_off + 256)
    assert torch.equal(o2, out[:, 256:]) and torch.equal(l2, lse[:, :, 256:])
    for q0, h0 in ((0, 3), (200, 9), (s_q - 40, 15)):
        n = 40
        inp = inputs.prefill_inputs(cfg, q_rows=(q_off + q0, q_off + q0 + n))
        sub = dict(inp, q_nope=inp["q_nope"][:, :, h0:h0 + 1], q_pe=inp["q_pe"][:, :, h0:h0 + 1])
        ro, rl = oracle_prefill(oracle, cfg, sub, q_offset=q_off + q0, head_begin=h0)
        check_out(out[:, q0:q0 + n, h0:h0 + 1], ro, torch.bfloat16, "rows %d head %d" % (q0, h0))
        check_lse(lse[:, h0:h0 + 1, q0:q0 + n], rl, "lse rows %d head %d" % (q0, h0))


# ------------------------------------------------------------------- decode ----
def run_decode(cfg, inp, n_splits, partials=True):
    d = mla.dims(cfg.n_heads, cfg.d_kv, cfg.d_nope, cfg.d_rope, cfg.d_v, cfg.rope_base)
    B, H = cfg.batch, cfg.n_heads
    po = torch.empty(n_splits, B, H, cfg.d_kv, device="cuda") if partials else None
    pl = torch.empty(n_splits, B, H, device="cuda") if partials else None
    o, l = mla.decode_splitkv(d, inp["q_nope"], inp["q_pe"], inp["c_cache"], inp["kpe_cache"], inp["w_kv_b"],
                              n_splits=n_splits, part_out=po, part_lse=pl)
    torch.cuda.synchronize()
    return o, l, po, pl


def test_decode_full_size(oracle):
    cfg = configs.DECODE
    inp = inputs.decode_inputs(cfg)
    o, l, po, pl = run_decode(cfg, dev(inp), cfg.n_splits)
    for b in (0, 37, 63):
        sub = inputs.decode_inputs(cfg, batches=(b, b + 1))
        n = np_inputs(sub)
        ro, rl, rpo, rpl = oracle.mla_decode(**n, n_splits=cfg.n_splits, base=cfg.rope_base)
        check_out(o[b:b + 1], ro, torch.bfloat16, "decode out b=%d" % b)
        check_lse(l[b:b + 1], rl, "decode lse b=%d" % b)
        check_out(po[:, b:b + 1], rpo, torch.bfloat16, "partials b=%d" % b)
        check_lse(pl[:, b:b + 1], rpl, "partial lse b=%d" % b)


@pytest.mark.parametrize("dtype,L,n_splits", [
    ("bf16", 1000, 1), ("bf16", 1000, 2), ("bf16", 1000, 8), ("bf16", 1000, 13), ("bf16", 5, 8),
    ("bf16", 1, 1), ("bf16", 5000, 40), ("f32", 333, 13), ("f32", 64, 3)])
def test_decode_splits(oracle, dtype, L, n_splits):
    if dtype == "bf16":
        cfg = dataclasses.replace(configs.DECODE, batch=3, kv_len=L, n_splits=n_splits)
    else:
        cfg = configs.Decode("dec_f32", "f32", batch=2, kv_len=L, n_splits=n_splits, n_heads=4, d_kv=64,
                             d_nope=32, d_rope=16, d_v=32)
    inp = inputs.decode_inputs(cfg)
    o, l, po, pl = run_decode(cfg, dev(inp), n_splits)
    ro, rl, rpo, rpl = oracle.mla_decode(**np_inputs(inp), n_splits=n_splits, base=cfg.rope_base)
    check_out(o, ro, cfg.torch_dtype)
    check_lse(l, rl)
    check_out(po, rpo, cfg.torch_dtype, "partials")
    check_lse(pl, rpl, "partial lse")
    o2, l2, _, _ = run_decode(cfg, dev(inp), n_splits, partials=False)
    assert torch.equal(o2, o) and torch.equal(l2, l)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_lse_combine(oracle, out_dtype):
    g = np.random.default_rng(5)
    n, rows, D = 7, 300, 136
    po = g.standard_normal((n, rows, D)).astype(np.float32)
    pl = (4 * g.standard_normal((n, rows))).astype(np.float32)
    pl[3, :40] = -np.inf
    pl[:, 7] = -np.inf                       # a row with no keys at all
    po[:, 7] = 0
    o, l = mla.lse_combine(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), out_dtype=out_dtype)
    torch.cuda.synchronize()
    ro, rl = oracle.lse_combine(po, pl)
    check_out(o, ro, out_dtype)
    check_lse(l, rl)


def test_empty_calls_are_noops():
    cfg = configs.TINY
    inp = dev(inputs.prefill_inputs(cfg))
    d = mla.dims_of(cfg)
    z = {k: (v[:, :0] if k in ("q_nope", "q_pe") else v) for k, v in inp.items()}
    o, l = mla.latent_attn_fwd(d, z["q_nope"], z["q_pe"], z["c_kv"], z["k_pe"], z["w_kv_b"], z["rms_w"])
    assert o.shape[1] == 0 and l.shape[2] == 0


# ------------------------------------------------- tensor cores vs CUDA cores ----
@pytest.mark.parametrize("absorbed", [False, True])
def test_tensor_core_path_matches_simt_path(absorbed):
    """Same bf16 call through both kernel families (the SIMT one forced)."""
    cfg = dataclasses.replace(RAGGED, s_kv=700, s_q=500, q_offset=200, batch=1, head_shard=4)
    d_in = dev(inputs.prefill_inputs(cfg))
    o_tc, l_tc = run_prefill(cfg, d_in, absorbed=absorbed)
    path_tc = mla.last_path()
    assert path_tc == mla.PATH_TC
    mla.set_path_override(1)
    try:
        o_s, l_s = run_prefill(cfg, d_in, absorbed=absorbed)
        assert mla.last_path() == mla.PATH_SIMT
    finally:
        mla.set_path_override(0)
    check_out(o_tc, o_s.float(), torch.bfloat16, "tc vs simt (path %d)" % path_tc)
    check_lse(l_tc, l_s)


def test_explicit_bf16_uses_tensor_cores():
    cfg = dataclasses.replace(RAGGED, batch=1)
    d_in = dev(inputs.prefill_inputs(cfg))
    run_prefill(cfg, d_in)
    assert mla.last_path() == mla.PATH_TC


def test_decode_tensor_core_path_matches_simt_path():
    cfg = dataclasses.replace(configs.DECODE, batch=2, kv_len=2500, n_splits=3)
    inp = dev(inputs.decode_inputs(cfg))
    o_tc, l_tc, po_tc, pl_tc = run_decode(cfg, inp, cfg.n_splits)
    assert mla.last_path() == mla.PATH_TC
    mla.set_path_override(1)
    try:
        o_s, l_s, po_s, pl_s = run_decode(cfg, inp, cfg.n_splits)
        assert mla.last_path() == mla.PATH_SIMT
    finally:
        mla.set_path_override(0)
    check_out(o_tc, o_s.float(), torch.bfloat16, "decode tc vs simt")
    check_lse(l_tc, l_s)
    check_out(po_tc, po_s, torch.bfloat16, "partials tc vs simt")
    check_lse(pl_tc, pl_s)


# --------------------------------------------------------------------- TPLA ----
def tpla_cfg(dtype, L, n_splits, n_heads=None):
    if dtype == "bf16":
        return dataclasses.replace(configs.DECODE, batch=3, kv_len=L, n_splits=n_splits,
                                   n_heads=n_heads or configs.DECODE.n_heads)
    return configs.Decode("dec_f32", "f32", batch=2, kv_len=L, n_splits=n_splits, n_heads=n_heads or 4, d_kv=64,
                          d_nope=32, d_rope=16, d_v=32)


def run_tpla(cfg, d_inp, g, cache=None):
    d = mla.dims(cfg.n_heads, cfg.d_kv, cfg.d_nope, cfg.d_rope, cfg.d_v, cfg.rope_base)
    cache = d_inp["c_cache"] if cache is None else cache
    o, sl = mla.tpla_decode(d, d_inp["q_nope"], d_inp["q_pe"], cache, d_inp["kpe_cache"], d_inp["w_kv_b"],
                            n_shards=g, n_splits=cfg.n_splits)
    torch.cuda.synchronize()
    return o, sl


@pytest.mark.parametrize("dtype,L,n_splits,g,heads", [
    ("bf16", 1000, 1, 2, None), ("bf16", 1000, 8, 2, None), ("bf16", 1000, 13, 4, None),
    ("bf16", 5, 8, 2, None), ("bf16", 1, 1, 2, None), ("bf16", 777, 4, 2, 64),
    ("f32", 333, 13, 2, None), ("f32", 64, 3, 4, None), ("f32", 50, 2, 2, 3)])
def test_tpla_decode(oracle, dtype, L, n_splits, g, heads):
    """Decode over a cache normalised shard by shard (the call's contract): the same
    seeded cache values go to both sides."""
    cfg = tpla_cfg(dtype, L, n_splits, heads)
    inp = inputs.decode_inputs(cfg)
    o, sl = run_tpla(cfg, dev(inp), g)
    if dtype == "bf16":
        assert mla.last_path() == mla.PATH_TC
    n = np_inputs(inp)
    ro, rsl = oracle.tpla_decode(n["q_nope"], n["q_pe"], n["c_cache"], n["kpe_cache"], n["w_kv_b"], None,
                                 shards=g, base=cfg.rope_base)
    check_out(o, ro, cfg.torch_dtype, "tpla out")
    check_lse(sl, rsl, "tpla shard lse")


def test_tpla_one_shard_is_plain_decode():
    cfg = tpla_cfg("bf16", 1000, 8)
    inp = dev(inputs.decode_inputs(cfg))
    o1, sl = run_tpla(cfg, inp, 1)
    o, l, _, _ = run_decode(cfg, inp, cfg.n_splits, partials=False)
    assert torch.equal(o1, o) and torch.equal(sl[0], l)


def test_tpla_shard_decodes_sum_to_the_two_shard_decode():
    """What two tensor-parallel ranks would each compute and then all-reduce: each latent
    shard decoded on its own by the product call (a one-shard TPLA decode over the shard's
    latent columns and the matching W_kv_b columns, the RoPE band whole), the two outputs
    added, equals the two-shard TPLA decode; each shard's LSE is its shard LSE."""
    cfg = tpla_cfg("bf16", 1000, 4)
    inp = dev(inputs.decode_inputs(cfg))
    o2, sl2 = run_tpla(cfg, inp, 2)
    ds = cfg.d_kv // 2
    scfg = dataclasses.replace(cfg, d_kv=ds)
    total = torch.zeros_like(o2, dtype=torch.float32)
    for i in range(2):
        sub = dict(inp, c_cache=inp["c_cache"][..., i * ds:(i + 1) * ds].contiguous(),
                   w_kv_b=inp["w_kv_b"][:, i * ds:(i + 1) * ds].contiguous())
        o, sl = run_tpla(scfg, sub, 1)
        total += o.float()
        check_lse(sl[0], sl2[i], "shard %d lse" % i)
    check_out(o2, total, torch.bfloat16, "sum of shard decodes")


def test_tpla_tensor_core_path_matches_simt_path():
    cfg = tpla_cfg("bf16", 2500, 3)
    inp = dev(inputs.decode_inputs(cfg))
    o_tc, l_tc = run_tpla(cfg, inp, 2)
    assert mla.last_path() == mla.PATH_TC
    mla.set_path_override(1)
    try:
        o_s, l_s = run_tpla(cfg, inp, 2)
        assert mla.last_path() == mla.PATH_SIMT
    finally:
        mla.set_path_override(0)
    check_out(o_tc, o_s.float(), torch.bfloat16, "tpla tc vs simt")
    check_lse(l_tc, l_s)


@pytest.mark.parametrize("dtype,rows,d,g", [("bf16", 1000, 512, 1), ("bf16", 1000, 512, 2), ("bf16", 333, 512, 2),
                                            ("bf16", 77, 2048, 4), ("f32", 101, 256, 2), ("bf16", 333, 512, 4),
                                            ("f32", 257, 64, 4), ("f32", 100, 30, 3), ("bf16", 50, 36, 3)])
def test_rmsnorm_shards(oracle, dtype, rows, d, g):
    """The per-shard latent norm (the TPLA cache write) against the oracle's RMSNorm of
    each shard slice; vector and scalar layouts both covered."""
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = inputs.to_torch(inputs.normal_rows(3, inputs.DEC_C_CACHE, rows, d, 2.0), tdt, (rows, d))
    w = inputs.norm_weight(d, tdt, seed=3)
    y = mla.rmsnorm(x.cuda(), w.cuda(), n_shards=g, eps=1e-6)
    torch.cuda.synchronize()
    xs, ws, ds = to64(x), to64(w), d // g
    ref = np.concatenate([oracle.rmsnorm(np.ascontiguousarray(xs[:, i * ds:(i + 1) * ds]), ws[i * ds:(i + 1) * ds],
                                         1e-6) for i in range(g)], 1)
    check_out(y, ref, tdt, "rmsnorm shards")


def test_tpla_cache_write_then_decode(oracle):
    """The whole TPLA chain on the GPU -- per-shard RMSNorm of the raw latent, then the
    decode -- against the oracle from the raw latent.  The normalised cache is rounded
    to bf16 before the decode reads it; over 2000 keys that rounding averages out in the
    log-sum-exp, so the usual bars apply."""
    cfg = tpla_cfg("bf16", 2000, 4)
    inp = inputs.decode_inputs(cfg)
    w = inputs.norm_weight(cfg.d_kv, cfg.torch_dtype)
    d_inp = dev(inp)
    cache = mla.rmsnorm(d_inp["c_cache"], w.cuda(), n_shards=2)
    o, sl = run_tpla(cfg, d_inp, 2, cache=cache)
    n = np_inputs(inp)
    ro, rsl = oracle.tpla_decode(n["q_nope"], n["q_pe"], n["c_cache"], n["kpe_cache"], n["w_kv_b"], to64(w),
                                 shards=2, base=cfg.rope_base)
    check_out(o, ro, torch.bfloat16, "tpla chain out")
    check_lse(sl, rsl, "tpla chain lse")


def test_tpla_full_size_sampled(oracle):
    """The bench's TPLA workload (64 sequences x 32768 keys, 128 heads, 8 splits, two
    shards) in the bench's launch configuration; sequences 0 and 63 against the oracle."""
    cfg = configs.DECODE
    inp = inputs.decode_inputs(cfg)
    o, sl = run_tpla(cfg, dev(inp), 2)
    assert mla.last_path() == mla.PATH_TC
    for b in (0, 63):
        n = np_inputs(inputs.decode_inputs(cfg, batches=(b, b + 1)))
        ro, rsl = oracle.tpla_decode(n["q_nope"], n["q_pe"], n["c_cache"], n["kpe_cache"], n["w_kv_b"], None,
                                     shards=2, base=cfg.rope_base)
        check_out(o[b:b + 1], ro, torch.bfloat16, "tpla out b=%d" % b)
        check_lse(sl[:, b:b + 1], rsl, "tpla lse b=%d" % b)


@pytest.mark.parametrize("dtype,rows,d,g", [("bf16", 1000, 512, 1), ("bf16", 777, 512, 2), ("bf16", 50, 1024, 1),
                                            ("f32", 333, 256, 2), ("f32", 9000, 128, 1), ("bf16", 333, 512, 4),
                                            ("f32", 100, 30, 3), ("bf16", 50, 36, 3), ("bf16", 60001, 512, 2),
                                            ("bf16", 20000, 512, 4)])
def test_rmsnorm_bwd(oracle, dtype, rows, d, g):
    """The per-shard RMSNorm backward against the oracle's, fused and two-kernel paths;
    dw (fp32, a sum over rows) must also come out bit-identical on a second call.  The
    60001-row case walks each warp's ring of staged rows many times round (and ends on a
    ragged last stride); the 20000-row, four-shard case takes the two-kernel path with
    its 16-byte dw pass over many partial rows."""
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = inputs.to_torch(inputs.normal_rows(4, inputs.DEC_C_CACHE, rows, d, 2.0), tdt, (rows, d))
    gy = inputs.to_torch(inputs.normal_rows(5, inputs.DEC_KPE_CACHE, rows, d), tdt, (rows, d))
    w = inputs.norm_weight(d, tdt, seed=4)
    dx, dw = mla.rmsnorm_bwd(x.cuda(), w.cuda(), gy.cuda(), n_shards=g, eps=1e-6)
    dx2, dw2 = mla.rmsnorm_bwd(x.cuda(), w.cuda(), gy.cuda(), n_shards=g, eps=1e-6)
    torch.cuda.synchronize()
    rdx, rdw = oracle.rmsnorm_bwd(to64(x), to64(w), to64(gy), shards=g, eps=1e-6)
    check_out(dx, rdx, tdt, "rmsnorm bwd dx")
    np.testing.assert_allclose(to64(dw), rdw, rtol=1e-4, atol=1e-4 * max(1.0, np.abs(rdw).max()))
    assert torch.equal(dw, dw2) and torch.equal(dx, dx2)


def test_rmsnorm_bwd_no_rows_zeroes_dw():
    x = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(512, dtype=torch.bfloat16, device="cuda")
    dw = torch.full((512,), 7.0, device="cuda")
    mla.rmsnorm_bwd(x, w, x, dw=dw)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw).item() == 0


# ------------------------------------------------ inputs far from unit scale ----
def _scaled(inp, q=1.0, w=1.0):
    out = dict(inp)
    out["q_nope"] = (inp["q_nope"].float() * q).to(torch.bfloat16)
    out["q_pe"] = (inp["q_pe"].float() * q).to(torch.bfloat16)
    out["rms_w"] = (inp["rms_w"].float() * w).to(torch.bfloat16)
    return out


LARGE = configs.Prefill("large_bf16", "bf16", batch=1, s_kv=600, s_q=600, q_offset=0, n_heads=4, d_kv=512,
                        d_nope=128, d_rope=64, d_v=128, head_shard=4)


@pytest.mark.parametrize("absorbed", [False, True])
def test_large_scores_on_the_simt_route(oracle, absorbed):
    """q x 100 and a norm weight of 8 (scores up to ~3000): the CUDA-core kernels, which
    keep fp32 intermediates (selected with mla_set_path_override(1), the route include/mla.h
    names for scores this large), meet the bars scaled to the magnitudes: bf16 output
    rounding grows with |out| and fp32 score rounding with |score|."""
    inp = _scaled(inputs.prefill_inputs(LARGE), q=100.0, w=8.0)
    ro, rl = oracle_prefill(oracle, LARGE, inp, absorbed=absorbed)
    mla.set_path_override(1)
    try:
        o, l = run_prefill(LARGE, dev(inp), absorbed=absorbed)
        assert mla.last_path() == mla.PATH_SIMT
    finally:
        mla.set_path_override(0)
    g, r = to64(o), ro
    assert np.all(np.isfinite(g))
    assert np.abs(g - r).max() <= 3e-2 * max(1.0, np.abs(r).max())
    assert np.linalg.norm(g - r) / np.linalg.norm(r) <= 1e-2
    assert np.abs(to64(l) - rl).max() <= 1e-3 * max(1.0, np.abs(rl).max() / 300.0)


@pytest.mark.parametrize("qs,ws", [(1.0, 1.0), (4.0, 4.0), (100.0, 8.0)])
def test_tensor_core_error_grows_with_the_scores_as_documented(oracle, qs, ws):
    """The tensor-core path's score operands are fp16 (11-bit significand): its LSE error
    is bounded by about 2^-11 of the largest |lse| (include/mla.h), its outputs stay finite
    and within 1e-2 relative L2.  At unit scale that bound is inside the 1e-3 bar."""
    inp = _scaled(inputs.prefill_inputs(LARGE), q=qs, w=ws)
    ro, rl = oracle_prefill(oracle, LARGE, inp)
    o, l = run_prefill(LARGE, dev(inp))
    assert mla.last_path() == mla.PATH_TC
    g = to64(o)
    assert np.all(np.isfinite(g)) and np.all(np.isfinite(to64(l)))
    assert np.linalg.norm(g - ro) / np.linalg.norm(ro) <= 1e-2
    assert np.abs(to64(l) - rl).max() <= 2.0 ** -11 * max(2.0, np.abs(rl).max())
