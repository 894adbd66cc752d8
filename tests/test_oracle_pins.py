"""Pins for the CPU oracle: each stage is tied to something other than itself.

* RMSNorm  -- closed form for a constant row; torch's own rms_norm (a library routine).
* RoPE     -- identity at position 0; the half-split rotation as a complex product
              z * exp(i * pos * base^(-2t/d)) (textbook rotation); norm preservation;
              composition; relative-position invariance of dot products.
* Attention -- the whole explicit path rebuilt from library routines (torch rms_norm,
              torch.matmul, numpy complex rotation, torch scaled_dot_product_attention,
              torch.logsumexp); closed form for all-zero queries; brute force in
              50-digit arithmetic on a 3-key case.
* Forms     -- explicit == absorbed (LAGA, Fig. 2 and "What carries the argument");
              concatenated query shards == one call (LAGA, sequence-parallel ranks);
              head ranges concatenate (LAGA, "H_r slice", paper section 3.3).
* Decode    -- split partials merged by the log-sum-exp rescale equal the unsplit
              result (Helix, "Assumptions", paper section 2.1.1); decode at position
              L-1 equals the last row of a prefill over the same latent.
* TPLA      -- one shard is plain latent decode; g shards equal the sum of g independent
              latent decodes over the shard slices (TPLA, "The reading"), and the same
              sum rebuilt from library routines (torch rms_norm per shard, matmul,
              softmax, logsumexp).
* Backward  -- every entry of every gradient of the explicit path against central finite
              differences of the (pinned) forward in fp64, for causal with an offset,
              non-causal and a head range (LAGA, "What carries the argument": the method's
              gradients match the baseline's).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

BASE = 10000.0
EPS = 1e-6


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


# ----------------------------------------------------------------- RMSNorm ----
def test_rmsnorm_constant_row_closed_form(oracle):
    d = 48
    w = _rand(d, 1)
    for alpha in (-3.0, 0.25, 7.5):
        x = np.full((1, d), alpha)
        y = oracle.rmsnorm(x, w, EPS)
        expect = w * alpha / math.sqrt(alpha * alpha + EPS)
        np.testing.assert_allclose(y[0], expect, rtol=1e-15, atol=0)


def test_rmsnorm_matches_torch_library(oracle):
    x = _rand((37, 64), 2) * 3.0
    w = _rand(64, 3)
    y = oracle.rmsnorm(x, w, EPS)
    ref = F.rms_norm(torch.from_numpy(x), (64,), weight=torch.from_numpy(w), eps=EPS).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-14)


def test_rmsnorm_unit_mean_square_and_scale_invariance(oracle):
    x = _rand((9, 512), 4)
    y = oracle.rmsnorm(x, np.ones(512), 0.0)
    np.testing.assert_allclose((y * y).mean(-1), 1.0, rtol=1e-13)
    y2 = oracle.rmsnorm(x * 17.0, np.ones(512), 0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-13, atol=1e-14)


# -------------------------------------------------------------------- RoPE ----
def _rope_complex(x, pos, d):
    """Textbook form: the pair (x_t, x_{t+d/2}) as a complex number times e^{i*pos*theta_t}."""
    h = d // 2
    z = x[..., :h] + 1j * x[..., h:]
    theta = BASE ** (-2.0 * np.arange(h) / d)
    z = z * np.exp(1j * np.asarray(pos, dtype=np.float64)[..., None] * theta)
    return np.concatenate([z.real, z.imag], -1)


def test_rope_position_zero_is_identity(oracle):
    x = _rand((5, 64), 5)
    np.testing.assert_array_equal(oracle.rope(x, 0.0, BASE), x)


@pytest.mark.parametrize("d", [16, 64])
def test_rope_matches_complex_rotation(oracle, d):
    x = _rand((50, d), 6)
    pos = np.arange(50) * 331.0 + 7.0
    y = oracle.rope(x, pos, BASE)
    # one ulp of theta (pow in C vs numpy) moves the angle by pos * 2.2e-16
    atol = 8 * pos.max() * np.finfo(np.float64).eps * np.abs(x).max()
    np.testing.assert_allclose(y, _rope_complex(x, pos, d), rtol=0, atol=atol)


def test_rope_norm_composition_relative(oracle):
    d = 64
    x = _rand((8, d), 7)
    y = oracle.rope(x, 1234.0, BASE)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    two = oracle.rope(oracle.rope(x, 100.0, BASE), 23.0, BASE)
    np.testing.assert_allclose(two, oracle.rope(x, 123.0, BASE), rtol=1e-11, atol=1e-12)
    q, k = _rand(d, 8), _rand(d, 9)
    a = oracle.rope(q[None], 500.0, BASE)[0] @ oracle.rope(k[None], 470.0, BASE)[0]
    b = oracle.rope(q[None], 30.0, BASE)[0] @ oracle.rope(k[None], 0.0, BASE)[0]
    assert abs(a - b) < 1e-11


# ---------------------------------------------- whole path from library calls ----
def _make(B, S, H, dk, dn, dr, dv, seed, s_q=None, q_off=0):
    s_q = S if s_q is None else s_q
    g = np.random.default_rng(seed)
    return dict(
        q_nope=g.standard_normal((B, s_q, H, dn)),
        q_pe=g.standard_normal((B, s_q, H, dr)),
        c_kv=g.standard_normal((B, S, dk)),
        k_pe=g.standard_normal((B, S, dr)),
        w_kv_b=g.standard_normal((H * (dn + dv), dk)) / math.sqrt(dk),
        rms_w=1.0 + 0.1 * g.standard_normal(dk),
    )


def _library_explicit(inp, n_heads, q_off, causal, head_begin=0, scale=None):
    """The explicit MLA path composed from library routines only."""
    qn = torch.from_numpy(inp["q_nope"])
    B, s_q, hc, dn = qn.shape
    dr = inp["q_pe"].shape[-1]
    S, dk = inp["c_kv"].shape[1:]
    W = torch.from_numpy(inp["w_kv_b"]).reshape(n_heads, -1, dk)
    dv = W.shape[1] - dn
    scale = 1.0 / math.sqrt(dn + dr) if scale is None else scale
    chat = F.rms_norm(torch.from_numpy(inp["c_kv"]), (dk,), weight=torch.from_numpy(inp["rms_w"]), eps=EPS)
    kv = torch.einsum("bsk,hnk->bhsn", chat, W[head_begin:head_begin + hc])  # [B,hc,S,dn+dv]
    kn, v = kv[..., :dn], kv[..., dn:]
    qpos = q_off + np.arange(s_q)
    qr = torch.from_numpy(_rope_complex(inp["q_pe"], qpos[None, :, None].repeat(hc, 2), dr))
    kr = torch.from_numpy(_rope_complex(inp["k_pe"], np.arange(S)[None, :], dr))
    q = torch.cat([qn, qr], -1).permute(0, 2, 1, 3)                  # [B,hc,s_q,dqk]
    k = torch.cat([kn, kr[:, None].expand(B, hc, S, dr)], -1)        # [B,hc,S,dqk]
    mask = torch.ones(s_q, S, dtype=torch.bool)
    if causal:
        mask = torch.from_numpy(np.arange(S)[None, :] <= qpos[:, None])
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    s = torch.matmul(q, k.transpose(-1, -2)) * scale
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, -1)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy()


@pytest.mark.parametrize("q_off,causal,s_q,head_begin,hc", [
    (0, True, 24, 0, 3), (9, True, 11, 1, 2), (0, False, 20, 0, 3), (5, False, 7, 2, 1)])
def test_explicit_matches_library_composition(oracle, q_off, causal, s_q, head_begin, hc):
    H, S, dk, dn, dr, dv = 3, 24, 40, 12, 8, 10
    inp = _make(2, S, hc, dk, dn, dr, dv, 11, s_q=s_q)
    inp["w_kv_b"] = _rand((H * (dn + dv), dk), 12, 1 / math.sqrt(dk))
    out, lse = oracle.mla_explicit(**inp, n_heads=H, q_offset=q_off, causal=causal,
                                   head_begin=head_begin, eps=EPS)
    ref_o, ref_l = _library_explicit(inp, H, q_off, causal, head_begin)
    np.testing.assert_allclose(out, ref_o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def test_zero_queries_give_uniform_softmax(oracle):
    H, S, dk, dn, dr, dv = 2, 16, 32, 8, 8, 8
    inp = _make(1, S, H, dk, dn, dr, dv, 13)
    inp["q_nope"][:] = 0.0
    inp["q_pe"][:] = 0.0
    out, lse = oracle.mla_explicit(**inp, n_heads=H, causal=True, eps=EPS)
    n = np.arange(1, S + 1)
    np.testing.assert_allclose(lse[0], np.log(n)[None, :].repeat(H, 0), rtol=0, atol=1e-14)
    chat = F.rms_norm(torch.from_numpy(inp["c_kv"][0]), (dk,), weight=torch.from_numpy(inp["rms_w"]), eps=EPS)
    W = torch.from_numpy(inp["w_kv_b"]).reshape(H, dn + dv, dk)
    v = torch.einsum("sk,hnk->hsn", chat, W)[..., dn:].numpy()         # [H,S,dv]
    mean_v = np.cumsum(v, 1) / n[None, :, None]
    np.testing.assert_allclose(out[0].transpose(1, 0, 2), mean_v, rtol=1e-12, atol=1e-13)


def test_brute_force_high_precision(oracle):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    H, S, dk, dn, dr, dv = 1, 3, 4, 2, 2, 2
    inp = _make(1, S, H, dk, dn, dr, dv, 14)
    out, lse = oracle.mla_explicit(**inp, n_heads=H, causal=True, eps=EPS)
    c, w, W = inp["c_kv"][0], inp["rms_w"], inp["w_kv_b"]
    chat = []
    for j in range(S):
        ms = mp.fsum(mp.mpf(x) ** 2 for x in c[j]) / dk
        chat.append([mp.mpf(c[j][k]) * mp.mpf(w[k]) / mp.sqrt(ms + mp.mpf(EPS)) for k in range(dk)])

    def rot(x, pos):
        h = dr // 2
        y = [None] * dr
        for t in range(h):
            a = mp.mpf(pos) * mp.power(mp.mpf(BASE), -mp.mpf(2 * t) / dr)
            y[t] = mp.mpf(x[t]) * mp.cos(a) - mp.mpf(x[t + h]) * mp.sin(a)
            y[t + h] = mp.mpf(x[t + h]) * mp.cos(a) + mp.mpf(x[t]) * mp.sin(a)
        return y

    K = [[mp.fsum(mp.mpf(W[d][k]) * chat[j][k] for k in range(dk)) for d in range(dn + dv)] for j in range(S)]
    kr = [rot(inp["k_pe"][0][j], j) for j in range(S)]
    scale = 1 / mp.sqrt(dn + dr)
    for i in range(S):
        q = [mp.mpf(x) for x in inp["q_nope"][0][i][0]]
        qr = rot(inp["q_pe"][0][i][0], i)
        s = [scale * (mp.fsum(q[d] * K[j][d] for d in range(dn)) + mp.fsum(qr[t] * kr[j][t] for t in range(dr)))
             for j in range(i + 1)]
        z = mp.fsum(mp.exp(x) for x in s)
        o = [mp.fsum(mp.exp(s[j]) * K[j][dn + d] for j in range(i + 1)) / z for d in range(dv)]
        assert abs(float(mp.log(z)) - lse[0, 0, i]) < 1e-13
        for d in range(dv):
            assert abs(float(o[d]) - out[0, i, 0, d]) < 1e-13


# ------------------------------------------------------------ form identities ----
@pytest.mark.parametrize("q_off,causal", [(0, True), (16, True), (0, False)])
def test_explicit_equals_absorbed(oracle, q_off, causal):
    H, S, dk, dn, dr, dv = 4, 48, 64, 32, 16, 32
    inp = _make(2, S, H, dk, dn, dr, dv, 21, s_q=S - q_off)
    a = oracle.mla_explicit(**inp, n_heads=H, q_offset=q_off, causal=causal, eps=EPS)
    b = oracle.mla_absorbed(**inp, n_heads=H, q_offset=q_off, causal=causal, eps=EPS)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-10)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-10)


def test_query_shards_concatenate(oracle):
    H, S, dk, dn, dr, dv = 4, 64, 32, 16, 8, 16
    inp = _make(1, S, H, dk, dn, dr, dv, 22)
    full_o, full_l = oracle.mla_explicit(**inp, n_heads=H, eps=EPS)
    P = 8
    for r in range(P):
        sl = slice(r * S // P, (r + 1) * S // P)
        part = dict(inp, q_nope=inp["q_nope"][:, sl], q_pe=inp["q_pe"][:, sl])
        o, l = oracle.mla_explicit(**part, n_heads=H, q_offset=sl.start, eps=EPS)
        np.testing.assert_array_equal(o, full_o[:, sl])
        np.testing.assert_array_equal(l, full_l[:, :, sl])


def test_head_ranges_concatenate(oracle):
    H, S, dk, dn, dr, dv = 6, 20, 32, 16, 8, 16
    inp = _make(1, S, H, dk, dn, dr, dv, 23)
    full_o, full_l = oracle.mla_explicit(**inp, n_heads=H, eps=EPS)
    for h0, hc in ((0, 2), (2, 3), (5, 1)):
        part = dict(inp, q_nope=inp["q_nope"][:, :, h0:h0 + hc], q_pe=inp["q_pe"][:, :, h0:h0 + hc])
        o, l = oracle.mla_explicit(**part, n_heads=H, head_begin=h0, eps=EPS)
        np.testing.assert_array_equal(o, full_o[:, :, h0:h0 + hc])
        np.testing.assert_array_equal(l, full_l[:, h0:h0 + hc])


# ------------------------------------------------------------------- decode ----
def _decode_inputs(B, H, L, dk, dn, dr, dv, seed):
    g = np.random.default_rng(seed)
    return dict(q_nope=g.standard_normal((B, H, dn)), q_pe=g.standard_normal((B, H, dr)),
                c_cache=g.standard_normal((B, L, dk)), kpe_cache=g.standard_normal((B, L, dr)),
                w_kv_b=g.standard_normal((H * (dn + dv), dk)) / math.sqrt(dk))


@pytest.mark.parametrize("L,n_splits", [(100, 1), (100, 2), (100, 3), (100, 8), (100, 13), (10, 13)])
def test_decode_split_combine_equals_unsplit(oracle, L, n_splits):
    B, H, dk, dn, dr, dv = 2, 3, 32, 16, 8, 16
    inp = _decode_inputs(B, H, L, dk, dn, dr, dv, 31)
    out, lse, po, pl = oracle.mla_decode(**inp, n_splits=n_splits)
    o_lat, l = oracle.lse_combine(po.reshape(n_splits, -1, dk), pl.reshape(n_splits, -1))
    W = inp["w_kv_b"].reshape(H, dn + dv, dk)[:, dn:]                    # W_V per head
    o = np.einsum("hdk,bhk->bhd", W, o_lat.reshape(B, H, dk))
    np.testing.assert_allclose(o, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l.reshape(B, H), lse, rtol=0, atol=1e-12)
    chunk = -(-L // n_splits)
    for s in range(n_splits):
        if s * chunk >= L:
            assert np.all(np.isneginf(pl[s])) and np.all(po[s] == 0)


def test_lse_combine_matches_library(oracle):
    g = np.random.default_rng(41)
    n, rows, D = 5, 7, 9
    po, pl = g.standard_normal((n, rows, D)), 3 * g.standard_normal((n, rows))
    pl[2, 3] = -np.inf
    out, lse = oracle.lse_combine(po, pl)
    t = torch.from_numpy(pl)
    ref_l = torch.logsumexp(t, 0)
    ref_o = (torch.softmax(t, 0)[..., None] * torch.from_numpy(po)).sum(0)
    np.testing.assert_allclose(lse, ref_l.numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(out, ref_o.numpy(), rtol=0, atol=1e-13)
    one_o, one_l = oracle.lse_combine(po[:1], pl[:1])
    np.testing.assert_array_equal(one_o, po[0])
    np.testing.assert_array_equal(one_l, pl[0])


def test_decode_equals_last_prefill_row(oracle):
    H, S, dk, dn, dr, dv = 3, 33, 32, 16, 8, 16
    inp = _make(2, S, H, dk, dn, dr, dv, 51, s_q=1)
    o_ref, l_ref = oracle.mla_explicit(**inp, n_heads=H, q_offset=S - 1, eps=EPS)
    cache = oracle.rmsnorm(inp["c_kv"], inp["rms_w"], EPS)
    kpe = oracle.rope(inp["k_pe"], np.arange(S)[None, :].repeat(2, 0).astype(np.float64), BASE)
    out, lse, _, _ = oracle.mla_decode(inp["q_nope"][:, 0], inp["q_pe"][:, 0], cache, kpe,
                                       inp["w_kv_b"], n_splits=4)
    np.testing.assert_allclose(out, o_ref[:, 0], rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, l_ref[:, :, 0], rtol=0, atol=1e-11)


def _tpla_inputs(B, H, L, dk, dn, dr, dv, seed):
    inp = _decode_inputs(B, H, L, dk, dn, dr, dv, seed)
    g = np.random.default_rng(seed + 1)
    c_raw = inp.pop("c_cache") * (1.0 + 2.0 * g.random((1, 1, dk)))   # shards differ in scale
    return dict(inp, c_raw=c_raw, rms_w=1.0 + 0.2 * g.standard_normal(dk))


def test_tpla_one_shard_is_latent_decode(oracle):
    B, H, L, dk, dn, dr, dv = 2, 3, 57, 32, 16, 8, 16
    inp = _tpla_inputs(B, H, L, dk, dn, dr, dv, 61)
    out, slse = oracle.tpla_decode(**inp, shards=1, eps=EPS)
    cache = oracle.rmsnorm(inp["c_raw"].reshape(-1, dk), inp["rms_w"], EPS).reshape(B, L, dk)
    ref, lse, _, _ = oracle.mla_decode(inp["q_nope"], inp["q_pe"], cache, inp["kpe_cache"],
                                       inp["w_kv_b"], n_splits=3)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(slse[0], lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shards", [2, 4])
def test_tpla_shards_sum_of_slice_decodes(oracle, shards):
    B, H, L, dk, dn, dr, dv = 2, 3, 41, 32, 16, 8, 16
    inp = _tpla_inputs(B, H, L, dk, dn, dr, dv, 71)
    out, slse = oracle.tpla_decode(**inp, shards=shards, eps=EPS)
    ds, acc = dk // shards, 0.0
    for i in range(shards):
        sl = slice(i * ds, (i + 1) * ds)
        ci = np.ascontiguousarray(inp["c_raw"][..., sl]).reshape(-1, ds)
        ci = oracle.rmsnorm(ci, inp["rms_w"][sl], EPS).reshape(B, L, ds)
        oi, li, _, _ = oracle.mla_decode(inp["q_nope"], inp["q_pe"], ci, inp["kpe_cache"],
                                         np.ascontiguousarray(inp["w_kv_b"][:, sl]), n_splits=2,
                                         scale=oracle.default_scale(dn, dr))
        acc = acc + oi
        np.testing.assert_allclose(slse[i], li, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, acc, rtol=0, atol=1e-12)
    full, _, _, _ = oracle.mla_decode(inp["q_nope"], inp["q_pe"],
                                      oracle.rmsnorm(inp["c_raw"].reshape(-1, dk), inp["rms_w"], EPS)
                                      .reshape(B, L, dk), inp["kpe_cache"], inp["w_kv_b"])
    assert np.abs(out - full).max() > 1e-3          # sharding really changes the result


def test_tpla_normalised_cache_mode(oracle):
    """rms_w=None reads the cache as already normalised: it equals normalising first."""
    B, H, L, dk, dn, dr, dv, G = 2, 3, 29, 32, 16, 8, 16, 4
    inp = _tpla_inputs(B, H, L, dk, dn, dr, dv, 91)
    out, slse = oracle.tpla_decode(**inp, shards=G, eps=EPS)
    ds = dk // G
    c = inp["c_raw"].reshape(-1, G, ds)
    chat = np.stack([oracle.rmsnorm(np.ascontiguousarray(c[:, i]), inp["rms_w"][i * ds:(i + 1) * ds], EPS)
                     for i in range(G)], 1).reshape(B, L, dk)
    o2, l2 = oracle.tpla_decode(**dict(inp, c_raw=chat, rms_w=None), shards=G)
    np.testing.assert_allclose(o2, out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, slse, rtol=0, atol=1e-13)


def test_tpla_matches_library_composition(oracle):
    B, H, L, dk, dn, dr, dv, G = 2, 4, 37, 32, 16, 8, 16, 2
    inp = _tpla_inputs(B, H, L, dk, dn, dr, dv, 81)
    out, slse = oracle.tpla_decode(**inp, shards=G, eps=EPS)
    t = {k: torch.from_numpy(v) for k, v in inp.items()}
    W = t["w_kv_b"].reshape(H, dn + dv, dk)
    q_abs = torch.einsum("bhd,hdk->bhk", t["q_nope"], W[:, :dn])
    qr = torch.from_numpy(_rope_complex(inp["q_pe"], np.full((B, H), L - 1.0), dr))
    scale = 1.0 / math.sqrt(dn + dr)
    ref_o = torch.zeros(B, H, dv, dtype=torch.float64)
    ds = dk // G
    for i in range(G):
        sl = slice(i * ds, (i + 1) * ds)
        c = F.rms_norm(t["c_raw"][..., sl], (ds,), t["rms_w"][sl], EPS)       # [B,L,ds]
        s = (torch.einsum("bhk,blk->bhl", q_abs[..., sl], c)
             + torch.einsum("bhr,blr->bhl", qr, t["kpe_cache"])) * scale
        o_lat = torch.einsum("bhl,blk->bhk", torch.softmax(s, -1), c)
        ref_o += torch.einsum("hdk,bhk->bhd", W[:, dn:, sl], o_lat)
        np.testing.assert_allclose(slse[i], torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, ref_o.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("shards", [1, 2, 4])
def test_rmsnorm_backward_matches_finite_differences(oracle, shards):
    rows, d = 5, 24
    x, w, G = _rand((rows, d), 111) * 2.0, 1.0 + 0.3 * _rand(d, 112), _rand((rows, d), 113)
    dx, dw = oracle.rmsnorm_bwd(x, w, G, shards=shards, eps=EPS)
    ds = d // shards

    def loss(x_, w_):
        y = np.concatenate([oracle.rmsnorm(np.ascontiguousarray(x_[:, i * ds:(i + 1) * ds]),
                                           w_[i * ds:(i + 1) * ds], EPS) for i in range(shards)], 1)
        return float((y * G).sum())

    h = 1e-6
    for arr, grad in ((x, dx), (w, dw)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + h
            up = loss(x, w)
            arr[idx] = keep - h
            fd[idx] = (up - loss(x, w)) / (2 * h)
            arr[idx] = keep
        np.testing.assert_allclose(grad, fd, rtol=0, atol=1e-7)


@pytest.mark.parametrize("q_off,causal,s_q,head_begin,hc", [(4, True, 5, 0, 3), (0, False, 4, 0, 3),
                                                            (2, True, 3, 1, 2)])
def test_explicit_backward_matches_finite_differences(oracle, q_off, causal, s_q, head_begin, hc):
    B, S, H, dk, dn, dr, dv = 2, 9, 3, 16, 8, 8, 8
    inp = _make(B, S, H, dk, dn, dr, dv, 101, s_q=s_q, q_off=q_off)
    inp["q_nope"], inp["q_pe"] = inp["q_nope"][:, :, :hc].copy(), inp["q_pe"][:, :, :hc].copy()
    inp["rms_w"] = 1.0 + 0.3 * _rand(dk, 102)
    G = _rand((B, s_q, hc, dv), 103)
    kw = dict(n_heads=H, q_offset=q_off, causal=causal, head_begin=head_begin, eps=EPS)
    grads = oracle.mla_explicit_bwd(**inp, dout=G, **kw)

    def loss(d):
        out, _ = oracle.mla_explicit(**d, **kw)
        return float((out * G).sum())

    h = 1e-5
    for name in ("q_nope", "q_pe", "c_kv", "k_pe", "w_kv_b", "rms_w"):
        x = inp[name]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            keep = x[idx]
            x[idx] = keep + h
            up = loss(inp)
            x[idx] = keep - h
            dn_ = loss(inp)
            x[idx] = keep
            fd[idx] = (up - dn_) / (2 * h)
        assert np.abs(fd).max() > 0, name
        np.testing.assert_allclose(grads[name], fd, rtol=0, atol=1e-7 * max(1.0, np.abs(fd).max()),
                                   err_msg=name)
    if causal:   # keys no query sees carry no gradient
        n_vis = q_off + s_q
        assert np.all(grads["c_kv"][:, n_vis:] == 0) and np.all(grads["k_pe"][:, n_vis:] == 0)
    # heads outside the range get no weight gradient
    Wg = grads["w_kv_b"].reshape(H, dn + dv, dk)
    for hh in range(H):
        if not head_begin <= hh < head_begin + hc:
            assert np.all(Wg[hh] == 0)


def test_golden_rows_unchanged(oracle):
    """Regression anchor: the oracle still gives the stored rows on the seeded tiny case."""
    import os
    from head_latent_attention_rmsnorm_gb300 import configs, inputs
    cfg = configs.TINY
    inp = {k: v.double().numpy() for k, v in inputs.prefill_inputs(cfg, seed=0).items()}
    out, lse = oracle.mla_explicit(**inp, n_heads=cfg.n_heads, causal=True, base=cfg.rope_base,
                                   eps=cfg.rms_eps)
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_fp32_oracle_rows.txt")
    for line in open(path):
        if line.startswith("#"):
            continue
        f = line.split()
        i, h = int(f[0]), int(f[1])
        assert abs(lse[0, h, i] - float(f[2])) < 1e-12
        np.testing.assert_allclose(out[0, i, h, :8], [float(x) for x in f[3:]], rtol=0, atol=1e-12)
