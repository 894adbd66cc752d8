"""The oracle's pins repeated over seeded random small shapes, so that a mistake that
hides at one shape (a band width that happens to be a multiple of something, a head
count of one, a square causal mask) still fails somewhere:

* the explicit path against its composition from library routines (torch rms_norm,
  einsum, complex rotation, scaled_dot_product_attention, logsumexp);
* explicit == absorbed (LAGA, Fig. 2 and "What carries the argument");
* split-KV decode partials merged by the log-sum-exp rescale == one split (Helix,
  "Assumptions");
* every gradient of the explicit path against central finite differences;
* TPLA's g-shard decode == the sum of g latent decodes over the shard slices.

Shapes: B 1-2, heads 1-5 with a random head range, 1-40 keys, the query rows a random
slice (causal: inside the keys; non-causal: possibly past them), d_kv 8-40, d_nope
4-12, d_rope 2-8 (even), d_v 4-10.
"""
import numpy as np
import pytest

from test_oracle_pins import EPS, _library_explicit, _make

CASES = 16


def _shape(seed):
    g = np.random.default_rng(1000 + seed)
    B, H = int(g.integers(1, 3)), int(g.integers(1, 6))
    S = int(g.integers(1, 41))
    dk, dn = int(g.choice([8, 16, 24, 40])), int(g.choice([4, 8, 12]))
    dr, dv = int(g.choice([2, 4, 6, 8])), int(g.choice([4, 8, 10]))
    causal = bool(g.integers(0, 2))
    s_q = int(g.integers(1, S + 1))
    q_off = int(g.integers(0, S - s_q + 1)) if causal else int(g.integers(0, S + 6))
    h0 = int(g.integers(0, H))
    hc = int(g.integers(1, H - h0 + 1))
    return B, H, S, dk, dn, dr, dv, causal, s_q, q_off, h0, hc


@pytest.mark.parametrize("seed", range(CASES))
def test_explicit_against_library_and_absorbed(oracle, seed):
    B, H, S, dk, dn, dr, dv, causal, s_q, q_off, h0, hc = _shape(seed)
    inp = _make(B, S, hc, dk, dn, dr, dv, 2000 + seed, s_q=s_q)
    inp["w_kv_b"] = np.random.default_rng(3000 + seed).standard_normal((H * (dn + dv), dk)) / np.sqrt(dk)
    kw = dict(n_heads=H, q_offset=q_off, causal=causal, head_begin=h0, eps=EPS)
    out, lse = oracle.mla_explicit(**inp, **kw)
    ref_o, ref_l = _library_explicit(inp, H, q_off, causal, h0)
    np.testing.assert_allclose(out, ref_o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)
    a_o, a_l = oracle.mla_absorbed(**inp, **kw)
    np.testing.assert_allclose(a_o, out, rtol=0, atol=1e-10)
    np.testing.assert_allclose(a_l, lse, rtol=0, atol=1e-10)


@pytest.mark.parametrize("seed", range(CASES))
def test_decode_splits_against_one_split(oracle, seed):
    g = np.random.default_rng(4000 + seed)
    B, H, L = int(g.integers(1, 3)), int(g.integers(1, 6)), int(g.integers(1, 60))
    dk, dn = int(g.choice([8, 16, 24, 40])), int(g.choice([4, 8, 12]))
    dr, dv = int(g.choice([2, 4, 6, 8])), int(g.choice([4, 8, 10]))
    n = int(g.integers(1, L + 4))   # may leave trailing splits empty
    inp = dict(q_nope=g.standard_normal((B, H, dn)), q_pe=g.standard_normal((B, H, dr)),
               c_cache=g.standard_normal((B, L, dk)), kpe_cache=g.standard_normal((B, L, dr)),
               w_kv_b=g.standard_normal((H * (dn + dv), dk)) / np.sqrt(dk))
    one_o, one_l, _, _ = oracle.mla_decode(**inp, n_splits=1)
    out, lse, po, pl = oracle.mla_decode(**inp, n_splits=n)
    np.testing.assert_allclose(out, one_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, one_l, rtol=0, atol=1e-12)
    # the partials merged by the combine give the latent output that W_V up-projects
    o_lat, l = oracle.lse_combine(po.reshape(n, -1, dk), pl.reshape(n, -1))
    W_V = inp["w_kv_b"].reshape(H, dn + dv, dk)[:, dn:]
    np.testing.assert_allclose(np.einsum("hdk,bhk->bhd", W_V, o_lat.reshape(B, H, dk)), out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l.reshape(B, H), lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_backward_against_finite_differences(oracle, seed):
    """Every entry of every gradient (LAGA, "What carries the argument": the gradients
    are part of the equivalence) against central differences of the forward."""
    g = np.random.default_rng(5000 + seed)
    B, H, S = int(g.integers(1, 3)), int(g.integers(1, 4)), int(g.integers(2, 8))
    dk, dn, dr, dv = int(g.choice([4, 8])), int(g.choice([2, 4])), int(g.choice([2, 4])), int(g.choice([2, 4]))
    causal = bool(g.integers(0, 2))
    s_q = int(g.integers(1, S + 1))
    q_off = int(g.integers(0, S - s_q + 1)) if causal else int(g.integers(0, S + 3))
    h0 = int(g.integers(0, H))
    hc = int(g.integers(1, H - h0 + 1))
    inp = _make(B, S, hc, dk, dn, dr, dv, 6000 + seed, s_q=s_q)
    inp["w_kv_b"] = g.standard_normal((H * (dn + dv), dk)) / np.sqrt(dk)
    dout = g.standard_normal((B, s_q, hc, dv))
    kw = dict(n_heads=H, q_offset=q_off, causal=causal, head_begin=h0, eps=EPS)
    grads = oracle.mla_explicit_bwd(**inp, dout=dout, **kw)

    def loss():
        return float((oracle.mla_explicit(**inp, **kw)[0] * dout).sum())

    h = 1e-5
    for name in ("q_nope", "q_pe", "c_kv", "k_pe", "w_kv_b", "rms_w"):
        x = inp[name]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            keep = x[idx]
            x[idx] = keep + h
            up = loss()
            x[idx] = keep - h
            fd[idx] = (up - loss()) / (2 * h)
            x[idx] = keep
        np.testing.assert_allclose(grads[name], fd, rtol=0, atol=1e-7 * max(1.0, np.abs(fd).max()), err_msg=name)


@pytest.mark.parametrize("seed", range(8))
def test_tpla_shards_sum_of_slice_decodes(oracle, seed):
    """TPLA ("The reading"): g shards, each normalised and attended on its own, summed
    after the up-projection, equal g independent latent decodes over the slices."""
    g = np.random.default_rng(7000 + seed)
    B, H, L = int(g.integers(1, 3)), int(g.integers(1, 5)), int(g.integers(1, 50))
    shards = int(g.choice([1, 2, 4]))
    ds = int(g.choice([2, 4, 8]))
    dk, dn, dr, dv = shards * ds, int(g.choice([4, 8])), int(g.choice([2, 4, 6])), int(g.choice([4, 6]))
    inp = dict(q_nope=g.standard_normal((B, H, dn)), q_pe=g.standard_normal((B, H, dr)),
               c_raw=g.standard_normal((B, L, dk)) * (1.0 + 2.0 * g.random((1, 1, dk))),
               kpe_cache=g.standard_normal((B, L, dr)),
               w_kv_b=g.standard_normal((H * (dn + dv), dk)) / np.sqrt(dk), rms_w=1.0 + 0.2 * g.standard_normal(dk))
    out, slse = oracle.tpla_decode(**inp, shards=shards, eps=EPS)
    acc = 0.0
    for i in range(shards):
        sl = slice(i * ds, (i + 1) * ds)
        ci = oracle.rmsnorm(np.ascontiguousarray(inp["c_raw"][..., sl]).reshape(-1, ds), inp["rms_w"][sl], EPS)
        oi, li, _, _ = oracle.mla_decode(inp["q_nope"], inp["q_pe"], ci.reshape(B, L, ds), inp["kpe_cache"],
                                         np.ascontiguousarray(inp["w_kv_b"][:, sl]),
                                         n_splits=int(g.integers(1, L + 2)), scale=oracle.default_scale(dn, dr))
        acc = acc + oi
        np.testing.assert_allclose(slse[i], li, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, acc, rtol=0, atol=1e-12)
