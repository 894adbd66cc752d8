"""The work and memory accounting behind the bench's figures, checked on the host.

- The visible (query, key) pair count that every TFLOP/s figure divides by, against a
  brute-force count of the causal mask (LAGA page, "What carries the argument": causal
  attention with a per-rank query offset).
- The simulated sequence-parallel ranks partition the causal triangle: their pair
  counts add up to the single-rank count, and rank r rebuilds K/V for the first
  (r + 1) / R of the keys.
- The activation-memory closed form the bench prints beside the allocator's peak equals
  the library's own workspace query (the C ABI's ``*_workspace`` calls, which need no
  GPU), up to the 256-byte alignment of each workspace buffer.
"""
import ctypes
import dataclasses

import pytest

from head_latent_attention_rmsnorm_gb300 import configs, mla


def brute_pairs(s_q, s_kv, q_offset, causal):
    return sum(1 for i in range(s_q) for j in range(s_kv) if not causal or j <= q_offset + i)


@pytest.mark.parametrize("case", [
    dict(s_q=7, s_kv=7, q_offset=0, causal=True),       # the square causal triangle
    dict(s_q=5, s_kv=9, q_offset=4, causal=True),       # a rank's rows ending at the last key
    dict(s_q=3, s_kv=20, q_offset=2, causal=True),      # keys past the last query row
    dict(s_q=6, s_kv=4, q_offset=0, causal=False),
    dict(s_q=4, s_kv=5, q_offset=9, causal=False),      # queries past the keys
    dict(s_q=1, s_kv=1, q_offset=0, causal=True),
])
def test_visible_pairs_match_brute_force(case):
    cfg = dataclasses.replace(configs.TINY, **case)
    assert cfg.pairs() == brute_pairs(**case)
    assert cfg.kv_needed() == (min(case["q_offset"] + case["s_q"], case["s_kv"]) if case["causal"]
                               else case["s_kv"])


def test_sequence_parallel_ranks_partition_the_causal_triangle():
    full = configs.SP8_RANK7.s_kv
    ranks = [dataclasses.replace(configs.SP8_RANK7, q_offset=o) for o in configs.SP8_RANK7.sweep_offsets]
    assert len(ranks) == 8 and sum(r.s_q for r in ranks) == full
    assert sum(r.pairs() for r in ranks) == full * (full + 1) // 2
    for r, cfg in enumerate(ranks):
        assert cfg.kv_needed() == (r + 1) * full // 8
    # the headline call (rank 7): 128 heads x 320 flops per pair, plus K/V for every key
    f = configs.SP8_RANK7.flops()
    assert f["attention"] == 128 * 2 * (192 + 128) * sum(min(14336 + i + 1, full) for i in range(2048))
    assert f["reconstruct"] == 2 * full * 512 * 128 * 256
    assert 3.1265e12 < f["total"] < 3.1275e12


RAGGED = dataclasses.replace(configs.V2LITE, name="ragged", batch=2, s_kv=300, s_q=200, q_offset=77, n_heads=8,
                             head_shard=3)
PAST_KEYS = dataclasses.replace(configs.V2LITE, name="past_keys", batch=2, s_kv=100, s_q=30, q_offset=120,
                                n_heads=8, head_shard=3, causal=False)


@pytest.mark.parametrize("cfg", [configs.V2LITE, configs.V3, configs.SP8_RANK7, RAGGED, PAST_KEYS],
                         ids=lambda c: c.name)
@pytest.mark.parametrize("form", ["explicit", "absorbed", "fused"])
def test_activation_closed_form_matches_the_workspace_query(cfg, form):
    mla.lib()
    d = mla.dims_of(cfg)
    args = (ctypes.byref(d), mla.MLA_BF16, cfg.batch, cfg.s_q, cfg.s_kv, cfg.q_offset, int(cfg.causal),
            cfg.n_heads)
    for hs in sorted({1, 3, 16, cfg.n_heads}):
        if hs > cfg.n_heads:
            continue
        if form == "fused":
            ws = mla.mla_latent_attn_fused_workspace(*args)
            closed = cfg.activation_bytes(False, 0)
        else:
            f = mla.mla_absorbed_attn_workspace if form == "absorbed" else mla.mla_latent_attn_workspace
            ws = f(*args, hs)
            closed = cfg.activation_bytes(form == "absorbed", hs)
        need = closed["total"] - closed["outputs"]
        if form == "absorbed" and cfg.s_q < 128 and 128 % cfg.s_q:
            # the absorbed tensor-core path tiles query rows by 128; other row counts take
            # the CUDA-core route, whose workspace (fp32 intermediates, no 16-bit weight
            # copy) the closed form does not describe
            continue
        assert 0 <= ws - need < 16 * 256, (hs, ws, need)


def test_decode_bytes_are_the_call_tensors_bytes():
    """The decode GB/s figure divides by the bytes of what a call must move: the cache,
    W_kv_b and the queries in, the output and its LSE out (Helix, "What carries the
    argument": decode is bound by reading the KV cache)."""
    import torch

    from head_latent_attention_rmsnorm_gb300 import inputs
    cfg = dataclasses.replace(configs.DECODE, batch=3, kv_len=50)
    t = inputs.decode_inputs(cfg)
    nbytes = lambda x: x.numel() * x.element_size()  # noqa: E731
    assert cfg.cache_bytes() == nbytes(t["c_cache"]) + nbytes(t["kpe_cache"])
    out = torch.empty(cfg.batch, cfg.n_heads, cfg.d_v, dtype=cfg.torch_dtype)
    lse = torch.empty(cfg.batch, cfg.n_heads, dtype=torch.float32)
    assert cfg.algorithmic_bytes() == sum(nbytes(v) for v in t.values()) + nbytes(out) + nbytes(lse)
    # at the bench's size the cache is 98 % of the bytes
    assert configs.DECODE.cache_bytes() / configs.DECODE.algorithmic_bytes() > 0.98
