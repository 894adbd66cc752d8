"""The seeded input generators that the oracle, the parity tests and the bench share.

The sharded parity cases regenerate one simulated rank's query rows, or a range of
decode sequences, on their own and compare against the oracle run on the full
tensors; that is only sound if a row range drawn alone equals the same rows of the
full draw bit for bit.  Also checked: distinct seeds and tensor ids give distinct
streams, and the draws have the stated distribution (N(0, std^2), rounded once).
"""
import dataclasses

import numpy as np
import pytest
import torch

from head_latent_attention_rmsnorm_gb300 import configs, inputs


@pytest.mark.parametrize("r0,r1", [(0, 1000), (0, 1), (250, 777), (255, 257), (512, 768), (999, 1000), (300, 300)])
def test_row_range_equals_rows_of_the_full_draw(r0, r1):
    full = inputs.normal_rows(5, 3, 1000, 24, 0.5)
    part = inputs.normal_rows(5, 3, 1000, 24, 0.5, r0, r1)
    assert part.shape == (r1 - r0, 24) and part.dtype == np.float32
    assert np.array_equal(part, full[r0:r1])


def test_streams_differ_by_seed_tensor_id_and_block():
    n = 2 * inputs.BLOCK
    a = inputs.normal_rows(0, 1, n, 16)
    assert np.array_equal(a, inputs.normal_rows(0, 1, n, 16))   # deterministic
    assert not np.array_equal(a, inputs.normal_rows(1, 1, n, 16))
    assert not np.array_equal(a, inputs.normal_rows(0, 2, n, 16))
    assert not np.array_equal(a[:inputs.BLOCK], a[inputs.BLOCK:])   # each block its own stream


def test_draws_have_the_stated_distribution():
    x = inputs.normal_rows(9, 4, 4096, 256, 0.25).astype(np.float64)
    assert abs(x.mean()) < 5 * 0.25 / np.sqrt(x.size)
    assert abs(x.std() / 0.25 - 1) < 0.01
    t = inputs.to_torch(x.astype(np.float32), torch.bfloat16, (4096, 256))
    assert t.dtype == torch.bfloat16 and t.shape == (4096, 256)
    assert torch.equal(t, torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16))   # rounded once


def test_prefill_query_rows_of_a_rank_are_rows_of_the_whole_sequence():
    cfg = dataclasses.replace(configs.TINY, batch=2)
    whole = inputs.prefill_inputs(cfg, q_rows=(0, cfg.s_kv))
    for lo, hi in ((0, 64), (64, 128), (37, 101)):
        part = inputs.prefill_inputs(cfg, q_rows=(lo, hi))
        for k in ("q_nope", "q_pe"):
            assert torch.equal(part[k], whole[k][:, lo:hi]), (k, lo, hi)
        for k in ("c_kv", "k_pe", "w_kv_b", "rms_w"):
            assert torch.equal(part[k], whole[k]), k
    # the default rows are the config's own [q_offset, q_offset + s_q)
    off = dataclasses.replace(cfg, q_offset=64, s_q=64)
    assert torch.equal(inputs.prefill_inputs(off)["q_nope"], whole["q_nope"][:, 64:128])


def test_decode_sequence_range_is_rows_of_the_whole_batch():
    cfg = dataclasses.replace(configs.DECODE, batch=5, kv_len=300, n_heads=4)
    whole = inputs.decode_inputs(cfg)
    part = inputs.decode_inputs(cfg, batches=(2, 4))
    for k in ("q_nope", "q_pe", "c_cache", "kpe_cache"):
        assert torch.equal(part[k], whole[k][2:4]), k
    assert torch.equal(part["w_kv_b"], whole["w_kv_b"])
    assert "w_kv_b" not in inputs.decode_inputs(cfg, batches=(0, 1), with_weights=False)
