"""The bounded device wait behind MLA_ERR_DEVICE_TIMEOUT, made to run out on purpose.

Every mbarrier wait in the library's kernels gives up after a time limit, records the
timeout in a device error word and lets the kernel return instead of hanging the GPU.
mla_selftest_bounded_wait launches one tiny kernel whose single wait is on an mbarrier
that no thread ever arrives at (nothing else in flight), with a limit of a millisecond:
the status must then read MLA_ERR_DEVICE_TIMEOUT once, MLA_OK on the next check, and the
context must still run an ordinary call correctly."""
import dataclasses

import pytest
import torch

from head_latent_attention_rmsnorm_gb300 import build as mla_build
from head_latent_attention_rmsnorm_gb300 import configs, inputs, mla

from parity import check_lse, check_out, np_inputs

pytestmark = pytest.mark.gpu

TIMEOUT = -8


def test_bounded_wait_runs_out_and_the_context_stays_usable(oracle):
    mla_build.build()
    torch.cuda.synchronize()
    assert mla.mla_check_device_error(None) == 0          # nothing pending before
    stream = torch.cuda.current_stream().cuda_stream
    assert mla.mla_selftest_bounded_wait(1000, stream) == 0
    assert mla.mla_check_device_error(stream) == TIMEOUT   # the wait gave up and said so
    assert mla.mla_check_device_error(stream) == 0         # the word was cleared
    # the same context still computes: a small decode against the oracle
    cfg = dataclasses.replace(configs.DECODE, batch=2, kv_len=300, n_splits=2)
    inp = inputs.decode_inputs(cfg)
    d = mla.dims(cfg.n_heads, cfg.d_kv, cfg.d_nope, cfg.d_rope, cfg.d_v, cfg.rope_base)
    t = {k: v.cuda() for k, v in inp.items()}
    o, l = mla.decode_splitkv(d, t["q_nope"], t["q_pe"], t["c_cache"], t["kpe_cache"], t["w_kv_b"],
                              n_splits=cfg.n_splits)
    torch.cuda.synchronize()
    ro, rl, _, _ = oracle.mla_decode(**np_inputs(inp), n_splits=cfg.n_splits, base=cfg.rope_base)
    check_out(o, ro, torch.bfloat16, "decode after the timeout")
    check_lse(l, rl, "decode lse after the timeout")
    assert mla.mla_check_device_error(stream) == 0


def test_bounded_wait_twice_in_a_row():
    mla_build.build()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        assert mla.mla_selftest_bounded_wait(500, stream) == 0
        assert mla.mla_check_device_error(stream) == TIMEOUT
    assert mla.mla_check_device_error(stream) == 0
