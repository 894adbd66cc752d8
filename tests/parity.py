"""Tolerances and comparison helpers shared by the GPU parity tests.

Bars (the workload description's): fp32 storage -> max |err| <= 1e-4; bf16 storage
with fp32 accumulation -> max |err| <= 3e-2 and relative L2 <= 1e-2; log-sum-exp ->
max |err| <= 1e-3.
"""
import numpy as np
import torch

F32_ABS = 1e-4
BF16_ABS = 3e-2
BF16_REL_L2 = 1e-2
LSE_ABS = 1e-3


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def check_out(gpu, ref, dtype, what="out"):
    g, r = to64(gpu), to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), what + ": non-finite values"
    err = np.abs(g - r).max() if g.size else 0.0
    if dtype == torch.float32:
        assert err <= F32_ABS, "%s: max abs err %.3e > %.0e" % (what, err, F32_ABS)
        return err, 0.0
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert err <= BF16_ABS, "%s: max abs err %.3e > %.0e" % (what, err, BF16_ABS)
    assert rel <= BF16_REL_L2, "%s: rel L2 %.3e > %.0e" % (what, rel, BF16_REL_L2)
    return err, rel


def check_lse(gpu, ref, what="lse"):
    g, r = to64(gpu), to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    both_inf = np.isneginf(g) & np.isneginf(r)
    assert np.array_equal(np.isneginf(g), np.isneginf(r)), what + ": -inf pattern differs"
    d = np.abs(np.where(both_inf, 0.0, np.where(both_inf, 0.0, g) - np.where(both_inf, 0.0, r)))
    err = d.max() if d.size else 0.0
    assert err <= LSE_ABS, "%s: max abs err %.3e > %.0e" % (what, err, LSE_ABS)
    return err


def np_inputs(inp: dict) -> dict:
    return {k: to64(v) for k, v in inp.items()}
