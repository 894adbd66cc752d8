"""The Python binding checks its tensor arguments before it calls the library: the
kernels dereference every pointer on the GPU and read exactly the sizes and dtypes the
C ABI's layouts state, so host tensors, mixed dtypes or wrong sizes must be refused up
front rather than read out of bounds.  These run without a GPU."""
import pytest
import torch

from head_latent_attention_rmsnorm_gb300 import configs, inputs, mla

CFG = configs.TINY


def host_prefill():
    t = inputs.prefill_inputs(CFG)
    return mla.dims_of(CFG), t


def host_decode():
    dcfg = configs.Decode("dec_small", "f32", batch=2, kv_len=40, n_splits=2, n_heads=4, d_kv=64, d_nope=32,
                          d_rope=16, d_v=32)
    d = mla.dims(dcfg.n_heads, dcfg.d_kv, dcfg.d_nope, dcfg.d_rope, dcfg.d_v)
    return d, inputs.decode_inputs(dcfg)


def test_prefill_wrappers_refuse_host_tensors():
    d, t = host_prefill()
    args = (t["q_nope"], t["q_pe"], t["c_kv"], t["k_pe"], t["w_kv_b"], t["rms_w"])
    for fn in (mla.latent_attn_fwd, mla.absorbed_attn_fwd, mla.latent_attn_fused_fwd):
        with pytest.raises(ValueError, match="CUDA device"):
            fn(d, *args)
    out = torch.zeros(1, CFG.s_q, CFG.n_heads, CFG.d_v)
    lse = torch.zeros(1, CFG.n_heads, CFG.s_q)
    with pytest.raises(ValueError, match="CUDA device"):
        mla.latent_attn_bwd(d, *args, out, lse, out)


def test_decode_wrappers_refuse_host_tensors():
    d, t = host_decode()
    args = (t["q_nope"], t["q_pe"], t["c_cache"], t["kpe_cache"], t["w_kv_b"])
    with pytest.raises(ValueError, match="CUDA device"):
        mla.decode_splitkv(d, *args, n_splits=2)
    with pytest.raises(ValueError, match="CUDA device"):
        mla.tpla_decode(d, *args, n_shards=2, n_splits=2)


def test_row_wrappers_refuse_host_tensors():
    x = torch.zeros(8, 64)
    w = torch.ones(64)
    with pytest.raises(ValueError, match="CUDA device"):
        mla.rmsnorm(x, w)
    with pytest.raises(ValueError, match="CUDA device"):
        mla.rmsnorm_bwd(x, w, x)
    with pytest.raises(ValueError, match="CUDA device"):
        mla.lse_combine(torch.zeros(2, 8, 64), torch.zeros(2, 8))


def test_tensor_check():
    cpu = torch.device("cpu")
    x = torch.zeros(4, 6)
    mla._expect("x", x, 24, torch.float32, cpu)                  # passes
    mla._expect("x", None, 24, torch.float32, cpu)               # optional argument absent
    with pytest.raises(TypeError, match="dtype"):
        mla._expect("x", x.to(torch.bfloat16), 24, torch.float32, cpu)
    with pytest.raises(ValueError, match="elements"):
        mla._expect("x", x, 25, torch.float32, cpu)
    with pytest.raises(ValueError, match="contiguous"):
        mla._expect("x", x.t(), 24, torch.float32, cpu)
    with pytest.raises(ValueError, match="on meta"):
        mla._expect("x", torch.zeros(4, 6, device="meta"), 24, torch.float32, cpu)
    with pytest.raises(TypeError, match="torch.Tensor"):
        mla._expect("x", [0.0] * 24, 24, torch.float32, cpu)
