"""The five workloads of this library, as plain data (no arithmetic).

Dimensions follow the LAGA page (DeepSeek-V3: n_h=128, d_kv=512, per-head K/V
128+128, RoPE band 64 -- "What carries the argument") and the TPLA page's decode
regime (32K context, 576-dim latent per token -- "If this is right").
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Prefill:
    name: str
    dtype: str            # "f32" | "bf16"
    batch: int
    s_kv: int             # tokens in the (gathered) latent
    s_q: int              # query rows of this call
    q_offset: int         # absolute position of query row 0
    n_heads: int
    d_kv: int
    d_nope: int
    d_rope: int
    d_v: int
    head_shard: int
    causal: bool = True
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    sweep_offsets: tuple = field(default_factory=tuple)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def pairs(self) -> int:
        """Visible (query, key) pairs per (batch, head): the causal work."""
        if not self.causal:
            return self.s_q * self.s_kv
        return sum(min(self.q_offset + i + 1, self.s_kv) for i in range(self.s_q))

    def kv_needed(self) -> int:
        return min(self.q_offset + self.s_q, self.s_kv) if self.causal else self.s_kv

    def flops(self) -> dict:
        """Algorithmic FLOPs of one explicit call (masked pairs excluded)."""
        dqk = self.d_nope + self.d_rope
        attn = self.batch * self.n_heads * self.pairs() * 2 * (dqk + self.d_v)
        recon = 2 * self.batch * self.kv_needed() * self.d_kv * self.n_heads * (self.d_nope + self.d_v)
        return {"attention": attn, "reconstruct": recon, "total": attn + recon}

    def backward_flops(self) -> dict:
        """Algorithmic FLOPs of one backward call (masked pairs excluded), without the
        recomputation an implementation chooses: per visible pair and head dV = P^T dO and
        dP = dO V^T (2 d_v each), dQ = dS K and dK = dS^T Q (2 (d_nope + d_rope) each); per
        key and head the weight gradient dW = dKV^T chat and the latent gradient
        dchat = dKV W (2 d_kv (d_nope + d_v) each)."""
        dqk = self.d_nope + self.d_rope
        pairs = self.batch * self.n_heads * self.pairs()
        attn = pairs * 2 * (2 * self.d_v + 2 * dqk)
        recon = 2 * (2 * self.batch * self.kv_needed() * self.d_kv * self.n_heads * (self.d_nope + self.d_v))
        return {"attention": attn, "reconstruct": recon, "dkv_kernel": pairs * 2 * (self.d_v + dqk),
                "dq_kernel": pairs * 2 * dqk, "total": attn + recon}

    def absorbed_flops(self) -> dict:
        """Algorithmic FLOPs of one absorbed-form call: latent-space attention over
        d_kv + d_rope score dims and d_kv value dims, plus the absorb (q_nope -> q_abs) and
        un-absorb (o_lat -> out) products."""
        attn = self.batch * self.n_heads * self.pairs() * 2 * ((self.d_kv + self.d_rope) + self.d_kv)
        rows = self.batch * self.s_q * self.n_heads
        absorb = 2 * rows * self.d_nope * self.d_kv
        unabsorb = 2 * rows * self.d_kv * self.d_v
        return {"attention": attn, "absorb": absorb, "unabsorb": unabsorb, "total": attn + absorb + unabsorb}

    def activation_bytes(self, absorbed: bool, head_shard: int) -> dict:
        """Closed form of the per-call intermediates a caller allocates (outputs + the
        workspace the library asks for), in bytes, at the tensor-core path's storage
        (16-bit intermediates).  The head-dependent part is what separates the two forms
        (the LAGA page's per-token footprint: n_h (d_nope + d_v) against n_h d_kv):
        explicit K_nope and V^T of one head shard, absorbed q_abs and o_lat of one; with
        head_shard = 0 the fused explicit form, which keeps no K/V at all."""
        kv_pad = (self.kv_needed() + 127) // 128 * 128
        rows = self.batch * self.s_q
        out = rows * self.n_heads * self.d_v * 2 + rows * self.n_heads * 4
        positions = max(self.kv_needed(), self.q_offset + self.s_q)
        common = (self.batch * kv_pad * (self.d_kv + self.d_rope) * 2 + rows * self.n_heads * self.d_rope * 2
                  + positions * (self.d_rope // 2) * 8)   # normalised latent, rotated bands, RoPE table
        if absorbed:
            w16 = head_shard * (self.d_nope + self.d_v) * self.d_kv * 2
            shard = 2 * rows * head_shard * self.d_kv * 2
        else:
            w16 = self.n_heads * (self.d_nope + self.d_v) * self.d_kv * 2
            shard = self.batch * head_shard * kv_pad * (self.d_nope + self.d_v) * 2
        return {"outputs": out, "common": common, "w16": w16, "per_shard": shard,
                "total": out + common + w16 + shard}


@dataclass(frozen=True)
class Decode:
    name: str
    dtype: str
    batch: int
    kv_len: int
    n_splits: int
    n_heads: int
    d_kv: int
    d_nope: int
    d_rope: int
    d_v: int
    rope_base: float = 10000.0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def cache_bytes(self) -> int:
        el = 4 if self.dtype == "f32" else 2
        return self.batch * self.kv_len * (self.d_kv + self.d_rope) * el

    def algorithmic_bytes(self) -> int:
        """Bytes one decode call must move at least: the latent cache, W_kv_b, q in, out."""
        el = 4 if self.dtype == "f32" else 2
        w = self.n_heads * (self.d_nope + self.d_v) * self.d_kv * el
        q = self.batch * self.n_heads * (self.d_nope + self.d_rope) * el
        o = self.batch * self.n_heads * self.d_v * el + self.batch * self.n_heads * 4
        return self.cache_bytes() + w + q + o

    def flops(self) -> int:
        att = self.batch * self.n_heads * self.kv_len * 2 * ((self.d_kv + self.d_rope) + self.d_kv)
        absorb = 2 * self.batch * self.n_heads * self.d_nope * self.d_kv
        unabsorb = 2 * self.batch * self.n_heads * self.d_kv * self.d_v
        return att + absorb + unabsorb


TINY = Prefill("tiny_fp32", "f32", batch=1, s_kv=128, s_q=128, q_offset=0, n_heads=4, d_kv=64,
               d_nope=32, d_rope=16, d_v=32, head_shard=2, sweep_offsets=(0, 64))
V2LITE = Prefill("v2lite_prefill_s4096_h16", "bf16", batch=1, s_kv=4096, s_q=4096, q_offset=0,
                 n_heads=16, d_kv=512, d_nope=128, d_rope=64, d_v=128, head_shard=16)
V3 = Prefill("v3_prefill_s4096_h128", "bf16", batch=1, s_kv=4096, s_q=4096, q_offset=0,
             n_heads=128, d_kv=512, d_nope=128, d_rope=64, d_v=128, head_shard=16)
SP8_RANK7 = Prefill("v3_sp8_rank7_skv16384_q2048", "bf16", batch=1, s_kv=16384, s_q=2048,
                    q_offset=14336, n_heads=128, d_kv=512, d_nope=128, d_rope=64, d_v=128,
                    head_shard=16, sweep_offsets=tuple(2048 * r for r in range(8)))
DECODE = Decode("v3_decode_b64_l32768_split8", "bf16", batch=64, kv_len=32768, n_splits=8,
                n_heads=128, d_kv=512, d_nope=128, d_rope=64, d_v=128)

ALL = {c.name: c for c in (TINY, V2LITE, V3, SP8_RANK7, DECODE)}
