"""The multi-rank partitioning on CPU: two gloo ranks, oracle arithmetic.

Each rank takes its block of query positions (LAGA sequence-parallel view), of heads
(head-parallel view) or of decode key splits (Helix KV-parallel view) with
`sharding`, computes it with the oracle, and the blocks are exchanged with
all_gather; the concatenation (or the log-sum-exp merge of the split partials) must
equal the single-process result.  A TPLA rank decodes with its latent shard (its own
RMSNorm, local softmax, its slice of W_kv_b), and the all-reduced sum must equal the
two-shard TPLA decode.  In the backward, each sequence-parallel rank's latent, RoPE
band and weight gradients are all-reduced and must equal one call's, with the query
gradients reassembling by rows.  Also checks the max-over-ranks timing reduction the
benchmark uses.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs():
    g = np.random.default_rng(3)
    B, S, H, dk, dn, dr, dv = 1, 40, 4, 32, 16, 8, 16
    return dict(q_nope=g.standard_normal((B, S, H, dn)), q_pe=g.standard_normal((B, S, H, dr)),
                c_kv=g.standard_normal((B, S, dk)), k_pe=g.standard_normal((B, S, dr)),
                w_kv_b=g.standard_normal((H * (dn + dv), dk)) / np.sqrt(dk), rms_w=np.ones(dk)), H


def _worker(rank, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    from head_latent_attention_rmsnorm_gb300 import sharding
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        inp, H = _inputs()
        S = inp["c_kv"].shape[1]
        # sequence-parallel rank: a block of query rows over the full latent
        q0, n = sharding.query_shard(S, WORLD, rank)
        part = dict(inp, q_nope=inp["q_nope"][:, q0:q0 + n], q_pe=inp["q_pe"][:, q0:q0 + n])
        o, l = oracle.mla_explicit(**part, n_heads=H, q_offset=q0)
        outs = [None] * WORLD
        dist.all_gather_object(outs, (q0, o, l))
        # head-parallel rank
        h0, hc = sharding.head_shard(H, WORLD, rank)
        part = dict(inp, q_nope=inp["q_nope"][:, :, h0:h0 + hc], q_pe=inp["q_pe"][:, :, h0:h0 + hc])
        ho, hl = oracle.mla_explicit(**part, n_heads=H, head_begin=h0)
        houts = [None] * WORLD
        dist.all_gather_object(houts, (h0, ho, hl))
        # KV-parallel decode: each rank owns a block of the splits
        cache = oracle.rmsnorm(inp["c_kv"], inp["rms_w"], 1e-6)
        kpe = oracle.rope(inp["k_pe"], np.arange(S)[None, :].astype(float), 10000.0)
        n_splits = 5
        _, _, po, pl = oracle.mla_decode(inp["q_nope"][:, -1], inp["q_pe"][:, -1], cache, kpe, inp["w_kv_b"],
                                         n_splits=n_splits)
        s0, sc = sharding.split_shard(n_splits, WORLD, rank)
        parts = [None] * WORLD
        dist.all_gather_object(parts, (po[s0:s0 + sc], pl[s0:s0 + sc]))
        # TPLA tensor-parallel rank: its latent shard, every head; outputs all-reduced
        k0, kd = sharding.latent_shard(inp["c_kv"].shape[-1], WORLD, rank)
        sl = slice(k0, k0 + kd)
        to, _ = oracle.tpla_decode(inp["q_nope"][:, -1], inp["q_pe"][:, -1],
                                   np.ascontiguousarray(inp["c_kv"][..., sl]), kpe,
                                   np.ascontiguousarray(inp["w_kv_b"][:, sl]), 1.0 + 0.1 * np.arange(kd) / kd,
                                   shards=1, scale=oracle.default_scale(inp["q_nope"].shape[-1], kpe.shape[-1]))
        tsum = torch.from_numpy(np.ascontiguousarray(to))
        dist.all_reduce(tsum, op=dist.ReduceOp.SUM)
        t = torch.tensor([float(rank + 1)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            q.put((outs, houts, parts, t.item(), tsum.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_partitions_reassemble(oracle):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    outs, houts, parts, tmax, tpla_sum = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    inp, H = _inputs()
    full_o, full_l = oracle.mla_explicit(**inp, n_heads=H)
    o = np.concatenate([x[1] for x in sorted(outs, key=lambda x: x[0])], 1)
    l = np.concatenate([x[2] for x in sorted(outs, key=lambda x: x[0])], 2)
    np.testing.assert_array_equal(o, full_o)
    np.testing.assert_array_equal(l, full_l)
    ho = np.concatenate([x[1] for x in sorted(houts, key=lambda x: x[0])], 2)
    np.testing.assert_array_equal(ho, full_o)
    S = inp["c_kv"].shape[1]
    cache = oracle.rmsnorm(inp["c_kv"], inp["rms_w"], 1e-6)
    kpe = oracle.rope(inp["k_pe"], np.arange(S)[None, :].astype(float), 10000.0)
    do, dl, _, _ = oracle.mla_decode(inp["q_nope"][:, -1], inp["q_pe"][:, -1], cache, kpe, inp["w_kv_b"], n_splits=1)
    po = np.concatenate([p[0] for p in parts], 0)
    pl = np.concatenate([p[1] for p in parts], 0)
    n = po.shape[0]
    o_lat, lse = oracle.lse_combine(po.reshape(n, -1, po.shape[-1]), pl.reshape(n, -1))
    np.testing.assert_allclose(lse.reshape(dl.shape), dl, rtol=0, atol=1e-12)
    dk, dn = inp["c_kv"].shape[-1], inp["q_nope"].shape[-1]
    W = inp["w_kv_b"].reshape(H, -1, dk)[:, dn:]
    out = np.einsum("hdk,bhk->bhd", W, o_lat.reshape(1, H, dk))
    np.testing.assert_allclose(out, do, rtol=0, atol=1e-12)
    assert tmax == float(WORLD)
    # the all-reduced TPLA rank outputs = the two-shard TPLA decode (norm weight as the ranks drew it)
    dkv = inp["c_kv"].shape[-1]
    w_norm = np.concatenate([1.0 + 0.1 * np.arange(dkv // WORLD) / (dkv // WORLD)] * WORLD)
    ref, _ = oracle.tpla_decode(inp["q_nope"][:, -1], inp["q_pe"][:, -1], inp["c_kv"], kpe, inp["w_kv_b"], w_norm,
                                shards=WORLD)
    np.testing.assert_allclose(tpla_sum, ref, rtol=0, atol=1e-12)


def test_block_partition_covers_exactly():
    from head_latent_attention_rmsnorm_gb300 import sharding
    for n in (0, 1, 7, 128, 16384):
        for world in (1, 2, 3, 8):
            covered = []
            for r in range(world):
                b, c = sharding.block(n, world, r)
                covered.extend(range(b, b + c))
            assert covered == list(range(n))


def test_latent_shard_needs_even_split():
    from head_latent_attention_rmsnorm_gb300 import sharding
    assert [sharding.latent_shard(512, 2, r) for r in range(2)] == [(0, 256), (256, 256)]
    with pytest.raises(ValueError):
        sharding.latent_shard(512, 3, 0)


def _bwd_inputs():
    g = np.random.default_rng(5)
    B, S, H, dk, dn, dr, dv = 1, 24, 3, 16, 8, 4, 8
    inp = dict(q_nope=g.standard_normal((B, S, H, dn)), q_pe=g.standard_normal((B, S, H, dr)),
               c_kv=g.standard_normal((B, S, dk)), k_pe=g.standard_normal((B, S, dr)),
               w_kv_b=g.standard_normal((H * (dn + dv), dk)) / np.sqrt(dk), rms_w=1.0 + 0.2 * g.standard_normal(dk))
    return inp, g.standard_normal((B, S, H, dv)), H


def _bwd_worker(rank, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    from head_latent_attention_rmsnorm_gb300 import sharding
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        inp, dout, H = _bwd_inputs()
        S = inp["c_kv"].shape[1]
        q0, n = sharding.query_shard(S, WORLD, rank)
        part = dict(inp, q_nope=inp["q_nope"][:, q0:q0 + n].copy(), q_pe=inp["q_pe"][:, q0:q0 + n].copy())
        g = oracle.mla_explicit_bwd(**part, dout=dout[:, q0:q0 + n].copy(), n_heads=H, q_offset=q0)
        # the gradients of what every rank shares (the gathered latent, its RoPE band, the
        # weights) are summed over the ranks: the reduce-scatter / all-reduce that mirrors
        # the forward's all-gather; the query gradients stay with their rank's rows
        summed = {}
        for k in ("c_kv", "k_pe", "w_kv_b", "rms_w"):
            t = torch.from_numpy(np.ascontiguousarray(g[k]))
            dist.all_reduce(t, op=dist.ReduceOp.SUM)
            summed[k] = t.numpy()
        rows = [None] * WORLD
        dist.all_gather_object(rows, (q0, g["q_nope"], g["q_pe"]))
        if rank == 0:
            q.put((summed, rows))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_backward_gradients_sum_to_one_call(oracle):
    """LAGA, "If this is right": sequence-parallel ranks give the gradients of one call.
    Two gloo ranks each back-propagate their block of query rows; the summed latent, RoPE
    band and weight gradients equal one call's, and the query gradients reassemble."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bwd_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    summed, rows = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    inp, dout, H = _bwd_inputs()
    full = oracle.mla_explicit_bwd(**inp, dout=dout, n_heads=H)
    for k in ("c_kv", "k_pe", "w_kv_b", "rms_w"):
        np.testing.assert_allclose(summed[k], full[k], rtol=0, atol=1e-12 * max(1.0, np.abs(full[k]).max()),
                                   err_msg=k)
    rows = sorted(rows, key=lambda x: x[0])
    np.testing.assert_array_equal(np.concatenate([r[1] for r in rows], 1), full["q_nope"])
    np.testing.assert_array_equal(np.concatenate([r[2] for r in rows], 1), full["q_pe"])
