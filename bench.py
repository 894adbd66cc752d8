#!/usr/bin/env python3
"""Benchmark of MLA attention from the compressed latent on GB300.

One step = one explicit (LAGA per-rank) prefill call on the largest single-GPU
prefill workload: the simulated sequence-parallel rank 7 of 8 on DeepSeek-V3 dims
(bf16, 16384 gathered latent rows + k_pe, the last 2048 query rows at offset 14336,
128 heads rebuilt in head shards of 16, causal).  The headline ``value`` is its
TFLOP/s (algorithmic FLOPs: visible causal pairs x 2 x (192 + 128) per head plus the
K/V reconstruction GEMM), timed per call with CUDA events on the launching stream,
a 256 MB buffer written between timed calls; ``roofline`` is the attention kernel's,
``e2e`` the same call with its inputs copied from pinned host memory and its outputs
copied back inside every timed step (uploads and downloads on streams of their own,
overlapping the neighbouring steps' calls; the serial form beside it), ``cpu_baseline`` the fp64 oracle on a sample of
the same workload on the host's cores.  After the headline, rank 0 at N = 1 also
times, with the same step count, the V2-Lite and V3-shaped prefills, the V3 absorbed
form (``other_prefill_configs``), the split-KV decode (``decode``: HBM GB/s), the TPLA
decode, and measures the allocator's peak memory of the explicit against the
absorbed form beside its closed form (``activation_memory``); --no-extras skips them.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own copy of the workload (independent problems,
no collective on the data path: weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA prefill fwd TFLOP/s (% of BF16 peak); decode HBM GB/s (% of 8 TB/s)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12   # SMs x FP32 lanes x FMA x max clock
# DRAM bytes (read + write) per launch of the dominant kernels, keyed by (kernel,
# workload, absorbed), from the ncu captures summarised under profiles/ (absent until the
# current kernel has been captured on that workload).  The decode capture runs B = 8; its
# traffic grows in proportion to the batch, so the B = 64 launch is 8x that.
NCU_TRAFFIC = {("tc_attn", "v2lite_prefill_s4096_h16", False): 61.52e6,
               ("tc_attn", "v3_sp8_rank7_skv16384_q2048", False): 282.72e6,
               ("tc_fused_attn", "v2lite_prefill_s4096_h16", True): 34.19e6,
               ("tc_decode_attn", "v3_decode_b64_l32768_split8", False): 313.52e6 * 8}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks ----
class ClockSampler:
    """Polls SM clock and clock-event reasons through NVML (read-only queries)."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        self.samples, self.max_mhz, self.ok = [], None, False
        self._stop = threading.Event()
        try:
            import torch
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            props = torch.cuda.get_device_properties(device_index)
            bus = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id, props.pci_device_id)
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(h)) != 0:
                    return
            self.nv, self.h = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0 and \
                    self._reasons_fn(self.h, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(0.005)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "note": "NVML unavailable"}
        mhz = [s[0] for s in self.samples]
        seen = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    seen.add(name)
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": sorted(seen),
                "samples": len(self.samples)}


# ----------------------------------------------------------------- helpers ----
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], device="cuda", dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def randn(shape, std, dtype, g):
    import torch
    return (torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) * std).to(dtype)


def prefill_setup(cfg, seed=0, absorbed=False, fused=False):
    import torch
    from head_latent_attention_rmsnorm_gb300 import mla
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    dt = cfg.torch_dtype
    B, S, H = cfg.batch, cfg.s_q, cfg.n_heads
    t = dict(q_nope=randn((B, S, H, cfg.d_nope), 1.0, dt, g), q_pe=randn((B, S, H, cfg.d_rope), 1.0, dt, g),
             c_kv=randn((B, cfg.s_kv, cfg.d_kv), 1.0, dt, g), k_pe=randn((B, cfg.s_kv, cfg.d_rope), 1.0, dt, g),
             w_kv_b=randn((H * (cfg.d_nope + cfg.d_v), cfg.d_kv), cfg.d_kv ** -0.5, dt, g),
             rms_w=torch.ones(cfg.d_kv, dtype=dt, device="cuda"))
    d = mla.dims_of(cfg)
    out = torch.empty(B, S, H, cfg.d_v, dtype=dt, device="cuda")
    lse = torch.empty(B, H, S, dtype=torch.float32, device="cuda")
    if fused:
        nbytes = mla.mla_latent_attn_fused_workspace(ctypes.byref(d), 1 if dt == torch.bfloat16 else 0, B, S,
                                                     cfg.s_kv, cfg.q_offset, int(cfg.causal), H)
    else:
        wsq = mla.mla_absorbed_attn_workspace if absorbed else mla.mla_latent_attn_workspace
        nbytes = wsq(ctypes.byref(d), 1 if dt == torch.bfloat16 else 0, B, S, cfg.s_kv, cfg.q_offset,
                     int(cfg.causal), H, cfg.head_shard)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    return d, t, out, lse, ws


def prefill_call(cfg, d, t, out, lse, ws, stream, absorbed=False, fused=False):
    from head_latent_attention_rmsnorm_gb300 import mla
    if fused:
        st = mla.lib().mla_latent_attn_fused_fwd(
            ctypes.byref(d), mla.MLA_BF16 if cfg.dtype == "bf16" else mla.MLA_F32, cfg.batch, cfg.s_q, cfg.s_kv,
            cfg.q_offset, int(cfg.causal), 0, cfg.n_heads, t["q_nope"].data_ptr(), t["q_pe"].data_ptr(),
            t["c_kv"].data_ptr(), t["k_pe"].data_ptr(), t["w_kv_b"].data_ptr(), t["rms_w"].data_ptr(), out.data_ptr(),
            lse.data_ptr(), ws.data_ptr(), ws.numel(), stream)
        if st != 0:
            raise RuntimeError("mla_latent_attn_fused_fwd: " + mla.mla_status_string(st))
        return
    f = mla.lib().mla_absorbed_attn_fwd if absorbed else mla.lib().mla_latent_attn_fwd
    st = f(ctypes.byref(d), mla.MLA_BF16 if cfg.dtype == "bf16" else mla.MLA_F32, cfg.batch, cfg.s_q, cfg.s_kv,
           cfg.q_offset, int(cfg.causal), 0, cfg.n_heads, cfg.head_shard, t["q_nope"].data_ptr(), t["q_pe"].data_ptr(),
           t["c_kv"].data_ptr(), t["k_pe"].data_ptr(), t["w_kv_b"].data_ptr(), t["rms_w"].data_ptr(), out.data_ptr(),
           lse.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    if st != 0:
        raise RuntimeError(("mla_absorbed_attn_fwd: " if absorbed else "mla_latent_attn_fwd: ") +
                           mla.mla_status_string(st))


def decode_setup(cfg, seed=1):
    import torch
    from head_latent_attention_rmsnorm_gb300 import mla
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    dt = cfg.torch_dtype
    B, H, L = cfg.batch, cfg.n_heads, cfg.kv_len
    t = dict(q_nope=randn((B, H, cfg.d_nope), 1.0, dt, g), q_pe=randn((B, H, cfg.d_rope), 1.0, dt, g),
             c_cache=randn((B, L, cfg.d_kv), 1.0, dt, g), kpe_cache=randn((B, L, cfg.d_rope), 1.0, dt, g),
             w_kv_b=randn((H * (cfg.d_nope + cfg.d_v), cfg.d_kv), cfg.d_kv ** -0.5, dt, g))
    d = mla.dims(cfg.n_heads, cfg.d_kv, cfg.d_nope, cfg.d_rope, cfg.d_v, cfg.rope_base)
    out = torch.empty(B, H, cfg.d_v, dtype=dt, device="cuda")
    lse = torch.empty(B, H, dtype=torch.float32, device="cuda")
    nbytes = mla.mla_decode_workspace(ctypes.byref(d), 1 if dt == torch.bfloat16 else 0, B, L, cfg.n_splits)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    return d, t, out, lse, ws


def decode_call(cfg, d, t, out, lse, ws, stream):
    from head_latent_attention_rmsnorm_gb300 import mla
    st = mla.lib().mla_decode_splitkv(ctypes.byref(d), mla.MLA_BF16 if cfg.dtype == "bf16" else mla.MLA_F32,
                                      cfg.batch, cfg.kv_len, cfg.n_splits, t["q_nope"].data_ptr(),
                                      t["q_pe"].data_ptr(), t["c_cache"].data_ptr(), t["kpe_cache"].data_ptr(),
                                      t["w_kv_b"].data_ptr(), out.data_ptr(), lse.data_ptr(), None, None,
                                      ws.data_ptr(), ws.numel(), stream)
    if st != 0:
        raise RuntimeError("mla_decode_splitkv: " + mla.mla_status_string(st))


def tpla_setup(cfg, n_shards, seed=1):
    """The decode workload with its latent cache normalised per shard (the cache write of
    a TPLA deployment) and a workspace for the TPLA decode over ``n_shards`` shards."""
    import torch
    from head_latent_attention_rmsnorm_gb300 import inputs, mla
    d, t, out, _, _ = decode_setup(cfg, seed)
    dt = cfg.torch_dtype
    w = inputs.norm_weight(cfg.d_kv, dt).cuda()
    t["c_raw"], t["norm_w"] = t["c_cache"], w
    t["c_cache"] = mla.rmsnorm(t["c_raw"], w, n_shards=n_shards)
    slse = torch.empty(n_shards, cfg.batch, cfg.n_heads, dtype=torch.float32, device="cuda")
    nbytes = mla.mla_tpla_decode_workspace(ctypes.byref(d), mla.MLA_BF16 if cfg.dtype == "bf16" else mla.MLA_F32,
                                           cfg.batch, cfg.kv_len, cfg.n_splits, n_shards)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    return d, t, out, slse, ws


def tpla_call(cfg, n_shards, d, t, out, slse, ws, stream):
    from head_latent_attention_rmsnorm_gb300 import mla
    st = mla.lib().mla_tpla_decode(ctypes.byref(d), mla.MLA_BF16 if cfg.dtype == "bf16" else mla.MLA_F32,
                                   cfg.batch, cfg.kv_len, cfg.n_splits, n_shards, t["q_nope"].data_ptr(),
                                   t["q_pe"].data_ptr(), t["c_cache"].data_ptr(), t["kpe_cache"].data_ptr(),
                                   t["w_kv_b"].data_ptr(), out.data_ptr(), slse.data_ptr(), ws.data_ptr(),
                                   ws.numel(), stream)
    if st != 0:
        raise RuntimeError("mla_tpla_decode: " + mla.mla_status_string(st))


def tpla_extra(dcfg, stream, hbm_peak, n_shards=2, steps=10, warmup=3):
    """TPLA decode (latent cut into two shards, each attended by all heads with its own
    softmax, outputs summed) on the decode workload, and the per-shard RMSNorm that
    writes its cache, timed over the whole cache: reported beside the headline."""
    import torch
    from head_latent_attention_rmsnorm_gb300 import mla
    d, t, out, slse, ws = tpla_setup(dcfg, n_shards)
    fn = lambda: tpla_call(dcfg, n_shards, d, t, out, slse, ws, stream)  # noqa: E731
    ms = statistics.mean(timed(fn, steps, warmup, 1))
    nbytes = dcfg.algorithmic_bytes()
    normed = torch.empty_like(t["c_raw"])
    nfn = lambda: mla.rmsnorm(t["c_raw"], t["norm_w"], n_shards=n_shards, out=normed)  # noqa: E731
    n_ms = statistics.mean(timed(nfn, steps, warmup, 1))
    n_bytes = 2 * t["c_raw"].numel() * t["c_raw"].element_size() + t["norm_w"].numel() * 2
    # its backward over the same rows (x, dy read; dx written)
    dw = torch.empty(dcfg.d_kv, dtype=torch.float32, device="cuda")
    bws = torch.empty(mla.mla_rmsnorm_bwd_workspace(mla.MLA_BF16, t["c_raw"].numel() // dcfg.d_kv, dcfg.d_kv,
                                                    n_shards), dtype=torch.uint8, device="cuda")
    bfn = lambda: mla.rmsnorm_bwd(t["c_raw"], t["norm_w"], t["c_cache"], n_shards=n_shards, dx=normed, dw=dw,  # noqa: E731
                                  workspace=bws)
    b_ms = statistics.mean(timed(bfn, steps, warmup, 1))
    b_bytes = 3 * t["c_raw"].numel() * t["c_raw"].element_size()
    del dw, bws
    mla.profile_reset()
    mla.profile_enable(True)
    fn()
    prof = mla.profile_all()
    mla.profile_enable(False)
    path = mla.last_path()
    del d, t, out, slse, ws, normed
    torch.cuda.empty_cache()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": dcfg.name + "_tpla%d" % n_shards, "n_shards": n_shards, "ms_per_call": round(ms, 4),
            "GB/s": round(gbs, 1), "bytes_per_call": nbytes, "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
            "kernel_path": path_name(path),
            "kernels": {k: {"launches": v[0], "ms": round(v[1], 4)} for k, v in prof.items()},
            "cache_rmsnorm": {"rows": dcfg.batch * dcfg.kv_len, "ms": round(n_ms, 4), "bytes": n_bytes,
                              "GB/s": round(n_bytes / (n_ms * 1e-3) / 1e9, 1),
                              "frac_of_measured_hbm": round(n_bytes / (n_ms * 1e-3) / 1e9 / hbm_peak, 4)},
            "cache_rmsnorm_bwd": {"rows": dcfg.batch * dcfg.kv_len, "ms": round(b_ms, 4), "bytes": b_bytes,
                                  "GB/s": round(b_bytes / (b_ms * 1e-3) / 1e9, 1),
                                  "frac_of_measured_hbm": round(b_bytes / (b_ms * 1e-3) / 1e9 / hbm_peak, 4)}}


def timed(fn, steps, warmup, world, flush=None):
    """Per-call CUDA-event times (ms) of `steps` calls after `warmup` calls."""
    import torch
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        if flush is not None:
            flush.zero_()
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for a, b in ev:
        if flush is not None:
            flush.zero_()
        a.record(s)
        fn()
        b.record(s)
    torch.cuda.synchronize()
    barrier(world)
    return [a.elapsed_time(b) for a, b in ev]


def path_name(path: int) -> str:
    """The kernel family the library reports for its last call (mla_last_path)."""
    from head_latent_attention_rmsnorm_gb300 import mla
    return {mla.PATH_SIMT: "simt", mla.PATH_TC: "tcgen05",
            mla.PATH_TC_FUSED: "tcgen05 fused"}.get(path, "?")


def dominant(prof: dict, candidates):
    best = None
    for k in candidates:
        if k in prof and (best is None or prof[k][1] > prof[best][1]):
            best = k
    return best


def prefill_measure(cfg, stream, steps, warmup, world, flush, peaks, peak_kind, absorbed=False, fused=False):
    """One prefill workload: per-call time of `steps` calls after `warmup` (L2 flushed
    between calls), then a second pass with a CUDA-event pair around every launch for
    the per-kernel split and the dominant kernel's roofline.  The fused form's FLOPs are
    counted as the explicit form's (the method's own work; its extra reconstructions are
    the kernel's overhead)."""
    from head_latent_attention_rmsnorm_gb300 import mla
    d, t, out, lse, ws = prefill_setup(cfg, absorbed=absorbed, fused=fused)
    fn = lambda: prefill_call(cfg, d, t, out, lse, ws, stream, absorbed=absorbed, fused=fused)  # noqa: E731
    fn()
    import torch
    torch.cuda.synchronize()
    path = mla.last_path()
    n0 = mla.launch_count()
    times = timed(fn, steps, warmup, world, flush)
    launches = (mla.launch_count() - n0) * steps // (steps + warmup)
    mla.profile_enable(True)
    mla.profile_reset()
    timed(fn, steps, warmup, world, flush)
    prof = mla.profile_all()
    mla.profile_enable(False)
    ms = max_over_ranks(statistics.mean(times), world)
    fl = cfg.absorbed_flops() if absorbed else cfg.flops()
    calls = steps + warmup
    kern = dominant(prof, ("tc_latent_attn", "attn_simt") if absorbed else
                    (("tc_fused_attn",) if fused else ("tc_attn", "attn_simt")))
    roof = None
    if kern:
        n, kms = prof[kern]
        # the fused kernel does the reconstruction too
        per_launch = (fl["total"] if fused else fl["attention"]) * calls / n
        ach = per_launch / (kms / n * 1e-3) / 1e12
        if kern.startswith("tc_"):
            peak, bound, note = peaks.get("bf16_tflops", 1900.0), "tensor", "bf16 dense burst, " + peak_kind
        else:
            peak, bound, note = FP32_ALU_TFLOPS, "alu", "fp32 FMA lanes x max clock (SIMT kernel)"
        roof = {"kernel": kern, "bound": bound, "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "traffic": NCU_TRAFFIC.get((kern, cfg.name, absorbed or fused)),
                "peak_kind": note, "launches": n, "avg_launch_us": round(kms / n * 1e3, 2),
                "flops_per_launch": per_launch,
                "share_of_step": round(kms / (sum(v[1] for v in prof.values()) or 1), 3)}
    form = "absorbed" if absorbed else ("fused" if fused else "explicit")
    res = {"workload": cfg.name + ("" if form == "explicit" else "_" + form), "form": form,
           "ms_per_call": round(ms, 4), "TFLOP/s": round(world * fl["total"] / (ms * 1e-3) / 1e12, 2),
           "frac_of_bf16_peak": round(fl["total"] / (ms * 1e-3) / 1e12 / peaks.get("bf16_tflops", 1900.0), 4),
           "flops_per_call": fl["total"], "tokens_per_s": round(world * cfg.batch * cfg.s_q / (ms * 1e-3), 1),
           "head_shard": cfg.head_shard, "kernel_path": path_name(path),
           "steps": steps, "warmup": warmup, "gpu_launches": launches, "roofline": roof,
           "kernels": {k: {"launches": v[0], "ms": round(v[1], 4)} for k, v in prof.items()}}
    return res, (d, t, out, lse, ws, fn)


def decode_measure(dcfg, stream, steps, warmup, world, peaks, peak_kind):
    """The split-KV decode workload (inputs larger than L2): per-call time and the
    decode kernel's HBM roofline."""
    import torch
    from head_latent_attention_rmsnorm_gb300 import mla
    dd, dt_, dout, dlse, dws = decode_setup(dcfg)
    fn = lambda: decode_call(dcfg, dd, dt_, dout, dlse, dws, stream)  # noqa: E731
    fn()
    torch.cuda.synchronize()
    path = mla.last_path()
    times = timed(fn, steps, warmup, world)
    mla.profile_enable(True)
    mla.profile_reset()
    timed(fn, steps, warmup, world)
    prof = mla.profile_all()
    mla.profile_enable(False)
    ms = max_over_ranks(statistics.mean(times), world)
    dbytes = dcfg.algorithmic_bytes()
    gbs = world * dbytes / (ms * 1e-3) / 1e9
    calls = steps + warmup
    kd = dominant(prof, ("tc_decode_attn", "attn_simt"))
    droof = None
    hbm = peaks.get("hbm_gbs", 6800.0)
    if kd:
        n, kms = prof[kd]
        per_launch = dcfg.cache_bytes() * calls / n
        ach = per_launch / (kms / n * 1e-3) / 1e9
        droof = {"kernel": kd, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                 "frac": round(ach / hbm, 4), "traffic": NCU_TRAFFIC.get((kd, dcfg.name, False)),
                 "peak_kind": "copy bandwidth, " + peak_kind, "launches": n, "avg_launch_us": round(kms / n * 1e3, 2),
                 "bytes_per_launch": per_launch}
    del dd, dt_, dout, dlse, dws
    torch.cuda.empty_cache()
    return {"workload": dcfg.name, "value": round(gbs, 1), "unit": "GB/s", "ms_per_call": round(ms, 4),
            "bytes_per_call": dbytes, "frac_of_8TBps": round(gbs / world / 8000.0, 4),
            "frac_of_measured_hbm": round(gbs / world / hbm, 4),
            "tokens_per_s": round(world * dcfg.batch / (ms * 1e-3), 1), "steps": steps, "warmup": warmup,
            "kernel_path": path_name(path), "roofline": droof,
            "l2": "inputs (2.4 GB) larger than L2",
            "kernels": {k: {"launches": v[0], "ms": round(v[1], 4)} for k, v in prof.items()}}


def backward_measure(cfg, stream, steps, warmup, flush, peaks, peak_kind):
    """The backward call (mla_latent_attn_bwd) of workload `cfg` for a random upstream
    gradient, given the forward's out and lse: per-call time, the per-kernel split and the
    two attention-backward kernels' rooflines (their algorithmic FLOPs: dV + dK for the
    key-stationary kernel, dQ for the query-stationary one)."""
    import torch
    from head_latent_attention_rmsnorm_gb300 import mla
    d, t, out, lse, ws = prefill_setup(cfg)
    prefill_call(cfg, d, t, out, lse, ws, stream)
    del ws
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    dout = randn(out.shape, 1.0, out.dtype, g)
    grads = {"q_nope": torch.empty_like(t["q_nope"]), "q_pe": torch.empty_like(t["q_pe"]),
             "c_kv": torch.empty_like(t["c_kv"]), "k_pe": torch.empty_like(t["k_pe"]),
             "w_kv_b": torch.zeros(t["w_kv_b"].shape, dtype=torch.float32, device="cuda"),
             "rms_w": torch.empty(cfg.d_kv, dtype=torch.float32, device="cuda")}
    nbytes = mla.mla_latent_attn_bwd_workspace(ctypes.byref(d), mla.MLA_BF16, cfg.batch, cfg.s_q, cfg.s_kv,
                                               cfg.q_offset, int(cfg.causal), cfg.n_heads, cfg.head_shard)
    bws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def fn():
        mla.latent_attn_bwd(d, t["q_nope"], t["q_pe"], t["c_kv"], t["k_pe"], t["w_kv_b"], t["rms_w"], out, lse, dout,
                            q_offset=cfg.q_offset, causal=cfg.causal, head_shard=cfg.head_shard, grads=grads,
                            workspace=bws, stream=stream)
    fn()
    torch.cuda.synchronize()
    path = mla.last_path()
    times = timed(fn, steps, warmup, 1, flush)
    mla.profile_enable(True)
    mla.profile_reset()
    timed(fn, steps, warmup, 1, flush)
    prof = mla.profile_all()
    mla.profile_enable(False)
    ms = statistics.mean(times)
    fl = cfg.backward_flops()
    calls = steps + warmup
    roof = {}
    peak = peaks.get("bf16_tflops", 1900.0)
    for kern, key in (("tc_bwd_dkv", "dkv_kernel"), ("tc_bwd_dq", "dq_kernel")):
        if kern in prof:
            n, kms = prof[kern]
            per_launch = fl[key] * calls / n
            ach = per_launch / (kms / n * 1e-3) / 1e12
            roof[kern] = {"bound": "tensor", "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                          "frac": round(ach / peak, 4), "launches": n, "avg_launch_us": round(kms / n * 1e3, 2),
                          "flops_per_launch": per_launch, "peak_kind": "bf16 dense burst, " + peak_kind}
    del d, t, out, lse, dout, grads, bws
    torch.cuda.empty_cache()
    return {"workload": cfg.name + "_backward", "ms_per_call": round(ms, 4),
            "TFLOP/s": round(fl["total"] / (ms * 1e-3) / 1e12, 2),
            "frac_of_bf16_peak": round(fl["total"] / (ms * 1e-3) / 1e12 / peak, 4), "flops_per_call": fl["total"],
            "flops_counted": "dV, dP, dQ, dK per visible pair and head; dW and dchat per key and head (no recompute)",
            "kernel_path": path_name(path), "steps": steps, "warmup": warmup,
            "roofline": roof, "kernels": {k: {"launches": v[0], "ms": round(v[1], 4)} for k, v in prof.items()}}


def activation_memory():
    """Peak device memory the CUDA caching allocator sees for one prefill call (outputs +
    workspace), explicit against absorbed, at head shards of 16 and of all heads, on the
    V3-shaped prefill and the simulated SP=8 rank 7; each beside its closed form."""
    import torch
    from head_latent_attention_rmsnorm_gb300 import configs, mla
    res = {}
    for cfg in (configs.V3, configs.SP8_RANK7):
        d, t, _, _, _ = prefill_setup(cfg)
        r = {}
        for absorbed in (False, True):
            for hs in (16, cfg.n_heads):
                torch.cuda.synchronize()
                torch.cuda.empty_cache()
                base = torch.cuda.memory_allocated()
                torch.cuda.reset_peak_memory_stats()
                fn = mla.absorbed_attn_fwd if absorbed else mla.latent_attn_fwd
                o, l = fn(d, t["q_nope"], t["q_pe"], t["c_kv"], t["k_pe"], t["w_kv_b"], t["rms_w"], head_shard=hs,
                          q_offset=cfg.q_offset)
                torch.cuda.synchronize()
                key = "%s_hs%d" % ("absorbed" if absorbed else "explicit", hs)
                cf = cfg.activation_bytes(absorbed, hs)
                r[key + "_MB"] = round((torch.cuda.max_memory_allocated() - base) / 1e6, 1)
                r[key + "_closed_form_MB"] = round(cf["total"] / 1e6, 1)
                del o, l
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        o, l = mla.latent_attn_fused_fwd(d, t["q_nope"], t["q_pe"], t["c_kv"], t["k_pe"], t["w_kv_b"], t["rms_w"],
                                         q_offset=cfg.q_offset)
        torch.cuda.synchronize()
        r["fused_MB"] = round((torch.cuda.max_memory_allocated() - base) / 1e6, 1)
        cf = cfg.activation_bytes(False, 0)
        r["fused_closed_form_MB"] = round(cf["total"] / 1e6, 1)
        del o, l
        per_tok = {"explicit": cfg.n_heads * (cfg.d_nope + cfg.d_v) * 2, "absorbed": cfg.n_heads * 2 * cfg.d_kv * 2}
        r["per_token_head_bytes_all_heads"] = per_tok
        r["closed_form"] = ("outputs + normalised latent and rotated bands + RoPE table + fp16 W rows + "
                            "per shard: explicit K_nope,V^T = B*kv_pad*hs*(d_nope+d_v)*2; absorbed q_abs,o_lat = "
                            "2*B*s_q*hs*d_kv*2; fused: nothing per shard")
        res[cfg.name] = r
        del d, t
        torch.cuda.empty_cache()
    res["counts"] = "out + lse + workspace, torch.cuda.max_memory_allocated() minus the inputs"
    return res


def e2e_measure(cfg, bufs, steps, warmup, world):
    """The headline call end to end through the C ABI: every step copies the inputs from
    pinned host memory to the device, runs the call and copies out + lse back."""
    import torch
    d, t, out, lse, ws, fn = bufs
    host_in = {k: v.cpu().pin_memory() for k, v in t.items()}
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    host_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    def step():
        for k, v in host_in.items():
            t[k].copy_(v, non_blocking=True)
        fn()
        host_out.copy_(out, non_blocking=True)
        host_lse.copy_(lse, non_blocking=True)

    times = timed(step, steps, warmup, world)
    serial_ms = max_over_ranks(statistics.mean(times), world)
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * 4
    ms = max_over_ranks(e2e_pipelined(cfg, bufs, host_in, steps, warmup, world), world)
    flops = world * cfg.flops()["total"]
    return {"value": round(flops / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "steps": steps,
            "mode": "pipelined: two input and two output sets, uploads on one stream and downloads on "
                    "another, ordered by events, so step i+1's upload and step i-1's download run "
                    "beside step i's call; the region spans the first upload to the last download",
            "serial": {"value": round(flops / (serial_ms * 1e-3) / 1e12, 3), "ms_per_step": round(serial_ms, 4),
                       "mode": "upload, call and download one after another on the call's stream"}}


def e2e_pipelined(cfg, bufs, host_in, steps, warmup, world):
    """Mean ms per step of `steps` pipelined steps (after `warmup`), timed from an event
    before the first upload to one after the last download, on the call's stream."""
    import torch
    d, t, out, lse, ws, _ = bufs
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    sets = [(t, out, lse), ({k: torch.empty_like(v) for k, v in t.items()}, torch.empty_like(out),
                            torch.empty_like(lse))]
    h_out = [(torch.empty(out.shape, dtype=out.dtype).pin_memory(),
              torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for _ in range(2)]
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    stream = comp.cuda_stream

    def run(n, start_ev):
        up.wait_event(start_ev)
        down.wait_event(start_ev)
        for i in range(n):
            j = i & 1
            ti, oj, lj = sets[j]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(in_free[j])
                for k, v in host_in.items():
                    ti[k].copy_(v, non_blocking=True)
                in_ready[j].record(up)
            comp.wait_event(in_ready[j])
            if i >= 2:
                comp.wait_event(out_free[j])
            prefill_call(cfg, d, ti, oj, lj, ws, stream)
            in_free[j].record(comp)
            out_ready[j].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(out_ready[j])
                h_out[j][0].copy_(oj, non_blocking=True)
                h_out[j][1].copy_(lj, non_blocking=True)
                out_free[j].record(down)
        for j in range(min(n, 2)):
            comp.wait_event(out_free[j])

    s0 = torch.cuda.Event()
    s0.record(comp)
    run(warmup, s0)
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    run(steps, a)
    b.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    ok = torch.equal(h_out[(steps - 1) & 1][0].to(out.device), out) if steps >= 1 else True
    if not ok:
        raise RuntimeError("pipelined end-to-end output differs from the device-resident call's")
    return a.elapsed_time(b) / steps


# -------------------------------------------------------------- our arm ----
HEADLINE = "v3_sp8_rank7_skv16384_q2048"


def run_ours(args, world, rank, local):
    import torch
    from head_latent_attention_rmsnorm_gb300 import build as mla_build
    from head_latent_attention_rmsnorm_gb300 import configs, mla

    if rank == 0:
        mla_build.build()
    barrier(world)
    mla.lib()
    peaks, peak_kind = load_peaks()
    pcfg = configs.ALL[HEADLINE]
    stream = torch.cuda.current_stream().cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    steps, warmup = args.steps, args.warmup

    # ---- the headline: the simulated SP=8 rank 7 (the largest single-GPU prefill)
    with ClockSampler(local) as clk:
        head, bufs = prefill_measure(pcfg, stream, steps, warmup, world, flush, peaks, peak_kind)
    value = head["TFLOP/s"]
    p_ms = head["ms_per_call"]
    e2e = None
    try:
        with ClockSampler(local) as clk_e2e:
            e2e = e2e_measure(pcfg, bufs, max(1, min(steps, 20)), min(warmup, 3), world)
        e2e["clocks"] = clk_e2e.summary()
    except Exception as ex:  # keep the kernel numbers even if pinning fails
        e2e = {"value": None, "unit": "TFLOP/s", "error": str(ex)[:200]}
    del bufs
    torch.cuda.empty_cache()

    # ---- beside the headline, with the same step count: the other prefill workloads,
    # the absorbed form, the decode (rank 0 at N = 1 only, so replicas are not slowed)
    side, decode, mem, tpla = {}, None, None, None
    if rank == 0 and world == 1 and not args.no_extras:
        with ClockSampler(local) as clk_side:
            for cfg, absorbed, fused in ((configs.V2LITE, False, False), (configs.V3, False, False),
                                         (configs.V3, True, False), (configs.V2LITE, False, True),
                                         (configs.V3, False, True), (configs.SP8_RANK7, False, True)):
                r, bufs = prefill_measure(cfg, stream, steps, warmup, 1, flush, peaks, peak_kind, absorbed=absorbed,
                                          fused=fused)
                side[r["workload"]] = r
                del bufs
                torch.cuda.empty_cache()
            for cfg in (configs.V2LITE, configs.SP8_RANK7):
                r = backward_measure(cfg, stream, steps, warmup, flush, peaks, peak_kind)
                side[r["workload"]] = r
            del flush
            torch.cuda.empty_cache()
            decode = decode_measure(configs.DECODE, stream, steps, warmup, 1, peaks, peak_kind)
        side["clocks"] = clk_side.summary()
        mem = activation_memory()
        tpla = tpla_extra(configs.DECODE, stream, peaks.get("hbm_gbs", 6800.0))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_headline()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(p_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded torch.randn, N(0,1); W_kv_b N(0,1/512))",
        "config": {"workload": pcfg.name, "batch": pcfg.batch, "seq_len_kv": pcfg.s_kv, "query_rows": pcfg.s_q,
                   "q_offset": pcfg.q_offset, "n_heads": pcfg.n_heads, "head_shard": pcfg.head_shard,
                   "causal": True, "flops_per_step": pcfg.flops()["total"],
                   "l2": "256 MB buffer written between timed calls",
                   "kernel_path": head["kernel_path"], "parallelism": "replicas" if world > 1 else "single"},
        "frac_of_bf16_peak": head["frac_of_bf16_peak"],
        "tokens_per_s": head["tokens_per_s"],
        "clocks": clk.summary(),
        "e2e": e2e,
        "gpu_launches": head["gpu_launches"],
        "roofline": head["roofline"],
        "cpu_baseline": cpu,
        "kernels_prefill": head["kernels"],
        "decode": decode,
        "other_prefill_configs": side or None,
        "tpla_decode": tpla,
        "activation_memory": mem,
        "peaks": {"kind": peak_kind, "hbm_gbs": peaks.get("hbm_gbs"), "bf16_tflops": peaks.get("bf16_tflops")},
    }
    print(json.dumps(line), flush=True)


def run_case(args):
    """Only `warmup + steps` calls of one workload, no timing or report: the target of
    ncu captures.  --only prefill|backward|decode|tpla; --workload picks a prefill config by
    name (backward: one forward call, then the backward calls)."""
    import torch
    from head_latent_attention_rmsnorm_gb300 import build as mla_build
    from head_latent_attention_rmsnorm_gb300 import configs, mla
    mla_build.build()
    mla.lib()
    stream = torch.cuda.current_stream().cuda_stream
    if args.only == "prefill":
        cfg = configs.ALL[args.workload] if args.workload else configs.ALL[HEADLINE]
        d, t, out, lse, ws = prefill_setup(cfg, absorbed=args.absorbed, fused=args.fused)
        fn = lambda: prefill_call(cfg, d, t, out, lse, ws, stream, absorbed=args.absorbed, fused=args.fused)  # noqa: E731
    elif args.only == "backward":
        cfg = configs.ALL[args.workload] if args.workload else configs.ALL[HEADLINE]
        d, t, out, lse, ws = prefill_setup(cfg)
        prefill_call(cfg, d, t, out, lse, ws, stream)
        del ws
        g = torch.Generator(device="cuda")
        g.manual_seed(3)
        dout = randn(out.shape, 1.0, out.dtype, g)

        def fn():
            mla.latent_attn_bwd(d, t["q_nope"], t["q_pe"], t["c_kv"], t["k_pe"], t["w_kv_b"], t["rms_w"], out, lse,
                                dout, q_offset=cfg.q_offset, causal=cfg.causal, head_shard=cfg.head_shard,
                                stream=stream)
    else:
        cfg = configs.DECODE
        if args.batch:
            import dataclasses
            cfg = dataclasses.replace(cfg, batch=args.batch)
        if args.only == "tpla":
            d, t, out, slse, ws = tpla_setup(cfg, 2)
            fn = lambda: tpla_call(cfg, 2, d, t, out, slse, ws, stream)  # noqa: E731
        else:
            d, t, out, lse, ws = decode_setup(cfg)
            fn = lambda: decode_call(cfg, d, t, out, lse, ws, stream)  # noqa: E731
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    st = mla.mla_check_device_error(None)
    print("%s %s: %d calls, path %d, device status %s" % (args.only, cfg.name, args.warmup + args.steps,
                                                       mla.last_path(), mla.mla_status_string(st)))
    if st != 0:
        sys.exit(1)


# -------------------------------------------------------- oracle (CPU) ----
def oracle_prefill_sample(cfg, rows: int, heads: int):
    """Time the oracle on the last `rows` query rows of workload `cfg`, heads [0, heads).

    Returns (seconds, algorithmic FLOPs of the sample, threads used).  The sample's FLOPs
    are its own: the visible pairs of those rows and heads x 2 x (qk + v dims), plus the
    K/V reconstruction of those heads over every key the rows see."""
    import dataclasses

    import oracle
    from head_latent_attention_rmsnorm_gb300 import inputs
    q0 = cfg.q_offset + cfg.s_q - rows
    full = inputs.prefill_inputs(cfg, q_rows=(q0, q0 + rows))
    sub = dataclasses.replace(cfg, s_q=rows, q_offset=q0, n_heads=heads)
    inp = {k: v.double().numpy() for k, v in full.items()}
    inp["q_nope"] = inp["q_nope"][:, :, :heads].copy()
    inp["q_pe"] = inp["q_pe"][:, :, :heads].copy()
    t0 = time.perf_counter()
    oracle.mla_explicit(**inp, n_heads=cfg.n_heads, q_offset=q0, causal=True, base=cfg.rope_base, eps=cfg.rms_eps)
    dt = time.perf_counter() - t0
    return dt, sub.flops()["total"], int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


CPU_SAMPLE = (512, 48)    # rows, heads of the cpu_baseline leg (10-20 s of the host's cores)
REF_SAMPLE = (32, 8)      # rows, heads of each step of the --impl reference arm (~3 s on 8 cores)


def cpu_baseline_headline():
    from head_latent_attention_rmsnorm_gb300 import configs
    oracle_build()
    cfg = configs.ALL[HEADLINE]
    rows, heads = CPU_SAMPLE
    dt, fl, cores = oracle_prefill_sample(cfg, rows, heads)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "seconds": round(dt, 3),
            "sample": "fp64 oracle, %s: the last %d query rows (positions %d-%d), heads 0-%d, K/V rebuilt "
                      "for every key they see" % (cfg.name, rows, cfg.q_offset + cfg.s_q - rows,
                                                   cfg.q_offset + cfg.s_q - 1, heads - 1)}


def oracle_build():
    import oracle
    oracle.build()


def run_reference(args, world, rank):
    """The oracle as the reference arm (rank 0 only), on the headline workload."""
    if rank != 0:
        return
    from head_latent_attention_rmsnorm_gb300 import configs
    oracle_build()
    cfg = configs.ALL[HEADLINE]
    rows, heads = REF_SAMPLE
    for _ in range(args.warmup):
        oracle_prefill_sample(cfg, rows, heads)
    times, fl, cores = [], 0, 1
    for _ in range(args.steps):
        dt, fl, cores = oracle_prefill_sample(cfg, rows, heads)
        times.append(dt)
    ms = statistics.mean(times) * 1e3
    v = fl / (ms * 1e-3) / 1e12
    sample = ("fp64 oracle, %s: the last %d query rows, heads 0-%d, K/V rebuilt for every key they see"
              % (cfg.name, rows, heads - 1))
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded PCG64, N(0,1))",
            "config": {"workload": cfg.name, "sample_rows": rows, "sample_heads": heads},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the side workloads (V2-Lite, V3, absorbed, decode, TPLA) and the memory measurement")
    ap.add_argument("--absorbed", action="store_true", help="--only prefill: the absorbed form")
    ap.add_argument("--fused", action="store_true", help="--only prefill: the fused explicit form")
    ap.add_argument("--only", choices=("prefill", "backward", "decode", "tpla"), default=None,
                    help="run only this workload's calls, without timing (profiling target)")
    ap.add_argument("--workload", default=None, help="prefill workload name for --only prefill")
    ap.add_argument("--batch", type=int, default=0, help="decode batch for --only decode (default 64)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup(args)
    if args.only:
        run_case(args)
        return
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
