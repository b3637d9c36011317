"""Benchmark of one MLA decode step on B300.

A step is the whole hot path over one batch: append the new token's cache row
(S1), absorb the query (S2), latent split-KV attention (S3) and the W_UV / W_O
expansion (S4/S5), for the DeepSeek-V2-shaped layer (d=5120, n_h=128, d_h=128,
d_c=512, d_r=64, d_cq=1536, bf16) at batch 64 with 4096 cached tokens per
sequence, timed through mla_decode_step (one library call per step); the
per-stage breakdown and the attention call's roofline come from a second loop
through the four entry points. Inputs are synthetic (h ~ N(0,1), W ~ N(0, 1/fan_in), seeded) and
resident in HBM; the cache (302 MB) and weights (298 MB) exceed the 126 MB L2,
so no flush is needed between steps.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]

Under torchrun each rank runs its own batch on its own GPU (weak scaling: the
sequences of a decode batch are independent, so no collective touches the data
path); rank 0 prints one JSON line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode tokens/s and latent-cache GB/s (fraction of roofline), 1×B300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(kernel: str = "decode_pair") -> str:
    """Hash of an attention kernel's sources (the kernel a committed traffic
    figure was measured on, and the headers it includes)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "head_latent_attention_24_b300", "csrc")
    for n in (f"{kernel}.cu", f"{kernel}.cuh", "tc_ptx.cuh", "tmap.cuh", "internal.cuh"):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_hash: str, record: str = "decode_attn_v2_traffic.json"):
    """DRAM bytes per launch of a kernel from its committed ncu summary, if it
    was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", record)
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != kernel_hash:
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled during the timed
    region: the driver's NVML library polled every ~1 ms from a thread (the
    region lasts tens of milliseconds)."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.ident = None
        try:
            import torch
            props = torch.cuda.get_device_properties(gpu_index)
            uuid = getattr(props, "uuid", None)
            if uuid is not None:
                self.ident = ("uuid", "GPU-" + str(uuid))
            elif hasattr(props, "pci_bus_id"):
                self.ident = ("pci", "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                                          getattr(props, "pci_device_id", 0)))
        except Exception:  # noqa: BLE001
            self.ident = None
        self.samples = []
        self.stop_flag = threading.Event()
        self.t = None
        self.err = None

    def _poll(self):
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            # NVML numbers GPUs without regard to CUDA_VISIBLE_DEVICES: find
            # this process's device by its UUID (or PCI bus id) instead.
            h = ctypes.c_void_p()
            if self.ident and self.ident[0] == "uuid":
                rc = nv.nvmlDeviceGetHandleByUUID(self.ident[1].encode(), ctypes.byref(h))
            elif self.ident and self.ident[0] == "pci":
                rc = nv.nvmlDeviceGetHandleByPciBusId_v2(self.ident[1].encode(), ctypes.byref(h))
            else:
                raise RuntimeError("no UUID or PCI bus id for the CUDA device")
            if rc != 0:
                raise RuntimeError(f"NVML handle lookup for {self.ident} failed ({rc})")
            clk, mx, reasons = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
            NVML_CLOCK_SM = 1
            if nv.nvmlDeviceGetMaxClockInfo(h, NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            while not self.stop_flag.is_set():
                if nv.nvmlDeviceGetClockInfo(h, NVML_CLOCK_SM, ctypes.byref(clk)) == 0 and \
                        get_reasons(h, ctypes.byref(reasons)) == 0:
                    self.samples.append((clk.value, int(reasons.value)))
                time.sleep(0.001)
            nv.nvmlShutdown()
        except Exception as e:  # noqa: BLE001
            self.err = f"{type(e).__name__}: {e}"

    def start(self):
        self.t = threading.Thread(target=self._poll, daemon=True)
        self.t.start()
        time.sleep(0.05)

    def stop(self):
        self.stop_flag.set()
        if self.t is not None:
            self.t.join(timeout=5)
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0,
                    "reasons": [f"no NVML samples ({self.err})" if self.err else "no NVML samples"]}
        sm = [c for c, _ in self.samples]
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": getattr(self, "max_mhz", None),
                "samples": len(sm), "sm_mhz_min": min(sm), "reasons": sorted(reasons),
                "device": self.ident[1] if self.ident else None}


def roofline_of(nbytes: float, flops: float, seconds: float, peaks: dict) -> dict:
    """Roofline of one call: the slower of its bytes at the measured HBM copy
    bandwidth and its FLOPs at the measured burst bf16 rate (the call is timed
    on its own), with the achieved rate in that bound's unit."""
    hbm_t = nbytes / (peaks["hbm_gbs"] * 1e9)
    tc_t = flops / (peaks["bf16_tflops"] * 1e12)
    if hbm_t >= tc_t:
        out = {"bound": "hbm", "achieved": round(nbytes / seconds / 1e9, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        out = {"bound": "tensor", "achieved": round(flops / seconds / 1e12, 1), "peak": peaks["bf16_tflops"],
               "unit": "TFLOP/s"}
    out["frac"] = round(max(hbm_t, tc_t) / seconds, 4)
    out["roofline_us"] = round(max(hbm_t, tc_t) * 1e6, 2)
    sus = peaks.get("bf16_tflops_sustained")
    if sus:
        out["frac_vs_sustained_tensor_peak"] = round(max(hbm_t, flops / (sus * 1e12)) / seconds, 4)
    return out


def plan_balance(seqlens, chunks: int, granule: int):
    """Rows per chunk of the equal-row split plan (the same rule the library's
    plan kernel applies): max over mean of the busy chunks."""
    total = int(np.sum(seqlens))
    cl = -(-total // chunks)
    cl = max(granule, -(-cl // granule) * granule)
    rows = [min(cl, total - c * cl) for c in range(chunks) if c * cl < total]
    return round(max(rows) / (sum(rows) / len(rows)), 4), len(rows)


class L2Flush:
    """Empties L2 before a timed call: writes a 256 MB buffer (twice L2), then
    reads another 256 MB one, so that L2 ends up holding clean lines. Without
    the read the timed kernel would pay for writing back up to 126 MB of the
    flush's dirty lines."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        self.r = torch.ones(64 << 20, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.fill_(1)
        self.r.sum()


def attention_workloads(device, peaks, iters: int = 20):
    """mla_decode_attn alone on the other decode workloads (random caches of
    the workload's shape; CUDA events, median of `iters` calls)."""
    import torch
    import head_latent_attention_24_b300 as M
    import mla_synth as S
    out = {}
    for name in ("minimind", "v2_ragged", "v2_long"):
        shp = S.workload(name)
        seqlens = (S.draw_context_lengths(shp) + 1).astype(np.int32)
        B, max_len = len(seqlens), int(seqlens.max())
        g = torch.Generator(device=device)
        g.manual_seed(shp.seed)
        cache = torch.randn((B, max_len, shp.D), generator=g, device=device, dtype=torch.bfloat16)
        q = torch.randn((B, shp.n_h, shp.D), generator=g, device=device, dtype=torch.bfloat16)
        q[..., :shp.d_c] *= (shp.d_h / shp.d_c) ** 0.5
        h = M.mla_create(shp.d, shp.n_h, shp.d_h, shp.d_c, shp.d_r, shp.d_cq, M.MLA_BF16, max_len)
        try:
            ws = torch.empty(M.mla_decode_workspace_size(h, B, max_len), dtype=torch.uint8, device=device)
            o = torch.empty((B, shp.n_h, shp.d_c), dtype=torch.bfloat16, device=device)
            lse = torch.empty((B, shp.n_h), dtype=torch.float32, device=device)
            sl = torch.as_tensor(seqlens).to(device)
            flush = L2Flush(device) if B * max_len * shp.D * 2 < (256 << 20) else None
            for _ in range(3):
                M.mla_decode_attn(h, q, cache, B, max_len, sl, o, lse, ws, ws.numel())
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
            for e0, e1 in evs:
                if flush is not None:
                    flush()   # the cache is smaller than two L2s: start each call cold
                e0.record()
                M.mla_decode_attn(h, q, cache, B, max_len, sl, o, lse, ws, ws.numel())
                e1.record()
            torch.cuda.synchronize()
            st, bits = M.mla_get_device_status(h)
            if st != M.MLA_OK:
                raise RuntimeError(f"{name}: device status {st} bits {bits}")
            us = statistics.median(e0.elapsed_time(e1) * 1e3 for e0, e1 in evs)
            rows = int(seqlens.sum())
            nbytes = rows * shp.D * 2
            flops = 2.0 * rows * shp.n_h * (shp.D + shp.d_c)
            r = roofline_of(nbytes, flops, us * 1e-6, peaks)
            r.update({"attn_us": round(us, 2), "GBps": round(nbytes / us / 1e3, 1), "cache_bytes": nbytes,
                      "tokens_per_s": round(B / (us * 1e-6), 1), "batch": B, "rows": rows,
                      "l2": "flushed before each call (256 MB write, then 256 MB read)" if flush is not None
                      else "cache larger than L2",
                      "decode_path": {M.MLA_DECODE_SIMT: "simt", M.MLA_DECODE_TCGEN05: "tcgen05"}[
                          M.mla_get_decode_path(h)]})
            if name == "minimind":
                r["traffic"] = committed_traffic(kernel_source_hash("decode_narrow"),
                                                 "decode_narrow_minimind_traffic.json")
            if name == "v2_ragged":
                bal, busy = plan_balance(seqlens, h_chunks(M, h, B, max_len, device), 64)
                r["split_rows_max_over_mean"] = bal
                r["split_chunks_busy"] = busy
                r["seqlen_min_max"] = [int(seqlens.min()), int(seqlens.max())]
            out[name] = r
        finally:
            M.mla_destroy(h)
            del cache
            torch.cuda.empty_cache()
    return out


def premerged_comparison(M, dec, shp, h_new, pos, device, iters: int = 15):
    """S2 and S4/S5 two ways on the benchmark's batch: the two-step factors
    (W_UQ then W_UK^T; W_UV then W_O) against the pre-merged maps W_QK and
    W_OUV. L2 is flushed (L2Flush) before every timed call, as in the step,
    where each weight byte is read once."""
    import torch
    B = shp.batch
    dt = torch.bfloat16
    W_QK = torch.empty((shp.n_h, shp.d_c, shp.d_cq), dtype=dt, device=device)
    W_OUV = torch.empty((shp.d, shp.n_h * shp.d_c), dtype=dt, device=device)
    M.mla_premerge_query_weights(dec.handle, dec.W["W_UQ"], dec.W["W_UK"], W_QK)
    M.mla_premerge_output_weights(dec.handle, dec.W["W_UV"], dec.W["W_O"], W_OUV)
    flush = L2Flush(device)
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(iters):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return round(statistics.median(ts), 2), M.mla_last_launch_count(dec.handle)

    W = dec.W
    a2, l_a2 = timed(lambda: M.mla_absorb_q(dec.handle, h_new, B, W["W_DQ"], W["W_UQ"], W["W_QR"], W["W_UK"], pos,
                                            dec.q_abs, dec.ws, dec.ws.numel()))
    a1, l_a1 = timed(lambda: M.mla_absorb_q_premerged(dec.handle, h_new, B, W["W_DQ"], W_QK, W["W_QR"], pos,
                                                      dec.q_abs, dec.ws, dec.ws.numel()))
    o2, l_o2 = timed(lambda: M.mla_out_proj(dec.handle, dec.o_lat, B, W["W_UV"], W["W_O"], dec.u, dec.ws,
                                            dec.ws.numel()))
    o1, l_o1 = timed(lambda: M.mla_out_proj_premerged(dec.handle, dec.o_lat, B, W_OUV, dec.u))
    nb = lambda *ts: round(sum(t.numel() * 2 for t in ts) / 1e6, 1)
    res = {
        "batch": B,
        "absorb_two_step": {"us": a2, "launches": l_a2, "weight_MB": nb(W["W_DQ"], W["W_UQ"], W["W_QR"], W["W_UK"])},
        "absorb_premerged": {"us": a1, "launches": l_a1, "weight_MB": nb(W["W_DQ"], W_QK, W["W_QR"])},
        "out_proj_two_step": {"us": o2, "launches": l_o2, "weight_MB": nb(W["W_UV"], W["W_O"])},
        "out_proj_premerged": {"us": o1, "launches": l_o1, "weight_MB": nb(W_OUV)},
        "l2": "flushed before every call (256 MB write, then 256 MB read)",
    }
    del W_QK, W_OUV, flush
    torch.cuda.empty_cache()
    return res


def prefill_workload(device, peaks, B: int = 2, T: int = 4096, iters: int = 10):
    """The MHA path on the V2 shape for T new tokens per sequence (no earlier
    context): K/V materialised for the T cache rows, queries projected, causal
    multi-head attention, W_O. Times each call (CUDA events, median) and the
    attention's FLOP rate against the burst bf16 peak (causal: query t attends
    t + 1 rows; 2 * n_h * (d_h + d_r + d_h) FLOPs per query-row pair)."""
    import torch
    import head_latent_attention_24_b300 as M
    shp = v2_shape()
    n_h, d_h, d_r, d_c, d = shp.n_h, shp.d_h, shp.d_r, shp.d_c, shp.d
    g = torch.Generator(device=device)
    g.manual_seed(shp.seed + 7)

    def w(r, c):
        return (torch.randn((r, c), generator=g, device=device) / c ** 0.5).to(torch.bfloat16)

    W = {"W_DKV": w(d_c, d), "W_KR": w(d_r, d), "W_DQ": w(shp.d_cq, d), "W_UQ": w(n_h * d_h, shp.d_cq),
         "W_QR": w(n_h * d_r, shp.d_cq), "W_UK": w(n_h * d_h, d_c), "W_UV": w(n_h * d_h, d_c), "W_O": w(d, n_h * d_h)}
    h = M.mla_create(d, n_h, d_h, d_c, d_r, shp.d_cq, M.MLA_BF16, T)
    try:
        x = torch.randn((B * T, d), generator=g, device=device).to(torch.bfloat16)
        cache = torch.zeros((B, T, shp.D), dtype=torch.bfloat16, device=device)
        seq = torch.arange(B, dtype=torch.int32, device=device).repeat_interleave(T)
        pos = torch.arange(T, dtype=torch.int32, device=device).repeat(B)
        k_c = torch.empty((B, T, n_h, d_h), dtype=torch.bfloat16, device=device)
        v_c = torch.empty_like(k_c)
        q = torch.empty((B, T, n_h, d_h + d_r), dtype=torch.bfloat16, device=device)
        o = torch.empty((B, T, n_h, d_h), dtype=torch.bfloat16, device=device)
        lse = torch.empty((B, T, n_h), dtype=torch.float32, device=device)
        u = torch.empty((B * T, d), dtype=torch.bfloat16, device=device)
        ws = torch.empty(M.mla_absorb_q_workspace_size(h, B * T), dtype=torch.uint8, device=device)
        q_pos0 = torch.zeros(B, dtype=torch.int32, device=device)
        calls = {
            "append": lambda: M.mla_append_cache(h, x, B * T, W["W_DKV"], W["W_KR"], seq, pos, cache, B, T),
            "materialise_kv": lambda: M.mla_materialise_kv(h, cache, B * T, W["W_UK"], W["W_UV"], k_c, v_c),
            "project_q": lambda: M.mla_project_q(h, x, B * T, W["W_DQ"], W["W_UQ"], W["W_QR"], pos, q, ws,
                                                 ws.numel()),
            "mha_attn": lambda: M.mla_mha_attn(h, q, B, T, k_c, v_c, cache, T, q_pos0, o, lse),
            "project_out": lambda: M.mla_project_out(h, o, B * T, W["W_O"], u),
        }
        out = {"batch": B, "new_tokens": T, "context": 0}
        for name, fn in calls.items():
            for _ in range(2):
                fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(iters):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
            out[name + "_us"] = round(statistics.median(ts), 1)
        st, bits = M.mla_get_device_status(h)
        if st != M.MLA_OK:
            raise RuntimeError(f"prefill: device status {st} bits {bits}")
        flops = 2.0 * B * n_h * (2 * d_h + d_r) * (T * (T + 1) / 2)
        t_attn = out["mha_attn_us"] * 1e-6
        out["mha_attn_tflops"] = round(flops / t_attn / 1e12, 1)
        out["mha_attn_frac_of_burst_bf16"] = round(flops / t_attn / 1e12 / peaks["bf16_tflops"], 4)
        total = sum(out[k + "_us"] for k in calls)
        out["tokens_per_s"] = round(B * T / (total * 1e-6), 1)
        return out
    finally:
        M.mla_destroy(h)
        torch.cuda.empty_cache()


def h_chunks(M, h, B, max_len, device):
    """Split-KV chunk count the attention call uses (CTA pairs of the
    tensor-core kernel): from the SM count."""
    import torch
    return torch.cuda.get_device_properties(device).multi_processor_count // 2


# --------------------------------------------------------------------------- workload
def v2_shape():
    import mla_synth as S
    return S.workload("v2")


def make_inputs(shp, device, rank=0):
    """Weights (the same layer on every rank) and this rank's new-token inputs,
    on the device, from seeded torch generators."""
    import torch
    import mla_synth as S
    g = torch.Generator(device=device)
    g.manual_seed(shp.seed * 7919)
    W = {}
    for name in S.WEIGHT_NAMES:
        r, c = shp.weight_shape(name)
        W[name] = (torch.randn((r, c), generator=g, device=device) * (1.0 / shp.fan_in(name)) ** 0.5).to(
            torch.bfloat16).contiguous()
    g.manual_seed(shp.seed * 7919 + 1 + rank)
    h_new = torch.randn((shp.batch, shp.d), generator=g, device=device).to(torch.bfloat16).contiguous()
    return W, h_new


def context_seq_id(b: int, rank: int) -> int:
    """Generator id of sequence b of a rank's batch: distinct over ranks, so
    each rank serves its own sequences (data parallel over the batch)."""
    return b + 1000 * rank


def max_over_ranks(x: float, device) -> float:
    """The slowest rank's value of a per-rank time (the job ends with it)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(batch_per_rank: int, world: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return batch_per_rank * world * steps / (max_ms * 1e-3)


def build_cache(dec, shp, cache, device, rank=0):
    """Append every context token (positions 0..ctx-1 of each sequence) through
    mla_append_cache, in chunks; h of the context drawn per sequence."""
    import torch
    import mla_synth as S
    B, ctx = shp.batch, shp.ctx
    per = max(1, 32768 // ctx)
    for b0 in range(0, B, per):
        bs = list(range(b0, min(B, b0 + per)))
        x = torch.cat([S.context_h_device(shp, context_seq_id(b, rank), ctx, device) for b in bs], 0).contiguous()
        seq = torch.tensor(np.repeat(bs, ctx), dtype=torch.int32, device=device)
        pos = torch.tensor(np.tile(np.arange(ctx), len(bs)), dtype=torch.int32, device=device)
        dec.append(x, seq, pos, cache)
    torch.cuda.synchronize()


def oracle_sample(shp, W_dev, cache_h_fn, h_new_dev, budget_s=12.0, max_seqs=8):
    """Time the fp64 oracle's whole step on as many sequences as fit the
    budget (at least one). Returns (tokens/s, seconds, sequences, threads)."""
    import torch
    from oracle import mla as O
    W = {k: v.double().cpu().numpy() for k, v in W_dev.items()}
    h_new = h_new_dev.double().cpu().numpy()
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        threads = os.cpu_count()
    done, spent = 0, 0.0
    while done < max_seqs and (done == 0 or spent < budget_s):
        b = done
        h_ctx = cache_h_fn(b)
        t0 = time.perf_counter()
        O.decode_materialised([h_ctx], h_new[b:b + 1], W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base)
        spent += time.perf_counter() - t0
        done += 1
    return done / spent, spent, done, threads


# --------------------------------------------------------------------------- arms
def run_ours(args, rank, world, local_rank):
    import torch
    import head_latent_attention_24_b300 as M
    import mla_synth as S

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    shp = v2_shape()
    B, ctx = shp.batch, shp.ctx
    max_len = ctx + 1
    W, h_new = make_inputs(shp, device, rank)
    ls = M.LayerShape(shp.d, shp.n_h, shp.d_h, shp.d_c, shp.d_r, shp.d_cq, "bf16", shp.rope_base)
    dec = M.MLADecoder(ls, W, B, max_len, max_pos=max_len)
    if args.decode_path != "auto":
        M.mla_set_decode_path(dec.handle, {"simt": M.MLA_DECODE_SIMT, "tc": M.MLA_DECODE_TCGEN05}[args.decode_path])
    path = M.mla_get_decode_path(dec.handle)
    cache = torch.zeros((B, max_len, shp.D), dtype=torch.bfloat16, device=device)
    build_cache(dec, shp, cache, device, rank)
    pos = torch.full((B,), ctx, dtype=torch.int32, device=device)
    seqlens = pos + 1
    stream = torch.cuda.current_stream()

    def step_calls(evs):
        """The step through the four entry points, events between them."""
        evs[0].record(stream)
        M.mla_append_cache(dec.handle, h_new, B, dec.W["W_DKV"], dec.W["W_KR"], dec.tok_seq, pos, cache, B, max_len)
        M.mla_absorb_q(dec.handle, h_new, B, dec.W["W_DQ"], dec.W["W_UQ"], dec.W["W_QR"], dec.W["W_UK"], pos,
                       dec.q_abs, dec.ws, dec.ws.numel())
        evs[1].record(stream)
        M.mla_decode_attn(dec.handle, dec.q_abs, cache, B, max_len, seqlens, dec.o_lat, dec.lse, dec.ws,
                          dec.ws.numel())
        evs[2].record(stream)
        M.mla_out_proj(dec.handle, dec.o_lat, B, dec.W["W_UV"], dec.W["W_O"], dec.u, dec.ws, dec.ws.numel())
        evs[3].record(stream)

    for _ in range(args.warmup):
        dec.step(h_new, pos, cache, seqlens)
        step_calls([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    torch.cuda.synchronize()
    st, bits = M.mla_get_device_status(dec.handle)
    if st != M.MLA_OK:
        raise RuntimeError(f"device status after warm-up: {st} bits={bits}")

    # ---- the timed region: K steps through mla_decode_step (the product call)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    launches = 0
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(args.steps):
        dec.step(h_new, pos, cache, seqlens)
        launches += dec.launches
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = start.elapsed_time(end)
    total_ms = max_over_ranks(total_ms, device)

    # ---- per-stage breakdown (and the attention call's time for the roofline):
    # the same step through the four entry points, CUDA events between them
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for k in range(args.steps):
        step_calls(evs[k])
    torch.cuda.synchronize()
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    s12_ms = [e[0].elapsed_time(e[1]) for e in evs]
    s45_ms = [e[2].elapsed_time(e[3]) for e in evs]

    # ---- end to end through the public API: pinned host in, host out, every step
    h_host = torch.empty_like(h_new, device="cpu").pin_memory()
    h_host.copy_(h_new)
    pos_host = pos.cpu().pin_memory()
    sl_host = seqlens.cpu().pin_memory()
    u_host = torch.empty_like(dec.u, device="cpu").pin_memory()
    h_dev = torch.empty_like(h_new)
    pos_dev = torch.empty_like(pos)
    sl_dev = torch.empty_like(seqlens)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        h_dev.copy_(h_host, non_blocking=True)
        pos_dev.copy_(pos_host, non_blocking=True)
        sl_dev.copy_(sl_host, non_blocking=True)
        u = dec.step(h_dev, pos_dev, cache, sl_dev)
        u_host.copy_(u, non_blocking=True)
        stream.synchronize()
    e2e_eager_s = time.perf_counter() - t0
    # the same through the decoder's captured step (one graph launch per step;
    # positions and lengths travel as one [2, B4] copy)
    dec.capture(cache)
    ps_host = torch.zeros(tuple(dec.ps_in.shape), dtype=torch.int32).pin_memory()
    ps_host[0, :B].copy_(pos_host)
    ps_host[1, :B].copy_(sl_host)
    for _ in range(2):
        dec.replay()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        dec.h_in.copy_(h_host, non_blocking=True)
        dec.ps_in.copy_(ps_host, non_blocking=True)
        u = dec.replay()
        u_host.copy_(u, non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, device)
    e2e_eager_s = max_over_ranks(e2e_eager_s, device)

    st, bits = M.mla_get_device_status(dec.handle)
    if st != M.MLA_OK:
        raise RuntimeError(f"device status after timing: {st} bits={bits}")

    if rank != 0:
        return None

    peaks, peaks_src = load_peaks()
    cache_bytes = B * max_len * shp.D * 2
    flops = 2.0 * B * max_len * shp.n_h * (shp.D + shp.d_c)
    attn_s = statistics.mean(attn_ms) / 1e3
    achieved_gbs = cache_bytes / attn_s / 1e9
    achieved_tf = flops / attn_s / 1e12
    hbm = peaks["hbm_gbs"]
    roof = roofline_of(cache_bytes, flops, attn_s, peaks)
    kh = kernel_source_hash()
    traffic = committed_traffic(kh)
    tokens = B * world * args.steps
    value = job_tokens_per_s(B, world, args.steps, total_ms)
    weight_bytes = sum(v.numel() * 2 for v in W.values())
    step_roof_s = max((cache_bytes + weight_bytes) / (hbm * 1e9),
                      (flops + 2.0 * B * sum(v.numel() for v in W.values())) / (peaks["bf16_tflops"] * 1e12))
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded: h ~ N(0,1), W ~ N(0,1/fan_in), cache built by mla_append_cache)",
        "config": {
            "workload": "DeepSeek-V2-shaped MLA decode: d=5120, n_h=128, d_h=128, d_c=512, d_r=64, d_cq=1536; "
                        "batch 64 per GPU, context 4096 (+1 new token), bf16",
            "batch_per_gpu": B, "context": ctx, "global_batch": B * world,
            "l2": "no flush: inputs larger than L2 (cache 302 MB + weights 298 MB > 126 MB)",
            "decode_path": {M.MLA_DECODE_SIMT: "simt", M.MLA_DECODE_TCGEN05: "tcgen05"}[path],
        },
        "roofline": {
            "kernel": "mla_decode_attn (split plan + split-KV latent attention + LSE combine)",
            "bound": roof["bound"],
            "achieved": roof["achieved"],
            "peak": roof["peak"],
            "unit": roof["unit"],
            "frac": roof["frac"],
            "traffic": traffic,
            "peak_source": f"{peaks_src} " + ("hbm_gbs" if roof["bound"] == "hbm" else "bf16_tflops (burst)"),
            "roofline_us": roof["roofline_us"],
            "frac_vs_sustained_tensor_peak": roof.get("frac_vs_sustained_tensor_peak"),
            "algorithmic_bytes_per_launch": cache_bytes,
            "launch_us": round(attn_s * 1e6, 2),
            "frac_of_nominal_8TBps": round(achieved_gbs / NOMINAL_HBM_GBS, 4),
            "tensor_tflops": round(achieved_tf, 1),
            "tensor_frac_of_burst": round(achieved_tf / peaks["bf16_tflops"], 4),
        },
        "step_roofline_frac": round(step_roof_s / (total_ms / 1e3 / args.steps), 4),
        "e2e": {
            "value": round(job_tokens_per_s(B, world, args.steps, e2e_s * 1e3), 1),
            "unit": "tokens/s",
            "h2d_bytes_per_step": h_new.numel() * 2 + ps_host.numel() * 4,
            "d2h_bytes_per_step": dec.u.numel() * 2,
            "path": "MLADecoder.replay (the step captured as one CUDA graph); pinned host copies in the region",
            "eager_value": round(job_tokens_per_s(B, world, args.steps, e2e_eager_s * 1e3), 1),
        },
        "gpu_launches": launches,
        "clocks": clocks,
        "kernel_source_hash": kh,
        "four_call_step_ms_median": round(statistics.median(step_ms), 4),
        "step_breakdown_us": {"append_and_absorb": round(1e3 * statistics.median(s12_ms), 1),
                              "attention": round(1e3 * statistics.median(attn_ms), 1),
                              "out_proj": round(1e3 * statistics.median(s45_ms), 1)},
    }
    if world == 1 and not args.no_workloads:
        out["attention_workloads"] = attention_workloads(device, peaks)
        out["premerged_comparison"] = premerged_comparison(M, dec, shp, h_new, pos, device)
        out["prefill"] = prefill_workload(device, peaks)
    if world == 1 and not args.no_cpu_baseline:
        import mla_synth as S

        def ctx_h(b):
            return S.context_h_device(shp, b, ctx, device).double().cpu().numpy()

        v, spent, nseq, threads = oracle_sample(shp, W, ctx_h, h_new, budget_s=args.cpu_budget)
        out["cpu_baseline"] = {"value": round(v, 4), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                               "host_cpus": os.cpu_count(),
                               "sample": f"{nseq} of the {B} sequences (one decode token each, full 4097-row "
                                         f"context, fp64 materialised K/V) in {spent:.1f} s"}
    return out


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, over a bounded sample of the
    same workload (rank 0 only). A reference step is one sequence of the batch:
    its decode token over the full 4097-row context through the fp64
    materialised definition (k_C, v_C per head, two-pass softmax, W_O). W
    untimed and K timed steps run over the batch's sequences in turn, so
    K x ms_per_step is the measured time."""
    if rank != 0:
        return None
    import torch
    from oracle import mla as O
    import mla_synth as S
    shp = v2_shape()
    B, ctx = shp.batch, shp.ctx
    rng_dev = "cuda" if torch.cuda.is_available() else "cpu"
    W, h_new = make_inputs(shp, rng_dev)
    Wh = {k: v.double().cpu().numpy() for k, v in W.items()}
    hn = h_new.double().cpu().numpy()
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        threads = os.cpu_count()

    def one(b):
        h_ctx = S.context_h_device(shp, b, ctx, rng_dev).double().cpu().numpy()
        t0 = time.perf_counter()
        O.decode_materialised([h_ctx], hn[b:b + 1], Wh, shp.n_h, shp.d_h, shp.d_r, shp.rope_base)
        return time.perf_counter() - t0

    for w in range(args.warmup):
        one(w % B)
    times = [one((args.warmup + k) % B) for k in range(args.steps)]
    total_s = sum(times)
    per_seq = total_s / len(times)
    value = 1.0 / per_seq
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world, "steps": len(times),
        "warmup": args.warmup, "ms_per_step": round(per_seq * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "DeepSeek-V2-shaped MLA decode: d=5120, n_h=128, d_h=128, d_c=512, d_r=64, "
                               "d_cq=1536; batch 64, context 4096 (+1), fp64 oracle on host cores",
                   "batch_per_gpu": B, "context": ctx,
                   "step": "one sequence of the batch: its decode token over the full context"},
        "measured_s": round(total_s, 3),
        "full_batch_ms_extrapolated": round(per_seq * B * 1e3, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{len(times)} sequences of the {B}-sequence batch, one decode token each, "
                                   f"full 4097-row context, measured in {total_s:.1f} s"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-path", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other workloads' attention timings")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local_rank)
    if out is not None:
        print(json.dumps(out), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
