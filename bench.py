"""Benchmark: decode-attention µs per layer-step and effective KV GB/s (% of HBM peak).

One step = one pass of the whole hot path on one layer, through kvq_flash_decode_append:
the decode kernel encodes the new token's K and V rows into the resident store, runs the
split-K fused-dequant flash-decode over the whole sequence (new token included), and a
second kernel, chained to it by programmatic dependent launch, merges the per-warp
partial results into the output and advances seq_lens by one: two launches per step
(record mode; plans whose partials do not fit the record layout merge in place inside the
decode kernel, one launch).  The store grows by one token per step.  Inputs are resident
in HBM when the timed region starts; the L2 is flushed before every timed step by reading
a 2 x L2 buffer (leaving clean lines, so the timed kernel pays no write-back), outside its
events, with a bounded ~100 µs GPU wait queued after it so that the events time the GPU
work, not host launch latency.  That wait spins a fixed number of SM cycles, so its own
event-timed length gives the SM clock of every step.

The headline time is the 10%-trimmed mean of the K per-step event times (the event clock
ticks in ~2 µs steps, which a median would round to); the median, p10/p90 and a
1000-step distribution with per-step clock bins are reported beside it.

Default workload: 8B-class decode layer, one sequence, 32 query heads on 8 KV heads,
head_dim 128, kv_len 65536, q8_0 K and V; the sweep adds every codec arm at kv_len 4096,
16384 and 65536 (kernel-only timings).  `value` is effective KV GB/s: the KV bytes one
decode reads (kv_len x kv_heads x bytes per token-head of K and V, scales included)
divided by the step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload layer8b|longctx|ragged|resident] [--codec q8_0/q8_0]
                    [--kv-len L] [--variant 0|1|2] [--no-sweep]
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DIST_STEPS = 1000                     # steps of the per-step distribution block
METRIC = "decode-attention µs/layer-step & effective KV GB/s (% of HBM peak) vs kv_len"
FALLBACK_HBM_GBS = 6800.0
ROW_BYTES = {"bf16": lambda d: 2 * d, "f16": lambda d: 2 * d, "q8_0": lambda d: d + d // 16,
             "q4s": lambda d: d // 2 + d // 16}

WORKLOADS = {
    "layer8b": dict(batch=1, hq=32, hkv=8, d=128, kv_len=65536, dist="normal", scaled=False,
                    codec="q8_0/q8_0"),
    "longctx": dict(batch=1, hq=32, hkv=2, d=256, kv_len=204800, dist="normal", scaled=True,
                    codec="q8_0/q8_0"),
    "ragged": dict(batch=64, hq=32, hkv=8, d=128, kv_len=None, dist="normal", scaled=False,
                   codec="q8_0/q8_0"),
    "resident": dict(batch=1, hq=32, hkv=8, d=128, kv_len=65536, dist="t3", scaled=True,
                     codec="q8_0/q8_0"),
}


def token_head_bytes(codec_pair: str, d: int) -> int:
    kc, vc = codec_pair.split("/")
    return ROW_BYTES[kc](d) + ROW_BYTES[vc](d)


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                j = json.load(f)
            for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if key in j:
                    return float(j[key]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def decode_source_files() -> list:
    """The device-code sources the decode kernels are built from: the tensor-core decode
    instantiation units and every header they include, directly or not (the prefill
    kernels' own headers are not among them), sorted."""
    csrc = os.path.join(ROOT, "flash_decode_quantized_gb300", "csrc")
    files = sorted(n for n in os.listdir(csrc) if n.startswith("mma_") and n.endswith(".cu"))
    todo, seen = list(files), set(files)
    while todo:
        for line in open(os.path.join(csrc, todo.pop())):
            m = re.match(r'\s*#include\s+"([^"]+)"', line)
            if m and m.group(1) not in seen and os.path.exists(os.path.join(csrc, m.group(1))):
                seen.add(m.group(1))
                todo.append(m.group(1))
    return sorted(seen)


def kernel_sources_sha() -> str:
    """Hash of decode_source_files(), in order."""
    csrc = os.path.join(ROOT, "flash_decode_quantized_gb300", "csrc")
    h = hashlib.sha256()
    for name in decode_source_files():
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_sha: str, workload_key: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == workload_key and parts[1] == kernel_sha:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- device side

def device_rows(torch, gen, n, hkv, d, dist, scales):
    if dist == "normal":
        x = torch.randn((n, hkv, d), generator=gen, device="cuda", dtype=torch.float32)
    else:  # Student-t, 3 degrees of freedom: N / sqrt(chi2_3 / 3)
        z = torch.randn((n, hkv, d), generator=gen, device="cuda", dtype=torch.float32)
        c = torch.randn((3, n, hkv, d), generator=gen, device="cuda", dtype=torch.float32)
        x = z / torch.sqrt((c * c).sum(0) / 3.0)
    if scales is not None:
        x = x * scales
    return x.to(torch.bfloat16)


class Layer:
    """One decode layer's resident stores plus per-step inputs, on the current device."""

    def __init__(self, kvq, torch, wl, codec_pair, seq_lens, capacity_extra, seed, page_size=256):
        self.kvq, self.torch = kvq, torch
        self.hq, self.hkv, self.d = wl["hq"], wl["hkv"], wl["d"]
        self.kc, self.vc = codec_pair.split("/")
        self.batch = len(seq_lens)
        self.page_size = page_size
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        ks = vs = None
        if wl["scaled"]:
            lo, hi = math.log(0.25), math.log(4.0)
            ks = torch.exp(torch.rand((self.hkv, self.d), generator=gen, device="cuda") * (hi - lo) + lo)
            vs = torch.exp(torch.rand((self.hkv, self.d), generator=gen, device="cuda") * (hi - lo) + lo)
        self.k_scales, self.v_scales, self.dist = ks, vs, wl["dist"]
        caps = [int(L) + capacity_extra for L in seq_lens]
        pages = [max(1, -(-c // page_size)) for c in caps]
        total = int(sum(pages))
        perm = torch.randperm(total, generator=gen, device="cuda").to(torch.int32)
        self.max_pages = max(pages)
        pt = torch.full((self.batch, self.max_pages), -1, dtype=torch.int32, device="cuda")
        pos = 0
        for b, n in enumerate(pages):
            pt[b, :n] = perm[pos:pos + n]
            pos += n
        self.page_table = pt
        self.k_store = kvq.kvq_store_create(self.kc, self.hkv, self.d, page_size, total)
        self.v_store = kvq.kvq_store_create(self.vc, self.hkv, self.d, page_size, total)
        self.seq_lens = torch.zeros(self.batch, dtype=torch.int32, device="cuda")
        for b, L in enumerate(seq_lens):
            done = 0
            while done < L:
                n = min(32768, int(L) - done)
                seq = torch.tensor([done], dtype=torch.int32, device="cuda")
                kr = device_rows(torch, gen, n, self.hkv, self.d, self.dist, ks)
                vr = device_rows(torch, gen, n, self.hkv, self.d, self.dist, vs)
                kvq.kvq_append(self.k_store, kr[None], seq, pt[b:b + 1].contiguous())
                kvq.kvq_append(self.v_store, vr[None], seq, pt[b:b + 1].contiguous())
                done += n
        self.seq_lens.copy_(torch.tensor(list(seq_lens), dtype=torch.int32))
        self.host_lens = [int(L) for L in seq_lens]
        self.q = torch.randn((self.batch, self.hq, self.d), generator=gen, device="cuda").to(torch.bfloat16)
        self.new_k = device_rows(torch, gen, 1, self.hkv, self.d, self.dist, ks).view(1, 1, self.hkv, self.d).expand(self.batch, 1, self.hkv, self.d).contiguous()
        self.new_v = device_rows(torch, gen, 1, self.hkv, self.d, self.dist, vs).view(1, 1, self.hkv, self.d).expand(self.batch, 1, self.hkv, self.d).contiguous()
        self.out = torch.empty((self.batch, self.hq, self.d), dtype=torch.float32, device="cuda")
        self.hint = max(caps)
        self.ws = None

    def prepare(self, variant, chunk_tokens=0):
        n = self.kvq.kvq_decode_workspace_bytes(self.k_store, self.v_store, self.batch, self.hq,
                                                self.hint, chunk_tokens, variant)
        self.ws = self.torch.empty(n, dtype=self.torch.uint8, device="cuda")
        self.kvq.kvq_decode_workspace_init(self.ws)
        self.variant, self.chunk = variant, chunk_tokens

    def append(self, new_k=None, new_v=None):
        # one launch: encode the step's K and V rows, then seq_lens += 1
        self.kvq.kvq_append_kv(self.k_store, self.v_store, self.new_k if new_k is None else new_k,
                               self.new_v if new_v is None else new_v, self.seq_lens, self.page_table,
                               advance=True)
        self.host_lens = [L + 1 for L in self.host_lens]

    def decode(self, q=None):
        return self.kvq.kvq_flash_decode(self.q if q is None else q, self.k_store, self.v_store,
                                         self.seq_lens, self.page_table, out=self.out,
                                         max_len_hint=self.hint, workspace=self.ws,
                                         chunk_tokens=self.chunk, variant=self.variant)

    def step(self, q=None, new_k=None, new_v=None):
        """One decode step of the layer: append the new token's K and V rows, attend,
        advance seq_lens.  One fused launch on the tensor-core kernel; the CUDA-core
        variant runs kvq_append_kv + kvq_flash_decode."""
        if self.variant == 1:
            self.append(new_k, new_v)
            return self.decode(q)
        nk = self.new_k if new_k is None else new_k
        nv = self.new_v if new_v is None else new_v
        out = self.kvq.kvq_flash_decode_append(
            self.q if q is None else q, nk.view(self.batch, self.hkv, self.d),
            nv.view(self.batch, self.hkv, self.d), self.k_store, self.v_store, self.seq_lens,
            self.page_table, advance=True, out=self.out, max_len_hint=self.hint, workspace=self.ws,
            chunk_tokens=self.chunk, variant=self.variant)
        self.host_lens = [L + 1 for L in self.host_lens]
        return out

    def unfused(self, target="f16"):
        """The separate-pass arm (stock build of halobench record clm-0022): dequantize K and
        V into 16-bit stores with kvq_dequantize, then a 16-bit kvq_flash_decode."""
        kvq, torch = self.kvq, self.torch
        if getattr(self, "kd", None) is None:
            pages = self.k_store.num_pages
            self.kd = kvq.kvq_store_create(target, self.hkv, self.d, self.page_size, pages)
            self.vd = kvq.kvq_store_create(target, self.hkv, self.d, self.page_size, pages)
            n = kvq.kvq_decode_workspace_bytes(self.kd, self.vd, self.batch, self.hq, self.hint, 0, 0)
            self.ws16 = torch.empty(n, dtype=torch.uint8, device="cuda")
            kvq.kvq_decode_workspace_init(self.ws16)
        kvq.kvq_dequantize(self.k_store, self.kd, self.seq_lens, self.page_table)
        kvq.kvq_dequantize(self.v_store, self.vd, self.seq_lens, self.page_table)
        return kvq.kvq_flash_decode(self.q, self.kd, self.vd, self.seq_lens, self.page_table, out=self.out,
                                    max_len_hint=self.hint, workspace=self.ws16)

    def multi(self, tokens):
        """Decode of `tokens` query tokens per sequence (the last `tokens` positions being
        drafts) with kvq_flash_decode_multi."""
        kvq, torch = self.kvq, self.torch
        key = f"_multi{tokens}"
        if not hasattr(self, key):
            q = torch.randn((self.batch, self.hq, tokens, self.d), device="cuda").to(torch.bfloat16)
            n = kvq.kvq_decode_workspace_bytes(self.k_store, self.v_store, self.batch, self.hq * tokens,
                                               self.hint, 0, 0)
            ws = torch.empty(n, dtype=torch.uint8, device="cuda")
            kvq.kvq_decode_workspace_init(ws)
            out = torch.empty((self.batch, self.hq, tokens, self.d), dtype=torch.float32, device="cuda")
            setattr(self, key, (q, ws, out))
        q, ws, out = getattr(self, key)
        return kvq.kvq_flash_decode_multi(q, self.k_store, self.v_store, self.seq_lens, self.page_table,
                                          out=out, max_len_hint=self.hint, workspace=ws)

    def kv_bytes(self):
        return sum(self.host_lens) * self.hkv * token_head_bytes(f"{self.kc}/{self.vc}", self.d)


def l2_flusher(torch):
    """Evicts the KV store from L2 by reading a buffer of twice the L2 size.  Reading
    (not writing) leaves only clean lines behind, so the timed kernel pays no write-back
    of the flush traffic."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    buf = torch.ones(2 * l2 // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty((), dtype=torch.float32, device="cuda")

    def flush():
        torch.sum(buf, dim=0, out=sink)
    return flush


LEAD_CYCLES = 200_000


def gpu_lead(torch):
    """Keeps the GPU busy ~100 µs (a wait of LEAD_CYCLES SM clock cycles) so that the host
    has enqueued the whole step before the GPU reaches the step's first event; otherwise
    the events would time host launch latency."""
    torch.cuda._sleep(LEAD_CYCLES)


def trimmed_mean(xs, frac=0.1):
    """Mean of the values left after dropping the lowest and highest `frac` of them."""
    xs = sorted(xs)
    k = int(len(xs) * frac)
    core = xs[k:len(xs) - k] or xs
    return sum(core) / len(core)


def timed_steps(torch, fn, flush, n):
    """n calls of fn, each after an L2 flush and the cycle-count lead, each bracketed by
    CUDA events on the current stream.  Returns (ms per call, SM MHz per call); the clock
    of a call is LEAD_CYCLES over its lead's event-timed length (an estimate within the
    event clock's ~2 µs resolution, ~2%)."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(n):
        flush()
        ev[i][0].record()
        gpu_lead(torch)
        ev[i][1].record()
        fn()
        ev[i][2].record()
    torch.cuda.synchronize()
    ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(n)]
    mhz = [LEAD_CYCLES / max(ev[i][0].elapsed_time(ev[i][1]), 1e-6) / 1e3 for i in range(n)]
    return ms, mhz


def step_stats(ms, mhz=None):
    """Trimmed mean, median, p10/p90 (µs) of per-step times; with clocks, per-step SM clock
    bins (steps, trimmed mean and median time per bin)."""
    out = {"steps": len(ms), "trimmed_mean_us": round(trimmed_mean(ms) * 1e3, 2),
           "median_us": round(statistics.median(ms) * 1e3, 2),
           "p10_p90_us": [round(float(np.percentile(ms, 10)) * 1e3, 2),
                          round(float(np.percentile(ms, 90)) * 1e3, 2)]}
    if mhz:
        out["sm_mhz_median"] = round(statistics.median(mhz), 0)
        bins = {}
        for lo, hi, name in ((1980, 1e9, ">=1980"), (1880, 1980, "1880-1980"), (0, 1880, "<1880")):
            sel = [t for t, f in zip(ms, mhz) if lo <= f < hi]
            if sel:
                bins[name] = {"steps": len(sel), "trimmed_mean_us": round(trimmed_mean(sel) * 1e3, 2),
                              "median_us": round(statistics.median(sel) * 1e3, 2)}
        out["clock_bins_mhz"] = bins
    return out


def bench_config(wl_name, wl, codec, kv_len_desc, world):
    """The workload this run measures; both arms print the same dict."""
    return {"workload": f"{wl_name}: B={wl['batch']}, Hq={wl['hq']}, Hkv={wl['hkv']}, D={wl['d']}, "
                        f"kv_len={kv_len_desc}",
            "codec": codec, "kv_len": kv_len_desc,
            "l2": "GPU arm: KV store evicted from L2 before every timed step by reading a 2xL2 buffer "
                  "(clean lines), outside the step's events; CPU oracle arm: not applicable",
            "parallelism": f"replicas x{world}"}


def max_over_ranks(torch, x: float, world: int, device) -> float:
    """The slowest rank's value (all ranks call this; a no-op on one process)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_gbs(kv_bytes_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job effective KV GB/s: every replica reads kv_bytes_per_rank per step, and a
    step takes the slowest rank's time."""
    return world * kv_bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def read_probe_gbs(torch, kvq, flush, gib: float = 2.0) -> float:
    """Achievable read bandwidth on this GPU now: kvq_read_probe over a `gib` GiB buffer
    (16x the L2), median of 10 event-timed launches."""
    buf = torch.ones(int(gib * (1 << 30)) // 16 * 16, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    ms = []
    for it in range(12):
        flush()
        gpu_lead(torch)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        kvq.kvq_read_probe(buf, sink)
        e1.record()
        torch.cuda.synchronize()
        if it >= 2:
            ms.append(e0.elapsed_time(e1))
    n = buf.numel()
    del buf
    torch.cuda.empty_cache()
    return n / (statistics.median(ms) * 1e-3) / 1e9


def time_decode_only(torch, layer, flush, iters, fn=None):
    fn = fn or layer.decode
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for i in range(iters):
        flush()
        gpu_lead(torch)
        ev[i][0].record()
        fn()
        ev[i][1].record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def run_mine(args, rank, world):
    import torch
    from flash_decode_quantized_gb300 import kvq

    torch.cuda.set_device(rank % max(1, torch.cuda.device_count()))
    wl = dict(WORKLOADS[args.workload])
    codec = args.codec or wl["codec"]
    if wl["kv_len"] is None:
        from workloads import ragged_lengths
        seq_lens = [int(x) for x in ragged_lengths(1234 + rank, wl["batch"])]
    else:
        seq_lens = [args.kv_len or wl["kv_len"]] * wl["batch"]
    # timed, e2e (three passes), unfused, the 1000-step distribution
    extra = args.warmup + 4 * max(args.steps, 20) + 128 + DIST_STEPS + 16
    layer = Layer(kvq, torch, wl, codec, seq_lens, extra, seed=1000 + rank)
    layer.prepare(args.variant, args.chunk_tokens)
    flush = l2_flusher(torch)
    probe = read_probe_gbs(torch, kvq, flush)
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush()
        layer.step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    K = args.steps
    kv_bytes = []
    launches0 = kvq.kvq_launch_count()

    def one_step():
        layer.step()
        kv_bytes.append(layer.kv_bytes())
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step_ms, step_mhz = timed_steps(torch, one_step, flush, K)   # synchronizes at the end
        wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    launches = kvq.kvq_launch_count() - launches0
    # the step is the decode kernel plus its PDL-chained merge kernel (the CUDA-core
    # variant: append + decode + combine)
    dec_ms = step_ms
    # 10%-trimmed mean over the K per-step event pairs: robust to the event clock's ~2 us
    # ticks (which a median rounds to) and to the odd step an nvidia-smi sample stalls
    ms_per_step = max_over_ranks(torch, trimmed_mean(step_ms), world, "cuda")
    kvb = statistics.mean(kv_bytes)
    value = job_gbs(kvb, world, ms_per_step)
    peak, peak_kind = hbm_peak()
    dec_mean = trimmed_mean(dec_ms)
    achieved = kvb / (dec_mean * 1e-3) / 1e9
    sha = kernel_sources_sha()
    key = f"{args.workload}:{codec}:{seq_lens[0] if len(set(seq_lens)) == 1 else 'ragged'}"
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(sha, key),
                "kernel": "decode_mma_kernel with the fused append + record_merge_kernel (kvq_flash_decode_append), timed together per step" if args.variant != 1 else "kvq_append_kv + decode_simt + combine",
                "peak_source": f"{peak_kind} copy bandwidth",
                "decode_us": round(dec_mean * 1e3, 2),
                "decode_us_median": round(statistics.median(dec_ms) * 1e3, 2),
                "decode_us_p10_p90": [round(float(np.percentile(dec_ms, 10)) * 1e3, 2),
                                      round(float(np.percentile(dec_ms, 90)) * 1e3, 2)],
                "cv": round(statistics.pstdev(dec_ms) / statistics.mean(dec_ms), 4),
                "stat": "10%-trimmed mean of per-step CUDA-event times",
                "clock_bins_mhz": step_stats(step_ms, step_mhz)["clock_bins_mhz"],
                "read_probe_gbs": round(probe, 1), "frac_of_read_probe": round(achieved / probe, 4)}

    e2e = measure_e2e(torch, kvq, layer, flush, max(20, K))
    e2e["value"] = round(world * e2e.pop("kvb") / (e2e["ms"] * 1e-3) / 1e9, 1)
    # the same step as two launches (kvq_append_kv, then kvq_flash_decode), for comparison
    unfused = None
    if args.variant != 1:
        ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for i in range(K):
            flush()
            gpu_lead(torch)
            ev2[i][0].record()
            layer.append()
            ev2[i][1].record()
            layer.decode()
            ev2[i][2].record()
        torch.cuda.synchronize()
        unfused = {"step_us": round(statistics.mean(a.elapsed_time(c) for a, _, c in ev2) * 1e3, 2),
                   "decode_us": round(statistics.mean(b.elapsed_time(c) for _, b, c in ev2) * 1e3, 2)}

    # a longer run of the same step for its distribution: per-step times and SM clocks
    dist_ms, dist_mhz = timed_steps(torch, layer.step, flush, DIST_STEPS)
    distribution = step_stats(dist_ms, dist_mhz)
    distribution["timing"] = ("the timed step repeated after the timed region, each after an L2 "
                              "flush; clock per step from the cycle-count lead's event-timed length")

    sweep = extras = None
    if rank == 0 and args.workload == "layer8b":
        if not args.no_sweep:
            sweep = run_sweep(torch, kvq, args, flush, peak)
        if not args.no_extras:
            extras = run_extras(torch, kvq, args, flush, peak)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_layer_step": round(ms_per_step * 1e3, 2),
        "us_per_step_mean": round(statistics.mean(step_ms) * 1e3, 2),
        "us_per_step_max": [round(max(step_ms) * 1e3, 2), int(np.argmax(step_ms))],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, device-generated bf16 rows encoded on device)",
        "config": bench_config(args.workload, wl, codec, kv_len_desc(wl, seq_lens[0]), world),
        "run": {"kv_bytes_per_step": int(kvb), "variant": args.variant, "chunk_tokens": args.chunk_tokens,
                "lead": "~100 us cycle-count GPU wait before each step so that events exclude host launch latency"},
        "roofline": roofline,
        "distribution": distribution,
        "unfused_step": unfused,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 3),
        "kernel_sha": sha,
        "frac_of_8TBs": round(achieved / 8000.0, 4),
    }
    if sweep is not None:
        result["sweep"] = sweep
        result["slopes"] = depth_slopes([(r["codec"], r["kv_len"], r["us"]) for r in sweep], "layer8b")
    if extras is not None:
        result["workloads"] = extras
        lc = [(r["codec"], r["kv_len"], r["us"]) for r in extras if r["workload"] == "longctx"]
        result.setdefault("slopes", {}).update(depth_slopes(lc, "longctx"))
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args, wl, codec, seq_lens[0] if wl["kv_len"] else 4096)
    return result


def depth_slopes(points, tag):
    """Least-squares us = a + b * kv_len per codec arm (the pages' marginal cost per 1k KV
    tokens is b * 1000): {"<tag> <codec>": {"us_per_1k_tokens": b*1000, "intercept_us": a}}."""
    by = {}
    for codec, L, us in points:
        by.setdefault(codec, []).append((L, us))
    out = {}
    for codec, pts in by.items():
        if len(pts) < 2:
            continue
        xs = np.array([p[0] for p in pts], dtype=np.float64)
        ys = np.array([p[1] for p in pts], dtype=np.float64)
        b, a = np.polyfit(xs, ys, 1)
        out[f"{tag} {codec}"] = {"us_per_1k_tokens": round(float(b) * 1000, 4), "intercept_us": round(float(a), 2)}
    return out


def measure_e2e(torch, kvq, layer, flush, iters):
    """The same step through the public API with host buffers.  Each of the K steps has its
    own pinned host slot for its inputs (q and the new token's K and V rows) and for its
    output.  Default (tensor-core variant): each step is one library call bound to its slots
    (kvq.DecodeAppendStep over pinned CPU tensors), and the kernel reads the inputs from and
    writes the output to host memory in place, so the transfers happen inside the step.
    `copy_engine`: the same loop with explicit pinned H2D and D2H copies around a call bound
    to device buffers.  The steps are enqueued back to back on one stream and the region
    ends with a synchronize (L2 not flushed: the serving pattern).  `sync_step`: one step at
    a time (synchronize after each, L2 evicted before it), median."""
    nq, nk, nv = layer.q.numel(), layer.new_k.numel(), layer.new_v.numel()
    n_in = nq + nk + nv
    host_in = torch.empty((iters, n_in), dtype=torch.bfloat16).pin_memory()
    for i in range(iters):
        host_in[i, :nq] = layer.q.reshape(-1).cpu()
        host_in[i, nq:nq + nk] = layer.new_k.reshape(-1).cpu()
        host_in[i, nq + nk:] = layer.new_v.reshape(-1).cpu()
    host_out = torch.empty((iters,) + tuple(layer.out.shape), dtype=torch.float32).pin_memory()
    bkd = (layer.batch, layer.hkv, layer.d)

    def timed(run_one, sync_each=False, n=iters):
        for i in range(3):   # warm the path
            run_one(i)
        torch.cuda.synchronize()
        if sync_each:
            out = []
            for i in range(n):
                flush()
                torch.cuda.synchronize()
                t1 = time.perf_counter()
                run_one(i)
                torch.cuda.synchronize()
                out.append((time.perf_counter() - t1) * 1e3)
            return statistics.median(out)
        kvb = 0
        t0 = time.perf_counter()
        for i in range(n):
            run_one(i)
            kvb += layer.kv_bytes()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) * 1e3 / n, kvb / n

    # explicit copies around a step bound to device buffers
    dev_in = torch.empty(n_in, dtype=torch.bfloat16, device="cuda")
    q_d = dev_in[:nq].view(layer.q.shape)
    k_d = dev_in[nq:nq + nk].view(bkd)
    v_d = dev_in[nq + nk:].view(bkd)
    if layer.variant == 1:
        def dev_step():
            layer.step(q_d, k_d.view(layer.new_k.shape), v_d.view(layer.new_v.shape))
    else:
        bound = kvq.DecodeAppendStep(q_d, k_d, v_d, layer.k_store, layer.v_store, layer.seq_lens,
                                     layer.page_table, layer.out, layer.ws, layer.hint,
                                     chunk_tokens=layer.chunk, variant=layer.variant)

        def dev_step():
            bound()
            layer.host_lens = [L + 1 for L in layer.host_lens]

    def copy_one(i):
        dev_in.copy_(host_in[i], non_blocking=True)
        dev_step()
        host_out[i].copy_(layer.out, non_blocking=True)

    ce_ms, ce_kvb = timed(copy_one)
    ce = {"ms": round(ce_ms, 5), "value": round(ce_kvb / (ce_ms * 1e-3) / 1e9, 1),
          "timing": "pinned H2D copy of the step's inputs, the step (bound to device buffers), "
                    "pinned D2H copy of its output, per step; back to back, one synchronize"}
    if layer.variant == 1:
        sync_ms = timed(copy_one, sync_each=True, n=min(iters, 20))
        return {"ms": round(ce_ms, 5), "unit": "GB/s", "h2d_bytes_per_step": int(n_in * 2),
                "d2h_bytes_per_step": int(layer.out.numel() * 4), "kvb": ce_kvb,
                "timing": ce["timing"],
                "sync_step": {"ms": round(sync_ms, 5), "value": round(layer.kv_bytes() / (sync_ms * 1e-3) / 1e9, 1),
                              "timing": "one step at a time, synchronize after it, L2 evicted before, median"}}

    # zero-copy: one call per step, bound to its pinned host slots
    steps = []
    for i in range(iters):
        hq = host_in[i, :nq].view(layer.q.shape)
        hk = host_in[i, nq:nq + nk].view(bkd)
        hv = host_in[i, nq + nk:].view(bkd)
        steps.append(kvq.DecodeAppendStep(hq, hk, hv, layer.k_store, layer.v_store, layer.seq_lens,
                                          layer.page_table, host_out[i], layer.ws, layer.hint,
                                          chunk_tokens=layer.chunk, variant=layer.variant))

    def zc_one(i):
        steps[i]()
        layer.host_lens = [L + 1 for L in layer.host_lens]

    ms, kvb = timed(zc_one)
    sync_ms = timed(zc_one, sync_each=True, n=min(iters, 20))
    # the same zero-copy call timed on the device, L2 evicted before each (cold, like the
    # headline), next to the warm back-to-back loop above
    ctr = [0]

    def zc_next():
        zc_one(ctr[0] % iters)
        ctr[0] += 1
    ev_ms, _ = timed_steps(torch, zc_next, flush, min(iters, 50))
    ev_t = trimmed_mean(ev_ms)
    return {"ms": round(ms, 5), "unit": "GB/s", "h2d_bytes_per_step": int(n_in * 2),
            "d2h_bytes_per_step": int(layer.out.numel() * 4), "kvb": kvb,
            "timing": f"host wall clock over {iters} back-to-back steps, each one library call whose "
                      "kernel reads the step's inputs from its pinned host slot and writes the output "
                      "to its pinned host slot (zero-copy over the host link), one synchronize at the end",
            "copy_engine": ce,
            "l2_evicted": {"ms": round(ev_t, 5), "value": round(layer.kv_bytes() / (ev_t * 1e-3) / 1e9, 1),
                           "timing": "CUDA events around each zero-copy step (inputs read from and output "
                                     "written to pinned host memory inside it), L2 evicted before each, "
                                     f"10%-trimmed mean of {len(ev_ms)}"},
            "sync_step": {"ms": round(sync_ms, 5),
                          "value": round(layer.kv_bytes() / (sync_ms * 1e-3) / 1e9, 1),
                          "timing": "one step at a time: the zero-copy step + synchronize, L2 evicted before, median"}}


def prefill_cells(torch, kvq, flush):
    """Chunked prefill attention at the 8B-class layer shape (pp512 at depth 32768): the f16
    control, q8_0 K+V fused, and a separate dequantize pass + the f16 kernel; one row each
    (medians of 6 event-timed launches, L2 evicted before each)."""
    out = []
    # the 512 chunk tokens are appended, then attend causally over the 33280-token store
    depth, T = 32768, 512
    times = {}
    for arm in ("f16/f16", "q8_0/q8_0"):
        layer = Layer(kvq, torch, WORKLOADS["layer8b"], arm, [depth + T], 0, seed=92)
        qp = torch.randn((1, T, layer.hq, layer.d), device="cuda").to(torch.bfloat16)
        outp = torch.empty((1, T, layer.hq, layer.d), dtype=torch.float32, device="cuda")

        def pf(layer=layer, qp=qp, outp=outp):
            kvq.kvq_prefill_attention(qp, layer.k_store, layer.v_store, layer.seq_lens, layer.page_table, out=outp)
        time_decode_only(torch, layer, flush, 2, pf)
        ms = statistics.median(time_decode_only(torch, layer, flush, 6, pf))
        times[arm] = ms
        flops = 4.0 * layer.d * layer.hq * sum(depth + i + 1 for i in range(T))
        row = {"workload": "prefill_attention", "depth": depth, "chunk_tokens": T, "codec": arm,
               "us": round(ms * 1e3, 1), "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
        if arm == "q8_0/q8_0":
            row["vs_f16_time"] = round(ms / times["f16/f16"], 3)
            # unfused arm: the quantized store dequantized to f16 first, then the f16 kernel
            kd = kvq.kvq_store_create("f16", layer.hkv, layer.d, layer.page_size, layer.k_store.num_pages)
            vd = kvq.kvq_store_create("f16", layer.hkv, layer.d, layer.page_size, layer.k_store.num_pages)

            def unf(layer=layer, qp=qp, outp=outp, kd=kd, vd=vd):
                kvq.kvq_dequantize(layer.k_store, kd, layer.seq_lens, layer.page_table)
                kvq.kvq_dequantize(layer.v_store, vd, layer.seq_lens, layer.page_table)
                kvq.kvq_prefill_attention(qp, kd, vd, layer.seq_lens, layer.page_table, out=outp)
            time_decode_only(torch, layer, flush, 2, unf)
            um = statistics.median(time_decode_only(torch, layer, flush, 6, unf))
            row["unfused_f16_us"] = round(um * 1e3, 1)
            del kd, vd
        out.append(row)
        del layer
        torch.cuda.empty_cache()
    return out


def run_extras(torch, kvq, args, flush, peak):
    """The other workloads at full size: the long-context depth sweep (f16 control vs
    q8_0 K+V, GQA 16:1, D=256), the 64-sequence ragged paged batch, and the resident
    append + decode loop (128 steps from a 65536-token heavy-tailed prefix)."""
    out = []
    wl = WORKLOADS["longctx"]
    for L in (32768, 131072, 204800):
        base = None
        for arm in ("f16/f16", "q8_0/q8_0"):
            layer = Layer(kvq, torch, wl, arm, [L], 0, seed=88)
            layer.prepare(args.variant, 0)
            time_decode_only(torch, layer, flush, 3)
            ms = statistics.median(time_decode_only(torch, layer, flush, 10))
            gbs = layer.kv_bytes() / (ms * 1e-3) / 1e9
            base = ms if arm == "f16/f16" else base
            row = {"workload": "longctx", "kv_len": L, "codec": arm, "us": round(ms * 1e3, 2),
                   "gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "vs_f16_time": round(ms / base, 3)}
            if arm == "q8_0/q8_0":
                time_decode_only(torch, layer, flush, 2, layer.unfused)
                um = statistics.median(time_decode_only(torch, layer, flush, 8, layer.unfused))
                row["unfused_f16_us"] = round(um * 1e3, 2)
                row["unfused_vs_f16_time"] = round(um / base, 3)
            out.append(row)
            del layer
            torch.cuda.empty_cache()
    # prefill-side bulk encode: one kvq_append_kv of a 65536-token prompt's K and V rows
    # (8B-class layer shape) into fresh q8_0 / q4s stores, bf16 read + codes and scales written
    wl8 = WORKLOADS["layer8b"]
    for arm in ("q8_0/q8_0", "q4s/q4s"):
        kc, vc = arm.split("/")
        n = 65536
        pages = n // 256
        ks = kvq.kvq_store_create(kc, wl8["hkv"], wl8["d"], 256, pages)
        vs = kvq.kvq_store_create(vc, wl8["hkv"], wl8["d"], 256, pages)
        rows_k = torch.randn((1, n, wl8["hkv"], wl8["d"]), device="cuda").to(torch.bfloat16)
        rows_v = torch.randn((1, n, wl8["hkv"], wl8["d"]), device="cuda").to(torch.bfloat16)
        pt = torch.arange(pages, dtype=torch.int32, device="cuda")[None]
        seq = torch.zeros(1, dtype=torch.int32, device="cuda")
        ev = []
        for it in range(6):
            flush()
            gpu_lead(torch)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            kvq.kvq_append_kv(ks, vs, rows_k, rows_v, seq, pt, advance=False)
            e1.record()
            ev.append((e0, e1))
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in ev[1:])
        moved = 2 * rows_k.numel() * 2 + n * wl8["hkv"] * token_head_bytes(arm, wl8["d"])
        out.append({"workload": "prefill_encode", "tokens": n, "codec": arm, "us": round(ms * 1e3, 2),
                    "gbs_moved": round(moved / (ms * 1e-3) / 1e9, 1),
                    "note": "bf16 K and V rows read, codes and scales written, one launch"})
        del ks, vs, rows_k, rows_v
        torch.cuda.empty_cache()
    out.extend(prefill_cells(torch, kvq, flush))
    depth, T = 32768, 512
    # the same chunk at the long-context shape (GQA 16:1, head_dim 256)
    ptimes = {}
    for arm in ("f16/f16", "q8_0/q8_0"):
        layer = Layer(kvq, torch, WORKLOADS["longctx"], arm, [depth + T], 0, seed=94)
        qp = torch.randn((1, T, layer.hq, layer.d), device="cuda").to(torch.bfloat16)
        outp = torch.empty((1, T, layer.hq, layer.d), dtype=torch.float32, device="cuda")

        def pf2(layer=layer, qp=qp, outp=outp):
            kvq.kvq_prefill_attention(qp, layer.k_store, layer.v_store, layer.seq_lens, layer.page_table, out=outp)
        time_decode_only(torch, layer, flush, 2, pf2)
        ms = statistics.median(time_decode_only(torch, layer, flush, 6, pf2))
        ptimes[arm] = ms
        flops = 4.0 * layer.d * layer.hq * sum(depth + i + 1 for i in range(T))
        row = {"workload": "prefill_attention_longctx", "depth": depth, "chunk_tokens": T, "codec": arm,
               "us": round(ms * 1e3, 1), "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
        if arm == "q8_0/q8_0":
            row["vs_f16_time"] = round(ms / ptimes["f16/f16"], 3)
        out.append(row)
        del layer
        torch.cuda.empty_cache()
    # speculative-draft verification: T query tokens per sequence in one decode, against
    # T single-token decodes of the same cache (8B-class layer, 65536 tokens, q8_0 K+V)
    layer = Layer(kvq, torch, WORKLOADS["layer8b"], "q8_0/q8_0", [65536], 0, seed=91)
    layer.prepare(args.variant, 0)
    time_decode_only(torch, layer, flush, 3)
    one = statistics.median(time_decode_only(torch, layer, flush, 10))
    for T in (2, 4):
        fn = (lambda T=T: layer.multi(T))
        time_decode_only(torch, layer, flush, 3, fn)
        ms = statistics.median(time_decode_only(torch, layer, flush, 10, fn))
        out.append({"workload": "spec_verify", "kv_len": 65536, "codec": "q8_0/q8_0", "query_tokens": T,
                    "us": round(ms * 1e3, 2), "single_token_us": round(one * 1e3, 2),
                    "vs_T_single_decodes": round(ms / (T * one), 3),
                    "gbs": round(layer.kv_bytes() / (ms * 1e-3) / 1e9, 1)})
    del layer
    torch.cuda.empty_cache()
    # the same at long context (GQA 16:1, D = 256, 131072 tokens, q8_0 K+V): two draft tokens
    # are 32 query rows per KV head
    layer = Layer(kvq, torch, WORKLOADS["longctx"], "q8_0/q8_0", [131072], 0, seed=93)
    layer.prepare(args.variant, 0)
    time_decode_only(torch, layer, flush, 3)
    one = statistics.median(time_decode_only(torch, layer, flush, 10))
    fn = (lambda: layer.multi(2))
    time_decode_only(torch, layer, flush, 3, fn)
    ms = statistics.median(time_decode_only(torch, layer, flush, 10, fn))
    out.append({"workload": "spec_verify_longctx", "kv_len": 131072, "codec": "q8_0/q8_0", "query_tokens": 2,
                "us": round(ms * 1e3, 2), "single_token_us": round(one * 1e3, 2),
                "vs_T_single_decodes": round(ms / (2 * one), 3),
                "gbs": round(layer.kv_bytes() / (ms * 1e-3) / 1e9, 1)})
    del layer
    torch.cuda.empty_cache()
    from workloads import ragged_lengths
    lens = [int(x) for x in ragged_lengths(1234, 64)]
    for arm in ("q8_0/q8_0", "q4s/q4s"):
        layer = Layer(kvq, torch, WORKLOADS["ragged"], arm, lens, 0, seed=89)
        layer.prepare(args.variant, 0)
        time_decode_only(torch, layer, flush, 2)
        ms = statistics.median(time_decode_only(torch, layer, flush, 8))
        gbs = layer.kv_bytes() / (ms * 1e-3) / 1e9
        out.append({"workload": "ragged", "batch": 64, "total_tokens": sum(lens), "codec": arm,
                    "us": round(ms * 1e3, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)})
        del layer
        torch.cuda.empty_cache()
    for arm in ("q8_0/q8_0", "q8_0/q4s"):
        layer = Layer(kvq, torch, WORKLOADS["resident"], arm, [65536], 3 + 3 * 128 + 32, seed=90)
        layer.prepare(args.variant, 0)
        for _ in range(3):
            layer.step()
        torch.cuda.synchronize()
        tph = layer.hkv * token_head_bytes(arm, layer.d)

        def loop_bytes(L0):   # KV bytes the 128 steps from length L0 read
            return sum(L0 + i + 1 for i in range(128)) * tph
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        L0 = int(layer.seq_lens.item())
        e0.record()
        for _ in range(128):
            layer.step()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 128
        gbs = loop_bytes(L0) / 128 / (ms * 1e-3) / 1e9
        row = {"workload": "resident", "steps": 128, "codec": arm, "us_per_step": round(ms * 1e3, 2),
               "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
               "note": "128 back-to-back fused append+decode steps, L2 not flushed between steps"}
        # the same 128 steps captured once in a CUDA graph, timed over one replay
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(128):
                    layer.step()
            graph.replay()
            torch.cuda.synchronize()
            L0 = int(layer.seq_lens.item())
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            assert int(layer.seq_lens.item()) == L0 + 128
            gms = e0.elapsed_time(e1) / 128
            row["graph_us_per_step"] = round(gms * 1e3, 2)
            row["graph_gbs"] = round(loop_bytes(L0) / 128 / (gms * 1e-3) / 1e9, 1)
        except Exception as exc:   # report, keep the rest of the run
            row["graph_error"] = str(exc)[:200]
        out.append(row)
        del layer
        torch.cuda.empty_cache()
    return out


def run_sweep(torch, kvq, args, flush, peak):
    """Kernel-only decode timings for every codec arm at kv_len 4096 / 16384 / 65536."""
    wl = WORKLOADS["layer8b"]
    arms = ["bf16/bf16", "q8_0/bf16", "q8_0/q8_0", "q4s/q4s", "q8_0/q4s", "q4s/q8_0", "q4s/bf16"]
    rows = []
    for L in (4096, 16384, 65536):
        base = None
        for arm in arms:
            layer = Layer(kvq, torch, wl, arm, [L], 0, seed=77)
            layer.prepare(args.variant, 0)
            time_decode_only(torch, layer, flush, 3)
            ms = time_decode_only(torch, layer, flush, 20)
            med = statistics.median(ms)
            gbs = layer.kv_bytes() / (med * 1e-3) / 1e9
            if arm == "bf16/bf16":
                base = med
            row = {"kv_len": L, "codec": arm, "us": round(med * 1e3, 2),
                   "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                   "vs_bf16_time": round(med / base, 3),
                   "cv": round(statistics.pstdev(ms) / statistics.mean(ms), 4)}
            if arm in ("q8_0/q8_0", "q4s/q4s"):
                # the same decode with a separate dequantize-to-f16 pass first
                time_decode_only(torch, layer, flush, 2, layer.unfused)
                um = statistics.median(time_decode_only(torch, layer, flush, 10, layer.unfused))
                row["unfused_f16_us"] = round(um * 1e3, 2)
                row["fused_speedup"] = round(um / med, 3)
            rows.append(row)
            del layer
            torch.cuda.empty_cache()
    return rows


# ----------------------------------------------------------------------------- CPU oracle

def _oracle_step(wl, codec, L, kv_heads, seed):
    """The oracle on a bounded sample of one step: dequantize `kv_heads` KV heads' prefixes
    and attend with their query heads.  Returns (seconds, KV bytes of the sample)."""
    from oracle import attention as oatt
    from oracle import codec as ocodec
    from workloads import make_inputs
    kc, vc = codec.split("/")
    g = wl["hq"] // wl["hkv"]
    inp = make_inputs([L], g * kv_heads, kv_heads, wl["d"], seed=seed, dist=wl["dist"],
                      channel_scaled=wl["scaled"])
    q = ocodec.bf16_bits_to_f64(inp.q)
    t0 = time.perf_counter()
    d = wl["d"]
    kd = ocodec.dequantized(inp.k_rows[0].reshape(-1, d), kc).reshape(L, kv_heads, d)
    vd = ocodec.dequantized(inp.v_rows[0].reshape(-1, d), vc).reshape(L, kv_heads, d)
    oatt.attention(q, [kd], [vd], kv_heads, 1 / math.sqrt(d))
    dt = time.perf_counter() - t0
    return dt, L * kv_heads * token_head_bytes(codec, d)


def cpu_baseline(args, wl, codec, L):
    cores = len(os.sched_getaffinity(0))
    times, nbytes = [], 0
    budget = 20.0
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < budget and len(times) < 8:
        dt, b = _oracle_step(wl, codec, L, 1, seed=99 + len(times))
        times.append(dt)
        nbytes += b
    value = nbytes / sum(times) / 1e9
    return {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(times)} x (1 KV head of {wl['hkv']}, its {wl['hq'] // wl['hkv']} query heads, "
                      f"kv_len {L}, {codec}): float64 NumPy dequantize + attention",
            "ms_per_layer_step_scaled": round(statistics.mean(times) * wl["hkv"] * 1e3, 1)}


def kv_len_desc(wl, kv_len):
    return str(kv_len) if wl["kv_len"] is not None else "U[1024,32768]"


def run_reference(args, world):
    wl = dict(WORKLOADS[args.workload])
    codec = args.codec or wl["codec"]
    L = args.kv_len or wl["kv_len"] or 16384
    cores = len(os.sched_getaffinity(0))
    for i in range(args.warmup):
        _oracle_step(wl, codec, min(L, 4096), 1, seed=5 + i)
    times, nbytes = [], []
    for i in range(args.steps):
        dt, b = _oracle_step(wl, codec, L, 1, seed=50 + i)
        times.append(dt)
        nbytes.append(b)
    ms = statistics.mean(times) * 1e3
    value = sum(nbytes) / sum(times) / 1e9
    sample = (f"each step: 1 KV head of {wl['hkv']} with its {wl['hq'] // wl['hkv']} query heads, "
              f"kv_len {L}, {codec} (float64 NumPy oracle: dequantize + attention)")
    return {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded NumPy)", "impl": "reference",
            "config": bench_config(args.workload, wl, codec, kv_len_desc(wl, L), world),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--workload", default="layer8b", choices=list(WORKLOADS))
    ap.add_argument("--codec", default=None)
    ap.add_argument("--kv-len", type=int, default=None)
    ap.add_argument("--variant", type=int, default=0)
    ap.add_argument("--chunk-tokens", type=int, default=0)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads' cells")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the chunked prefill cells (pp512 at depth 32768) and print them")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)))
        return
    if args.prefill_only:
        if rank == 0:
            import torch
            from flash_decode_quantized_gb300 import kvq
            cells = prefill_cells(torch, kvq, l2_flusher(torch))
            print(json.dumps({"metric": "chunked prefill attention us (pp512 at depth 32768, 8B-class layer)",
                              "unit": "us", "higher_is_better": False, "cells": cells,
                              "gpu_launches": kvq.kvq_launch_count()}))
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res = run_mine(args, rank, world)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
