"""Benchmark of the two-stage compressed decode path on one GB300 per rank.

One step = one pass of the whole hot path over one batch of the 32K workload
(batch 8, Llama3.1-8B-shaped GQA layer: 32 query / 8 KV heads, d_head 128,
32768-token prompt, budget 1024): SnapKV stage-1 eviction, KT build, then 64
decode steps of (append, HSA decode).  Four identical passes are captured in
one CUDA graph and replayed (exactly K passes timed); inputs stay resident in HBM.  `value` is decode tokens per
second over whole passes (B x 64 tokens per pass, stage 1 included); the
decode-only rate, the stage-1 time and the HSA kernel's roofline are reported
beside it.  The prompt K/V (1.07 GB) is streamed every pass, which exceeds
the 129 MB L2, so no explicit L2 flush is inserted.  `e2e` runs the same
passes from host buffers: each pass copies K and the query / decode inputs
from page-locked host memory, reads the kept V rows in place across the host
link, and copies the outputs back.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs an independent replica (weak scaling, no
collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "HSA decode steps/sec (tokens/s) + achieved HBM GB/s vs roofline, 32K ctx"
WORKLOAD = "b8_32k"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "hsa_decode_b8_32k.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the e4m3-storage pass")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of the source the HSA launch depends on: the kernel file, the device
    helpers, the HsaArgs structure and the host function that plans and launches it."""
    csrc = os.path.join(ROOT, "two_stage_kv_gb300", "csrc")

    def read(f):
        with open(os.path.join(csrc, f)) as fh:
            return fh.read()

    def between(text, start, end):
        i = text.index(start)
        return text[i:text.index(end, i)]

    h = hashlib.sha256()
    h.update(read("rkv_hsa.cu").encode())
    h.update(read("rkv_common.cuh").encode())
    h.update(between(read("rkv_internal.h"), "struct HsaArgs {", "};").encode())
    h.update(between(read("rkv_api.cu"), "rkv_status hsa_common(", "\n}\n").encode())
    return h.hexdigest()[:16]


def ncu_traffic_per_launch():
    """DRAM bytes per HSA launch from the committed ncu summary, if it was taken
    on the current kernel source (else None): (cold, caches flushed by ncu;
    warm, a launch of the graph loop with the caches as the loop leaves them)."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None, None
    with open(PROFILE_SUMMARY) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None, None
    warm = d.get("warm_dram_bytes_read")
    if warm is not None:
        warm += d.get("warm_dram_bytes_write", 0)
    return d.get("dram_bytes_per_launch"), warm


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[3:7]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# multi-rank helpers (one independent replica per rank, no data-path collective)
# ---------------------------------------------------------------------------


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank timing over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Units processed by all ranks divided by the slowest rank's time (weak scaling)."""
    return world * units_per_rank / seconds_max


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


def hsa_bytes_per_launch(wl, B1, k2, n):
    """Algorithmic bytes one fused HSA launch must move at candidate count n (all
    pairs): KT rows of the k1 kept channels, the K and V rows of the selected
    blocks, the queries, the fp32 outputs, plus the appended token (read k/v,
    write the cache rows, read-modify-write its KT column)."""
    nblk = -(-n // wl.blk)
    k2e = min(k2, nblk)
    toks = min(k2e * wl.blk, n)
    per_pair = (wl.k1 * nblk * 2 + 2 * toks * wl.D * 2 + wl.G * wl.D * 2 + wl.G * wl.D * 4
                + 4 * wl.D * 2 + 2 * (2 * wl.D * 2))
    return per_pair * wl.B * wl.Hkv


def hsa_bytes_per_launch_fp8(wl, B1, k2, n):
    """hsa_bytes_per_launch for e4m3 storage: one byte per KT entry and per
    cached K / V element (queries, outputs and the appended token's inputs as
    before)."""
    nblk = -(-n // wl.blk)
    k2e = min(k2, nblk)
    toks = min(k2e * wl.blk, n)
    per_pair = (wl.k1 * nblk + 2 * toks * wl.D + wl.G * wl.D * 2 + wl.G * wl.D * 4
                + 2 * wl.D * 2 + 2 * wl.D + 2 * (2 * wl.D))
    return per_pair * wl.B * wl.Hkv


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    from two_stage_kv_gb300 import pipeline, synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = synth.WORKLOADS[WORKLOAD]
    li = synth.layer_inputs(wl)
    t = lambda bits: pipeline.bf16_tensor(bits, dev)  # noqa: E731
    k, v, qo = t(li.k), t(li.v), t(li.q_obs)
    qd, kn, vn = t(li.q_dec), t(li.k_new), t(li.v_new)
    L = pipeline.Layer(wl, k, v, qo, device=dev)
    B1, k2 = L.bud.B1, L.bud.k2
    out_all = torch.empty(wl.steps, wl.B, wl.Hq, wl.D, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def tev():
        # timing events recorded as graph nodes (cudaEventRecordExternal)
        return torch.cuda.Event(enable_timing=True, external=True)

    # phase-boundary events only: event nodes between every launch would add
    # several microseconds per decode step to the graph
    ev = {"s0": tev(), "s1": tev(), "s2": tev(), "d1": tev()}

    def one_pass(record=True, lay=None, q_=None, kn_=None, vn_=None, out_=None):
        lay = L if lay is None else lay
        q_ = qd if q_ is None else q_
        kn_ = kn if kn_ is None else kn_
        vn_ = vn if vn_ is None else vn_
        out_ = out_all if out_ is None else out_
        if record:
            ev["s0"].record()
        lay.stage1_select(pooled=False)
        if record:
            ev["s1"].record()
        lay.compact_kt()
        if record:
            ev["s2"].record()
        for s in range(wl.steps):
            lay.step(q_[s], kn_[s], vn_[s], out=out_[s], selections=False)
        if record:
            ev["d1"].record()

    # two score passes, the fused pool + select (one CTA, or a cluster of up to 8
    # for prefixes of up to 2048 pooling groups; pool and select apart beyond),
    # compaction with the KT build, and the fused append + HSA steps
    E_pool, L_pref = wl.P // 2 + 1, wl.S - wl.W
    nq_pool = -(-L_pref // E_pool)
    fused_ps = E_pool <= 32 and nq_pool <= 8 * 256
    launches_per_pass = 2 + (1 if fused_ps else 2) + 1 + wl.steps
    with torch.cuda.stream(stream):
        one_pass(record=False)          # sets kernel attributes outside capture
    torch.cuda.synchronize()
    # several identical passes per graph: one graph launch serves ppg passes, and
    # the phase events (recorded in the graph's last pass) time a pass that
    # follows another pass, as passes do in steady state
    ppg = next(p for p in (4, 2, 1) if args.steps % p == 0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(ppg):
            one_pass(record=(i == ppg - 1))
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    with torch.cuda.stream(stream):
        for _ in range(-(-args.warmup // ppg)):     # at least W warm-up passes
            graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    tA, tB = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        tA.record()
        for _ in range(args.steps // ppg):          # exactly K passes
            graph.replay()
        tB.record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(tA.elapsed_time(tB), dev)
    ms_pass = ms_total / args.steps
    tokens_per_pass = wl.B * wl.steps
    value = whole_job_rate(tokens_per_pass * args.steps, world, ms_total / 1e3)

    # per-kernel times from the last replay of the timed region
    stage1_ms = ev["s0"].elapsed_time(ev["s1"])
    kt_ms = ev["s1"].elapsed_time(ev["s2"])
    decode_ms = ev["s2"].elapsed_time(ev["d1"])
    # the decode phase is 64 back-to-back HSA launches (append fused in): the
    # average launch duration includes the gaps between launches (conservative)
    hsa_avg_us = decode_ms * 1e3 / wl.steps
    bytes_avg = sum(hsa_bytes_per_launch(wl, B1, k2, B1 + s + 1) for s in range(wl.steps)) / wl.steps
    peak, peak_kind = peaks()
    achieved = bytes_avg / (hsa_avg_us * 1e-6) / 1e9
    traffic, traffic_warm = ncu_traffic_per_launch()
    roofline = {"kernel": "hsa_decode_kernel", "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                # (cold: caches flushed by ncu, all 2*D KT rows of a CTA's blocks prefetched from DRAM;
                # warm: a launch inside the graph loop, the state the timed region runs in)
                "traffic_warm": traffic_warm,
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured" else
                "fallback 6.8 TB/s", "bytes_per_launch": int(bytes_avg), "avg_launch_us": round(hsa_avg_us, 3),
                "timing": "decode-phase events of the last timed pass / 64 launches (gaps included)",
                "l2": "warm within a pass: inputs > L2 but the 190 MB compacted cache is re-read each step",
                # the same achieved rate against GB300's nominal HBM3e rate, and the
                # target fraction this kernel is held to (not met while frac < target)
                "peak_nominal": NOMINAL_HBM_GBS, "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "target_frac": 0.70, "target_met": bool(achieved / peak >= 0.70)}

    # e4m3 storage of the compacted cache (a storage option; the headline stays
    # bf16): the same pass with rkv_compact_kt_fp8 and rkv_hsa_decode_fp8, fixed
    # power-of-two scales for this workload's value range (keys to about +-56,
    # values to about +-14), timed as its own graph
    fp8 = None
    if not args.no_fp8:
        ks_ = torch.full((wl.B, wl.Hkv), 0.125, dtype=torch.float32, device=dev)
        vs_ = torch.full((wl.B, wl.Hkv), 1.0 / 32, dtype=torch.float32, device=dev)
        L.enable_fp8(ks_, vs_)
        out8 = torch.empty_like(out_all)
        ev8 = {"s2": tev(), "d1": tev()}

        def pass_fp8():
            L.stage1_select(pooled=False)
            L.compact_kt_fp8()
            ev8["s2"].record()
            for s_ in range(wl.steps):
                L.step_fp8(qd[s_], kn[s_], vn[s_], out=out8[s_], selections=False)
            ev8["d1"].record()
        with torch.cuda.stream(stream):
            pass_fp8()
        torch.cuda.synchronize()
        g8 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g8, stream=stream):
            pass_fp8()
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                g8.replay()
        torch.cuda.synchronize()
        steps8 = max(3, min(args.steps, 50))
        t8a, t8b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t8a.record()
            for _ in range(steps8):
                g8.replay()
            t8b.record()
        torch.cuda.synchronize()
        ms8 = max_over_ranks(t8a.elapsed_time(t8b), dev) / steps8
        dec8_ms = ev8["s2"].elapsed_time(ev8["d1"])
        hsa8_us = dec8_ms * 1e3 / wl.steps
        bytes8 = sum(hsa_bytes_per_launch_fp8(wl, B1, k2, B1 + s_ + 1) for s_ in range(wl.steps)) / wl.steps
        ach8 = bytes8 / (hsa8_us * 1e-6) / 1e9
        ref = out_all.double()
        rel = ((out8.double() - ref).norm(dim=-1) / ref.norm(dim=-1).clamp_min(1e-30)).mean().item()
        fp8 = {"tokens_per_s": round(whole_job_rate(tokens_per_pass * steps8, world, ms8 * steps8 / 1e3), 1),
               "ms_per_step": round(ms8, 5), "k_scale": 0.125, "v_scale": 1.0 / 32,
               "roofline": {"kernel": "hsa_decode_kernel (e4m3)", "bound": "hbm", "achieved": round(ach8, 1),
                            "peak": peak, "unit": "GB/s", "frac": round(ach8 / peak, 4),
                            "bytes_per_launch": int(bytes8), "avg_launch_us": round(hsa8_us, 3)},
               "mean_rel_diff_vs_bf16_outputs": round(rel, 5)}

    # e2e: host buffers, host-link traffic of the pass's inputs and D2H of its
    # outputs inside the timed region.  K (all of it feeds stage 1), q_obs and
    # the decode inputs are copied to the device; V stays in page-locked host
    # memory and the compaction reads only its B1 kept rows per (b, h) across the
    # link.  Two device input sets: the copies of pass i+1 cross the link while
    # pass i computes (a pass reuses a set once the pass two before it, and its
    # D2H, are done).
    e2e = None
    if not args.no_e2e:
        v_host = v.cpu().pin_memory()
        host_in = [x.cpu().pin_memory() for x in (k, qo, qd, kn, vn)]
        sets = []
        for _ in range(2):
            inp = [torch.empty_like(x) for x in (k, qo, qd, kn, vn)]
            lay = pipeline.Layer(wl, inp[0], v_host, inp[1], device=dev)
            o_ = torch.empty_like(out_all)
            with torch.cuda.stream(stream):
                for d_, h_ in zip(inp, host_in):
                    d_.copy_(h_)
                one_pass(record=False, lay=lay, q_=inp[2], kn_=inp[3], vn_=inp[4], out_=o_)
            torch.cuda.synchronize()
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_, stream=stream):
                one_pass(record=False, lay=lay, q_=inp[2], kn_=inp[3], vn_=inp[4], out_=o_)
            sets.append(dict(inp=inp, out=o_, graph=g_, lay=lay))
        torch.cuda.synchronize()
        # the host-resident V gives the same outputs as the device-resident one
        with torch.cuda.stream(stream):
            graph.replay()
            sets[0]["graph"].replay()
        torch.cuda.synchronize()
        e2e_same = bool(torch.equal(out_all, sets[0]["out"]))
        host_out = [torch.empty(out_all.shape, dtype=out_all.dtype, pin_memory=True) for _ in range(2)]
        v_rows = wl.B * wl.Hkv * B1 * wl.D * v.element_size()
        h2d = sum(x.numel() * x.element_size() for x in host_in) + v_rows
        d2h = host_out[0].numel() * host_out[0].element_size()
        e2e_steps = max(4, min(args.steps, 20))
        copy_stream = torch.cuda.Stream(device=dev)
        ev_copied = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e0.record(copy_stream)
        for i in range(e2e_steps):
            st_ = sets[i % 2]
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(ev_done[i % 2])
                for d_, h_ in zip(st_["inp"], host_in):
                    d_.copy_(h_, non_blocking=True)
                ev_copied[i % 2].record(copy_stream)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_copied[i % 2])
                st_["graph"].replay()
                host_out[i % 2].copy_(st_["out"], non_blocking=True)
                ev_done[i % 2].record(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
        e2e = {"value": round(whole_job_rate(tokens_per_pass * e2e_steps, world, e2e_ms / 1e3), 1),
               "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
               "ms_per_step": round(e2e_ms / e2e_steps, 4),
               "v_rows_read_from_host_per_step": int(v_rows), "outputs_equal_device_resident_v": e2e_same,
               "note": "K, q_obs and decode inputs copied from page-locked host memory each pass; V stays in "
                       "page-locked host memory and the compaction reads its kept rows over the host link; "
                       "two device input sets: a pass's copies overlap the previous pass's compute"}

    from two_stage_kv_gb300 import rkv
    flags = rkv.rkv_read_device_flags()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_pass, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": wl.B, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": wl.D,
                   "context": wl.S, "budget": wl.t, "B1": B1, "k2_blocks": k2, "block": wl.blk, "k1": wl.k1,
                   "decode_steps_per_pass": wl.steps, "parallelism": f"replicas x{world}",
                   "l2": "no flush: every pass streams the 1.07 GB prompt K/V (> 129 MB L2)",
                   "graph": f"one CUDA graph per {ppg} passes (phase times from its last pass)"},
        "decode_only": {"tokens_per_s": round(wl.B * wl.steps / (decode_ms / 1e3) * world, 1),
                        "steps_per_s": round(wl.steps / (decode_ms / 1e3), 1), "ms": round(decode_ms, 4)},
        "stage1_ms": round(stage1_ms, 4), "compact_kt_ms": round(kt_ms, 4),
        "roofline": roofline, "e2e": e2e, "fp8": fp8, "gpu_launches": launches_per_pass * args.steps,
        "clocks": clk, "device_flags": flags,
    }
    if world > 1:
        torch.distributed.destroy_process_group()
    return line


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

_ORACLE_SAMPLE = r"""
import json, math, sys, time
sys.path.insert(0, {root!r})
import numpy as np
import oracle
from two_stage_kv_gb300 import synth
wl = synth.WORKLOADS[{wl!r}]
budget_s = {budget_s}
start = {start}
stride = {stride}
max_pairs = {max_pairs}
f = synth.bf16_bits_to_f64
qd = synth.q_decode(wl)
kn, vn = synth.kv_new(wl)
qo = synth.q_obs(wl, 0, qd)
r, B1, k2 = oracle.budget_split(wl.S, wl.t, wl.blk, wl.W)
scale = 1 / math.sqrt(wl.D)
G = wl.G
done = 0
t_total = 0.0
pairs = [(b, h) for b in range(wl.B) for h in range(wl.Hkv)]
limit = min(len(pairs), max_pairs)
while done < limit and (done == 0 or t_total < budget_s):
    b, h = pairs[(start + done * stride) % len(pairs)]
    kb, vb = synth.kv_slice(wl, 0, b, h, qd)
    K, V = f(kb), f(vb)
    t0 = time.perf_counter()
    keep, _ = oracle.snap_keep(f(qo[b, h * G:(h + 1) * G]), K, B1, wl.W, wl.P, scale)
    Kc = np.zeros((B1 + wl.steps, wl.D)); Vc = np.zeros_like(Kc)
    Kc[:B1] = K[keep]; Vc[:B1] = V[keep]
    kmax, kmin = oracle.build_kt(Kc, B1, wl.blk)
    n = B1
    for s in range(wl.steps):
        Kc[n] = f(kn[s, b, h]); Vc[n] = f(vn[s, b, h])
        kmax, kmin = oracle.kt_append(kmax, kmin, n, Kc[n], wl.blk)
        n += 1
        oracle.hsa_decode(f(qd[s, b, h * G:(h + 1) * G]), Kc, Vc, n, kmax, kmin, wl.blk, wl.k1, k2, scale)
    t_total += time.perf_counter() - t0
    done += 1
print(json.dumps({{"pairs": done, "total_pairs": len(pairs), "seconds": t_total}}))
"""


def _oracle_env():
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    return env


def oracle_sample(budget_s: float, start: int = 0, max_pairs: int = 1 << 30):
    """Times the oracle (1 thread) on whole (batch, KV head) pairs of one pass: at
    least one pair, then more while the budget lasts (at most max_pairs),
    starting from pair `start`."""
    code = _ORACLE_SAMPLE.format(root=ROOT, wl=WORKLOAD, budget_s=budget_s, start=start, stride=1,
                                 max_pairs=max_pairs)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=_oracle_env())
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    from two_stage_kv_gb300 import synth
    wl = synth.WORKLOADS[WORKLOAD]
    pass_s = d["seconds"] * d["total_pairs"] / d["pairs"]      # pairs are independent
    value = wl.B * wl.steps / pass_s
    return value, d, pass_s


def oracle_parallel(budget_s: float, procs: int):
    """The oracle on all host cores: `procs` single-threaded processes, each
    taking every procs-th (batch, KV head) pair of one pass (pairs are
    independent).  Returns (pairs done, total pairs, slowest process's compute
    seconds)."""
    from two_stage_kv_gb300 import synth
    wl = synth.WORKLOADS[WORKLOAD]
    total = wl.B * wl.Hkv
    procs = max(1, min(procs, total))
    per = (total + procs - 1) // procs
    runs = []
    for i in range(procs):
        code = _ORACLE_SAMPLE.format(root=ROOT, wl=WORKLOAD, budget_s=budget_s, start=i, stride=procs,
                                     max_pairs=per)
        runs.append(subprocess.Popen([sys.executable, "-c", code], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                     text=True, env=_oracle_env()))
    done, slowest = 0, 0.0
    for r in runs:
        out, err = r.communicate()
        if r.returncode != 0:
            raise RuntimeError(err[-2000:])
        d = json.loads(out.strip().splitlines()[-1])
        done += d["pairs"]
        slowest = max(slowest, d["seconds"])
    return done, total, slowest


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline_obj(budget_s=15.0):
    from two_stage_kv_gb300 import synth
    wl = synth.WORKLOADS[WORKLOAD]
    cores = host_cores()
    done, total, secs = oracle_parallel(budget_s, cores)
    pass_s = secs * total / done
    value = wl.B * wl.steps / pass_s
    v1, d1, _ = oracle_sample(min(budget_s, 10.0))
    return {"value": round(value, 3), "unit": "tokens/s", "cores": min(cores, total), "kind": "oracle",
            "sample": f"{done} of {total} (batch, KV head) pairs of one pass (stage 1, KT, {wl.steps} decode steps) "
                      f"split over {min(cores, total)} single-threaded processes, slowest {secs:.1f} s of "
                      f"compute, scaled by pair count; numpy fp64",
            "single_thread": {"value": round(v1, 3), "cores": 1,
                              "sample": f"{d1['pairs']} pairs in {d1['seconds']:.1f} s on one thread, scaled"}}


def run_reference(args):
    from two_stage_kv_gb300 import synth
    wl = synth.WORKLOADS[WORKLOAD]
    # each step = one bounded sample (one pair's share of a pass); the run is time-boxed
    steps_run, secs, pairs = 0, 0.0, 0
    tbox = 150.0
    for i in range(args.warmup + args.steps):
        value, d, pass_s = oracle_sample(0.0, start=i, max_pairs=1)     # exactly one pair per step
        if i >= args.warmup:
            steps_run += 1
            secs += d["seconds"]
            pairs += d["pairs"]
        if secs > tbox:
            break
    pass_s = secs * (wl.B * wl.Hkv) / max(pairs, 1)
    value = wl.B * wl.steps / pass_s
    cores = 1
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1,
            "steps": steps_run, "warmup": args.warmup, "ms_per_step": round(secs / max(steps_run, 1) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": wl.B, "context": wl.S, "budget": wl.t,
                       "decode_steps_per_pass": wl.steps},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{pairs} (batch, KV head) pairs, one per step, each a full share of one "
                                       f"pass; scaled by the 64 pairs of the batch"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    line = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline_obj()
        print(json.dumps(line))


if __name__ == "__main__":
    main()
