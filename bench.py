"""Benchmark of the GDN recurrent-state decode step on GB300.

Headline: GDN decode tokens/s at B=256, Hk=16, Hv=32, dk=dv=128 (bf16
activations, fp32 state pool of 512 slots), and the decode kernel's achieved
HBM bandwidth against the measured peak. One "step" is one decode step of the
whole batch: gating, q/k normalisation, slot gather, fused update + readout,
round + scatter -- all inside one kernel launch. The same JSON line also
carries narrow-state decode, the ReplaySSM step and the T=4 verify window,
the speculative-step baseline, and a Mamba2 layer's decode and ReplaySSM step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs under torch.distributed.run, one process per GPU, each with its
own replica of the batch (the step has no cross-sequence exchange): weak
scaling, barrier + synchronize around the timed region, max time over ranks.
--impl reference times the CPU oracle (the plain fp64 C implementation) on
the host cores for the same metric and workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN decode tokens/s at B=256,Hv=32,d=128; achieved HBM GB/s vs GB300 peak"
B, HK, HV, DK, DV = 256, 16, 32, 128, 128
NUM_SLOTS = 2 * B
L_RING, T_VERIFY = 16, 4
# Mamba2 layer: groups, heads, state dim, head dim
M2_G, M2_H, M2_N, M2_P = 8, 128, 128, 64
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0  # dense bf16 burst, one earlier measurement on a GB300
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, ~8 TB/s nominal
KERNEL_SOURCES = ["gdn_decode.cuh", "gdn_device.cuh", "gdn_launch.cuh"]


# ------------------------------------------------------------------ bytes


def decode_bytes_per_token(state_bytes: int, in_bytes: int = 2, out_bytes: int = 4) -> int:
    """Algorithmic HBM bytes of one decode step of one sequence (all heads):
    state read + write, q and k (per key head), v, a, b, output, slot index."""
    return (2 * HV * DK * DV * state_bytes + 2 * HK * DK * in_bytes + HV * DV * in_bytes + 2 * HV * in_bytes +
            HV * DV * out_bytes + 4)


def replay_unit_bytes(count: int, T: int, fold: bool, ckpt_bytes: int, in_bytes: int = 2, out_bytes: int = 4,
                      read_bytes: int = 0) -> int:
    """Algorithmic bytes of one ReplaySSM call for one (sequence, value head):
    checkpoint read, the `count` buffered ring entries read (raw k + the fp32
    record {alpha, beta, w}), T tokens of inputs (q/k shared by Hv/Hk value
    heads), T appended entries (raw k, raw v, record), T outputs, pointers,
    and on a fold the checkpoint write. With a read copy of `read_bytes` per
    element, a call that does not fold reads only the copy; a fold reads and
    writes the master and writes the copy, and the tokens after it use the
    fresh copy without reading it back."""
    rec = (4 + DV) * 4
    cells = DK * DV
    if read_bytes:
        state = cells * (2 * ckpt_bytes + read_bytes) if fold else cells * read_bytes
    else:
        state = cells * ckpt_bytes * (2 if fold else 1)
    inputs = T * (2 * DK * in_bytes * HK // HV + DV * in_bytes + 2 * in_bytes)
    return (state + count * (DK * in_bytes + rec) + inputs + T * (DK * in_bytes + DV * in_bytes + rec) +
            T * DV * out_bytes + 16)


def mamba2_decode_bytes_per_token(state_bytes: int, in_bytes: int = 2, out_bytes: int = 4) -> int:
    """Algorithmic bytes of one Mamba2 decode step of one sequence (all heads): state read +
    write, B and C (per group), x, dt, output, slot index."""
    return (2 * M2_H * M2_N * M2_P * state_bytes + 2 * M2_G * M2_N * in_bytes + M2_H * M2_P * in_bytes +
            M2_H * in_bytes + M2_H * M2_P * out_bytes + 4)


def mamba2_replay_unit_bytes(count: int, fold: bool, ckpt_bytes: int, in_bytes: int = 2, out_bytes: int = 4) -> int:
    """Algorithmic bytes of one Mamba2 ReplaySSM step of one (sequence, head): checkpoint read,
    `count` buffered entries (raw B + the fp32 record {alpha, delta, 1, 0, w}), the token's
    inputs (B, C shared by H/G heads), the appended entry (raw B, raw x, record), the output,
    pointers, and on a fold the checkpoint write."""
    rec = (4 + M2_P) * 4
    state = M2_N * M2_P * ckpt_bytes
    inputs = 2 * M2_N * in_bytes * M2_G // M2_H + M2_P * in_bytes + in_bytes
    return (state * (2 if fold else 1) + count * (M2_N * in_bytes + rec) + inputs +
            (M2_N * in_bytes + M2_P * in_bytes + rec) + M2_P * out_bytes + 16)


def spec_bytes_per_seq(T: int, state_bytes: int, in_bytes: int = 2, out_bytes: int = 4) -> int:
    """Algorithmic bytes of one speculative step with one state copy per window token, one
    sequence (all heads): the source state read, T state copies written, T tokens of inputs,
    T outputs, T + 1 slot indices."""
    state = HV * DK * DV * state_bytes
    return (state * (1 + T) + T * (2 * HK * DK * in_bytes + HV * DV * in_bytes + 2 * HV * in_bytes) +
            T * HV * DV * out_bytes + 4 * (1 + T))


# ------------------------------------------------------------------ helpers


def load_peaks() -> tuple[float, str, str]:
    """The HBM peak fractions are taken against: the measured copy bandwidth of the GB300s
    when MEASURED_PEAKS.json is present, else the fallback figure; with how it was measured."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", str(d.get("how", ""))[:160]
    except Exception:
        return FALLBACK_HBM_GBS, "fallback", "one earlier copy-bandwidth measurement on a GB300"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "hybrid_ssm_gated_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic() -> float | None:
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source."""
    import re

    path = os.path.join(ROOT, "profiles", "decode_kernel_b256_dram_traffic.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    sha = re.search(r"^kernel_source_sha: (\w+)", text, re.M)
    val = re.search(r"^dram_bytes_per_launch: (\d+)", text, re.M)
    if not sha or not val or sha.group(1) != kernel_source_hash():
        return None
    return float(val.group(1))


def pci_bus_id(dev: int) -> str | None:
    for name in ("libcudart.so", "libcudart.so.13", "libcudart.so.12"):
        try:
            rt = ctypes.CDLL(name)
            buf = ctypes.create_string_buffer(64)
            if rt.cudaDeviceGetPCIBusId(buf, 64, dev) == 0:
                return buf.value.decode()
        except OSError:
            continue
    return None


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev: int):
        self.proc = None
        self.target = None
        bus = pci_bus_id(dev)
        try:
            rows = subprocess.run(["nvidia-smi", "--query-gpu=index,pci.bus_id", "--format=csv,noheader"],
                                  capture_output=True, text=True, timeout=20).stdout.strip().splitlines()
            for r in rows:
                idx, b = [x.strip() for x in r.split(",")]
                if bus and b.lower().endswith(bus.lower()[-12:]):
                    self.target = idx
            if self.target is None and len(rows) == 1:
                self.target = rows[0].split(",")[0].strip()
        except Exception:
            self.target = None

    def __enter__(self):
        if self.target is not None:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=20)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ ranks


def reduce_max(x: float, world: int, device="cpu") -> float:
    """Max of x over the ranks of the default process group (timing only)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, elapsed_ms_max: float, world: int) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (elapsed_ms_max / 1e3)


# ------------------------------------------------------------------ GPU arm


def gpu_arm(args, rank: int, world: int) -> dict | None:
    import numpy as np
    import torch
    import torch.distributed as dist

    from hybrid_ssm_gated_gb300 import build, gdn
    from hybrid_ssm_gated_gb300 import workload as wl

    build.build()
    gdn.lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = wl.WORKLOADS["decode_b256_f32"].with_(seed=rank)
    A_log, dt_bias = (torch.from_numpy(t).to(dev) for t in wl.head_params(w))
    slots = torch.from_numpy(wl.slots(w)).to(dev)
    gen = torch.Generator(device=dev).manual_seed(1234 + rank)

    def randn(*shape, dtype=torch.bfloat16, std=1.0):
        return (torch.randn(*shape, generator=gen, device=dev) * std).to(dtype)

    q, k = randn(B, HK, DK), randn(B, HK, DK)
    v, a, b = randn(B, HV, DV), randn(B, HV), randn(B, HV)
    out = torch.empty(B, HV, DV, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x: float) -> float:
        return reduce_max(x, world, dev)

    def timed(fn, steps, warmup, per_launch=True):
        """Run warmup, then `steps` timed calls; returns (elapsed ms over ranks, mean launch ms)."""
        for _ in range(warmup):
            fn()
        barrier()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)] \
            if per_launch else []
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(steps):
            if per_launch:
                evs[i][0].record(stream)
            fn()
            if per_launch:
                evs[i][1].record(stream)
        t1.record(stream)
        barrier()
        elapsed = t0.elapsed_time(t1)
        launch = statistics.fmean(s.elapsed_time(e) for s, e in evs) if per_launch else elapsed / steps
        return max_over_ranks(elapsed), launch

    peak, peak_kind, peak_how = load_peaks()
    result = {}

    # -------- headline: decode, fp32 state pool
    pool = (torch.randn(NUM_SLOTS, HV, DV, DK, generator=gen, device=dev) * 0.1).float()
    step = lambda: gdn.gdn_decode_step(pool, slots, q, k, v, a, b, A_log, dt_bias, out, err, stream)
    sampler = ClockSampler(dev.index)
    for _ in range(args.warmup):
        step()
    with sampler:
        elapsed, launch_ms = timed(step, args.steps, 0)
    clocks = sampler.summary()
    bpt = decode_bytes_per_token(4)
    tok_s = job_tokens_per_s(B * args.steps, elapsed, world)
    achieved = bpt * B / (launch_ms / 1e3) / 1e9
    result.update({
        "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "gdn_decode_b256_fp32_state", "B": B, "Hk": HK, "Hv": HV, "dk": DK, "dv": DV,
                   "state_dtype": "fp32", "in_dtype": "bf16", "out_dtype": "fp32", "num_slots": NUM_SLOTS,
                   "slots": "seeded permutation", "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: 512 MiB of state read+written per step (L2 129 MB)"},
        "hbm_gbs": achieved,
        "bytes_per_token": bpt,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic(), "peak_kind": peak_kind, "peak_how": peak_how,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "kernel": "gdn::decode_kernel<float, dk=128> (16 consumer warps in groups of 4, 6 chunk stages)",
                     "launch_us": launch_ms * 1e3,
                     "algorithmic_bytes_per_launch": bpt * B},
        "clocks": clocks,
        "gpu_launches": args.steps,
    })
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during the headline run")

    # -------- e2e through the public API with host buffers: every step copies its inputs from pinned
    # host memory and its output back, pipelined as a serving loop would run it -- step i+1's inputs go
    # up on one copy stream and step i-1's output comes down on another while step i computes (two
    # device buffers of each)
    pin = lambda t: t.cpu().pin_memory()
    hin = tuple(pin(t) for t in (q, k, v, a, b, slots))
    dbuf = [tuple(torch.empty_like(t) for t in (q, k, v, a, b, slots)) for _ in range(2)]
    douts = [torch.empty_like(out) for _ in range(2)]
    houts = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    in_ready, kern_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_run(nsteps: int, start: torch.cuda.Event) -> None:
        def h2d(i):
            j = i % 2
            up.wait_event(start)
            if i >= 2:
                up.wait_event(kern_done[j])  # step i-2 has read buffer j
            with torch.cuda.stream(up):
                for d, h in zip(dbuf[j], hin):
                    d.copy_(h, non_blocking=True)
                in_ready[j].record(up)

        h2d(0)
        for i in range(nsteps):
            j = i % 2
            if i + 1 < nsteps:
                h2d(i + 1)
            stream.wait_event(in_ready[j])
            if i >= 2:
                stream.wait_event(out_done[j])  # step i-2's output has left buffer j
            dq, dk_, dv_, da, db, ds = dbuf[j]
            gdn.gdn_decode_step(pool, ds, dq, dk_, dv_, da, db, A_log, dt_bias, douts[j], err, stream)
            kern_done[j].record(stream)
            down.wait_event(kern_done[j])
            with torch.cuda.stream(down):
                houts[j].copy_(douts[j], non_blocking=True)
                out_done[j].record(down)
        stream.wait_event(out_done[(nsteps - 1) % 2])  # the last output is in host memory

    e2e_steps = max(10, args.steps // 4)
    for _ in range(max(3, args.warmup // 4)):
        w0 = ev()
        w0.record(stream)
        e2e_run(2, w0)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps, e0)
    e1.record(stream)
    barrier()
    e_elapsed = max_over_ranks(e0.elapsed_time(e1))
    h2d = sum(t.numel() * t.element_size() for t in hin)
    result["e2e"] = {"value": world * B * e2e_steps / (e_elapsed / 1e3), "unit": "tokens/s",
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": houts[0].numel() * houts[0].element_size(),
                     "steps": e2e_steps, "ms_per_step": e_elapsed / e2e_steps,
                     "pipeline": "inputs up and outputs down on two copy streams, overlapped with the kernel"}
    result["gpu_launches"] += e2e_steps
    del pool

    # -------- other modes (same JSON line)
    modes = {}
    msteps = max(20, args.steps // 10)
    for name, sdt, ss in (("decode_bf16_state", torch.bfloat16, 2), ("decode_fp16_state", torch.float16, 2)):
        p = (torch.randn(NUM_SLOTS, HV, DV, DK, generator=gen, device=dev) * 0.1).to(sdt)
        el, lm = timed(lambda: gdn.gdn_decode_step(p, slots, q, k, v, a, b, A_log, dt_bias, out, err, stream),
                       msteps, args.warmup)
        bt = decode_bytes_per_token(ss)
        gbs = bt * B / (lm / 1e3) / 1e9
        modes[name] = {"tokens_per_s": world * B * msteps / (el / 1e3), "us_per_step": el / msteps * 1e3,
                       "hbm_gbs": gbs, "frac": gbs / peak, "bytes_per_token": bt}
        result["gpu_launches"] += msteps
        del p

    offsets = wl.start_offsets(wl.WORKLOADS["replay_b256_f32"])
    slot_np = wl.slots(w)
    for ckname, cdt, cs, rdt, rs in (("fp32", torch.float32, 4, None, 0), ("bf16", torch.bfloat16, 2, None, 0),
                                     ("fp32_bf16read", torch.float32, 4, torch.bfloat16, 2)):
        cache = gdn.ReplayCache.allocate(NUM_SLOTS, HV, DK, DV, L_RING, cdt, torch.bfloat16, device=dev,
                                         read_dtype=rdt)
        cache.ckpt.normal_(0, 0.1, generator=gen)
        if rdt is not None:
            cache.ckpt_read.copy_(cache.ckpt.to(rdt))
        counts = np.zeros(NUM_SLOTS, dtype=np.int64)
        counts[slot_np] = offsets
        cache.pos.copy_(torch.from_numpy(np.repeat(counts[:, None], HV, 1).astype(np.int32)))
        # warm the ring so buffered entries hold real data: run L steps first
        out1 = torch.empty(B, 1, HV, DV, device=dev)
        rstep = lambda: gdn.gdn_replay_step(cache, slots, q, k, v, a, b, A_log, dt_bias, out1, err, stream)
        for _ in range(L_RING):
            rstep()
        torch.cuda.synchronize()
        c = (cache.pos - cache.ckpt_pos)[slots.long(), 0].cpu().numpy().astype(np.int64)
        rsteps = max(32, (args.steps // 20) // L_RING * L_RING)
        total_bytes = 0
        cc = c.copy()
        for _ in range(rsteps):  # host replay of the ring counts: fold when an append would overflow
            fold = cc + 1 > L_RING
            total_bytes += HV * sum(replay_unit_bytes(int(x), 1, bool(f), cs, read_bytes=rs)
                                    for x, f in zip(cc, fold))
            cc = np.where(fold, 0, cc) + 1
        el, lm = timed(rstep, rsteps, 3)
        gbs = total_bytes / rsteps / (lm / 1e3) / 1e9
        modes[f"replay_step_{ckname}_ckpt"] = {
            "tokens_per_s": world * B * rsteps / (el / 1e3), "us_per_step": el / rsteps * 1e3, "hbm_gbs": gbs,
            "frac": gbs / peak, "bytes_per_token": total_bytes / rsteps / B, "L": L_RING,
            "start_offsets": "uniform in [0, 15]",
            "state_write_bytes_per_token": HV * DK * DV * (cs + rs) / L_RING,
            "speedup_vs_decode": (result["ms_per_step"] * 1e3 if cs == 4 else modes["decode_bf16_state"]["us_per_step"])
            / (el / rsteps * 1e3)}
        result["gpu_launches"] += rsteps

        # verify T=4 + rollback, accepted uniform in {0..3}
        T = T_VERIFY
        q4, k4 = randn(B, T, HK, DK), randn(B, T, HK, DK)
        v4, a4, b4 = randn(B, T, HV, DV), randn(B, T, HV), randn(B, T, HV)
        out4 = torch.empty(B, T, HV, DV, device=dev)
        acc = torch.randint(0, T, (B,), generator=gen, device=dev, dtype=torch.int32)

        def vround():
            gdn.gdn_verify_window(cache, slots, q4, k4, v4, a4, b4, A_log, dt_bias, out4, err, stream)
            gdn.gdn_rollback(cache, slots, acc, T, err, stream)

        vrounds = max(16, args.steps // 40)
        torch.cuda.synchronize()
        cv = (cache.pos - cache.ckpt_pos)[slots.long(), 0].cpu().numpy().astype(np.int64)
        acc_np = acc.cpu().numpy().astype(np.int64)
        el, lm = timed(vround, vrounds, 3)
        vbytes = 0
        for _ in range(3 + vrounds):  # host replay of the counts through warm-up and timed rounds
            fold = cv + T > L_RING
            vbytes_round = HV * sum(replay_unit_bytes(int(x), T, bool(f), cs, read_bytes=rs)
                                   for x, f in zip(cv, fold))
            cv = np.where(fold, 0, cv) + 1 + acc_np
            vbytes = vbytes_round  # bytes of the last round (the counts cycle; rounds differ little)
        accepted_tokens = float((acc.float() + 1).sum().item())
        vgbs = vbytes / (el / vrounds / 1e3) / 1e9
        modes[f"verify_T4_{ckname}_ckpt"] = {
            "window_tokens_per_s": world * B * T * vrounds / (el / 1e3),
            "accepted_tokens_per_s": world * accepted_tokens * vrounds / (el / 1e3),
            "us_per_round": el / vrounds * 1e3, "T": T, "L": L_RING, "hbm_gbs": vgbs, "frac": vgbs / peak,
            "bytes_per_round": vbytes}
        result["gpu_launches"] += 2 * vrounds
        del cache
    # the baseline the verify window replaces: T=4 window with one state copy per token
    T = T_VERIFY
    perm = torch.randperm(B * (T + 1), generator=gen, device=dev).to(torch.int32)
    ssrc, sdst = perm[:B].contiguous(), perm[B:].reshape(B, T).contiguous()
    q4, k4 = randn(B, T, HK, DK), randn(B, T, HK, DK)
    v4, a4, b4 = randn(B, T, HV, DV), randn(B, T, HV), randn(B, T, HV)
    out4 = torch.empty(B, T, HV, DV, device=dev)
    for sname, sdt, ss in (("fp32", torch.float32, 4), ("bf16", torch.bfloat16, 2)):
        sp = (torch.randn(B * (T + 1), HV, DV, DK, generator=gen, device=dev) * 0.1).to(sdt)
        srounds = max(16, args.steps // 40)
        el, lm = timed(lambda: gdn.gdn_spec_step(sp, ssrc, sdst, q4, k4, v4, a4, b4, A_log, dt_bias, out4, err, stream),
                       srounds, 3)
        sb = spec_bytes_per_seq(T, ss) * B
        sgbs = sb / (lm / 1e3) / 1e9
        modes[f"spec_T4_{sname}_state"] = {
            "window_tokens_per_s": world * B * T * srounds / (el / 1e3), "us_per_round": el / srounds * 1e3,
            "T": T, "hbm_gbs": sgbs, "frac": sgbs / peak, "bytes_per_round": sb,
            "state_write_bytes_per_window_token": HV * DK * DV * ss}
        result["gpu_launches"] += srounds
        del sp
    result["gpu_launches"] += mamba2_modes(modes, timed, peak, args, world, dev, gen, err, stream)
    result["gpu_launches"] += prefill_modes(modes, timed, args, world, dev, gen, err, stream)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during the mode runs")
    result["modes"] = modes
    result["drift"] = {"workload_decays": drift_modes(dev, gen, err, stream),
                       "long_memory": drift_modes(dev, gen, err, stream, a_shift=-5.0)}
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during the drift runs")
    return result


def fp32_alu_peak_tflops(dev) -> tuple[float, str]:
    """FP32 FMA peak: SMs x 128 FP32 lanes x 2 flops x the maximum SM clock."""
    import torch

    props = torch.cuda.get_device_properties(dev)
    mhz = None
    try:
        q = subprocess.run(["nvidia-smi", "-i", str(dev.index), "--query-gpu=clocks.max.sm",
                            "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
        mhz = float(q.stdout.strip().splitlines()[0])
    except Exception:
        pass
    if not mhz:
        mhz = 2070.0
    sms = props.multi_processor_count
    return sms * 128 * 2 * mhz * 1e6 / 1e12, f"{sms} SMs x 128 x 2 x {mhz:.0f} MHz"


def prefill_mma_flops(B: int, Hv: int, dv: int, tokens: int, interval: int = 64) -> int:
    """MMA flops of the chunked tensor-core prefill for B sequences of `tokens` tokens: per chunk of 64 tokens
    (the write-back interval dividing 64) and 128 state rows, S0 [K;Q]^T (128x128x128), [K;Q] K^T (128x64x128),
    Y T^T and delta^T P^T (128x64x64 each), delta^T K~ (128x128x64), at 2 flops a multiply-add."""
    chunks = B * Hv * (dv // 128) * ((tokens + min(64, interval) - 1) // min(64, interval))
    return chunks * 2 * (128 * 128 * 128 + 128 * 64 * 128 + 2 * 128 * 64 * 64 + 128 * 128 * 64)


def prefill_bytes(B: int, Hk: int, Hv: int, dk: int, dv: int, tokens: int, state_bytes: int, in_bytes: int = 2,
                  out_bytes: int = 4) -> int:
    """Algorithmic HBM bytes of a prefill call: every token's q, k, v, a, b read and output written, and each
    (sequence, head) state read once and written once."""
    per_token = 2 * Hk * dk * in_bytes + Hv * dv * in_bytes + 2 * Hv * in_bytes + Hv * dv * out_bytes
    return B * tokens * per_token + 2 * B * Hv * dv * dk * state_bytes


def prefill_modes(modes, timed, args, world, dev, gen, err, stream) -> int:
    """Prefill of 19 sequences of 2048 tokens (Hk=16, Hv=32, dk=dv=128, bf16 activations), state written
    back every 64 tokens, fp32 and bf16 state: tokens/s. The fp32 state runs the sequential kernel: its rate
    is the rule's 7 dk dv flops per token and head against the FP32 FMA peak. The bf16 state runs the
    chunked kernel on the tcgen05 tensor cores (TF32 operands): its rate is the MMA flops per launch against
    a TF32 peak, the measured bf16 GEMM rate times the nominal dense TF32 / BF16 ratio (1.1 / 2.25 PFLOP/s),
    with its HBM fraction beside it. Returns the number of timed launches."""
    import numpy as np
    import torch

    from hybrid_ssm_gated_gb300 import gdn
    from hybrid_ssm_gated_gb300 import workload as wl

    w = wl.WORKLOADS["prefill_b19_f32"]
    total = w.B * w.prefill_len
    cu = torch.from_numpy(np.arange(w.B + 1, dtype=np.int32) * w.prefill_len).to(dev)
    slots = torch.from_numpy(wl.slots(w)).to(dev)
    A_log, dt_bias = (torch.from_numpy(t).to(dev) for t in wl.head_params(w))
    rnd = lambda *shape: torch.randn(*shape, generator=gen, device=dev).to(torch.bfloat16)
    q, k, v = rnd(total, w.Hk, w.dk), rnd(total, w.Hk, w.dk), rnd(total, w.Hv, w.dv)
    a, b = rnd(total, w.Hv), rnd(total, w.Hv)
    out = torch.empty(total, w.Hv, w.dv, device=dev)
    peak, peak_note = fp32_alu_peak_tflops(dev)
    flops = 7 * w.dk * w.dv * w.Hv * total
    mma_flops = prefill_mma_flops(w.B, w.Hv, w.dv, w.prefill_len)
    bf16_peak, bf16_note = 0.0, "MEASURED_PEAKS.json absent"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16_peak, bf16_note = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        bf16_peak, bf16_note = FALLBACK_BF16_TFLOPS, "fallback"
    tf32_peak = bf16_peak * 1.1 / 2.25
    hbm_peak, _, _ = load_peaks()
    calls = max(5, args.steps // 200)
    for name, sdt in (("fp32", torch.float32), ("bf16", torch.bfloat16)):
        pool = (torch.randn(w.num_slots, w.Hv, w.dv, w.dk, generator=gen, device=dev) * 0.1).to(sdt)
        el, lm = timed(lambda: gdn.gdn_prefill(pool, slots, cu, q, k, v, a, b, A_log, dt_bias, out, err, 64, stream),
                       calls, 3)
        entry = {"tokens_per_s": world * total * calls / (el / 1e3), "us_per_call": el / calls * 1e3,
                 "sequences": w.B, "tokens_per_sequence": w.prefill_len, "state_write_interval": 64}
        nbytes = prefill_bytes(w.B, w.Hk, w.Hv, w.dk, w.dv, w.prefill_len, pool.element_size())
        gbs = nbytes / (lm / 1e3) / 1e9
        if name == "fp32":
            tf = flops / (lm / 1e3) / 1e12
            entry.update({"kernel": "prefill_kernel (sequential, FP32 FMA)", "bound": "alu", "alu_tflops": tf,
                          "alu_peak_tflops": peak, "frac": tf / peak, "peak_derivation": peak_note,
                          "flops_per_token": flops / total})
        else:
            tf = mma_flops / (lm / 1e3) / 1e12
            entry.update({"kernel": "prefill_tc_kernel (chunked, tcgen05 TF32)", "bound": "tensor",
                          "tensor_tflops": tf, "tf32_peak_tflops": tf32_peak, "frac": tf / tf32_peak,
                          "peak_derivation": f"{bf16_note} bf16 {bf16_peak:.0f} TFLOP/s x 1.1 / 2.25",
                          "mma_flops_per_launch": mma_flops})
        entry.update({"hbm_gbs": gbs, "hbm_frac": gbs / hbm_peak})
        modes[f"prefill_{name}_state"] = entry
        del pool
    return 2 * calls


def mamba2_modes(modes, timed, peak, args, world, dev, gen, err, stream) -> int:
    """Mamba2 layer (B = 256, 8 groups, 128 heads, state 128, head dim 64): decode with an fp32 /
    bf16 state pool of 2B slots, and the ReplaySSM step (L = 16, start offsets in [0, 15]) with an
    fp32 / bf16 checkpoint. Returns the number of timed launches."""
    import numpy as np
    import torch

    from hybrid_ssm_gated_gb300 import gdn
    from hybrid_ssm_gated_gb300 import workload as wl

    w = wl.WORKLOADS["mamba2_b256_f32"]
    A_log, dt_bias, D = (torch.from_numpy(t).to(dev) for t in wl.mamba2_params(w))
    slots = torch.from_numpy(wl.slots(w)).to(dev)
    rnd = lambda *shape: torch.randn(*shape, generator=gen, device=dev).to(torch.bfloat16)
    x, dt, Bm, Cm = rnd(B, M2_H, M2_P), rnd(B, M2_H), rnd(B, M2_G, M2_N), rnd(B, M2_G, M2_N)
    out = torch.empty(B, M2_H, M2_P, device=dev)
    launches = 0
    msteps = max(20, args.steps // 10)
    decode_us = {}
    for name, sdt, ss in (("fp32", torch.float32, 4), ("bf16", torch.bfloat16, 2)):
        pool = (torch.randn(2 * B, M2_H, M2_P, M2_N, generator=gen, device=dev) * 0.1).to(sdt)
        el, lm = timed(lambda: gdn.mamba2_decode_step(pool, slots, x, dt, Bm, Cm, A_log, dt_bias, D, out, err, stream),
                       msteps, args.warmup)
        bt = mamba2_decode_bytes_per_token(ss)
        gbs = bt * B / (lm / 1e3) / 1e9
        decode_us[name] = el / msteps * 1e3
        modes[f"mamba2_decode_{name}_state"] = {
            "tokens_per_s": world * B * msteps / (el / 1e3), "us_per_step": decode_us[name], "hbm_gbs": gbs,
            "frac": gbs / peak, "bytes_per_token": bt}
        launches += msteps
        del pool
    offsets = wl.start_offsets(wl.WORKLOADS["mamba2_replay_b256_f32"])
    slot_np = wl.slots(w)
    for ckname, cdt, cs in (("fp32", torch.float32, 4), ("bf16", torch.bfloat16, 2)):
        cache = gdn.ReplayCache.allocate(2 * B, M2_H, M2_N, M2_P, L_RING, cdt, torch.bfloat16, device=dev)
        cache.ckpt.normal_(0, 0.1, generator=gen)
        counts = np.zeros(2 * B, dtype=np.int64)
        counts[slot_np] = offsets
        cache.pos.copy_(torch.from_numpy(np.repeat(counts[:, None], M2_H, 1).astype(np.int32)))
        out1 = torch.empty(B, 1, M2_H, M2_P, device=dev)
        rstep = lambda: gdn.mamba2_replay_step(cache, slots, x, dt, Bm, Cm, A_log, dt_bias, D, out1, err, stream)
        for _ in range(L_RING):  # the ring holds real entries before timing
            rstep()
        torch.cuda.synchronize()
        cc = (cache.pos - cache.ckpt_pos)[slots.long(), 0].cpu().numpy().astype(np.int64)
        rsteps = max(32, (args.steps // 20) // L_RING * L_RING)
        total = 0
        for _ in range(rsteps):  # host replay of the ring counts: fold when an append would overflow
            fold = cc + 1 > L_RING
            total += M2_H * sum(mamba2_replay_unit_bytes(int(c), bool(f), cs) for c, f in zip(cc, fold))
            cc = np.where(fold, 0, cc) + 1
        el, lm = timed(rstep, rsteps, 3)
        gbs = total / rsteps / (lm / 1e3) / 1e9
        us = el / rsteps * 1e3
        modes[f"mamba2_replay_step_{ckname}_ckpt"] = {
            "tokens_per_s": world * B * rsteps / (el / 1e3), "us_per_step": us, "hbm_gbs": gbs, "frac": gbs / peak,
            "bytes_per_token": total / rsteps / B, "L": L_RING, "start_offsets": "uniform in [0, 15]",
            "speedup_vs_decode": decode_us[ckname] / us,
            "state_write_bytes_per_token": M2_H * M2_N * M2_P * cs / L_RING}
        launches += rsteps
        del cache
    return launches


def drift_modes(dev, gen, err, stream, steps: int = 200, a_shift: float = 0.0) -> dict:
    """Low-precision drift on one token stream (untimed). B = 256 sequences, 32 heads, d = 128, bf16
    activations, 200 steps from one common initial state (N(0, 0.1) in bf16, so every storage dtype
    starts from the same values), through:
      - decode with an fp32, bf16 and fp16 state pool (the state is rounded on every step);
      - the ReplaySSM step (L = 16, every ring empty at the start) with a bf16 checkpoint, and with an
        fp32 master checkpoint plus a bf16 read copy (the state is rounded only when the ring folds).
    The reference is the fp32-state decode of the same stream, on every (sequence, head); the parity
    tests check that run against the fp64 oracle within 1e-4 and the low-precision modes against the
    oracle with the same rounding points. For each mode: the largest |output - reference| over all
    steps, the RMS of that difference, the state after the last fold (or the final state, for decode)
    against the reference state at the same position, and the requantisations of each (sequence,
    head)'s stored state: one per step for decode, one per fold for replay, counted from the
    checkpoint pointers the kernels move. The ReplaySSM article (section "缓存输入而非状态", its
    precision paragraph) says replay requantises the low-precision checkpoint about L times less
    often. a_shift is added to A_log: -5 gives decays of 0.97 to 0.99 per token, a long memory in
    which roundings accumulate (the workload's own gates forget a rounding within a few tokens)."""
    import torch

    from hybrid_ssm_gated_gb300 import gdn
    from hybrid_ssm_gated_gb300 import workload as wl

    w = wl.WORKLOADS["decode_b256_bf16"]
    A_log, dt_bias = (torch.from_numpy(t).to(dev) for t in wl.head_params(w))
    A_log = A_log + a_shift
    slots = torch.from_numpy(wl.slots(w)).to(dev)
    sl = slots.long()
    bf, f16, f32 = torch.bfloat16, torch.float16, torch.float32
    S0 = (torch.randn(NUM_SLOTS, HV, DV, DK, generator=gen, device=dev) * 0.1).to(bf)
    pools = {"fp32": S0.to(f32), "bf16": S0.clone(), "fp16": S0.to(f16)}
    caches = {}
    for name, cdt, rdt in (("bf16", bf, None), ("fp32_bf16copy", f32, bf)):
        c = gdn.ReplayCache.allocate(NUM_SLOTS, HV, DK, DV, L_RING, cdt, bf, device=dev, read_dtype=rdt)
        c.ckpt.copy_(S0.to(cdt))
        if rdt is not None:
            c.ckpt_read.copy_(S0)
        caches[name] = c
    modes = ["decode_bf16", "decode_fp16", "replay_bf16_ckpt", "replay_fp32_master_bf16_copy"]
    outs = {m: torch.empty(B, HV, DV, device=dev) for m in ["decode_fp32"] + modes}
    out_max = {m: torch.zeros((), device=dev) for m in modes}
    out_sq = {m: torch.zeros((), dtype=torch.float64, device=dev) for m in modes}
    folds = {m: torch.zeros((), dtype=torch.int64, device=dev) for m in modes[2:]}
    snap = None  # the reference state after the last multiple of L tokens, where the last fold stands
    for t in range(steps):
        rnd = lambda *shape: torch.randn(*shape, generator=gen, device=dev).to(bf)
        q, k, v, a, b = rnd(B, HK, DK), rnd(B, HK, DK), rnd(B, HV, DV), rnd(B, HV), rnd(B, HV)
        for m, p in (("decode_fp32", pools["fp32"]), ("decode_bf16", pools["bf16"]), ("decode_fp16", pools["fp16"])):
            gdn.gdn_decode_step(p, slots, q, k, v, a, b, A_log, dt_bias, outs[m], err, stream)
        for m, c in (("replay_bf16_ckpt", caches["bf16"]), ("replay_fp32_master_bf16_copy", caches["fp32_bf16copy"])):
            before = c.ckpt_pos[sl].clone()
            gdn.gdn_replay_step(c, slots, q, k, v, a, b, A_log, dt_bias, outs[m], err, stream)
            folds[m] += (c.ckpt_pos[sl] != before).sum()
        for m in modes:
            d = outs[m] - outs["decode_fp32"]
            out_max[m] = torch.maximum(out_max[m], d.abs().max())
            out_sq[m] += (d.double() ** 2).sum()
        if (t + 1) % L_RING == 0:
            snap = pools["fp32"][sl].clone()
    ref = pools["fp32"][sl]
    units = B * HV
    state = {
        "decode_bf16": (pools["bf16"][sl].float() - ref).abs().max(),
        "decode_fp16": (pools["fp16"][sl].float() - ref).abs().max(),
        "replay_bf16_ckpt": (caches["bf16"].ckpt[sl].float() - snap).abs().max(),
        "replay_fp32_master_bf16_copy": (caches["fp32_bf16copy"].ckpt_read[sl].float() - snap).abs().max(),
    }
    master = float((caches["fp32_bf16copy"].ckpt[sl] - snap).abs().max())
    rep = {"steps": steps, "B": B, "L": L_RING, "A_log_shift": a_shift, "reference": "fp32-state decode of the same stream",
           "fields": "out_max, out_rms, state_max vs the reference; requantisations per (sequence, head)"}
    for m in modes:
        rq = steps if m.startswith("decode") else float(folds[m]) / units
        rep[m] = [float(f"{float(out_max[m]):.4g}"), float(f"{(float(out_sq[m]) / (units * DV * steps)) ** 0.5:.4g}"),
                  float(f"{float(state[m]):.4g}"), rq]
    rep["replay_fp32_master_bf16_copy_master_max"] = float(f"{master:.4g}")
    rep["requant_ratio_decode_over_replay"] = float(f"{steps / rep['replay_bf16_ckpt'][3]:.4g}")
    return rep


def summary(res: dict) -> dict:
    """Every configuration of the line in a few characters, the last key of the line."""
    m = res["modes"]
    peak = res["roofline"]["peak"]
    g = lambda x: float(f"{x:.3g}")
    f = lambda x: round(x, 3)
    row = lambda tok, frac: [g(tok), f(frac), f(frac * peak / NOMINAL_HBM_GBS)]
    s = {"fields": "tokens/s, frac of measured HBM peak, frac of nominal 8 TB/s (prefill: FP32 ALU frac)",
         "decode_fp32": row(res["value"], res["roofline"]["frac"])}
    for k, v in m.items():
        tok = v.get("tokens_per_s", v.get("window_tokens_per_s"))
        if k.startswith("prefill"):
            s[k] = [g(tok), f(v["frac"])]
        else:
            s[k] = row(tok, v["frac"])
        if "speedup_vs_decode" in v:
            s[k].append(round(v["speedup_vs_decode"], 3))
    d = res.get("drift")
    if d:
        s["drift_rms_out"] = {v: [d[v][k][1] for k in ("decode_bf16", "replay_bf16_ckpt",
                                                       "replay_fp32_master_bf16_copy")] for v in d}
        s["requant_decode_replay"] = [d["workload_decays"]["decode_bf16"][3],
                                      d["workload_decays"]["replay_bf16_ckpt"][3]]
    cb = res.get("cpu_baseline")
    if cb:
        s["oracle_tok_s"] = [g(cb["value"]), cb["cores"], g(cb.get("value_1_thread", 0.0))]
    return s


# ------------------------------------------------------------------ CPU oracle


def oracle_decode_rate(seconds: float = 15.0, sample_seqs: int = 32, seconds_1t: float = 5.0) -> dict:
    """Time the CPU oracle on a bounded sample of the headline workload:
    `sample_seqs` sequences x all 32 heads per step, steps repeated until
    `seconds` of wall time, all host cores; then the same on one thread for
    about `seconds_1t`."""
    import numpy as np

    import oracle
    from hybrid_ssm_gated_gb300 import workload as wl

    w = wl.WORKLOADS["decode_b256_f32"].with_(B=sample_seqs, num_slots=sample_seqs, slot_mode="identity")
    pool = np.stack([wl.slot_state(w, s) for s in range(sample_seqs)])
    A_log, dt_bias = wl.head_params(w)
    slots = wl.slots(w)
    cores = os.cpu_count() or 1
    run = lambda x: oracle.decode_step(pool, "f32", slots, x["q"], x["k"], x["v"], x["a"], x["b"], "bf16", A_log,
                                       dt_bias, nthreads=cores)
    x0 = wl.step_inputs(w, 0)
    ts = time.perf_counter()
    run(x0)  # calibration step
    steps = int(min(2000, max(1, seconds / max(time.perf_counter() - ts, 1e-6))))
    xs = [wl.step_inputs(w, s) for s in range(1, steps + 1)]
    ts = time.perf_counter()
    for x in xs:
        run(x)
    el = time.perf_counter() - ts
    # one thread: a few steps of the same sample
    run1 = lambda x: oracle.decode_step(pool, "f32", slots, x["q"], x["k"], x["v"], x["a"], x["b"], "bf16", A_log,
                                        dt_bias, nthreads=1)
    ts1 = time.perf_counter()
    n1 = 0
    while n1 < len(xs) and (n1 == 0 or time.perf_counter() - ts1 < seconds_1t):
        run1(xs[n1])
        n1 += 1
    el1 = time.perf_counter() - ts1
    return {"value": sample_seqs * steps / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{sample_seqs} of the 256 sequences x {HV} heads x {steps} decode steps of the B=256 "
                      f"workload (fp32 state, bf16 inputs), fp64 C oracle, OpenMP over (sequence, head)",
            "seconds": el, "value_1_thread": sample_seqs * n1 / el1,
            "sample_1_thread": f"the same sample, {n1} steps on one thread", "seconds_1_thread": el1}


def reference_arm(args, rank: int, world: int) -> None:
    """The oracle as the reference arm: W untimed and K timed steps, each one oracle decode step over a
    bounded sample of the headline workload's sequences (all 32 heads), sized so that the whole run takes
    about two minutes on the host cores."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from hybrid_ssm_gated_gb300 import workload as wl

    nseq = 32
    w = wl.WORKLOADS["decode_b256_f32"].with_(B=nseq, num_slots=nseq, slot_mode="identity")
    pool = np.stack([wl.slot_state(w, s) for s in range(nseq)])
    A_log, dt_bias = wl.head_params(w)
    slots = wl.slots(w)
    xs = [wl.step_inputs(w, s) for s in range(8)]
    cores = os.cpu_count() or 1

    def run(n, x):
        oracle.decode_step(pool, "f32", slots[:n], x["q"][:n], x["k"][:n], x["v"][:n], x["a"][:n], x["b"][:n],
                           "bf16", A_log, dt_bias, nthreads=cores)

    run(nseq, xs[0])  # builds the oracle and pages the library in
    ts = time.perf_counter()
    run(nseq, xs[1])
    per_seq = (time.perf_counter() - ts) / nseq
    n = int(min(nseq, max(1, round(120.0 / (args.steps + args.warmup) / per_seq))))
    for i in range(args.warmup):
        run(n, xs[i % 8])
    ts = time.perf_counter()
    for i in range(args.steps):
        run(n, xs[i % 8])
    el = time.perf_counter() - ts
    v = n * args.steps / el
    cb = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
          "sample": f"a sample of {n} of the 256 sequences x {HV} heads per step of the B=256 workload "
                    f"(fp32 state, bf16 inputs), {args.steps} timed steps after {args.warmup}, fp64 C oracle, "
                    f"OpenMP over (sequence, head); tokens/s counts the sampled sequences",
          "seconds": el}
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "gdn_decode_b256_fp32_state", "B": B, "Hk": HK, "Hv": HV, "dk": DK, "dv": DV,
                       "state_dtype": "fp32", "in_dtype": "bf16"},
            "cpu_baseline": cb, "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ profiling cases


def run_case(args) -> None:
    """Run a few untimed launches of one kernel for a profiler (no JSON line).

    decode:  B sequences, fp32/bf16/fp16 state pool of 2B slots.
    replay:  ReplaySSM steps, L=16 ring pre-filled to start offsets in [0, 15]; with
             --read-dtype, an fp32 checkpoint plus a read copy of that dtype.
    verify:  T=4 verify windows + rollbacks on the same cache.
    spec:    T=4 speculative steps with one state copy per window token, pool of 5B slots.
    mamba2_decode / mamba2_replay: the Mamba2 layer (8 groups, 128 heads, state 128, head dim 64),
             decode on a pool of 2B slots, or ReplaySSM steps with L=16 and offsets in [0, 15].
    prefill: B sequences of 2048 tokens, state written back every 64 tokens.
    """
    import numpy as np
    import torch

    from hybrid_ssm_gated_gb300 import build, gdn

    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev).manual_seed(0)
    Bc = args.B
    sdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[args.state_dtype]
    rnd = lambda *s: torch.randn(*s, generator=g, device=dev).to(torch.bfloat16)
    A_log = torch.rand(HV, generator=g, device=dev) * 2
    dt_bias = torch.rand(HV, generator=g, device=dev) * 2 - 1
    slots = torch.randperm(2 * Bc, generator=g, device=dev)[:Bc].to(torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if args.case == "prefill":
        Tp = 2048
        cu = torch.arange(Bc + 1, device=dev, dtype=torch.int32) * Tp
        q, k, v = rnd(Bc * Tp, HK, DK), rnd(Bc * Tp, HK, DK), rnd(Bc * Tp, HV, DV)
        a, b = rnd(Bc * Tp, HV), rnd(Bc * Tp, HV)
        pool = (torch.randn(2 * Bc, HV, DV, DK, generator=g, device=dev) * 0.1).to(sdt)
        out = torch.empty(Bc * Tp, HV, DV, device=dev)
        for _ in range(args.steps):
            gdn.gdn_prefill(pool, slots, cu, q, k, v, a, b, A_log, dt_bias, out, err, 64)
    elif args.case.startswith("mamba2"):
        from hybrid_ssm_gated_gb300 import workload as wl

        A2, dt2, D2 = (torch.from_numpy(t).to(dev) for t in wl.mamba2_params(wl.WORKLOADS["mamba2_b256_f32"]))
        x, dtt, Bm, Cm = rnd(Bc, M2_H, M2_P), rnd(Bc, M2_H), rnd(Bc, M2_G, M2_N), rnd(Bc, M2_G, M2_N)
        out = torch.empty(Bc, M2_H, M2_P, device=dev)
        if args.case == "mamba2_decode":
            pool = (torch.randn(2 * Bc, M2_H, M2_P, M2_N, generator=g, device=dev) * 0.1).to(sdt)
            for _ in range(args.steps):
                gdn.mamba2_decode_step(pool, slots, x, dtt, Bm, Cm, A2, dt2, D2, out, err)
        else:
            cache = gdn.ReplayCache.allocate(2 * Bc, M2_H, M2_N, M2_P, L_RING, sdt, torch.bfloat16, device=dev)
            cache.ckpt.normal_(0, 0.1, generator=g)
            off = torch.randint(0, L_RING, (2 * Bc, 1), generator=g, device=dev).to(torch.int32)
            cache.pos.copy_(off.expand(2 * Bc, M2_H))
            for _ in range(args.steps):
                gdn.mamba2_replay_step(cache, slots, x, dtt, Bm, Cm, A2, dt2, D2, out, err)
    elif args.case == "decode":
        pool = (torch.randn(2 * Bc, HV, DV, DK, generator=g, device=dev) * 0.1).to(sdt)
        q, k, v, a, b = rnd(Bc, HK, DK), rnd(Bc, HK, DK), rnd(Bc, HV, DV), rnd(Bc, HV), rnd(Bc, HV)
        out = torch.empty(Bc, HV, DV, device=dev)
        for _ in range(args.steps):
            gdn.gdn_decode_step(pool, slots, q, k, v, a, b, A_log, dt_bias, out, err)
    elif args.case == "spec":
        T = T_VERIFY
        pool = (torch.randn(Bc * (T + 1), HV, DV, DK, generator=g, device=dev) * 0.1).to(sdt)
        perm = torch.randperm(Bc * (T + 1), generator=g, device=dev).to(torch.int32)
        src, dst = perm[:Bc].contiguous(), perm[Bc:].reshape(Bc, T).contiguous()
        q, k, v, a, b = rnd(Bc, T, HK, DK), rnd(Bc, T, HK, DK), rnd(Bc, T, HV, DV), rnd(Bc, T, HV), rnd(Bc, T, HV)
        out = torch.empty(Bc, T, HV, DV, device=dev)
        for _ in range(args.steps):
            gdn.gdn_spec_step(pool, src, dst, q, k, v, a, b, A_log, dt_bias, out, err)
    else:
        T = T_VERIFY if args.case == "verify" else 1
        rdt = {None: None, "bf16": torch.bfloat16, "f16": torch.float16}[args.read_dtype]
        cache = gdn.ReplayCache.allocate(2 * Bc, HV, DK, DV, L_RING, sdt, torch.bfloat16, device=dev, read_dtype=rdt)
        cache.ckpt.normal_(0, 0.1, generator=g)
        if rdt is not None:
            cache.ckpt_read.copy_(cache.ckpt.to(rdt))
        off = torch.randint(0, L_RING, (2 * Bc, 1), generator=g, device=dev).to(torch.int32)
        cache.pos.copy_(off.expand(2 * Bc, HV))
        q, k, v, a, b = rnd(Bc, T, HK, DK), rnd(Bc, T, HK, DK), rnd(Bc, T, HV, DV), rnd(Bc, T, HV), rnd(Bc, T, HV)
        out = torch.empty(Bc, T, HV, DV, device=dev)
        acc = torch.randint(0, T, (Bc,), generator=g, device=dev, dtype=torch.int32)
        for _ in range(args.steps):
            if T == 1:
                gdn.gdn_replay_step(cache, slots, q, k, v, a, b, A_log, dt_bias, out, err)
            else:
                gdn.gdn_verify_window(cache, slots, q, k, v, a, b, A_log, dt_bias, out, err)
                gdn.gdn_rollback(cache, slots, acc, T, err)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise SystemExit(f"device error word {int(err.item())}")
    print(f"case {args.case} ok")


# ------------------------------------------------------------------ main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["decode", "replay", "verify", "spec", "mamba2_decode", "mamba2_replay",
                                       "prefill"],
                    help="run --steps untimed launches of one kernel for a profiler and exit")
    ap.add_argument("--B", type=int, default=B, help="batch of --case")
    ap.add_argument("--state-dtype", default="f32", choices=["f32", "bf16", "f16"], help="state dtype of --case")
    ap.add_argument("--read-dtype", default=None, choices=["bf16", "f16"],
                    help="read copy of the replay/verify checkpoint of --case (needs --state-dtype f32)")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    import torch

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    res = gpu_arm(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = oracle_decode_rate()
        res["summary"] = summary(res)  # last: a compact copy of every configuration's figures
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
