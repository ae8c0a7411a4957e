"""Benchmark of the AFD FFN-side step (fan-in -> router -> permute -> grouped
SwiGLU experts + shared expert -> combine -> per-peer split) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload v2lite_prefill|decode|skewed|fanin]

One step = afd_ffn_forward over one freshly packed fan-in (for the decode
workload: all 26 layers, each re-packed).  Timing: CUDA events around each
forward on the library's stream; the packs (the attention side's remote
write) and an L2 flush run between the timed windows.  Rank 0 prints one
JSON line.  --impl reference times the CPU oracle (the plain C reference of
the same computation) on a bounded sample of the same workload.
"""
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

METRIC = "FFN-side MoE tokens/s + TFLOP/s (V2-Lite shape, bf16); % of roofline, 1xGB300"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return PEAKS_FALLBACK, "fallback"


def dist_init(n_gpus):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, ws):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v, ws):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index):
        fd, self.path = tempfile.mkstemp(prefix="afd_clocks_", suffix=".csv")
        self.f = os.fdopen(fd, "w")
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
        self.f.close()

    def summary(self):
        if not self.proc:
            os.unlink(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# algorithmic work (roofline numerators)
# ---------------------------------------------------------------------------
def stage_work(w, T, nz=None):
    """Algorithmic FLOPs / bytes per launch of each stage for T tokens (nz:
    experts with rows, whose weights the GEMMs read; all E by default)."""
    H, I, Is, k, E = w.hidden, w.inter, w.shared_inter, w.topk, w.num_experts
    nz = E if nz is None else nz
    ab = w.act_bytes
    # the routed partial outputs y reach the combine as 24-bit floats (3
    # bytes: its weighted sum may cancel, so bf16 is too coarse) and the
    # shared output s as fp32
    return {
        "router": {"flops": 2 * T * H * E, "bytes": T * H * ab + H * E * 4 + T * k * 8},
        # each token row read once from its slot, each routed copy written
        # once (the shared expert reads its rows in place)
        "gather": {"bytes": T * H * ab + T * k * H * ab},
        # weights of the experts with rows + the shared expert, rows in, outputs
        "gemm_swiglu": {"flops": 2 * T * H * 2 * (k * I + Is),
                        "bytes": (nz * 2 * I + 2 * Is) * H * 2 + (T * k + T) * H * ab
                        + (T * k * I + T * Is) * ab},
        "gemm_down": {"flops": 2 * T * H * (k * I + Is),
                      "bytes": (nz * I + Is) * H * 2 + (T * k * I + T * Is) * ab
                      + T * k * H * 3 + T * H * 4},
        "combine_split": {"bytes": T * k * H * 3 + T * H * 4 + T * H * ab + T * k * 8},
    }


def with_gemm_pair(work):
    """Work of the one-launch GEMM pair (stage "gemm"): the SwiGLU and down
    projections' FLOPs and bytes together."""
    sw, dn = work.get("gemm_swiglu"), work.get("gemm_down")
    if sw and dn:
        work["gemm"] = {"flops": sw["flops"] + dn["flops"], "bytes": sw["bytes"] + dn["bytes"]}
    return work


def stage_work_grouped(w, T, Rr, nz=None):
    """Algorithmic work per stage of the grouped form: Rr routed rows arrive
    grouped (no router, no combine: the rows' outputs go back)."""
    H, I, Is = w.hidden, w.inter, w.shared_inter
    nz = w.num_experts if nz is None else nz
    ab = w.act_bytes
    return {
        # each received row read once and placed once
        "gather": {"bytes": Rr * H * ab * 2},
        "gemm_swiglu": {"flops": 2 * H * 2 * (Rr * I + T * Is),
                        "bytes": (nz * 2 * I + 2 * Is) * H * 2 + (Rr + T) * H * ab
                        + (Rr * I + T * Is) * ab},
        "gemm_down": {"flops": 2 * H * (Rr * I + T * Is),
                      "bytes": (nz * I + Is) * H * 2 + (Rr * I + T * Is) * ab + Rr * H * ab
                      + T * H * 4},
        "combine_split": {"bytes": Rr * H * ab * 2 + T * H * (4 + ab)},
    }


def path_roofline_grouped(w, T, Rr, counts_nonzero, pk):
    """Roofline of one grouped forward: FLOP = 6 H (Rr I + T I_s); bytes =
    weights of every expert with rows + shared + rows and shared rows in +
    their outputs."""
    H, I, Is = w.hidden, w.inter, w.shared_inter
    flops = 6 * H * (Rr * I + T * Is)
    wbytes = counts_nonzero * 3 * H * I * 2 + 3 * H * Is * 2
    abytes = 2 * (Rr + T) * H * w.act_bytes
    t_flop = flops / (pk["bf16_tflops"] * 1e12)
    t_mem = (wbytes + abytes) / (pk["hbm_gbs"] * 1e9)
    return flops, wbytes + abytes, max(t_flop, t_mem), ("tensor" if t_flop >= t_mem else "hbm")


def path_roofline(w, T, counts_nonzero, pk):
    """Roofline time of one forward: max(FLOP / bf16 peak, bytes / HBM) with
    bytes = weights of every expert that received a token + shared + router
    weight + activations (x in, shared_x in, output)."""
    H, I, Is, E = w.hidden, w.inter, w.shared_inter, w.num_experts
    flops = T * w.flops_per_token()
    wbytes = counts_nonzero * 3 * H * I * 2 + 3 * H * Is * 2 + H * E * 4
    abytes = 3 * T * H * w.act_bytes
    t_flop = flops / (pk["bf16_tflops"] * 1e12)
    t_mem = (wbytes + abytes) / (pk["hbm_gbs"] * 1e9)
    return flops, wbytes + abytes, max(t_flop, t_mem), ("tensor" if t_flop >= t_mem else "hbm")


def traffic_from_profile(kernel, workload):
    """dram bytes per launch recorded by an ncu capture under profiles/, valid
    only while the kernel source is unchanged (sha256 recorded with it)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    src = vals.get("kernel_source")
    if not src or "dram_bytes_per_launch" not in vals:
        return None
    with open(os.path.join(ROOT, src), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != vals.get("kernel_source_sha256"):
            return None
    return float(vals["dram_bytes_per_launch"])


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, ws, rank, local):
    import numpy as np
    import torch
    from combine_peer_slot_gb300 import afd as A
    from combine_peer_slot_gb300 import runtime as R
    from combine_peer_slot_gb300 import workloads as W

    w = workload_of(args)
    T = w.total_tokens
    grouped = args.form == "grouped"
    run = R.Runner(w, max_total_tokens=T, flags=A.AFD_CFG_SPLIT_GEMMS if args.split_gemms else 0)
    # the tensor engine runs both projections as one launch unless split
    gemm_pair = not args.split_gemms
    if grouped:  # the Attention side routes: grouped rows, no router or combine here
        run.prepare_grouped(seed=w.seed)
    pack = run.pack_grouped_all if grouped else run.pack_all
    fwd = run.forward_grouped if grouped else run.forward
    stream = run.stream
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(w.layers)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(w.layers)]

    def step(timed_stats=None):
        fwd_ms = 0.0
        for layer in range(w.layers):
            pack(layer)
            flush.zero_()
            e0[layer].record(stream)
            rc = fwd(layer)
            e1[layer].record(stream)
            if rc:
                raise A.AfdError(rc, "afd_ffn_forward")
        torch.cuda.synchronize()
        if timed_stats is not None:  # stage events: read once per step, no wait between layers
            st, _ = A.afd_stage_times(run.ctx)
            for i, v in enumerate(st):
                timed_stats[i] += v
        for layer in range(w.layers):
            fwd_ms += e0[layer].elapsed_time(e1[layer])
        return fwd_ms

    for _ in range(args.warmup):
        step()
    if run.poll() != 0:
        raise RuntimeError("device error during warm-up")
    dev_index = getattr(torch.cuda.get_device_properties(local), "pci_bus_id", None) or local
    launches0 = A.afd_launch_count(run.ctx)
    total_ms = 0.0
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(dev_index) as clk:
        t_wall = time.perf_counter()
        for _ in range(args.steps):
            total_ms += step()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(ws)
    launches = A.afd_launch_count(run.ctx) - launches0
    status = run.poll()
    if status != 0:
        raise RuntimeError(f"device error in the timed region: {A.strerror(status)}")
    # stage pass: the same K steps again with an event on the launching stream
    # between every two stages (those events cost about 2 us each on the
    # device, so the timed pass above records only the two around a forward)
    A.afd_profile(run.ctx, True)
    stage_sum = [0.0] * A.AFD_NUM_STAGES
    stage_pass_ms = 0.0
    for _ in range(args.steps):
        stage_pass_ms += step(stage_sum)
    A.afd_profile(run.ctx, False)
    if run.poll() != 0:
        raise RuntimeError("device error in the stage pass")
    ms_step = total_ms / args.steps
    ms_step_max = max_over_ranks(ms_step, ws)
    tokens_step = T * w.layers
    value = sum_over_ranks(tokens_step, ws) / (ms_step_max / 1e3)

    # roofline of the whole path and of the dominant stage
    pk, pk_kind = peaks()
    cnt = run.workspace(A.AFD_WS_COUNTS, 4 * w.num_experts).cpu().numpy().view(np.int32)
    if grouped:
        Rr = int(sum(run.g_n))
        flops, nbytes, t_roof, bound = path_roofline_grouped(w, T, Rr, int((cnt > 0).sum()), pk)
    else:
        flops, nbytes, t_roof, bound = path_roofline(w, T, int((cnt > 0).sum()), pk)
    stages = {n: stage_sum[i] / (args.steps * w.layers) for i, n in enumerate(A.STAGE_NAMES)}
    if gemm_pair:  # one launch: its events bracket both projections
        stages["gemm"] = stages.pop("gemm_swiglu") + stages.pop("gemm_down")
    dom = max(stages, key=stages.get)
    nz = int((cnt > 0).sum())
    work = with_gemm_pair(stage_work_grouped(w, T, Rr, nz) if grouped else stage_work(w, T, nz)).get(dom, {})
    # a GEMM below the ridge point (peak FLOP/s / peak bytes/s) streams its
    # weights from HBM (decode-sized fan-ins): measured against HBM then
    gemm_tensor = dom.startswith("gemm") and "flops" in work and (
        "bytes" not in work
        or work["flops"] / (pk["bf16_tflops"] * 1e12) >= work["bytes"] / (pk["hbm_gbs"] * 1e9))
    if gemm_tensor:
        ach = work["flops"] / (stages[dom] / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"],
                "peak_source": f"{pk_kind} bf16_tflops (burst)",
                "algorithmic_flops_per_launch": work["flops"]}
    else:
        ach = work.get("bytes", 0) / (stages[dom] / 1e3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "peak_source": f"{pk_kind} hbm_gbs",
                "algorithmic_bytes_per_launch": work.get("bytes", 0)}
    roof["avg_launch_ms"] = stages[dom]
    roof["traffic"] = None if grouped else traffic_from_profile(dom, args.workload)

    # end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        dt = torch.bfloat16 if w.act == "bf16" else torch.float32
        # the peers' token rows and outputs in one buffer each (views per
        # peer), so a forward's inputs go up in one copy and its outputs
        # come back in one
        offs = [0]
        for n in w.seq_lens:
            offs.append(offs[-1] + n)
        xall = torch.cat([x[:n] for x, n in zip(run.x, w.seq_lens)]).contiguous()
        outall = torch.empty((max(T, 1), w.hidden), dtype=dt, device="cuda")
        run.x = [xall[offs[p]:offs[p + 1]] for p in range(w.num_peers)]
        run.out = [outall[offs[p]:offs[p + 1]] for p in range(w.num_peers)]
        hxall = xall.cpu().pin_memory()
        houtall = torch.empty((max(T, 1), w.hidden), dtype=dt).pin_memory()
        h2d = T * w.hidden * w.act_bytes
        d2h = T * w.hidden * w.act_bytes
        if grouped:  # also the routed rows in and their expert outputs back
            hrows = [r.cpu().pin_memory() if r is not None else None for r in run.g_rows]
            hy = [torch.empty_like(y, device="cpu").pin_memory() for y in run.g_y]
            h2d += sum(r.numel() * r.element_size() for r in hrows if r is not None)
            d2h += sum(n * w.hidden * w.act_bytes for n in run.g_n)

        # every forward's inputs go up from pinned host memory and its outputs
        # come back, on a copy stream beside the library's: the next
        # forward's inputs while this one runs (once its own inputs are
        # packed), its outputs once they are unpacked (before the next
        # unpack reuses the buffers)
        cs = torch.cuda.Stream()
        ev_in, ev_packed, ev_out, ev_d2h = (torch.cuda.Event() for _ in range(4))

        def copy_inputs():
            with torch.cuda.stream(cs):
                cs.wait_event(ev_packed)
                if T:
                    xall.copy_(hxall, non_blocking=True)
                if grouped:
                    for p in range(w.num_peers):
                        if hrows[p] is not None:
                            run.g_rows[p].copy_(hrows[p], non_blocking=True)
                ev_in.record(cs)

        def e2e_step():
            for layer in range(w.layers):
                stream.wait_event(ev_in)
                with torch.cuda.stream(stream):
                    pack(layer)
                    ev_packed.record(stream)
                copy_inputs()  # the next forward's inputs
                rc = fwd(layer)
                if rc:
                    raise A.AfdError(rc, "afd_ffn_forward")
                stream.wait_event(ev_d2h)
                with torch.cuda.stream(stream):
                    if grouped:
                        run.unpack_grouped_all()
                    else:
                        run.unpack_all()
                    ev_out.record(stream)
                with torch.cuda.stream(cs):
                    cs.wait_event(ev_out)
                    if T:
                        houtall[:T].copy_(outall[:T], non_blocking=True)
                    if grouped:
                        for p in range(w.num_peers):
                            if run.g_n[p]:
                                hy[p][:run.g_n[p]].copy_(run.g_y[p][:run.g_n[p]], non_blocking=True)
                    ev_d2h.record(cs)

        copy_inputs()  # the first forward's inputs
        for _ in range(max(2, args.warmup)):
            e2e_step()
        stream.synchronize()
        cs.synchronize()
        n_e2e = max(5, args.steps // 4)
        barrier(ws)
        t = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        stream.synchronize()
        cs.synchronize()
        t = (time.perf_counter() - t) / n_e2e
        t = max_over_ranks(t, ws)
        if run.poll() != 0:
            raise RuntimeError("device error in the end-to-end loop")
        # the last outputs copied out are the last ones unpacked
        if T and not torch.equal(houtall[:T], outall[:T].cpu()):
            raise RuntimeError("end-to-end outputs differ from the device's")
        e2e = {"value": sum_over_ranks(tokens_step, ws) / t, "unit": "tokens/s",
               "ms_per_step": t * 1e3, "h2d_bytes_per_step": h2d * w.layers,
               "d2h_bytes_per_step": d2h * w.layers,
               "note": "pinned host x -> device, pack, forward, unpack, device -> pinned host; every "
                       "forward's copies inside the timed region, on a copy stream: the next forward's "
                       "inputs while this one runs, its outputs once unpacked"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not grouped:
        cpu = cpu_baseline(w, budget_s=args.cpu_budget)

    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; no model weights or dataset)",
        "config": {"workload": args.workload + ("_grouped" if grouped else ""),
                   "peers": w.num_peers, "seq_lens": w.seq_lens,
                   "total_tokens": T, "hidden": w.hidden, "experts": w.num_experts,
                   "topk": w.topk, "inter": w.inter, "shared_inter": w.shared_inter,
                   "layers": w.layers, "parallelism": f"replicas{ws}",
                   "l2": "flushed (256 MB write) before every timed forward",
                   "stage_timing": "per-stage events on the launching stream in a second "
                                   "pass of the same K steps; the timed pass records only "
                                   "the events around each forward",
                   **({"form": "grouped: the Attention side routed (seeded distinct top-k "
                               "per token); rows grouped by expert arrive, their expert "
                               "outputs go back", "routed_rows": int(sum(run.g_n))}
                      if grouped else {})},
        "tflops": flops * w.layers / (ms_step_max / 1e3) / 1e12,
        "path_roofline": {"bound": bound, "roofline_ms": t_roof * 1e3 * w.layers,
                          "frac": t_roof * 1e3 * w.layers / ms_step_max,
                          "flops_per_layer": flops, "bytes_per_layer": nbytes,
                          "peak_source": pk_kind},
        "roofline": roof, "stages_ms": stages,
        "stage_pass_ms_per_step": stage_pass_ms / args.steps, "gpu_launches": launches,
        "wall_s_timed": t_wall, "clocks": clk.summary(), "e2e": e2e, "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(out))
    run.close()


def run_serve(args, ws, rank, local):
    """The device-resident work-item loop measured: every layer's item packed
    into a stage of its own (ring_depth = layers) before the timed region,
    then one step = the whole set served back to back, by the host-described
    step per item ("host"), by the loop's eager steps ("eager") or by one
    replay of the captured loop ("graph").  All three modes run in the same
    process on the same packs; --serve names the one reported as value."""
    import numpy as np
    import torch
    from combine_peer_slot_gb300 import afd as A
    from combine_peer_slot_gb300 import runtime as R

    w = workload_of(args)
    T, L = w.total_tokens, w.layers
    grouped = args.form == "grouped"
    run = R.Runner(w, max_total_tokens=T, ring_depth=L)
    if grouped:
        run.prepare_grouped(seed=w.seed)
    slots = list(range(w.num_peers))
    form = A.AFD_FORM_GROUPED if grouped else A.AFD_FORM_TOKENS
    rc, graph, graph_kernels = A.afd_serve_graph_create(run.ctx, slots, L, form)
    if rc:
        raise A.AfdError(rc, "afd_serve_graph_create")
    stream = run.stream
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def step(mode):
        for layer in range(L):
            if grouped:
                run.pack_grouped_all(layer, stage=layer)
            else:
                run.pack_all(layer, stage=layer)
        flush.zero_()
        e0.record(stream)
        if mode == "host":
            for layer in range(L):
                rc = (run.forward_grouped if grouped else run.forward)(layer, stage=layer)
                if rc:
                    raise A.AfdError(rc, "host-described step")
        elif mode == "eager":
            rc = A.afd_ffn_serve(run.ctx, slots, L, form)
            if rc:
                raise A.AfdError(rc, "afd_ffn_serve")
        else:
            rc = A.afd_serve_graph_launch(graph)
            if rc:
                raise A.AfdError(rc, "afd_serve_graph_launch")
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    modes = ["host", "eager", "graph"]
    for _ in range(args.warmup):
        for m in modes:
            step(m)
    if run.poll() != 0:
        raise RuntimeError("device error during warm-up")
    dev_index = getattr(torch.cuda.get_device_properties(local), "pci_bus_id", None) or local
    ms = {m: 0.0 for m in modes}
    launches = {m: 0 for m in modes}
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(dev_index) as clk:
        for _ in range(args.steps):
            for m in modes:  # interleaved, so the three see the same clocks
                l0 = A.afd_launch_count(run.ctx)
                ms[m] += step(m)
                launches[m] += A.afd_launch_count(run.ctx) - l0
    barrier(ws)
    status = run.poll()
    if status != 0:
        raise RuntimeError(f"device error in the timed region: {A.strerror(status)}")
    log, served = A.afd_serve_log(run.ctx, 64)
    assert [r[1] for r in log[-L:]] == list(range(L)), "items served out of layer order"
    # the pack kernels are the Attention side's, not the step's: two launches
    # per stage with the batched packs, two per peer and stage without
    pack_launches = L * 2 * (1 if run.batched else w.num_peers)
    launches = {m: v - pack_launches * args.steps for m, v in launches.items()}
    launches["graph"] = graph_kernels * args.steps
    per = {m: max_over_ranks(v / args.steps, ws) for m, v in ms.items()}
    tokens_step = T * L
    value = sum_over_ranks(tokens_step, ws) / (per[args.serve] / 1e3)
    pk, pk_kind = peaks()
    cnt = run.workspace(A.AFD_WS_COUNTS, 4 * w.num_experts).cpu().numpy().view(np.int32)
    if grouped:
        flops, nbytes, t_roof, bound = path_roofline_grouped(w, T, int(sum(run.g_n)),
                                                             int((cnt > 0).sum()), pk)
    else:
        flops, nbytes, t_roof, bound = path_roofline(w, T, int((cnt > 0).sum()), pk)
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per[args.serve],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; no model weights or dataset)",
        "config": {"workload": args.workload + ("_grouped" if grouped else "") + "_serve",
                   "serve": args.serve, "items_per_step": L, "ring_depth": L,
                   "peers": w.num_peers, "seq_lens": w.seq_lens, "total_tokens": T,
                   "layers": L, "parallelism": f"replicas{ws}",
                   "l2": "flushed (256 MB write) before every timed step",
                   "timing": "one event pair around the whole set of items; every item "
                             "packed into its own stage before the first event"},
        "serve_ms_per_step": per, "graph_kernels": graph_kernels,
        "gpu_launches": launches[args.serve], "gpu_launches_by_mode": launches,
        "path_roofline": {"bound": bound, "roofline_ms": t_roof * 1e3 * L,
                          "frac": t_roof * 1e3 * L / per[args.serve], "peak_source": pk_kind},
        "roofline": None, "clocks": clk.summary(), "e2e": None, "cpu_baseline": None,
        "items_served": served,
    }
    if rank == 0:
        print(json.dumps(out))
    A.afd_serve_graph_destroy(graph)
    run.close()


def run_ranks(args, ws, rank, local):
    """Token-level dispatch to --ffn-ranks FFN ranks on this one GPU: per
    step, every peer's send (afd_attn_dispatch), every rank's grouped step
    over the peers (the work-item loop, counts taken on the device), every
    peer's combine (afd_attn_combine), each part between its own event pair
    on the one stream, after an L2 flush.  The ranks run one after another
    here; on ffn_size GPUs they would run side by side (rank_ms lists each)."""
    import numpy as np
    import torch
    from combine_peer_slot_gb300 import afd as A
    from combine_peer_slot_gb300 import runtime as R

    w = workload_of(args)
    T, F = w.total_tokens, args.ffn_ranks
    rs = R.RankSet(w, F, layers=1)
    stream = rs.stream
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(F + 3)]
    slots = list(range(w.num_peers))

    def step():
        rs.route()                  # the Attention side's gate: not timed
        flush.zero_()
        ev[0].record(stream)
        rs.dispatch_all()
        ev[1].record(stream)
        for r in range(F):
            rc = A.afd_ffn_serve(rs.ranks[r], slots, 1, A.AFD_FORM_GROUPED)
            if rc:
                raise A.AfdError(rc, "afd_ffn_serve")
            ev[2 + r].record(stream)
        rs.combine_all()
        ev[F + 2].record(stream)
        torch.cuda.synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(F + 2)]

    for _ in range(args.warmup):
        step()
    if rs.poll() != (0, 0):
        raise RuntimeError("device error during warm-up")
    dev_index = getattr(torch.cuda.get_device_properties(local), "pci_bus_id", None) or local
    acc = np.zeros(F + 2)
    l0 = sum(A.afd_launch_count(c) for c in rs.ranks) + sum(A.afd_attn_launch_count(a) for a in rs.attn)
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(dev_index) as clk:
        for _ in range(args.steps):
            acc += np.array(step())
    barrier(ws)
    launches = (sum(A.afd_launch_count(c) for c in rs.ranks) +
                sum(A.afd_attn_launch_count(a) for a in rs.attn) - l0)
    st = rs.poll()
    if st != (0, 0):
        raise RuntimeError(f"device error in the timed region: {st}")
    per = acc / args.steps
    dispatch_ms, rank_ms, combine_ms = per[0], list(per[1:F + 1]), per[F + 1]
    ms_step = max_over_ranks(float(per.sum()), ws)
    value = sum_over_ranks(T, ws) / (ms_step / 1e3)
    rows = [[int(v) for v in A.afd_attn_rows(a, 0, F)] for a in rs.attn]
    rows_per_rank = [sum(r[q] for r in rows) for q in range(F)]
    pk, pk_kind = peaks()
    eb = w.act_bytes
    # algorithmic bytes: the send reads every token row once and writes the
    # T*k routed rows and the T shared rows; the combine reads those rows
    # back and writes the T outputs
    moved = (T * w.topk + T) * w.hidden * eb
    send_bytes = T * w.hidden * eb + moved
    recv_bytes = moved + T * w.hidden * eb
    def hbm(nbytes, ms):
        a = nbytes / (ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": a, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": a / pk["hbm_gbs"], "peak_source": f"{pk_kind} hbm_gbs",
                "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": ms, "traffic": None}
    flops_rank = [6 * w.hidden * (rows_per_rank[q] * w.inter +
                                  sum(len(range(q, n, F)) for n in w.seq_lens) * w.shared_inter)
                  for q in range(F)]
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; no model weights or dataset)",
        "config": {"workload": f"{args.workload}_ranks{F}", "ffn_size": F, "peers": w.num_peers,
                   "seq_lens": w.seq_lens, "total_tokens": T, "experts": w.num_experts,
                   "topk": w.topk, "routed_cap_multiplier": 2.0,
                   "parallelism": f"replicas{ws}; {F} FFN ranks served one after another",
                   "l2": "flushed (256 MB write) before every timed send",
                   "gate": "the library's router on each peer's tokens, before the timed region"},
        "dispatch_ms": dispatch_ms, "rank_ms": rank_ms, "combine_ms": combine_ms,
        "rows_per_rank": rows_per_rank,
        "rank_tflops": [flops_rank[q] / (rank_ms[q] / 1e3) / 1e12 for q in range(F)],
        "roofline": hbm(send_bytes, dispatch_ms), "combine_roofline": hbm(recv_bytes, combine_ms),
        "gpu_launches": launches, "clocks": clk.summary(), "e2e": None, "cpu_baseline": None,
    }
    out["roofline"]["kernel"] = "attn_dispatch"
    out["combine_roofline"]["kernel"] = "attn_combine"
    if rank == 0:
        print(json.dumps(out))
    rs.close()


# ---------------------------------------------------------------------------
# the CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_setup(w):
    """Pack the workload into a host dispatch window for the oracle (the
    oracle's own pack) and return what forward_tokens needs."""
    import numpy as np
    from combine_peer_slot_gb300 import workloads as W
    from oracle import oracle as O
    host = W.host_inputs(w)
    L = O.slot_layout(w.num_peers, 1, w.token_cap, w.topk, w.hidden, w.act_bytes, w.num_experts,
                      w.shared_inter > 0)
    win = np.zeros(L.window_bytes, np.uint8)
    for p, x in enumerate(host["x"]):
        O.pack_slot(win, L, 1, p, 0, 0, x, w.hidden, w.act_bytes, w.token_cap, w.num_experts,
                    w.shared_inter > 0, w.shared_inter > 0, p + 1)
    wt = W.weights_to_numpy(W.expert_weights(w, 0, "cpu"))
    wt["Wg"], wt["bias"] = host["Wg"], host["bias"]
    cfg = dict(num_regions=w.num_peers, ring_depth=1, token_cap=w.token_cap, hidden=w.hidden,
               act_bytes=w.act_bytes, num_experts=w.num_experts, topk=w.topk, inter=w.inter,
               shared_inter=w.shared_inter, renorm=w.renorm, max_total_tokens=0,
               routed_scaling=w.routed_scaling)
    return cfg, win, wt


def oracle_rate(w, cfg, win, wt, n_tokens, seed=0):
    import numpy as np
    from oracle import oracle as O
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(w.total_tokens, size=min(n_tokens, w.total_tokens), replace=False))
    nthreads = os.cpu_count() or 1
    t = time.perf_counter()
    O.forward_tokens(cfg, win, wt, 0, w.seq_lens, list(range(w.num_peers)), toks,
                     nthreads=nthreads)
    return len(toks), time.perf_counter() - t, nthreads


def cpu_baseline(w, budget_s=15.0):
    cfg, win, wt = oracle_setup(w)
    n, dt, nth = oracle_rate(w, cfg, win, wt, 32)
    rate = n / dt
    n_big = int(max(32, min(w.total_tokens, rate * budget_s)))
    n2, dt2, nth = oracle_rate(w, cfg, win, wt, n_big, seed=1)
    return {"value": n2 / dt2 * 1.0, "unit": "tokens/s", "cores": nth, "kind": "oracle",
            "sample": f"{n2} tokens drawn uniformly from the {w.total_tokens}-token fan-in of "
                      f"'{w.name}' (all layer-0 experts), {dt2:.1f} s of CPU work; "
                      f"tokens/s counts one layer per token"}


def run_reference(args, ws, rank):
    if rank != 0:
        return
    w = workload_of(args)
    cfg, win, wt = oracle_setup(w)
    n, dt, nth = oracle_rate(w, cfg, win, wt, 16)
    rate = n / dt
    per_step = int(max(4, min(w.total_tokens, rate * args.ref_budget / max(1, args.steps + args.warmup))))
    for i in range(args.warmup):
        oracle_rate(w, cfg, win, wt, per_step, seed=100 + i)
    tot_n, tot_t = 0, 0.0
    for i in range(args.steps):
        n, dt, nth = oracle_rate(w, cfg, win, wt, per_step, seed=i)
        tot_n += n
        tot_t += dt
    value = tot_n / tot_t
    sample = (f"{per_step} tokens per step drawn from the {w.total_tokens}-token fan-in of "
              f"'{w.name}' (layer 0), {args.steps} steps")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
           "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded; no model weights or dataset)",
           "config": {"workload": args.workload, "peers": w.num_peers,
                      "total_tokens": w.total_tokens, "hidden": w.hidden,
                      "experts": w.num_experts, "topk": w.topk, "inter": w.inter,
                      "shared_inter": w.shared_inter, "layers": w.layers,
                      "parallelism": "host cores"},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nth, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def workload_of(args):
    from combine_peer_slot_gb300 import workloads as W
    over = {}
    if getattr(args, "form", "tokens") == "grouped":  # a slot holds a peer's n * k routed rows
        w0 = W.get(args.workload)
        lens = [int(v) for v in args.seq_lens.split(",")] if args.seq_lens else w0.seq_lens
        over["token_cap"] = -(-max(lens) * w0.topk // 64) * 64
    if args.seq_lens:
        over["seq_lens"] = [int(v) for v in args.seq_lens.split(",")]
    if args.layers:
        over["layers"] = args.layers
    return W.custom(args.workload, **over) if over else W.get(args.workload)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="v2lite_prefill",
                    choices=["v2lite_prefill", "decode", "skewed", "fanin"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--split-gemms", action="store_true",
                    help="launch the SwiGLU and down GEMMs as two kernels (AFD_CFG_SPLIT_GEMMS)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=60.0)
    ap.add_argument("--seq-lens", default="",
                    help="comma-separated per-peer token counts replacing the workload's "
                         "(smaller profiling cases of the same shapes)")
    ap.add_argument("--form", choices=["tokens", "grouped"], default="tokens",
                    help="grouped: the Attention side routes and sends rows grouped by expert")
    ap.add_argument("--layers", type=int, default=0,
                    help="number of layers replacing the workload's (smaller profiling cases)")
    ap.add_argument("--ffn-ranks", type=int, default=0,
                    help="token-level dispatch to this many FFN ranks on this GPU: the peers' "
                         "send, every rank's grouped step, the peers' combine")
    ap.add_argument("--serve", choices=["host", "eager", "graph"], default=None,
                    help="measure the device-resident work-item loop: all layers' items "
                         "packed into stages, served by host-described steps, the loop's "
                         "eager steps or a replay of its captured graph (value = this mode)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, ws, rank)
    elif args.ffn_ranks:
        run_ranks(args, ws, rank, local)
    elif args.serve:
        run_serve(args, ws, rank, local)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
