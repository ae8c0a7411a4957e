"""The ncu summaries under profiles/ (host only): every quoted ncu command
leaves the GPU's clocks alone, every summary that records DRAM bytes names
its kernel source and either matches it or says it was captured on an
earlier revision, and the bench line's traffic figure for its dominant
kernel comes from a summary of the current source."""
import glob
import hashlib
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUMMARIES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.txt"))
                   + glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def commands(text):
    """Shell commands quoted in a summary, continuation lines joined."""
    lines = [re.sub(r"^#\s?", "", ln).strip() for ln in text.splitlines()]
    out, cur = [], ""
    for ln in lines:
        cur = f"{cur} {ln}" if cur else ln
        if cur.endswith("\\"):
            cur = cur[:-1].rstrip()
            continue
        out.append(cur)
        cur = ""
    return [c for c in out if re.match(r"ncu\s", c)]


def fields(text):
    vals = {}
    for ln in text.splitlines():
        if ":" in ln and not ln.startswith("#"):
            k, v = ln.split(":", 1)
            vals[k.strip()] = v.strip()
    return vals


def test_summaries_present():
    names = {os.path.basename(p) for p in SUMMARIES}
    for want in ("gemm_v2lite_prefill.txt", "gemm_decode.txt", "router_v2lite_prefill.txt",
                 "gather_v2lite_prefill.txt", "combine_split_v2lite_prefill.txt",
                 "plan_v2lite_prefill.txt", "launches_v2lite_prefill.md",
                 "launches_decode_26layers.md"):
        assert want in names, want


def test_every_ncu_command_keeps_the_clocks():
    seen = 0
    for p in SUMMARIES:
        for c in commands(open(p).read()):
            assert "--clock-control none" in c, (os.path.basename(p), c)
            seen += 1
    assert seen >= 10


def test_source_hashes_current_or_marked():
    for p in SUMMARIES:
        text = open(p).read()
        vals = fields(text)
        if "dram_bytes_per_launch" not in vals:
            continue
        src = vals.get("kernel_source")
        assert src and os.path.exists(os.path.join(ROOT, src)), os.path.basename(p)
        with open(os.path.join(ROOT, src), "rb") as f:
            current = hashlib.sha256(f.read()).hexdigest() == vals.get("kernel_source_sha256")
        assert current or "earlier revision" in text, os.path.basename(p)


def test_bench_traffic_from_current_summaries():
    for workload in ("v2lite_prefill", "decode"):
        t = bench.traffic_from_profile("gemm", workload)
        assert t is not None and t > 1e9, workload


def test_tracked_bench_lines_meet_the_targets():
    """The tracked bench lines: V2-Lite prefill at >= 60 % of its tensor
    roofline, the 26-layer decode pass at >= 70 % of its HBM roofline, each
    with clocks sampled under load and no slowdown reason, an end-to-end
    figure through host buffers and the dominant kernel's DRAM traffic."""
    import json
    for fname, bound, target in (("bench_v2lite_prefill.json", "tensor", 0.60),
                                 ("bench_decode_26layers.json", "hbm", 0.70)):
        with open(os.path.join(ROOT, "profiles", fname)) as f:
            line = json.load(f)
        pr = line["path_roofline"]
        assert pr["bound"] == bound and pr["frac"] >= target, (fname, pr["frac"])
        assert abs(pr["roofline_ms"] / line["ms_per_step"] - pr["frac"]) < 1e-9
        clk = line["clocks"]
        assert clk["samples"] >= 1 and clk["sm_mhz"] >= 0.95 * clk["sm_max_mhz"], clk
        assert not set(clk["reasons"]) & {"hw_slowdown", "hw_thermal_slowdown",
                                          "sw_thermal_slowdown"}, clk
        assert line["warmup"] >= 3 and line["gpu_launches"] > 0
        e2e = line["e2e"]
        assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
        assert e2e["ms_per_step"] >= line["ms_per_step"]
        assert line["roofline"]["traffic"] and 0 < line["roofline"]["frac"] <= 1.05
