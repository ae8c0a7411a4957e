"""The bench's algorithmic work per stage and the bound it measures each GEMM
against (host only: no GPU)."""
import bench
from combine_peer_slot_gb300 import workloads as W

PEAKS = {"bf16_tflops": 1940.7, "hbm_gbs": 6794.1}


def bound(work):
    t_flop = work["flops"] / (PEAKS["bf16_tflops"] * 1e12)
    t_mem = work["bytes"] / (PEAKS["hbm_gbs"] * 1e9)
    return "tensor" if t_flop >= t_mem else "hbm"


def test_gemm_work_counted_by_hand():
    """V2-Lite prefill, every expert with rows: the SwiGLU GEMM reads the
    64 experts' gate/up weights and the shared expert's, the routed and
    shared rows, and writes the SwiGLU outputs; FLOPs are 2 per MAC."""
    w = W.get("v2lite_prefill")
    T, H, I, Is, k, E = w.total_tokens, w.hidden, w.inter, w.shared_inter, w.topk, w.num_experts
    sw = bench.stage_work(w, T, E)["gemm_swiglu"]
    assert sw["flops"] == 2 * H * (T * k * 2 * I + T * 2 * Is)
    weights = (E * 2 * I * H + 2 * Is * H) * 2
    rows_in = (T * k + T) * H * 2
    rows_out = (T * k * I + T * Is) * 2
    assert sw["bytes"] == weights + rows_in + rows_out
    dn = bench.stage_work(w, T, E)["gemm_down"]
    assert dn["flops"] == 2 * H * (T * k * I + T * Is)
    # routed partials as 24-bit floats, the shared expert's output in fp32
    assert dn["bytes"] == (E * I * H + Is * H) * 2 + (T * k * I + T * Is) * 2 + T * k * H * 3 + T * H * 4


def test_gather_counts_each_row_once():
    """The gather reads every token row once from its slot and writes each
    of its k routed copies once; the shared rows are read in place."""
    w = W.get("v2lite_prefill")
    T, H, k = w.total_tokens, w.hidden, w.topk
    assert bench.stage_work(w, T)["gather"]["bytes"] == T * H * 2 + T * k * H * 2
    assert bench.stage_work_grouped(w, T, T * k)["gather"]["bytes"] == 2 * T * k * H * 2


def test_only_experts_with_rows_count():
    w = W.get("decode")
    T = w.total_tokens
    full = bench.stage_work(w, T, w.num_experts)["gemm_down"]["bytes"]
    fewer = bench.stage_work(w, T, w.num_experts - 10)["gemm_down"]["bytes"]
    assert full - fewer == 10 * w.inter * w.hidden * 2


def test_prefill_gemms_tensor_bound_decode_gemms_hbm_bound():
    for name, want in (("v2lite_prefill", "tensor"), ("decode", "hbm")):
        w = W.get(name)
        sw = bench.stage_work(w, w.total_tokens, w.num_experts)
        assert bound(sw["gemm_swiglu"]) == want, name
        assert bound(sw["gemm_down"]) == want, name


def test_grouped_form_matches_token_form_when_rows_agree():
    """The grouped form with Rr = T k routed rows does the GEMM work of the
    token form."""
    w = W.get("v2lite_prefill")
    T = w.total_tokens
    a = bench.stage_work(w, T, w.num_experts)
    b = bench.stage_work_grouped(w, T, T * w.topk, w.num_experts)
    assert a["gemm_swiglu"]["flops"] == b["gemm_swiglu"]["flops"]
    assert a["gemm_swiglu"]["bytes"] == b["gemm_swiglu"]["bytes"]
    assert a["gemm_down"]["flops"] == b["gemm_down"]["flops"]
    # the grouped form returns each row's output in the activation type,
    # the token form keeps 24 bits of it for its combine
    T, H, k = w.total_tokens, w.hidden, w.topk
    assert a["gemm_down"]["bytes"] - b["gemm_down"]["bytes"] == T * k * H * (3 - 2)


def test_stage_bytes_never_exceed_the_hbm_peak_at_recorded_times():
    """The algorithmic bytes bench.py counts for each stage, over that
    stage's time in a recorded bench line, stay under the measured HBM copy
    rate: an over-count (a row counted k times that is read once) would show
    as an impossible bandwidth.  Every expert's weights are counted (an upper
    bound)."""
    import json
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for name, fname in (("v2lite_prefill", "bench_v2lite_prefill.json"),
                        ("decode", "bench_decode_26layers.json")):
        with open(os.path.join(root, "profiles", fname)) as f:
            line = json.load(f)
        w = W.get(name)
        work = bench.with_gemm_pair(bench.stage_work(w, w.total_tokens))
        checked = 0
        for stage, ms in line["stages_ms"].items():
            nbytes = work.get(stage, {}).get("bytes")
            if nbytes:
                gbs = nbytes / (ms * 1e-3) / 1e9
                assert gbs <= PEAKS["hbm_gbs"] * 1.02, (name, stage, gbs)
                checked += 1
        assert checked >= 4, name


def test_gemm_pair_work_is_both_projections():
    w = W.get("v2lite_prefill")
    work = bench.with_gemm_pair(bench.stage_work(w, w.total_tokens))
    for key in ("flops", "bytes"):
        assert work["gemm"][key] == work["gemm_swiglu"][key] + work["gemm_down"][key]
