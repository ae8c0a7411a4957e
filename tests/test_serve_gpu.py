"""Device-resident work-item loop ([RFC]: Async AFD for Prefill on Ascend NPU,
"Asynchronous work-item contract" and "FFN execution modes"; [RFC]: Async GPU
Connector, "FFN main loop" and the device-side wait_any): each step waits on
the device for a ready stage, takes the layer and counts from the headers and
runs the FFN step with that layer's weights.  Checked against the
host-described step on a second context (bit for bit: the same kernels on the
same bytes) and against the CPU oracle.  Needs an sm_103a GPU."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from combine_peer_slot_gb300 import afd as A
from combine_peer_slot_gb300 import runtime as R
from combine_peer_slot_gb300 import workloads as W
from oracle import oracle as O
from tests import gpu_parity as G


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    A.lib()


def make(w, ring_depth, layers=3, **kw):
    return R.Runner(w, layers=layers, ring_depth=ring_depth, max_total_tokens=w.total_tokens, **kw)


def pack_item(run, stage, layer, counts, with_shared=None):
    """One Attention replica's send of a work item: peer p's first counts[p]
    tokens into its (p, stage) slot, tagged with the layer."""
    ws = (run.w.shared_inter > 0) if with_shared is None else with_shared
    seqs = []
    for p, n in enumerate(counts):
        run.seq += 1
        rc = A.afd_pack_slot(run.ctx, p, stage, layer, run.x[p].data_ptr() if n else 0, n, ws,
                             run.seq)
        assert rc == 0, A.strerror(rc)
        seqs.append(run.seq)
    return seqs


def slot_bytes(buf, run, p, stage, n):
    """(header, route_table rows, routed_x rows, flag) of return slot (p, stage)."""
    L, w = run.layout, run.w
    off = G.slot_off(run, p, stage)
    rb = w.hidden * w.act_bytes
    hdr = buf[off + L.header: off + L.header + 4 * (12 + w.num_experts)].copy()
    rt = buf[off + L.route_table: off + L.route_table + n * w.topk * 4].copy()
    rows = buf[off + L.routed_x: off + L.routed_x + n * rb].copy()
    flag = int(buf[:L.flags_bytes].view(np.uint64)[p * run.cfg.ring_depth + stage])
    return hdr, rt, rows, flag


def rows_f64(raw, w, n):
    if w.act == "bf16":
        return O.bf16_bits_to_f32(raw.view(np.uint16)).astype(np.float64).reshape(n, w.hidden)
    return raw.view(np.float32).astype(np.float64).reshape(n, w.hidden)


def check_item_against_oracle(run, stage, layer, counts):
    w = run.w
    win = run.window(A.AFD_DIR_DISPATCH).cpu().numpy()
    ret = run.window(A.AFD_DIR_RETURN).cpu().numpy()
    ret_orc = np.zeros_like(win)
    seen = np.zeros(w.num_peers * run.cfg.ring_depth, np.uint64)
    slots = list(range(w.num_peers))
    rc, r = O.ffn_forward(G.oracle_cfg(run), win.copy(), ret_orc, run.weights_numpy(layer), layer,
                          stage, list(counts), slots, seen)
    assert rc == 0
    start, got, ref = 0, [], []
    for p, n in enumerate(counts):
        h, rt, rows, _ = slot_bytes(ret, run, p, stage, n)
        ho, rto, _, _ = slot_bytes(ret_orc, run, p, stage, n)
        assert np.array_equal(h, ho), (p, stage)
        assert np.array_equal(rt, rto), (p, stage)
        if n:
            got.append(rows_f64(rows, w, n))
            ref.append(r["out64"][start:start + n])
        start += n
    if got:
        e = G.rel_err(np.concatenate(got), np.concatenate(ref))
        assert e <= G.tol_for(w), e


# stage -> (layer, counts per peer): stage 1 a partial fan-in, stage 2 one
# peer without tokens; layers out of order
ITEMS = {0: (2, [37, 91]), 1: (0, [20, 50]), 2: (1, [0, 91])}


@pytest.mark.parametrize("gemm", [A.AFD_GEMM_TENSOR, A.AFD_GEMM_TENSOR_1CTA, A.AFD_GEMM_SIMT])
def test_serve_takes_layer_and_counts_from_headers(gemm):
    w = W.custom("fanin", seq_lens=[37, 91])
    dev = make(w, 3, gemm=gemm)
    host = make(w, 3, gemm=gemm)
    for stage, (layer, counts) in ITEMS.items():
        pack_item(dev, stage, layer, counts)
        pack_item(host, stage, layer, counts)
    assert A.afd_ffn_serve(dev.ctx, [0, 1], 3) == 0
    for stage, (layer, counts) in ITEMS.items():
        assert A.afd_ffn_forward(host.ctx, layer, stage, counts, [0, 1]) == 0
    assert dev.poll() == 0 and host.poll() == 0
    log, served = A.afd_serve_log(dev.ctx)
    assert served == 3
    assert log == [(s, l, sum(c), 0) for s, (l, c) in ITEMS.items()]
    rd = dev.window(A.AFD_DIR_RETURN).cpu().numpy()
    rh = host.window(A.AFD_DIR_RETURN).cpu().numpy()
    for stage, (layer, counts) in ITEMS.items():
        for p, n in enumerate(counts):
            a, b = slot_bytes(rd, dev, p, stage, n), slot_bytes(rh, host, p, stage, n)
            for x, y in zip(a[:3], b[:3]):
                assert np.array_equal(x, y), (stage, p)
            assert a[3] == b[3] > 0
        check_item_against_oracle(dev, stage, layer, counts)


def test_serve_scan_order_serves_every_ready_stage():
    """Ready stages are served from the one after the stage served last: a
    stage that is not ready is passed over, and one that is ready waits for
    at most ring_depth - 1 others."""
    w = W.custom("fanin", seq_lens=[37, 91])
    run = make(w, 3)
    pack_item(run, 2, 0, [5, 6])
    pack_item(run, 1, 1, [7, 8])
    assert A.afd_ffn_serve(run.ctx, [0, 1], 2) == 0
    assert run.poll() == 0
    log, _ = A.afd_serve_log(run.ctx)
    assert [r[0] for r in log] == [1, 2]
    # next scan starts at stage 0: the stages packed now are served 0, 1, 2
    for stage in (2, 0, 1):
        pack_item(run, stage, stage, [stage + 1, 3])
    assert A.afd_ffn_serve(run.ctx, [0, 1], 3) == 0
    assert run.poll() == 0
    log, served = A.afd_serve_log(run.ctx)
    assert served == 5
    assert [r[:3] for r in log[-3:]] == [(0, 0, 4), (1, 1, 5), (2, 2, 6)]


def test_serve_graph_replays_new_items():
    """The loop captured once; each replay serves whatever the peers packed
    since (other layers, other counts) without a new capture."""
    w = W.custom("fanin", seq_lens=[37, 91])
    dev = make(w, 2)
    host = make(w, 2)
    rc, graph, kernels = A.afd_serve_graph_create(dev.ctx, [0, 1], 2)
    assert rc == 0, A.strerror(rc)
    assert kernels >= 2 * 7
    try:
        rounds = [{0: (1, [37, 91]), 1: (2, [3, 0])}, {0: (0, [1, 2]), 1: (1, [30, 90])}]
        for items in rounds:
            for stage, (layer, counts) in items.items():
                pack_item(dev, stage, layer, counts)
                pack_item(host, stage, layer, counts)
            assert A.afd_serve_graph_launch(graph) == 0
            for stage, (layer, counts) in items.items():
                assert A.afd_ffn_forward(host.ctx, layer, stage, counts, [0, 1]) == 0
            assert dev.poll() == 0 and host.poll() == 0
            rd = dev.window(A.AFD_DIR_RETURN).cpu().numpy()
            rh = host.window(A.AFD_DIR_RETURN).cpu().numpy()
            for stage, (layer, counts) in items.items():
                for p, n in enumerate(counts):
                    a, b = slot_bytes(rd, dev, p, stage, n), slot_bytes(rh, host, p, stage, n)
                    for x, y in zip(a, b):
                        assert np.array_equal(x, y), (stage, p)
                check_item_against_oracle(dev, stage, layer, counts)
        log, served = A.afd_serve_log(dev.ctx)
        assert served == 4
        assert [r[:2] for r in log] == [(0, 1), (1, 2), (0, 0), (1, 1)]
    finally:
        A.afd_serve_graph_destroy(graph)


def test_serve_timeout_then_recovers():
    """No stage ready: the bounded wait gives up with AFD_ERR_TIMEOUT, writes
    no return flag, and the context serves the next item once polled."""
    w = W.custom("fanin", seq_lens=[37, 91])
    run = make(w, 2, wait_timeout_ns=20_000_000)
    pack_item(run, 0, 0, [4, 4])
    pack_item(run, 1, 0, [4, 4])
    assert A.afd_ffn_serve(run.ctx, [0, 1], 3) == 0   # the third finds nothing
    assert run.poll() == A.AFD_ERR_TIMEOUT
    log, served = A.afd_serve_log(run.ctx)
    assert served == 2
    pack_item(run, 0, 1, [9, 10])
    assert A.afd_ffn_serve(run.ctx, [0, 1], 1) == 0
    assert run.poll() == 0
    log, served = A.afd_serve_log(run.ctx)
    assert served == 3 and log[-1][:3] == (0, 1, 19)
    check_item_against_oracle(run, 0, 1, [9, 10])


@pytest.mark.parametrize("case", ["layer_outside_table", "layers_disagree", "over_capacity",
                                  "shutdown"])
def test_serve_header_faults(case):
    """Faults the loop can only see in the headers stop it with the matching
    status; nothing is returned for the item."""
    w = W.custom("fanin", seq_lens=[37, 91])
    run = R.Runner(w, layers=2, ring_depth=1, wait_timeout_ns=20_000_000,
                   max_total_tokens=100 if case == "over_capacity" else w.total_tokens)
    want = {"layer_outside_table": A.AFD_ERR_LAYER, "layers_disagree": A.AFD_ERR_LAYER,
            "over_capacity": A.AFD_ERR_CAPACITY, "shutdown": A.AFD_ERR_SHUTDOWN}[case]
    if case == "layer_outside_table":
        pack_item(run, 0, 5, [3, 4])
    elif case == "layers_disagree":
        run.seq += 1
        assert A.afd_pack_slot(run.ctx, 0, 0, 0, run.x[0].data_ptr(), 3, 1, run.seq) == 0
        run.seq += 1
        assert A.afd_pack_slot(run.ctx, 1, 0, 1, run.x[1].data_ptr(), 4, 1, run.seq) == 0
    elif case == "over_capacity":
        pack_item(run, 0, 0, [37, 91])
    else:
        pack_item(run, 0, 0, [3, 4])
        assert A.afd_ffn_serve(run.ctx, [0, 1], 1) == 0
        assert run.poll() == 0
        run.seq += 1
        assert A.afd_announce_shutdown(run.ctx, 0, 0, run.seq) == 0
        run.seq += 1
        assert A.afd_pack_slot(run.ctx, 1, 0, 0, run.x[1].data_ptr(), 4, 1, run.seq) == 0
    ret0 = run.window(A.AFD_DIR_RETURN).cpu().numpy()[:run.layout.flags_bytes].copy()
    assert A.afd_ffn_serve(run.ctx, [0, 1], 1) == 0
    assert run.poll() == want
    ret = run.window(A.AFD_DIR_RETURN).cpu().numpy()
    assert np.array_equal(ret[:run.layout.flags_bytes], ret0)


@pytest.mark.parametrize("peers", [[0, 1], [1]])
def test_serve_grouped_form(peers):
    """The grouped form (the Attention side routed) through the loop: two
    stages with different layers; one peer alone takes the in-place path."""
    w = W.custom("fanin", seq_lens=[37, 91], token_cap=384)
    dev = make(w, 2)
    host = make(w, 2)
    for r in (dev, host):
        r.prepare_grouped(seed=3)
    ws = w.shared_inter > 0
    for stage, layer in ((0, 2), (1, 0)):
        for r in (dev, host):
            for p in peers:
                r.seq += 1
                rows = r.g_rows[p]
                n = w.seq_lens[p]
                assert A.afd_pack_grouped(r.ctx, p, stage, layer, rows.data_ptr(), r.g_n[p],
                                          r.g_list[p], r.x[p].data_ptr(), n, ws, r.seq) == 0
    assert A.afd_ffn_serve(dev.ctx, peers, 2, A.AFD_FORM_GROUPED) == 0
    for stage, layer in ((0, 2), (1, 0)):
        assert A.afd_ffn_forward_grouped(host.ctx, layer, stage, [host.g_n[p] for p in peers],
                                         [w.seq_lens[p] for p in peers], peers) == 0
    assert dev.poll() == 0 and host.poll() == 0
    log, _ = A.afd_serve_log(dev.ctx)
    assert log == [(0, 2, sum(w.seq_lens[p] for p in peers), sum(dev.g_n[p] for p in peers)),
                   (1, 0, sum(w.seq_lens[p] for p in peers), sum(dev.g_n[p] for p in peers))]
    rd = dev.window(A.AFD_DIR_RETURN).cpu().numpy()
    rh = host.window(A.AFD_DIR_RETURN).cpu().numpy()
    L = dev.layout
    for stage in (0, 1):
        for p in peers:
            off = G.slot_off(dev, p, stage)
            rb = w.hidden * w.act_bytes
            for field, n in ((L.header, 4 * (12 + w.num_experts)), (L.routed_x, dev.g_n[p] * rb),
                             (L.shared_x, w.seq_lens[p] * rb)):
                assert np.array_equal(rd[off + field: off + field + n], rh[off + field: off + field + n])


@pytest.mark.parametrize("workload", ["v2lite_prefill", "decode"])
def test_serve_full_size_matches_host_step(workload):
    """At full size (the bench's launch shapes): the same packed bytes served
    by the loop and by the host-described step on one context give
    bit-identical return windows (the device-described kernels against the
    host-described ones; the host step is checked against the oracle in
    test_parity_gpu.py)."""
    w = W.get(workload)
    run = R.Runner(w, layers=1, max_total_tokens=w.total_tokens)
    ret = []
    for mode in ("host", "serve"):
        run.pack_all(0)
        if mode == "host":
            assert run.forward(0) == 0
        else:
            assert A.afd_ffn_serve(run.ctx, list(range(w.num_peers)), 1) == 0
        assert run.poll() == 0
        win = run.window(A.AFD_DIR_RETURN)
        L = run.layout
        # payload of every return slot (the flags and echoed seqs differ)
        rb = w.hidden * w.act_bytes
        got = []
        for p, n in enumerate(w.seq_lens):
            off = L.flags_bytes + p * run.cfg.ring_depth * L.slot_bytes
            got.append(win[off + L.routed_x: off + L.routed_x + n * rb].cpu().numpy().copy())
            got.append(win[off + L.route_table: off + L.route_table + n * w.topk * 4].cpu().numpy().copy())
            hdr = win[off + L.header: off + L.header + 4 * (12 + w.num_experts)].cpu().numpy().copy()
            got.append(np.delete(hdr.view(np.int32), [3, 4]))   # all but seq / echo_seq
        ret.append(got)
    for a, b in zip(*ret):
        assert np.array_equal(a, b)
    run.close()
