"""Grouped form (the Attention side routes and sends its routed rows grouped by
expert; the FFN runs each row through its expert) against the CPU oracle,
through the C ABI (needs an sm_103a GPU)."""
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


def attention_routing(rng, n, E, k):
    """Distinct top-k experts per token (the Attention side's gate; any valid
    routing will do for the FFN side)."""
    return np.argsort(rng.random((n, E)), axis=1)[:, :k].astype(np.int32)


def grouped_rows(ids, x_bits, E):
    order = np.argsort(ids.reshape(-1), kind="stable")
    k = ids.shape[1]
    rows = np.ascontiguousarray(x_bits[order // k])
    return rows, np.bincount(ids.reshape(-1), minlength=E).astype(np.int32)


def to_dev(bits, act):
    return R.act_tensor(bits, act, "cuda")


def run_grouped(w, seed, with_shared=True, slots=None, zero_rows=(), gemm=A.AFD_GEMM_TENSOR):
    """Pack every peer in grouped form, run the GPU step and the oracle on the
    same rows; return (run, gpu y/s per peer, oracle y64/s64, rows per peer)."""
    rng = np.random.default_rng(seed)
    run = R.Runner(w, max_total_tokens=w.total_tokens, gemm=gemm)
    slots = list(range(w.num_peers)) if slots is None else slots
    ws = with_shared and w.shared_inter > 0
    rows_h, gls, R_ = {}, {}, {}
    L = O.slot_layout(w.num_peers, 1, w.token_cap, w.topk, w.hidden, w.act_bytes, w.num_experts,
                      w.shared_inter > 0)
    win = np.zeros(L.window_bytes, np.uint8)
    keep = []
    for p in slots:
        n = w.seq_lens[p]
        ids = attention_routing(rng, n, w.num_experts, w.topk)
        if p in zero_rows:
            ids = ids[:0]
        rows, gl = grouped_rows(ids, run.host["x"][p], w.num_experts)
        rows_h[p], gls[p], R_[p] = rows, gl, rows.shape[0]
        run.seq += 1
        rows_d = to_dev(rows, w.act) if rows.shape[0] else None
        keep.append(rows_d)
        rc = A.afd_pack_grouped(run.ctx, p, 0, 0, rows_d.data_ptr() if rows_d is not None else 0,
                                rows.shape[0], gl, run.x[p].data_ptr() if n else 0, n, ws,
                                run.seq)
        assert rc == 0, A.strerror(rc)
        run.last_seq[(p, 0)] = run.seq
        assert O.pack_grouped(win, L, 1, p, 0, 0, rows, gl, run.host["x"][p], w.hidden,
                              w.act_bytes, w.token_cap, w.num_experts, ws, w.shared_inter > 0,
                              run.seq) == 0
    rc = A.afd_ffn_forward_grouped(run.ctx, 0, 0, [R_[p] for p in slots],
                                   [w.seq_lens[p] for p in slots], slots)
    assert rc == 0, A.strerror(rc)
    dt = torch.bfloat16 if w.act == "bf16" else torch.float32
    ys, ss = {}, {}
    for p in slots:
        n = w.seq_lens[p]
        y = torch.empty((max(R_[p], 1), w.hidden), dtype=dt, device="cuda")
        s = torch.empty((max(n, 1), w.hidden), dtype=dt, device="cuda") if ws else None
        rc = A.afd_unpack_grouped(run.ctx, p, 0, y.data_ptr() if R_[p] else 0, R_[p],
                                  s.data_ptr() if s is not None else 0, n, run.last_seq[(p, 0)])
        assert rc == 0, A.strerror(rc)
        ys[p] = y[:R_[p]].float().cpu().numpy().astype(np.float64)
        ss[p] = s[:n].float().cpu().numpy().astype(np.float64) if s is not None else None
    assert run.poll() == 0
    ret = np.zeros_like(win)
    seen = np.zeros(w.num_peers, np.uint64)
    rc, y64, s64 = O.grouped_forward(G.oracle_cfg(run), win, ret, run.weights_numpy(0), 0, 0,
                                     [R_[p] for p in slots], [w.seq_lens[p] for p in slots],
                                     slots, seen)
    assert rc == 0
    return run, ys, ss, y64, s64, R_, ret, slots


def compare(w, run, ys, ss, y64, s64, R_, ret, slots):
    tol = G.tol_for(w)
    gpu_ret = run.window(A.AFD_DIR_RETURN).cpu().numpy()
    rb = rs = 0
    errs = []
    for p in slots:
        n = w.seq_lens[p]
        ref_y = y64[rb:rb + R_[p]]
        if R_[p]:
            e = G.rel_err(ys[p], ref_y)
            errs.append(e)
            assert e <= tol, (p, e)
        if ss[p] is not None and n:
            e = G.rel_err(ss[p], s64[rs:rs + n])
            errs.append(e)
            assert e <= tol, (p, e)
        assert np.array_equal(G.header(gpu_ret, run, p), G.header(ret, run, p))
        rb += R_[p]
        rs += n
    return max(errs) if errs else 0.0


def test_grouped_fanin():
    w = W.custom("fanin", token_cap=384)
    args = run_grouped(w, seed=5)
    print("grouped fanin max|err|/rms", compare(w, *args))


def test_grouped_routed_only_with_empty_peer():
    """The routed-only protocol (no shared rows: the shared expert runs on the
    Attention side) with a peer that sends no rows and the list reordered."""
    w = W.custom("fanin", seq_lens=[37, 20, 91], token_cap=384)
    args = run_grouped(w, seed=6, with_shared=False, slots=[2, 0, 1], zero_rows=(1,))
    compare(w, *args)


@pytest.mark.parametrize("gemm", [A.AFD_GEMM_TENSOR_1CTA, A.AFD_GEMM_SIMT])
def test_grouped_other_engines(gemm):
    """The same rows through the one-CTA tensor engine and the SIMT engine."""
    w = W.custom("fanin", token_cap=384)
    compare(w, *run_grouped(w, seed=7, gemm=gemm))


def test_grouped_bad_group_list_is_a_device_error():
    """A header whose group list does not sum to routed_tokens (corrupted in
    the window after the pack): the step stops with AFD_ERR_SHAPE and no
    return flag is written."""
    w = W.custom("fanin", seq_lens=[12], token_cap=64)
    run = R.Runner(w, max_total_tokens=w.total_tokens, wait_timeout_ns=20_000_000)
    rng = np.random.default_rng(8)
    ids = attention_routing(rng, 12, w.num_experts, w.topk)
    rows, gl = grouped_rows(ids, run.host["x"][0], w.num_experts)
    rows_d = to_dev(rows, w.act)
    run.seq += 1
    assert A.afd_pack_grouped(run.ctx, 0, 0, 0, rows_d.data_ptr(), rows.shape[0], gl,
                              run.x[0].data_ptr(), 12, True, run.seq) == 0
    win = run.window(A.AFD_DIR_DISPATCH)
    off = G.slot_off(run, 0) + run.layout.header + 4 * 12
    cnt0 = win[off:off + 4].clone().view(torch.int32)
    win[off:off + 4] = (cnt0 + 1).view(torch.uint8)
    assert A.afd_ffn_forward_grouped(run.ctx, 0, 0, [rows.shape[0]], [12], [0]) == 0
    assert run.poll() == A.AFD_ERR_SHAPE
    ret = run.window(A.AFD_DIR_RETURN).cpu().numpy()
    assert ret[:8].view(np.uint64)[0] == 0


@pytest.mark.parametrize("gemm", [A.AFD_GEMM_TENSOR, A.AFD_GEMM_TENSOR_1CTA])
@pytest.mark.parametrize("with_shared", [True, False])
def test_grouped_single_peer_in_place(gemm, with_shared):
    """One peer: the GEMMs read its grouped rows in its dispatch slot and write
    the outputs into its return slot (no gather, no scatter)."""
    w = W.custom("fanin", seq_lens=[91], token_cap=384)
    compare(w, *run_grouped(w, seed=9, gemm=gemm, with_shared=with_shared))
