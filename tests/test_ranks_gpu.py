"""Token-level dispatch to several FFN ranks on one GPU ([RFC]: Async GPU
Connector, "Data flow" and "Capacity and ring depth"): the Attention peers'
send (segments by destination rank, grouped by local expert, round-robin
shared rows), every rank's grouped step on its own experts, the peers'
combine -- against the CPU oracle.  Needs an sm_103a GPU."""
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


def layouts(rs):
    return [O.slot_layout_ranks(rs.w.num_peers, c.ring_depth, c.token_cap, c.topk, c.hidden,
                                rs.w.act_bytes, c.num_experts, c.shared_inter > 0,
                                O.routed_cap(c.token_cap, c.topk, rs.F, c.routed_cap_multiplier))
            for c in rs.cfgs]


def oracle_dispatch(rs, Ls, stage=0, layer=0, with_shared=True):
    """The oracle's send of every peer (same x bytes, the GPU gate's ids)."""
    w = rs.w
    wins = [np.zeros(L.window_bytes, np.uint8) for L in Ls]
    plans = []
    rcap = O.routed_cap(w.token_cap, w.topk, rs.F, rs.cfgs[0].routed_cap_multiplier)
    for p, n in enumerate(w.seq_lens):
        ids = rs.ids[p][:n].cpu().numpy()
        rc, dst, pos, rows = O.dispatch_ranks(wins, Ls, rs.cfgs[0].ring_depth, p, stage, layer,
                                              rs.host["x"][p], ids, w.num_experts, w.hidden,
                                              w.act_bytes, w.token_cap, rcap, with_shared,
                                              w.shared_inter > 0, rs.last_seq[(p, stage)])
        assert rc == 0, rc
        plans.append((dst, pos, rows))
    return wins, plans


def test_dispatch_bytes_match_oracle():
    """Every rank's dispatch window after the peers' sends, byte for byte:
    E = 10 over 4 ranks (not divisible), the shared rows round-robin."""
    w = W.custom("fanin", seq_lens=[37, 91], num_experts=10)
    rs = R.RankSet(w, 4)
    try:
        rs.route()
        rs.dispatch_all()
        assert rs.poll() == (0, 0)
        Ls = layouts(rs)
        wins, plans = oracle_dispatch(rs, Ls)
        for r in range(rs.F):
            got = rs.window(r, A.AFD_DIR_DISPATCH).cpu().numpy()
            assert got.size == wins[r].size
            for p in range(w.num_peers):
                assert A.afd_attn_rows(rs.attn[p], 0, rs.F)[r] == plans[p][2][r]
            assert np.array_equal(got, wins[r]), r
    finally:
        rs.close()


def run_round_trip(rs, with_shared=True):
    w = rs.w
    rs.route()
    rs.dispatch_all(with_shared=with_shared)
    rs.serve_all()
    rs.combine_all()
    assert rs.poll() == (0, 0)
    # the oracle: the same send, each rank's grouped step, each peer's combine
    Ls = layouts(rs)
    wins, plans = oracle_dispatch(rs, Ls, with_shared=with_shared)
    rets = [np.zeros_like(x) for x in wins]
    for r in range(rs.F):
        c = rs.cfgs[r]
        cfg = dict(num_regions=w.num_peers, ring_depth=c.ring_depth, token_cap=w.token_cap,
                   hidden=w.hidden, act_bytes=w.act_bytes, num_experts=c.num_experts, topk=w.topk,
                   inter=w.inter, shared_inter=w.shared_inter, renorm=w.renorm,
                   max_total_tokens=c.max_total_tokens, routed_scaling=w.routed_scaling,
                   ffn_rank=r, ffn_size=rs.F,
                   routed_cap=O.routed_cap(w.token_cap, w.topk, rs.F, c.routed_cap_multiplier))
        seen = np.zeros(w.num_peers * c.ring_depth, np.uint64)
        rc, y64, s64 = O.grouped_forward(cfg, wins[r], rets[r], rs.rank_weights_numpy(r), 0, 0,
                                         [int(pl[2][r]) for pl in plans], list(w.seq_lens),
                                         list(range(w.num_peers)), seen)
        assert rc == 0, rc
        # this rank's return window: headers and flags bit-exact, rows within tolerance
        got = rs.window(r, A.AFD_DIR_RETURN).cpu().numpy()
        L = Ls[r]
        assert np.array_equal(got[:L.flags_bytes], rets[r][:L.flags_bytes])
        for p in range(w.num_peers):
            off = L.flags_bytes + p * c.ring_depth * L.slot_bytes
            hb = 4 * (12 + c.num_experts)
            assert np.array_equal(got[off + L.header: off + L.header + hb],
                                  rets[r][off + L.header: off + L.header + hb]), (r, p)
        # the rows against the oracle's unrounded expert outputs (y64 in the
        # peers' order, s64 the peers' shared rows one after the other)
        errs = []
        for field, nrows, ref in (("routed_x", [int(pl[2][r]) for pl in plans], y64),
                                  ("shared_x", [O.rr_rows(n, r, rs.F) for n in w.seq_lens], s64)):
            base = 0
            for p in range(w.num_peers):
                n_p = nrows[p]
                off = L.flags_bytes + p * c.ring_depth * L.slot_bytes + getattr(L, field)
                nb = n_p * w.hidden * w.act_bytes
                if n_p and (field == "routed_x" or with_shared):
                    raw = got[off: off + nb]
                    a = (O.bf16_bits_to_f32(raw.view(np.uint16)) if w.act == "bf16"
                         else raw.view(np.float32)).reshape(n_p, -1)
                    errs.append(G.rel_err(a.astype(np.float64), ref[base: base + n_p]))
                base += n_p
        assert errs and max(errs) <= G.tol_for(w), (r, errs)
    worst = 0.0
    for p, n in enumerate(w.seq_lens):
        dst, pos, rows = plans[p]
        rc, out64, _ = O.attn_combine(rets, Ls, rs.cfgs[0].ring_depth, p, 0, n, w.topk, dst, pos,
                                      rs.wts[p][:n].cpu().numpy(), rows, with_shared, w.hidden,
                                      w.act_bytes, rs.last_seq[(p, 0)])
        assert rc == 0, rc
        gpu = rs.out[p][:n].float().cpu().numpy().astype(np.float64)
        e = G.rel_err(gpu, out64)
        worst = max(worst, e)
        assert e <= G.tol_for(w), (p, e)
    return worst


@pytest.mark.parametrize("E,F,seq_lens", [(16, 2, [37, 91]), (10, 4, [37, 91]), (16, 3, [91])])
def test_round_trip_matches_oracle(E, F, seq_lens):
    """Gate, send, each rank's grouped step, combine: the peers' outputs and
    every rank's return slots against the oracle's round trip on the same
    ids and weights (one peer: the ranks take the in-place path)."""
    w = W.custom("fanin", seq_lens=seq_lens, num_experts=E)
    rs = R.RankSet(w, F)
    try:
        print("max|err|/rms", run_round_trip(rs))
    finally:
        rs.close()


@pytest.mark.parametrize("gemm", [A.AFD_GEMM_TENSOR_1CTA, A.AFD_GEMM_SIMT])
def test_round_trip_other_engines_routed_only(gemm):
    """The routed-only protocol (no shared rows travel) on the other engines."""
    w = W.custom("fanin", seq_lens=[37, 91], num_experts=12)
    rs = R.RankSet(w, 3, gemm=gemm)
    try:
        run_round_trip(rs, with_shared=False)
    finally:
        rs.close()


def test_round_trip_fp32_simt():
    """fp32 activations (the tiny configuration: renormalised top-2 of 8,
    no shared expert) over 2 ranks on the SIMT engine."""
    w = W.get("tiny")
    rs = R.RankSet(w, 2, gemm=A.AFD_GEMM_SIMT)
    try:
        run_round_trip(rs, with_shared=False)
    finally:
        rs.close()


def test_segment_over_routed_cap_raises():
    """Every partial on rank 0 with the multiplier at 1.0: the send raises
    AFD_ERR_CAPACITY and no rank's flag is written."""
    w = W.custom("fanin", seq_lens=[37, 91])
    rs = R.RankSet(w, 2, multiplier=1.0)
    try:
        for p, n in enumerate(w.seq_lens):
            rs.ids[p][:n] = torch.arange(w.topk, dtype=torch.int32, device="cuda")
        rs.seq += 1
        assert A.afd_attn_dispatch(rs.attn[1], 0, 0, rs.x[1].data_ptr(), 91, rs.ids[1].data_ptr(),
                                   True, rs.seq) == 0
        assert A.afd_attn_poll_status(rs.attn[1]) == A.AFD_ERR_CAPACITY
        for r in range(rs.F):
            L = A.afd_slot_layout(rs.cfgs[r])
            assert not rs.window(r, A.AFD_DIR_DISPATCH)[:L.flags_bytes].any().item()
    finally:
        rs.close()


def test_empty_destination_creates_no_wait():
    """Ranks that get neither routed nor shared rows from a peer receive an
    empty message (header with no rows, flag written) and are not waited
    for: with those ranks never run, the combine still completes."""
    w = W.custom("fanin", seq_lens=[2], num_experts=16)
    rs = R.RankSet(w, 4, wait_timeout_ns=50_000_000)
    try:
        # both tokens choose experts of rank 0 (experts 0..3), so ranks 2 and
        # 3 get nothing (and no shared token: only tokens 0 and 1 exist)
        rs.ids[0][:2] = torch.tensor([[0, 1, 2, 3], [3, 2, 1, 0]], dtype=torch.int32, device="cuda")
        rs.wts[0][:2] = torch.rand((2, 4), device="cuda")
        rs.dispatch_all()
        assert A.afd_attn_rows(rs.attn[0], 0, 4) == [8, 0, 0, 0]
        rs.serve_all(ranks=[0, 1])       # rank 1 has shared token 1
        rs.combine_all()
        assert rs.poll() == (0, 0)
        for r in (2, 3):
            L = A.afd_slot_layout(rs.cfgs[r])
            win = rs.window(r, A.AFD_DIR_DISPATCH).cpu().numpy()
            h = win[L.flags_bytes + L.header: L.flags_bytes + L.header + 4 * 16].view(np.int32)
            assert h[7] == 2 and h[8] == 0 and h[9] == 0
            assert win[:8].view(np.uint64)[0] == rs.last_seq[(0, 0)]
        # the output: the rank-0 expert rows and rank 0 / 1's shared rows
        Ls = layouts(rs)
        wins, plans = oracle_dispatch(rs, Ls)
        assert list(plans[0][2]) == [8, 0, 0, 0]
    finally:
        rs.close()
