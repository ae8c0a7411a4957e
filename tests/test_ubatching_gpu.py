"""Two-stage micro-batching ([RFC]: Async AFD for Prefill on Ascend NPU, the
async_moe_ubatching mode; [RFC]: Async GPU Connector, "Capacity and ring
depth": ring_depth = the number of stages): each peer's batch is split into
two token-balanced stages whose slots are in flight together; the FFN side
serves stage 0 and stage 1 as separate work items and the peers rejoin the
outputs.  Needs an sm_103a GPU."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from combine_peer_slot_gb300 import afd as A
from combine_peer_slot_gb300 import runtime as R
from combine_peer_slot_gb300 import workloads as W
from tests import gpu_parity as G


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    A.lib()


def split_stages(w):
    """Token-balanced split of every peer's batch: stage 0 = the first half."""
    return {p: (n // 2, n - n // 2) for p, n in enumerate(w.seq_lens)}


def full_batch_outputs(w):
    run = R.Runner(w, max_total_tokens=w.total_tokens)
    G.run_and_compare_full(run)   # the single-stage step, checked against the oracle
    outs = [o[:n].clone() for o, n in zip(run.out, w.seq_lens)]
    run.close()
    return outs


def test_two_stages_token_form():
    w = W.custom("fanin", seq_lens=[37, 91])
    ref = full_batch_outputs(w)
    run = R.Runner(w, max_total_tokens=w.total_tokens, ring_depth=2)
    halves = split_stages(w)
    ws = w.shared_inter > 0
    seqs = {}
    # both stages packed before either is served: their slots are in flight together
    for stage in (0, 1):
        for p, (h0, h1) in halves.items():
            n = h0 if stage == 0 else h1
            x = run.x[p][:h0] if stage == 0 else run.x[p][h0:]
            run.seq += 1
            assert A.afd_pack_slot(run.ctx, p, stage, 0, x.data_ptr() if n else 0, n, ws,
                                   run.seq) == 0
            seqs[(p, stage)] = run.seq
    for stage in (0, 1):
        lens = [halves[p][stage] for p in range(w.num_peers)]
        assert A.afd_ffn_forward(run.ctx, 0, stage, lens, list(range(w.num_peers))) == 0
    outs = []
    for p, (h0, h1) in halves.items():
        o = torch.empty_like(ref[p])
        for stage, (a, b) in ((0, (0, h0)), (1, (h0, h0 + h1))):
            if b > a:
                assert A.afd_unpack_split(run.ctx, p, stage, o[a:b].data_ptr(), b - a,
                                          seqs[(p, stage)]) == 0
        outs.append(o)
    assert run.poll() == 0
    # the rejoined outputs are the single-batch outputs, bit for bit (every
    # token's routing, expert sums and combine are independent of the batch)
    for p in range(w.num_peers):
        assert torch.equal(outs[p], ref[p]), p


def test_two_stages_grouped_form():
    """The same with the grouped form (micro-batching requires the gate on the
    Attention side): stage-wise grouped rows, outputs rejoined per peer."""
    w = W.custom("fanin", seq_lens=[37, 91], token_cap=384)
    rng = np.random.default_rng(12)
    halves = split_stages(w)
    ids = {p: np.argsort(rng.random((n, w.num_experts)), axis=1)[:, :w.topk].astype(np.int32)
           for p, n in enumerate(w.seq_lens)}

    def serve(run, stages):
        """stages: list of (stage, {peer: (token range)}) -> per peer list of
        (token range, expert outputs per (token, j) in t*k + j order)."""
        ws = w.shared_inter > 0
        keep, meta = [], []
        for stage, ranges in stages:
            for p, (a, b) in ranges.items():
                sub = ids[p][a:b]
                order = np.argsort(sub.reshape(-1), kind="stable")
                rows = np.ascontiguousarray(run.host["x"][p][a:b][order // w.topk])
                gl = np.bincount(sub.reshape(-1), minlength=w.num_experts)
                rows_d = R.act_tensor(rows, w.act, "cuda") if rows.shape[0] else None
                keep.append(rows_d)
                run.seq += 1
                x = run.x[p][a:b]
                assert A.afd_pack_grouped(run.ctx, p, stage, 0,
                                          rows_d.data_ptr() if rows_d is not None else 0,
                                          rows.shape[0], gl, x.data_ptr() if b > a else 0, b - a,
                                          ws, run.seq) == 0
                meta.append((stage, p, a, b, order, rows.shape[0], run.seq))
        for stage, ranges in stages:
            ps = sorted(ranges)
            assert A.afd_ffn_forward_grouped(run.ctx, 0, stage,
                                             [(ranges[p][1] - ranges[p][0]) * w.topk for p in ps],
                                             [ranges[p][1] - ranges[p][0] for p in ps], ps) == 0
        res = {}
        for stage, p, a, b, order, nr, seq in meta:
            y = torch.empty((max(nr, 1), w.hidden), dtype=torch.bfloat16, device="cuda")
            s = torch.empty((max(b - a, 1), w.hidden), dtype=torch.bfloat16, device="cuda")
            assert A.afd_unpack_grouped(run.ctx, p, stage, y.data_ptr() if nr else 0, nr,
                                        s.data_ptr() if b > a else 0, b - a, seq) == 0
            # back to (token, j) order
            yy = torch.empty_like(y[:nr])
            yy[torch.from_numpy(order).cuda()] = y[:nr]
            res.setdefault(p, []).append((a, b, yy, s[:b - a]))
        assert run.poll() == 0
        return res

    one = R.Runner(w, max_total_tokens=w.total_tokens)
    ref = serve(one, [(0, {p: (0, n) for p, n in enumerate(w.seq_lens)})])
    two = R.Runner(w, max_total_tokens=w.total_tokens, ring_depth=2)
    got = serve(two, [(0, {p: (0, h0) for p, (h0, h1) in halves.items()}),
                      (1, {p: (h0, h0 + h1) for p, (h0, h1) in halves.items()})])
    for p in range(w.num_peers):
        (_, _, y_ref, s_ref), = ref[p]
        y_two = torch.cat([y for _, _, y, _ in sorted(got[p], key=lambda v: v[0])])
        s_two = torch.cat([s for _, _, _, s in sorted(got[p], key=lambda v: v[0])])
        assert torch.equal(y_two, y_ref) and torch.equal(s_two, s_ref), p
