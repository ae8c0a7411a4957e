"""GPU path against the CPU oracle through the C ABI (needs an sm_103a GPU)."""
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


def test_tiny_fp32():
    run = R.Runner(W.get("tiny"), gemm=A.AFD_GEMM_SIMT, canary=True)
    e, _ = G.run_and_compare_full(run)
    print("tiny max|err|/rms", e)


@pytest.mark.parametrize("gemm", [A.AFD_GEMM_TENSOR, A.AFD_GEMM_TENSOR_1CTA, A.AFD_GEMM_SIMT],
                         ids=["tcgen05_pair", "tcgen05_1cta", "simt"])
def test_fanin_bf16(gemm):
    run = R.Runner(W.get("fanin"), gemm=gemm, canary=True)
    e, _ = G.run_and_compare_full(run)
    print("fanin max|err|/rms", e)


@pytest.mark.parametrize("gemm", [A.AFD_GEMM_TENSOR, A.AFD_GEMM_TENSOR_1CTA],
                         ids=["tcgen05_pair", "tcgen05_1cta"])
def test_weights_copied_at_registration(gemm):
    """The tensor engines read the library's tiled weight copies: the
    caller's expert weights overwritten with NaN once afd_set_layer has
    returned leave every result as the oracle gives it on the original
    weights; a second registration of the same layer (same sizes, copies
    reused) then takes the new values."""
    w = W.get("fanin")
    run = R.Runner(w, gemm=gemm, canary=True)
    snap = run.weights_numpy(0)
    for key in ("W13", "Wd", "W13s", "Wds"):
        if run.weights[0][key] is not None:
            run.weights[0][key].fill_(float("nan"))
    torch.cuda.synchronize()
    run.weights_numpy = lambda layer: snap
    e, _ = G.run_and_compare_full(run)
    print("weights overwritten after registration: max|err|/rms", e)
    # register the NaN weights: every output row becomes NaN
    wt = run.weights[0]
    assert A.afd_set_layer(run.ctx, 0, run.Wg.data_ptr(), run.bias.data_ptr() if run.bias is not None else 0,
                           wt["W13"].data_ptr(), wt["Wd"].data_ptr(),
                           wt["W13s"].data_ptr() if wt["W13s"] is not None else 0,
                           wt["Wds"].data_ptr() if wt["Wds"] is not None else 0) == 0
    run.pack_all(0)
    assert run.forward(0) == 0
    outs = run.unpack_all()
    assert run.poll() == 0
    assert all(torch.isnan(o[:n].float()).all() for o, n in zip(outs, w.seq_lens) if n)
    run.close()


@pytest.mark.parametrize("workload", ["fanin", "v2lite_prefill"])
def test_serialised_launches(workload):
    """Every kernel launched after the previous one has finished (no
    programmatic dependent launch): the same results."""
    w = W.get(workload)
    run = R.Runner(w, max_total_tokens=w.total_tokens, flags=A.AFD_CFG_NO_PDL, canary=True)
    if workload == "fanin":
        G.run_and_compare_full(run)
    else:
        # the full-size step is compared with the oracle row by row in
        # test_v2lite_prefill_full_size; here the return window of the
        # serialised launches must equal the default launches' byte for byte
        ref = R.Runner(w, max_total_tokens=w.total_tokens, canary=True)
        wins = []
        for r in (run, ref):
            r.pack_all(0)
            assert r.forward(0) == 0
            assert r.poll() == 0
            wins.append(r.window(A.AFD_DIR_RETURN).cpu().numpy())
        assert np.array_equal(wins[0], wins[1])
        ref.close()
    run.close()


@pytest.mark.parametrize("workload", ["fanin", "v2lite_prefill", "decode"])
def test_gemm_pair_equals_split_gemms(workload):
    """The SwiGLU and down GEMMs as one launch (down units waiting on their
    token tile's SwiGLU units) and as two launches: the same return window,
    byte for byte (decode: the first layer)."""
    w = W.get(workload)
    wins = []
    for flags in (0, A.AFD_CFG_SPLIT_GEMMS):
        run = R.Runner(w, max_total_tokens=w.total_tokens, flags=flags, layers=1)
        for _ in range(2):  # the counters start from zero again on the second step
            run.pack_all(0)
            assert run.forward(0) == 0
            assert run.poll() == 0
        wins.append(run.window(A.AFD_DIR_RETURN).cpu().numpy())
        run.close()
    assert np.array_equal(wins[0], wins[1])


def test_batched_pack_unpack_equal_per_peer_calls():
    """afd_pack_slots / afd_unpack_splits (all peers in one call, an empty
    peer among them) leave the same dispatch and return windows and the same
    unpacked rows as afd_pack_slot / afd_unpack_split per peer."""
    w = W.custom("fanin", seq_lens=[37, 0, 91, 5])
    got = []
    for batched in (True, False):
        run = R.Runner(w, max_total_tokens=w.total_tokens, layers=1)
        run.batched = batched
        run.pack_all(0)
        disp = run.window(A.AFD_DIR_DISPATCH).cpu().numpy()
        assert run.forward(0) == 0
        outs = [o[:n].cpu() for o, n in zip(run.unpack_all(), w.seq_lens)]
        assert run.poll() == 0
        got.append((disp, run.window(A.AFD_DIR_RETURN).cpu().numpy(), outs))
        run.close()
    assert np.array_equal(got[0][0], got[1][0])
    assert np.array_equal(got[0][1], got[1][1])
    assert all(torch.equal(a, b) for a, b in zip(got[0][2], got[1][2]))


def test_fanin_reordered_with_empty_peer():
    w = W.custom("fanin", seq_lens=[37, 0, 91, 5])
    run = R.Runner(w, canary=True)
    G.run_and_compare_full(run, slots=[2, 1, 3, 0])


def test_fanin_subset_of_peers_and_repeat():
    """Only some peers in the fan-in; then a second round on the same slots
    (the flags must advance) gives the same answer."""
    w = W.custom("fanin", seq_lens=[37, 91, 64])
    run = R.Runner(w, canary=True)
    G.run_and_compare_full(run, slots=[2, 0])
    e2, _ = G.run_and_compare_full(run, slots=[2, 0])


def test_single_peer_ragged_tiles():
    """One peer, token counts that leave ragged 16/32/256 tails per expert."""
    w = W.custom("fanin", seq_lens=[301], num_experts=8, topk=2)
    run = R.Runner(w, canary=True)
    G.run_and_compare_full(run)


def test_large_fanin_small_rows():
    """T * k = 9200 partials (ranked inside the gather) while the combine has
    few enough items to release the flags itself: the return headers must
    still be written (by the return-header kernel)."""
    w = W.custom("fanin", seq_lens=[1200, 1100])
    run = R.Runner(w, max_total_tokens=w.total_tokens, canary=True)
    e, _ = G.run_and_compare_full(run)
    print("fanin 2300 tokens max|err|/rms", e)
    run.close()


def test_v2lite_prefill_full_size():
    """Every output row of the 13312-token fan-in against the oracle (which
    runs the same fan-in on all host cores), with routing, plan, headers and
    route tables bit-exact."""
    w = W.get("v2lite_prefill")
    run = R.Runner(w, max_total_tokens=w.total_tokens, canary=True)
    e, _ = G.run_and_compare_full(run)
    print("v2lite max|err|/rms", e)
    run.close()


def test_skewed_full_size():
    w = W.get("skewed")
    run = R.Runner(w, max_total_tokens=w.total_tokens, canary=True)
    e, _ = G.run_and_compare_full(run)
    print("skewed max|err|/rms", e)
    counts = G.ws_array(run, A.AFD_WS_COUNTS, w.num_experts, np.int32)
    assert (counts == 0).any() and counts.max() > 5 * counts.mean()
    run.close()


def test_decode_26_layers():
    """All 26 layers, every output row of each, through one context."""
    w = W.get("decode")
    run = R.Runner(w, max_total_tokens=w.total_tokens, canary=True)
    worst = 0.0
    for layer in range(w.layers):
        e, _ = G.run_and_compare_full(run, layer=layer)
        worst = max(worst, e)
    print("decode 26 layers: worst max|err|/rms", worst)
    run.close()


@pytest.mark.parametrize("gemm", [A.AFD_GEMM_TENSOR, A.AFD_GEMM_SIMT])
def test_fanin_peer_without_shared_rows(gemm):
    """A peer that sends no shared rows (shared_tokens = 0) beside peers that
    do: its tokens get no shared-expert term, while the shared expert reads
    the other peers' rows in place from their slots."""
    w = W.custom("fanin", seq_lens=[37, 20, 91])
    run = R.Runner(w, max_total_tokens=w.total_tokens, gemm=gemm, canary=True)
    run.pack_all(peers=[0, 2])
    run.pack_all(peers=[1], with_shared=False)
    e, _ = G.run_and_compare_full(run, pack=False)
    print("max|err|/rms", e)
