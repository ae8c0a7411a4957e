"""Edge cases of the FFN step against the CPU oracle: an empty fan-in, the
largest expert count and top-k the kernels cover, the most peers, top-k
equal to the expert count, hidden sizes that take the router's other
kernels.  Needs an sm_103a GPU."""
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


def test_all_peers_empty():
    """Every listed peer sends no tokens: no expert work, and each return
    slot still gets its header (num_tokens 0, no counts) and its flag."""
    w = W.custom("fanin", seq_lens=[0, 0, 0], token_cap=64)
    run = R.Runner(w, max_total_tokens=64, canary=True)
    run.pack_all(0)
    assert run.forward(0) == 0
    assert run.poll() == 0
    ret = run.window(A.AFD_DIR_RETURN).cpu().numpy()
    for p in range(3):
        h = G.header(ret, run, p)
        assert h[0] == 0x47444641 and h[7] == 0 and h[8] == 0 and not h[12:].any()
        assert ret[:run.layout.flags_bytes].view(np.uint64)[p] == run.last_seq[(p, 0)]


@pytest.mark.parametrize("shape", [
    dict(num_experts=256, topk=16, hidden=512, inter=64, shared_inter=64, seq_lens=[40, 7]),
    dict(num_experts=8, topk=8, hidden=256, inter=96, shared_inter=96, seq_lens=[19, 1, 33]),
    # without a shared expert a token's weighted sum of its k expert outputs
    # can cancel to far less than each of them; the expert outputs reach
    # the combine as 24-bit floats (16 significant bits, 2^-16 relative
    # rounding), far finer than the output's bf16 rounding
    dict(num_experts=8, topk=8, hidden=256, inter=96, shared_inter=0, seq_lens=[19, 1, 33]),
    dict(num_experts=16, topk=2, hidden=4096, inter=128, shared_inter=64, seq_lens=[33, 20]),
    dict(num_experts=64, topk=6, hidden=3072, inter=64, shared_inter=64, seq_lens=[25]),
    dict(num_experts=64, topk=6, hidden=3072, inter=64, shared_inter=0, seq_lens=[25]),
    # ~128 rows per expert take the 256-row tiles; hidden 320 and inter 176
    # give odd k-block counts (5 and 3, the last one partial), so the pair
    # GEMM's last stage carries a single k-block
    dict(num_experts=8, topk=2, hidden=320, inter=176, shared_inter=80, seq_lens=[300, 212]),
], ids=["E256_k16", "k_equals_E", "k_equals_E_no_shared", "hidden4096", "hidden3072",
        "hidden3072_no_shared", "wide_odd_k"])
def test_shapes_at_the_edges(shape):
    """Routing, plan and outputs against the oracle at the shapes' edges:
    256 experts with top-16 (the largest the router covers), top-k equal to
    the expert count, hidden above 2048 (the router's fallback kernels),
    wide token tiles over odd and partial k-block counts, layers with and
    without a shared expert."""
    w = W.custom("fanin", **shape)
    run = R.Runner(w, max_total_tokens=w.total_tokens, canary=True)
    e, _ = G.run_and_compare_full(run)
    print(shape, "max|err|/rms", e)
    run.close()


def test_sixty_four_peers():
    """The most peers a window holds, with ragged and empty slots, listed in
    a shuffled order."""
    rng = np.random.default_rng(64)
    lens = [int(v) for v in rng.integers(0, 9, size=A.AFD_MAX_PEERS)]
    w = W.custom("fanin", seq_lens=lens, token_cap=16)
    run = R.Runner(w, max_total_tokens=w.total_tokens, canary=True)
    slots = [int(v) for v in rng.permutation(A.AFD_MAX_PEERS)]
    e, _ = G.run_and_compare_full(run, slots=slots)
    print("64 peers, T =", sum(lens), "max|err|/rms", e)
    run.close()
