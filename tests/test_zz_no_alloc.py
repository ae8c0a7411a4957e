"""The allocation-free router entry point (afd_route_noalloc), for callers
that cannot call cudaMalloc (a serving process whose memory pool already
holds the device's free memory, or a plugin that must not trigger the
device-wide synchronisation an allocation can bring).

Its output must match the CPU oracle's router -- ids bit for bit, gate
weights within the 1e-6 relative tolerance the parity tests use -- on two
calls in a row that reuse its shared scratch array, and on the named fan-in
and skewed workloads also the router step of afd_ffn_forward.  The cases
reach every logits kernel the entry point can launch (bf16 with 16 or more
experts, bf16 with fewer, fp32, hidden above 2048) and both capacity limits
exactly.  Collected last on purpose."""
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


def case(name):
    """(workload, whether afd_ffn_forward's router is compared too)."""
    if name == "fanin":
        return W.get("fanin"), True
    if name == "skewed":
        return W.get("skewed"), True
    if name == "tiny_f32":            # fp32 activations, 8 experts top-2 renormalised
        return W.get("tiny"), False
    if name == "bf16_E8":             # bf16 with fewer than 16 experts
        return W.custom("fanin", num_experts=8, topk=2, seq_lens=[37, 91]), False
    if name == "logits_at_limit":     # n_tokens * E == AFD_NOALLOC_MAX_LOGITS
        n = A.AFD_NOALLOC_MAX_LOGITS // 64
        return W.custom("v2lite_prefill", seq_lens=[n // 2, n - n // 2]), False
    if name == "weights_at_limit":    # 4 * ceil(E / 4) * hidden == AFD_NOALLOC_MAX_ROUTER_WEIGHTS
        h = A.AFD_NOALLOC_MAX_ROUTER_WEIGHTS // 64
        return W.custom("v2lite_prefill", hidden=h, seq_lens=[33]), False
    raise KeyError(name)


def forward_router_outputs(w):
    """ids and gate weights from the existing entry point (afd_ffn_forward)."""
    run = R.Runner(w, layers=1)
    run.pack_all(0)
    assert run.forward(0) == 0 and run.poll() == 0
    T, k = w.total_tokens, w.topk
    ids = G.ws_array(run, A.AFD_WS_IDS, T * k, np.int32).reshape(T, k).copy()
    wts = G.ws_array(run, A.AFD_WS_WEIGHTS, T * k, np.float32).reshape(T, k).copy()
    run.close()
    return ids, wts


@pytest.mark.parametrize("name", ["fanin", "skewed", "tiny_f32", "bf16_E8", "logits_at_limit",
                                  "weights_at_limit"])
def test_noalloc_router_matches_oracle_twice(name):
    w, with_forward = case(name)
    host = W.host_inputs(w)
    X = np.concatenate([a for a, n in zip(host["x"], w.seq_lens) if n])
    T, k = w.total_tokens, w.topk
    assert X.shape == (T, w.hidden)
    if name == "logits_at_limit":
        assert T * w.num_experts == A.AFD_NOALLOC_MAX_LOGITS
    if name == "weights_at_limit":
        assert 4 * -(-w.num_experts // 4) * w.hidden == A.AFD_NOALLOC_MAX_ROUTER_WEIGHTS
    ids_ref, w_ref, _ = O.route(X, w.act_bytes, host["Wg"], host["bias"], k, w.renorm,
                                w.routed_scaling)
    x = R.act_tensor(X, w.act, "cuda")
    Wg = torch.from_numpy(host["Wg"]).cuda()
    bias = None if host["bias"] is None else torch.from_numpy(host["bias"]).cuda()
    stream = torch.cuda.current_stream()
    act = A.AFD_DTYPE_BF16 if w.act == "bf16" else A.AFD_DTYPE_F32
    for _ in range(2):
        ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        rc = A.afd_route_noalloc(x.data_ptr(), T, w.hidden, act, Wg.data_ptr(),
                                 bias.data_ptr() if bias is not None else 0, w.num_experts, k,
                                 w.renorm, w.routed_scaling, ids.data_ptr(), wts.data_ptr(),
                                 stream.cuda_stream)
        assert rc == A.AFD_OK, A.strerror(rc)
        torch.cuda.synchronize()
        got_ids, got_w = ids.cpu().numpy(), wts.cpu().numpy()
        assert np.array_equal(got_ids, ids_ref), f"{int((got_ids != ids_ref).sum())} ids differ"
        assert np.allclose(got_w, w_ref, rtol=1e-6, atol=0), np.abs(got_w / w_ref - 1).max()
    if with_forward:
        f_ids, f_w = forward_router_outputs(w)
        assert np.array_equal(got_ids, f_ids)
        assert np.allclose(got_w, f_w, rtol=1e-6, atol=0)


def test_noalloc_router_rejects_oversize():
    too_wide = A.AFD_NOALLOC_MAX_ROUTER_WEIGHTS // 64 + 8
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    rc = A.afd_route_noalloc(dummy.data_ptr(), 4, too_wide, A.AFD_DTYPE_BF16, dummy.data_ptr(),
                             0, 64, 6, 0, 1.0, dummy.data_ptr(), dummy.data_ptr(), 0)
    assert rc == A.AFD_ERR_CAPACITY
    too_many = A.AFD_NOALLOC_MAX_LOGITS // 64 + 1
    rc = A.afd_route_noalloc(dummy.data_ptr(), too_many, 2048, A.AFD_DTYPE_BF16, dummy.data_ptr(),
                             0, 64, 6, 0, 1.0, dummy.data_ptr(), dummy.data_ptr(), 0)
    assert rc == A.AFD_ERR_CAPACITY
