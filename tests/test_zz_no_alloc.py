"""The allocation-free router entry point (afd_route_noalloc), for callers
that cannot call cudaMalloc (a serving process whose memory pool already
holds the device's free memory, or a plugin that must not trigger the
device-wide synchronisation an allocation can bring).  Its output must
match the router step of afd_ffn_forward -- ids bit for bit, gate weights
within the 1e-6 relative tolerance the parity tests use -- on two calls in
a row that reuse its shared scratch array.  Collected last on purpose."""
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


def forward_router_outputs(w):
    """ids and gate weights from the existing entry point (afd_ffn_forward)."""
    run = R.Runner(w, layers=1)
    run.pack_all(0)
    assert run.forward(0) == 0 and run.poll() == 0
    T, k = w.total_tokens, w.topk
    ids = G.ws_array(run, A.AFD_WS_IDS, T * k, np.int32).reshape(T, k).copy()
    wts = G.ws_array(run, A.AFD_WS_WEIGHTS, T * k, np.float32).reshape(T, k).copy()
    x = torch.cat([t for t, n in zip(run.x, w.seq_lens) if n]).contiguous()
    return run, x, ids, wts


@pytest.mark.parametrize("name", ["fanin", "skewed"])
def test_noalloc_router_matches_forward_twice(name):
    w = W.get(name)
    run, x, ids_ref, w_ref = forward_router_outputs(w)
    T, k = w.total_tokens, w.topk
    stream = torch.cuda.current_stream()
    act = A.AFD_DTYPE_BF16 if w.act == "bf16" else A.AFD_DTYPE_F32
    bias = run.bias.data_ptr() if run.bias is not None else 0
    for _ in range(2):
        ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        rc = A.afd_route_noalloc(x.data_ptr(), T, w.hidden, act, run.Wg.data_ptr(), bias,
                                 w.num_experts, k, w.renorm, w.routed_scaling, ids.data_ptr(),
                                 wts.data_ptr(), stream.cuda_stream)
        assert rc == A.AFD_OK
        torch.cuda.synchronize()
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        assert np.allclose(wts.cpu().numpy(), w_ref, rtol=1e-6, atol=0)
    run.close()


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
