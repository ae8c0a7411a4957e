"""Failure detection on the GPU, injected on the host: corrupted headers, a
flag nothing sets (bounded wait must give up), shutdown, wrong layer or
shape, host pointers.  Every device wait here is bounded by a short
wait_timeout_ns; nothing faults, traps or hangs the GPU.  The error code is
compared with the oracle's on the same slot bytes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from combine_peer_slot_gb300 import afd as A
from combine_peer_slot_gb300 import runtime as R
from combine_peer_slot_gb300 import workloads as W
from oracle import oracle as O
from tests import gpu_parity as G

SHORT_WAIT_NS = 20_000_000  # 20 ms


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    A.lib()


def make_run(layers=2):
    w = W.custom("fanin", seq_lens=[5, 9], num_experts=8, topk=2, hidden=256, inter=64,
                 shared_inter=64)
    return R.Runner(w, layers=layers, wait_timeout_ns=SHORT_WAIT_NS)


def oracle_code(run, layer=0, lens=None, slots=(0, 1), seen=None):
    win = run.window(A.AFD_DIR_DISPATCH).cpu().numpy().copy()
    ret = np.zeros_like(win)
    seen = np.zeros(run.w.num_peers, np.uint64) if seen is None else seen
    lens = list(run.w.seq_lens) if lens is None else lens
    rc, _ = O.ffn_forward(G.oracle_cfg(run), win, ret, run.weights_numpy(min(layer, run.layers - 1)),
                          layer, 0, lens, list(slots), seen)
    return rc


def poke_header(run, peer, word, value):
    win = run.window(A.AFD_DIR_DISPATCH)
    off = G.slot_off(run, peer) + run.layout.header + 4 * word
    win[off:off + 4] = torch.tensor([value], dtype=torch.int32).view(torch.uint8).cuda()
    torch.cuda.synchronize()


@pytest.mark.parametrize("word,value,code", [
    (0, 0x1234, A.AFD_ERR_HEADER), (1, 7, A.AFD_ERR_HEADER), (11, 3, A.AFD_ERR_HEADER),
    (3, 999, A.AFD_ERR_SEQ), (4, 999, A.AFD_ERR_SEQ), (2, 2, A.AFD_ERR_SHUTDOWN),
    (5, 1, A.AFD_ERR_LAYER), (6, 1, A.AFD_ERR_STAGE), (7, 4, A.AFD_ERR_SHAPE),
    (9, 3, A.AFD_ERR_SHAPE)])
def test_corrupted_header(word, value, code):
    run = make_run()
    run.pack_all(0)
    poke_header(run, 1, word, value)
    assert oracle_code(run) == code
    assert run.forward(0) == A.AFD_OK          # launched; the device records the error
    assert run.poll() == code
    # nothing was consumed: repack and the context works again
    run.pack_all(0)
    assert run.forward(0) == A.AFD_OK and run.poll() == A.AFD_OK


def test_flag_never_set_times_out():
    run = make_run()
    run.pack_all(0)
    assert run.forward(0) == 0 and run.poll() == 0
    seen = np.array([run.last_seq[(0, 0)], run.last_seq[(1, 0)]], np.uint64)
    assert oracle_code(run, seen=seen) == O.ERR_TIMEOUT
    import time
    t0 = time.time()
    assert run.forward(0) == 0                 # same slots again: flags never advance
    assert run.poll() == A.AFD_ERR_TIMEOUT
    assert time.time() - t0 < 5.0
    run.pack_all(0)
    assert run.forward(0) == 0 and run.poll() == 0


def test_forward_queued_behind_a_failed_one():
    """A forward enqueued behind one that failed finds the sticky status: its
    header check skips and hands the router the abort token, so nothing
    waits out a timeout; the first error is the one reported, and the
    context works again afterwards."""
    import time
    w = W.custom("fanin", seq_lens=[5, 9], token_cap=64)
    run = R.Runner(w, layers=2, wait_timeout_ns=2_000_000_000)  # a router left waiting: > 2 s
    run.pack_all(0)
    assert run.forward(0) == 0 and run.poll() == 0   # warm (module loads, first launches)
    run.pack_all(0)
    assert run.forward(1) == 0                 # wrong layer: recorded on the device
    run.pack_all(0)
    t0 = time.time()
    assert run.forward(0) == 0                 # queued behind it
    assert run.poll() == A.AFD_ERR_LAYER
    assert time.time() - t0 < 1.0
    run.pack_all(0)
    assert run.forward(0) == 0 and run.poll() == 0


def test_shutdown_announced():
    run = make_run()
    run.pack_all(0, peers=[0])
    run.seq += 1
    assert A.afd_announce_shutdown(run.ctx, 1, 0, run.seq) == 0
    assert run.forward(0, slots=[0, 1]) == 0
    assert run.poll() == A.AFD_ERR_SHUTDOWN


def test_layer_and_shape_mismatch():
    run = make_run()
    run.pack_all(0)
    assert run.forward(1) == 0 and run.poll() == A.AFD_ERR_LAYER
    run.pack_all(0)
    assert oracle_code(run, lens=[5, 8]) == O.ERR_SHAPE
    assert A.afd_ffn_forward(run.ctx, 0, 0, [5, 8], [0, 1]) == 0
    assert run.poll() == A.AFD_ERR_SHAPE


def test_host_side_errors():
    run = make_run()
    cap = run.w.token_cap
    assert A.afd_ffn_forward(run.ctx, 0, 0, [5, cap + 1], [0, 1]) == A.AFD_ERR_CAPACITY
    assert A.afd_ffn_forward(run.ctx, 0, 0, [5, 9], [0, 0]) == A.AFD_ERR_ARG
    assert A.afd_ffn_forward(run.ctx, 0, 1, [5, 9], [0, 1]) == A.AFD_ERR_ARG
    assert A.afd_ffn_forward(run.ctx, 5, 0, [5, 9], [0, 1]) == A.AFD_ERR_LAYER
    host = torch.zeros((5, run.w.hidden), dtype=torch.bfloat16)
    assert A.afd_pack_slot(run.ctx, 0, 0, 0, host.data_ptr(), 5, 1, 10**6) == A.AFD_ERR_NOT_DEVICE
    assert A.afd_pack_slot(run.ctx, 0, 0, 0, run.x[0].data_ptr(), cap + 1, 1, 10**6) == A.AFD_ERR_CAPACITY
    run.pack_all(0)
    assert A.afd_pack_slot(run.ctx, 0, 0, 0, run.x[0].data_ptr(), 5, 1, 1) == A.AFD_ERR_SEQ
    hout = torch.zeros((5, run.w.hidden), dtype=torch.bfloat16)
    assert A.afd_unpack_split(run.ctx, 0, 0, hout.data_ptr(), 5, 1) == A.AFD_ERR_NOT_DEVICE
    assert run.poll() == 0


def test_batched_pack_unpack_host_side_errors():
    """afd_pack_slots / afd_unpack_splits check every entry before launching
    anything: a refused call leaves the slots and the seqs as they were."""
    run = make_run()
    cap, H = run.w.token_cap, run.w.hidden
    x0, x1 = run.x[0].data_ptr(), run.x[1].data_ptr()
    host = torch.zeros((5, H), dtype=torch.bfloat16)
    assert A.afd_pack_slots(run.ctx, [0, 0], 0, 0, [x0, x0], [5, 5], 1, [10, 11]) == A.AFD_ERR_ARG
    assert A.afd_pack_slots(run.ctx, [0, 1], 0, 0, [x0, host.data_ptr()], [5, 5], 1, [10, 11]) == \
        A.AFD_ERR_NOT_DEVICE
    assert A.afd_pack_slots(run.ctx, [0, 1], 0, 0, [x0, x1], [5, cap + 1], 1, [10, 11]) == A.AFD_ERR_CAPACITY
    assert A.afd_pack_slots(run.ctx, [0, 1], 1, 0, [x0, x1], [5, 5], 1, [10, 11]) == A.AFD_ERR_ARG
    run.pack_all(0)
    s0 = run.last_seq[(0, 0)]
    assert A.afd_pack_slots(run.ctx, [1, 0], 0, 0, [x1, x0], [5, 5], 1, [10**6, s0]) == A.AFD_ERR_SEQ
    out = torch.empty((5, H), dtype=torch.bfloat16, device="cuda")
    assert A.afd_unpack_splits(run.ctx, [0], 0, [host.data_ptr()], [5], [s0]) == A.AFD_ERR_NOT_DEVICE
    assert A.afd_unpack_splits(run.ctx, [0], 0, [out.data_ptr()], [cap + 1], [s0]) == A.AFD_ERR_CAPACITY
    # the refused packs left the slots alone: the step packed above still runs
    assert run.forward(0) == 0
    run.unpack_all()
    assert run.poll() == 0


def test_unpack_wrong_seq():
    run = make_run()
    run.pack_all(0)
    assert run.forward(0) == 0
    out = torch.empty((5, run.w.hidden), dtype=torch.bfloat16, device="cuda")
    s = run.last_seq[(0, 0)]
    assert A.afd_unpack_split(run.ctx, 0, 0, out.data_ptr(), 5, s + 1) == 0
    assert run.poll() == A.AFD_ERR_TIMEOUT
    assert A.afd_unpack_split(run.ctx, 0, 0, out.data_ptr(), 5, s - 1) == 0
    assert run.poll() == A.AFD_ERR_SEQ
    assert A.afd_unpack_split(run.ctx, 0, 0, out.data_ptr(), 4, s) == 0
    assert run.poll() == A.AFD_ERR_SHAPE
    assert A.afd_unpack_split(run.ctx, 0, 0, out.data_ptr(), 5, s) == 0
    assert run.poll() == 0
