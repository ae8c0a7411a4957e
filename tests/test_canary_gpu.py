"""Guard words after every slot field (AFD_CFG_CANARY), the memory checker's
stand-in: a forward leaves them intact, and a byte changed in any guard is
found, with its window and offset.  Needs an sm_103a GPU."""
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


def guard_offsets(run, peer):
    """A byte inside each guard of slot (peer, 0), and one in the flag array's."""
    L = run.layout
    base = G.slot_off(run, peer)
    ends = [L.route_table, L.routed_x, L.shared_idx, L.shared_x, L.slot_bytes]
    offs = [base + e - L.guard + 4 * i + 1 for i, e in enumerate(ends)]
    return [L.flags_bytes - L.guard + 5] + offs


def test_forward_leaves_guards_intact_and_a_changed_byte_is_found():
    w = W.get("fanin")
    run = R.Runner(w, canary=True)
    assert run.layout.guard == run.layout.align
    G.run_and_compare_full(run)  # checks the guards after the forward
    for direction in (A.AFD_DIR_DISPATCH, A.AFD_DIR_RETURN):
        win = run.window(direction)
        for off in guard_offsets(run, 1):
            old = int(win[off].item())
            win[off] = old ^ 0x5A
            torch.cuda.synchronize()
            rc, found_dir, found_off = A.afd_check_canaries(run.ctx)
            assert rc == A.AFD_ERR_CANARY
            assert (found_dir, found_off) == (direction, off & ~3)
            win[off] = old
            torch.cuda.synchronize()
            assert A.afd_check_canaries(run.ctx)[0] == A.AFD_OK
    run.close()


def test_no_guards_nothing_to_check():
    run = R.Runner(W.get("fanin"))
    assert run.layout.guard == 0
    assert A.afd_check_canaries(run.ctx)[0] == A.AFD_ERR_ARG
    run.close()
