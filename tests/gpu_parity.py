"""Helpers shared by the GPU parity tests: run a workload through the C ABI
and compare it with the CPU oracle on the same slot bytes."""
import numpy as np

from combine_peer_slot_gb300 import afd as A
from combine_peer_slot_gb300 import runtime as R
from oracle import oracle as O

BF16_TOL = 2e-2   # max |err| <= 2e-2 * rms(oracle), bf16 activations
F32_TOL = 1e-4    # max |err| <= 1e-4 * rms(oracle), fp32 activations


def oracle_cfg(run):
    """The oracle's configuration for a runner's context."""
    w = run.w
    return dict(num_regions=w.num_peers, ring_depth=run.cfg.ring_depth, token_cap=w.token_cap,
                hidden=w.hidden, act_bytes=w.act_bytes, num_experts=w.num_experts, topk=w.topk,
                inter=w.inter, shared_inter=w.shared_inter, renorm=w.renorm,
                max_total_tokens=run.cfg.max_total_tokens, routed_scaling=w.routed_scaling)


def tol_for(w):
    return BF16_TOL if w.act == "bf16" else F32_TOL


def ws_array(run, which, count, dtype):
    nbytes = count * np.dtype(dtype).itemsize
    if nbytes == 0:
        return np.zeros(0, dtype)
    return run.workspace(which, nbytes).cpu().numpy().view(dtype)


def slot_off(run, peer, stage=0, L=None):
    """Byte offset of slot (peer, stage) in layout L (the run's by default)."""
    L = run.layout if L is None else L
    return L.flags_bytes + (peer * run.cfg.ring_depth + stage) * L.slot_bytes


def return_rows(ret, run, peer, n, L=None):
    L = run.layout if L is None else L
    w = run.w
    off = slot_off(run, peer, L=L) + L.routed_x
    rb = w.hidden * w.act_bytes
    raw = ret[off: off + n * rb]
    if w.act == "bf16":
        return O.bf16_bits_to_f32(raw.view(np.uint16)).astype(np.float64).reshape(n, w.hidden)
    return raw.view(np.float32).astype(np.float64).reshape(n, w.hidden)


def route_table(ret, run, peer, n, L=None):
    L = run.layout if L is None else L
    off = slot_off(run, peer, L=L) + L.route_table
    return ret[off: off + n * run.w.topk * 4].view(np.int32).reshape(n, run.w.topk)


def header(buf, run, peer, L=None):
    L = run.layout if L is None else L
    off = slot_off(run, peer, L=L) + L.header
    return buf[off: off + 4 * (12 + run.w.num_experts)].view(np.int32)


def plain_layout(run):
    """The run's slot layout without guard words (the oracle's)."""
    cfg = A.afd_config.from_buffer_copy(run.cfg)
    cfg.flags = cfg.flags & ~A.AFD_CFG_CANARY
    return A.afd_slot_layout(cfg)


def plain_window(run, buf):
    """A window of a run created with canaries, re-laid without the guard
    words (every field moved to its offset in the plain layout), for the
    oracle, which knows no guards."""
    Lg = run.layout
    if not Lg.guard:
        return buf
    Lp = plain_layout(run)
    out = np.zeros(Lp.window_bytes, np.uint8)
    nslots = run.cfg.num_peers * run.cfg.ring_depth
    out[:nslots * 8] = buf[:nslots * 8]
    names = ["header", "route_table", "routed_x", "shared_idx", "shared_x"]
    starts = [getattr(Lp, n) for n in names] + [Lp.slot_bytes]
    for s_ in range(nslots):
        bg = Lg.flags_bytes + s_ * Lg.slot_bytes
        bp = Lp.flags_bytes + s_ * Lp.slot_bytes
        for i, n in enumerate(names):
            size = starts[i + 1] - starts[i]
            if size:
                out[bp + starts[i]: bp + starts[i] + size] = buf[bg + getattr(Lg, n): bg + getattr(Lg, n) + size]
    return out


def check_canaries(run):
    """Every guard word after the slot fields intact (runs with canaries)."""
    if run.layout.guard:
        rc, win, off = A.afd_check_canaries(run.ctx)
        assert rc == A.AFD_OK, f"guard word changed: window {win}, byte offset {off}"


def rel_err(got, ref):
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 1.0
    return float(np.abs(got - ref).max() / rms) if ref.size else 0.0


def check_plan_exact(run, T, ids_ref):
    """GPU ids / counts / offsets / perm / inv against the oracle's plan of the
    oracle's ids, bit for bit."""
    w = run.w
    k, E = w.topk, w.num_experts
    ids = ws_array(run, A.AFD_WS_IDS, T * k, np.int32).reshape(T, k)
    assert np.array_equal(ids, ids_ref), f"{int((ids != ids_ref).sum())} ids differ"
    counts, offsets, perm, inv = O.plan(ids_ref, E)
    assert np.array_equal(ws_array(run, A.AFD_WS_COUNTS, E, np.int32), counts)
    assert np.array_equal(ws_array(run, A.AFD_WS_OFFSETS, E + 1, np.int32), offsets)
    assert np.array_equal(ws_array(run, A.AFD_WS_PERM, T * k, np.int32), perm)
    assert np.array_equal(ws_array(run, A.AFD_WS_INV, T * k, np.int32), inv)
    return ids


def run_and_compare_full(run, slots=None, layer=0, pack=True):
    """Whole-fan-in comparison (sizes the oracle finishes in seconds); with
    pack=False the caller has packed the slots."""
    w = run.w
    slots = list(range(w.num_peers)) if slots is None else slots
    if pack:
        run.pack_all(layer)
    rc = run.forward(layer, slots=slots)
    assert rc == 0, A.strerror(rc)
    outs = run.unpack_all(peers=slots)
    st = run.poll()
    assert st == 0, (A.strerror(st), A.afd_debug_bounds(run.ctx))
    check_canaries(run)
    # the oracle reads and writes windows without guard words
    win = plain_window(run, run.window(A.AFD_DIR_DISPATCH).cpu().numpy())
    ret = plain_window(run, run.window(A.AFD_DIR_RETURN).cpu().numpy())
    Lp = plain_layout(run)
    c = oracle_cfg(run)
    ret_orc = np.zeros_like(win)
    seen = np.zeros(w.num_peers, np.uint64)
    lens = [w.seq_lens[p] for p in slots]
    rc, r = O.ffn_forward(c, win.copy(), ret_orc, run.weights_numpy(layer), layer, 0, lens, slots,
                          seen)
    assert rc == 0
    T, k = sum(lens), w.topk
    check_plan_exact(run, T, r["ids"])
    assert A.afd_last_expert_counts(run.ctx) == [int(v) for v in r["counts"]]
    wts = ws_array(run, A.AFD_WS_WEIGHTS, T * k, np.float32).reshape(T, k)
    assert np.allclose(wts, r["w"], rtol=1e-6, atol=0), np.abs(wts / r["w"] - 1).max()
    errs = []
    start = 0
    nflags = run.cfg.num_peers * run.cfg.ring_depth * 8
    for p in slots:
        n = w.seq_lens[p]
        assert np.array_equal(header(ret, run, p, Lp), header(ret_orc, run, p, Lp))
        assert ret[:nflags].view(np.uint64)[p] == ret_orc[:nflags].view(np.uint64)[p]
        if n:
            assert np.array_equal(route_table(ret, run, p, n, Lp), route_table(ret_orc, run, p, n, Lp))
            got = return_rows(ret, run, p, n, Lp)
            ref = r["out64"][start:start + n]
            errs.append((got, ref))
            o = outs[p][:n].float().cpu().numpy().astype(np.float64)
            assert np.array_equal(o, got), "unpacked rows differ from the return slot"
        start += n
    got = np.concatenate([g for g, _ in errs]) if errs else np.zeros((0, w.hidden))
    ref = np.concatenate([r for _, r in errs]) if errs else np.zeros((0, w.hidden))
    e = rel_err(got, ref)
    assert e <= tol_for(w), f"max|err|/rms = {e:.3e} > {tol_for(w)}"
    return e, r
