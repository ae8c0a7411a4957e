"""Helpers shared by the GPU parity tests: run a workload through the C ABI
and compare it with the CPU oracle on the same slot bytes."""
import numpy as np

from combine_peer_slot_gb300 import afd as A
from combine_peer_slot_gb300 import runtime as R
from oracle import oracle as O

BF16_TOL = 2e-2   # max |err| <= 2e-2 * rms(oracle), bf16 activations
F32_TOL = 1e-4    # max |err| <= 1e-4 * rms(oracle), fp32 activations


def tol_for(w):
    return BF16_TOL if w.act == "bf16" else F32_TOL


def ws_array(run, which, count, dtype):
    nbytes = count * np.dtype(dtype).itemsize
    if nbytes == 0:
        return np.zeros(0, dtype)
    return run.workspace(which, nbytes).cpu().numpy().view(dtype)


def slot_off(run, peer, stage=0):
    """Byte offset of slot (peer, stage); the runner uses one stage per peer."""
    L = run.layout
    return L.flags_bytes + (peer * run.cfg.ring_depth + stage) * L.slot_bytes


def return_rows(ret, run, peer, n):
    L, w = run.layout, run.w
    off = slot_off(run, peer) + L.routed_x
    rb = w.hidden * w.act_bytes
    raw = ret[off: off + n * rb]
    if w.act == "bf16":
        return O.bf16_bits_to_f32(raw.view(np.uint16)).astype(np.float64).reshape(n, w.hidden)
    return raw.view(np.float32).astype(np.float64).reshape(n, w.hidden)


def route_table(ret, run, peer, n):
    off = slot_off(run, peer) + run.layout.route_table
    return ret[off: off + n * run.w.topk * 4].view(np.int32).reshape(n, run.w.topk)


def header(buf, run, peer):
    off = slot_off(run, peer) + run.layout.header
    return buf[off: off + 4 * (12 + run.w.num_experts)].view(np.int32)


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
    assert run.poll() == 0
    win = run.window(A.AFD_DIR_DISPATCH).cpu().numpy()
    ret = run.window(A.AFD_DIR_RETURN).cpu().numpy()
    c = run.oracle_cfg()
    ret_orc = np.zeros_like(win)
    seen = np.zeros(w.num_peers, np.uint64)
    lens = [w.seq_lens[p] for p in slots]
    rc, r = O.ffn_forward(c, win.copy(), ret_orc, run.weights_numpy(layer), layer, 0, lens, slots,
                          seen)
    assert rc == 0
    T, k = sum(lens), w.topk
    check_plan_exact(run, T, r["ids"])
    wts = ws_array(run, A.AFD_WS_WEIGHTS, T * k, np.float32).reshape(T, k)
    assert np.allclose(wts, r["w"], rtol=1e-6, atol=0), np.abs(wts / r["w"] - 1).max()
    errs = []
    start = 0
    for p in slots:
        n = w.seq_lens[p]
        assert np.array_equal(header(ret, run, p), header(ret_orc, run, p))
        assert ret[:run.layout.flags_bytes].view(np.uint64)[p] == ret_orc[:run.layout.flags_bytes].view(np.uint64)[p]
        if n:
            assert np.array_equal(route_table(ret, run, p, n), route_table(ret_orc, run, p, n))
            got = return_rows(ret, run, p, n)
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


def sample_tokens(lens, per_peer=6, seed=0):
    rng = np.random.default_rng(seed)
    toks, start = [], 0
    for n in lens:
        if n:
            pick = {start, start + n - 1}
            pick.update((start + rng.integers(0, n, size=per_peer)).tolist())
            toks.extend(sorted(pick))
        start += n
    return np.array(toks, np.int32)


def run_and_compare_sampled(run, layer=0, per_peer=6, nthreads=0, check_routing=True):
    """Full-size comparison: routing, counts, offsets, permutation bit-exact
    over every token; outputs on sampled tokens (first, last and random rows
    of every peer) computed one by one by the oracle."""
    w = run.w
    slots = list(range(w.num_peers))
    lens = [w.seq_lens[p] for p in slots]
    run.pack_all(layer)
    rc = run.forward(layer)
    assert rc == 0, A.strerror(rc)
    assert run.poll() == 0
    win = run.window(A.AFD_DIR_DISPATCH).cpu().numpy()
    ret = run.window(A.AFD_DIR_RETURN).cpu().numpy()
    T, k = sum(lens), w.topk
    wts = run.weights_numpy(layer)
    if check_routing:
        X = np.concatenate([run.host["x"][p] for p in slots])
        ids_ref, w_ref, gap = O.route(X, w.act_bytes, wts["Wg"], wts["bias"], k, w.renorm,
                                      w.routed_scaling, nthreads=nthreads)
        check_plan_exact(run, T, ids_ref)
        g = ws_array(run, A.AFD_WS_WEIGHTS, T * k, np.float32).reshape(T, k)
        assert np.allclose(g, w_ref, rtol=1e-6, atol=0)
    toks = sample_tokens(lens, per_peer, seed=layer)
    c = run.oracle_cfg()
    ids_s, w_s, out_s = O.forward_tokens(c, win, wts, 0, lens, slots, toks, nthreads=nthreads)
    prefix = np.concatenate([[0], np.cumsum(lens)])
    got = np.zeros_like(out_s)
    for q, t in enumerate(toks):
        p = int(np.searchsorted(prefix, t, side="right") - 1)
        local = int(t - prefix[p])
        got[q] = return_rows(ret, run, slots[p], local + 1)[local]
        assert np.array_equal(route_table(ret, run, slots[p], local + 1)[local], ids_s[q])
    e = rel_err(got, out_s)
    assert e <= tol_for(w), f"max|err|/rms = {e:.3e} > {tol_for(w)}"
    # return headers: per-peer expert counts from the oracle's routing
    if check_routing:
        for i, p in enumerate(slots):
            h = header(ret, run, p)
            n = lens[i]
            assert h[7] == n and h[8] == n * k and h[3] == run.last_seq[(p, 0)]
            cnt = np.bincount(ids_ref[prefix[i]:prefix[i] + n].ravel(), minlength=w.num_experts)
            assert np.array_equal(h[12:], cnt)
    return e
