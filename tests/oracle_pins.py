"""Pins of the CPU oracle: checks against what the pages and mathematics fix.

Each check takes an oracle library handle, so the same checks run against
the real oracle (tests/test_oracle_pins.py) and against deliberately wrong
builds of it (the planted-mistake test), which must each fail at least one.
Independent formulations only: numpy matmuls, numpy's stable argsort and
bincount, closed forms, hand-derived fixtures.  Nothing here calls the CUDA
library.
"""
import math
import os

import numpy as np

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    import json
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# helpers: independent numpy formulations
# --------------------------------------------------------------------------
def np_silu(g):
    return g / (1.0 + np.exp(-g))


def act_to_f64(a, act_bytes):
    return O.bf16_bits_to_f32(a).astype(np.float64) if act_bytes == 2 else \
        np.asarray(a, np.float32).astype(np.float64)


def np_round_act(v, act_bytes):
    if act_bytes == 4:
        return v.astype(np.float32).astype(np.float64)
    import torch
    return torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def np_swiglu(X, W13, Wd, act_bytes):
    """Dense SwiGLU MLP with numpy matmuls: X [T, H], W13 [2I, H], Wd [H, I]."""
    I = W13.shape[0] // 2
    G = X @ W13[:I].T
    U = X @ W13[I:].T
    Hm = np_round_act(np_silu(G) * U, act_bytes)
    return Hm @ Wd.T


def rand_act(rng, shape, act_bytes, scale=1.0):
    a = (rng.standard_normal(shape) * scale).astype(np.float32)
    if act_bytes == 4:
        return a
    import torch
    return torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def make_problem(rng, *, seq_lens, hidden, E, k, inter, shared_inter, act_bytes,
                 renorm=False, scale=1.0, bias=False, ring_depth=1, num_regions=None,
                 token_cap=None):
    num_regions = num_regions or len(seq_lens)
    token_cap = token_cap or max(8, max(seq_lens))
    cfg = dict(num_regions=num_regions, ring_depth=ring_depth, token_cap=token_cap,
               hidden=hidden, act_bytes=act_bytes, num_experts=E, topk=k, inter=inter,
               shared_inter=shared_inter, renorm=renorm, max_total_tokens=0,
               routed_scaling=scale)
    xs = [rand_act(rng, (n, hidden), act_bytes) for n in seq_lens]
    Wt = dict(
        Wg=(rng.standard_normal((hidden, E)) / math.sqrt(hidden)).astype(np.float32),
        bias=(rng.standard_normal(E) * 0.5).astype(np.float32) if bias else None,
        W13=rand_act(rng, (E, 2 * inter, hidden), act_bytes, 1 / math.sqrt(hidden)),
        Wd=rand_act(rng, (E, hidden, inter), act_bytes, 1 / math.sqrt(inter)),
        W13s=rand_act(rng, (2 * shared_inter, hidden), act_bytes, 1 / math.sqrt(hidden))
        if shared_inter else None,
        Wds=rand_act(rng, (hidden, shared_inter), act_bytes, 1 / math.sqrt(shared_inter))
        if shared_inter else None)
    return cfg, xs, Wt


def run_forward(lib, cfg, xs, Wt, *, layer=0, stage=0, slots=None, seqs=None,
                with_shared=True, want_h=False):
    """Pack every peer into a host dispatch window, run the oracle step, and
    return (rc, result dict, return window, layout)."""
    L = O.slot_layout(cfg["num_regions"], cfg["ring_depth"], cfg["token_cap"], cfg["topk"],
                      cfg["hidden"], cfg["act_bytes"], cfg["num_experts"],
                      cfg["shared_inter"] > 0, lib=lib)
    win = np.zeros(L.window_bytes, np.uint8)
    ret = np.zeros(L.window_bytes, np.uint8)
    slots = list(range(len(xs))) if slots is None else slots
    seqs = seqs or [100 + i for i in range(len(xs))]
    for i, p in enumerate(slots):
        rc = O.pack_slot(win, L, cfg["ring_depth"], p, stage, layer, xs[i], cfg["hidden"],
                         cfg["act_bytes"], cfg["token_cap"], cfg["num_experts"],
                         with_shared and cfg["shared_inter"] > 0, cfg["shared_inter"] > 0,
                         seqs[i], lib=lib)
        assert rc == 0
    seen = np.zeros(cfg["num_regions"] * cfg["ring_depth"], np.uint64)
    rc, r = O.ffn_forward(cfg, win, ret, Wt, layer, stage, [x.shape[0] for x in xs], slots,
                          seen, want_h=want_h, lib=lib)
    return rc, r, win, ret, L


def return_rows(ret, L, cfg, peer, stage, n):
    off = L.flags_bytes + (peer * cfg["ring_depth"] + stage) * L.slot_bytes
    rb = cfg["hidden"] * cfg["act_bytes"]
    raw = ret[off + L.routed_x: off + L.routed_x + n * rb]
    dt = np.uint16 if cfg["act_bytes"] == 2 else np.float32
    return act_to_f64(raw.view(dt).reshape(n, cfg["hidden"]), cfg["act_bytes"])


def header_words(win, L, cfg, peer, stage):
    off = L.flags_bytes + (peer * cfg["ring_depth"] + stage) * L.slot_bytes + L.header
    return win[off: off + 4 * (12 + cfg["num_experts"])].view(np.int32)


# --------------------------------------------------------------------------
# checks
# --------------------------------------------------------------------------
def check_bf16(lib):
    import torch
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_to_f64(allbits, lib=lib)
    ref = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all((ours == ref) | both_nan)
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(4000).astype(np.float32) * 10,
                        (rng.standard_normal(500) * 1e-39).astype(np.float32),
                        np.array([0.0, -0.0, 3e38, -3e38, 1e-45, 65504.0], np.float32)])
    ref_bits = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f64_to_bf16(v.astype(np.float64), lib=lib), ref_bits)
    for case in _golden("bf16_rounding.json")["cases"]:
        assert int(O.f64_to_bf16([eval(case["value"])], lib=lib)[0]) == case["bits"], case


def check_layout(lib):
    for case in _golden("slot_layout_tiny.json")["cases"]:
        args = [case[n] for n in ("num_regions", "ring_depth", "token_cap", "topk", "hidden",
                                  "act_bytes", "num_experts", "has_shared")]
        assert O.slot_layout(*args, lib=lib).as_dict() == case["expect"]
    rng = np.random.default_rng(3)
    for _ in range(200):
        R, D = int(rng.integers(1, 17)), int(rng.integers(1, 3))
        cap, k = int(rng.integers(1, 5000)), int(rng.integers(1, 9))
        H, ab = int(rng.integers(1, 600)) * 8, int(rng.choice([2, 4]))
        E, sh = int(rng.integers(1, 257)), int(rng.integers(0, 2))
        L = O.slot_layout(R, D, cap, k, H, ab, E, sh, lib=lib).as_dict()
        row = H * ab
        fields = [("header", (12 + E) * 4), ("route_table", cap * k * 4),
                  ("routed_x", cap * row), ("shared_idx", cap * 4 * sh),
                  ("shared_x", cap * row * sh)]
        end = 0
        for name, size in fields:
            off = L[name]
            assert off % 256 == 0 and off % row == 0 and off % 4 == 0, (name, L)
            assert off >= end, "fields overlap"
            end = off + size
        assert end <= L["slot_bytes"] and L["slot_bytes"] % 256 == 0
        assert L["flags_bytes"] >= R * D * 8 and L["flags_bytes"] % row == 0
        assert L["window_bytes"] == L["flags_bytes"] + R * D * L["slot_bytes"]


def check_header_roundtrip(lib):
    g = _golden("header_magic.json")
    rng = np.random.default_rng(11)
    cfg, xs, Wt = make_problem(rng, seq_lens=[5, 3], hidden=64, E=4, k=2, inter=16,
                               shared_inter=16, act_bytes=2, ring_depth=2)
    L = O.slot_layout(2, 2, cfg["token_cap"], 2, 64, 2, 4, 1, lib=lib)
    win = np.zeros(L.window_bytes, np.uint8)
    assert O.pack_slot(win, L, 2, 1, 1, 7, xs[0], 64, 2, cfg["token_cap"], 4, 1, 1, 41,
                       shutdown=1, lib=lib) == 0
    h = header_words(win, L, cfg, 1, 1)
    assert bytes(h[:1].view(np.uint8)) == g["magic_bytes"].encode()
    assert int(h[0]) == g["magic_word_le"] and len(h) == g["fixed_words"] + 4
    assert int(h[2]) & g["shutdown_mask"]
    assert list(h[3:12]) == [41, 41, 7, 1, 5, 0, 5, 4, 16]
    flags = win[:L.flags_bytes].view(np.uint64)
    assert flags[1 * 2 + 1] == 41 and flags.sum() == 41
    off = L.flags_bytes + 3 * L.slot_bytes
    assert np.array_equal(win[off + L.routed_x: off + L.routed_x + xs[0].nbytes], xs[0].view(np.uint8).ravel())
    assert np.array_equal(win[off + L.shared_x: off + L.shared_x + xs[0].nbytes], xs[0].view(np.uint8).ravel())
    assert list(win[off + L.shared_idx: off + L.shared_idx + 20].view(np.int32)) == [0, 1, 2, 3, 4]
    rc, out = O.unpack_split(win, L, 2, 1, 1, 5, 64, 2, 4, 41, lib=lib)
    assert rc == 0 and np.array_equal(out, xs[0])
    assert O.unpack_split(win, L, 2, 1, 1, 5, 64, 2, 4, 42, lib=lib)[0] == O.ERR_TIMEOUT
    assert O.unpack_split(win, L, 2, 1, 1, 5, 64, 2, 4, 40, lib=lib)[0] == O.ERR_SEQ
    assert O.unpack_split(win, L, 2, 1, 1, 4, 64, 2, 4, 41, lib=lib)[0] == O.ERR_SHAPE
    win[off] ^= 1
    assert O.unpack_split(win, L, 2, 1, 1, 5, 64, 2, 4, 41, lib=lib)[0] == O.ERR_HEADER


def check_split(lib):
    for c in _golden("split_sizes.json")["cases"]:
        rc, sizes = O.split_sizes(c["total"], c["n_peers"], c["seq_lens"], lib=lib)
        assert rc == c["status"], c
        if rc == 0:
            assert sizes == c["sizes"]


def check_logit_order(lib):
    for c in _golden("logit_order.json")["cases"]:
        H = c["hidden"]
        x = np.zeros((1, H), np.float32)
        for h, v in c["x_nonzero"].items():
            x[0, int(h)] = v
        Wg = np.zeros((H, 2), np.float32)
        Wg[:, 0] = 1.0
        ids, w, gap, lg = O.route(x, 4, Wg, None, 1, False, 1.0, with_logits=True, lib=lib)
        assert float(lg[0, 0]) == c["expect"], (float(lg[0, 0]), c)


def check_router(lib):
    rng = np.random.default_rng(5)
    for ab, renorm, scale, bias in ((4, True, 1.0, False), (2, False, 2.5, True)):
        T, H, E, k = 96, 256, 16, 4
        x = rand_act(rng, (T, H), ab)
        Wg = (rng.standard_normal((H, E)) / 16).astype(np.float32)
        b = (rng.standard_normal(E) * 0.3).astype(np.float32) if bias else None
        ids, w, gap, lg = O.route(x, ab, Wg, b, k, renorm, scale, with_logits=True, lib=lib)
        X = act_to_f64(x, ab)
        L64 = X @ Wg.astype(np.float64) + (0 if b is None else b.astype(np.float64))
        bound = 1e-5 * (np.abs(X) @ np.abs(Wg.astype(np.float64)) + 1)
        assert np.all(np.abs(lg - L64) <= bound)
        order = np.argsort(-L64, axis=1, kind="stable")[:, :k]
        clear = np.sort(L64, axis=1)[:, ::-1]
        clear = (clear[:, k - 1] - clear[:, k]) > 2 * bound.max()
        assert np.array_equal(ids[clear], order[clear])
        P = np.exp(lg.astype(np.float64) - lg.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        wref = np.take_along_axis(P, ids, axis=1)
        if renorm:
            wref /= wref.sum(axis=1, keepdims=True)
            assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
        assert np.allclose(w, wref * scale, rtol=1e-6, atol=0)
        assert np.all(gap[clear] > 0)


def check_router_ties(lib):
    rng = np.random.default_rng(9)
    T, H, E, k = 400, 64, 8, 3
    x = rand_act(rng, (T, H), 4)
    Wg = (rng.standard_normal((H, E)) / 8).astype(np.float32)
    Wg[:, 5] = Wg[:, 2]
    ids, w, gap, lg = O.route(x, 4, Wg, None, k, False, 1.0, with_logits=True, lib=lib)
    assert np.array_equal(lg[:, 2], lg[:, 5])
    saw = 0
    for t in range(T):
        row = list(ids[t])
        if 5 in row:
            assert 2 in row and row.index(2) < row.index(5)
        if 2 in row and 5 not in row and row.index(2) == k - 1:
            saw += 1
    assert saw > 0, "no token exercised the boundary tie"


def check_plan(lib):
    rng = np.random.default_rng(13)
    for n, E in ((0, 4), (1, 1), (777, 16), (5000, 64)):
        ids = rng.integers(0, max(E // 2, 1), size=n).astype(np.int32)
        counts, offsets, perm, inv = O.plan(ids, E, lib=lib)
        assert np.array_equal(counts, np.bincount(ids, minlength=E))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        assert np.array_equal(perm, np.argsort(ids, kind="stable"))
        assert np.array_equal(inv[perm], np.arange(n))


def check_dense_swiglu(lib):
    """E = 1, k = 1: the layer is a plain dense SwiGLU MLP (plus the shared
    expert when present)."""
    rng = np.random.default_rng(17)
    for shared in (0, 24):
        cfg, xs, Wt = make_problem(rng, seq_lens=[6, 11], hidden=64, E=1, k=1, inter=40,
                                   shared_inter=shared, act_bytes=4)
        rc, r, win, ret, L = run_forward(lib, cfg, xs, Wt)
        assert rc == 0
        X = np.concatenate([act_to_f64(x, 4) for x in xs])
        ref = np_swiglu(X, act_to_f64(Wt["W13"][0], 4), act_to_f64(Wt["Wd"][0], 4), 4)
        if shared:
            ref = ref + np_swiglu(X, act_to_f64(Wt["W13s"], 4), act_to_f64(Wt["Wds"], 4), 4)
        assert np.all(r["w"] == 1.0)
        err = np.abs(r["out64"] - ref).max() / np.sqrt((ref ** 2).mean())
        assert err < 1e-6, err


def check_dense_mixture(lib):
    """sum over all experts with the unselected gates zeroed (numpy, dense)
    equals the routed layer."""
    rng = np.random.default_rng(19)
    for ab in (4, 2):
        cfg, xs, Wt = make_problem(rng, seq_lens=[9, 4, 12], hidden=64, E=8, k=3, inter=32,
                                   shared_inter=16, act_bytes=ab, renorm=(ab == 4))
        rc, r, win, ret, L = run_forward(lib, cfg, xs, Wt)
        assert rc == 0
        X = np.concatenate([act_to_f64(x, ab) for x in xs])
        T = X.shape[0]
        wdense = np.zeros((T, 8))
        np.put_along_axis(wdense, r["ids"], r["w"].astype(np.float64), axis=1)
        ref = np.zeros_like(X)
        for e in range(8):
            ref += wdense[:, e:e + 1] * np_swiglu(X, act_to_f64(Wt["W13"][e], ab),
                                                  act_to_f64(Wt["Wd"][e], ab), ab)
        ref += np_swiglu(X, act_to_f64(Wt["W13s"], ab), act_to_f64(Wt["Wds"], ab), ab)
        tol = 1e-6 if ab == 4 else 2e-3
        err = np.abs(r["out64"] - ref).max() / np.sqrt((ref ** 2).mean())
        assert err < tol, (ab, err)
        # the oracle's own dense-mixture entry agrees too
        xcat = np.concatenate(xs)
        dm = O.dense_mixture(xcat, ab, Wt, 8, 32, 16, wdense, lib=lib)
        assert np.abs(dm - r["out64"]).max() / np.sqrt((ref ** 2).mean()) < tol
        # returned rows are the fp64 result rounded once
        rows = np.concatenate([return_rows(ret, L, cfg, p, 0, xs[p].shape[0]) for p in range(3)])
        assert np.array_equal(rows, np_round_act(r["out64"], ab)) or ab == 2
        if ab == 2:
            assert np.abs(rows - r["out64"]).max() <= 2 ** -8 * np.abs(r["out64"]).max()


def check_identity_combine(lib):
    rng = np.random.default_rng(23)
    T, k, H = 7, 3, 5
    x = rng.standard_normal((T, H))
    s = rng.standard_normal((T, H))
    w = rng.random((T, k)).astype(np.float32)
    y = np.repeat(x[:, None, :], k, axis=1)
    out = O.combine(y, w, s, lib=lib)
    assert np.allclose(out, w.astype(np.float64).sum(1, keepdims=True) * x + s, rtol=1e-14)


def check_fanin_split(lib):
    """Each token's output depends on its own row only, so the fan-in result
    for a peer equals that peer run alone; a zero-length peer gets an empty
    slice; T = sum(seq_lens)."""
    rng = np.random.default_rng(29)
    cfg, xs, Wt = make_problem(rng, seq_lens=[5, 0, 9, 3], hidden=32, E=4, k=2, inter=16,
                               shared_inter=8, act_bytes=4)
    order = [2, 0, 3, 1]
    rc, r, win, ret, L = run_forward(lib, cfg, [xs[p] for p in order], Wt, slots=order)
    assert rc == 0 and r["ids"].shape[0] == sum(x.shape[0] for x in xs)
    for p in range(4):
        n = xs[p].shape[0]
        h = header_words(ret, L, cfg, p, 0)
        assert h[7] == n and h[8] == n * 2
        alone_cfg = dict(cfg)
        rc1, r1, _, ret1, _ = run_forward(lib, alone_cfg, [xs[p]], Wt, slots=[p])
        assert rc1 == 0
        if n:
            assert np.array_equal(return_rows(ret, L, cfg, p, 0, n),
                                  return_rows(ret1, L, cfg, p, 0, n))
            counts = np.bincount(r1["ids"].ravel(), minlength=4)
            assert list(h[12:]) == list(counts)


def check_hand_moe(lib):
    g = _golden("hand_moe.json")
    cfg = dict(num_regions=1, ring_depth=1, token_cap=4, hidden=2, act_bytes=4,
               num_experts=2, topk=1, inter=1, shared_inter=1, renorm=False,
               max_total_tokens=0, routed_scaling=1.0)
    Wt = {k: np.array(g[k], np.float32) for k in ("Wg", "W13", "Wd", "W13s", "Wds")}
    Wt["bias"] = None
    rc, r, win, ret, L = run_forward(lib, cfg, [np.array(g["x"], np.float32)], Wt)
    assert rc == 0 and r["ids"].tolist() == g["expect_ids"]
    s1, s3 = 1 / (1 + math.exp(-1)), 1 / (1 + math.exp(-3))
    expect = [2 * s1 ** 2 - 3 * s3, -2 * s1 ** 2 - 3 * s3]
    assert np.allclose(r["out64"][0], expect, atol=g["tolerance_abs"], rtol=0)


def check_fault_codes(lib):
    rng = np.random.default_rng(31)
    cfg, xs, Wt = make_problem(rng, seq_lens=[4, 6], hidden=32, E=4, k=2, inter=8,
                               shared_inter=8, act_bytes=2, token_cap=8)
    L = O.slot_layout(2, 1, 8, 2, 32, 2, 4, 1, lib=lib)

    def packed():
        win = np.zeros(L.window_bytes, np.uint8)
        for p in range(2):
            assert O.pack_slot(win, L, 1, p, 0, 3, xs[p], 32, 2, 8, 4, 1, 1, 10 + p, lib=lib) == 0
        return win

    def fwd(win, layer=3, stage=0, seq_lens=(4, 6), slots=(0, 1), seen=None, c=cfg):
        ret = np.zeros(L.window_bytes, np.uint8)
        seen = np.zeros(2, np.uint64) if seen is None else seen
        return O.ffn_forward(c, win, ret, Wt, layer, stage, list(seq_lens), list(slots), seen,
                             lib=lib)[0]

    assert fwd(packed()) == O.OK
    hdr = lambda win, p: L.flags_bytes + p * L.slot_bytes + L.header
    for word, val, code in ((0, 0x12345678, O.ERR_HEADER), (1, 2, O.ERR_HEADER),
                            (10, 5, O.ERR_HEADER), (11, 99, O.ERR_HEADER),
                            (3, 77, O.ERR_SEQ), (4, 77, O.ERR_SEQ), (2, 2, O.ERR_SHUTDOWN),
                            (5, 4, O.ERR_LAYER), (6, 1, O.ERR_STAGE), (7, 5, O.ERR_SHAPE),
                            (8, 3, O.ERR_SHAPE), (9, 2, O.ERR_SHAPE)):
        win = packed()
        win[hdr(win, 1) + 4 * word: hdr(win, 1) + 4 * word + 4] = np.array([val], np.int32).view(np.uint8)
        assert fwd(win) == code, (word, val, code)
    win = packed()
    sidx = L.flags_bytes + 1 * L.slot_bytes + L.shared_idx
    win[sidx + 4: sidx + 8] = np.array([3], np.int32).view(np.uint8)
    assert fwd(win) == O.ERR_SHAPE
    assert fwd(packed(), seq_lens=(4, 5)) == O.ERR_SHAPE
    assert fwd(packed(), seen=np.array([10, 0], np.uint64)) == O.ERR_TIMEOUT
    assert fwd(packed(), slots=(0, 0)) == O.ERR_ARG
    assert fwd(packed(), stage=1) == O.ERR_ARG
    assert fwd(packed(), seq_lens=(4, 9)) == O.ERR_CAPACITY
    assert fwd(packed(), c=dict(cfg, max_total_tokens=9)) == O.ERR_CAPACITY
    win = np.zeros(L.window_bytes, np.uint8)
    big = rand_act(rng, (9, 32), 2)
    assert O.pack_slot(win, L, 1, 0, 0, 3, big, 32, 2, 8, 4, 1, 1, 5, lib=lib) == O.ERR_CAPACITY
    # a consumed slot is not consumed again: the flag must advance
    win = packed()
    seen = np.zeros(2, np.uint64)
    assert fwd(win, seen=seen) == O.OK
    assert list(seen) == [10, 11]
    assert fwd(win, seen=seen) == O.ERR_TIMEOUT


def grouped_dispatch(ids, x, k, E):
    """The Attention side's grouped send for one peer: the flattened top-k
    ids sorted stably (numpy), the token rows in that order, bincount as the
    group list.  Returns (rows, group_list, order) with order[r] = t*k + j."""
    order = np.argsort(ids.reshape(-1), kind="stable")
    rows = np.ascontiguousarray(x[order // k])
    return rows, np.bincount(ids.reshape(-1), minlength=E).astype(np.int32), order


def run_grouped(lib, cfg, xs, Wt, ids_per_peer, *, layer=0, stage=0, seqs=None,
                with_shared=True):
    L = O.slot_layout(cfg["num_regions"], cfg["ring_depth"], cfg["token_cap"], cfg["topk"],
                      cfg["hidden"], cfg["act_bytes"], cfg["num_experts"],
                      cfg["shared_inter"] > 0, lib=lib)
    win = np.zeros(L.window_bytes, np.uint8)
    ret = np.zeros(L.window_bytes, np.uint8)
    seqs = seqs or [200 + i for i in range(len(xs))]
    orders, R = [], []
    for p, x in enumerate(xs):
        rows, gl, order = grouped_dispatch(ids_per_peer[p], x, cfg["topk"], cfg["num_experts"])
        rc = O.pack_grouped(win, L, cfg["ring_depth"], p, stage, layer, rows, gl, x,
                            cfg["hidden"], cfg["act_bytes"], cfg["token_cap"],
                            cfg["num_experts"], with_shared and cfg["shared_inter"] > 0,
                            cfg["shared_inter"] > 0, seqs[p], lib=lib)
        assert rc == 0, rc
        orders.append(order)
        R.append(rows.shape[0])
    seen = np.zeros(cfg["num_regions"] * cfg["ring_depth"], np.uint64)
    rc, y, sh = O.grouped_forward(cfg, win, ret, Wt, layer, stage, R, [x.shape[0] for x in xs],
                                  list(range(len(xs))), seen, lib=lib)
    return rc, y, sh, orders, R, win, ret, L


def check_grouped_dense(lib):
    """Grouped form, E = 1: every row goes through the one expert (a dense
    SwiGLU MLP, numpy) and the shared rows through the shared MLP."""
    rng = np.random.default_rng(23)
    cfg, xs, Wt = make_problem(rng, seq_lens=[5, 9], hidden=64, E=1, k=1, inter=40,
                               shared_inter=24, act_bytes=4)
    ids = [np.zeros((x.shape[0], 1), np.int32) for x in xs]
    rc, y, sh, orders, R, win, ret, L = run_grouped(lib, cfg, xs, Wt, ids)
    assert rc == 0
    X = np.concatenate([act_to_f64(x, 4) for x in xs])
    ref = np_swiglu(X, act_to_f64(Wt["W13"][0], 4), act_to_f64(Wt["Wd"][0], 4), 4)
    refs = np_swiglu(X, act_to_f64(Wt["W13s"], 4), act_to_f64(Wt["Wds"], 4), 4)
    for got, want in ((y, ref), (sh, refs)):
        err = np.abs(got - want).max() / np.sqrt((want ** 2).mean())
        assert err < 1e-6, err
    # the return slot carries the rows rounded once, and the group list echoed
    for p, x in enumerate(xs):
        n = x.shape[0]
        start = sum(r.shape[0] for r in xs[:p])
        assert np.array_equal(return_rows(ret, L, cfg, p, 0, n), np_round_act(y[start:start + n], 4))
        hw = header_words(ret, L, cfg, p, 0)
        assert hw[8] == n and hw[12] == n and hw[9] == n


def check_grouped_combine(lib):
    """The Attention side's combine of the grouped outputs (sum over j
    ascending of w[t,j] * y[row of (t,j)], then + s[t], fp64) equals the FFN-side
    routed layer on the same tokens and ids, exactly."""
    rng = np.random.default_rng(29)
    for ab in (4, 2):
        cfg, xs, Wt = make_problem(rng, seq_lens=[7, 0, 12], hidden=64, E=8, k=3, inter=32,
                                   shared_inter=16, act_bytes=ab, token_cap=48)
        rc, r, win0, ret0, L0 = run_forward(lib, cfg, xs, Wt)
        assert rc == 0
        k = cfg["topk"]
        prefix = np.cumsum([0] + [x.shape[0] for x in xs])
        ids_pp = [r["ids"][prefix[p]:prefix[p + 1]] for p in range(len(xs))]
        rc, y, sh, orders, R, win, ret, L = run_grouped(lib, cfg, xs, Wt, ids_pp)
        assert rc == 0
        rbase = np.cumsum([0] + R)
        for p in range(len(xs)):
            pos = np.empty(R[p], np.int64)
            pos[orders[p]] = np.arange(R[p])   # row of (t, j) for this peer
            for tl in range(xs[p].shape[0]):
                t = prefix[p] + tl
                acc = np.zeros(cfg["hidden"])
                for j in range(k):
                    acc = acc + np.float64(r["w"][t, j]) * y[rbase[p] + pos[tl * k + j]]
                acc = acc + sh[t]
                assert np.array_equal(acc, r["out64"][t]), (ab, p, tl)


def check_grouped_faults(lib):
    """Grouped form: a group list that does not sum to the row count, a row
    count other than the call's, too many rows."""
    rng = np.random.default_rng(31)
    cfg, xs, Wt = make_problem(rng, seq_lens=[6], hidden=32, E=4, k=2, inter=16,
                               shared_inter=0, act_bytes=4, token_cap=16)
    ids = [rng.integers(0, 4, size=(6, 2)).astype(np.int32)]
    rc, y, sh, orders, R, win, ret, L = run_grouped(lib, cfg, xs, Wt, ids)
    assert rc == 0
    def fwd(w, rows=None):
        seen = np.zeros(1, np.uint64)
        out = np.zeros_like(w)
        return O.grouped_forward(cfg, w, out, Wt, 0, 0, rows or R, [6], [0], seen, lib=lib)[0]
    assert fwd(win, rows=[R[0] - 1]) == O.ERR_SHAPE
    bad = win.copy()
    off = L.flags_bytes + L.header
    bad[off + 4 * 12: off + 4 * 13] = np.array([R[0] + 1], np.int32).view(np.uint8)
    assert fwd(bad) == O.ERR_SHAPE
    assert fwd(win, rows=[17]) == O.ERR_CAPACITY
    rows, gl, _ = grouped_dispatch(ids[0], xs[0], 2, 4)
    assert O.pack_grouped(win, L, 1, 0, 0, 0, rows, gl + np.array([1, 0, 0, 0], np.int32), xs[0],
                          32, 4, 16, 4, 0, 0, 301, lib=lib) == O.ERR_SHAPE


# --------------------------------------------------------------------------
# several FFN ranks
# --------------------------------------------------------------------------
def check_expert_range(lib):
    """Experts of FFN rank r among F (a reading: contiguous blocks, the first
    E mod F ranks one expert more): the blocks tile 0..E-1 in rank order,
    every rank holds at least one, and sizes differ by at most one, larger
    first."""
    for E in range(1, 41):
        for F in range(1, E + 1):
            got = [O.expert_range(E, F, r, lib=lib) for r in range(F)]
            nxt = 0
            for first, cnt in got:
                assert first == nxt and cnt >= 1, (E, F, got)
                nxt += cnt
            assert nxt == E
            sizes = [c for _, c in got]
            assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)


def check_routed_cap(lib):
    """routed_cap against hand-computed values of the page's formula
    (tests/golden/routed_cap.json)."""
    for c in _golden("routed_cap.json")["cases"]:
        got = O.routed_cap(c["token_cap"], c["topk"], c["ffn_size"], c["multiplier"], lib=lib)
        assert got == c["routed_cap"], (c, got)
    # the round-robin share: arange(r, n, F)
    for n in range(0, 30):
        for F in range(1, 7):
            for r in range(F):
                assert O.rr_rows(n, r, F, lib=lib) == len(range(r, n, F))


def ranks_setup(F, E, k, hidden, ab, token_cap, mult, has_shared, lib, num_regions=2,
                ring_depth=1):
    rcap = O.routed_cap(token_cap, k, F, mult, lib=lib)
    Ls, wins, rets = [], [], []
    for r in range(F):
        _, cnt = O.expert_range(E, F, r, lib=lib)
        L = O.slot_layout_ranks(num_regions, ring_depth, token_cap, k, hidden, ab, cnt, has_shared,
                                rcap, lib=lib)
        Ls.append(L)
        wins.append(np.zeros(L.window_bytes, np.uint8))
        rets.append(np.zeros(L.window_bytes, np.uint8))
    return rcap, Ls, wins, rets


def slot_field(win, L, region, stage, ring_depth, field, nbytes):
    off = L.flags_bytes + (region * ring_depth + stage) * L.slot_bytes + getattr(L, field)
    return win[off: off + nbytes]


def distinct_topk(rng, n, E, k):
    return np.argsort(rng.random((n, E)), axis=1)[:, :k].astype(np.int32)


def check_dispatch_ranks(lib):
    """One peer's send to F ranks, against the page's unit-test list: every
    partial routed exactly once, each destination's segment grouped by local
    expert (stable: numpy's stable argsort restricted to the rank's
    experts), E not divisible by F, the shared rows round-robin, an empty
    destination (a header with no rows, its flag still written), and a
    segment over routed_cap raising before anything is written."""
    rng = np.random.default_rng(41)
    H, ab, E, F, k, n, cap = 32, 4, 10, 4, 3, 11, 16
    rcap, Ls, wins, _ = ranks_setup(F, E, k, H, ab, cap, 2.0, True, lib)
    x = rand_act(rng, (n, H), ab)
    ids = distinct_topk(rng, n, E, k)
    rc, dst, pos, rows = O.dispatch_ranks(wins, Ls, 1, 1, 0, 3, x, ids, E, H, ab, cap, rcap, True,
                                          True, 77, lib=lib)
    assert rc == 0
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")
    seen = []
    for r in range(F):
        first, cnt = O.expert_range(E, F, r, lib=lib)
        mine = order[(flat[order] >= first) & (flat[order] < first + cnt)]
        assert rows[r] == mine.size
        table = slot_field(wins[r], Ls[r], 1, 0, 1, "route_table", 4 * mine.size).view(np.int32)
        assert np.array_equal(table, mine)          # grouped by local expert, stable
        seen.extend(table.tolist())
        assert np.array_equal(dst[mine], np.full(mine.size, r)) and np.array_equal(pos[mine], np.arange(mine.size))
        got = slot_field(wins[r], Ls[r], 1, 0, 1, "routed_x", mine.size * H * 4).view(np.float32)
        assert np.array_equal(got.reshape(-1, H), x[mine // k])
        h = slot_field(wins[r], Ls[r], 1, 0, 1, "header", 4 * (12 + cnt)).view(np.int32)
        share = np.arange(r, n, F)
        assert h[5] == 3 and h[7] == n and h[8] == mine.size and h[9] == share.size and h[10] == cnt
        assert np.array_equal(h[12:], np.bincount(flat - first, minlength=E)[:cnt]
                              if False else np.bincount(flat, minlength=E)[first:first + cnt])
        sidx = slot_field(wins[r], Ls[r], 1, 0, 1, "shared_idx", 4 * share.size).view(np.int32)
        assert np.array_equal(sidx, share)
        sx = slot_field(wins[r], Ls[r], 1, 0, 1, "shared_x", share.size * H * 4).view(np.float32)
        assert np.array_equal(sx.reshape(-1, H), x[share])
        assert wins[r][:Ls[r].flags_bytes].view(np.uint64)[1] == 77
    assert sorted(seen) == list(range(n * k))     # every partial exactly once
    # an empty destination: two tokens (ranks 2 and 3 get no shared row), all
    # ids among rank 0's experts
    rcap, Ls, wins, _ = ranks_setup(F, E, k, H, ab, cap, 2.0, True, lib)
    x2 = rand_act(rng, (2, H), ab)
    ids2 = np.array([[0, 1, 2], [2, 1, 0]], np.int32)
    rc, dst, pos, rows = O.dispatch_ranks(wins, Ls, 1, 0, 0, 0, x2, ids2, E, H, ab, cap, rcap, True,
                                          True, 5, lib=lib)
    assert rc == 0 and list(rows) == [6, 0, 0, 0]
    for r in (2, 3):
        _, cnt = O.expert_range(E, F, r, lib=lib)
        h = slot_field(wins[r], Ls[r], 0, 0, 1, "header", 4 * (12 + cnt)).view(np.int32)
        assert h[8] == 0 and h[9] == 0 and not h[12:].any()
        assert wins[r][:8].view(np.uint64)[0] == 5
    # overflow: every partial on rank 0 with the multiplier at 1.0 (even share
    # ceil(16 * 3 / 4) = 12 < 33 partials): raise, write nothing
    rcap, Ls, wins, _ = ranks_setup(F, E, k, H, ab, cap, 1.0, True, lib)
    ids3 = np.tile(np.array([0, 1, 2], np.int32), (n, 1))
    rc, _, _, _ = O.dispatch_ranks(wins, Ls, 1, 0, 0, 0, x, ids3, E, H, ab, cap, rcap, True, True, 9,
                                   lib=lib)
    assert rc == O.ERR_CAPACITY
    assert all(not w.any() for w in wins)


def ranks_round_trip(lib, F, E, ab, xs, Wt, ids, ws, with_shared, k, H, inter, shared_inter, cap):
    """Dispatch every peer to F ranks, run each rank's grouped step (its own
    expert slice of the weights), combine on the Attention side; returns the
    per-peer fp64 outputs."""
    P = len(xs)
    rcap, Ls, wins, rets = ranks_setup(F, E, k, H, ab, cap, 2.0, shared_inter > 0, lib,
                                       num_regions=P)
    plans = []
    for p in range(P):
        rc, dst, pos, rows = O.dispatch_ranks(wins, Ls, 1, p, 0, 0, xs[p], ids[p], E, H, ab, cap,
                                              rcap, with_shared, shared_inter > 0, 500 + p,
                                              lib=lib)
        assert rc == 0, rc
        plans.append((dst, pos, rows))
    for r in range(F):
        first, cnt = O.expert_range(E, F, r, lib=lib)
        cfg = dict(num_regions=P, ring_depth=1, token_cap=cap, hidden=H, act_bytes=ab,
                   num_experts=cnt, topk=k, inter=inter, shared_inter=shared_inter, renorm=False,
                   max_total_tokens=0, routed_scaling=1.0, ffn_rank=r, ffn_size=F,
                   routed_cap=rcap)
        Wr = dict(Wt)
        Wr["W13"] = np.ascontiguousarray(Wt["W13"][first:first + cnt])
        Wr["Wd"] = np.ascontiguousarray(Wt["Wd"][first:first + cnt])
        seen = np.zeros(P, np.uint64)
        rc, _, _ = O.grouped_forward(cfg, wins[r], rets[r], Wr, 0, 0,
                                     [int(plans[p][2][r]) for p in range(P)],
                                     [x.shape[0] for x in xs], list(range(P)), seen, lib=lib)
        assert rc == 0, (r, rc)
    outs = []
    for p in range(P):
        dst, pos, rows = plans[p]
        rc, out64, _ = O.attn_combine(rets, Ls, 1, p, 0, xs[p].shape[0], k, dst, pos, ws[p], rows,
                                      with_shared, H, ab, 500 + p, lib=lib)
        assert rc == 0, rc
        outs.append(out64)
    return outs


def check_ranks_round_trip(lib):
    """Token-level dispatch to F ranks, each rank's grouped step on its own
    experts and round-robin shared rows, then the Attention side's combine,
    equals the same step with one FFN rank, exactly (the same expert
    arithmetic on the same rows, the same summation order); for E divisible
    by F and not, with and without the shared expert, fp32 and bf16."""
    rng = np.random.default_rng(43)
    H, k, inter, Is = 64, 3, 32, 16
    for ab in (4, 2):
        for E, F, with_shared in ((8, 2, True), (10, 4, True), (6, 3, False), (9, 2, True)):
            cfg, xs, Wt = make_problem(rng, seq_lens=[7, 12], hidden=H, E=E, k=k, inter=inter,
                                       shared_inter=Is, act_bytes=ab, token_cap=48)
            ids = [distinct_topk(rng, x.shape[0], E, k) for x in xs]
            ws = [rng.random((x.shape[0], k)).astype(np.float32) for x in xs]
            one = ranks_round_trip(lib, 1, E, ab, xs, Wt, ids, ws, with_shared, k, H, inter, Is, 12)
            many = ranks_round_trip(lib, F, E, ab, xs, Wt, ids, ws, with_shared, k, H, inter, Is, 12)
            for p in range(len(xs)):
                assert np.array_equal(one[p], many[p]), (ab, E, F, p)
            # and the single rank is the grouped form of the FFN-side layer:
            # dense mixture with these ids and weights (numpy, tolerance)
            for p, x in enumerate(xs):
                X = act_to_f64(x, ab)
                ref = np.zeros_like(one[p])
                for t in range(X.shape[0]):
                    for j in range(k):
                        e = ids[p][t, j]
                        y = np_swiglu(X[t:t + 1], act_to_f64(Wt["W13"][e], ab),
                                      act_to_f64(Wt["Wd"][e], ab), ab)[0]
                        ref[t] += np.float64(ws[p][t, j]) * np_round_act(y, ab)
                if with_shared:
                    ref += np_round_act(np_swiglu(X, act_to_f64(Wt["W13s"], ab),
                                                  act_to_f64(Wt["Wds"], ab), ab), ab)
                err = np.abs(one[p] - ref).max() / np.sqrt((ref ** 2).mean())
                assert err < (1e-2 if ab == 2 else 1e-5), (ab, E, F, p, err)


def check_ranks_faults(lib):
    """An FFN rank's header checks: shared rows other than its round-robin
    share, or shared_idx not r, r + F, ...: AFD_ERR_SHAPE; more routed rows
    than routed_cap: AFD_ERR_CAPACITY."""
    rng = np.random.default_rng(47)
    H, ab, E, F, k, n, cap, inter = 32, 4, 6, 2, 2, 9, 16, 16
    cfg0, xs, Wt = make_problem(rng, seq_lens=[n], hidden=H, E=E, k=k, inter=inter,
                                shared_inter=16, act_bytes=ab, token_cap=cap)
    rcap, Ls, wins, rets = ranks_setup(F, E, k, H, ab, cap, 2.0, True, lib, num_regions=1)
    ids = distinct_topk(rng, n, E, k)
    rc, dst, pos, rows = O.dispatch_ranks(wins, Ls, 1, 0, 0, 0, xs[0], ids, E, H, ab, cap, rcap, True,
                                          True, 11, lib=lib)
    assert rc == 0
    r = 1
    first, cnt = O.expert_range(E, F, r, lib=lib)
    cfg = dict(cfg0, num_regions=1, num_experts=cnt, ffn_rank=r, ffn_size=F, routed_cap=rcap)
    Wr = dict(Wt, W13=np.ascontiguousarray(Wt["W13"][first:first + cnt]),
              Wd=np.ascontiguousarray(Wt["Wd"][first:first + cnt]))

    def fwd(w, R=None):
        return O.grouped_forward(cfg, w, np.zeros_like(w), Wr, 0, 0, [int(rows[r]) if R is None else R],
                                 [n], [0], np.zeros(1, np.uint64), lib=lib)[0]
    assert fwd(wins[r]) == 0
    hoff = Ls[r].flags_bytes + Ls[r].header
    bad = wins[r].copy()
    bad[hoff + 4 * 9: hoff + 4 * 10] = np.array([n], np.int32).view(np.uint8)   # all n tokens
    assert fwd(bad) == O.ERR_SHAPE
    bad = wins[r].copy()
    soff = Ls[r].flags_bytes + Ls[r].shared_idx
    bad[soff: soff + 4] = np.array([0], np.int32).view(np.uint8)   # rank 0's first token
    assert fwd(bad) == O.ERR_SHAPE
    assert fwd(wins[r], R=rcap + 1) == O.ERR_CAPACITY


ALL_CHECKS = [check_bf16, check_layout, check_header_roundtrip, check_split,
              check_logit_order, check_router, check_router_ties, check_plan,
              check_dense_swiglu, check_dense_mixture, check_identity_combine,
              check_fanin_split, check_hand_moe, check_fault_codes, check_grouped_dense,
              check_grouped_combine, check_grouped_faults, check_expert_range, check_routed_cap,
              check_dispatch_ranks, check_ranks_round_trip, check_ranks_faults]
