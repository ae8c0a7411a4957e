"""ctypes binding of the C oracle (afd_oracle.c) with numpy marshalling.

Test infrastructure only.  Each wrapper names the C function it calls; the
arithmetic and its citations live in afd_oracle.c.
"""
import ctypes as C
import os

import numpy as np

from . import build_oracle

OK, ERR_ARG, ERR_SHAPE, ERR_CAPACITY, ERR_HEADER, ERR_SEQ, ERR_LAYER, ERR_STAGE, \
    ERR_TIMEOUT, ERR_SHUTDOWN, ERR_SPLIT_UNEVEN = range(11)

HEADER_FIXED_WORDS = 12
(H_MAGIC, H_VERSION, H_FLAGS, H_SEQ, H_ECHO_SEQ, H_LAYER, H_STAGE, H_NUM_TOKENS,
 H_ROUTED_TOKENS, H_SHARED_TOKENS, H_NUM_EXPERTS, H_LEN) = range(12)


class Layout(C.Structure):
    _fields_ = [(n, C.c_int64) for n in (
        "header", "route_table", "routed_x", "shared_idx", "shared_x",
        "slot_bytes", "flags_bytes", "window_bytes", "align")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class Weights(C.Structure):
    _fields_ = [("Wg", C.c_void_p), ("bias", C.c_void_p), ("W13", C.c_void_p),
                ("Wd", C.c_void_p), ("W13s", C.c_void_p), ("Wds", C.c_void_p)]


class Cfg(C.Structure):
    _fields_ = [("num_regions", C.c_int), ("ring_depth", C.c_int),
                ("token_cap", C.c_int), ("hidden", C.c_int),
                ("act_bytes", C.c_int), ("num_experts", C.c_int),
                ("topk", C.c_int), ("inter", C.c_int), ("shared_inter", C.c_int),
                ("renorm", C.c_int), ("max_total_tokens", C.c_int),
                ("routed_scaling", C.c_float), ("ffn_rank", C.c_int), ("ffn_size", C.c_int),
                ("routed_cap", C.c_int64)]


_LIBS = {}


def load(path=None):
    """Load the oracle library (building it if needed); path selects a
    planted variant built elsewhere."""
    if path is None:
        path = build_oracle.ensure_built()
    if path in _LIBS:
        return _LIBS[path]
    lib = C.CDLL(path)
    P, I, I64, U64, F, V = C.c_void_p, C.c_int, C.c_int64, C.c_uint64, C.c_float, None
    sig = {
        "orc_bf16_to_f64": (C.c_double, [C.c_uint16]),
        "orc_f64_to_bf16": (C.c_uint16, [C.c_double]),
        "orc_slot_layout": (I, [I, I, I, I, I, I, I, I, P]),
        "orc_pack_slot": (I, [P, P, I, I, I, I, P, I, I, I, I, I, I, I, U64, I]),
        "orc_unpack_split": (I, [P, P, I, I, I, P, I, I, I, I, U64]),
        "orc_split_sizes": (I, [I, I, P, I, P]),
        "orc_route": (V, [P, I, I, I, P, P, I, I, I, F, P, P, P, P, I]),
        "orc_plan": (I, [P, I, I, P, P, P, P]),
        "orc_dense_mixture": (V, [P, I, I, I, I, I, I, P, P, P]),
        "orc_ffn_forward": (I, [P, P, P, P, I, I, P, P, I, P, P, P, P, P, P, P, P, P, P, I]),
        "orc_forward_tokens": (I, [P, P, P, I, P, P, I, P, I, P, P, P, I]),
        "orc_combine": (V, [P, P, P, I, I, I, P]),
        "orc_pack_grouped": (I, [P, P, I, I, I, I, P, I, P, P, I, I, I, I, I, I, I, U64]),
        "orc_grouped_forward": (I, [P, P, P, P, I, I, P, P, P, I, P, P, P, I]),
        "orc_num_threads": (I, []),
        "orc_slot_layout_ranks": (I, [I, I, I, I, I, I, I, I, I64, P]),
        "orc_expert_range": (V, [I, I, I, P, P]),
        "orc_routed_cap": (I64, [I, I, I, C.c_double]),
        "orc_rr_rows": (I, [I, I, I]),
        "orc_dispatch_ranks": (I, [P, P, I, I, I, I, I, P, I, P, I, I, I, I, I, I64, I, I, U64,
                                   P, P, P]),
        "orc_attn_combine": (I, [P, P, I, I, I, I, I, I, P, P, P, P, I, I, I, U64, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIBS[path] = lib
    return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# bf16
# --------------------------------------------------------------------------
def bf16_to_f64(bits, lib=None):
    lib = lib or load()
    return np.array([lib.orc_bf16_to_f64(int(b)) for b in np.ravel(bits)])


def f64_to_bf16(vals, lib=None):
    lib = lib or load()
    return np.array([lib.orc_f64_to_bf16(float(v)) for v in np.ravel(vals)],
                    dtype=np.uint16)


def bf16_bits_to_f32(bits):
    """Exact widening of bf16 bit patterns (uint16 array) to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# layout / pack / unpack / split
# --------------------------------------------------------------------------
def slot_layout(num_regions, ring_depth, token_cap, topk, hidden, act_bytes,
                num_experts, has_shared, lib=None):
    lib = lib or load()
    L = Layout()
    rc = lib.orc_slot_layout(num_regions, ring_depth, token_cap, topk, hidden,
                             act_bytes, num_experts, int(bool(has_shared)), C.byref(L))
    if rc:
        raise ValueError(f"orc_slot_layout rc={rc}")
    return L


def pack_slot(win, L, ring_depth, region, stage, layer, x, hidden, act_bytes,
              token_cap, num_experts, with_shared, has_shared, seq, shutdown=0,
              lib=None):
    """x: uint16 bf16 bits or float32 array [n, hidden]; win: uint8 array."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    return lib.orc_pack_slot(_p(win), C.byref(L), ring_depth, region, stage, layer,
                             _p(x), int(x.shape[0]), hidden, act_bytes, token_cap,
                             num_experts, int(with_shared), int(has_shared), seq,
                             int(shutdown))


def unpack_split(win, L, ring_depth, region, stage, n_tokens, hidden, act_bytes,
                 num_experts, expect_seq, lib=None):
    lib = lib or load()
    dt = np.uint16 if act_bytes == 2 else np.float32
    out = np.zeros((n_tokens, hidden), dtype=dt)
    rc = lib.orc_unpack_split(_p(win), C.byref(L), ring_depth, region, stage, _p(out),
                              n_tokens, hidden, act_bytes, num_experts, expect_seq)
    return rc, out


def split_sizes(total, n_peers, seq_lens, lib=None):
    lib = lib or load()
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    sizes = np.zeros(max(n_peers, 1), dtype=np.int32)
    rc = lib.orc_split_sizes(total, n_peers, _p(sl), int(sl.size), _p(sizes))
    return rc, sizes[:n_peers].tolist()


# --------------------------------------------------------------------------
# router / plan / experts
# --------------------------------------------------------------------------
def route(x, act_bytes, Wg, bias, k, renorm, scale, nthreads=0, with_logits=False,
          lib=None):
    lib = lib or load()
    x = np.ascontiguousarray(x)
    T, H = x.shape
    E = Wg.shape[1]
    Wg = _c(Wg, np.float32)
    bias = _c(bias, np.float32)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    gap = np.zeros(T, np.float64)
    lg = np.zeros((T, E), np.float32) if with_logits else None
    lib.orc_route(_p(x), act_bytes, T, H, _p(Wg), _p(bias), E, k, int(renorm),
                  float(scale), _p(ids), _p(w), _p(gap), _p(lg), nthreads)
    return (ids, w, gap, lg) if with_logits else (ids, w, gap)


def plan(ids, E, lib=None):
    lib = lib or load()
    ids = np.ascontiguousarray(ids, dtype=np.int32).ravel()
    n = ids.size
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(max(n, 1), np.int32)
    inv = np.zeros(max(n, 1), np.int32)
    rc = lib.orc_plan(_p(ids), n, E, _p(counts), _p(offsets), _p(perm), _p(inv))
    if rc:
        raise ValueError(f"orc_plan rc={rc}")
    return counts, offsets, perm[:n], inv[:n]


def _weights(wt):
    keep = {k: (_c(v, np.float32) if k in ("Wg", "bias") else
                (None if v is None else np.ascontiguousarray(v)))
            for k, v in wt.items()}
    W = Weights(*[None if keep.get(n) is None else keep[n].ctypes.data
                  for n, _ in Weights._fields_])
    return W, keep


def dense_mixture(x, act_bytes, Wdict, E, inter, shared_inter, wdense, lib=None):
    lib = lib or load()
    W, keep = _weights(Wdict)
    x = np.ascontiguousarray(x)
    T, H = x.shape
    out = np.zeros((T, H), np.float64)
    wd = np.ascontiguousarray(wdense, dtype=np.float64)
    lib.orc_dense_mixture(_p(x), act_bytes, T, H, E, inter, shared_inter, C.byref(W),
                          _p(wd), _p(out))
    return out


def combine(y, w, s=None, lib=None):
    lib = lib or load()
    T, k, H = y.shape
    y = np.ascontiguousarray(y, np.float64)
    w = np.ascontiguousarray(w, np.float32)
    s = None if s is None else np.ascontiguousarray(s, np.float64)
    out = np.zeros((T, H), np.float64)
    lib.orc_combine(_p(y), _p(w), _p(s), T, k, H, _p(out))
    return out


def make_cfg(c):
    """c: dict with num_regions, ring_depth, token_cap, hidden, act_bytes,
    num_experts, topk, inter, shared_inter, renorm, max_total_tokens,
    routed_scaling; for one FFN rank among several also ffn_rank, ffn_size
    and routed_cap (num_experts is then the rank's own count)."""
    return Cfg(c["num_regions"], c["ring_depth"], c["token_cap"], c["hidden"],
               c["act_bytes"], c["num_experts"], c["topk"], c["inter"],
               c["shared_inter"], int(c["renorm"]), c.get("max_total_tokens", 0),
               float(c.get("routed_scaling", 1.0)), int(c.get("ffn_rank", 0)),
               int(c.get("ffn_size", 1)), int(c.get("routed_cap", 0)))


def ffn_forward(c, in_win, ret_win, Wdict, layer, stage, seq_lens, slots, seen,
                want_h=False, nthreads=0, lib=None):
    """Run the whole FFN step on host windows; returns (rc, dict)."""
    lib = lib or load()
    cfg = make_cfg(c)
    W, keep = _weights(Wdict)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    sp = np.ascontiguousarray(slots, np.int32)
    T = int(sl.sum())
    k, E, H = c["topk"], c["num_experts"], c["hidden"]
    r = dict(ids=np.zeros((T, k), np.int32), w=np.zeros((T, k), np.float32),
             counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
             perm=np.zeros(max(T * k, 1), np.int32), inv=np.zeros(max(T * k, 1), np.int32),
             gap=np.zeros(max(T, 1), np.float64), out64=np.zeros((max(T, 1), H), np.float64))
    h = np.zeros((max(T, 1), k, c["inter"]), np.float64) if want_h else None
    rc = lib.orc_ffn_forward(C.byref(cfg), _p(in_win), _p(ret_win), C.byref(W), layer,
                             stage, _p(sl), _p(sp), int(sl.size), _p(seen),
                             _p(r["ids"]), _p(r["w"]), _p(r["counts"]), _p(r["offsets"]),
                             _p(r["perm"]), _p(r["inv"]), _p(r["gap"]), _p(r["out64"]),
                             _p(h), nthreads)
    r["perm"], r["inv"] = r["perm"][:T * k], r["inv"][:T * k]
    r["gap"], r["out64"] = r["gap"][:T], r["out64"][:T]
    if want_h:
        r["h"] = h[:T]
    return rc, r


def pack_grouped(win, L, ring_depth, region, stage, layer, rows, group_list, x, hidden,
                 act_bytes, token_cap, num_experts, with_shared, has_shared, seq, lib=None):
    """Grouped (Attention-side gate) dispatch: rows [R, hidden] grouped by
    expert with group_list [E] rows per expert; x [n, hidden] the peer's
    tokens (the shared rows)."""
    lib = lib or load()
    rows = np.ascontiguousarray(rows)
    x = np.ascontiguousarray(x)
    gl = np.ascontiguousarray(group_list, np.int32)
    return lib.orc_pack_grouped(_p(win), C.byref(L), ring_depth, region, stage, layer,
                                _p(rows), int(rows.shape[0]), _p(gl), _p(x), int(x.shape[0]),
                                hidden, act_bytes, token_cap, num_experts, int(with_shared),
                                int(has_shared), seq)


def grouped_forward(c, in_win, ret_win, Wdict, layer, stage, rows, seq_lens, slots, seen,
                    nthreads=0, lib=None):
    """FFN step of the grouped form on host windows; returns (rc, y64 [sum R, H],
    s64 [sum n, H])."""
    lib = lib or load()
    cfg = make_cfg(c)
    W, keep = _weights(Wdict)
    rw = np.ascontiguousarray(rows, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    sp = np.ascontiguousarray(slots, np.int32)
    H = c["hidden"]
    F, r = int(c.get("ffn_size", 1)), int(c.get("ffn_rank", 0))
    ns = sum(rr_rows(int(n), r, F, lib) for n in sl) if F > 1 else int(sl.sum())
    y = np.zeros((max(int(rw.sum()), 1), H), np.float64)
    s = np.zeros((max(ns, 1), H), np.float64)
    rc = lib.orc_grouped_forward(C.byref(cfg), _p(in_win), _p(ret_win), C.byref(W), layer, stage,
                                 _p(rw), _p(sl), _p(sp), int(sl.size), _p(seen), _p(y), _p(s),
                                 nthreads)
    return rc, y[:int(rw.sum())], s[:ns]


def forward_tokens(c, in_win, Wdict, stage, seq_lens, slots, tokens, nthreads=0,
                   lib=None):
    lib = lib or load()
    cfg = make_cfg(c)
    W, keep = _weights(Wdict)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    sp = np.ascontiguousarray(slots, np.int32)
    tk = np.ascontiguousarray(tokens, np.int32)
    n, k, H = tk.size, c["topk"], c["hidden"]
    ids = np.zeros((n, k), np.int32)
    w = np.zeros((n, k), np.float32)
    out = np.zeros((n, H), np.float64)
    rc = lib.orc_forward_tokens(C.byref(cfg), _p(in_win), C.byref(W), stage, _p(sl),
                                _p(sp), int(sl.size), _p(tk), n, _p(ids), _p(w),
                                _p(out), nthreads)
    if rc:
        raise ValueError(f"orc_forward_tokens rc={rc}")
    return ids, w, out


# --------------------------------------------------------------------------
# several FFN ranks: expert placement, capacity, dispatch, combine
# --------------------------------------------------------------------------
def slot_layout_ranks(num_regions, ring_depth, token_cap, topk, hidden, act_bytes, num_experts,
                      has_shared, routed_cap, lib=None):
    lib = lib or load()
    L = Layout()
    rc = lib.orc_slot_layout_ranks(num_regions, ring_depth, token_cap, topk, hidden, act_bytes,
                                   num_experts, int(bool(has_shared)), int(routed_cap), C.byref(L))
    if rc:
        raise ValueError(f"orc_slot_layout_ranks rc={rc}")
    return L


def expert_range(E, F, r, lib=None):
    """(first expert, count) of FFN rank r among F"""
    lib = lib or load()
    first, count = C.c_int(0), C.c_int(0)
    lib.orc_expert_range(E, F, r, C.byref(first), C.byref(count))
    return first.value, count.value


def routed_cap(token_cap, topk, F, multiplier, lib=None):
    return int((lib or load()).orc_routed_cap(token_cap, topk, F, float(multiplier)))


def rr_rows(n, r, F, lib=None):
    return int((lib or load()).orc_rr_rows(int(n), int(r), int(F)))


def dispatch_ranks(wins, layouts, ring_depth, region, stage, layer, x, ids, E, hidden, act_bytes,
                   token_cap, rcap, with_shared, has_shared, seq, lib=None):
    """One peer's send to len(wins) FFN ranks; returns (rc, dst [n*k], pos [n*k],
    rows per rank [F])."""
    lib = lib or load()
    F = len(wins)
    x = np.ascontiguousarray(x)
    ids = np.ascontiguousarray(ids, np.int32)
    n, k = ids.shape
    wp = (C.c_void_p * F)(*[w.ctypes.data for w in wins])
    Ls = (Layout * F)(*layouts)
    dst = np.full(max(n * k, 1), -1, np.int32)
    pos = np.full(max(n * k, 1), -1, np.int32)
    rows = np.zeros(F, np.int32)
    rc = lib.orc_dispatch_ranks(C.cast(wp, C.c_void_p), C.cast(Ls, C.c_void_p), F, ring_depth,
                                region, stage, layer, _p(x), n, _p(ids), k, E, hidden, act_bytes,
                                token_cap, int(rcap), int(bool(with_shared)),
                                int(bool(has_shared)), seq, _p(dst), _p(pos), _p(rows))
    return rc, dst[:n * k], pos[:n * k], rows


def attn_combine(rets, layouts, ring_depth, region, stage, n, k, dst, pos, w, rows, with_shared,
                 hidden, act_bytes, expect_seq, lib=None):
    """The Attention side's combine of F ranks' returns; (rc, out64 [n, H],
    out in the activation type (uint16 bf16 bits or float32))."""
    lib = lib or load()
    F = len(rets)
    rp = (C.c_void_p * F)(*[r.ctypes.data for r in rets])
    Ls = (Layout * F)(*layouts)
    dst = np.ascontiguousarray(dst, np.int32)
    pos = np.ascontiguousarray(pos, np.int32)
    w = np.ascontiguousarray(w, np.float32)
    rows = np.ascontiguousarray(rows, np.int32)
    out64 = np.zeros((max(n, 1), hidden), np.float64)
    out = np.zeros((max(n, 1), hidden), np.uint16 if act_bytes == 2 else np.float32)
    rc = lib.orc_attn_combine(C.cast(rp, C.c_void_p), C.cast(Ls, C.c_void_p), F, ring_depth,
                              region, stage, n, k, _p(dst), _p(pos), _p(w), _p(rows),
                              int(bool(with_shared)), hidden, act_bytes, expect_seq, _p(out64),
                              _p(out))
    return rc, out64[:n], out[:n]


def num_threads(lib=None):
    return (lib or load()).orc_num_threads()


def lib_path():
    return build_oracle.LIB if os.path.exists(build_oracle.LIB) else None
