"""ctypes binding of libafd_gb300.so (include/afd.h), argument marshalling only.

Every function keeps the C name.  Tensors are passed by data_ptr(); all
computation happens in the library's CUDA kernels.  Loading fails loudly
when the library has not been built: there is no other implementation.
"""
import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libafd_gb300.so")

AFD_OK = 0
(AFD_ERR_ARG, AFD_ERR_SHAPE, AFD_ERR_CAPACITY, AFD_ERR_HEADER, AFD_ERR_SEQ, AFD_ERR_LAYER,
 AFD_ERR_STAGE, AFD_ERR_TIMEOUT, AFD_ERR_SHUTDOWN, AFD_ERR_SPLIT_UNEVEN, AFD_ERR_NOT_DEVICE,
 AFD_ERR_CUDA, AFD_ERR_UNSUPPORTED, AFD_ERR_CANARY, AFD_ERR_BOUNDS) = range(1, 16)
AFD_DTYPE_F32, AFD_DTYPE_BF16 = 0, 1
AFD_GEMM_TENSOR, AFD_GEMM_SIMT, AFD_GEMM_TENSOR_1CTA = 0, 1, 2
AFD_CFG_NO_PDL = 1
AFD_CFG_CANARY = 2
AFD_CFG_SPLIT_GEMMS = 4
(AFD_DBG_GATHER_INV, AFD_DBG_GATHER_PERM, AFD_DBG_GATHER_GROUPED, AFD_DBG_COMBINE_INV,
 AFD_DBG_SCATTER_INV, AFD_DBG_GEMM_OUT) = range(1, 7)
AFD_DBG_NUM_SITES = 7
AFD_DIR_DISPATCH, AFD_DIR_RETURN = 0, 1
(AFD_WS_IDS, AFD_WS_WEIGHTS, AFD_WS_COUNTS, AFD_WS_OFFSETS, AFD_WS_PERM, AFD_WS_INV, AFD_WS_XP,
 AFD_WS_H, AFD_WS_Y, AFD_WS_HS, AFD_WS_S, AFD_WS_STATUS) = range(12)
AFD_HEADER_FIXED_WORDS = 12
AFD_NOALLOC_MAX_ROUTER_WEIGHTS = 262144
AFD_NOALLOC_MAX_LOGITS = 1048576
AFD_MAX_PEERS = 64
AFD_MAX_RING = 64
AFD_FORM_TOKENS, AFD_FORM_GROUPED = 0, 1
AFD_MAX_FFN_RANKS = 16


class afd_config(C.Structure):
    _fields_ = [("num_peers", C.c_int32), ("ring_depth", C.c_int32), ("token_cap", C.c_int32),
                ("max_total_tokens", C.c_int32), ("hidden", C.c_int32),
                ("num_experts", C.c_int32), ("topk", C.c_int32), ("inter", C.c_int32),
                ("shared_inter", C.c_int32), ("act_dtype", C.c_int32), ("renorm", C.c_int32),
                ("max_layers", C.c_int32), ("gemm", C.c_int32), ("flags", C.c_int32),
                ("routed_scaling", C.c_float), ("routed_cap_multiplier", C.c_float),
                ("wait_timeout_ns", C.c_int64), ("ffn_rank", C.c_int32), ("ffn_size", C.c_int32)]


class afd_layout(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("header", "route_table", "routed_x", "shared_idx",
                                         "shared_x", "slot_bytes", "flags_bytes",
                                         "window_bytes", "align", "guard")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class afd_stats(C.Structure):
    _fields_ = [("window_bytes", C.c_int64), ("workspace_bytes", C.c_int64),
                ("last_total_tokens", C.c_int32), ("num_sms", C.c_int32),
                ("forwards", C.c_int64)]


class AfdError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


_lib = None

# (name, restype, argtypes) -- mirrors include/afd.h
_P, _I, _I64, _U64, _F = C.c_void_p, C.c_int, C.c_int64, C.c_uint64, C.c_float
SIGNATURES = [
    ("afd_create", _I, [C.POINTER(afd_config), _P, C.POINTER(_P)]),
    ("afd_destroy", None, [_P]),
    ("afd_set_stream", _I, [_P, _P]),
    ("afd_slot_layout", _I, [C.POINTER(afd_config), C.POINTER(afd_layout)]),
    ("afd_split_sizes", _I, [_I, _I, C.POINTER(C.c_int), _I, C.POINTER(C.c_int)]),
    ("afd_set_layer", _I, [_P, _I, _P, _P, _P, _P, _P, _P]),
    ("afd_pack_slot", _I, [_P, _I, _I, _I, _P, _I, _I, _U64]),
    ("afd_announce_shutdown", _I, [_P, _I, _I, _U64]),
    ("afd_ffn_forward", _I, [_P, _I, _I, C.POINTER(C.c_int), C.POINTER(C.c_int), _I]),
    ("afd_unpack_split", _I, [_P, _I, _I, _P, _I, _U64]),
    ("afd_pack_slots", _I, [_P, _I, C.POINTER(C.c_int32), _I, _I, C.POINTER(_P), C.POINTER(C.c_int32), _I,
                            C.POINTER(_U64)]),
    ("afd_unpack_splits", _I, [_P, _I, C.POINTER(C.c_int32), _I, C.POINTER(_P), C.POINTER(C.c_int32),
                               C.POINTER(_U64)]),
    ("afd_pack_grouped", _I, [_P, _I, _I, _I, _P, _I, C.POINTER(C.c_int), _P, _I, _I, _U64]),
    ("afd_ffn_forward_grouped", _I, [_P, _I, _I, C.POINTER(C.c_int), C.POINTER(C.c_int),
                                     C.POINTER(C.c_int), _I]),
    ("afd_unpack_grouped", _I, [_P, _I, _I, _P, _I, _P, _I, _U64]),
    ("afd_poll_status", _I, [_P]),
    ("afd_get_window", _I, [_P, _I, C.POINTER(_P), C.POINTER(_I64)]),
    ("afd_get_workspace", _I, [_P, _I, C.POINTER(_P), C.POINTER(_I64)]),
    ("afd_get_stats", _I, [_P, C.POINTER(afd_stats)]),
    ("afd_last_expert_counts", _I, [_P, C.POINTER(C.c_int32), _I, C.POINTER(C.c_int)]),
    ("afd_launch_count", _I64, [_P]),
    ("afd_check_canaries", _I, [_P, C.POINTER(C.c_int), C.POINTER(_I64)]),
    ("afd_debug_bounds", _I, [_P, C.POINTER(C.c_int32), C.POINTER(_I64), C.POINTER(_I64)]),
    ("afd_debug_plant", _I, [_P, C.c_int32]),
    ("afd_strerror", C.c_char_p, [_I]),
    ("afd_profile", _I, [_P, _I]),
    ("afd_route_noalloc", _I, [_P, _I, _I, _I, _P, _P, _I, _I, _I, _F, _P, _P, _P]),
    ("afd_stage_times", _I, [_P, C.POINTER(C.c_float), _I, C.POINTER(C.c_int64)]),
    ("afd_ffn_serve", _I, [_P, C.POINTER(C.c_int), _I, _I, _I]),
    ("afd_serve_graph_create", _I, [_P, C.POINTER(C.c_int), _I, _I, _I, C.POINTER(_P),
                                    C.POINTER(_I64)]),
    ("afd_serve_graph_launch", _I, [_P]),
    ("afd_serve_graph_destroy", None, [_P]),
    ("afd_serve_log", _I, [_P, C.POINTER(C.c_int32), _I, C.POINTER(C.c_int),
                           C.POINTER(_I64)]),
    ("afd_get_config", _I, [_P, C.POINTER(afd_config)]),
    ("afd_expert_range", _I, [_I, _I, _I, C.POINTER(C.c_int), C.POINTER(C.c_int)]),
    ("afd_attn_create", _I, [C.POINTER(_P), _I, _I, _I, _P, C.POINTER(_P)]),
    ("afd_attn_destroy", None, [_P]),
    ("afd_attn_dispatch", _I, [_P, _I, _I, _P, _I, _P, _I, _U64]),
    ("afd_attn_combine", _I, [_P, _I, _P, _P, _I, _U64]),
    ("afd_attn_rows", _I, [_P, _I, C.POINTER(C.c_int)]),
    ("afd_attn_poll_status", _I, [_P]),
    ("afd_attn_launch_count", _I64, [_P]),
]
AFD_NUM_STAGES = 8
STAGE_NAMES = ("header_check", "router", "plan", "gather", "gemm_swiglu", "gemm_down",
               "combine_split", "return_header")


def lib(path=None):
    """Load the library once; raise if it is missing (build it with
    __graft_entry__.build() or combine_peer_slot_gb300/build.py).  The
    AFD_LIBRARY environment variable names another build to load instead
    (e.g. the bounds-checking libafd_gb300_dbg.so)."""
    global _lib
    if _lib is None:
        path = path or os.environ.get("AFD_LIBRARY") or LIB_PATH
        if not os.path.exists(path):
            raise ImportError(f"{path} is not built; run __graft_entry__.build()")
        L = C.CDLL(path)
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def strerror(code):
    return lib().afd_strerror(int(code)).decode()


def _check(rc, what):
    if rc != AFD_OK:
        raise AfdError(rc, what)
    return rc


def _ints(seq):
    arr = (C.c_int * max(len(seq), 1))(*[int(v) for v in seq])
    return arr


def make_config(num_peers, token_cap, hidden, num_experts, topk, inter, shared_inter=0,
                act="bf16", renorm=False, routed_scaling=1.0, ring_depth=1,
                max_total_tokens=0, max_layers=1, gemm=AFD_GEMM_TENSOR,
                routed_cap_multiplier=2.0, wait_timeout_ns=0, flags=0, ffn_rank=0, ffn_size=0):
    return afd_config(num_peers, ring_depth, token_cap, max_total_tokens, hidden, num_experts,
                      topk, inter, shared_inter,
                      AFD_DTYPE_BF16 if act == "bf16" else AFD_DTYPE_F32, int(bool(renorm)),
                      max_layers, gemm, int(flags), float(routed_scaling),
                      float(routed_cap_multiplier), int(wait_timeout_ns), int(ffn_rank),
                      int(ffn_size))


# ---- thin functional wrappers (same names as the C ABI) ----------------------
def afd_slot_layout(cfg):
    L = afd_layout()
    _check(lib().afd_slot_layout(C.byref(cfg), C.byref(L)), "afd_slot_layout")
    return L


def afd_split_sizes(total, n_peers, seq_lens):
    sizes = (C.c_int * max(n_peers, 1))()
    rc = lib().afd_split_sizes(int(total), int(n_peers), _ints(seq_lens), len(seq_lens), sizes)
    return rc, [int(sizes[i]) for i in range(n_peers)] if rc == AFD_OK else None


def afd_create(cfg, stream=0):
    ctx = C.c_void_p()
    _check(lib().afd_create(C.byref(cfg), C.c_void_p(int(stream)), C.byref(ctx)), "afd_create")
    return ctx


def afd_destroy(ctx):
    lib().afd_destroy(ctx)


def afd_set_stream(ctx, stream):
    return _check(lib().afd_set_stream(ctx, C.c_void_p(int(stream))), "afd_set_stream")


def afd_set_layer(ctx, layer, Wg, bias, W13, Wd, W13_s=0, Wd_s=0):
    """Pointers as ints (tensor.data_ptr())."""
    return _check(lib().afd_set_layer(ctx, int(layer), Wg, bias or None, W13, Wd,
                                      W13_s or None, Wd_s or None), "afd_set_layer")


def afd_pack_slot(ctx, peer, stage, layer, x_ptr, n_tokens, with_shared, seq):
    return lib().afd_pack_slot(ctx, peer, stage, layer, x_ptr or None, n_tokens,
                               int(bool(with_shared)), seq)


def afd_announce_shutdown(ctx, peer, stage, seq):
    return lib().afd_announce_shutdown(ctx, peer, stage, seq)


def afd_ffn_forward(ctx, layer, stage, seq_lens, slots):
    return lib().afd_ffn_forward(ctx, int(layer), int(stage), _ints(seq_lens), _ints(slots),
                                 len(slots))


def afd_unpack_split(ctx, peer, stage, out_ptr, n_tokens, expect_seq):
    return lib().afd_unpack_split(ctx, peer, stage, out_ptr or None, n_tokens, expect_seq)


def afd_pack_slots(ctx, peers, stage, layer, x_ptrs, n_tokens, with_shared, seqs):
    n = len(peers)
    return lib().afd_pack_slots(ctx, n, (C.c_int32 * n)(*peers), int(stage), int(layer),
                                (_P * n)(*[p or None for p in x_ptrs]), (C.c_int32 * n)(*n_tokens),
                                int(bool(with_shared)), (_U64 * n)(*seqs))


def afd_unpack_splits(ctx, peers, stage, out_ptrs, n_tokens, expect_seqs):
    n = len(peers)
    return lib().afd_unpack_splits(ctx, n, (C.c_int32 * n)(*peers), int(stage),
                                   (_P * n)(*[p or None for p in out_ptrs]), (C.c_int32 * n)(*n_tokens),
                                   (_U64 * n)(*expect_seqs))


def afd_pack_grouped(ctx, peer, stage, layer, rows_ptr, n_rows, group_list, x_ptr, n_tokens,
                     with_shared, seq):
    return lib().afd_pack_grouped(ctx, peer, stage, layer, rows_ptr or None, n_rows,
                                  _ints(group_list), x_ptr or None, n_tokens,
                                  int(bool(with_shared)), seq)


def afd_ffn_forward_grouped(ctx, layer, stage, n_rows, seq_lens, slots):
    return lib().afd_ffn_forward_grouped(ctx, int(layer), int(stage), _ints(n_rows),
                                         _ints(seq_lens), _ints(slots), len(slots))


def afd_unpack_grouped(ctx, peer, stage, y_ptr, n_rows, s_ptr, n_tokens, expect_seq):
    return lib().afd_unpack_grouped(ctx, peer, stage, y_ptr or None, n_rows, s_ptr or None,
                                    n_tokens, expect_seq)


def afd_poll_status(ctx):
    return lib().afd_poll_status(ctx)


def afd_get_window(ctx, direction):
    p, n = C.c_void_p(), C.c_int64()
    _check(lib().afd_get_window(ctx, direction, C.byref(p), C.byref(n)), "afd_get_window")
    return p.value, n.value


def afd_get_workspace(ctx, which):
    p, n = C.c_void_p(), C.c_int64()
    _check(lib().afd_get_workspace(ctx, which, C.byref(p), C.byref(n)), "afd_get_workspace")
    return p.value, n.value


def afd_get_stats(ctx):
    s = afd_stats()
    _check(lib().afd_get_stats(ctx, C.byref(s)), "afd_get_stats")
    return s


def afd_last_expert_counts(ctx, n=256):
    """Per-expert counts of the last step (a list of num_experts ints)."""
    buf = (C.c_int32 * n)()
    ne = C.c_int(0)
    _check(lib().afd_last_expert_counts(ctx, buf, n, C.byref(ne)), "afd_last_expert_counts")
    return [int(v) for v in buf[:min(n, ne.value)]]


def afd_check_canaries(ctx):
    """(status, window, byte offset of the first changed guard word)."""
    w, off = C.c_int(-1), C.c_int64(-1)
    rc = lib().afd_check_canaries(ctx, C.byref(w), C.byref(off))
    return rc, w.value, off.value


def afd_debug_bounds(ctx):
    """(status, site, index, limit) of the first failed bounds check of the
    debug build; AFD_ERR_UNSUPPORTED from the release build."""
    site, idx, lim = C.c_int32(0), C.c_int64(-1), C.c_int64(-1)
    rc = lib().afd_debug_bounds(ctx, C.byref(site), C.byref(idx), C.byref(lim))
    return rc, site.value, idx.value, lim.value


def afd_debug_plant(ctx, site):
    return lib().afd_debug_plant(ctx, int(site))


def afd_launch_count(ctx):
    return int(lib().afd_launch_count(ctx))


def afd_profile(ctx, enable):
    return _check(lib().afd_profile(ctx, int(bool(enable))), "afd_profile")


def afd_stage_times(ctx):
    """(per-stage milliseconds summed over the forwards since the previous
    call, number of those forwards)"""
    ms = (C.c_float * AFD_NUM_STAGES)()
    n = C.c_int64(0)
    _check(lib().afd_stage_times(ctx, ms, AFD_NUM_STAGES, C.byref(n)), "afd_stage_times")
    return [float(v) for v in ms], int(n.value)


def afd_route_noalloc(x_ptr, n_tokens, hidden, act_dtype, Wg_ptr, bias_ptr, num_experts, topk,
                      renorm, routed_scaling, ids_ptr, weights_ptr, stream=0):
    """Router step with no device allocation (see include/afd.h)."""
    return lib().afd_route_noalloc(x_ptr or None, int(n_tokens), int(hidden), int(act_dtype),
                                   Wg_ptr or None, bias_ptr or None, int(num_experts),
                                   int(topk), int(bool(renorm)), float(routed_scaling),
                                   ids_ptr or None, weights_ptr or None,
                                   C.c_void_p(int(stream)))


def afd_ffn_serve(ctx, slots, n_items, form=AFD_FORM_TOKENS):
    """n_items steps of the device-resident work-item loop over the peers in slots."""
    return lib().afd_ffn_serve(ctx, _ints(slots), len(slots), int(n_items), int(form))


def afd_serve_graph_create(ctx, slots, n_items, form=AFD_FORM_TOKENS):
    """(status, graph handle, kernels in the graph)"""
    g, k = C.c_void_p(), C.c_int64(0)
    rc = lib().afd_serve_graph_create(ctx, _ints(slots), len(slots), int(n_items), int(form),
                                      C.byref(g), C.byref(k))
    return rc, g, int(k.value)


def afd_serve_graph_launch(graph):
    return lib().afd_serve_graph_launch(graph)


def afd_serve_graph_destroy(graph):
    lib().afd_serve_graph_destroy(graph)


def afd_serve_log(ctx, max_records=64):
    """(records [(stage, layer, tokens, rows)] oldest first, items served)"""
    recs = (C.c_int32 * (4 * max(max_records, 1)))()
    n, served = C.c_int(0), C.c_int64(0)
    _check(lib().afd_serve_log(ctx, recs, int(max_records), C.byref(n), C.byref(served)),
           "afd_serve_log")
    return [tuple(recs[4 * j:4 * j + 4]) for j in range(n.value)], int(served.value)


def afd_get_config(ctx):
    c = afd_config()
    _check(lib().afd_get_config(ctx, C.byref(c)), "afd_get_config")
    return c


def afd_expert_range(num_experts, ffn_size, ffn_rank):
    """(first expert, count) of FFN rank ffn_rank among ffn_size"""
    first, count = C.c_int(0), C.c_int(0)
    _check(lib().afd_expert_range(int(num_experts), int(ffn_size), int(ffn_rank),
                                  C.byref(first), C.byref(count)), "afd_expert_range")
    return first.value, count.value


def afd_attn_create(ranks, peer, num_experts, stream=0):
    """One Attention peer over the FFN-rank contexts ranks (rank order)."""
    arr = (C.c_void_p * max(len(ranks), 1))(*[r.value if isinstance(r, C.c_void_p) else r
                                                for r in ranks])
    a = C.c_void_p()
    _check(lib().afd_attn_create(arr, len(ranks), int(peer), int(num_experts),
                                 C.c_void_p(int(stream)), C.byref(a)), "afd_attn_create")
    return a


def afd_attn_destroy(a):
    lib().afd_attn_destroy(a)


def afd_attn_dispatch(a, stage, layer, x_ptr, n_tokens, ids_ptr, with_shared, seq):
    return lib().afd_attn_dispatch(a, int(stage), int(layer), x_ptr or None, int(n_tokens),
                                   ids_ptr or None, int(bool(with_shared)), seq)


def afd_attn_combine(a, stage, w_ptr, out_ptr, n_tokens, expect_seq):
    return lib().afd_attn_combine(a, int(stage), w_ptr or None, out_ptr or None, int(n_tokens),
                                  expect_seq)


def afd_attn_rows(a, stage, ffn_size):
    rows = (C.c_int * ffn_size)()
    _check(lib().afd_attn_rows(a, int(stage), rows), "afd_attn_rows")
    return list(rows)


def afd_attn_poll_status(a):
    return lib().afd_attn_poll_status(a)


def afd_attn_launch_count(a):
    return int(lib().afd_attn_launch_count(a))
