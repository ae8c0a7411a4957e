"""The C-ABI library without a GPU: it loads, exports every function that
include/afd.h declares, and its host-only logic (slot layout, split sizes,
argument validation) agrees with the independent oracle and the fixtures."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from combine_peer_slot_gb300 import afd as A
from combine_peer_slot_gb300 import build as B
from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if B.needs_build():
        B.build()
    return A.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "afd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(afd_\w+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/afd.h but not exported"
    bound = {n for n, _, _ in A.SIGNATURES}
    assert set(names) == bound, set(names) ^ bound


def test_strerror(lib):
    for code in range(0, 16):
        assert A.strerror(code) and A.strerror(code) != "unknown status"
    assert A.strerror(99) == "unknown status"


def test_release_build_has_no_bounds_checks(lib):
    # the checks are compiled out: the record calls answer UNSUPPORTED
    # before they look at the context
    assert A.afd_debug_bounds(None)[0] == A.AFD_ERR_UNSUPPORTED
    assert A.afd_debug_plant(None, A.AFD_DBG_GEMM_OUT) == A.AFD_ERR_UNSUPPORTED


def test_layout_matches_oracle(golden, lib):
    for case in golden("slot_layout_tiny.json")["cases"]:
        cfg = A.make_config(case["num_regions"], case["token_cap"], case["hidden"],
                            case["num_experts"], case["topk"], 64,
                            shared_inter=64 if case["has_shared"] else 0,
                            act="f32" if case["act_bytes"] == 4 else "bf16",
                            ring_depth=case["ring_depth"], gemm=A.AFD_GEMM_SIMT)
        got = A.afd_slot_layout(cfg).as_dict()
        assert got.pop("guard") == 0
        assert got == case["expect"]
    rng = np.random.default_rng(2)
    for _ in range(300):
        P, D = int(rng.integers(1, 65)), int(rng.integers(1, 9))
        cap, k = int(rng.integers(1, 20000)), int(rng.integers(1, 17))
        H, E = int(rng.integers(1, 293)) * 8, int(rng.integers(k, 257))  # router tile fits
        act = str(rng.choice(["bf16", "f32"]))
        Is = int(rng.choice([0, 64]))
        cfg = A.make_config(P, cap, H, E, k, 64, shared_inter=Is, act=act, ring_depth=D,
                            gemm=A.AFD_GEMM_SIMT)
        ours = A.afd_slot_layout(cfg).as_dict()
        assert ours.pop("guard") == 0
        ref = O.slot_layout(P, D, cap, k, H, 2 if act == "bf16" else 4, E, Is > 0).as_dict()
        assert ours == ref


def test_canary_layout_adds_one_guard_after_every_field(lib):
    """AFD_CFG_CANARY: the flag array and every slot field are followed by one
    alignment unit of guard words, so each field sits after the guards of
    the fields before it and stays aligned."""
    rng = np.random.default_rng(5)
    for _ in range(200):
        P, D = int(rng.integers(1, 65)), int(rng.integers(1, 9))
        cap, k = int(rng.integers(1, 20000)), int(rng.integers(1, 17))
        H, E = int(rng.integers(1, 293)) * 8, int(rng.integers(k, 257))
        act = str(rng.choice(["bf16", "f32"]))
        Is = int(rng.choice([0, 64]))
        kw = dict(shared_inter=Is, act=act, ring_depth=D, gemm=A.AFD_GEMM_SIMT)
        plain = A.afd_slot_layout(A.make_config(P, cap, H, E, k, 64, **kw)).as_dict()
        g = A.afd_slot_layout(A.make_config(P, cap, H, E, k, 64, flags=A.AFD_CFG_CANARY, **kw)).as_dict()
        a = plain["align"]
        assert g["guard"] == a and g["align"] == a and plain["guard"] == 0
        fields = ["header", "route_table", "routed_x"] + (["shared_idx", "shared_x"] if Is else [])
        for i, f in enumerate(fields):
            assert g[f] == plain[f] + i * a and g[f] % a == 0
        assert g["slot_bytes"] == plain["slot_bytes"] + len(fields) * a
        assert g["flags_bytes"] == plain["flags_bytes"] + a
        assert g["window_bytes"] == g["flags_bytes"] + P * D * g["slot_bytes"]


def test_split_sizes(golden, lib):
    for c in golden("split_sizes.json")["cases"]:
        rc, sizes = A.afd_split_sizes(c["total"], c["n_peers"], c["seq_lens"])
        assert rc == c["status"], c
        if rc == 0:
            assert sizes == c["sizes"]


def test_config_validation(lib):
    ok = A.make_config(4, 8192, 2048, 64, 6, 1408, 2816)
    assert A.afd_slot_layout(ok).window_bytes > 0
    bad = [dict(num_peers=0), dict(num_peers=65), dict(topk=65), dict(hidden=0),
           dict(ring_depth=0), dict(ring_depth=A.AFD_MAX_RING + 1), dict(routed_cap_multiplier=0.5), dict(act_dtype=7)]
    for b in bad:
        cfg = A.make_config(4, 8192, 2048, 64, 6, 1408, 2816)
        for k, v in b.items():
            setattr(cfg, k, v)
        assert A.lib().afd_slot_layout(C.byref(cfg), C.byref(A.afd_layout())) == A.AFD_ERR_ARG, b
    unsupported = [dict(hidden=2044), dict(num_experts=300, topk=2), dict(topk=17),
                   dict(inter=1400), dict(act_dtype=A.AFD_DTYPE_F32)]
    for b in unsupported:
        cfg = A.make_config(4, 8192, 2048, 64, 6, 1408, 2816)
        for k, v in b.items():
            setattr(cfg, k, v)
        assert A.lib().afd_slot_layout(C.byref(cfg), C.byref(A.afd_layout())) == A.AFD_ERR_UNSUPPORTED, b


def test_noalloc_rejects_without_touching_the_device(lib):
    assert A.afd_route_noalloc(0, 4, 4104, A.AFD_DTYPE_BF16, 0, 0, 64, 6, 0, 1.0, 0, 0) == A.AFD_ERR_CAPACITY
    assert A.afd_route_noalloc(0, 4, 100, A.AFD_DTYPE_BF16, 0, 0, 64, 6, 0, 1.0, 0, 0) == A.AFD_ERR_ARG
    assert A.afd_route_noalloc(0, 0, 2048, A.AFD_DTYPE_BF16, 0, 0, 64, 6, 0, 1.0, 0, 0) == A.AFD_OK


def test_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(A.AfdError) as e:
        A.afd_create(A.make_config(2, 128, 1024, 16, 4, 512, 512))
    assert e.value.code == A.AFD_ERR_CUDA


def test_serve_rejects_bad_arguments_without_a_context(lib):
    """The work-item loop's host checks come before any device work."""
    assert A.afd_ffn_serve(None, [0], 1) == A.AFD_ERR_ARG
    rc, g, _ = A.afd_serve_graph_create(None, [0], 1)
    assert rc == A.AFD_ERR_ARG and not g.value
    assert A.afd_serve_graph_launch(None) == A.AFD_ERR_ARG
    A.afd_serve_graph_destroy(None)
    with pytest.raises(A.AfdError):
        A.afd_serve_log(None)


def test_rank_layout_and_experts_match_oracle(lib):
    """An FFN rank's slot layout under token-level dispatch (routed fields
    sized by routed_cap) and the expert placement, against the oracle."""
    rng = np.random.default_rng(5)
    for _ in range(200):
        F = int(rng.integers(1, A.AFD_MAX_FFN_RANKS + 1))
        E = int(rng.integers(F, 257))
        r = int(rng.integers(0, F))
        first, cnt = A.afd_expert_range(E, F, r)
        assert (first, cnt) == O.expert_range(E, F, r)
        cap, k = int(rng.integers(1, 5000)), int(rng.integers(1, 17))
        H = int(rng.integers(1, 129)) * 8
        mult = float(rng.choice([1.0, 1.5, 2.0, 3.0]))
        act = str(rng.choice(["bf16", "f32"]))
        Is = int(rng.choice([0, 64]))
        cfg = A.make_config(int(rng.integers(1, 9)), cap, H, cnt, min(k, cnt), 64,
                            shared_inter=Is, act=act, ring_depth=int(rng.integers(1, 4)),
                            gemm=A.AFD_GEMM_SIMT, routed_cap_multiplier=mult, ffn_rank=r,
                            ffn_size=F)
        ours = A.afd_slot_layout(cfg).as_dict()
        assert ours.pop("guard") == 0
        rcap = O.routed_cap(cap, min(k, cnt), F, mult)
        ref = O.slot_layout_ranks(cfg.num_peers, cfg.ring_depth, cap, min(k, cnt), H,
                                  2 if act == "bf16" else 4, cnt, Is > 0, rcap).as_dict()
        assert ours == ref
    assert lib.afd_expert_range(4, 5, 0, None, None) == A.AFD_ERR_ARG


def test_rank_config_validation(lib):
    base = dict(num_peers=2, token_cap=64, hidden=256, num_experts=8, topk=2, inter=64)
    for bad in (dict(ffn_size=A.AFD_MAX_FFN_RANKS + 1), dict(ffn_size=2, ffn_rank=2),
                dict(ffn_size=-1), dict(ffn_size=0, ffn_rank=1)):
        cfg = A.make_config(**{**base, **bad})
        with pytest.raises(A.AfdError) as e:
            A.afd_slot_layout(cfg)
        assert e.value.code == A.AFD_ERR_ARG, bad
    assert A.afd_slot_layout(A.make_config(**base, ffn_size=4, ffn_rank=3)).window_bytes > 0


def test_attn_rejects_bad_arguments_without_a_context(lib):
    import ctypes as C
    a = C.c_void_p()
    assert lib.afd_attn_create(None, 2, 0, 16, None, C.byref(a)) == A.AFD_ERR_ARG
    assert A.afd_attn_dispatch(None, 0, 0, 0, 0, 0, False, 1) == A.AFD_ERR_ARG
    assert A.afd_attn_combine(None, 0, 0, 0, 0, 1) == A.AFD_ERR_ARG
    assert A.afd_attn_poll_status(None) == A.AFD_ERR_ARG
    A.afd_attn_destroy(None)
