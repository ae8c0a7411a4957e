"""Cases run against the bounds-checking debug build (libafd_gb300_dbg.so),
in a process of their own that loads that build (AFD_LIBRARY).  Called by
tests/test_debug_bounds_gpu.py; prints one JSON line.

Clean runs: the debug build gives the oracle's results on the token form
(both gather orders, the three GEMM engines) and the grouped form, and no
check fails; nor on the full-size V2-Lite prefill fan-in and all 26 layers of
the decode-shaped pass.  Planted runs: for each check site, afd_debug_plant makes every
check there fail on valid indices (the bound is taken as 0, so the access is
skipped and no index out of range is used); the step must then report
AFD_ERR_BOUNDS and the record must name the site, after which a clean step
on the same context matches the oracle again."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from combine_peer_slot_gb300 import afd as A  # noqa: E402
from combine_peer_slot_gb300 import runtime as R  # noqa: E402
from combine_peer_slot_gb300 import workloads as W  # noqa: E402
from tests import gpu_parity as G  # noqa: E402
from tests import test_grouped_gpu as TG  # noqa: E402


def workload(name):
    if name == "fanin":        # position-order gather (T * k <= 8192)
        return W.get("fanin")
    if name == "token_order":  # T * k = 9200 > 8192: token-order gather
        return W.custom("fanin", seq_lens=[1200, 1100])
    if name == "grouped":
        return W.custom("fanin", token_cap=384)
    raise KeyError(name)


def clean_token_form(name, gemm):
    w = workload(name)
    run = R.Runner(w, max_total_tokens=w.total_tokens, gemm=gemm)
    err, _ = G.run_and_compare_full(run)
    rc = A.afd_debug_bounds(run.ctx)
    run.close()
    return {"err": err, "bounds": rc[0]}


def clean_grouped():
    w = workload("grouped")
    args = TG.run_grouped(w, seed=5)
    err = TG.compare(w, *args)
    rc = A.afd_debug_bounds(args[0].ctx)
    args[0].close()
    return {"err": err, "bounds": rc[0]}


def clean_full_size(name):
    """A full-size workload through the debug build (every layer of it): no
    check fails and every step ends without error (its outputs are compared
    with the oracle by the release build's parity tests)."""
    w = W.get(name)
    run = R.Runner(w, max_total_tokens=w.total_tokens)
    for layer in range(w.layers):
        run.pack_all(layer)
        assert run.forward(layer) == A.AFD_OK
        run.unpack_all()
    st = run.poll()
    rc = A.afd_debug_bounds(run.ctx)
    run.close()
    return {"step": st, "bounds": rc[0], "layers": w.layers}


def planted(site, name, gemm=A.AFD_GEMM_TENSOR):
    """One step with `site` planted, then a clean step on the same context."""
    w = workload(name)
    run = R.Runner(w, max_total_tokens=w.total_tokens, gemm=gemm)
    assert A.afd_debug_plant(run.ctx, site) == A.AFD_OK
    if name == "grouped":
        run.prepare_grouped(seed=5)
        run.pack_grouped_all()
        rc_fwd = run.forward_grouped()
    else:
        run.pack_all(0)
        rc_fwd = run.forward(0)
    torch.cuda.synchronize()
    step = run.poll()
    rec = A.afd_debug_bounds(run.ctx)
    assert A.afd_debug_plant(run.ctx, 0) == A.AFD_OK
    out = {"forward": rc_fwd, "step": step, "bounds": rec[0], "site": rec[1], "index": rec[2],
           "limit": rec[3]}
    if name != "grouped":
        err, _ = G.run_and_compare_full(run)
        out["after_err"] = err
        out["after_bounds"] = A.afd_debug_bounds(run.ctx)[0]
    run.close()
    return out


def main():
    assert torch.cuda.is_available()
    A.lib()
    assert A.afd_debug_bounds(None)[0] == A.AFD_ERR_ARG, "not the debug build"
    res = {
        "clean_fanin_tc2": clean_token_form("fanin", A.AFD_GEMM_TENSOR),
        "clean_fanin_1cta": clean_token_form("fanin", A.AFD_GEMM_TENSOR_1CTA),
        "clean_fanin_simt": clean_token_form("fanin", A.AFD_GEMM_SIMT),
        "clean_token_order": clean_token_form("token_order", A.AFD_GEMM_TENSOR),
        "clean_grouped": clean_grouped(),
        "full_v2lite_prefill": clean_full_size("v2lite_prefill"),
        "full_decode": clean_full_size("decode"),
        "planted": {
            "gather_inv": planted(A.AFD_DBG_GATHER_INV, "token_order"),
            "gather_perm": planted(A.AFD_DBG_GATHER_PERM, "fanin"),
            "gather_grouped": planted(A.AFD_DBG_GATHER_GROUPED, "grouped"),
            "combine_inv": planted(A.AFD_DBG_COMBINE_INV, "fanin"),
            "scatter_inv": planted(A.AFD_DBG_SCATTER_INV, "grouped"),
            "gemm_out_tc2": planted(A.AFD_DBG_GEMM_OUT, "fanin"),
            "gemm_out_1cta": planted(A.AFD_DBG_GEMM_OUT, "fanin", A.AFD_GEMM_TENSOR_1CTA),
            "gemm_out_simt": planted(A.AFD_DBG_GEMM_OUT, "fanin", A.AFD_GEMM_SIMT),
        },
    }
    print(json.dumps(res))


if __name__ == "__main__":
    main()
