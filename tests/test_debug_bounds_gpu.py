"""The bounds-checking debug build (-DAFD_DEBUG_BOUNDS), the memory checker's
stand-in for indices the kernels take from earlier kernels' outputs: it
matches the oracle with no failed check, and every check site reports a
planted failure (tests/debug_bounds_cases.py, run in a process of its own
that loads libafd_gb300_dbg.so).  Needs an sm_103a GPU."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from combine_peer_slot_gb300 import afd as A
from combine_peer_slot_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def debug_results():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if B.needs_build(debug=True):
        B.build(debug=True)
    env = dict(os.environ, AFD_LIBRARY=B.LIB_DBG)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_bounds_cases.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("case", ["clean_fanin_tc2", "clean_fanin_1cta", "clean_fanin_simt",
                                  "clean_token_order", "clean_grouped"])
def test_debug_build_matches_oracle_without_failed_checks(debug_results, case):
    r = debug_results[case]
    assert r["bounds"] == A.AFD_OK
    assert r["err"] <= 2e-2


@pytest.mark.parametrize("case", ["full_v2lite_prefill", "full_decode"])
def test_debug_build_full_size_without_failed_checks(debug_results, case):
    r = debug_results[case]
    assert r["step"] == A.AFD_OK
    assert r["bounds"] == A.AFD_OK


SITES = {"gather_inv": A.AFD_DBG_GATHER_INV, "gather_perm": A.AFD_DBG_GATHER_PERM,
         "gather_grouped": A.AFD_DBG_GATHER_GROUPED, "combine_inv": A.AFD_DBG_COMBINE_INV,
         "scatter_inv": A.AFD_DBG_SCATTER_INV, "gemm_out_tc2": A.AFD_DBG_GEMM_OUT,
         "gemm_out_1cta": A.AFD_DBG_GEMM_OUT, "gemm_out_simt": A.AFD_DBG_GEMM_OUT}


@pytest.mark.parametrize("name", sorted(SITES))
def test_planted_failure_is_reported_at_its_site(debug_results, name):
    r = debug_results["planted"][name]
    assert r["forward"] == A.AFD_OK          # launched; the failure shows in the step's status
    assert r["step"] == A.AFD_ERR_BOUNDS
    assert r["bounds"] == A.AFD_ERR_BOUNDS
    assert r["site"] == SITES[name]
    assert r["limit"] == 0 and r["index"] >= 0  # a valid index, refused by the planted bound
    if "after_err" in r:                        # the context recovers: a clean step matches
        assert r["after_bounds"] == A.AFD_OK
        assert r["after_err"] <= 2e-2
