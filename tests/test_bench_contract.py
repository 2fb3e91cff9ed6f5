"""Host-side bookkeeping of bench.py that the JSON line depends on (no GPU)."""
import os
import sys
from types import SimpleNamespace

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_step_flop_is_the_layers_gemm_flop():
    L, M = bench.LIN, bench.MOE
    assert bench.STEP_FLOP == 6 * L["M"] * L["N"] * L["K"] + 6 * M["T"] * M["N"] * M["K"]


def test_launch_count_per_step():
    """Dense layer: 2 dual quants + GEMM (fwd), dual quant + GEMM (dX), GEMM
    (dW) in saved-quant mode, two more row/column quants in recompute mode;
    MoE: 2 grouped dual quants + weight dual quant + 3 GEMMs; MXFP4: QDQ +
    packed quant."""
    m = SimpleNamespace(SAVE_QUANT=0, RECOMPUTE=1)
    assert bench.Workload.launches(SimpleNamespace(m=m, mode=0)) == 6 + 6 + 2
    assert bench.Workload.launches(SimpleNamespace(m=m, mode=1)) == 8 + 6 + 2


def test_traffic_is_reported_only_for_the_measured_gemm_source():
    kinds = {"linear_dw_gemm": [0.0, 10], "moe_fwd_gemm": [0.0, 10], "moe_dx_gemm": [0.0, 10],
             "moe_dw_gemm": [0.0, 10]}
    rec = bench.GEMM_DRAM_TRAFFIC.get(bench.gemm_source_hash())
    if rec is None:  # the kernel changed since the counters were taken: no traffic claim
        assert bench.gemm_traffic(kinds) is None
    else:
        assert bench.gemm_traffic(kinds) == sum(rec.values()) / 4
    assert bench.gemm_traffic({"unmeasured_gemm": [0.0, 1]}) is None
