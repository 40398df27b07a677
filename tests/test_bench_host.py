"""Host-side logic of bench.py and layer.py (no GPU): the launch counts the
bench claims per step, the traffic table's source check, and the
single-launch limits the layer applies against those the header states."""
import os
import re
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _ml(**kw):
    base = dict(fmt="w2", fused=True, single_launch=True, k=8, E=384, side_sms=0, cache_fp8=False, batch=64)
    base.update(kw)
    ml = types.SimpleNamespace(**base)
    ml.use_gemm = lambda T: T >= 2048 and ml.fmt in ("w2", "fp8")
    ml.mx_tensor_path = lambda: ml.fmt == "mixed"
    return ml


def test_launches_per_step_by_path():
    import bench
    assert bench.launches_per_step(_ml(), 8) == 1                       # the whole step in one launch
    assert bench.launches_per_step(_ml(), 33) == 4                      # T*k > 256: the four calls
    assert bench.launches_per_step(_ml(single_launch=False), 8) == 4    # route, permute, FC1+FC2, combine
    assert bench.launches_per_step(_ml(fused=False, single_launch=False), 8) == 7
    assert bench.launches_per_step(_ml(), 8192) == 6                    # tensor-core prefill
    assert bench.launches_per_step(_ml(fmt="mixed"), 64) == 10
    assert bench.launches_per_step(_ml(fmt="mixed", cache_fp8=True), 64) == 10
    assert bench.launches_per_step(_ml(fmt="mxfp4"), 8) == 6
    assert bench.launches_per_step(_ml(fmt="w2host", side_sms=16), 8) == 13
    assert bench.launches_per_step(_ml(fmt="fp8", E=256, batch=64), 16384) == 4 + 4 * 4


def test_traffic_entries_check_their_sources():
    import bench
    assert bench._traffic("no such workload") is None
    for name, ent in bench._TRAFFIC.items():
        for f in ent["src"]:  # every hashed source exists
            assert os.path.exists(os.path.join(ROOT, "bit_moe_expert_top_gb300", "csrc", f)), (name, f)
        t = bench._traffic(name)
        assert t is None or t == ent["bytes"]


def test_single_launch_limits_match_the_header():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    m = re.search(r"Limits: T\*k <= (\d+), k <= (\d+), E <= (\d+)", src)
    assert m, "moe_w2_decode_layer limits not found in the header"
    lay = open(os.path.join(ROOT, "bit_moe_expert_top_gb300", "layer.py")).read()
    cond = f"T * k <= {m.group(1)} and k <= {m.group(2)} and E <= {m.group(3)}"
    assert cond in lay, cond
