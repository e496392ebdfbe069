"""Host-side pieces of bench.py that need no GPU: the roofline peak taken
from the measured-peaks file, and the traffic record keyed by kernel source."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _peak(tmp_path, obj):
    p = tmp_path / "peaks.json"
    p.write_text(json.dumps(obj))
    return bench.hbm_peak(str(p))


def test_measured_hbm_peak_is_found_under_any_key_layout(tmp_path):
    assert _peak(tmp_path, {"hbm_gbs": 6779.4, "bf16_tflops": 1913.4}) == (6779.4, "measured")
    assert _peak(tmp_path, {"hbm": {"copy_gbs": 6779.4}}) == (6779.4, "measured")
    assert _peak(tmp_path, {"hbm_copy_tbs": 6.7794})[0] == 6779.4  # TB/s
    # a clock is not a bandwidth; the burst figure goes before the sustained one
    assert _peak(tmp_path, {"hbm_clock_mhz": 3996, "hbm_gbs": 6779.4})[0] == 6779.4
    assert _peak(tmp_path, {"hbm_gbs_sustained": 6500.0, "hbm_gbs_burst": 6779.4})[0] == 6779.4


def test_fallback_peak_without_a_measurement(tmp_path):
    assert _peak(tmp_path, {"bf16_tflops": 1900.0}) == (bench.FALLBACK_HBM_GBS, "fallback")
    assert bench.hbm_peak(str(tmp_path / "absent.json")) == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "bad.json").write_text("{not json")
    assert bench.hbm_peak(str(tmp_path / "bad.json"))[1] == "fallback"


def test_traffic_record_is_used_only_for_the_kernel_source_it_was_taken_on():
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    (key, val), = rec.items()
    assert key == "moe_stack_fused@stack30_b1_h2048_i768_e128_k2"
    got = bench.recorded_traffic("moe_stack_fused", "stack30_b1_h2048_i768_e128_k2")
    if val["source_hash"] == bench.kernel_source_hash():
        assert got == val["dram_bytes_per_launch"]
    else:  # kernels changed since the capture: the bench reports no traffic
        assert got is None
    # about the algorithmic 582 MB per 30-layer launch, never below it
    assert 582e6 <= val["dram_bytes_per_launch"] < 2 * 582e6
