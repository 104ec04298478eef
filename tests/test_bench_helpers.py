"""Host logic of bench.py's measurement (no GPU): which tensor peak a
roofline divides by, and when a committed ncu summary's DRAM traffic
applies to the kernel source being timed."""
import bench


PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def test_burst_peak_at_full_clock():
    v, why = bench.tensor_peak(PEAKS, "measured", {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0,
                                                   "reasons": []})
    assert v == 1900.0 and "burst" in why


def test_sustained_peak_under_power_cap_or_low_clock():
    v, _ = bench.tensor_peak(PEAKS, "measured", {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0,
                                                 "reasons": ["sw_power_cap"]})
    assert v == 1700.0
    v, _ = bench.tensor_peak(PEAKS, "measured", {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0,
                                                 "reasons": []})
    assert v == 1700.0
    # no clock record: the burst figure
    assert bench.tensor_peak(PEAKS, "measured", None)[0] == 1900.0


def test_fallback_peaks_when_a_key_is_missing():
    v, why = bench.tensor_peak({}, "fallback", {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0,
                                                "reasons": []})
    assert v == bench.FALLBACK_PEAKS["bf16_tflops"] and "fallback" in why


def test_profiled_traffic_follows_the_source(tmp_path):
    src = tmp_path / "kernel.cu"
    src.write_text("__global__ void k() {}\n")
    prof = tmp_path / "summary.txt"
    prof.write_text("# command: ncu ...\n"
                    f"source_sha256_16: {bench.source_hash(str(src))}\n"
                    "dram_bytes_per_launch: 12345\n")
    assert bench.profiled_traffic(str(prof), str(src)) == 12345.0
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.profiled_traffic(str(prof), str(src)) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.txt"), str(src)) is None
