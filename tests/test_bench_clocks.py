"""bench.py's clock handling on the host (no GPU): the in-band clock note,
the tensor roofline beside the burst peak, and the window of nvidia-smi
samples."""
import bench


def test_tensor_peak_at_the_kernel_clock():
    peaks = {"bf16_tflops": 1808.6, "source": "measured"}
    clocks = {"sm_max_mhz": 2032.0, "kernel_sm_mhz": {"gate_up": 1300.0, "down": 1250.0}}
    peak, kind, at = bench._tensor_peak(peaks, clocks)
    assert peak == 1808.6 and "burst" in kind
    # 4096 multiply-adds per clock per SM over 148 SMs
    assert abs(at["peak_tflops"] - 2 * 4096 * 148 * 1300e6 / 1e12) < 1e-9
    assert at["sm_mhz"] == 1300.0
    _, _, at2 = bench._tensor_peak(peaks, clocks, slot="down")
    assert at2["sm_mhz"] == 1250.0
    # e4m3: twice both figures
    peak8, _, at8 = bench._tensor_peak(peaks, clocks, fp8=True)
    assert peak8 == 2 * 1808.6 and abs(at8["peak_tflops"] - 2 * at["peak_tflops"]) < 1e-9
    # no in-band record: nothing beside the burst figure
    assert bench._tensor_peak(peaks, {"sm_max_mhz": 2032.0})[2] is None
    assert bench._tensor_peak(peaks, None)[2] is None


def test_inband_cap_note():
    c = {"sm_max_mhz": 2032.0, "kernel_sm_mhz": {"gate_up": 1300.0, "down": 1320.0}}
    bench._note_inband_cap(c)
    assert "1300-1320 MHz" in c["inband_below_max"]
    c = {"sm_max_mhz": 2032.0, "kernel_sm_mhz": {"gate_up": 2000.0}}
    bench._note_inband_cap(c)
    assert "inband_below_max" not in c
    c = {"sm_max_mhz": 2032.0, "kernel_sm_mhz": {}}
    bench._note_inband_cap(c)
    assert "inband_below_max" not in c


def test_sampler_window_reaches_past_the_timed_region():
    """nvidia-smi reports a clock change about 0.1 s late, so the window of
    samples taken into the record extends SMI_LAG_S past its end."""
    assert 0.1 <= bench.SMI_LAG_S <= 0.3
