"""bench.py host logic without a GPU: every workload is named in the seed and
dtype tables, carries what the timing, roofline, e2e and oracle legs read, and
a tensor-bound workload states the peak ratio of its own dtype."""
import bench


NEEDED = ["name", "unit", "bound", "default_steps", "kernel", "launches_per_step", "kernel_launches",
          "oracle_grain", "config", "setup", "step", "kernel_only", "e2e_step", "flops_per_step",
          "units_per_step", "kernel_units", "oracle_prepare", "oracle_step", "oracle_units",
          "oracle_sample_text"]


def test_every_workload_is_complete():
    for key, cls in bench.WORKLOADS.items():
        assert key in bench.SEEDS and key in bench.DTYPES, key
        wl = cls()
        for attr in NEEDED:
            assert hasattr(wl, attr), (key, attr)
        assert wl.bound in ("hbm", "tensor")
        assert wl.unit == ("GB/s" if wl.bound == "hbm" else "TFLOP/s")


def test_tensor_peaks_take_the_library_gemm_of_their_dtype():
    """The roofline peak of a tensor-bound workload is a library GEMM of its
    own operand type; the fallback is the nominal ratio of that type."""
    assert getattr(bench.Prefill(), "tensor_fmt", "nvfp4") == "nvfp4"
    assert bench.Fp8Blockwise().tensor_fmt == bench.W4a8().tensor_fmt == "fp8"
    assert bench.peak_text(bench.Prefill()) == "bf16_tflops_sustained x 6 (nominal FP4:BF16)"
    assert bench.peak_text(bench.Fp8Blockwise()) == "bf16_tflops_sustained x 2 (nominal FP8:BF16)"
    assert bench.peak_text(bench.W4a8()) == "bf16_tflops_sustained x 2 (nominal FP8:BF16)"


def test_library_peak_reports_a_missing_path():
    """Without a GPU the library GEMM cannot run: the peak is None with the
    reason, so the roofline falls back to the nominal ratio."""
    burst, sustained, why = bench.library_peak("nvfp4", "cpu", n=256, reps=1, seconds=0.01)
    assert burst is None and sustained is None and "unavailable" in why


def test_quantize_counts_one_read_of_x():
    wl = bench.QuantizeNvfp4()
    assert wl.units_per_step() == 8192 * 8192 * 2 + 8192 * 8192 // 2 + 8192 * 8192 // 16


def test_fp8_workloads_measure_flops_of_the_full_shape():
    for cls in (bench.Fp8Blockwise, bench.W4a8):
        wl = cls()
        wl.M, wl.N, wl.K = 8192, 28672, 8192
        assert wl.flops_per_step() == 2.0 * 8192 * 28672 * 8192
        assert wl.units_per_step() == wl.kernel_units() == wl.flops_per_step()
        assert wl.launches_per_step == 2 and wl.kernel_launches == 1
