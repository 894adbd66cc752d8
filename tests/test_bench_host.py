"""Host-side logic of bench.py: the clock record that decides whether a timed run is
kept, the kernel-family names, the choice of the dominant kernel, and that every
stored DRAM-traffic figure names a kernel the library times and a workload it has."""
import bench
from head_latent_attention_rmsnorm_gb300 import configs, mla


def test_clock_summary_decodes_event_reasons():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.ok, cs.max_mhz = True, 2070
    cs.samples = [(2070, 0x4), (2070, 0x0), (1980, 0x8 | 0x4), (2055, 0x20), (2070, 0x40)]
    s = cs.summary()
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["samples"] == 5
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_clock_summary_without_nvml():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.ok, cs.max_mhz, cs.samples = False, None, []
    s = cs.summary()
    assert s["sm_mhz"] is None and s["reasons"] == [] and s["samples"] == 0


def test_path_names():
    assert bench.path_name(mla.PATH_SIMT) == "simt"
    assert bench.path_name(mla.PATH_TC) == "tcgen05"
    assert bench.path_name(mla.PATH_TC_FUSED) == "tcgen05 fused"
    assert bench.path_name(mla.PATH_NONE) == "?"


def test_dominant_kernel_is_the_largest_candidate_present():
    prof = {"prep": (55, 0.87), "tc_gemm": (55, 1.20), "tc_attn": (55, 4.18)}
    assert bench.dominant(prof, ("tc_attn", "attn_simt")) == "tc_attn"
    assert bench.dominant(prof, ("tc_gemm", "prep")) == "tc_gemm"
    assert bench.dominant(prof, ("attn_simt",)) is None


def test_traffic_table_names_timed_kernels_and_known_workloads():
    for kern, workload, _ in bench.NCU_TRAFFIC:
        assert kern in mla.KERNELS, kern
        assert workload in configs.ALL, workload
    assert bench.HEADLINE in configs.ALL


def test_every_profiled_launch_has_a_reported_name():
    """Each launch site's profiling scope names a kernel family that the per-kernel
    breakdown reports, so no launch drops out of it."""
    import glob
    import os
    import re
    csrc = os.path.join(os.path.dirname(mla.__file__), "csrc")
    names = set()
    for f in glob.glob(os.path.join(csrc, "*.cu")):
        names |= set(re.findall(r'ProfScope \w+\("(\w+)"', open(f).read()))
    assert len(names) > 10
    assert names <= set(mla.KERNELS), names - set(mla.KERNELS)


def test_header_lists_the_profiled_names():
    """include/mla.h documents the names mla_profile_kernel answers to; they are the
    binding's and the launch sites'."""
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mla.h")).read()
    block = hdr[hdr.index("Names:"):hdr.index("mla_profile_reset:")]
    assert set(re.findall(r'"(\w+)"', block)) == set(mla.KERNELS)
