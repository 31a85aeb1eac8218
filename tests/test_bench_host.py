"""Host-side logic of bench.py that needs no GPU: the FLOP conventions, the
list of workload shapes timed in the `workloads` object, and the sources that
key the committed DRAM figures."""
import os

import bench
from synthetic_inputs import WORKLOADS


def test_backward_summary_both_conventions():
    # B=2 H=16 N=4096 D=128 causal: 7 GEMMs = 481.0 GFLOP, 5 GEMMs = 343.6 GFLOP
    s = bench.backward_summary(0.2, 0.25, 2, 16, 4096, 128, True, peak=1000.0)
    assert abs(s["ms"] - 0.45) < 1e-12
    assert abs(s["tflops_7gemm"] - 14 * 2 * 16 * 4096 ** 2 * 128 / 2 / 0.45e-3 / 1e12) < 1e-9
    assert abs(s["tflops_5gemm"] / s["tflops_7gemm"] - 5 / 7) < 1e-12
    assert abs(s["frac_5gemm"] - s["tflops_5gemm"] / 1000.0) < 1e-12
    # the split is the sum of the two kernels' work
    kf = bench.kernel_flops(2, 16, 4096, 128, True)
    assert abs(kf["bwd_dq"] + kf["bwd_dkdv"] - bench.backward_flops(2, 16, 4096, 128, True)["7gemm"]) < 1


def test_workload_keys_cover_every_shape_and_mask():
    keys = bench.workload_keys()
    names = {k for k, _, _ in keys}
    assert len(names) == len(keys)  # unique
    assert len(keys) == sum(len(w.causal) for w in WORKLOADS.values())
    assert "fwd_bf16_b4h16n2048d128_causal" in names and "fwd_bf16_b4h16n2048d128_noncausal" in names
    assert "bwd_bf16_b2h16n4096d128_causal" in names
    assert "fwdbwd_bf16_b1h32n32768d64_causal" in names


def test_kernel_sources_exist():
    for kn in ("fwd", "bwd_dq", "bwd_dkdv", "bwd_atomic"):
        for D in (64, 128, 192, 256):
            for p in bench.kernel_sources(kn, D):
                assert os.path.exists(os.path.join(bench.ROOT, p)), p
    assert any(p.endswith("fwd_f32.cu") for p in bench.kernel_sources("fwd", 64, "f32"))
    assert any(p.endswith("bwd_dq_k128.cu") for p in bench.kernel_sources("bwd_dq", 64))
