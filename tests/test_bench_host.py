"""Host-side pieces of bench.py that need no GPU: every workload name it
accepts resolves to a workload description, the JSON line's dtype label, and
the FLOP convention."""
import pytest

import attn_inputs
import bench


def test_every_bench_workload_exists_and_has_a_dtype_label():
    for name in bench.FWD_WORKLOADS + (bench.WORKLOAD,):
        w = attn_inputs.WORKLOADS[name]
        assert bench.dtype_label(w) in ("f16", "bf16", "f32", "e4m3+bf16", "e4m3+f16")
    for name in bench.CSR_WORKLOADS:
        w = attn_inputs.CSR_WORKLOADS[name]
        assert bench.dtype_label(w) in ("f16", "bf16", "f32")
    assert bench.dtype_label(attn_inputs.WORKLOADS["causal_fp8qk_b4_n8192"]) == "e4m3+bf16"


def test_flop_convention():
    # causal: 4 N^2 D H / 2 per sequence, four sequences of the training workload
    assert bench.attention_flops([8192] * 4, [8192] * 4, 32, 128, True) == pytest.approx(2.199023255552e12)
    # full cross attention of the Vx page's shape
    assert bench.attention_flops([8192], [2048], 1, 64, False) == pytest.approx(4.294967296e9)


def test_step_time_spread():
    assert bench.spread([3.0, 1.0, 2.0, 10.0]) == {"median": 2.5, "min": 1.0, "max": 10.0}


def test_forward_algorithmic_bytes():
    # causal N=256, H=2, D=64, fp16 q, k, v and o: three inputs read, o and f32 lse written
    assert bench.fwd_algorithmic_bytes([256], [256], 2, 64, 2, 2, 2) == 3 * 256 * 2 * 64 * 2 + 256 * 2 * 64 * 2 + 4 * 256 * 2
    # cross f32 8192 x 2048, D=64, H=1
    assert bench.fwd_algorithmic_bytes([8192], [2048], 1, 64, 4, 4, 4) == (8192 + 2 * 2048 + 8192) * 64 * 4 + 4 * 8192
    assert set(bench.SUB_WORKLOADS) <= set(bench.FWD_WORKLOADS)
