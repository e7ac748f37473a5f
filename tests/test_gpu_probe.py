"""The FP32 pipe probe (sgemm_f32_fma_probe): argument checks, and a measured rate that lies
between half and 105% of the derived peak (SMs x 128 FP32 lanes x 2 FLOP x the GPU's
maximum SM clock), the figure the GEMM kernels are held against."""
import ctypes

import pytest
import torch

import dense_fp32_matrix_08_gb300 as sg

pytestmark = pytest.mark.gpu


def _max_sm_mhz():
    import subprocess
    out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits",
                          "-i", "0"], capture_output=True, text=True, timeout=60)
    return float(out.stdout.strip().splitlines()[0])


def test_probe_arguments():
    t, ms = ctypes.c_double(0.0), ctypes.c_float(0.0)
    assert sg.lib.sgemm_f32_fma_probe(0, 1, ctypes.byref(t), ctypes.byref(ms)) == -1
    assert sg.lib.sgemm_f32_fma_probe((1 << 24) + 1, 1, ctypes.byref(t), ctypes.byref(ms)) == -1
    assert sg.lib.sgemm_f32_fma_probe(16, 0, ctypes.byref(t), ctypes.byref(ms)) == -2
    assert sg.lib.sgemm_f32_fma_probe(16, 101, ctypes.byref(t), ctypes.byref(ms)) == -2
    assert sg.lib.sgemm_f32_fma_probe(16, 1, None, ctypes.byref(ms)) == -3
    assert sg.lib.sgemm_f32_fma_probe(16, 1, ctypes.byref(t), None) == 0  # ms is optional


def test_probe_rate_against_derived_peak():
    r = sg.sgemm_f32_fma_probe(1 << 16, 3)
    assert r["status"] == 0
    props = torch.cuda.get_device_properties(0)
    derived = props.multi_processor_count * 128 * 2 * _max_sm_mhz() * 1e6 / 1e12
    assert r["ms"] > 0
    assert 0.5 * derived < r["tflops"] <= 1.05 * derived, (r, derived)
