"""sgemm_f32_cluster_capacity: the cluster capacities the planner decides with.

For the configurations whose shared memory holds a partial tile, clusters of 2 to 8 CTAs
must fit a whole number of clusters, at most the CTAs the SMs hold unclustered; the cluster
thin kernels report clusters of 1, 2, 4 and 8 only; configurations that cannot finish a
split in a cluster report 0.
"""
import ctypes

import pytest
import torch

import dense_fp32_matrix_08_gb300 as sg

pytestmark = pytest.mark.gpu


def test_arguments():
    n = ctypes.c_int(-5)
    assert sg.lib.sgemm_f32_cluster_capacity(-1, 2, ctypes.byref(n)) == -1
    assert sg.lib.sgemm_f32_cluster_capacity(sg.sgemm_f32_num_variants(), 2, ctypes.byref(n)) == -1
    assert sg.lib.sgemm_f32_cluster_capacity(35, 0, ctypes.byref(n)) == -2
    assert sg.lib.sgemm_f32_cluster_capacity(35, 9, ctypes.byref(n)) == -2
    assert sg.lib.sgemm_f32_cluster_capacity(35, 2, None) == -3


def test_gemm_configurations():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for v, per_sm in ((35, 3), (39, 4), (32, 4), (2, 4)):
        assert sg.sgemm_f32_cluster_capacity(v, 1) == (0, 0)
        for cl in range(2, 9):
            rc, ctas = sg.sgemm_f32_cluster_capacity(v, cl)
            assert rc == 0
            assert 0 < ctas <= sms * per_sm and ctas % cl == 0, (v, cl, ctas)
    # a 128 x 256 tile does not fit the shared memory of its own K ring: never clustered
    for cl in range(1, 9):
        assert sg.sgemm_f32_cluster_capacity(0, cl) == (0, 0)


def test_thin_cluster_kernels():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for v in (43, 44):
        for cl in (1, 2, 4, 8):
            rc, ctas = sg.sgemm_f32_cluster_capacity(v, cl)
            assert rc == 0 and 0 < ctas <= sms and ctas % cl == 0, (v, cl, ctas)
        for cl in (3, 5, 6, 7):
            assert sg.sgemm_f32_cluster_capacity(v, cl) == (0, 0)
