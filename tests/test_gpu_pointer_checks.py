"""Host-side rejection of pointers the GPU cannot use. Only the check itself
runs here (fo_check_device_pointers enqueues nothing): device, pinned host
and managed-by-torch CUDA memory pass, pageable host memory is refused, and
the binding refuses a CPU tensor before it reaches the library."""
import numpy as np
import pytest
import torch

from ag_gemm_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    return torch.device("cuda:0")


def test_device_and_pinned_memory_pass(dev):
    d = torch.empty(1024, device=dev)
    pinned = torch.empty(1024).pin_memory()
    assert B.fo_check_device_pointers([d.data_ptr(), d[16:].data_ptr(), pinned.data_ptr()]) == B.FO_OK
    assert B.fo_check_device_pointers([]) == B.FO_OK


def test_pageable_host_memory_is_refused(dev):
    host = np.zeros(4096, dtype=np.float32)
    cpu_tensor = torch.empty(1024)
    d = torch.empty(1024, device=dev)
    assert B.fo_check_device_pointers([host.ctypes.data]) == B.FO_ERR_INVALID_ARG
    assert B.fo_check_device_pointers([d.data_ptr(), cpu_tensor.data_ptr()]) == B.FO_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors_before_the_library(dev):
    plan = B.fo_plan("gemm_rs", 2, 256, 256, 512)
    ws = torch.zeros(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    X = [torch.zeros(256, 256, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    W = [torch.zeros(256, 256, dtype=torch.bfloat16) for _ in range(2)]        # on the host: refused
    Y = [torch.empty(128, 256, device=dev) for _ in range(2)]
    with pytest.raises(ValueError):
        B.fo_gemm_rs(plan, X, W, Y, ws)
    assert B.fo_plan_last_launches(plan) == 0
