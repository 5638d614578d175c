"""Failure detection without a GPU fault: a bounded device-side wait that runs out is
reported as TSI_ERR_TIMEOUT through the device error word, and the context stays usable
(tsi_selftest_wait_timeout drives the same bounded-wait helper as the tensor-core kernels)."""
import pytest
import torch

import top_selection_indexer_gb300 as tsi
from workloads.gen import draw

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_the_context_survives(cuda_lib):
    cuda_lib.device_status()  # start from a clear error word
    cuda_lib.selftest_wait_timeout()
    with pytest.raises(tsi.TSIError) as info:
        cuda_lib.device_status()
    assert info.value.status == tsi.ERR_TIMEOUT
    cuda_lib.device_status()  # the word was cleared by the read above
    # the context still runs kernels: a small indexer call on integer inputs
    qI = draw((1, 300, 64, 128), "int8", "e4m3", 1, "cuda")
    kI = draw((1, 300, 128), "int8", "e4m3", 2, "cuda")
    w = draw((1, 300, 64), "pow2", "bf16", 3, "cuda")
    idx = cuda_lib.indexer_topk(qI, kI, w, 64)
    cuda_lib.device_status()
    assert int(idx[0, 0, 0]) == 0 and int(idx[0, 0, 1]) == -1  # row 0 holds key 0 only
    assert torch.all(idx[0, 299] >= 0)
