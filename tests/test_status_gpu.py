"""Failure detection without a fault: a device wait that can never complete
ends after its bound with a status the host reads, and the context stays
usable afterwards."""
import pytest
import torch

import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert kvq.device_status() == kvq.KVQ_OK
    kvq.selftest_wait_timeout(2_000_000)  # 2 ms on an mbarrier nothing arrives at
    assert kvq.device_status() == kvq.KVQ_ERR_TIMEOUT
    assert kvq.device_status() == kvq.KVQ_OK  # read-and-clear
    kv = inputs.sweep_kv(256, 256, seed=1).cuda()
    st = kvq.kv_rotate_quant_pack(kv, 256)
    torch.cuda.synchronize()
    assert int(st.k_scales.count_nonzero()) > 0
    assert kvq.device_status() == kvq.KVQ_OK
