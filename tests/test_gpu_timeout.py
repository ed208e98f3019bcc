"""The device-side timeout path of the tensor-core write kernels.  With the test hook
armed (rkv_debug_wait_fault), a barrier wait of the W_c3 kernel runs out: the second
CTA of every pair leaves one stage's loads out, so its leader's full barrier never
completes, and every wait is limited to 2e5 cycles.  The kernel must report
RKV_ERR_DEVICE_TIMEOUT in the status word, drain what it issued, free its tensor
memory and return; the next calls on the same context must succeed and reproduce
the records of the call before the fault bit for bit."""
import numpy as np
import pytest
import torch

import rkv_workload as wl
from reference_residual_kv_gb300 import rkv

from _gpu_common import gen_inputs, host_records, run_gpu

pytestmark = pytest.mark.gpu


def test_wait_expiry_reports_timeout_and_context_survives():
    cfg = wl.CONFIGS["llama3.1-8b-kv"].replace(L=1, T=512, N=2, D=64, d_ff=256, d_c=64)
    kv, w = gen_inputs(cfg)
    bufs, (kv_d, W1, W2, W3) = run_gpu(cfg, kv, w)
    assert bufs.device_status() == 0
    before = host_records(cfg, bufs)

    rkv.rkv_debug_wait_fault(200_000, 0)
    bufs.compress(kv_d, W1, W2, W3)          # the launch itself succeeds
    torch.cuda.synchronize()
    assert bufs.device_status() == rkv.RKV_ERR_DEVICE_TIMEOUT

    for _ in range(2):                       # the hook was one-shot
        bufs.status.zero_()
        bufs.compress(kv_d, W1, W2, W3)
        torch.cuda.synchronize()
        assert bufs.device_status() == 0
        after = host_records(cfg, bufs)
        for key in ("idx", "q", "hdr", "z"):
            assert np.array_equal(after[key], before[key]), key
