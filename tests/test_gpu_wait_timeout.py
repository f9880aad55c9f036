"""The bounded-wait error path on the GPU, without a fault or a hang.

The kernels wait for their bulk copies on mbarriers, each wait bounded; a wait
that runs out sets TQ_DEVERR_TIMEOUT and the kernel returns. Here one thread
waits on an mbarrier nothing arrives on (`tq_selftest_wait_timeout`), so the
wait runs out by its deadline: the status bit must reach the host through
`tq_device_error`, be cleared by that read, and the device must stay usable
(a decode after it matches the oracle).
"""
import time

import numpy as np
import pytest
import torch

import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import GpuCase, compare_decode, oracle_decode, raw_kv, to_f32_np

pytestmark = pytest.mark.gpu

TQ_DEVERR_TIMEOUT = 8


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def test_wait_runs_out_reports_and_device_stays_usable():
    tq.tq_device_error()   # start from a clear word
    t0 = time.perf_counter()
    tq.tq_selftest_wait_timeout(0.05)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert tq.tq_device_error() & TQ_DEVERR_TIMEOUT
    assert 0.04 <= elapsed < 5.0, elapsed     # the deadline, not an endless wait
    assert tq.tq_device_error() == 0          # the read cleared it
    # a decode on the same device afterwards
    kspec, vspec = wl._spec("prod", 3, 21), wl._spec("mse", 3, 22)
    w = wl.Workload("after_timeout", 1, 1, 2, 16, 128, (700,), 2, torch.bfloat16, 1.0, 5, kspec, vspec,
                    block_tokens=128, shuffle_blocks=False, append_per_step=0, prefill_chunk=1024)
    case = GpuCase(w, layers=[0])
    case.prefill()
    q = wl.queries(w, 0, 0, "cuda")
    out = to_f32_np(case.decode(0, q))
    assert tq.tq_device_error() == 0
    K, V = raw_kv(w, 0, 0, 700, "cuda")
    qn = to_f32_np(q).astype(np.float64)
    for h in range(2):
        compare_decode(out[0, h * 8:(h + 1) * 8], oracle_decode(w, K[h], V[h], qn[0, h * 8:(h + 1) * 8]))


def test_wait_timeout_argument_range():
    for s in (0.0, -1.0, 1.5, float("nan")):
        with pytest.raises(tq.TQError):
            tq.tq_selftest_wait_timeout(s)
