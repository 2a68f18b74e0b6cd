"""The failure path of the bounded device waits, without a fault.

Every pipeline's waits on a barrier give up after a limit of the GPU's global
timer, raise a device flag and let the kernel exit; qm_device_status() then
reports QM_ETIMEOUT. qm_check_wait_timeout runs one warp that waits on a barrier
nothing completes, with a short limit: the wait must run out, be reported once,
and leave the context usable.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import packed_qmatmul_gb300 as qm
from packed_qmatmul_gb300 import synth


def _lib():
    from packed_qmatmul_gb300 import build

    build.build()
    return qm.load_library()


@pytest.mark.gpu
def test_wait_that_runs_out_is_reported_and_cleared():
    lib = _lib()
    torch.cuda.set_device(0)
    torch.cuda.synchronize()
    assert lib.qm_device_status(None) == qm.QM_OK
    t0 = time.perf_counter()
    assert lib.qm_check_wait_timeout(50_000_000, None) == qm.QM_OK  # 50 ms, enqueued
    st = lib.qm_device_status(None)
    el = time.perf_counter() - t0
    assert st == qm.QM_ETIMEOUT, (st, lib.qm_last_error())
    assert lib.qm_last_error().decode().startswith("device:")
    assert 0.04 < el < 5.0, el  # the limit, not a hang
    assert lib.qm_device_status(None) == qm.QM_OK  # reported once, then cleared
    # the context is still usable: a product runs and checks out
    g = synth.rng(5)
    w = synth.affine_weight(g, 64, 256, bits=4, group_size=64)
    qw = qm.QWeight.from_arrays(w)
    x = torch.from_numpy(synth.activations(g, 2, 256).view(np.int16)).cuda().view(torch.bfloat16)
    y = qm.apply(qw, x)
    ref = x.float() @ qm.dequant(qw, torch.float32).T
    assert torch.allclose(y.float(), ref, rtol=2e-2, atol=2e-2)
    assert lib.qm_device_status(None) == qm.QM_OK


def test_wait_check_refuses_a_limit_out_of_range():
    lib = _lib()
    assert lib.qm_check_wait_timeout(0, None) == qm.QM_EINVAL
    assert lib.qm_last_error().decode().startswith("limit:")
    assert lib.qm_check_wait_timeout(11 * 10**9, None) == qm.QM_EINVAL
