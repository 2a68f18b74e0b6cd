"""qm_apply_experts_static: the experts product for callers that cannot
allocate device memory (a plug-in inside a host program that owns all device
allocations, or a loop that must not pay cudaMalloc's implicit
synchronization). It keeps its routing tables in a 1 MiB array the library
reserves per GPU, so the caller passes only inputs and outputs.

This file is collected last on purpose: should it fail, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import packed_qmatmul_gb300 as qm
from packed_qmatmul_gb300 import synth
from wutil import bf16_half_ulp, check_product, row_norms, to_oracle


def _lib():
    from packed_qmatmul_gb300 import build

    build.build()
    return qm.load_library()


def _bf16_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


# (format, E, n, k, T, topk): the first two take the decode path in both entry
# points; the third has experts averaging over 32 positions, where
# qm_apply_experts takes the tensor cores and the static entry point does not
CASES = (("mxfp4", 8, 96, 512, 40, 2), ("affine", 5, 64, 256, 23, 3), ("q8_0", 4, 128, 256, 80, 2))


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point():
    _lib()
    torch.cuda.set_device(0)
    # calls in a row with different routing sizes: each must not see anything
    # the one before left in the shared array
    for call, (kind, E, n, k, T, topk) in enumerate(CASES):
        g = synth.rng(1300 + call)
        if kind == "mxfp4":
            w = synth.mxfp4_weight(g, n, k, lead=(E,))
        elif kind == "affine":
            w = synth.affine_weight(g, n, k, bits=4, group_size=64, lead=(E,))
        else:
            w = synth.q8_0_weight(g, n, k, lead=(E,))
        ids = synth.expert_ids(g, T, topk, E)
        ids[1, 0] = -1
        ids[T - 1, topk - 1] = E + 2
        x = synth.activations(g, T, k)
        qw = qm.QWeight.from_arrays(w)
        ids_d = torch.from_numpy(ids).cuda()
        x_d = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        y_ws = qm.apply_experts(qw, ids_d, x_d)  # the entry point with caller workspace
        y_st = torch.full_like(y_ws, float("nan"))
        qm.qm_apply_experts_static(qw, ids_d, x_d, y_st)
        torch.cuda.synchronize()
        qm.qm_device_status()
        a, b = _bf16_f64(y_st), _bf16_f64(y_ws)
        assert np.all(np.isfinite(a))
        a2, b2 = a.reshape(T * topk, n), b.reshape(T * topk, n)
        flat = ids.reshape(-1)
        inr = (flat >= 0) & (flat < E)
        assert np.all(a2[~inr] == 0)
        tensor = T * topk > 32 * E
        if not tensor:
            # the same decode path: the same bits
            assert np.array_equal(y_st.view(torch.int16).cpu().numpy(), y_ws.view(torch.int16).cpu().numpy()), call
        # the product tolerance of the parity tests, with the workspace entry
        # point's result as the reference
        xn = np.linalg.norm(x_d.float().cpu().numpy().astype(np.float64), axis=1)
        wv = qm.dequant(qw, torch.float32).cpu().numpy().astype(np.float64)
        wn = np.linalg.norm(wv, axis=-1)  # [E, n]
        bound = np.zeros((T * topk, n))
        bound[inr] = 1e-2 * xn[np.arange(T * topk)[inr] // topk][:, None] * wn[flat[inr]] / np.sqrt(k)
        assert np.all(np.abs(a2 - b2) <= bound + bf16_half_ulp(a2) + bf16_half_ulp(b2)), call
        assert np.linalg.norm(a2 - b2) <= 4e-3 * max(np.linalg.norm(b2), 1e-30)
        # and both against the oracle
        ow = to_oracle(w)
        ref = oracle.apply_experts(ow, ids, x).reshape(T * topk, n)
        rows = np.where(inr)[0]
        wr = row_norms(ow).reshape(E, n)[flat[rows]]
        for got, what in ((a2, "static"), (b2, "workspace")):
            check_product(got[rows], ref[rows], wr, xn[rows // topk], k, f"{what} call {call}")


def test_static_scratch_refuses_oversize_routing():
    # refused on the host before any device work
    lib = _lib()
    w = qm._CWeight()
    w.format, w.bits, w.group_size, w.ndim = qm.QM_MXFP4, 4, 32, 3
    w.shape[0], w.shape[1], w.shape[2] = 32, 64, 64
    w.codes, w.scales = 4096, 8192
    st = lib.qm_apply_experts_static(ctypes.byref(w), 4096, qm.QM_I32, 1 << 20, 4, 8192, 1 << 20,
                                     qm.QM_BF16, 16384, None)
    assert st == qm.QM_EINVAL
    assert lib.qm_last_error().decode().startswith("workspace:")
