"""The C boundary on the host: the library loads, exports what include/qm.h
declares, and refuses bad arguments naming the part -- all without a GPU
(every case here fails validation before any CUDA call)."""
import ctypes
import os
import re

import pytest

import packed_qmatmul_gb300 as qm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from packed_qmatmul_gb300 import build

    build.build()
    return qm.load_library()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^\s*(?:qm_status|size_t|const char\*|int32_t)\s+(qm_\w+)\s*\(",
                                    text, re.M))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"qm_dequant", "qm_apply", "qm_take", "qm_apply_experts", "qm_experts_route",
            "qm_apply_experts_workspace", "qm_experts_route_workspace", "qm_device_status", "qm_last_error"} <= names
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert lib.qm_version() >= 100


def _w(fmt=qm.QM_AFFINE, bits=4, gs=64, shape=(16, 64), codes=256, scales=512, biases=768, ndim=2, flags=0):
    w = qm._CWeight()
    w.format, w.bits, w.group_size, w.scale_dtype, w.ndim = fmt, bits, gs, qm.QM_BF16, ndim
    for i, s in enumerate(shape):
        w.shape[i] = s
    w.codes, w.scales, w.biases = codes, scales, biases
    w.flags = flags
    return w


def _dequant_err(lib, w, out=1024, dt=qm.QM_BF16):
    st = lib.qm_dequant(ctypes.byref(w), dt, out, None)
    return st, lib.qm_last_error().decode()


@pytest.mark.parametrize("mut,part", [
    (dict(shape=(16, 48)), "codes"),          # k not a multiple of 32
    (dict(bits=7), "w"),                      # affine widths are 2, 3, 4, 5, 6 and 8
    (dict(gs=16), "w"),
    (dict(shape=(16, 96), gs=64), "scales"),  # k not a multiple of group_size
    (dict(codes=0), "codes"),
    (dict(codes=264), "codes"),                # misaligned
    (dict(scales=0), "scales"),
    (dict(biases=8), "biases"),
    (dict(fmt=7), "w"),
    (dict(ndim=1), "w"),
    (dict(flags=2), "w"),                      # no such flag
    (dict(fmt=qm.QM_Q8_0, bits=0, gs=0), "scales"),  # Q8_0 takes no scales part
    (dict(fmt=qm.QM_MXFP4, bits=0, gs=0, scales=512), "biases"),
])
def test_invalid_weights_name_the_part(lib, mut, part):
    st, msg = _dequant_err(lib, _w(**mut))
    assert st == qm.QM_EINVAL
    assert msg.startswith(part + ":"), msg


def test_invalid_output(lib):
    st, msg = _dequant_err(lib, _w(), out=0)
    assert st == qm.QM_EINVAL and msg.startswith("out:")
    st, msg = _dequant_err(lib, _w(), dt=9)
    assert st == qm.QM_EINVAL and msg.startswith("out:")


def test_empty_weight_is_ok(lib):
    st, _ = _dequant_err(lib, _w(shape=(0, 64), codes=0, scales=0, biases=0), out=0)
    assert st == qm.QM_OK


def test_take_axis_rules(lib):
    w = _w(shape=(3, 16, 64), ndim=3)
    for axis, ok in ((2, False), (-1, False), (3, False), (-4, False)):
        st = lib.qm_take(ctypes.byref(w), axis, 4096, qm.QM_I32, 4, 2048, 2304, 2560, qm.QM_BF16,
                         None, None)
        assert st == qm.QM_EINVAL and lib.qm_last_error().decode().startswith("axis:")


def test_take_needs_an_output(lib):
    st = lib.qm_take(ctypes.byref(_w()), 0, 4096, qm.QM_I32, 4, None, None, None, qm.QM_BF16, None,
                     None)
    assert st == qm.QM_EINVAL and lib.qm_last_error().decode().startswith("out:")


def test_apply_validation(lib):
    w = _w()
    st = lib.qm_apply(ctypes.byref(w), 4096, 1, qm.QM_F16, 8192, None)
    assert st == qm.QM_ENOTSUP and lib.qm_last_error().decode().startswith("x:")
    st = lib.qm_apply(ctypes.byref(w), 4096, -1, qm.QM_BF16, 8192, None)
    assert st == qm.QM_EINVAL
    st = lib.qm_apply(ctypes.byref(w), 4096, 0, qm.QM_BF16, 8192, None)  # M = 0: nothing to do
    assert st == qm.QM_OK
    w3 = _w(shape=(2, 16, 64), ndim=3)
    st = lib.qm_apply(ctypes.byref(w3), 4096, 1, qm.QM_BF16, 8192, None)
    assert st == qm.QM_ENOTSUP and lib.qm_last_error().decode().startswith("w:")


def test_experts_validation(lib):
    w2 = _w()
    st = lib.qm_apply_experts(ctypes.byref(w2), 4096, qm.QM_I32, 4, 2, 8192, 4, qm.QM_BF16, 16384,
                              32768, 1 << 20, None)
    assert st == qm.QM_EINVAL and lib.qm_last_error().decode().startswith("w:")
    w3 = _w(shape=(4, 16, 64), ndim=3)
    st = lib.qm_apply_experts(ctypes.byref(w3), 4096, qm.QM_I32, 4, 2, 8192, 5, qm.QM_BF16, 16384,
                              32768, 1 << 20, None)
    assert st == qm.QM_EINVAL and lib.qm_last_error().decode().startswith("x:")
    st = lib.qm_apply_experts(ctypes.byref(w3), 4096, qm.QM_I32, 4, 2, 8192, 4, qm.QM_BF16, 16384,
                              32768, 16, None)
    assert st == qm.QM_EINVAL and lib.qm_last_error().decode().startswith("workspace:")


@pytest.mark.parametrize("T,topk", [(1 << 20, 1 << 12), (3, (1 << 62)), ((1 << 31), 1)])
def test_experts_refuse_positions_past_int32(lib, T, topk):
    # routing stores positions as int32: T*topk past 2^31-1 is refused before
    # anything multiplies them (a wrapped product would index out of bounds)
    w3 = _w(shape=(4, 16, 64), ndim=3)
    st = lib.qm_apply_experts(ctypes.byref(w3), 4096, qm.QM_I32, T, topk, 8192, T, qm.QM_BF16, 16384,
                              32768, 1 << 40, None)
    assert st == qm.QM_EINVAL and lib.qm_last_error().decode().startswith("ids:"), lib.qm_last_error()
    st = lib.qm_apply_experts_static(ctypes.byref(w3), 4096, qm.QM_I32, T, topk, 8192, T, qm.QM_BF16,
                                     16384, None)
    assert st == qm.QM_EINVAL and lib.qm_last_error().decode().startswith("ids:"), lib.qm_last_error()
    assert lib.qm_apply_experts_workspace(ctypes.byref(w3), T, topk) == 0


def test_route_refuses_positions_past_int32(lib):
    st = lib.qm_experts_route(4096, qm.QM_I32, 1 << 31, 8, 8192, 8192, 8192, 16384, 1 << 40, None)
    assert st == qm.QM_EINVAL and lib.qm_last_error().decode().startswith("ids:")


def test_workspace_query(lib):
    w3 = _w(fmt=qm.QM_MXFP4, bits=0, gs=0, shape=(32, 5760, 2880), ndim=3, biases=0)
    assert lib.qm_apply_experts_workspace(ctypes.byref(w3), 0, 4) == 0
    a = lib.qm_apply_experts_workspace(ctypes.byref(w3), 64, 4)
    b = lib.qm_apply_experts_workspace(ctypes.byref(w3), 4096, 4)
    assert 0 < a < b and a % 256 == 0 and b % 256 == 0
    assert a < 4096 * 4 * 2880 * 2 <= b  # many positions per expert: routed rows of x too
    bad = _w(shape=(16, 64))  # not a stack of experts
    assert lib.qm_apply_experts_workspace(ctypes.byref(bad), 64, 4) == 0
    assert lib.qm_experts_route_workspace(0, 32) == 0
    r = lib.qm_experts_route_workspace(256, 32)
    assert 0 < r <= a and r % 256 == 0


def test_descriptor_follows_assigned_parts():
    # the binding builds the descriptor once and rebuilds it when a field is
    # assigned: the library must always see the current tensors' addresses
    import torch

    codes = torch.zeros((16, 32), dtype=torch.int32)
    scales = torch.zeros((16, 4), dtype=torch.int16)
    biases = torch.zeros((16, 4), dtype=torch.int16)
    w = qm.QWeight("affine", (16, 256), codes, scales, biases, bits=4, group_size=64)
    first = w._ref()
    assert w._ref() is first  # cached between calls
    d = first._obj
    assert (d.codes, d.scales, d.biases) == (codes.data_ptr(), scales.data_ptr(), biases.data_ptr())
    assert (d.format, d.bits, d.group_size, d.ndim, d.shape[0], d.shape[1]) == (qm.QM_AFFINE, 4, 64, 2, 16, 256)
    other = torch.zeros_like(codes)
    w.codes = other
    d2 = w._ref()._obj
    assert d2.codes == other.data_ptr() and d2.scales == scales.data_ptr()
    w.flags = qm.QM_WEIGHT_STATIC
    assert w._ref()._obj.flags == qm.QM_WEIGHT_STATIC


def test_empty_inputs_return_ok_without_work(lib):
    # nothing to compute: every entry point accepts it before touching a pointer
    w = _w(shape=(16, 64))
    assert lib.qm_take(ctypes.byref(w), 0, None, qm.QM_I32, 0, 2048, 2304, 2560, qm.QM_BF16, None, None) == qm.QM_OK
    assert lib.qm_take(ctypes.byref(w), 0, None, qm.QM_I64, 0, None, None, None, qm.QM_BF16, 4096, None) == qm.QM_OK
    w3 = _w(shape=(4, 16, 64), ndim=3)
    for T, topk in ((0, 4), (8, 0)):
        st = lib.qm_apply_experts(ctypes.byref(w3), None, qm.QM_I32, T, topk, None, T, qm.QM_BF16, None,
                                  None, 0, None)
        assert st == qm.QM_OK, (T, topk, lib.qm_last_error())
    assert lib.qm_apply(ctypes.byref(_w(shape=(0, 64), codes=0, scales=0, biases=0)), 4096, 3, qm.QM_BF16,
                        8192, None) == qm.QM_OK  # n = 0
    # a negative count is refused, naming ids
    st = lib.qm_take(ctypes.byref(w), 0, 4096, qm.QM_I32, -1, 2048, 2304, 2560, qm.QM_BF16, None, None)
    assert st == qm.QM_EINVAL and lib.qm_last_error().decode().startswith("ids:")


def test_mxfp4_blocks_validation(lib):
    # MXFP4 in GGUF's blocks: one part, [.., n, k/32*17]; scales and biases refused
    def err(**kw):
        base = dict(fmt=qm.QM_MXFP4_BLOCKS, bits=0, gs=0, shape=(16, 64), scales=0, biases=0)
        base.update(kw)
        st, msg = _dequant_err(lib, _w(**base))
        return st, msg

    for kw, part in ((dict(scales=512), "scales"), (dict(biases=768), "biases"), (dict(bits=8), "w"),
                     (dict(gs=64), "w"), (dict(shape=(16, 48)), "codes"), (dict(codes=8), "codes")):
        st, msg = err(**kw)
        assert st == qm.QM_EINVAL and msg.startswith(part + ":"), (kw, msg)
    w3 = _w(fmt=qm.QM_MXFP4_BLOCKS, bits=0, gs=0, shape=(32, 5760, 2880), ndim=3, scales=0, biases=0)
    ws = lib.qm_apply_experts_workspace(ctypes.byref(w3), 64, 4)
    assert 0 < ws == lib.qm_experts_route_workspace(256, 32)  # plain kernels: routing tables only
    qw = qm.QWeight("mxfp4_blocks", (3, 16, 64), None)
    assert qw.part_shapes((3, 5)) == ((3, 5, 34), None, None)


def test_quantize_q8_0_validation(lib):
    def err(*args):
        st = lib.qm_quantize_q8_0(*args)
        return st, lib.qm_last_error().decode()
    st, msg = err(4096, 7, 4, 64, 8192, None)
    assert st == qm.QM_EINVAL and msg.startswith("x:")
    st, msg = err(4096, qm.QM_F32, 4, 48, 8192, None)
    assert st == qm.QM_EINVAL and msg.startswith("x:")
    st, msg = err(4100, qm.QM_F32, 4, 64, 8192, None)
    assert st == qm.QM_EINVAL and msg.startswith("x:")
    st, msg = err(4096, qm.QM_F32, 4, 64, 8194, None)
    assert st == qm.QM_EINVAL and msg.startswith("out:")
    st, msg = err(4096, qm.QM_F32, 4, 64, 4096 + 512, None)  # the blocks would overwrite x
    assert st == qm.QM_EINVAL and msg.startswith("out:")
    assert lib.qm_quantize_q8_0(None, qm.QM_F32, 0, 64, None, None) == qm.QM_OK  # nothing to do


def _many(lib, ws, x, M, ys, dt=qm.QM_BF16):
    warr = (ctypes.POINTER(qm._CWeight) * max(len(ws), 1))(*[ctypes.pointer(w) for w in ws])
    yarr = (ctypes.c_void_p * max(len(ys), 1))(*ys)
    st = lib.qm_apply_many(warr, len(ws), x, M, dt, yarr, None)
    return st, lib.qm_last_error().decode()


def test_apply_many_validation(lib):
    a, b = _w(), _w(shape=(32, 64), codes=1024, scales=2048, biases=3072)
    # counts outside 1 .. QM_MAX_MANY
    assert _many(lib, [], 4096, 1, [])[0] == qm.QM_EINVAL
    st, msg = _many(lib, [a] * (qm.QM_MAX_MANY + 1), 4096, 1, [8192 + 256 * i for i in range(9)])
    assert st == qm.QM_EINVAL and msg.startswith("count:")
    # a bad weight is named by its index and part
    st, msg = _many(lib, [a, _w(codes=0)], 4096, 1, [8192, 9216])
    assert st == qm.QM_EINVAL and msg.startswith("ws[1]: codes"), msg
    # weights must share format, widths and k
    st, msg = _many(lib, [a, _w(bits=8)], 4096, 1, [8192, 9216])
    assert st == qm.QM_EINVAL and msg.startswith("ws[1]:") and "bits" in msg, msg
    st, msg = _many(lib, [a, _w(shape=(16, 128))], 4096, 1, [8192, 9216])
    assert st == qm.QM_EINVAL and msg.startswith("ws[1]: k"), msg
    # outputs: present, aligned, apart from x and from each other
    st, msg = _many(lib, [a, b], 4096, 1, [8192, 0])
    assert st == qm.QM_EINVAL and msg.startswith("ys[1]: NULL"), msg
    st, msg = _many(lib, [a, b], 4096, 1, [8192, 9224])
    assert st == qm.QM_EINVAL and msg.startswith("ys[1]:") and "aligned" in msg, msg
    st, msg = _many(lib, [a, b], 4096, 1, [8192, 8208])  # ys[0] is 32 bytes long
    assert st == qm.QM_EINVAL and msg == "ys[1]: overlaps ys[0]", msg
    st, msg = _many(lib, [a, b], 4096, 1, [4160, 9216])  # x is 128 bytes long
    assert st == qm.QM_EINVAL and msg == "ys[0]: overlaps x", msg
    # activations are bfloat16; M = 0 does nothing
    assert _many(lib, [a, b], 4096, 1, [8192, 9216], dt=qm.QM_F16)[0] == qm.QM_ENOTSUP
    assert _many(lib, [a, b], 4096, -1, [8192, 9216])[0] == qm.QM_EINVAL
    assert _many(lib, [a, b], 4096, 0, [8192, 9216])[0] == qm.QM_OK
