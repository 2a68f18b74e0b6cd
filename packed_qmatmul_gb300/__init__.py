"""GB300-native weight-only quantized products over packed block formats.

A thin ctypes binding over libqm (include/qm.h). Every function marshals its
arguments and calls the C entry point of the same name; every step of the
work runs in the library's CUDA kernels. PyTorch supplies device memory and
the current stream. There is no CPU fallback: if libqm.so is missing or fails
to load, the first call raises.

Formats (see include/qm.h): MLX affine (uint32 codes + per-group scales and
biases), GGUF Q8_0 (34-byte blocks of 32 values) and MXFP4 (e2m1 codes, two
per byte, plus e8m0 scales per 32 values).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

__all__ = [
    "QM_AFFINE", "QM_Q8_0", "QM_MXFP4", "QM_MXFP4_BLOCKS", "QM_Q4_K", "QM_Q6_K", "QM_WEIGHT_STATIC", "QM_F32", "QM_BF16", "QM_F16", "QM_I32", "QM_I64",
    "QMError", "QWeight", "library_path", "load_library",
    "qm_dequant", "qm_quantize_q8_0", "qm_apply", "qm_apply_many", "qm_take", "qm_apply_experts", "qm_apply_experts_workspace",
    "qm_experts_route_workspace",
    "qm_experts_route", "qm_apply_experts_static", "qm_check_wait_timeout", "qm_device_status", "qm_last_error",
    "qm_version",
    "dequant", "quantize_q8_0", "apply", "apply_many", "take", "apply_experts", "route",
]

QM_OK, QM_EINVAL, QM_ECUDA, QM_ETIMEOUT, QM_ENOTSUP = 0, 1, 2, 3, 4
QM_AFFINE, QM_Q8_0, QM_MXFP4, QM_MXFP4_BLOCKS, QM_Q4_K, QM_Q6_K = 0, 1, 2, 3, 4, 5
QM_F32, QM_BF16, QM_F16 = 0, 1, 2
QM_I32, QM_I64 = 0, 1
QM_WEIGHT_STATIC = 1
QM_MAX_NDIM = 4
QM_MAX_MANY = 8

_STATUS = {QM_EINVAL: "QM_EINVAL", QM_ECUDA: "QM_ECUDA", QM_ETIMEOUT: "QM_ETIMEOUT",
           QM_ENOTSUP: "QM_ENOTSUP"}
_FORMATS = {"affine": QM_AFFINE, "q8_0": QM_Q8_0, "mxfp4": QM_MXFP4, "mxfp4_blocks": QM_MXFP4_BLOCKS,
            "q4_k": QM_Q4_K, "q6_k": QM_Q6_K}
_DTYPES = {torch.float32: QM_F32, torch.bfloat16: QM_BF16, torch.float16: QM_F16}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class QMError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


class _CWeight(ctypes.Structure):
    _fields_ = [
        ("format", ctypes.c_int32), ("bits", ctypes.c_int32), ("group_size", ctypes.c_int32),
        ("scale_dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * QM_MAX_NDIM),
        ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p),
        ("flags", ctypes.c_uint32),
    ]


def library_path() -> str:
    return os.environ.get("QM_LIBRARY") or os.path.join(_HERE, "libqm.so")


def load_library():
    """Loads libqm.so (built by packed_qmatmul_gb300/build.py); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libqm.so not found at {path}: run "
                               "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(path)
        i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        wp = ctypes.POINTER(_CWeight)
        sigs = {
            "qm_dequant": ([wp, i32, vp, vp], i32),
            "qm_quantize_q8_0": ([vp, i32, i64, i64, vp, vp], i32),
            "qm_check_wait_timeout": ([ctypes.c_uint64, vp], i32),
            "qm_apply": ([wp, vp, i64, i32, vp, vp], i32),
            "qm_apply_many": ([ctypes.POINTER(wp), i32, vp, i64, i32, ctypes.POINTER(vp), vp], i32),
            "qm_take": ([wp, i32, vp, i32, i64, vp, vp, vp, i32, vp, vp], i32),
            "qm_apply_experts_workspace": ([wp, i64, i64], sz),
            "qm_experts_route_workspace": ([i64, i64], sz),
            "qm_apply_experts": ([wp, vp, i32, i64, i64, vp, i64, i32, vp, vp, sz, vp], i32),
            "qm_experts_route": ([vp, i32, i64, i64, vp, vp, vp, vp, sz, vp], i32),
            "qm_apply_experts_static": ([wp, vp, i32, i64, i64, vp, i64, i32, vp, vp], i32),
            "qm_device_status": ([vp], i32),
            "qm_last_error": ([], ctypes.c_char_p),
            "qm_version": ([], i32),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(status: int):
    if status != QM_OK:
        msg = load_library().qm_last_error().decode()
        raise QMError(status, msg)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("libqm takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- weights
class QWeight:
    """A packed weight: format, logical shape [..., n, k] and device parts.

    Parts are device tensors whose bytes are the format's (any integer dtype of
    the right byte size; uint32 codes may be held as int32). The descriptor
    passed to the library is built once and rebuilt when a field is assigned;
    parts are read through their tensors' addresses at that time.
    """

    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        if name != "_cref":
            object.__setattr__(self, "_cref", None)

    def __init__(self, fmt, shape: Sequence[int], codes: torch.Tensor,
                 scales: Optional[torch.Tensor] = None, biases: Optional[torch.Tensor] = None,
                 bits: int = 0, group_size: int = 0, scale_dtype: int = QM_BF16, flags: int = 0):
        self.format = _FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
        self.shape = tuple(int(s) for s in shape)
        self.codes, self.scales, self.biases = codes, scales, biases
        self.bits = int(bits)
        self.group_size = int(group_size)
        self.scale_dtype = int(scale_dtype)
        self.flags = int(flags)

    @classmethod
    def from_arrays(cls, d: dict, device="cuda", flags: int = 0) -> "QWeight":
        """From a dict of NumPy parts as packed_qmatmul_gb300.synth returns."""
        import numpy as np

        def dev(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            view = {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16}.get(a.dtype)
            t = torch.from_numpy(a.view(view) if view is not None else a)
            return t.to(device)

        sdt = QM_F16 if d.get("scale_dtype") == "f16" else QM_BF16
        return cls(d["format"], d["shape"], dev(d["codes"]), dev(d.get("scales")),
                   dev(d.get("biases")), bits=d.get("bits", 0), group_size=d.get("group_size", 0),
                   scale_dtype=sdt, flags=flags)

    def _ref(self):
        """ctypes reference to the descriptor (cached)."""
        ref = self._cref
        if ref is None:
            ref = ctypes.byref(self._c())
            object.__setattr__(self, "_cref", ref)
        return ref

    def _pointer(self):
        """ctypes pointer to the same cached descriptor (for arrays of weights)."""
        ref = self._ref()
        cached = self.__dict__.get("_cptr")
        if cached is None or cached[0] is not ref:  # the descriptor was rebuilt
            cached = (ref, ctypes.pointer(ref._obj))
            object.__setattr__(self, "_cptr", cached)
        return cached[1]

    def _c(self) -> _CWeight:
        w = _CWeight()
        w.format, w.bits, w.group_size, w.scale_dtype = (self.format, self.bits, self.group_size,
                                                          self.scale_dtype)
        w.ndim = len(self.shape)
        for i, s in enumerate(self.shape[:QM_MAX_NDIM]):
            w.shape[i] = s
        w.codes, w.scales, w.biases = _ptr(self.codes), _ptr(self.scales), _ptr(self.biases)
        w.flags = self.flags
        return w

    def part_shapes(self, lead: Sequence[int]):
        """Byte shapes of (codes, scales, biases) for leading dims `lead` + [n]."""
        k = self.shape[-1]
        if self.format == QM_AFFINE:
            cb, sb = k * self.bits // 8, k // self.group_size * 2
            return (tuple(lead) + (cb,), tuple(lead) + (sb,), tuple(lead) + (sb,))
        if self.format == QM_Q8_0:
            return (tuple(lead) + (k // 32 * 34,), None, None)
        if self.format == QM_MXFP4_BLOCKS:
            return (tuple(lead) + (k // 32 * 17,), None, None)
        if self.format == QM_Q4_K:
            return (tuple(lead) + (k // 256 * 144,), None, None)
        if self.format == QM_Q6_K:
            return (tuple(lead) + (k // 256 * 210,), None, None)
        return (tuple(lead) + (k // 2,), tuple(lead) + (k // 32,), None)


# ---------------------------------------------------------------- C entry points
def qm_version() -> int:
    return load_library().qm_version()


def qm_last_error() -> str:
    return load_library().qm_last_error().decode()


def qm_dequant(w: QWeight, out: torch.Tensor, stream=None) -> None:
    _check(load_library().qm_dequant(w._ref(), _DTYPES[out.dtype], _ptr(out),
                                     _stream(stream)))


def qm_quantize_q8_0(x: torch.Tensor, blocks: torch.Tensor, stream=None) -> None:
    k = x.shape[-1]
    rows = x.numel() // k if k else 0
    _check(load_library().qm_quantize_q8_0(_ptr(x), _DTYPES[x.dtype], rows, k, _ptr(blocks),
                                           _stream(stream)))


def qm_apply(w: QWeight, x: torch.Tensor, y: torch.Tensor, stream=None) -> None:
    M = x.shape[0] if x.dim() == 2 else 1
    _check(load_library().qm_apply(w._ref(), _ptr(x), M, _DTYPES[x.dtype], _ptr(y),
                                   _stream(stream)))


_WARR = [ctypes.POINTER(_CWeight) * max(i, 1) for i in range(QM_MAX_MANY + 1)]
_PARR = [ctypes.c_void_p * max(i, 1) for i in range(QM_MAX_MANY + 1)]


_MANY = {}


def _weight_array(ws):
    """The C array of descriptor pointers for these weights, kept per tuple of
    weights and rebuilt when any of their descriptors was (a cached entry holds
    its descriptors, so a weight reusing an id cannot match a stale one)."""
    key = tuple(map(id, ws))
    hit = _MANY.get(key)
    if hit is not None and tuple([w._cref for w in ws]) == hit[0]:  # descriptors compare by identity
        return hit[1]
    refs = tuple(w._ref() for w in ws)
    arr = _WARR[len(ws)](*[w._pointer() for w in ws])
    if len(_MANY) >= 1024:
        _MANY.clear()
    _MANY[key] = (refs, arr)
    return arr


def qm_apply_many(ws: Sequence[QWeight], x: torch.Tensor, ys: Sequence[torch.Tensor], stream=None) -> None:
    """ys[i] = x times ws[i]^T for weights that read the same x (one launch at M = 1)."""
    M = x.shape[0] if x.dim() == 2 else 1
    n = len(ws)
    if n > QM_MAX_MANY or len(ys) != n:  # the C call refuses these; keep the arrays in range
        raise QMError(QM_EINVAL, f"count: {n} weights and {len(ys)} outputs (1 .. {QM_MAX_MANY} each)")
    warr = _weight_array(ws)
    yarr = _PARR[n](*[_ptr(y) for y in ys])
    _check(load_library().qm_apply_many(warr, n, _ptr(x), M, _DTYPES[x.dtype], yarr, _stream(stream)))


def qm_take(w: QWeight, axis: int, ids: torch.Tensor, out_codes=None, out_scales=None,
            out_biases=None, out_dense: Optional[torch.Tensor] = None, stream=None) -> None:
    id_type = QM_I64 if ids.dtype == torch.int64 else QM_I32
    out_dtype = _DTYPES[out_dense.dtype] if out_dense is not None else QM_F32
    _check(load_library().qm_take(w._ref(), axis, _ptr(ids), id_type, ids.numel(),
                                  _ptr(out_codes), _ptr(out_scales), _ptr(out_biases), out_dtype,
                                  _ptr(out_dense), _stream(stream)))


def qm_apply_experts_workspace(w: QWeight, T: int, topk: int) -> int:
    return load_library().qm_apply_experts_workspace(w._ref(), T, topk)


def qm_experts_route_workspace(P: int, E: int) -> int:
    return load_library().qm_experts_route_workspace(P, E)


def qm_apply_experts(w: QWeight, ids: torch.Tensor, x: torch.Tensor, y: torch.Tensor,
                     workspace: torch.Tensor, stream=None) -> None:
    T, topk = ids.shape
    id_type = QM_I64 if ids.dtype == torch.int64 else QM_I32
    _check(load_library().qm_apply_experts(
        w._ref(), _ptr(ids), id_type, T, topk, _ptr(x), x.shape[0], _DTYPES[x.dtype],
        _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def qm_apply_experts_static(w: QWeight, ids: torch.Tensor, x: torch.Tensor, y: torch.Tensor,
                            stream=None) -> None:
    """qm_apply_experts with the library's own 1 MiB routing scratch (no workspace)."""
    T, topk = ids.shape
    id_type = QM_I64 if ids.dtype == torch.int64 else QM_I32
    _check(load_library().qm_apply_experts_static(
        w._ref(), _ptr(ids), id_type, T, topk, _ptr(x), x.shape[0], _DTYPES[x.dtype],
        _ptr(y), _stream(stream)))


def qm_experts_route(ids: torch.Tensor, E: int, counts: torch.Tensor, offsets: torch.Tensor,
                     perm: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    id_type = QM_I64 if ids.dtype == torch.int64 else QM_I32
    _check(load_library().qm_experts_route(
        _ptr(ids), id_type, ids.numel(), E, _ptr(counts), _ptr(offsets), _ptr(perm),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def qm_check_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load_library().qm_check_wait_timeout(limit_ns, _stream(stream)))


def qm_device_status(stream=None) -> None:
    _check(load_library().qm_device_status(_stream(stream)))


# ---------------------------------------------------------------- conveniences
def dequant(w: QWeight, dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    out = torch.empty(w.shape, dtype=dtype, device=w.codes.device)
    qm_dequant(w, out, stream)
    return out


def quantize_q8_0(x: torch.Tensor, stream=None) -> QWeight:
    """The float weight x [..., n, k] (float32, bfloat16 or float16) stored as GGUF Q8_0."""
    k = x.shape[-1]
    blocks = torch.empty(tuple(x.shape[:-1]) + (k // 32 * 34,), dtype=torch.uint8, device=x.device)
    qm_quantize_q8_0(x, blocks, stream)
    return QWeight("q8_0", tuple(x.shape), blocks)


def apply(w: QWeight, x: torch.Tensor, stream=None) -> torch.Tensor:
    y = torch.empty((x.shape[0], w.shape[-2]), dtype=x.dtype, device=x.device)
    qm_apply(w, x, y, stream)
    return y


def apply_many(ws: Sequence[QWeight], x: torch.Tensor, stream=None) -> list:
    ys = [torch.empty((x.shape[0], w.shape[-2]), dtype=x.dtype, device=x.device) for w in ws]
    qm_apply_many(ws, x, ys, stream)
    return ys


def take(w: QWeight, axis: int, ids: torch.Tensor, dense_dtype=None, packed=True, stream=None):
    """Returns (packed QWeight or None, dense tensor or None)."""
    ndim = len(w.shape)
    ax = axis + ndim if axis < 0 else axis
    n = ids.numel()
    out_shape = w.shape[:ax] + (n,) + w.shape[ax + 1:]
    dev = w.codes.device
    outs = [None, None, None]
    tw = None
    if packed:
        shapes = w.part_shapes(out_shape[:-1])
        outs = [None if s is None else torch.empty(s, dtype=torch.uint8, device=dev) for s in shapes]
        tw = QWeight(w.format, out_shape, outs[0], outs[1], outs[2], bits=w.bits,
                     group_size=w.group_size, scale_dtype=w.scale_dtype)
    dense = None if dense_dtype is None else torch.empty(out_shape, dtype=dense_dtype, device=dev)
    qm_take(w, axis, ids, outs[0], outs[1], outs[2], dense, stream)
    return tw, dense


def apply_experts(w: QWeight, ids: torch.Tensor, x: torch.Tensor, stream=None) -> torch.Tensor:
    T, topk = ids.shape
    y = torch.empty((T, topk, w.shape[-2]), dtype=x.dtype, device=x.device)
    ws = torch.empty(max(qm_apply_experts_workspace(w, T, topk), 256), dtype=torch.uint8,
                     device=x.device)
    qm_apply_experts(w, ids, x, y, ws, stream)
    return y


def route(ids: torch.Tensor, E: int, stream=None):
    P = ids.numel()
    dev = ids.device
    counts = torch.empty(max(E, 1), dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(P, 1), dtype=torch.int32, device=dev)
    ws = torch.empty(max(qm_experts_route_workspace(P, E), 256), dtype=torch.uint8, device=dev)
    qm_experts_route(ids, E, counts, offsets, perm, ws, stream)
    return counts[:E], offsets, perm[:P]
