"""The oracle: a plain float64 CPU restatement of the packed weight formats.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only code that may import this
package. The CUDA library neither imports nor links it, and this package
imports nothing from the library.

The arithmetic lives in ``qm_oracle.c`` (plain C, compiled with gcc, OpenMP
over output rows). This module builds it on first use and wraps it for NumPy
arrays. Format and dtype codes here are the oracle's own:

    format: AFFINE = 0 (MLX affine), Q8_0 = 1 (GGUF), MXFP4 = 2 (scales apart),
            MXFP4_BLOCKS = 3 (MXFP4 in GGUF's 17-byte blocks),
            Q4_K = 4, Q6_K = 5 (GGUF's 256-value super-blocks)
    dtype : F32 = 0, BF16 = 1, F16 = 2   (16-bit data is passed as uint16 bits)

Sources, by page title and section:
  "GPTQModel wiki: MLX Apple Silicon" -- "Concepts: method, checkpoint,
      runtime, and tensor layout"; "Packed layouts and exact transcoding".
  "Nx_quant (raven-ml.dev API docs)" -- "Weights"; "Products".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

AFFINE, Q8_0, MXFP4, MXFP4_BLOCKS, Q4_K, Q6_K = 0, 1, 2, 3, 4, 5
F32, BF16, F16 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile qm_oracle.c into liboracle.so next to it (gcc -O2 -fopenmp)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # QM_ORACLE_LIB names a prebuilt variant of this library; the
            # mutation tests use it to load copies with planted mistakes.
            path = os.environ.get("QM_ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            i32, i64, vp, dp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            u16 = ctypes.c_uint16
            lib.or_f16_to_f64.argtypes = [u16]
            lib.or_f16_to_f64.restype = ctypes.c_double
            lib.or_bf16_to_f64.argtypes = [u16]
            lib.or_bf16_to_f64.restype = ctypes.c_double
            lib.or_e2m1_to_f64.argtypes = [i32]
            lib.or_e2m1_to_f64.restype = ctypes.c_double
            lib.or_e8m0_to_f64.argtypes = [i32]
            lib.or_e8m0_to_f64.restype = ctypes.c_double
            lib.or_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.or_f32_to_bf16.restype = u16
            lib.or_f32_to_f16.argtypes = [ctypes.c_float]
            lib.or_f32_to_f16.restype = u16
            lib.or_affine_code.argtypes = [vp, i32, i64]
            lib.or_affine_code.restype = ctypes.c_uint32
            lib.or_mxfp4_code.argtypes = [vp, i64]
            lib.or_mxfp4_code.restype = i32
            lib.or_row_values.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, i64, vp]
            lib.or_row_values.restype = None
            lib.or_dequant.argtypes = [i32, i32, i32, i32, i64, i64, vp, vp, vp, i32, vp]
            lib.or_dequant.restype = None
            lib.or_apply.argtypes = [i32, i32, i32, i32, i64, i64, vp, vp, vp, vp, i32, i64, dp]
            lib.or_apply.restype = None
            lib.or_apply_entries.argtypes = [i32, i32, i32, i32, i64, i64, vp, vp, vp, vp, i32,
                                             i64, vp, vp, dp]
            lib.or_apply_entries.restype = None
            lib.or_quantize_q8_0.argtypes = [vp, i64, i64, vp]
            lib.or_quantize_q8_0.restype = None
            lib.or_take_part.argtypes = [vp, i64, i64, i64, vp, i32, i64, vp]
            lib.or_take_part.restype = None
            lib.or_route.argtypes = [vp, i32, i64, i64, vp, vp, vp]
            lib.or_route.restype = i64
            lib.or_apply_experts.argtypes = [i32, i32, i32, i32, i64, i64, i64, vp, vp, vp,
                                             vp, i32, i64, i64, vp, i64, i32, dp]
            lib.or_apply_experts.restype = None
            lib.or_apply_experts_entries.argtypes = [i32, i32, i32, i32, i64, i64, i64, vp, vp,
                                                     vp, vp, i32, i64, i64, vp, i64, i32, i64,
                                                     vp, vp, dp]
            lib.or_apply_experts_entries.restype = None
            lib.or_round_array.argtypes = [vp, i64, i32, vp]
            lib.or_round_array.restype = None
            lib.or_decode_array.argtypes = [vp, i64, i32, dp]
            lib.or_decode_array.restype = None
            lib.or_num_threads.argtypes = []
            lib.or_num_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous arrays"
    return a.ctypes.data


def _ids_flag(ids: np.ndarray) -> int:
    if ids.dtype == np.int32:
        return 0
    if ids.dtype == np.int64:
        return 1
    raise TypeError("ids must be int32 or int64")


def num_threads() -> int:
    return _load().or_num_threads()


# ---------------------------------------------------------------- scalars
def f16_to_f64(h: int) -> float:
    return _load().or_f16_to_f64(h)


def bf16_to_f64(h: int) -> float:
    return _load().or_bf16_to_f64(h)


def e2m1_to_f64(code: int) -> float:
    return _load().or_e2m1_to_f64(code)


def e8m0_to_f64(s: int) -> float:
    return _load().or_e8m0_to_f64(s)


def f32_to_bf16(f: float) -> int:
    return _load().or_f32_to_bf16(f)


def f32_to_f16(f: float) -> int:
    return _load().or_f32_to_f16(f)


def round_array(a: np.ndarray, dtype: int) -> np.ndarray:
    """float32 array rounded once to dtype (16-bit results as uint16 bits)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.float32 if dtype == F32 else np.uint16)
    _load().or_round_array(_ptr(a), a.size, dtype, _ptr(out))
    return out


def decode_array(bits: np.ndarray, dtype: int) -> np.ndarray:
    """bf16 (dtype BF16) or f16 (dtype F16) bit patterns -> float64."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().or_decode_array(_ptr(bits), bits.size, dtype, _ptr(out))
    return out


def affine_code(row_words: np.ndarray, bits: int, i: int) -> int:
    row_words = np.ascontiguousarray(row_words, dtype=np.uint32)
    return _load().or_affine_code(_ptr(row_words), bits, i)


def mxfp4_code(row_bytes: np.ndarray, i: int) -> int:
    row_bytes = np.ascontiguousarray(row_bytes, dtype=np.uint8)
    return _load().or_mxfp4_code(_ptr(row_bytes), i)


# ---------------------------------------------------------------- weights
class Weight:
    """A packed weight as the oracle reads it: parts as NumPy arrays.

    shape is the logical [..., n, k]; the parts carry the same leading axes.
    """

    def __init__(self, fmt, shape, codes, scales=None, biases=None, bits=0,
                 group_size=32, scale_dtype=BF16):
        self.fmt = fmt
        self.shape = tuple(int(s) for s in shape)
        self.codes = np.ascontiguousarray(codes)
        self.scales = None if scales is None else np.ascontiguousarray(scales)
        self.biases = None if biases is None else np.ascontiguousarray(biases)
        self.bits = bits if fmt == AFFINE else {Q8_0: 8, Q6_K: 6}.get(fmt, 4)
        self.group_size = group_size if fmt == AFFINE else {Q4_K: 256, Q6_K: 256}.get(fmt, 32)
        self.scale_dtype = scale_dtype

    @property
    def k(self):
        return self.shape[-1]

    @property
    def rows(self):
        r = 1
        for s in self.shape[:-1]:
            r *= s
        return r

    def _args(self):
        return (self.fmt, self.bits, self.group_size, self.scale_dtype)

    def parts(self):
        return {"codes": self.codes, "scales": self.scales, "biases": self.biases}


def row_values(w: Weight, r: int) -> np.ndarray:
    v = np.empty(w.k, dtype=np.float32)
    _load().or_row_values(*w._args(), w.k, _ptr(w.codes), _ptr(w.scales), _ptr(w.biases),
                          r, _ptr(v))
    return v


def dequant(w: Weight, dtype: int) -> np.ndarray:
    """Every value of w rounded once to dtype; 16-bit results as uint16 bits."""
    out = np.empty(w.shape, dtype=np.float32 if dtype == F32 else np.uint16)
    _load().or_dequant(*w._args(), w.rows, w.k, _ptr(w.codes), _ptr(w.scales),
                       _ptr(w.biases), dtype, _ptr(out))
    return out


def _x_dtype(x: np.ndarray, xdt):
    if xdt is not None:
        return xdt
    return F32 if x.dtype == np.float32 else BF16


def apply(w: Weight, x: np.ndarray, xdt=None) -> np.ndarray:
    """y[m, j] = sum_i x[m, i] * w[j, i] in float64 (unrounded), x [M, k]."""
    x = np.ascontiguousarray(x)
    M = x.shape[0]
    y = np.empty((M, w.rows), dtype=np.float64)
    _load().or_apply(*w._args(), w.rows, w.k, _ptr(w.codes), _ptr(w.scales), _ptr(w.biases),
                     _ptr(x), _x_dtype(x, xdt), M, _ptr(y))
    return y


def apply_entries(w: Weight, x: np.ndarray, m_idx, j_idx, xdt=None) -> np.ndarray:
    x = np.ascontiguousarray(x)
    m_idx = np.ascontiguousarray(m_idx, dtype=np.int64)
    j_idx = np.ascontiguousarray(j_idx, dtype=np.int64)
    # the C routine reads both index arrays and x's rows unchecked
    if m_idx.ndim != 1 or m_idx.shape != j_idx.shape:
        raise ValueError(f"apply_entries: m_idx {m_idx.shape} and j_idx {j_idx.shape} must be equal 1-D arrays")
    if m_idx.size and (m_idx.min() < 0 or m_idx.max() >= x.shape[0] or j_idx.min() < 0 or j_idx.max() >= w.rows):
        raise ValueError("apply_entries: an index is out of range")
    out = np.empty(m_idx.shape[0], dtype=np.float64)
    _load().or_apply_entries(*w._args(), w.rows, w.k, _ptr(w.codes), _ptr(w.scales),
                             _ptr(w.biases), _ptr(x), _x_dtype(x, xdt), m_idx.shape[0],
                             _ptr(m_idx), _ptr(j_idx), _ptr(out))
    return out


def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    """Float32 x [..., n, k] (k a multiple of 32) as Q8_0 blocks [..., n, k/32*34]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    k = x.shape[-1]
    if k % 32:
        raise ValueError("k must be a multiple of 32")
    rows = x.size // k if k else 0
    out = np.empty(x.shape[:-1] + (k // 32 * 34,), dtype=np.uint8)
    _load().or_quantize_q8_0(_ptr(x), rows, k, _ptr(out))
    return out


def take_part(part: np.ndarray, axis: int, ids: np.ndarray) -> np.ndarray:
    """Gather along `axis` of one packed part; out-of-range ids give zero bytes."""
    part = np.ascontiguousarray(part)
    ids = np.ascontiguousarray(ids)
    shape = part.shape
    outer = int(np.prod(shape[:axis], dtype=np.int64))
    length = shape[axis]
    inner = int(np.prod(shape[axis + 1:], dtype=np.int64)) * part.itemsize
    out = np.empty(shape[:axis] + (ids.size,) + shape[axis + 1:], dtype=part.dtype)
    _load().or_take_part(_ptr(part), outer, length, inner, _ptr(ids), _ids_flag(ids), ids.size,
                         _ptr(out))
    return out


def take(w: Weight, axis: int, ids: np.ndarray) -> Weight:
    """take ~axis p w: each packed part gathered along axis, nothing decoded."""
    if axis < 0:
        axis += len(w.shape)
    if axis < 0 or axis >= len(w.shape) - 1:
        raise ValueError("axis")
    shape = w.shape[:axis] + (int(np.asarray(ids).size),) + w.shape[axis + 1:]
    parts = {name: (None if p is None else take_part(p, axis, ids))
             for name, p in w.parts().items()}
    return Weight(w.fmt, shape, parts["codes"], parts["scales"], parts["biases"], bits=w.bits,
                  group_size=w.group_size, scale_dtype=w.scale_dtype)


def route(ids: np.ndarray, E: int):
    """Stable sort of flattened positions by expert: (counts, offsets, perm, n_out)."""
    ids = np.ascontiguousarray(ids).reshape(-1)
    P = ids.size
    counts = np.empty(E, dtype=np.int64)
    offsets = np.empty(E + 1, dtype=np.int64)
    perm = np.empty(max(P, 1), dtype=np.int64)
    n_out = _load().or_route(_ptr(ids), _ids_flag(ids), P, E, _ptr(counts), _ptr(offsets),
                             _ptr(perm))
    return counts, offsets, perm[: offsets[E]].copy(), int(n_out)


def apply_experts(w: Weight, ids: np.ndarray, x: np.ndarray, xdt=None) -> np.ndarray:
    """y[t, j, :] = w[ids[t, j]] applied to x's row (zeros for ids outside [0, E))."""
    E, n, k = w.shape
    ids = np.ascontiguousarray(ids)
    T, topk = ids.shape
    x = np.ascontiguousarray(x)
    y = np.empty((T, topk, n), dtype=np.float64)
    _load().or_apply_experts(*w._args(), E, n, k, _ptr(w.codes), _ptr(w.scales),
                             _ptr(w.biases), _ptr(ids), _ids_flag(ids), T, topk, _ptr(x),
                             x.shape[0], _x_dtype(x, xdt), _ptr(y))
    return y


def apply_experts_entries(w: Weight, ids: np.ndarray, x: np.ndarray, p_idx, j_idx,
                          xdt=None) -> np.ndarray:
    E, n, k = w.shape
    ids = np.ascontiguousarray(ids)
    T, topk = ids.shape
    x = np.ascontiguousarray(x)
    p_idx = np.ascontiguousarray(p_idx, dtype=np.int64)
    j_idx = np.ascontiguousarray(j_idx, dtype=np.int64)
    out = np.empty(p_idx.shape[0], dtype=np.float64)
    _load().or_apply_experts_entries(*w._args(), E, n, k, _ptr(w.codes), _ptr(w.scales),
                                     _ptr(w.biases), _ptr(ids), _ids_flag(ids), T, topk,
                                     _ptr(x), x.shape[0], _x_dtype(x, xdt), p_idx.shape[0],
                                     _ptr(p_idx), _ptr(j_idx), _ptr(out))
    return out
