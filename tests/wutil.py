"""Test helpers: synthetic weights as oracle weights, and the product tolerance.

Nothing here decodes a format or forms a product; the oracle and the library
do that. The tolerance is the one the product contract states (see
``check_product``).
"""
import numpy as np

import oracle

FMT = {"affine": oracle.AFFINE, "q8_0": oracle.Q8_0, "mxfp4": oracle.MXFP4, "mxfp4_blocks": oracle.MXFP4_BLOCKS}
SDT = {"bf16": oracle.BF16, "f16": oracle.F16, None: oracle.BF16}


def to_oracle(w: dict) -> "oracle.Weight":
    return oracle.Weight(FMT[w["format"]], w["shape"], w["codes"], w.get("scales"),
                         w.get("biases"), bits=w.get("bits", 0),
                         group_size=w.get("group_size", 32), scale_dtype=SDT[w.get("scale_dtype")])


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return oracle.decode_array(bits, oracle.BF16)


def bf16_half_ulp(y: np.ndarray) -> np.ndarray:
    """Half a unit in the last place of bfloat16 at |y| (8 significant bits)."""
    a = np.abs(y)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def row_norms(wq: "oracle.Weight") -> np.ndarray:
    """||w_j||_2 of every dequantized row, float64."""
    v = oracle.dequant(wq, oracle.F32).reshape(-1, wq.k).astype(np.float64)
    return np.sqrt((v * v).sum(axis=1))


def check_product(y_gpu: np.ndarray, y_ref: np.ndarray, wnorm: np.ndarray, xnorm: np.ndarray,
                  k: int, what: str = ""):
    """The product contract, element by element and as a whole.

    y_gpu: the library's result decoded to float64 [M, n]; y_ref: the oracle's
    unrounded float64 product [M, n]; wnorm [n] (or [M, n] where each output
    row has its own matrix, as with experts), xnorm [M] the row norms.

    Per element: |y_gpu - y_ref| <= 1e-2 * ||w_j|| * ||x_m|| / sqrt(k) plus half
    a bfloat16 ulp of y_gpu -- the single final rounding to x's dtype that the
    product's definition itself applies. As a whole: relative Frobenius error
    <= 4e-3. Returns a dict of statistics.
    """
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite outputs"
    wnorm = np.asarray(wnorm, dtype=np.float64)
    xnorm = np.asarray(xnorm, dtype=np.float64)
    bound = 1e-2 * (np.outer(xnorm, wnorm) if wnorm.ndim == 1 else xnorm[:, None] * wnorm) / np.sqrt(k)
    err = np.abs(y_gpu - y_ref)
    allowed = bound + bf16_half_ulp(y_gpu)
    bad = err > allowed
    fro = np.linalg.norm(y_gpu - y_ref) / max(np.linalg.norm(y_ref), 1e-300)
    stats = dict(max_err=float(err.max(initial=0.0)), n_bad=int(bad.sum()),
                 literal_over=int((err > bound).sum()), fro=float(fro),
                 max_ratio=float((err / np.maximum(bound, 1e-300)).max(initial=0.0)))
    assert stats["n_bad"] == 0, f"{what}: {stats}"
    assert fro <= 4e-3, f"{what}: {stats}"
    return stats
