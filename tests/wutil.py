"""Test helpers: synthetic weights as oracle weights, and the product tolerance.

Nothing here decodes a format or forms a product; the oracle and the library
do that. The tolerance is the one the product contract states (see
``check_product``).
"""
import numpy as np

import oracle

FMT = {"affine": oracle.AFFINE, "q8_0": oracle.Q8_0, "mxfp4": oracle.MXFP4, "mxfp4_blocks": oracle.MXFP4_BLOCKS,
       "q4_k": oracle.Q4_K, "q6_k": oracle.Q6_K}
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


# Magnitudes from here up round to infinity in bfloat16: halfway between its
# largest finite value, (2 - 2^-7) * 2^127, and 2^128.
BF16_OVERFLOW = 2.0 ** 128 - 2.0 ** 119


def expected_nonfinite(y_ref: np.ndarray):
    """Where the oracle's product, rounded once to bfloat16, is NaN, +inf or -inf."""
    nan = np.isnan(y_ref)
    big = ~nan & (np.abs(y_ref) >= BF16_OVERFLOW)
    return nan, big & (y_ref > 0), big & (y_ref < 0)


def check_product(y_gpu: np.ndarray, y_ref: np.ndarray, wnorm: np.ndarray, xnorm: np.ndarray,
                  k: int, what: str = ""):
    """The product contract, element by element and as a whole.

    y_gpu: the library's result decoded to float64 [M, n]; y_ref: the oracle's
    unrounded float64 product [M, n]; wnorm [n] (or [M, n] where each output
    row has its own matrix, as with experts), xnorm [M] the row norms.

    Non-finite results exactly: NaN where the oracle's product is NaN, and an
    infinity of the same sign where it is infinite or, rounded once to
    bfloat16, overflows (the per-element definition of "Nx_quant", "Products":
    values and products are IEEE arithmetic, so an infinite value meets its
    activation as IEEE says). Every other element must be finite and, per
    element: |y_gpu - y_ref| <= 1e-2 * ||w_j|| * ||x_m|| / sqrt(k) plus half a
    bfloat16 ulp of y_gpu -- the single final rounding to x's dtype that the
    product's definition itself applies. As a whole, over the finite elements:
    relative Frobenius error <= 4e-3. Returns a dict of statistics.
    """
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    nan, pinf, ninf = expected_nonfinite(y_ref)
    for name, want, got in (("NaN", nan, np.isnan(y_gpu)), ("+inf", pinf, np.isposinf(y_gpu)),
                            ("-inf", ninf, np.isneginf(y_gpu))):
        if not np.array_equal(want, got):
            idx = np.argwhere(want != got)[:8].tolist()
            raise AssertionError(f"{what}: {name} pattern differs from the oracle at {idx} "
                                 f"(gpu {[y_gpu[tuple(i)] for i in idx]}, oracle {[y_ref[tuple(i)] for i in idx]})")
    fin = ~(nan | pinf | ninf)
    wnorm = np.asarray(wnorm, dtype=np.float64)
    xnorm = np.asarray(xnorm, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        bound = 1e-2 * (np.outer(xnorm, wnorm) if wnorm.ndim == 1 else xnorm[:, None] * wnorm) / np.sqrt(k)
        bound = np.broadcast_to(bound, y_ref.shape)
        err = np.abs(np.where(fin, y_gpu, 0.0) - np.where(fin, y_ref, 0.0))
        allowed = bound + bf16_half_ulp(np.where(fin, y_gpu, 0.0))
    bad = fin & ~(err <= allowed)
    d = np.where(fin, y_gpu, 0.0) - np.where(fin, y_ref, 0.0)
    r = np.where(fin, y_ref, 0.0)
    fro = np.linalg.norm(d) / max(np.linalg.norm(r), 1e-300)
    with np.errstate(invalid="ignore", divide="ignore"):
        ratio = np.where(fin & (bound > 0), err / np.where(bound > 0, bound, 1.0), 0.0)
    stats = dict(max_err=float(err.max(initial=0.0)), n_bad=int(bad.sum()),
                 literal_over=int((fin & (err > bound)).sum()), fro=float(fro),
                 max_ratio=float(np.nan_to_num(ratio, nan=np.inf).max(initial=0.0)),
                 n_nonfinite=int((~fin).sum()))
    assert stats["n_bad"] == 0, f"{what}: {stats}"
    assert fro <= 4e-3, f"{what}: {stats}"
    return stats
