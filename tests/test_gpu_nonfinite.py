"""Products where weight values or activations are infinite or NaN, or large
enough that a block-scaled sum could overflow where the true product does not.

"Nx_quant (raven-ml.dev API docs)", section "Products": every value of a
weight is a float32 value (val dequant) -- an MXFP4 value past float32's
range is infinite (codes of magnitude 4 or more at scale byte 253, 2 or more
at 254), the scale byte 255 makes its group NaN, a GGUF block whose float16
scale is infinite or NaN gives infinite or NaN values -- and apply sums x
times those values (val apply). The non-finite results therefore follow from
IEEE arithmetic on each element, whatever the order of the sum, and the tests
compare them exactly (wutil.check_product): NaN where the oracle has NaN, an
infinity of the same sign where it has one. Every finite result keeps the
ordinary tolerance.

M = 1 and 8 run the decode kernel, M = 33 and 130 the tensor-core kernel;
apply_experts runs both of its paths.
"""
import numpy as np
import pytest
import torch

import oracle
import packed_qmatmul_gb300 as qm
from packed_qmatmul_gb300 import synth
from wutil import bf16_to_f64, check_product, row_norms, to_oracle

pytestmark = pytest.mark.gpu

MS = [1, 8, 33, 130]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from packed_qmatmul_gb300 import build

    build.build()
    qm.load_library()
    torch.cuda.set_device(0)


def _host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _norms(ow, x):
    with np.errstate(over="ignore", invalid="ignore"):
        return row_norms(ow), np.linalg.norm(oracle.decode_array(x, oracle.BF16), axis=1)


def _apply(w, x, what):
    ow = to_oracle(w)
    got = bf16_to_f64(_host(qm.apply(qm.QWeight.from_arrays(w), _dev_bf16(x))))
    ref = oracle.apply(ow, x)
    wn, xn = _norms(ow, x)
    return check_product(got, ref, wn, xn, ow.k, what), ref


def _experts(w, ids, x, what):
    E, n, k = w["shape"]
    T, topk = ids.shape
    ow = to_oracle(w)
    y = qm.apply_experts(qm.QWeight.from_arrays(w), torch.from_numpy(ids).cuda(), _dev_bf16(x))
    got = bf16_to_f64(_host(y)).reshape(T * topk, n)
    ref = oracle.apply_experts(ow, ids, x).reshape(T * topk, n)
    flat = ids.reshape(-1)
    out = (flat < 0) | (flat >= E)
    assert np.all(got[out] == 0), what
    rows = np.where(~out)[0]
    wn, xn = _norms(ow, x)
    xr = rows // topk if x.shape[0] == T else rows
    return check_product(got[rows], ref[rows], wn.reshape(E, n)[flat[rows]], xn[xr], k, what)


# ---------------------------------------------------------------- MXFP4
def _mxfp4_every_byte(g, k=512, lead=()):
    """Rows 0..255: row r has one group (r mod k/32) at scale byte r and the
    others at the ordinary bytes 118..126; codes uniform."""
    n = 256
    w = synth.mxfp4_weight(g, n, k, lead=lead)
    sc = w["scales"].reshape(-1, n, k // 32)
    for r in range(n):
        sc[:, r, r % (k // 32)] = r
    return w


@pytest.mark.parametrize("M", MS)
def test_mxfp4_every_scale_byte(M):
    # activations of about 2^-10, so that no partial sum of the terms at scale
    # byte 252 (values up to 1.5 * 2^127) can leave float32's range: the
    # finite results are then order-free, and bytes 253 and 254 give the
    # infinities (and, with both signs, NaNs) of their values
    g = synth.rng(1400 + M)
    w = _mxfp4_every_byte(g)
    x = synth.activations(g, M, 512, sigma=2.0 ** -10)
    stats, ref = _apply(w, x, f"mxfp4 every scale byte M={M}")
    assert stats["n_nonfinite"] >= 3 * M  # rows at 253, 254 and 255 at least


@pytest.mark.parametrize("sigma", [1e-30, 2.0 ** -10])
@pytest.mark.parametrize("M", [1, 8])
def test_mxfp4_large_scales_small_activations(M, sigma):
    # every group at scale bytes 200..252 (2^73 .. 2^125) with tiny activations:
    # each group's sum is formed at its true size, so nothing overflows that
    # the exact product does not
    g = synth.rng(1410 + M)
    w = synth.mxfp4_weight(g, 96, 512, scale_lo=200, scale_hi=252)
    x = synth.activations(g, M, 512, sigma=sigma)
    stats, _ = _apply(w, x, f"mxfp4 large scales sigma={sigma} M={M}")
    assert stats["n_nonfinite"] == 0


@pytest.mark.parametrize("T", [16, 80])
def test_mxfp4_every_scale_byte_experts(T):
    # expert 0 holds the 256 rows of every scale byte, expert 1 ordinary ones;
    # T = 16 x 2 positions run the decode path, T = 80 x 2 the tensor cores
    g = synth.rng(1420 + T)
    w = _mxfp4_every_byte(g, lead=(2,))
    sc = w["scales"]
    sc[1] = g.integers(118, 127, size=sc[1].shape)
    ids = synth.expert_ids(g, T, 2, 2)
    ids[0, 1] = -1
    x = synth.activations(g, T, 512, sigma=2.0 ** -10)
    _experts(w, ids, x, f"mxfp4 every byte experts T={T}")


# ---------------------------------------------------------------- Q8_0
def _q8_0_nonfinite(g, k=256):
    """Every non-finite float16 d (both infinities, every NaN pattern) as one
    block of its own row, plus rows whose infinite d meets quants of one
    sign only (so products of one sign give an infinity, not a NaN)."""
    pats = np.concatenate([np.arange(0x7C00, 0x8000), np.arange(0xFC00, 0x10000)]).astype(np.uint16)
    n = len(pats) + 4
    w = synth.q8_0_weight(g, n, k)
    b = w["codes"].reshape(n, k // 32, 34)
    for r, d in enumerate(pats):
        blk = r % (k // 32)
        b[r, blk, 0], b[r, blk, 1] = d & 0xFF, d >> 8
    for i, (d, qs) in enumerate(((0x7C00, 1), (0x7C00, -1), (0xFC00, 1), (0xFC00, -1))):
        r = len(pats) + i
        b[r, 3, 0], b[r, 3, 1] = d & 0xFF, d >> 8
        q = g.integers(1, 128, size=32) * qs
        b[r, 3, 2:] = q.astype(np.int8).view(np.uint8)
    return w


@pytest.mark.parametrize("M", MS)
def test_q8_0_every_nonfinite_scale(M):
    g = synth.rng(1430 + M)
    w = _q8_0_nonfinite(g)
    x = synth.activations(g, M, 256)
    x[0] = synth.to_bf16_bits(np.abs(oracle.decode_array(x[0], oracle.BF16)).astype(np.float32))  # token 0 >= 0
    if M > 1:
        x[1, 100] = 0  # an infinite value times a zero activation: NaN
    stats, ref = _apply(w, x, f"q8_0 non-finite d M={M}")
    # one-signed rows give infinities for the non-negative token
    assert np.isposinf(ref[0, -4]) and np.isneginf(ref[0, -3])


@pytest.mark.parametrize("T", [16, 80])
def test_q8_0_nonfinite_scale_experts(T):
    g = synth.rng(1440 + T)
    w1 = _q8_0_nonfinite(g)
    n = w1["shape"][0]
    w0 = synth.q8_0_weight(g, n, 256)
    w = dict(w1, shape=(2, n, 256), codes=np.stack([w1["codes"], w0["codes"]]))
    ids = synth.expert_ids(g, T, 2, 2)
    x = synth.activations(g, T, 256)
    _experts(w, ids, x, f"q8_0 non-finite experts T={T}")


# ---------------------------------------------------------------- affine
def _affine_special(g, bits, gs, sdt):
    """Rows whose group 1 has a special scale or bias: infinities, NaNs,
    magnitudes at which code * scale + bias overflows float32 for some codes,
    and large finite ones on both sides of the exceptional threshold."""
    k = 512
    if sdt == "f16":
        cases = [(0x7C00, None), (0xFC00, None), (0x7E00, None), (None, 0x7C00), (None, 0xFC00), (None, 0x7E00),
                 (0x7BFF, 0x7BFF)]
        enc = synth.to_f16_bits
    else:
        cases = [(0x7F80, None), (0xFF80, None), (0x7FC0, None), (None, 0x7F80), (None, 0xFF80), (None, 0x7FC0),
                 (0x7E00, None),   # 2^125: 4-bit codes of 8 or more overflow to infinity
                 (0x7E80, None),   # 2^126
                 (0x7B80, None),   # 2^120: finite values, per element
                 (0x7AC0, None),   # 1.5 * 2^118: finite values, block-scaled
                 (None, 0x7F00),   # bias 2^127
                 (0x7E00, 0xFF00)]  # 2^125 and -2^127
        enc = synth.to_bf16_bits
    w = synth.affine_weight(g, 48, k, bits=bits, group_size=gs, scale_dtype=sdt)
    for r, (s, b) in enumerate(cases):
        if s is not None:
            w["scales"][r, 1] = s
        if b is not None:
            w["biases"][r, 1] = b
    if sdt == "bf16":  # and a row with every group at 2^120: finite values, summed per element
        w["scales"][len(cases), :] = enc(np.float32(2.0 ** 120))[()]
    return w


@pytest.mark.parametrize("bits,gs,sdt", [(4, 64, "bf16"), (8, 32, "bf16"), (4, 32, "f16"), (3, 64, "bf16"),
                                         (6, 32, "bf16")])
@pytest.mark.parametrize("M", MS)
def test_affine_special_scales(bits, gs, sdt, M):
    g = synth.rng(1450 + M + bits + gs)
    w = _affine_special(g, bits, gs, sdt)
    x = synth.activations(g, M, 512, sigma=2.0 ** -12)
    stats, _ = _apply(w, x, f"affine{bits} gs{gs} {sdt} special scales M={M}")
    assert stats["n_nonfinite"] >= 6 * M


# ---------------------------------------------------------------- activations
@pytest.mark.parametrize("M", [1, 8, 33])
def test_mxfp4_blocks_every_scale_byte(M):
    # MXFP4 in GGUF's 17-byte blocks: row r has one block at scale byte r
    g = synth.rng(1425 + M)
    n, k = 256, 512
    w = synth.mxfp4_blocks_weight(g, n, k)
    b = w["codes"].reshape(n, k // 32, 17)
    for r in range(n):
        b[r, r % (k // 32), 0] = r
    x = synth.activations(g, M, k, sigma=2.0 ** -10)
    stats, _ = _apply(w, x, f"mxfp4 blocks every scale byte M={M}")
    assert stats["n_nonfinite"] >= 3 * M


@pytest.mark.parametrize("kind", ["affine", "q8_0", "mxfp4", "mxfp4_blocks"])
@pytest.mark.parametrize("M", MS)
def test_nonfinite_activations(kind, M):
    # ordinary weights, activations holding infinities and NaNs: each output
    # is what IEEE gives for its terms (an infinity times a zero value is NaN)
    g = synth.rng(1460 + M)
    n, k = 80, 512
    if kind == "affine":
        w = synth.affine_weight(g, n, k, bits=4, group_size=64)
    elif kind == "q8_0":
        w = synth.q8_0_weight(g, n, k)
    elif kind == "mxfp4":
        w = synth.mxfp4_weight(g, n, k)
    else:
        w = synth.mxfp4_blocks_weight(g, n, k)
    x = synth.activations(g, M, k)
    x[0, 7] = 0x7F80                 # +inf
    if M > 1:
        x[1, 300] = 0xFFC0           # NaN
        x[M - 1, 31], x[M - 1, 480] = 0xFF80, 0x7F80  # -inf and +inf
    _apply(w, x, f"{kind} non-finite activations M={M}")
