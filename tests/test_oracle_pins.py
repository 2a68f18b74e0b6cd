"""Pins for the oracle: what the pages and the mathematics fix, checked without
calling the oracle's own formulas a second time.

Each test names the fact it pins. Library routines used as independent
references: NumPy's float16, PyTorch's bfloat16 conversion, torch.matmul in
float64, NumPy fancy indexing.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from packed_qmatmul_gb300 import synth
from wutil import to_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def _parse_value(s):
    s = s.strip()
    if s in ("nan", "inf", "-inf"):
        return float(s)
    if "2^" in s:
        sign = -1.0 if s.startswith("-") else 1.0
        s = s.lstrip("-")
        mant, _, exp = s.partition("2^")
        mant = float(mant.rstrip("*")) if mant else 1.0
        return sign * mant * 2.0 ** int(exp)
    return float(s)


def _same(a, b):
    """Equal values, NaN equal to NaN, and the sign of zero compared."""
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


# ------------------------------------------------------------ scalar codes
def test_e2m1_table_from_page():
    seen = 0
    for line in _golden_lines("e2m1_values.txt"):
        code, val = line.split()
        assert _same(oracle.e2m1_to_f64(int(code)), float(val)), line
        seen += 1
    assert seen == 16


def test_e2m1_closed_form():
    # OCP e2m1: exponent bits e (bias 1), one mantissa bit m; e == 0 is subnormal
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        assert _same(oracle.e2m1_to_f64(c), -mag if s else mag)


def test_e8m0_and_overflow_facts():
    for line in _golden_lines("e8m0_facts.txt"):
        kind, sbyte, code, val = line.split()
        want = _parse_value(val)
        if kind == "scale":
            assert _same(oracle.e8m0_to_f64(int(sbyte)), want), line
        else:
            # one MXFP4 row of 32 values, value 0 carries `code`
            codes = np.zeros((1, 16), np.uint8)
            codes[0, 0] = int(code)
            w = oracle.Weight(oracle.MXFP4, (1, 32), codes, np.array([[int(sbyte)]], np.uint8))
            got = float(oracle.dequant(w, oracle.F32)[0, 0])
            assert _same(got, float(np.float32(want))), (line, got)
    for s in range(255):
        assert oracle.e8m0_to_f64(s) == math.ldexp(1.0, s - 127)


# ------------------------------------------------------------ float formats
def test_f16_decode_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode_array(bits, oracle.F16)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_bf16_decode_exhaustive_vs_torch():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode_array(bits, oracle.BF16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def _special_f32():
    g = np.random.default_rng(11)
    r = g.integers(0, 2**32, size=400_000, dtype=np.uint64).astype(np.uint32)
    # ties and near-ties for bf16 (low 16 bits 0x8000 +- 1) and f16 (low 13 bits)
    base = g.integers(0, 2**32, size=20_000, dtype=np.uint64).astype(np.uint32)
    ties = np.concatenate([
        (base & 0xFFFF0000) | 0x8000, (base & 0xFFFF0000) | 0x7FFF, (base & 0xFFFF0000) | 0x8001,
        (base & 0xFFFFE000) | 0x1000, (base & 0xFFFFE000) | 0x0FFF, (base & 0xFFFFE000) | 0x1001,
    ]).astype(np.uint32)
    specials = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0x00000001,
                         0x007FFFFF, 0x00800000, 0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0x477FE000,
                         0x477FEFFF, 0x477FF000, 0x33800000, 0x33000000, 0x33000001, 0x387FC000,
                         0x38800000], dtype=np.uint32)
    return np.concatenate([r, ties, specials]).view(np.float32)


def test_round_to_bf16_vs_torch():
    f = _special_f32()
    got = oracle.round_array(f, oracle.BF16)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x7F) != 0)


def test_round_to_f16_vs_numpy():
    f = _special_f32()
    got = oracle.round_array(f, oracle.F16)
    with np.errstate(over="ignore"):
        want = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)


# ------------------------------------------------------------ packing order
def test_packing_worked_examples():
    n = 0
    for line in _golden_lines("packing_examples.txt"):
        head, _, tail = line.partition(":")
        f = head.split()
        if f[0] == "affine":
            bits = int(f[1])
            words = np.array([int(h, 16) for h in f[2:]], dtype=np.uint32)
            codes = [int(c) for c in tail.split()]
            got = [oracle.affine_code(words, bits, i) for i in range(len(codes))]
            assert got == codes, line
        elif f[0] == "mxfp4":
            b = np.array([int(f[1], 16)], dtype=np.uint8)
            lo, hi = (int(c) for c in tail.split())
            assert (oracle.mxfp4_code(b, 0), oracle.mxfp4_code(b, 1)) == (lo, hi), line
        elif f[0] == "q8_0":
            hdr = bytes.fromhex(f[1])
            d = float(f[2])
            q = np.arange(-16, 16, dtype=np.int8)
            blk = np.frombuffer(hdr + q.tobytes(), dtype=np.uint8).reshape(1, 34).copy()
            w = oracle.Weight(oracle.Q8_0, (1, 32), blk)
            got = oracle.dequant(w, oracle.F32)[0].astype(np.float64)
            assert np.array_equal(got, d * q.astype(np.float64)), line
        elif f[0] == "mxfp4_blocks":
            blk = np.frombuffer(bytes.fromhex(f[1] + f[2]), dtype=np.uint8).reshape(1, 17).copy()
            codes = [int(c) for c in tail.split()]
            w = oracle.Weight(oracle.MXFP4_BLOCKS, (1, 32), blk)
            got = oracle.dequant(w, oracle.F32)[0]
            table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # the page's magnitudes
            scale = 2.0 ** (int(f[1], 16) - 127)
            want = [(-1.0 if c & 8 else 1.0) * table[c & 7] * scale for c in codes]
            assert all(_same(float(a), b) for a, b in zip(got, want)), line
        n += 1
    assert n >= 17


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_pack_unpack_round_trip(bits):
    g = np.random.default_rng(bits)
    k = 256
    codes = g.integers(0, 1 << bits, size=k)
    stream = 0
    for i, c in enumerate(codes):
        stream |= int(c) << (i * bits)
    words = np.array([(stream >> (32 * t)) & 0xFFFFFFFF for t in range(k * bits // 32)],
                     dtype=np.uint32)
    got = np.array([oracle.affine_code(words, bits, i) for i in range(k)])
    assert np.array_equal(got, codes)


def test_mxfp4_nibble_order_in_a_row():
    # value 2i in byte i's low nibble, 2i+1 in its high one
    codes = np.array([[0x21, 0x43, 0x65, 0x07] + [0] * 12], dtype=np.uint8)
    w = oracle.Weight(oracle.MXFP4, (1, 32), codes, np.array([[127]], np.uint8))
    v = oracle.dequant(w, oracle.F32)[0, :8]
    assert list(v) == [0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 0.0]


# ------------------------------------------------------------ dequant
def test_affine_unit_scale_returns_codes():
    g = np.random.default_rng(5)
    for bits in (4, 8):
        w = synth.affine_weight(g, 8, 128, bits=bits, group_size=64)
        w["scales"][:] = 0x3F80  # 1.0
        w["biases"][:] = 0
        v = oracle.dequant(to_oracle(w), oracle.F32)
        per = 32 // bits
        words = w["codes"].astype(np.uint64)
        want = np.stack([(words >> (bits * t)) & ((1 << bits) - 1) for t in range(per)], -1)
        assert np.array_equal(v, want.reshape(8, 128).astype(np.float32))


@pytest.mark.parametrize("bits", [2, 3, 5, 6])
def test_affine_cross_word_widths_dequant(bits):
    # "GPTQModel wiki: MLX Apple Silicon", "Packed layouts and exact transcoding":
    # widths that do not divide 32 continue one little-endian bit stream across
    # words. Codes packed here by a Python integer stream; value = code*scale + bias.
    g = np.random.default_rng(20 + bits)
    rows, k, gs = 6, 256, 64
    codes = g.integers(0, 1 << bits, size=(rows, k))
    words = np.empty((rows, k * bits // 32), np.uint32)
    for r in range(rows):
        stream = 0
        for i, c in enumerate(codes[r]):
            stream |= int(c) << (i * bits)
        words[r] = [(stream >> (32 * t)) & 0xFFFFFFFF for t in range(k * bits // 32)]
    one = np.full((rows, k // gs), 0x3F80, np.uint16)   # bf16 1.0
    zero = np.zeros((rows, k // gs), np.uint16)
    w = oracle.Weight(oracle.AFFINE, (rows, k), words, one, zero, bits=bits, group_size=gs)
    assert np.array_equal(oracle.dequant(w, oracle.F32), codes.astype(np.float32))
    sc = synth.normal_bf16(g, (rows, k // gs), 0.02)
    bi = synth.normal_bf16(g, (rows, k // gs), 0.02)
    w = oracle.Weight(oracle.AFFINE, (rows, k), words, sc, bi, bits=bits, group_size=gs)
    s64 = torch.from_numpy(sc.view(np.int16)).view(torch.bfloat16).double().numpy()
    b64 = torch.from_numpy(bi.view(np.int16)).view(torch.bfloat16).double().numpy()
    want = (codes * np.repeat(s64, gs, axis=1) + np.repeat(b64, gs, axis=1)).astype(np.float32)
    assert np.array_equal(oracle.dequant(w, oracle.F32), want)


def test_affine_reconstruction_per_group():
    # value = code * scale + bias with the group's scale and bias: checked in
    # float64 (exact for these magnitudes), rounded once to float32
    g = np.random.default_rng(6)
    for bits, gs in ((4, 32), (4, 64), (4, 128), (8, 64)):
        w = synth.affine_weight(g, 16, 256, bits=bits, group_size=gs)
        v = oracle.dequant(to_oracle(w), oracle.F32)
        words = w["codes"].astype(np.uint64)
        per = 32 // bits
        codes = np.stack([(words >> (bits * t)) & ((1 << bits) - 1) for t in range(per)], -1)
        codes = codes.reshape(16, 256).astype(np.float64)
        s = torch.from_numpy(w["scales"].view(np.int16)).view(torch.bfloat16).double().numpy()
        b = torch.from_numpy(w["biases"].view(np.int16)).view(torch.bfloat16).double().numpy()
        want = (codes * np.repeat(s, gs, axis=1) + np.repeat(b, gs, axis=1)).astype(np.float32)
        assert np.array_equal(v, want), (bits, gs)


def test_affine_f16_scales():
    g = np.random.default_rng(7)
    w = synth.affine_weight(g, 4, 64, bits=8, group_size=32)
    s = (np.abs(g.standard_normal(w["scales"].shape)) * 0.01).astype(np.float16)
    b = (g.standard_normal(w["biases"].shape) * 0.01).astype(np.float16)
    w["scales"], w["biases"], w["scale_dtype"] = s.view(np.uint16), b.view(np.uint16), "f16"
    v = oracle.dequant(to_oracle(w), oracle.F32)
    codes = np.stack([(w["codes"].astype(np.uint64) >> (8 * t)) & 255 for t in range(4)], -1)
    codes = codes.reshape(4, 64).astype(np.float64)
    want = codes * np.repeat(s.astype(np.float64), 32, 1) + np.repeat(b.astype(np.float64), 32, 1)
    assert np.array_equal(v, want.astype(np.float32))


def test_mxfp4_exhaustive_codes_and_scales():
    # one row: 256 groups (scale bytes 0..255), each holding codes 0..15 twice
    k = 32 * 256
    codes = np.tile(np.array([(2 * i % 16) | (((2 * i + 1) % 16) << 4) for i in range(16)],
                             np.uint8), 256).reshape(1, k // 2)
    scales = np.arange(256, dtype=np.uint8).reshape(1, 256)
    w = oracle.Weight(oracle.MXFP4, (1, k), codes, scales)
    table = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    want = np.empty(k, np.float64)
    for i in range(k):
        c, s = i % 16, i // 32
        mag = table[c & 7] * 2.0 ** (s - 127) if s < 255 else math.nan
        want[i] = -mag if c & 8 else mag
    with np.errstate(over="ignore"):
        want32 = want.astype(np.float32)
    got = oracle.dequant(w, oracle.F32)[0]
    nan = np.isnan(want32)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want32[~nan].view(np.uint32))
    # bf16 holds every finite value exactly; f16 rounds once from float32
    got_bf = oracle.dequant(w, oracle.BF16)[0]
    want_bf = torch.from_numpy(want32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_bf[~nan], want_bf[~nan])
    assert np.array_equal(torch.from_numpy(want_bf.view(np.int16)).view(torch.bfloat16)
                          .float().numpy()[~nan], want32[~nan])
    got_h = oracle.dequant(w, oracle.F16)[0]
    with np.errstate(over="ignore"):
        want_h = want32.astype(np.float16).view(np.uint16)
    assert np.array_equal(got_h[~nan], want_h[~nan])


def test_q8_0_exhaustive_scales_and_quants():
    # every float16 scale pattern times every int8 quant: d * q is exact in float32
    d = np.arange(65536, dtype=np.uint16)
    q = np.arange(-128, 128, dtype=np.int16).astype(np.int8)
    blocks = np.empty((65536, 8, 34), np.uint8)
    blocks[:, :, 0] = (d & 0xFF)[:, None]
    blocks[:, :, 1] = (d >> 8)[:, None]
    blocks[:, :, 2:] = q.view(np.uint8).reshape(8, 32)[None]
    w = oracle.Weight(oracle.Q8_0, (65536, 256), blocks.reshape(65536, 272))
    got = oracle.dequant(w, oracle.F32)
    with np.errstate(invalid="ignore", over="ignore"):
        want = (d.view(np.float16).astype(np.float64)[:, None] * q.astype(np.float64)[None])
        want32 = want.astype(np.float32)
    nan = np.isnan(want32)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want32[~nan].view(np.uint32))
    assert np.array_equal(want32[~nan].astype(np.float64), want[~nan])  # exactness


def test_zero_bytes_decode_to_zero():
    for fmt, codes, scales, biases in (
        (oracle.AFFINE, np.zeros((2, 8), np.uint32), np.zeros((2, 1), np.uint16),
         np.zeros((2, 1), np.uint16)),
        (oracle.Q8_0, np.zeros((2, 68), np.uint8), None, None),
        (oracle.MXFP4, np.zeros((2, 32), np.uint8), np.zeros((2, 2), np.uint8), None),
        (oracle.MXFP4_BLOCKS, np.zeros((2, 34), np.uint8), None, None),
    ):
        k = 64
        w = oracle.Weight(fmt, (2, k), codes, scales, biases, bits=4, group_size=64)
        assert not np.any(oracle.dequant(w, oracle.F32))


def _blocks_to_apart(blocks, k):
    # GGUF's blocks ("Nx_quant", "Weights", Mxfp4_blocks: the scale byte, then
    # byte j holding value j low and value j + 16 high) to the scales-apart
    # layout (Mxfp4: value 2i low and 2i + 1 high in byte i), by NumPy indexing
    rows = blocks.shape[0]
    b = blocks.reshape(rows, k // 32, 17)
    scales = b[:, :, 0].copy()
    body = b[:, :, 1:]
    codes = np.concatenate([body & 0xF, body >> 4], axis=2).reshape(rows, k)  # value order
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scales


def test_mxfp4_blocks_transcode_identity():
    # GGUF's blocks and the scales-apart layout hold the same values; the two
    # decoders read different byte positions, so a wrong nibble, byte or scale
    # position in either shows up as a mismatch
    g = np.random.default_rng(17)
    rows, k = 64, 256
    blocks = g.integers(0, 256, size=(rows, k // 32 * 17), dtype=np.int64).astype(np.uint8)
    b = blocks.reshape(rows, k // 32, 17)
    b[:, :, 0] = g.integers(100, 140, size=(rows, k // 32))  # finite scales ...
    b[0, 0, 0], b[1, 3, 0], b[2, 5, 0] = 255, 0, 254         # ... and the edges
    packed, scales = _blocks_to_apart(blocks, k)
    wb = oracle.Weight(oracle.MXFP4_BLOCKS, (rows, k), blocks)
    wa = oracle.Weight(oracle.MXFP4, (rows, k), packed, scales)
    for dt in (oracle.F32, oracle.BF16, oracle.F16):
        a, c = oracle.dequant(wb, dt), oracle.dequant(wa, dt)
        if dt == oracle.F32:
            nan = np.isnan(a)
            assert np.array_equal(nan, np.isnan(c)) and nan[0, :32].all() and not nan[0, 32:].any()
            assert np.array_equal(a[~nan].view(np.uint32), c[~nan].view(np.uint32))
        else:
            assert np.array_equal(a, c)
    x = synth.activations(g, 3, k)
    with np.errstate(invalid="ignore", over="ignore"):
        ya, yc = oracle.apply(wb, x), oracle.apply(wa, x)
    assert np.array_equal(np.isnan(ya), np.isnan(yc))
    ok = ~np.isnan(ya)
    assert np.array_equal(ya[ok], yc[ok])


def test_q8_0_to_affine_transcode_identity():
    # "GPTQModel wiki: MLX Apple Silicon", "Packed layouts and exact transcoding":
    # Q8_0 maps to 8-bit affine, group 32, code = q + 128, bias = -128 d. The
    # two decoders are independent, and must give the same float32 values.
    g = np.random.default_rng(8)
    wq = synth.q8_0_weight(g, 32, 256)
    blk = wq["codes"].reshape(32, 8, 34)
    d = blk[:, :, 0].astype(np.uint16) | (blk[:, :, 1].astype(np.uint16) << 8)
    q = blk[:, :, 2:].view(np.int8).astype(np.int64).reshape(32, 256)
    c = (q + 128).astype(np.uint64).reshape(32, 64, 4)
    words = (c[..., 0] | (c[..., 1] << 8) | (c[..., 2] << 16) | (c[..., 3] << 24)).astype(np.uint32)
    bias = (-128.0 * d.view(np.float16).astype(np.float64)).astype(np.float16)
    wa = oracle.Weight(oracle.AFFINE, (32, 256), words, d, bias.view(np.uint16), bits=8,
                       group_size=32, scale_dtype=oracle.F16)
    a = oracle.dequant(wa, oracle.F32)
    b = oracle.dequant(to_oracle(wq), oracle.F32)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_quantize_q8_0_round_trip():
    # "Nx_quant", "val quantize_q8_0": d = amax/127 stored at float16, quants
    # round(v * (1/d)) halves away from zero at float32. Dequant lands within
    # half a step of the input.
    g = np.random.default_rng(9)
    x = g.standard_normal((8, 128)).astype(np.float32)
    xb = x.reshape(8, 4, 32)
    amax = np.abs(xb).max(-1)
    d16 = (amax / np.float32(127)).astype(np.float16)
    inv = (np.float32(1) / d16.astype(np.float32))
    prod = xb * inv[..., None]
    q = (np.sign(prod) * np.floor(np.abs(prod) + np.float32(0.5))).astype(np.int8)
    blocks = np.concatenate([d16.view(np.uint8).reshape(8, 4, 2), q.view(np.uint8)], -1)
    w = oracle.Weight(oracle.Q8_0, (8, 128), blocks.reshape(8, 136))
    v = oracle.dequant(w, oracle.F32).reshape(8, 4, 32)
    step = d16.astype(np.float32)[..., None]
    assert np.all(np.abs(v - xb) <= 0.5 * step * 1.002 + 1e-7)


def _q8_block(x32):
    b = oracle.quantize_q8_0(np.asarray(x32, np.float32).reshape(1, 32))[0]
    return int(b[0]) | (int(b[1]) << 8), b[2:].view(np.int8)


def test_quantize_q8_0_stated_cases():
    # "Nx_quant", "val quantize_q8_0": d = amax / 127 stored at float16 rounded
    # to nearest; quants round(v * (1/d)), halves away from zero; 0 where d is 0
    x = np.zeros(32, np.float32)
    x[:6] = [127.0, 2.5, -2.5, 0.5, -0.5, 126.5]    # d = 1 exactly
    h, q = _q8_block(x)
    assert h == 0x3C00 and list(q[:6]) == [127, 3, -3, 1, -1, 127] and not q[6:].any()
    h, q = _q8_block(np.zeros(32))                 # d = 0: zero bytes
    assert h == 0 and not q.any()
    # 1/d infinite (amax below about 127 * 2^-128): zero bytes, which decode to +0.
    tiny = np.zeros(32, np.float32)
    tiny[3] = np.float32(1e-39)
    h, q = _q8_block(tiny)
    assert h == 0 and not q.any()
    # an infinity: scale +inf, quants 0, whatever its sign
    for s in (1.0, -1.0):
        xi = np.linspace(-1, 1, 32).astype(np.float32)
        xi[7] = s * np.inf
        h, q = _q8_block(xi)
        assert h == 0x7C00 and not q.any()
    # a NaN: a NaN scale and quants 0, an infinity in the block or not
    for extra in (False, True):
        xn = np.linspace(-1, 1, 32).astype(np.float32)
        xn[31] = np.nan
        if extra:
            xn[0] = np.inf
        h, q = _q8_block(xn)
        assert (h & 0x7C00) == 0x7C00 and (h & 0x3FF) != 0 and not q.any()
    # d past float16's largest: the scale is +inf, the quants as usual
    big = np.zeros(32, np.float32)
    big[0], big[1] = 127.0 * 70000.0, -63.5 * 70000.0
    h, q = _q8_block(big)
    assert h == 0x7C00 and q[0] == 127 and q[1] == -64


def test_quantize_q8_0_fixed_point_on_exact_blocks():
    # x = d * q with a float16 d and |q| reaching 127: amax / 127 is d exactly,
    # v * (1/d) lands within an ulp of q, so quantizing gives the same bytes back
    g = np.random.default_rng(12)
    rows, k = 16, 256
    d = (np.abs(g.standard_normal((rows, k // 32))) * 0.01 + 1e-3).astype(np.float16)
    q = g.integers(-127, 128, size=(rows, k // 32, 32)).astype(np.int8)
    q[:, :, 5] = np.where(g.random((rows, k // 32)) < 0.5, 127, -127)
    x = (d.astype(np.float32)[..., None] * q.astype(np.float32)).reshape(rows, k)
    blocks = np.concatenate([d.view(np.uint8).reshape(rows, k // 32, 2), q.view(np.uint8)], -1)
    assert np.array_equal(oracle.quantize_q8_0(x), blocks.reshape(rows, k // 32 * 34))


def test_quantize_q8_0_dequant_within_half_a_step():
    # the quants round v / d at float32 (half a step), and the stored d is d
    # rounded to float16 (a relative 2^-11), which moves a decoded value by at
    # most 127 * 2^-11 steps more
    g = np.random.default_rng(13)
    x = (g.standard_normal((8, 512)) * np.exp(g.standard_normal((8, 1)))).astype(np.float32)
    blocks = oracle.quantize_q8_0(x)
    v = oracle.dequant(oracle.Weight(oracle.Q8_0, x.shape, blocks), oracle.F32).reshape(8, 16, 32)
    d = blocks.reshape(8, 16, 34)[:, :, :2].copy().view(np.float16).astype(np.float32)
    err = np.abs(v - x.reshape(8, 16, 32))
    assert np.all(err <= (0.5 + 127 * 2.0 ** -11) * d * 1.002 + 1e-7)
    assert err.max() > 0.5 * d.min()  # the bound is not vacuous


# ------------------------------------------------------------ take
@pytest.mark.parametrize("kind", ["affine", "q8_0", "mxfp4"])
def test_take_commutes_with_dequant(kind):
    g = np.random.default_rng(10)
    mk = {"affine": lambda lead: synth.affine_weight(g, 12, 128, lead=lead),
          "q8_0": lambda lead: synth.q8_0_weight(g, 12, 128, lead=lead),
          "mxfp4": lambda lead: synth.mxfp4_weight(g, 12, 128, lead=lead)}[kind]
    for lead, axis in (((), 0), ((3,), 0), ((3,), 1), ((2, 3), 1)):
        w = to_oracle(mk(lead))
        L = w.shape[axis]
        ids = np.array([L - 1, 0, -1, L, 2, 2, -L], dtype=np.int64)
        t = oracle.take(w, axis, ids)
        got = oracle.dequant(t, oracle.F32)
        full = oracle.dequant(w, oracle.F32)
        inr = (ids >= 0) & (ids < L)
        want = np.take(full, np.where(inr, ids, 0), axis=axis)
        mask_shape = [1] * want.ndim
        mask_shape[axis] = ids.size
        want = np.where(inr.reshape(mask_shape), want, 0.0)
        assert np.array_equal(got, want), (kind, lead, axis)
        for name, part in t.parts().items():
            if part is not None:
                zero = np.take(part, np.where(~inr)[0], axis=axis)
                assert not np.any(zero), name


def test_take_rejects_last_axis():
    w = to_oracle(synth.mxfp4_weight(np.random.default_rng(1), 4, 64))
    with pytest.raises(ValueError):
        oracle.take(w, 1, np.array([0], np.int32))
    with pytest.raises(ValueError):
        oracle.take(w, -1, np.array([0], np.int32))


# ------------------------------------------------------------ products
FORMATS = ["affine4", "affine8", "q8_0", "mxfp4"]


def _weight(kind, g, n, k, lead=()):
    if kind == "affine4":
        return synth.affine_weight(g, n, k, bits=4, group_size=64, lead=lead)
    if kind == "affine8":
        return synth.affine_weight(g, n, k, bits=8, group_size=32, lead=lead)
    if kind == "q8_0":
        return synth.q8_0_weight(g, n, k, lead=lead)
    return synth.mxfp4_weight(g, n, k, lead=lead)


@pytest.mark.parametrize("kind", FORMATS)
def test_one_hot_input_returns_a_column(kind):
    g = np.random.default_rng(12)
    n, k = 5, 64
    w = to_oracle(_weight(kind, g, n, k))
    v = oracle.dequant(w, oracle.F32)
    x = np.zeros((k, k), np.uint16)
    x[np.arange(k), np.arange(k)] = 0x3F80  # bf16 1.0 on the diagonal: x row m = e_m
    y = oracle.apply(w, x)
    assert np.array_equal(y, v.T.astype(np.float64))


@pytest.mark.parametrize("kind", FORMATS)
def test_product_vs_torch_float64(kind):
    g = np.random.default_rng(13)
    n, k, M = 7, 192, 3  # n != k: a transposed operand cannot pass
    w = to_oracle(_weight(kind, g, n, k))
    x = synth.activations(g, M, k)
    y = oracle.apply(w, x)
    v = torch.from_numpy(oracle.dequant(w, oracle.F32)).double()
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double()
    want = torch.matmul(xd, v.T).numpy()
    assert y.shape == (M, n)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)
    ent = oracle.apply_entries(w, x, [0, 2, 1], [6, 0, 3])
    assert np.allclose(ent, [want[0, 6], want[2, 0], want[1, 3]], rtol=1e-12, atol=1e-12)



def test_apply_entries_rejects_bad_indices():
    # the C routine reads the index arrays and x's rows unchecked: mismatched
    # or out-of-range indices are refused before it runs
    g = synth.rng(77)
    w = to_oracle(synth.q8_0_weight(g, 8, 64))
    x = synth.activations(g, 3, 64)
    with pytest.raises(ValueError):
        oracle.apply_entries(w, x, [0, 1, 2], [0, 1])
    with pytest.raises(ValueError):
        oracle.apply_entries(w, x, [3], [0])
    with pytest.raises(ValueError):
        oracle.apply_entries(w, x, [0], [8])

def test_product_all_ones_codes_zero_bias():
    # codes all 1, bias 0: y = sum over groups of s_g * (sum of x over the group)
    g = np.random.default_rng(14)
    n, k, gs = 3, 256, 64
    w = synth.affine_weight(g, n, k, bits=4, group_size=gs)
    w["codes"][:] = 0x11111111
    w["biases"][:] = 0
    x = synth.activations(g, 2, k)
    y = oracle.apply(to_oracle(w), x)
    s = torch.from_numpy(w["scales"].view(np.int16)).view(torch.bfloat16).double().numpy()
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    xg = xd.reshape(2, k // gs, gs).sum(-1)
    assert np.allclose(y, xg @ s.T, rtol=1e-13, atol=1e-13)


def test_product_brute_force_tiny():
    # n = 2, k = 32, M = 1: the sum written out term by term from hand-chosen codes
    codes = np.zeros((2, 16), np.uint8)
    codes[0, 0] = 0x92   # v0 = 1.0, v1 = -0.5 (code 9)
    codes[1, 15] = 0x70  # v30 = 0, v31 = 6
    w = oracle.Weight(oracle.MXFP4, (2, 32), codes, np.array([[128], [126]], np.uint8))
    xf = np.zeros(32, np.float32)
    xf[0], xf[1], xf[31] = 3.0, 2.0, -1.5
    x = synth.to_bf16_bits(xf).reshape(1, 32)
    y = oracle.apply(w, x)
    assert y[0, 0] == 2.0 * (1.0 * 3.0 + (-0.5) * 2.0)
    assert y[0, 1] == 0.5 * (6.0 * -1.5)


# ------------------------------------------------------------ routing
def test_route_brute_force():
    g = np.random.default_rng(15)
    for E, T, topk in ((4, 7, 2), (32, 64, 4), (1, 5, 1)):
        ids = synth.expert_ids(g, T, topk, E).astype(np.int64)
        ids.reshape(-1)[::5] = -1
        ids.reshape(-1)[1::7] = E
        counts, offsets, perm, n_out = oracle.route(ids, E)
        flat = ids.reshape(-1)
        inr = (flat >= 0) & (flat < E)
        assert n_out == int((~inr).sum())
        assert np.array_equal(counts, np.bincount(flat[inr], minlength=E))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        assert sorted(perm.tolist()) == np.where(inr)[0].tolist()
        keys = [(int(flat[p]), int(p)) for p in perm]
        assert keys == sorted(keys)


# ------------------------------------------------------------ apply_experts
def test_experts_single_expert_reduces_to_apply():
    g = np.random.default_rng(16)
    w = synth.mxfp4_weight(g, 6, 64, lead=(1,))
    x = synth.activations(g, 5, 64)
    ids = np.zeros((5, 1), np.int32)
    y = oracle.apply_experts(to_oracle(w), ids, x)
    w2 = dict(w, shape=(6, 64), codes=w["codes"][0], scales=w["scales"][0])
    assert np.array_equal(y[:, 0, :], oracle.apply(to_oracle(w2), x))


def test_experts_out_of_range_gives_zeros_whatever_x_holds():
    g = np.random.default_rng(17)
    w = to_oracle(synth.mxfp4_weight(g, 6, 64, lead=(3,)))
    x = synth.activations(g, 2, 64)
    x[1, :] = 0x7FC0  # NaN row
    ids = np.array([[0, 3], [-1, 7]], np.int64)
    y = oracle.apply_experts(w, ids, x)
    assert np.all(y[0, 1] == 0) and np.all(y[1] == 0) and np.all(np.signbit(y[1]) == 0)
    assert np.all(np.isfinite(y[0, 0]))


def test_experts_row_independent_of_other_positions():
    g = np.random.default_rng(18)
    w = to_oracle(synth.mxfp4_weight(g, 8, 64, lead=(4,)))
    x = synth.activations(g, 6, 64)
    ids = synth.expert_ids(g, 6, 2, 4)
    y = oracle.apply_experts(w, ids, x)
    ids2 = ids.copy()
    ids2[1:] = np.roll(ids2[1:], 1, axis=1)
    y2 = oracle.apply_experts(w, ids2, x)
    assert np.array_equal(y[0], y2[0])


def test_experts_broadcast_equals_repeated_rows():
    g = np.random.default_rng(19)
    w = to_oracle(synth.affine_weight(g, 8, 128, lead=(3,)))
    x = synth.activations(g, 4, 128)
    ids = synth.expert_ids(g, 4, 2, 3)
    a = oracle.apply_experts(w, ids, x)
    b = oracle.apply_experts(w, ids, np.repeat(x, 2, axis=0))
    assert np.array_equal(a, b)
    for t in range(4):
        for j in range(2):
            sub = oracle.Weight(w.fmt, (8, 128), w.codes[ids[t, j]], w.scales[ids[t, j]],
                                w.biases[ids[t, j]], bits=4, group_size=64)
            assert np.array_equal(a[t, j], oracle.apply(sub, x[t:t + 1])[0])


def test_experts_entries_are_per_matrix_products():
    # sampled entries of apply_experts: entry (p, j) is row j of expert
    # ids[p]'s matrix against p's row of x -- the product of apply on that one
    # matrix (pinned above against torch.matmul) -- and zero where ids[p] is out
    # of range, whatever x holds
    g = np.random.default_rng(20)
    E, n, k, T, topk = 3, 7, 96, 5, 2
    w = to_oracle(synth.affine_weight(g, n, k, bits=4, group_size=32, lead=(E,)))
    x = synth.activations(g, T, k)
    x[4] = 0x7FC0  # NaN row, used only by out-of-range positions below
    ids = synth.expert_ids(g, T, topk, E)
    ids[4] = (-1, E)
    p_idx = np.array([0, 1, 3, 5, 8, 9, 2, 6])
    j_idx = np.array([0, 6, 3, 2, 5, 1, 4, 0])
    ent = oracle.apply_experts_entries(w, ids, x, p_idx, j_idx)
    for e, (p, j) in enumerate(zip(p_idx, j_idx)):
        t, s = divmod(int(p), topk)
        eid = int(ids[t, s])
        if not 0 <= eid < E:
            assert ent[e] == 0 and not np.signbit(ent[e])
            continue
        sub = oracle.Weight(w.fmt, (n, k), w.codes[eid], w.scales[eid], w.biases[eid], bits=4,
                            group_size=32)
        assert ent[e] == oracle.apply(sub, x[t:t + 1])[0, j]
    # per-position rows of x (x_rows = T * topk) pick row p, not row p // topk
    xp = synth.activations(g, T * topk, k)
    ent2 = oracle.apply_experts_entries(w, ids, xp, p_idx[:4], j_idx[:4])
    for e in range(4):
        t, s = divmod(int(p_idx[e]), topk)
        eid = int(ids[t, s])
        sub = oracle.Weight(w.fmt, (n, k), w.codes[eid], w.scales[eid], w.biases[eid], bits=4,
                            group_size=32)
        assert ent2[e] == oracle.apply(sub, xp[p_idx[e]:p_idx[e] + 1])[0, j_idx[e]]


# ------------------------------------------------------------ Q4_K and Q6_K
# "Nx_quant (raven-ml.dev API docs)", "Weights": Q4_K is 144 bytes per 256
# values (float16 d and dmin, 12 bytes of 6-bit scales and mins for eight
# sub-blocks of 32, 128 bytes of 4-bit quants), value d * sc * q - dmin * m;
# Q6_K is 210 bytes per 256 values (128 bytes of low 4 bits, 64 of high 2
# bits, sixteen int8 scales of sub-blocks of 16, float16 d), value
# d * sc * (q - 32). The arrangement inside the fields is ggml's block layout
# (the page names it); the packers below write it from the description,
# independently of the oracle's readers.
def _pack_q4_k(d, dmin, sc, m, q):
    """One Q4_K block from d, dmin (float16 bit patterns), scales and mins [8]
    (0..63) and quants [256] (0..15)."""
    blk = np.zeros(144, np.uint8)
    blk[0], blk[1], blk[2], blk[3] = d & 0xFF, d >> 8, dmin & 0xFF, dmin >> 8
    s = np.zeros(12, np.int64)
    for j in range(8):
        if j < 4:  # six bits in bytes 0..3 (scale) and 4..7 (min)
            s[j] |= sc[j] & 63
            s[4 + j] |= m[j] & 63
        else:      # low four bits in a nibble of bytes 8..11, top two on bytes 0..7's top bits
            s[8 + j - 4] |= (sc[j] & 15) | ((m[j] & 15) << 4)
            s[j - 4] |= (sc[j] >> 4) << 6
            s[j] |= (m[j] >> 4) << 6
    blk[4:16] = s.astype(np.uint8)
    for c in range(4):  # run c: values 64c .. 64c+31 low nibbles, 64c+32 .. 64c+63 high ones
        for l in range(32):
            blk[16 + 32 * c + l] = q[64 * c + l] | (q[64 * c + 32 + l] << 4)
    return blk


def _pack_q6_k(d, sc, q):
    """One Q6_K block from d (float16 bits), int8 scales [16] and quants [256] (0..63)."""
    blk = np.zeros(210, np.uint8)
    for h in range(2):
        for t in range(4):
            for l in range(32):
                v = q[128 * h + 32 * t + l]
                i = 64 * h + l + 32 * (t % 2)
                blk[i] |= (v & 15) << (4 if t >= 2 else 0)
                blk[128 + 32 * h + l] |= (v >> 4) << (2 * t)
    blk[192:208] = np.asarray(sc, np.int8).view(np.uint8)
    blk[208], blk[209] = d & 0xFF, d >> 8
    return blk


def _f16(v):
    return int(np.float16(v).view(np.uint16))


def test_k_quants_zero_block_decodes_to_zeros():
    # the page: a block of zero bytes decodes to zeros, -0. in Q6_K
    for fmt, nb, neg in ((oracle.Q4_K, 144, False), (oracle.Q6_K, 210, True)):
        w = oracle.Weight(fmt, (3, 512), np.zeros((3, 2 * nb), np.uint8))
        v = oracle.dequant(w, oracle.F32)
        assert np.all(v == 0) and np.all(np.signbit(v) == neg), fmt


def test_q4_k_values_from_the_fields():
    # every sub-block with its own scale and min (the 6-bit ranges' edges
    # included) and quants covering 0..15: value i = d * sc[i // 32] * q[i] -
    # dmin * m[i // 32], rounded once to float32
    g = np.random.default_rng(40)
    for trial in range(20):
        sc = g.integers(0, 64, 8)
        m = g.integers(0, 64, 8)
        if trial == 0:
            sc[:] = [0, 63, 1, 62, 32, 31, 48, 15]
            m[:] = [63, 0, 62, 1, 31, 32, 15, 48]
        q = g.integers(0, 16, 256)
        d = float(np.float16(abs(g.standard_normal()) * 0.01))
        dmin = float(np.float16(abs(g.standard_normal()) * 0.01))
        blk = _pack_q4_k(_f16(d), _f16(dmin), sc, m, q)
        v = oracle.dequant(oracle.Weight(oracle.Q4_K, (1, 256), blk[None]), oracle.F32)[0]
        j = np.arange(256) // 32
        want = (d * sc[j] * q - dmin * m[j]).astype(np.float32)  # exact in float64, one rounding
        assert np.array_equal(v.view(np.uint32), want.view(np.uint32)), trial


def test_q6_k_values_from_the_fields():
    g = np.random.default_rng(41)
    for trial in range(20):
        sc = g.integers(-128, 128, 16)
        q = g.integers(0, 64, 256)
        if trial == 0:
            sc[:] = [-128, 127, 0, 1, -1, 64, -64, 5, 7, -9, 100, -100, 2, 3, 4, 6]
            q[:64] = np.arange(64)
        d = float(np.float16(abs(g.standard_normal()) * 0.001))
        blk = _pack_q6_k(_f16(d), sc, q)
        v = oracle.dequant(oracle.Weight(oracle.Q6_K, (1, 256), blk[None]), oracle.F32)[0]
        want = (d * sc[np.arange(256) // 16] * (q - 32.0)).astype(np.float32)
        assert np.array_equal(v.view(np.uint32), want.view(np.uint32)), trial


def test_q4_k_to_affine_transcode_identity():
    # "GPTQModel wiki: MLX Apple Silicon", "Packed layouts and exact
    # transcoding": Q4_K is affine 4-bit with groups of 32, scale d * sc and
    # bias -dmin * m. With d and dmin powers of two both are exact in bfloat16,
    # and the affine decoder (another code path) must give the same bits.
    g = np.random.default_rng(42)
    rows, k = 6, 512
    blocks, qs, scl, bia = [], [], [], []
    for r in range(rows):
        rb = []
        for b in range(k // 256):
            sc, m, q = g.integers(0, 64, 8), g.integers(0, 64, 8), g.integers(0, 16, 256)
            d, dmin = 2.0 ** int(g.integers(-14, 0)), 2.0 ** int(g.integers(-14, 0))
            rb.append(_pack_q4_k(_f16(d), _f16(dmin), sc, m, q))
            qs.append(q)
            scl.extend(d * sc)
            bia.extend(-dmin * m)
        blocks.append(np.concatenate(rb))
    q = np.concatenate(qs).reshape(rows, k).astype(np.uint64)
    words = np.zeros((rows, k // 8), np.uint64)
    for i in range(8):
        words |= q[:, i::8] << np.uint64(4 * i)
    wa = oracle.Weight(oracle.AFFINE, (rows, k), words.astype(np.uint32),
                       synth.to_bf16_bits(np.array(scl, np.float32)).reshape(rows, k // 32),
                       synth.to_bf16_bits(np.array(bia, np.float32)).reshape(rows, k // 32), bits=4, group_size=32)
    wk = oracle.Weight(oracle.Q4_K, (rows, k), np.stack(blocks))
    a, b = oracle.dequant(wa, oracle.F32), oracle.dequant(wk, oracle.F32)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_q6_k_to_affine_transcode_identity():
    # Q6_K as affine 6-bit with groups of 16: code q, scale d * sc, bias
    # -32 * d * sc; exact in bfloat16 for d a power of two
    g = np.random.default_rng(43)
    rows, k = 5, 512
    blocks, qs, scl = [], [], []
    for r in range(rows):
        rb = []
        for b in range(k // 256):
            sc, q = g.integers(-128, 128, 16), g.integers(0, 64, 256)
            d = 2.0 ** int(g.integers(-14, -2))
            rb.append(_pack_q6_k(_f16(d), sc, q))
            qs.append(q)
            scl.extend(d * sc)
        blocks.append(np.concatenate(rb))
    q = np.concatenate(qs).reshape(rows, k)
    bits = ((q[:, :, None] >> np.arange(6)) & 1).reshape(rows, k * 6)  # little-endian stream
    words = (bits.reshape(rows, -1, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(axis=2)
    s = np.array(scl, np.float32).reshape(rows, k // 16)
    wa = oracle.Weight(oracle.AFFINE, (rows, k), words.astype(np.uint32), synth.to_bf16_bits(s),
                       synth.to_bf16_bits(-32.0 * s), bits=6, group_size=16)
    wk = oracle.Weight(oracle.Q6_K, (rows, k), np.stack(blocks))
    a, b = oracle.dequant(wa, oracle.F32), oracle.dequant(wk, oracle.F32)
    same = (a.view(np.uint32) == b.view(np.uint32)) | ((a == 0) & (b == 0))  # (q - 32) * 0 is -0. in Q6_K
    assert same.all()
