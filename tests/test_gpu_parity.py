"""Parity of the CUDA path (through the C entry points) with the oracle.

Dequant, take and routing must match bit for bit (NaN payloads aside);
products must meet the stated bound element by element (see
wutil.check_product) and the relative Frobenius bound.
"""
import numpy as np
import pytest
import torch

import oracle
import packed_qmatmul_gb300 as qm
from packed_qmatmul_gb300 import synth
from wutil import bf16_to_f64, check_product, row_norms, to_oracle

pytestmark = pytest.mark.gpu

ODT = {torch.float32: oracle.F32, torch.bfloat16: oracle.BF16, torch.float16: oracle.F16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from packed_qmatmul_gb300 import build

    build.build()
    qm.load_library()
    torch.cuda.set_device(0)


def _host(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> NumPy with the same bytes (16-bit floats as uint16)."""
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _bits_equal(a: np.ndarray, b: np.ndarray, dt) -> bool:
    """Equal bit patterns, with every NaN equal to every other NaN."""
    if dt == torch.float32:
        fa, fb = a.astype(np.float32), b.astype(np.float32)
        nan = np.isnan(fa)
        return np.array_equal(nan, np.isnan(fb)) and np.array_equal(fa[~nan].view(np.uint32),
                                                                     fb[~nan].view(np.uint32))
    ea = (a & 0x7F80) == 0x7F80 if dt == torch.bfloat16 else (a & 0x7C00) == 0x7C00
    ma = (a & 0x7F) != 0 if dt == torch.bfloat16 else (a & 0x3FF) != 0
    eb = (b & 0x7F80) == 0x7F80 if dt == torch.bfloat16 else (b & 0x7C00) == 0x7C00
    mb = (b & 0x7F) != 0 if dt == torch.bfloat16 else (b & 0x3FF) != 0
    na, nb = ea & ma, eb & mb
    return np.array_equal(na, nb) and np.array_equal(a[~na], b[~nb])


KINDS = ["affine4_g32", "affine4_g64", "affine4_g128", "affine8_g32", "affine8_g64",
         "affine8_g128", "q8_0", "mxfp4"]


def _make(kind, g, n, k, lead=()):
    if kind.startswith("affine"):
        bits = int(kind[6])
        gs = int(kind.split("_g")[1])
        return synth.affine_weight(g, n, k, bits=bits, group_size=gs, lead=lead)
    if kind == "q8_0":
        return synth.q8_0_weight(g, n, k, lead=lead)
    return synth.mxfp4_weight(g, n, k, lead=lead)


# ---------------------------------------------------------------- dequant
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16])
def test_dequant_bit_exact(kind, dt):
    g = synth.rng(100)
    for n, k, lead in ((37, 256, ()), (5, 1024, (3,)), (1, 128, (2, 2))):
        w = _make(kind, g, n, k, lead)
        got = _host(qm.dequant(qm.QWeight.from_arrays(w), dt))
        want = oracle.dequant(to_oracle(w), ODT[dt])
        assert _bits_equal(got, want, dt), (kind, n, k, lead)


def test_dequant_config1_seed0():
    w, _ = synth.small_affine_config(0)
    got = _host(qm.dequant(qm.QWeight.from_arrays(w), torch.bfloat16))
    assert np.array_equal(got, oracle.dequant(to_oracle(w), oracle.BF16))


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16])
def test_dequant_mxfp4_every_code_and_scale(dt):
    k = 32 * 256
    codes = np.tile(np.array([(2 * i % 16) | (((2 * i + 1) % 16) << 4) for i in range(16)], np.uint8),
                    256).reshape(1, k // 2)
    scales = np.arange(256, dtype=np.uint8).reshape(1, 256)
    w = dict(format="mxfp4", shape=(1, k), codes=codes, scales=scales, biases=None)
    got = _host(qm.dequant(qm.QWeight.from_arrays(w), dt))
    assert _bits_equal(got, oracle.dequant(to_oracle(w), ODT[dt]), dt)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16])
def test_dequant_q8_0_every_scale_and_quant(dt):
    d = np.arange(65536, dtype=np.uint16)
    q = np.arange(-128, 128, dtype=np.int16).astype(np.int8)
    blocks = np.empty((65536, 8, 34), np.uint8)
    blocks[:, :, 0] = (d & 0xFF)[:, None]
    blocks[:, :, 1] = (d >> 8)[:, None]
    blocks[:, :, 2:] = q.view(np.uint8).reshape(8, 32)[None]
    w = dict(format="q8_0", shape=(65536, 256), codes=blocks.reshape(65536, 272))
    got = _host(qm.dequant(qm.QWeight.from_arrays(w), dt))
    assert _bits_equal(got, oracle.dequant(to_oracle(w), ODT[dt]), dt)


# ---------------------------------------------------------------- take
@pytest.mark.parametrize("kind", ["affine4_g64", "affine8_g32", "q8_0", "mxfp4"])
@pytest.mark.parametrize("id64", [False, True])
def test_take_packed_and_dense(kind, id64):
    g = synth.rng(200)
    for lead, axis in (((), 0), ((3,), 0), ((3,), 1), ((2, 3), 1)):
        w = _make(kind, g, 24, 256, lead)
        ow = to_oracle(w)
        L = ow.shape[axis]
        ids = np.array([L - 1, 0, -1, L, 2, 2, -L, 1, L + 7], dtype=np.int64 if id64 else np.int32)
        tw, dense = qm.take(qm.QWeight.from_arrays(w), axis, torch.from_numpy(ids).cuda(),
                            dense_dtype=torch.bfloat16)
        ot = oracle.take(ow, axis, ids)
        for name, part in (("codes", tw.codes), ("scales", tw.scales), ("biases", tw.biases)):
            want = ot.parts()[name]
            if want is None:
                assert part is None
                continue
            assert np.array_equal(_host(part).view(np.uint8).reshape(-1),
                                  want.view(np.uint8).reshape(-1)), (kind, lead, axis, name)
        assert np.array_equal(_host(dense), oracle.dequant(ot, oracle.BF16)), (kind, lead, axis)


def test_take_embedding_shape():
    # the embedding-table shape, scaled down: affine 4-bit gs64, k = 1024
    g = synth.rng(4)
    w = synth.affine_weight(g, 4096, 1024, bits=4, group_size=64)
    ids = synth.uniform_ids(g, 512, 4096)
    tw, dense = qm.take(qm.QWeight.from_arrays(w), 0, torch.from_numpy(ids).cuda(),
                        dense_dtype=torch.bfloat16)
    ot = oracle.take(to_oracle(w), 0, ids)
    assert np.array_equal(_host(tw.codes).view(np.uint32), ot.codes)
    assert np.array_equal(_host(dense), oracle.dequant(ot, oracle.BF16))


# ---------------------------------------------------------------- products
def _check_apply(w, x, what):
    ow = to_oracle(w)
    y = qm.apply(qm.QWeight.from_arrays(w), _dev_bf16(x))
    got = bf16_to_f64(_host(y))
    ref = oracle.apply(ow, x)
    xn = np.linalg.norm(oracle.decode_array(x, oracle.BF16), axis=1)
    return check_product(got, ref, row_norms(ow), xn, ow.k, what)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 16])
def test_apply_decode(kind, M):
    g = synth.rng(300 + M)
    for n, k in ((48, 256), (300, 512), (17, 1024)):
        w = _make(kind, g, n, k)
        x = synth.activations(g, M, k)
        _check_apply(w, x, f"{kind} M={M} n={n} k={k}")


@pytest.mark.parametrize("M", [1, 8])
def test_apply_config1_seed0(M):
    w, xs = synth.small_affine_config(0)
    _check_apply(w, xs[M], f"config1 M={M}")


@pytest.mark.parametrize("kind", ["affine4_g64", "affine8_g64", "q8_0", "mxfp4"])
def test_apply_split_k(kind):
    # few rows, long k: the decode path splits k over a cluster
    g = synth.rng(400)
    for n, k, M in ((64, 4096, 1), (40, 14336, 4), (1024, 3072, 2)):
        w = _make(kind, g, n, k)
        x = synth.activations(g, M, k)
        _check_apply(w, x, f"{kind} split n={n} k={k} M={M}")


@pytest.mark.parametrize("kind", ["affine4_g64", "q8_0", "mxfp4"])
def test_apply_larger_m(kind):
    g = synth.rng(500)
    for n, k, M in ((64, 256, 17), (96, 512, 33)):
        w = _make(kind, g, n, k)
        x = synth.activations(g, M, k)
        _check_apply(w, x, f"{kind} n={n} k={k} M={M}")


def test_apply_activation_range():
    # activations far from 1 in magnitude: the power-of-two rescale keeps them exact
    g = synth.rng(600)
    w = _make("affine4_g64", g, 64, 512)
    for sigma in (1e-30, 1e-6, 1e4, 1e30):
        x = synth.activations(g, 4, 512, sigma=sigma)
        _check_apply(w, x, f"sigma={sigma}")


@pytest.mark.parametrize("M", [1, 8, 16])
def test_apply_mxfp4_scale_range(M):
    # e8m0 scales over the range a product stays finite in: row r < 201 has
    # every group at scale byte r (from 2^-127, below float32's normal range,
    # up to 2^73), the rows after it mix them; three rows hold one group at
    # 255, which makes every value of the group NaN and so the row's outputs
    g = synth.rng(650 + M)
    n, k = 256, 512
    w = synth.mxfp4_weight(g, n, k)
    sc = np.empty((n, k // 32), np.uint8)
    sc[:201] = np.arange(201, dtype=np.uint8)[:, None]
    sc[201:] = g.integers(0, 201, size=(n - 201, k // 32))
    nanrows = [7, 150, 230]
    for r, grp in zip(nanrows, (0, 9, 15)):
        sc[r, grp] = 255
    w["scales"] = sc
    x = synth.activations(g, M, k)
    ow = to_oracle(w)
    got = bf16_to_f64(_host(qm.apply(qm.QWeight.from_arrays(w), _dev_bf16(x))))
    ref = oracle.apply(ow, x)
    assert np.all(np.isnan(ref[:, nanrows])) and np.all(np.isnan(got[:, nanrows]))
    keep = np.setdiff1d(np.arange(n), nanrows)
    xn = np.linalg.norm(oracle.decode_array(x, oracle.BF16), axis=1)
    check_product(got[:, keep], ref[:, keep], row_norms(ow)[keep], xn, k, f"mxfp4 scales M={M}")


def test_apply_deterministic():
    g = synth.rng(700)
    w = _make("q8_0", g, 256, 4096)
    qw = qm.QWeight.from_arrays(w)
    x = _dev_bf16(synth.activations(g, 4, 4096))
    a = _host(qm.apply(qw, x))
    b = _host(qm.apply(qw, x))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("n", [64, 1024])
def test_apply_static_weight_chain(M, n):
    # weights marked static are streamed before the previous kernel in the stream
    # ends; the activations, which that kernel writes, must still be read after it
    g = synth.rng(710 + M)
    k = n
    ws = [_make("affine4_g64", g, n, k) for _ in range(4)]
    x0 = synth.activations(g, M, k)
    ys = {}
    for flags in (0, qm.QM_WEIGHT_STATIC):
        qws = [qm.QWeight.from_arrays(w, flags=flags) for w in ws]
        x = _dev_bf16(x0)
        outs = []
        for qw in qws:  # each product reads the one before it, no sync between
            x = qm.apply(qw, x)
            outs.append(x)
        ys[flags] = [_host(o) for o in outs]
    for a, b in zip(ys[0], ys[qm.QM_WEIGHT_STATIC]):
        assert np.array_equal(a, b)
    xin = x0
    for i, w in enumerate(ws):
        ow = to_oracle(w)
        got = bf16_to_f64(ys[qm.QM_WEIGHT_STATIC][i])
        ref = oracle.apply(ow, xin)
        xn = np.linalg.norm(oracle.decode_array(xin, oracle.BF16), axis=1)
        check_product(got, ref, row_norms(ow), xn, k, f"static chain step {i}")
        xin = ys[qm.QM_WEIGHT_STATIC][i]


# ---------------------------------------------------------------- routing and experts
@pytest.mark.parametrize("id64", [False, True])
def test_route_bit_exact(id64):
    g = synth.rng(800)
    for E, T, topk in ((32, 64, 4), (8, 700, 2), (3, 5, 1), (256, 1024, 8)):
        ids = synth.expert_ids(g, T, topk, E).astype(np.int64 if id64 else np.int32)
        flat = ids.reshape(-1)
        flat[::7] = -1
        flat[3::11] = E + 3
        counts, offsets, perm = qm.route(torch.from_numpy(ids).cuda(), E)
        oc, oo, op, n_out = oracle.route(ids, E)
        assert np.array_equal(counts.cpu().numpy(), oc)
        assert np.array_equal(offsets.cpu().numpy(), oo)
        pm = perm.cpu().numpy()
        assert np.array_equal(pm[: oo[E]], op)
        out_pos = np.where((flat < 0) | (flat >= E))[0]
        assert np.array_equal(pm[oo[E]:], out_pos)


@pytest.mark.parametrize("kind", ["affine4_g64", "q8_0", "mxfp4"])
@pytest.mark.parametrize("broadcast", [True, False])
def test_apply_experts_small(kind, broadcast):
    g = synth.rng(900)
    E, n, k, T, topk = 4, 40, 256, 6, 2
    w = _make(kind, g, n, k, lead=(E,))
    ids = synth.expert_ids(g, T, topk, E)
    ids[1, 0] = -1
    ids[4, 1] = E
    x = synth.activations(g, T if broadcast else T * topk, k)
    if broadcast:
        x[1] = 0x7FC0  # NaN row: its in-range position sees it, the other gives zeros
    else:
        x[2] = 0x7FC0  # position (1, 0), out of range: zeros whatever the row holds
    ow = to_oracle(w)
    y = qm.apply_experts(qm.QWeight.from_arrays(w), torch.from_numpy(ids).cuda(), _dev_bf16(x))
    got = bf16_to_f64(_host(y)).reshape(T * topk, n)
    ref = oracle.apply_experts(ow, ids, x).reshape(T * topk, n)
    flat = ids.reshape(-1)
    out = (flat < 0) | (flat >= E)
    assert np.all(got[out] == 0) and not np.any(np.signbit(got[out]))
    ok = ~out & np.all(np.isfinite(ref), axis=1)
    rows = np.where(ok)[0]
    xr = rows // topk if broadcast else rows
    xn = np.linalg.norm(oracle.decode_array(x, oracle.BF16), axis=1)[xr]
    wn = row_norms(ow).reshape(E, n)[flat[rows]]
    bound = 1e-2 * xn[:, None] * wn / np.sqrt(k)
    err = np.abs(got[rows] - ref[rows])
    from wutil import bf16_half_ulp
    assert np.all(err <= bound + bf16_half_ulp(got[rows])), err.max()
    nanrows = ~out & ~np.all(np.isfinite(ref), axis=1)
    assert np.all(np.isnan(got[nanrows]))


def _check_experts(w, ids, x, what):
    """y of apply_experts against the oracle: zeros out of range, the product
    tolerance per in-range row; returns the device result [P, n] as float64."""
    E, n, k = w["shape"]
    T, topk = ids.shape
    ow = to_oracle(w)
    y = qm.apply_experts(qm.QWeight.from_arrays(w), torch.from_numpy(ids).cuda(), _dev_bf16(x))
    got = bf16_to_f64(_host(y)).reshape(T * topk, n)
    ref = oracle.apply_experts(ow, ids, x).reshape(T * topk, n)
    flat = ids.reshape(-1)
    out = (flat < 0) | (flat >= E)
    assert np.all(got[out] == 0) and not np.any(np.signbit(got[out])), what
    rows = np.where(~out)[0]
    xr = rows // topk if x.shape[0] == T else rows
    xn = np.linalg.norm(oracle.decode_array(x, oracle.BF16), axis=1)[xr]
    wn = row_norms(ow).reshape(E, n)[flat[rows]]
    check_product(got[rows], ref[rows], wn, xn, k, what)
    return got


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("T", [24, 160])
def test_apply_experts_chunks(kind, T):
    # experts with many positions (several chunks or tiles), empty experts,
    # positions out of range, per-token and per-position activations; T = 24
    # takes the decode path, T = 160 (over 32 positions per expert) the tensor cores
    g = synth.rng(910)
    E, n, k = 6, 100, 512
    w = _make(kind, g, n, k, lead=(E,))
    topk = 2
    ids = synth.expert_ids(g, T, topk, E)
    ids[:, 0] = 2           # expert 2: 24+ positions, more than one chunk
    ids[:, 1] = np.where(ids[:, 1] == 2, 5, ids[:, 1])
    ids[ids == 4] = 3       # expert 4 empty
    ids[3, 1] = -7
    ids[9, 1] = E
    for rows in (T, T * topk):
        x = synth.activations(g, rows, k)
        _check_experts(w, ids, x, f"{kind} x_rows={rows}")


def test_apply_experts_all_out_of_range():
    g = synth.rng(920)
    w = _make("mxfp4", g, 64, 256, lead=(4,))
    ids = np.full((5, 2), 9, dtype=np.int32)
    ids[0, 0] = -1
    y = qm.apply_experts(qm.QWeight.from_arrays(w), torch.from_numpy(ids).cuda(),
                         _dev_bf16(synth.activations(g, 5, 256)))
    h = _host(y)
    assert np.all(h.view(np.uint16) == 0)


@pytest.mark.parametrize("T", [16, 200])
def test_apply_experts_rows_independent_of_other_experts(T):
    # a row's bits depend on its own row and expert only (decode and tensor paths)
    g = synth.rng(930)
    E, n, k, topk = 8, 96, 512, 2
    w = _make("affine4_g64", g, n, k, lead=(E,))
    qw = qm.QWeight.from_arrays(w)
    x = _dev_bf16(synth.activations(g, T, k))
    ids1 = synth.expert_ids(g, T, topk, E)
    ids2 = ids1.copy()
    ids2[::3, 1] = (ids2[::3, 1] + 3) % E
    ids2[ids2[:, 0] == ids2[:, 1], 1] = (ids2[ids2[:, 0] == ids2[:, 1], 1] + 1) % E
    y1 = _host(qm.apply_experts(qw, torch.from_numpy(ids1).cuda(), x)).reshape(T * topk, n)
    y2 = _host(qm.apply_experts(qw, torch.from_numpy(ids2).cuda(), x)).reshape(T * topk, n)
    same = (ids1 == ids2).reshape(-1)
    assert same.sum() > 0 and (~same).sum() > 0
    assert np.array_equal(y1[same].view(np.uint16), y2[same].view(np.uint16))


@pytest.mark.parametrize("T", [64, 1024, 4096])
def test_apply_experts_moe_shape_sampled(T):
    # 32 MXFP4 experts [5760, 2880], T tokens x 4: every output row of a
    # sample of positions against the oracle
    w, ids, x = synth.moe_config(T)
    E, n, k = w["shape"]
    T, topk = ids.shape
    ow = to_oracle(w)
    y = qm.apply_experts(qm.QWeight.from_arrays(w), torch.from_numpy(ids).cuda(), _dev_bf16(x))
    got = bf16_to_f64(_host(y)).reshape(T * topk, n)
    pos = np.sort(synth.rng(940 + T).choice(T * topk, size=16, replace=False))
    sub_ids = ids.reshape(-1)[pos].reshape(-1, 1).astype(np.int32)
    sub_x = x[pos // topk]
    ref = oracle.apply_experts(ow, sub_ids, sub_x).reshape(len(pos), n)
    xn = np.linalg.norm(oracle.decode_array(sub_x, oracle.BF16), axis=1)
    used = np.unique(sub_ids[:, 0])
    sub_w = dict(w, shape=(len(used), n, k), codes=w["codes"][used], scales=w["scales"][used])
    wn = row_norms(to_oracle(sub_w)).reshape(len(used), n)[np.searchsorted(used, sub_ids[:, 0])]
    check_product(got[pos], ref, wn, xn, k, f"moe T={T} positions {pos.tolist()}")


@pytest.mark.parametrize("bits,gs", [(4, 64), (8, 32), (4, 128)])
def test_f16_scales_every_entry_point(bits, gs):
    # affine scales and biases stored as float16 (the other dtype the format
    # allows): dequant bit-exact, take, decode and tensor-core products, experts
    g = synth.rng(1220 + bits + gs)
    n, k = 200, 1024
    w = synth.affine_weight(g, n, k, bits=bits, group_size=gs, scale_dtype="f16")
    ow = to_oracle(w)
    qw = qm.QWeight.from_arrays(w)
    for dt in (torch.bfloat16, torch.float16, torch.float32):
        got = _host(qm.dequant(qw, dt))
        assert _bits_equal(got, oracle.dequant(ow, ODT[dt]), dt), dt
    ids = synth.uniform_ids(g, 50, n)
    tw, dense = qm.take(qw, 0, torch.from_numpy(ids).cuda(), dense_dtype=torch.bfloat16)
    ot = oracle.take(ow, 0, ids)
    for name, part in (("codes", tw.codes), ("scales", tw.scales), ("biases", tw.biases)):
        assert np.array_equal(_host(part).view(np.uint8).reshape(-1),
                              ot.parts()[name].view(np.uint8).reshape(-1)), name
    assert np.array_equal(_host(dense), oracle.dequant(ot, oracle.BF16))
    for M in (1, 3, 16, 64, 200):
        x = synth.activations(g, M, k)
        _check_apply(w, x, f"f16 scales bits={bits} gs={gs} M={M}")
    E = 4
    we = synth.affine_weight(g, 96, 512, bits=bits, group_size=gs, lead=(E,), scale_dtype="f16")
    for T in (6, 80):  # decode path, then the tensor cores
        ide = synth.expert_ids(g, T, 2, E)
        _check_experts(we, ide, synth.activations(g, T, 512), f"f16 scales experts T={T}")


# ---------------------------------------------------------------- long pipelines
@pytest.mark.parametrize("kind,n,k", [("affine4_g64", 40000, 1024), ("affine8_g32", 20000, 512),
                                      ("q8_0", 12000, 1024), ("mxfp4", 30000, 256)])
@pytest.mark.parametrize("M", [1, 3])
def test_apply_many_stages_per_cta(kind, n, k, M):
    # many more stages per CTA than shared-memory slots: slots are refilled
    # several times while different teams work on them
    g = synth.rng(1000 + M)
    w = _make(kind, g, n, k)
    x = synth.activations(g, M, k)
    _check_apply(w, x, f"{kind} n={n} k={k} M={M}")


def test_apply_lm_head_shape_sampled():
    # the full lm_head shape (151936 x 1024, affine 4-bit gs64) at M = 1,
    # checked on sampled outputs the oracle computes one by one
    g = synth.rng(1100)
    w = synth.affine_weight(g, 151936, 1024, bits=4, group_size=64)
    x = synth.activations(g, 1, 1024)
    ow = to_oracle(w)
    y = bf16_to_f64(_host(qm.apply(qm.QWeight.from_arrays(w), _dev_bf16(x))))[0]
    j = np.unique(np.concatenate([g.integers(0, 151936, 3000), [0, 1, 151935, 151904]]))
    ref = oracle.apply_entries(ow, x, np.zeros_like(j), j)
    wn = np.array([np.linalg.norm(oracle.row_values(ow, int(r)).astype(np.float64)) for r in j])
    xn = np.linalg.norm(oracle.decode_array(x, oracle.BF16), axis=1)
    check_product(y[j][None], ref[None], wn, xn, 1024, "lm_head sampled")


# ---------------------------------------------------------------- prefill (tensor cores)
@pytest.mark.parametrize("kind", KINDS)
def test_apply_prefill(kind):
    # several weight and token tiles along both axes (token tiles of 128 or
    # 256), ragged M and n, k not a multiple of 256
    g = synth.rng(1200)
    for n, k, M in ((200, 512, 130), (256, 1024, 64), (130, 384, 257), (136, 512, 192), (130, 384, 385)):
        if kind == "q8_0" and k % 256:
            k = 512  # Q8_0 rows must be 16-byte multiples for the TMA path
        w = _make(kind, g, n, k)
        x = synth.activations(g, M, k)
        _check_apply(w, x, f"{kind} prefill n={n} k={k} M={M}")


@pytest.mark.parametrize("kind", ["affine4_g64", "affine8_g32", "q8_0", "mxfp4"])
def test_apply_prefill_split_k(kind):
    # few weight tiles and a long k: a cluster splits k and adds its partial
    # sums across CTAs (ragged M and n included)
    g = synth.rng(1210)
    for n, k, M in ((256, 4096, 17), (200, 4096, 64), (384, 2048, 128), (130, 8192, 100)):
        w = _make(kind, g, n, k)
        x = synth.activations(g, M, k)
        _check_apply(w, x, f"{kind} split-k n={n} k={k} M={M}")


def test_apply_prefill_split_k_deterministic():
    g = synth.rng(1211)
    qw = qm.QWeight.from_arrays(synth.q8_0_weight(g, 512, 4096))
    x = _dev_bf16(synth.activations(g, 96, 4096))
    a = _host(qm.apply(qw, x))
    b = _host(qm.apply(qw, x))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("n,k", [(4096, 4096), (14336, 4096), (4096, 14336)])
def test_apply_prefill_q8_0_full_shape_sampled(n, k):
    # the Q8_0 prefill shapes at M = 2048, in the launch configuration the
    # benchmark times, checked on sampled outputs (tile corners included)
    g = synth.rng(1201 + n + k)
    w = synth.q8_0_weight(g, n, k)
    x = synth.activations(g, 2048, k)
    ow = to_oracle(w)
    y = bf16_to_f64(_host(qm.apply(qm.QWeight.from_arrays(w), _dev_bf16(x))))
    m_idx = np.concatenate([g.integers(0, 2048, 2000), [0, 2047, 127, 128, 191, 192, 383, 384, 1919, 1920]])
    j_idx = np.concatenate([g.integers(0, n, 2000), [0, n - 1, 128, 127, n - 128, 129, 1, 255, 256, n - 129]])
    ref = oracle.apply_entries(ow, x, m_idx, j_idx)
    wn = np.array([np.linalg.norm(oracle.row_values(ow, int(r)).astype(np.float64)) for r in j_idx])
    xn = np.linalg.norm(oracle.decode_array(x[m_idx], oracle.BF16), axis=1)
    got = y[m_idx, j_idx]
    bound = 1e-2 * xn * wn / np.sqrt(k)
    from wutil import bf16_half_ulp
    assert np.all(np.abs(got - ref) <= bound + bf16_half_ulp(got)), np.max(np.abs(got - ref) / bound)
    assert np.linalg.norm(got - ref) <= 4e-3 * np.linalg.norm(ref)


def test_apply_q8_0_decode_full_shapes_sampled():
    # the Q8_0 shapes at M = 1 and 16 (the decode kernel, k split over clusters)
    g = synth.rng(1205)
    for n, k, M in ((14336, 4096, 1), (4096, 14336, 1), (4096, 4096, 16)):
        w = synth.q8_0_weight(g, n, k)
        x = synth.activations(g, M, k)
        ow = to_oracle(w)
        y = bf16_to_f64(_host(qm.apply(qm.QWeight.from_arrays(w), _dev_bf16(x))))
        j = np.unique(np.concatenate([g.integers(0, n, 1500), [0, 1, 31, 32, n - 1]]))
        m = g.integers(0, M, j.size)
        ref = oracle.apply_entries(ow, x, m, j)
        wn = np.array([np.linalg.norm(oracle.row_values(ow, int(r)).astype(np.float64)) for r in j])
        xn = np.linalg.norm(oracle.decode_array(x, oracle.BF16), axis=1)[m]
        from wutil import bf16_half_ulp
        got = y[m, j]
        bound = 1e-2 * xn * wn / np.sqrt(k)
        assert np.all(np.abs(got - ref) <= bound + bf16_half_ulp(got)), (n, k, M)
        assert np.linalg.norm(got - ref) <= 4e-3 * np.linalg.norm(ref)


def test_embedding_table_full_dequant_and_take():
    # the whole 151936 x 1024 affine 4-bit gs64 table: dequant to bf16 bit for
    # bit, and a take of 4096 uniform ids, packed and decoded, bit for bit
    g = synth.rng(5)
    w = synth.affine_weight(g, 151936, 1024, bits=4, group_size=64)
    ow = to_oracle(w)
    qw = qm.QWeight.from_arrays(w)
    got = _host(qm.dequant(qw, torch.bfloat16))
    want = oracle.dequant(ow, oracle.BF16)
    assert np.array_equal(got, want)
    del got
    ids = synth.uniform_ids(g, 4096, 151936)
    tw, dense = qm.take(qw, 0, torch.from_numpy(ids).cuda(), dense_dtype=torch.bfloat16)
    assert np.array_equal(_host(dense), want[ids])
    ot = oracle.take(ow, 0, ids)
    for name, part in (("codes", tw.codes), ("scales", tw.scales), ("biases", tw.biases)):
        assert np.array_equal(_host(part).view(np.uint8).reshape(-1), ot.parts()[name].view(np.uint8).reshape(-1))


# ---------------------------------------------------------------- MXFP4 in GGUF's blocks
# "Nx_quant", "Weights", Mxfp4_blocks: per 32 values the scale byte, then byte j
# holding value j low and value j + 16 high. Dequant and take decode it in their
# own kernels; products run the plain per-row kernels.
def _blocks(g, n, k, lead=()):
    w = synth.mxfp4_blocks_weight(g, n, k, lead=lead)
    b = w["codes"].reshape(-1, 17)
    b[0, 0], b[1, 0], b[2, 0], b[3, 0] = 255, 0, 254, 1  # NaN, 2^-127, 2^127, 2^-126 groups
    return w


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16])
def test_mxfp4_blocks_dequant_bit_exact(dt):
    g = synth.rng(700)
    for n, k, lead in ((37, 256, ()), (5, 1024, (3,)), (1, 128, (2, 2))):
        w = _blocks(g, n, k, lead)
        got = _host(qm.dequant(qm.QWeight.from_arrays(w), dt))
        want = oracle.dequant(to_oracle(w), ODT[dt])
        assert _bits_equal(got, want, dt), (n, k, lead)


@pytest.mark.parametrize("id64", [False, True])
def test_mxfp4_blocks_take(id64):
    g = synth.rng(701)
    for lead, axis in (((), 0), ((3,), 0), ((3,), 1)):
        w = _blocks(g, 24, 256, lead)
        ow = to_oracle(w)
        L = ow.shape[axis]
        ids = np.array([L - 1, 0, -1, L, 2, 2, 1], dtype=np.int64 if id64 else np.int32)
        tw, dense = qm.take(qm.QWeight.from_arrays(w), axis, torch.from_numpy(ids).cuda(),
                            dense_dtype=torch.bfloat16)
        ot = oracle.take(ow, axis, ids)
        assert tw.scales is None and tw.biases is None
        assert np.array_equal(_host(tw.codes).view(np.uint8).reshape(-1), ot.codes.reshape(-1)), (lead, axis)
        assert _bits_equal(_host(dense), oracle.dequant(ot, oracle.BF16), torch.bfloat16), (lead, axis)


@pytest.mark.parametrize("M", [1, 2, 8, 16, 33, 130])
def test_mxfp4_blocks_apply(M):
    # k a multiple of 512: M <= 16 streams the 17-byte blocks through the
    # tensor-map GEMV (one CTA per stage, a k split over a cluster, many stages
    # per CTA), M >= 17 decodes them for the tensor cores (128- and 256-token tiles)
    g = synth.rng(702 + M)
    for n, k in ((80, 512), (64, 4096), (9000, 512)):
        w = synth.mxfp4_blocks_weight(g, n, k)
        _check_apply(w, synth.activations(g, M, k), f"mxfp4 blocks n={n} k={k} M={M}")


def test_mxfp4_blocks_one_token_full_shape_sampled():
    # 14336 x 4096 in GGUF blocks (31 MB) at M = 1: the tensor-map GEMV, checked
    # on sampled outputs the oracle computes one by one
    g = synth.rng(706)
    w = synth.mxfp4_blocks_weight(g, 14336, 4096)
    x = synth.activations(g, 1, 4096)
    ow = to_oracle(w)
    y = bf16_to_f64(_host(qm.apply(qm.QWeight.from_arrays(w), _dev_bf16(x))))[0]
    j = np.unique(np.concatenate([g.integers(0, 14336, 1500), [0, 1, 14335]]))
    ref = oracle.apply_entries(ow, x, np.zeros_like(j), j)
    wn = np.array([np.linalg.norm(oracle.row_values(ow, int(r)).astype(np.float64)) for r in j])
    xn = np.linalg.norm(oracle.decode_array(x, oracle.BF16), axis=1)
    check_product(y[j][None], ref[None], wn, xn, 4096, "mxfp4 blocks 14336x4096 sampled")


def test_mxfp4_blocks_apply_experts():
    g = synth.rng(705)
    w = synth.mxfp4_blocks_weight(g, 48, 256, lead=(4,))
    ids = synth.expert_ids(g, 16, 2, 4).astype(np.int32)
    ids[3, 1] = 4   # out of range: zeros
    ids[7, 0] = -1
    _check_experts(w, ids, synth.activations(g, 16, 256), "mxfp4 blocks experts")
    # k a multiple of 512: the grouped tensor-map GEMV
    w = synth.mxfp4_blocks_weight(g, 64, 512, lead=(8,))
    ids = synth.expert_ids(g, 24, 2, 8).astype(np.int32)
    ids[5, 0] = 8
    _check_experts(w, ids, synth.activations(g, 24, 512), "mxfp4 blocks experts k=512")
    # more than 32 positions per expert: the grouped tensor-core GEMM
    w = synth.mxfp4_blocks_weight(g, 160, 1024, lead=(4,))
    ids = synth.expert_ids(g, 96, 2, 4).astype(np.int32)
    ids[9, 1] = -1
    _check_experts(w, ids, synth.activations(g, 96, 1024), "mxfp4 blocks experts tensor path")


# ---------------------------------------------------------------- quantize_q8_0
def _quantize_cases(g, rows, k):
    x = (g.standard_normal((rows, k)) * np.exp(2 * g.standard_normal((rows, 1)))).astype(np.float32)
    b = x.reshape(rows, k // 32, 32)
    b[0, 0] = 0.0                                 # d = 0
    b[0, 1, :] = 0.0; b[0, 1, 4] = 1e-39          # 1/d past float32's range: zero bytes
    b[0, 2, 7] = np.inf; b[0, 3, 9] = -np.inf     # infinities: scale +inf, quants 0
    b[0, 4, 31] = np.nan; b[0, 5, 0] = np.nan; b[0, 5, 1] = np.inf   # NaN, with and without inf
    b[0, 6, :] = 0.0; b[0, 6, :6] = [127.0, 2.5, -2.5, 0.5, -0.5, 126.5]   # halves away from zero
    b[0, 7] *= np.float32(1e6)                     # d past float16's largest
    b[1] *= np.float32(1e-5)                       # float16 subnormal scales
    b[2] *= np.float32(1e-30)                      # scales below float16's range: stored as 0
    b[3, :, :] = -b[3, :, :1]                      # blocks of one repeated value
    return x


def test_quantize_q8_0_bit_exact():
    # "Nx_quant", val quantize_q8_0: the blocks' bytes, every stated case included
    g = np.random.default_rng(800)
    rows, k = 48, 512
    x = _quantize_cases(g, rows, k)
    want = oracle.quantize_q8_0(x)
    got = qm.quantize_q8_0(torch.from_numpy(x).cuda())
    assert np.array_equal(_host(got.codes), want)
    w = dict(format="q8_0", shape=(rows, k), codes=want)
    assert _bits_equal(_host(qm.dequant(got, torch.float32)), oracle.dequant(to_oracle(w), oracle.F32),
                       torch.float32)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_quantize_q8_0_reads_16_bit_inputs_at_float32(dt):
    # x of a 16-bit dtype is read at float32: the blocks equal the float32 case's
    g = np.random.default_rng(801)
    x = _quantize_cases(g, 40, 256)
    xt = torch.from_numpy(x).to(dt)
    want = oracle.quantize_q8_0(xt.float().numpy())
    got = qm.quantize_q8_0(xt.cuda())
    assert np.array_equal(_host(got.codes), want)


def test_quantize_q8_0_large_and_lead_axes():
    # a [3, 700, 4096] weight: many blocks per launch, leading axes flattened
    g = np.random.default_rng(802)
    x = g.standard_normal((3, 700, 4096)).astype(np.float32) * np.float32(0.02)
    got = qm.quantize_q8_0(torch.from_numpy(x).cuda())
    assert got.shape == (3, 700, 4096)
    assert np.array_equal(_host(got.codes).reshape(-1), oracle.quantize_q8_0(x.reshape(-1, 4096)).reshape(-1))


# ---------------------------------------------------------------- affine 2, 3, 5 and 6 bits
# "GPTQModel wiki: MLX Apple Silicon", "Packed layouts and exact transcoding":
# one little-endian bit stream per row, so 3-, 5- and 6-bit codes cross words.
WIDTHS = [2, 3, 5, 6]


@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("gs", [32, 64, 128])
def test_affine_widths_dequant_and_take(bits, gs):
    g = synth.rng(1500 + 10 * bits + gs)
    for n, k, lead in ((37, 256, ()), (5, 1024, (3,)), (3, 128, (2, 2))):
        w = synth.affine_weight(g, n, k, bits=bits, group_size=gs, lead=lead)
        ow = to_oracle(w)
        qw = qm.QWeight.from_arrays(w)
        for dt in (torch.float32, torch.bfloat16, torch.float16):
            assert _bits_equal(_host(qm.dequant(qw, dt)), oracle.dequant(ow, ODT[dt]), dt), (n, k, lead, dt)
        L = ow.shape[0]
        ids = np.array([L - 1, 0, -1, L, 2 % L, 1 % L], dtype=np.int32)
        tw, dense = qm.take(qw, 0, torch.from_numpy(ids).cuda(), dense_dtype=torch.bfloat16)
        ot = oracle.take(ow, 0, ids)
        for name, part in (("codes", tw.codes), ("scales", tw.scales), ("biases", tw.biases)):
            assert np.array_equal(_host(part).view(np.uint8).reshape(-1), ot.parts()[name].view(np.uint8).reshape(-1))
        assert np.array_equal(_host(dense), oracle.dequant(ot, oracle.BF16))


@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("M", [1, 3, 16, 33, 130])
def test_affine_widths_apply(bits, M):
    # M = 1: the one-token kernel; 3 and 16: the plain kernel; 33 and 130: the
    # tensor cores (k = 96 rows are no 16-byte multiple: the plain kernel)
    g = synth.rng(1600 + 10 * bits + M)
    for gs, n, k in ((32, 96, 512), (64, 200, 1024), (128, 130, 2048), (32, 40, 96)):
        w = synth.affine_weight(g, n, k, bits=bits, group_size=gs)
        _check_apply(w, synth.activations(g, M, k), f"affine{bits} gs{gs} n={n} k={k} M={M}")


@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("T", [12, 100])
def test_affine_widths_experts(bits, T):
    g = synth.rng(1700 + bits + T)
    E, n, k = 4, 72, 512
    w = synth.affine_weight(g, n, k, bits=bits, group_size=64, lead=(E,))
    ids = synth.expert_ids(g, T, 2, E)
    ids[2, 1] = -1
    _check_experts(w, ids, synth.activations(g, T, k), f"affine{bits} experts T={T}")


# ---------------------------------------------------------------- GGUF Q4_K and Q6_K
# "Nx_quant", "Weights": Q4_K (144-byte blocks of 256 values: d, dmin, 6-bit
# scales and mins, 4-bit quants) and Q6_K (210-byte blocks: 6-bit quants,
# int8 sub-block scales, d), each arranged as ggml's block layout.
def _kquant(kind, g, n, k, lead=()):
    w = (synth.q4_k_weight if kind == "q4_k" else synth.q6_k_weight)(g, n, k, lead=lead)
    nb = 144 if kind == "q4_k" else 210
    b = w["codes"].reshape(-1, nb)
    if b.shape[0] >= 6:  # special blocks: all zero bytes, an infinite d, a NaN d, a subnormal d
        b[0] = 0
        dpos = 0 if kind == "q4_k" else 208
        for i, d in ((1, 0x7C00), (2, 0x7E00), (3, 0x0001)):
            b[i, dpos], b[i, dpos + 1] = d & 0xFF, d >> 8
        if kind == "q4_k":
            b[4, 2], b[4, 3] = 0x00, 0xFC  # dmin = -inf
    return w


@pytest.mark.parametrize("kind", ["q4_k", "q6_k"])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16])
def test_kquant_dequant_bit_exact(kind, dt):
    g = synth.rng(1800)
    for n, k, lead in ((37, 256, ()), (5, 1024, (3,)), (2, 512, (2, 2))):
        w = _kquant(kind, g, n, k, lead)
        got = _host(qm.dequant(qm.QWeight.from_arrays(w), dt))
        assert _bits_equal(got, oracle.dequant(to_oracle(w), ODT[dt]), dt), (kind, n, k, lead)


@pytest.mark.parametrize("kind", ["q4_k", "q6_k"])
def test_kquant_take(kind):
    g = synth.rng(1801)
    for lead, axis in (((), 0), ((3,), 0), ((3,), 1)):
        w = _kquant(kind, g, 24, 512, lead)
        ow = to_oracle(w)
        L = ow.shape[axis]
        ids = np.array([L - 1, 0, -1, L, 2, 2, 1], dtype=np.int32)
        tw, dense = qm.take(qm.QWeight.from_arrays(w), axis, torch.from_numpy(ids).cuda(),
                            dense_dtype=torch.bfloat16)
        ot = oracle.take(ow, axis, ids)
        assert tw.scales is None and tw.biases is None
        assert np.array_equal(_host(tw.codes).view(np.uint8).reshape(-1), ot.codes.reshape(-1)), (lead, axis)
        assert _bits_equal(_host(dense), oracle.dequant(ot, oracle.BF16), torch.bfloat16), (lead, axis)


@pytest.mark.parametrize("kind", ["q4_k", "q6_k"])
@pytest.mark.parametrize("M", [1, 3, 16, 33, 130])
def test_kquant_apply(kind, M):
    g = synth.rng(1810 + M)
    for n, k in ((96, 256), (200, 1024), (33, 2048)):
        w = (synth.q4_k_weight if kind == "q4_k" else synth.q6_k_weight)(g, n, k)
        _check_apply(w, synth.activations(g, M, k), f"{kind} n={n} k={k} M={M}")


@pytest.mark.parametrize("kind", ["q4_k", "q6_k"])
@pytest.mark.parametrize("M", [1, 33])
def test_kquant_apply_nonfinite_scales(kind, M):
    # blocks whose d (or Q4_K's dmin) is infinite or NaN: the per-element values'
    # infinities and NaNs, compared exactly
    g = synth.rng(1820 + M)
    w = _kquant(kind, g, 64, 512)
    _check_apply(w, synth.activations(g, M, 512), f"{kind} special blocks M={M}")


@pytest.mark.parametrize("kind", ["q4_k", "q6_k"])
@pytest.mark.parametrize("T", [12, 100])
def test_kquant_experts(kind, T):
    g = synth.rng(1830 + T)
    E = 4
    w = (synth.q4_k_weight if kind == "q4_k" else synth.q6_k_weight)(g, 64, 512, lead=(E,))
    ids = synth.expert_ids(g, T, 2, E)
    ids[1, 0] = E
    _check_experts(w, ids, synth.activations(g, T, 512), f"{kind} experts T={T}")


@pytest.mark.parametrize("kind", ["q8_0", "mxfp4_blocks", "q6_k"])
def test_one_token_rows_off_word_boundaries(kind):
    # GGUF block rows of 102 or 170 (Q8_0), 51 or 85 (MXFP4 blocks) and 210 or
    # 630 (Q6_K) bytes: row starts fall on every byte offset within a word
    g = synth.rng(1900)
    shapes = ((37, 256), (9, 768)) if kind == "q6_k" else ((37, 96), (9, 160))
    for n, k in shapes:
        if kind == "q8_0":
            w = synth.q8_0_weight(g, n, k)
        elif kind == "mxfp4_blocks":
            w = synth.mxfp4_blocks_weight(g, n, k)
        else:
            w = synth.q6_k_weight(g, n, k)
        _check_apply(w, synth.activations(g, 1, k), f"{kind} n={n} k={k} M=1")


@pytest.mark.parametrize("kind", ["affine4_g64", "q8_0", "mxfp4"])
def test_one_token_long_and_ragged_k(kind):
    # the one-token kernel at long k (16 and 17 chunks of 1024 inputs), and a
    # k that ends inside a chunk
    g = synth.rng(2000)
    for n, k in ((40, 16384), (40, 16448), (33, 1088)):
        w = _make(kind, g, n, k)
        _check_apply(w, synth.activations(g, 1, k), f"{kind} n={n} k={k} M=1")


# ---------------------------------------------------------------- several weights, one x
def _many_kind(kind, g, n, k):
    if kind == "q4_k":
        return synth.q4_k_weight(g, n, k)
    if kind == "q6_k":
        return synth.q6_k_weight(g, n, k)
    if kind == "mxfp4_blocks":
        return synth.mxfp4_blocks_weight(g, n, k)
    if kind == "affine3_g64":
        return synth.affine_weight(g, n, k, bits=3, group_size=64)
    return _make(kind, g, n, k)


def _apply_many_vs_apply(arrays, M, g, static=True):
    flags = qm.QM_WEIGHT_STATIC if static else 0
    ws = [qm.QWeight.from_arrays(a, flags=flags) for a in arrays]
    k = arrays[0]["shape"][-1]
    x = synth.activations(g, M, k)
    xd = _dev_bf16(x)
    got = qm.apply_many(ws, xd)
    for w, y in zip(ws, got):
        want = qm.apply(w, xd)
        assert torch.equal(y.view(torch.int16), want.view(torch.int16)), w.shape
    return ws, x, got


@pytest.mark.parametrize("kind", ["affine4_g64", "affine8_g64", "affine3_g64", "q8_0", "mxfp4",
                                  "mxfp4_blocks", "q4_k", "q6_k"])
@pytest.mark.parametrize("M", [1, 3])
def test_apply_many_bit_identical_to_apply(kind, M):
    # at M = 1 the weights run as one grid; the outputs are those of one call per weight
    g = synth.rng(2100 + M)
    for shapes in (((2048, 1024), (1024, 1024), (1024, 1024)), ((17, 512), (300, 512), (1, 512), (64, 512))):
        _apply_many_vs_apply([_many_kind(kind, g, n, k) for n, k in shapes], M, g)


def test_apply_many_against_the_oracle():
    g = synth.rng(2200)
    arrays = [synth.affine_weight(g, n, 1024, bits=4, group_size=64) for n in (2048, 1024, 1024)]
    _, x, got = _apply_many_vs_apply(arrays, 1, g, static=False)
    for a, y in zip(arrays, got):
        ow = to_oracle(a)
        xn = np.linalg.norm(oracle.decode_array(x, oracle.BF16), axis=1)
        check_product(bf16_to_f64(_host(y)), oracle.apply(ow, x), row_norms(ow), xn, ow.k, "apply_many")


def test_apply_many_edge_cases():
    g = synth.rng(2300)
    # an empty weight among others; the most weights a call takes; one weight
    arrays = [synth.affine_weight(g, n, 256, bits=4, group_size=64) for n in (5, 0, 7, 1, 2, 3, 4, 9)]
    _apply_many_vs_apply(arrays, 1, g)
    _apply_many_vs_apply(arrays[:1], 1, g)
    # a weight above 24 MB keeps its own launch (the streaming GEMV), the others still agree
    big = [synth.affine_weight(g, 50000, 1024, bits=4, group_size=64),
           synth.affine_weight(g, 64, 1024, bits=4, group_size=64)]
    _apply_many_vs_apply(big, 1, g)
    # non-finite values (MXFP4 scale bytes 254/255) go element by element in the fused grid too
    w1 = synth.mxfp4_weight(g, 40, 256)
    w1["scales"][3, 2] = 254
    w1["scales"][7, 0] = 255
    w2 = synth.mxfp4_weight(g, 24, 256)
    ws, x, got = _apply_many_vs_apply([w1, w2], 1, g)
    ow = to_oracle(w1)
    xn = np.linalg.norm(oracle.decode_array(x, oracle.BF16), axis=1)
    check_product(bf16_to_f64(_host(got[0])), oracle.apply(ow, x), row_norms(ow), xn, ow.k, "many nonfinite")


@pytest.mark.parametrize("gs", [32, 64, 128])
@pytest.mark.parametrize("M", [2, 5, 8])
def test_register_mma_decode(gs, M):
    # affine 4-bit at 2..8 tokens: weight tiles in registers on mma.sync; every
    # k split (k = 256, 512, 1024 and up), ragged row counts, f16 scales, and a
    # weight tall enough that CTAs stride over tiles
    g = synth.rng(2400 + gs + M)
    for n, k in ((17, 256), (300, 512), (48, 1024), (40, 3072)):
        w = synth.affine_weight(g, n, k, bits=4, group_size=gs)
        _check_apply(w, synth.activations(g, M, k), f"gs{gs} n={n} k={k} M={M}")
    w = synth.affine_weight(g, 64, 1024, bits=4, group_size=gs, scale_dtype="f16")
    _check_apply(w, synth.activations(g, M, 1024), f"gs{gs} f16 scales M={M}")
    if gs == 64:
        w = synth.affine_weight(g, 40000, 512, bits=4, group_size=gs)
        _check_apply(w, synth.activations(g, M, 512), f"gs{gs} n=40000 M={M}")
