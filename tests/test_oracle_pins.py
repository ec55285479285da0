"""Pins for the CPU oracle: each check ties the oracle to something other than itself
(printed values, closed forms, library routines, brute force, invariants).
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import nvfp4_oracle as O

F32 = np.float32


# --------------------------------------------------------------------------- E2M1

def test_e2m1_decode_matches_format_table(golden):
    g = golden("e2m1_values.json")["codes_to_values"]
    got = O.e2m1_decode(np.arange(16))
    for code, val in g.items():
        assert got[int(code)] == val
        assert math.copysign(1.0, got[int(code)]) == math.copysign(1.0, val)


def _brute_e2m1(v: float) -> int:
    """argmin over the 8 magnitudes; on a tie pick the even code; sign from v."""
    mag = abs(v)
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    if mag > 6.0:
        best = 7
    else:
        dists = [abs(mag - g) for g in grid]
        dmin = min(dists)
        cands = [i for i, d in enumerate(dists) if d == dmin]
        even = [i for i in cands if i % 2 == 0]
        best = even[0] if even else cands[0]
    return best | (8 if math.copysign(1.0, v) < 0 else 0)


def test_e2m1_encode_brute_force_sweep(golden):
    g = golden("e2m1_values.json")
    rng = np.random.default_rng(0)
    mids = [float(k) for k in g["round_to_nearest_even_midpoints"]]
    vals = list(np.linspace(-7, 7, 2801)) + mids + [-m for m in mids]
    vals += list(rng.uniform(-8, 8, 5000)) + [0.0, -0.0, 1e-30, -1e-30, 6.0, 6.0001, 1e30, -1e30]
    # fp32 neighbours of every midpoint
    for m in mids:
        vals += [float(np.nextafter(F32(m), F32(0))), float(np.nextafter(F32(m), F32(10)))]
    v = np.array(vals, dtype=np.float32)
    got = O.e2m1_encode(v)
    want = np.array([_brute_e2m1(float(x)) for x in v], dtype=np.uint8)
    np.testing.assert_array_equal(got, want)
    for k, code in g["round_to_nearest_even_midpoints"].items():
        assert O.e2m1_encode(np.array([float(k)]))[0] == code
        assert O.e2m1_encode(np.array([-float(k)]))[0] == code | 8
    for k, code in g["saturation"].items():
        assert O.e2m1_encode(np.array([float(k)]))[0] == code


# --------------------------------------------------------------------------- E4M3

def test_ue4m3_decode_matches_format_table(golden):
    for b, val in golden("e4m3_values.json")["bytes_to_values"].items():
        assert O.ue4m3_decode(np.array([int(b)]))[0] == val


def test_ue4m3_decode_matches_torch_float8():
    b = np.arange(0, 127, dtype=np.uint8)  # every finite non-negative byte
    t = torch.from_numpy(b.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.ue4m3_decode(b), t)


def test_ue4m3_encode_matches_torch_float8():
    vals = O.ue4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(1)
    sweep = np.exp2(rng.uniform(-14, 10, 20000))
    s = np.concatenate([vals, mids, sweep, [0.0, 447.9, 448.0, 460.0, 1e9, np.inf]]).astype(np.float32)
    for x in mids.astype(np.float32):  # fp32 neighbours of each midpoint
        s = np.append(s, [np.nextafter(x, F32(0)), np.nextafter(x, F32(1e4))])
    want = torch.from_numpy(np.minimum(s, F32(448.0))).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.ue4m3_encode(s), want)


# --------------------------------------------------------------------------- bf16

def test_bf16_conversion_matches_torch():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(100000) * np.exp2(rng.uniform(-30, 30, 100000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(O.f32_to_bf16_bits(x), want)
    back = torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(O.bf16_bits_to_f32(want), back)


# --------------------------------------------------------------------------- global scale

def test_global_scale_examples(golden):
    for ex in golden("gs_examples.json")["examples"]:
        x = np.array([[ex["amax"], -ex["amax"] / 3] + [0.0] * 14], dtype=np.float32)
        assert O.global_scale(x) == F32(ex["gs"])
        assert O.quantize(x).gs == F32(ex["gs"])


def test_block_with_global_amax_gets_max_scale():
    rng = np.random.default_rng(3)
    for _ in range(50):
        x = (rng.standard_normal((8, 256)) * np.exp2(rng.uniform(-20, 20))).astype(np.float32)
        q = O.quantize(x)
        r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        assert q.sf[r, c // 16] == 0x7E  # 448


# --------------------------------------------------------------------------- quantiser

def _on_grid_tensor(rng, M, K, gs):
    """Codes drawn at random, every block holding a +-6 code, scales drawn at random."""
    codes = rng.integers(0, 16, (M, K)).astype(np.uint8)
    codes[:, ::16] = np.where(rng.random((M, K // 16)) < 0.5, 7, 15)
    sf = rng.integers(1, 127, (M, K // 16)).astype(np.uint8)
    return codes, sf, O.dequantize(codes, sf, gs).astype(np.float32)


def test_quantize_is_exact_on_grid():
    """quantize(dequantize(q)) == q when every block's max is a +-6 code (spec fixed point)."""
    rng = np.random.default_rng(4)
    for gs in [F32(1.0), F32(0.125), F32(2.0 ** -10)]:
        codes, sf, x = _on_grid_tensor(rng, 16, 256, gs)
        q = O.quantize(x, gs=gs)
        np.testing.assert_array_equal(q.sf, sf)
        # code 8 decodes to -0.0, whose sign the quantiser keeps: the round trip is the identity
        np.testing.assert_array_equal(q.codes, codes)


def test_quantize_error_bound():
    """|x - deq(q(x))| <= half the E2M1 grid step at |x/d| (or the saturation excess) times d."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 512)) * np.exp(rng.standard_normal((64, 1)))).astype(np.float32)
    x[:, 7] *= 30.0  # outlier channel
    q = O.quantize(x)
    d = np.repeat(O.ue4m3_decode(q.sf) * float(q.gs), 16, axis=1)
    y = x.astype(np.float64) / d
    a = np.abs(y)
    half_step = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))
    bound = np.where(a > 6, a - 6, half_step) * d * (1 + 1e-6)
    err = np.abs(x - O.dequantize(q.codes, q.sf, q.gs))
    assert np.all(err <= bound)
    # saturation only comes from the E4M3 rounding of the block scale (at most 2^-4 relative)
    assert a.max() <= 6.0 * (1 + 2.0 ** -4) * (1 + 1e-6)


def test_roundtrip_cosine_matches_page_precision(golden):
    g = golden("page_precision.json")
    rng = np.random.default_rng(6)
    x = rng.standard_normal((256, 7168)).astype(np.float32)
    q = O.quantize(x)
    c4 = O.cosine(O.dequantize(q.codes, q.sf, q.gs), x)
    assert abs(c4 - g["nvfp4_roundtrip_cosine"]) < 7e-4
    s = F32(np.abs(x).max() / 448)
    b = O.ue4m3_encode((np.abs(x) / s).astype(np.float32))
    c8 = O.cosine(np.sign(x) * O.ue4m3_decode(b) * s, x)
    assert abs(c8 - g["fp8_e4m3_roundtrip_cosine"]) < 1e-4


def test_quantize_zero_and_degenerate_blocks():
    x = np.zeros((2, 64), dtype=np.float32)
    q = O.quantize(x)
    assert q.gs == 0 and not q.sf.any() and not q.codes.any()
    x[1, 20] = 3.0  # one non-zero block; the others stay zero-coded
    q = O.quantize(x)
    assert q.sf[0].sum() == 0 and q.sf[1, 1] == 0x7E and q.sf[1, 0] == 0
    assert O.e2m1_decode(q.codes[1, 20]) == 6.0
    # a value far below its block's resolution keeps its sign on a zero code
    x = np.array([[6.0, -1e-6] + [0.0] * 14], dtype=np.float32)
    q = O.quantize(x)
    assert q.codes[0, 1] == 8 and q.codes[0, 2] == 0
    # a static gs far too small saturates the scale at 448 and the codes at +-6
    q = O.quantize(np.full((1, 16), -5.0, dtype=np.float32), gs=1e-6)
    assert q.sf[0, 0] == 0x7E and (q.codes == 15).all()


def test_pack_low_nibble_is_even_element():
    codes = np.array([[1, 2, 15, 8]], dtype=np.uint8)
    np.testing.assert_array_equal(O.pack_codes(codes), [[0x21, 0x8F]])
    np.testing.assert_array_equal(O.unpack_codes(O.pack_codes(codes)), codes)


# --------------------------------------------------------------------------- scale layout

def test_sf_layout_fixture(golden):
    g = golden("sf_layout.json")
    off = O.sf_swizzle_offsets(g["rows"], g["K"])
    for e in g["offsets"]:
        assert off[e["r"], e["c"]] == e["offset"], e


@pytest.mark.parametrize("rows,K", [(1, 64), (127, 128), (128, 256), (200, 512), (300, 7168)])
def test_sf_layout_is_a_padded_bijection(rows, K):
    off = O.sf_swizzle_offsets(rows, K)
    R, C = O.sf_padded_shape(rows, K)
    assert off.shape == (R, C) and R % 128 == 0 and C % 4 == 0
    assert sorted(off.ravel().tolist()) == list(range(R * C)) == list(range(O.sf_bytes(rows, K)))
    # a row's 4 consecutive scale columns are 4 consecutive bytes (one 32-bit word)
    assert np.all(off[:, 1::4] == off[:, 0::4] + 1) and np.all(off[:, 3::4] == off[:, 0::4] + 3)
    sf = np.random.default_rng(7).integers(0, 127, (rows, K // 16)).astype(np.uint8)
    buf = O.swizzle_sf(sf, K)
    np.testing.assert_array_equal(O.unswizzle_sf(buf, rows, K), sf)
    pad = np.ones(R * C, bool)
    pad[off[:rows, : K // 16].ravel()] = False
    assert not buf[pad].any()


def test_sf_layout_32_row_slices_fill_one_word_per_chunk():
    """A 32-row slice starting 32 j rows into a 128-row block owns 32-bit word j of every one
    of the block's 32 sixteen-byte chunks, one chunk per row (what a 32-row GEMM tile's scale
    staging relies on when it moves word j into place)."""
    rows, K = 256, 512
    off = O.sf_swizzle_offsets(rows, K)
    for b in range(rows // 128):
        for j in range(4):
            sl = off[128 * b + 32 * j:128 * b + 32 * (j + 1), :]
            for q in range(sl.shape[1] // 4):  # each 512-byte block of 4 scale columns
                blk = sl[:, 4 * q:4 * q + 4]
                assert len(set((blk // 512).ravel().tolist())) == 1
                assert set(((blk % 16) // 4).ravel().tolist()) == {j}
                chunks = (blk[:, 0] % 512) // 16
                assert sorted(chunks.tolist()) == list(range(32))


# --------------------------------------------------------------------------- linear

def _frac_f32(v):
    return Fraction(float(v))


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (2, 3, 32), (4, 4, 64), (3, 2, 48)])
def test_linear_brute_force_exact_sum(M, N, K):
    """Each term is an exact rational product; compare with an exact rational sum."""
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    xq = O.quantize(x)
    wq = O.quantize(w)
    got = O.linear(xq, wq.codes, wq.sf, wq.gs)
    lut = [0, Fraction(1, 2), 1, Fraction(3, 2), 2, 3, 4, 6]

    def val(code, sfb):
        e, m = sfb >> 3, sfb & 7
        s = Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        v = lut[code & 7] * s
        return -v if code & 8 else v

    for i, j in itertools.product(range(M), range(N)):
        acc, mag = Fraction(0), Fraction(0)
        for k in range(K):
            t = (val(int(xq.codes[i, k]), int(xq.sf[i, k // 16])) * _frac_f32(xq.gs)
                 * val(int(wq.codes[j, k]), int(wq.sf[j, k // 16])) * _frac_f32(wq.gs))
            acc += t
            mag += abs(t)
        # fp64 summation of K terms: |error| <= (K + 4) * 2^-53 * sum |terms|
        assert abs(Fraction(float(got[i, j])) - acc) <= (K + 4) * Fraction(1, 2 ** 53) * mag


def test_ws2_is_weight_side_only():
    """The activation carries gs and the weight ws2 (page 2): folding the activation scale
    into the weight side as well multiplies the output by that factor again (the
    '~4000x too small' failure mode)."""
    rng = np.random.default_rng(8)
    xq = O.quantize(rng.standard_normal((4, 64)).astype(np.float32))
    wq = O.quantize((rng.standard_normal((8, 64)) * 0.02).astype(np.float32))
    good = O.linear(xq, wq.codes, wq.sf, wq.gs)
    wrong = O.linear(xq, wq.codes, wq.sf, wq.gs * xq.gs)
    np.testing.assert_allclose(wrong, good * float(xq.gs), rtol=1e-7)  # fp32 product of the two scales
    assert 1.0 / float(xq.gs) > 500  # with N(0,1) activations the error is a ~10^3x shrink


def test_grouped_linear_is_block_diagonal_linear():
    """G groups of K inputs -> N outputs each equal one linear with a block-diagonal weight."""
    rng = np.random.default_rng(12)
    M, G, K, N = 5, 3, 64, 32
    xq = O.quantize(rng.standard_normal((M, G * K)).astype(np.float32))
    ws = [O.quantize((rng.standard_normal((N, K)) * 0.02).astype(np.float32)) for _ in range(G)]
    got = O.grouped_linear(xq, [w.codes for w in ws], [w.sf for w in ws], [w.gs for w in ws])
    big = np.zeros((G * N, G * K))
    for g, w in enumerate(ws):
        big[g * N:(g + 1) * N, g * K:(g + 1) * K] = O.dequantize(w.codes, w.sf, w.gs)
    want = O.dequantize(xq.codes, xq.sf, xq.gs) @ big.T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)
    assert got.shape == (M, G * N)


# --------------------------------------------------------------------------- RMSNorm

def test_rmsnorm_against_library_and_closed_forms():
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((6, 256)) * 3).astype(np.float32)
    gamma = (1 + 0.1 * rng.standard_normal(256)).astype(np.float32)
    eps = 1e-6
    yb, y, inv = O.rmsnorm(x, gamma, eps)
    want = torch.nn.functional.rms_norm(torch.from_numpy(x).double(), (256,), torch.from_numpy(gamma).double(), eps)
    np.testing.assert_allclose(y, want.numpy(), rtol=1e-13)
    # bf16 rounding of the fp64 value: within half a bf16 ulp (2^-8 relative) plus the fp32 step
    assert np.all(np.abs(yb - y) <= np.abs(y) * (2.0 ** -8) * 1.0001 + 1e-30)
    # a constant row c normalises to sign(c) * gamma / sqrt(1 + eps / c^2)
    c = np.full((1, 256), -2.5, np.float32)
    _, yc, _ = O.rmsnorm(c, gamma, eps)
    np.testing.assert_allclose(yc[0], -gamma / np.sqrt(1 + eps / 6.25), rtol=1e-15)
    # scale invariance away from eps
    _, y2, _ = O.rmsnorm(x * 64, gamma, eps)
    np.testing.assert_allclose(y2, y, rtol=2e-7)  # differs by ~eps / (2 mean(x^2)) ~ 6e-8


# --------------------------------------------------------------------------- router

def test_signed_e4m3_matches_torch_float8():
    rng = np.random.default_rng(14)
    v = np.concatenate([rng.standard_normal(20000) * np.exp2(rng.uniform(-12, 9, 20000)),
                        [0.0, -0.0, 448.0, -448.0, 500.0, -1e9]]).astype(np.float32)
    want = torch.from_numpy(np.clip(v, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode_signed(v)
    np.testing.assert_array_equal(got[v != 0], want[v != 0])  # torch maps -0 to 0x80 as well; zeros checked below
    assert got[-6 + 0] == 0 and got[-5] == 0x80
    back = torch.from_numpy(want.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.e4m3_decode_signed(want), back)


def test_router_weight_fp8_roundtrip_precision(golden):
    """The gate's FP8 round trip keeps cosine ~0.9997 to the bf16 weight (page 1's FP8 figure)."""
    rng = np.random.default_rng(15)
    wq = O.quantize((rng.standard_normal((384, 7168)) * 0.02).astype(np.float32))
    wg = O.router_weight(wq.codes, wq.sf, wq.gs)
    w = O.dequantize(wq.codes, wq.sf, wq.gs)
    c = O.cosine(wg, w)
    assert abs(c - golden("page_precision.json")["fp8_e4m3_roundtrip_cosine"]) < 2e-4
    np.testing.assert_array_equal(O.bf16_bits_to_f32(O.f32_to_bf16_bits(wg.astype(np.float32))), wg)  # bf16 values


def _router_weight_by_library_casts(codes, sf, ws2, e2m1_table, bf16_before_fp8=True):
    """The gate weight's dequantise -> FP8-E4M3 round trip built from torch's own casts: the OCP
    E2M1 table (golden), torch's float8_e4m3fn decode of the scales, fp32 products, torch's bf16
    cast, fp32 amax / 448 and reciprocal, torch's float8_e4m3fn cast, and a final bf16 cast."""
    vals = torch.tensor([float(e2m1_table[str(c)]) for c in range(16)], dtype=torch.float32)
    scale = torch.from_numpy(np.repeat(sf, 16, axis=1)[:, : codes.shape[1]].copy()).view(torch.float8_e4m3fn).float()
    w = (vals[torch.from_numpy(codes.astype(np.int64))] * scale) * torch.tensor(ws2, dtype=torch.float32)
    if bf16_before_fp8:
        w = w.to(torch.bfloat16).float()
    s = w.abs().max() / torch.tensor(448.0, dtype=torch.float32)
    q = (w * (torch.tensor(1.0, dtype=torch.float32) / s)).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy(), (q.float() * s).to(torch.bfloat16).float().numpy()


def test_router_weight_against_library_casts(golden):
    """router_weight equals the same chain spelled with library casts, element for element, on a
    random gate and on a hand-picked one where the bf16 rounding ahead of the FP8 step changes
    FP8 codes (page 1, the router-gate FP8 round trip: NVFP4 dequantised to bf16 first)."""
    table = golden("e2m1_values.json")["codes_to_values"]
    rng = np.random.default_rng(17)
    wq = O.quantize((rng.standard_normal((64, 1024)) * 0.02).astype(np.float32))
    _, want = _router_weight_by_library_casts(wq.codes, wq.sf, wq.gs, table)
    np.testing.assert_array_equal(O.router_weight(wq.codes, wq.sf, wq.gs), want)
    # two 16-element blocks with different scales: without the bf16 rounding, codes 7, 12 and 13
    # of the FP8 tensor come out one step higher
    codes = np.array([[8, 4, 4, 0, 1, 0, 2, 13, 10, 14, 8, 9, 15, 11, 10, 8,
                       8, 14, 4, 13, 10, 0, 6, 13, 8, 0, 12, 11, 13, 2, 1, 13]], dtype=np.uint8)
    sf = np.array([[41, 86]], dtype=np.uint8)
    ws2 = np.float32(float.fromhex("0x1.a3d184p-8"))
    q_bf16, want = _router_weight_by_library_casts(codes, sf, ws2, table)
    q_plain, plain = _router_weight_by_library_casts(codes, sf, ws2, table, bf16_before_fp8=False)
    assert (q_bf16 != q_plain).sum() == 3
    got = O.router_weight(codes, sf, ws2)
    np.testing.assert_array_equal(got, want)
    assert not np.array_equal(got, plain)


def test_router_topk_against_library():
    rng = np.random.default_rng(16)
    x = rng.standard_normal((40, 64))
    wg = rng.standard_normal((24, 64)) * 0.1
    ids, w, p = O.router(x, wg, 5)
    tp = torch.softmax(torch.from_numpy(x @ wg.T), dim=1)
    tv, ti = torch.topk(tp, 5, dim=1)
    np.testing.assert_array_equal(ids, ti.numpy())
    np.testing.assert_allclose(w, (tv / tv.sum(1, keepdim=True)).numpy(), rtol=1e-14)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-15)
    # ties go to the lower expert id
    ids2, _, _ = O.router(np.zeros((1, 64)), np.zeros((24, 64)), 3)
    np.testing.assert_array_equal(ids2[0], [0, 1, 2])


# --------------------------------------------------------------------------- SiLU

def test_silu_closed_form_and_library():
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert O.silu(np.array([800.0]))[0] == 800.0
    assert O.silu(np.array([-800.0]))[0] == 0.0
    g = np.linspace(-30, 30, 10001)
    np.testing.assert_allclose(O.silu(g), torch.nn.functional.silu(torch.from_numpy(g)).numpy(),
                               rtol=1e-15, atol=1e-300)


# --------------------------------------------------------------------------- routing

@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (5, 2, 3), (16, 2, 8), (64, 8, 384), (7, 4, 5)])
def test_route_against_stable_sort_and_invariants(T, k, E):
    rng = np.random.default_rng(T * 7 + k)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)  # duplicates within a token allowed
    r = O.route(ids, E)
    flat = ids.ravel()
    np.testing.assert_array_equal(r.counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(r.offsets, np.concatenate([[0], np.cumsum(r.counts)]))
    np.testing.assert_array_equal(r.sorted_idx, np.argsort(flat, kind="stable"))
    assert sorted(r.sorted_idx.tolist()) == list(range(T * k))
    np.testing.assert_array_equal(r.sorted_idx[r.inv_idx], np.arange(T * k))
    for e in range(E):
        seg = r.sorted_idx[r.offsets[e]:r.offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


def test_route_brute_force_rank():
    ids = np.array([[2, 0], [2, 2], [1, 0]], dtype=np.int32)
    r = O.route(ids, 4)
    np.testing.assert_array_equal(r.counts, [2, 1, 3, 0])
    np.testing.assert_array_equal(r.sorted_idx, [1, 5, 4, 0, 2, 3])
    np.testing.assert_array_equal(r.inv_idx, [3, 0, 4, 5, 2, 1])
    with pytest.raises(ValueError):
        O.route(np.array([[4]]), 4)


# --------------------------------------------------------------------------- MoE

def _expert(rng, H, I):
    w13 = O.quantize((rng.standard_normal((2 * I, H)) * 0.02).astype(np.float32))
    w2 = O.quantize((rng.standard_normal((H, I)) * 0.02).astype(np.float32))
    return O.Expert(w13.codes, w13.sf, w13.gs, w2.codes, w2.sf, w2.gs)


def test_moe_single_expert_is_two_linears_with_silu_gate():
    rng = np.random.default_rng(9)
    T, H, I = 6, 64, 32
    ex = _expert(rng, H, I)
    x = rng.standard_normal((T, H)).astype(np.float32)
    a2 = [F32(0.004)]
    res = O.moe_forward(x, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32),
                        lambda e: ex, 1, a2)
    xq = O.quantize(x)
    gu = O.linear(xq, ex.w13_codes, ex.w13_sf, ex.w13_ws2)
    g, u = gu[:, :I], gu[:, I:]
    h = g * u / (1 + np.exp(-g))
    hq = O.quantize(h.astype(np.float32), gs=a2[0])
    want = O.linear(hq, ex.w2_codes, ex.w2_sf, ex.w2_ws2)
    np.testing.assert_allclose(res.y, want, rtol=1e-12, atol=1e-15)
    assert res.y.shape == (T, H)  # output width is the hidden size (page 3)


def test_moe_weights_select_experts_and_shared_adds():
    rng = np.random.default_rng(10)
    T, H, I, E, k = 5, 32, 16, 4, 2
    exps = [_expert(rng, H, I) for _ in range(E)]
    shared = _expert(rng, H, I)
    x = rng.standard_normal((T, H)).astype(np.float32)
    ids = np.array([[e, (e + 1) % E] for e in range(T)], np.int32) % E
    a2 = [F32(0.003)] * (E + 1)
    w_one = np.array([[1.0, 0.0]] * T, np.float32)
    only_first = O.moe_forward(x, ids, w_one, lambda e: exps[e], E, a2)
    single = O.moe_forward(x, ids[:, :1], np.ones((T, 1), np.float32), lambda e: exps[e], E, a2)
    np.testing.assert_allclose(only_first.y, single.y, rtol=1e-13, atol=1e-16)
    w = rng.random((T, k)).astype(np.float32)
    both = O.moe_forward(x, ids, w, lambda e: exps[e], E, a2)
    with_shared = O.moe_forward(x, ids, w, lambda e: exps[e], E, a2, shared=shared)
    sh_only = O.moe_forward(x, np.zeros((T, 1), np.int32), np.zeros((T, 1), np.float32),
                            lambda e: exps[e], E, a2, shared=shared)
    np.testing.assert_allclose(with_shared.y, both.y + sh_only.y, rtol=1e-12, atol=1e-15)


def test_moe_token_permutation_equivariance():
    rng = np.random.default_rng(11)
    T, H, I, E, k = 6, 32, 16, 3, 2
    exps = [_expert(rng, H, I) for _ in range(E)]
    x = rng.standard_normal((T, H)).astype(np.float32)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    a2 = [F32(0.003)] * (E + 1)
    p = rng.permutation(T)
    base = O.moe_forward(x, ids, w, lambda e: exps[e], E, a2)
    perm = O.moe_forward(x[p], ids[p], w[p], lambda e: exps[e], E, a2)
    np.testing.assert_allclose(perm.y, base.y[p], rtol=1e-13, atol=1e-16)
    # a subset of tokens gives the same rows (the global scale and routing still cover all
    # tokens); only the fp64 summation order of the batched library matmul may differ
    sub = O.moe_forward(x, ids, w, lambda e: exps[e], E, a2, tokens=[4, 1])
    np.testing.assert_allclose(sub.y, base.y[[4, 1]], rtol=1e-13, atol=1e-18)
    # per-expert jobs through another mapper (as a process pool runs them) give the same result
    mapped = O.moe_forward(x, ids, w, lambda e: exps[e], E, a2, mapper=lambda f, jobs: [f(j) for j in jobs[::-1]][::-1])
    np.testing.assert_array_equal(mapped.y, base.y)
