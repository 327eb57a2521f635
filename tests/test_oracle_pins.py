"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

None of these re-types an oracle formula and compares it with itself; each one
compares the oracle with a printed value, a closed form, a library routine, an
invariant, or brute force on a tiny domain.
"""
import math

import numpy as np
import pytest
import scipy.linalg

import workloads
from conftest import read_golden

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def unpack_codes(codes: np.ndarray, C: int) -> np.ndarray:
    lo = codes & 15
    hi = codes >> 4
    out = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out[:, :C]


# ------------------------------------------------------------------ E2M1


def test_e2m1_all_codes_round_trip(orc):
    for c in range(16):
        v = orc.e2m1_decode([c])[0]
        assert abs(v) == GRID[c & 7]
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)
        assert orc.e2m1_rne([v])[0] == c


def test_e2m1_rne_golden_cases(orc):
    rows = read_golden("e2m1_rne_cases.txt")
    x = np.array([float(r[0]) for r in rows], np.float32)
    want = np.array([int(r[1], 16) for r in rows], np.uint8)
    got = orc.e2m1_rne(x)
    bad = [(rows[i][0], hex(got[i]), rows[i][1]) for i in np.nonzero(got != want)[0]]
    assert not bad, bad


def test_e2m1_rne_is_nearest_brute_force(orc):
    rng = np.random.default_rng(5)
    q = np.concatenate([rng.uniform(-7, 7, 200000), rng.uniform(-0.3, 0.3, 20000)]).astype(np.float32)
    codes = orc.e2m1_rne(q)
    g = GRID[codes & 7]
    a = np.abs(q.astype(np.float64))
    d_best = np.min(np.abs(np.minimum(a, 6.0)[:, None] - GRID[None, :]), axis=1)
    assert np.all(np.abs(np.minimum(a, 6.0) - g) == d_best)
    nz = q != 0
    assert np.all(((codes[nz] & 8) != 0) == (q[nz] < 0))


# ------------------------------------------------------------------ E4M3


def test_e4m3_golden_values(orc):
    for code_hex, val in read_golden("e4m3_values.txt"):
        v = orc.e4m3_decode([int(code_hex, 16)])[0]
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val))


def test_e4m3_all_256_codes_round_trip(orc):
    vals = orc.e4m3_decode(np.arange(256))
    for b in range(256):
        if b in (0x7F, 0xFF):
            assert math.isnan(vals[b])
            continue
        assert math.isfinite(vals[b])
        assert orc.e4m3_rne_satfinite([vals[b]])[0] == b
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0), "non-negative codes must increase with the value"
    assert pos.max() == 448.0


def test_e4m3_rne_brute_force(orc):
    finite = orc.e4m3_decode(np.arange(0x7F)).astype(np.float64)  # 0 .. 448, codes 0..0x7E
    mids = (finite[:-1] + finite[1:]) / 2
    rng = np.random.default_rng(11)
    xs = np.concatenate([
        mids, np.nextafter(mids, 0), np.nextafter(mids, 1000), finite,
        np.exp(rng.uniform(np.log(1e-4), np.log(600.0), 200000)),
        [0.0, 448.0, 448.5, 463.9, 464.0, 480.0, 1e30, np.inf],
    ]).astype(np.float32)
    got = orc.e4m3_rne_satfinite(xs)
    x = xs.astype(np.float64)
    for i in range(x.size):
        if x[i] > 448.0:
            want = 0x7E
        else:
            d = np.abs(finite - x[i])
            best = np.nonzero(d == d.min())[0]
            want = best[0] if best.size == 1 else [b for b in best if b % 2 == 0][0]
        assert got[i] == want, (xs[i], hex(got[i]), hex(want))


# ------------------------------------------------------------------ Philox


def test_philox_known_answers(orc):
    for row in read_golden("philox4x32_10_kat.txt"):
        w = [int(v, 16) for v in row]
        out = orc.philox4x32_10(w[0:4], w[4:6])
        assert [int(v) for v in out] == w[6:10]


def test_sr_word_stream_layout(orc):
    seed = 0x1234_5678_9ABC_DEF0
    idx = np.array([0, 1, 2, 3, 4, 7, 1 << 33, (1 << 33) + 2, 12345678901], np.uint64)
    words = orc.sr_words(seed, idx)
    for i, w in zip(idx.tolist(), words.tolist()):
        blk = i >> 2
        out = orc.philox4x32_10([blk & 0xFFFFFFFF, blk >> 32, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
        assert w == int(out[i & 3])


# ------------------------------------------------------------------ RHT


def test_rht_matches_sylvester_hadamard(orc):
    H = scipy.linalg.hadamard(16).astype(np.float64)
    cols = orc.rht16(np.eye(16, dtype=np.float32), 0)  # row k = transform of e_k
    assert np.array_equal(cols.T.astype(np.float64) * 4.0, H)
    assert np.array_equal(H @ H.T, 16 * np.eye(16))


def test_rht_signs_and_orthogonality(orc):
    rng = np.random.default_rng(3)
    H = scipy.linalg.hadamard(16).astype(np.float64)
    for seed in (0, 1, 99, 2**40 + 5):
        mask = orc.rht_sign_mask(seed)
        sigma = np.array([-1.0 if (mask >> j) & 1 else 1.0 for j in range(16)])
        v = rng.standard_normal((64, 16)).astype(np.float32)
        y = orc.rht16(v, mask).astype(np.float64)
        ref = 0.25 * (v.astype(np.float64) * sigma) @ H.T
        assert np.allclose(y, ref, rtol=0, atol=1e-6 * np.abs(v).max())
        assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(v.astype(np.float64), axis=1), rtol=1e-6)
    assert len({orc.rht_sign_mask(s) for s in range(32)}) > 24


def test_rht_involution_without_signs(orc):
    v = np.random.default_rng(4).standard_normal((32, 16)).astype(np.float32)
    back = orc.rht16(orc.rht16(v, 0), 0)  # (H/4)(H/4) = H H^T / 16 = I
    assert np.allclose(back, v, rtol=0, atol=4e-7 * np.abs(v).max())


# ------------------------------------------------------------------ SR


@pytest.mark.parametrize("q", [0.3, 0.8, 1.2, 1.9, 2.7, 3.01, 4.9, 5.999, -3.3, -0.1])
def test_sr_unbiased_and_between_neighbours(orc, q):
    n = 1 << 16
    words = orc.sr_words(77, np.arange(n, dtype=np.uint64))
    codes = orc.e2m1_sr(np.full(n, q, np.float32), words)
    vals = orc.e2m1_decode(codes[:4096])  # decode via the oracle on a subset
    a = abs(q)
    lo = GRID[GRID <= a].max()
    hi = GRID[GRID > a].min()
    mags = GRID[codes & 7]
    assert set(np.unique(mags)).issubset({lo, hi})
    assert np.all(np.abs(vals) == mags[:4096])
    p = (a - lo) / (hi - lo)
    mean = mags.mean()
    sigma = (hi - lo) * math.sqrt(p * (1 - p) / n)
    assert abs(mean - a) <= 3 * sigma + 1e-12


def test_sr_seed_behaviour(orc):
    x = workloads.gradients(32, 64, seed=4)
    a = orc.quantize(x, rounding=orc.ROUND_SR, sr_seed=1)
    b = orc.quantize(x, rounding=orc.ROUND_SR, sr_seed=1)
    c = orc.quantize(x, rounding=orc.ROUND_SR, sr_seed=2)
    assert np.array_equal(a.codes, b.codes) and np.array_equal(a.sf, b.sf)
    assert not np.array_equal(a.codes, c.codes)


# ------------------------------------------------------------- quantizer


def _mixed_matrix(rows=64, cols=256, seed=21):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x[: rows // 4] = rng.standard_t(3, (rows // 4, cols)) * 0.05
    x[rows // 4: rows // 2] = rng.uniform(-1, 1, (rows // 4, cols))
    x[rows // 2:, ::37] *= 30.0
    x[3, 16:32] = 0.0  # one all-zero block
    x[5, 32:48] = 0.0
    x[5, 40] = 7.0  # one single-outlier block
    return workloads.bf16_bits(x)


def _true_block_sse(y64, sf_bytes_rm, s_t, orc, tile_rows=1):
    """FP64 SSE of each block (1 x 16) or tile (16 x 16) of y64 [R, C] for the
    given per-block scale bytes [R, C/16] (one per row of a tile, all equal),
    each value sent to the nearest grid magnitude by brute force."""
    R, C = y64.shape
    eff = orc.e4m3_decode(sf_bytes_rm).astype(np.float64) * s_t  # [R, nb]
    e = np.repeat(eff, 16, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        a = np.where(e > 0, np.abs(y64) / e, 0.0)
    a = np.minimum(a, 6.0)
    g = GRID[np.argmin(np.abs(a[..., None] - GRID), axis=-1)]
    xhat = np.sign(y64) * g * e
    sq = ((y64 - xhat) ** 2).reshape(R // tile_rows, tile_rows, C // 16, 16)
    return sq.sum(axis=(1, 3))  # [R / tile_rows, nb]


def _block_max(y64, tile_rows):
    R, C = y64.shape
    return np.abs(y64).reshape(R // tile_rows, tile_rows, C // 16, 16).max(axis=(1, 3))


def _check_choice_against_brute_force(orc, x, y64_out, tile_rows, **kw):
    """The oracle's 4/6 output against the definition, block by block:

    * each candidate's scale byte is E4M3(a_b / (M s_t)) with the product and
      the quotient rounded to FP32 ("Four Over Six", first section: the block
      maximum is mapped to 4 or to 6), a_b found here with numpy's max over the
      block or tile in the output orientation;
    * the kept candidate has the lower FP64 squared error, brute-forced over
      the grid with that candidate's scale, ties to 6, except where the two
      errors agree to 1e-6 relative (FP32 near-ties, counted and returned);
    * the 4/6 output carries the kept candidate's scale byte in every row of
      the block or tile.
    y64_out is the input in the output orientation (x itself, or x^T for
    transposed calls).  Returns the number of near-ties."""
    R, C = y64_out.shape
    nb = C // 16
    rm = orc.SF_ROWMAJOR
    q46 = orc.quantize(x, sf_layout=rm, **kw)
    q6 = orc.quantize(x, scale_rule=orc.SCALE_6, sf_layout=rm, **kw)
    q4 = orc.quantize(x, scale_rule=orc.SCALE_4, sf_layout=rm, **kw)
    assert (q46.rows, q46.cols) == (R, C)
    s_t = q46.tensor_scale
    assert np.float32(s_t) == np.float32(np.float32(np.abs(y64_out).max()) / np.float32(2688.0))
    ab = _block_max(y64_out, tile_rows).astype(np.float32)  # exact: bf16 values
    tiles = lambda a: a.reshape(R // tile_rows, tile_rows, nb)  # noqa: E731
    for M, q in ((6, q6), (4, q4)):
        t = np.float32(np.float32(M) * np.float32(s_t))
        with np.errstate(divide="ignore", invalid="ignore"):
            raw = np.where(t > 0, ab / t, np.float32(0)).astype(np.float32)
        want = orc.e4m3_rne_satfinite(raw)
        got = tiles(q.sf.reshape(R, nb))
        assert np.all(got == got[:, :1, :]), "one scale per tile"
        bad = np.argwhere(got[:, 0, :] != want)
        assert bad.size == 0, f"M={M}: {len(bad)} scale bytes differ from E4M3(a_b / (M s_t)), first {bad[:4]}"
    sf6, sf4 = tiles(q6.sf.reshape(R, nb))[:, 0, :], tiles(q4.sf.reshape(R, nb))[:, 0, :]
    E6 = _true_block_sse(y64_out, q6.sf.reshape(R, nb), s_t, orc, tile_rows)
    E4 = _true_block_sse(y64_out, q4.sf.reshape(R, nb), s_t, orc, tile_rows)
    chose4 = ((q46.choice[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(R, -1)[:, :nb].astype(bool)
    assert np.all(tiles(chose4) == tiles(chose4)[:, :1, :]), "one choice per tile"
    chose4 = tiles(chose4)[:, 0, :]
    same = sf4 == sf6  # identical candidates: a tie, 6 wins
    assert not np.any(chose4 & same)
    near = (np.abs(E4 - E6) <= 1e-6 * np.maximum(E4, E6)) & ~same
    ok = ~near & ~same
    wrong = np.argwhere(chose4[ok] != (E4 < E6)[ok])
    assert wrong.size == 0, f"{len(wrong)} choices disagree with the FP64 brute force outside the near-tie window"
    assert 0.02 < chose4.mean() < 0.98  # both candidates are exercised
    sf46 = tiles(q46.sf.reshape(R, nb))[:, 0, :]
    assert np.array_equal(sf46, np.where(chose4, sf4, sf6))
    return int(near.sum())


@pytest.mark.parametrize("layout", ["rows", "transposed", "2d", "2d_transposed"])
def test_choice_matches_brute_force(orc, layout):
    x = _mixed_matrix()
    y64 = workloads.bf16_to_f32(x).astype(np.float64)
    kw = {"transpose": layout in ("transposed", "2d_transposed"), "block_2d": layout.startswith("2d")}
    y_out = np.ascontiguousarray(y64.T) if kw["transpose"] else y64
    n_near = _check_choice_against_brute_force(orc, x, y_out, 16 if kw["block_2d"] else 1, **kw)
    assert n_near <= 0.01 * y_out.size / (256 if kw["block_2d"] else 16)


def test_candidate_scales_on_weight_rows_with_exact_ties(orc):
    """Rows of the q_proj-shaped weight (seed 2000): there amax is 1.1484375,
    s_t is 7/16384 exactly, and many a_b / (4 s_t) land exactly on E4M3
    rounding ties, where a_b times a rounded reciprocal 1/(4 s_t) falls on the
    wrong side.  The oracle must follow the quotient on every block."""
    x = workloads.student_t(1024, 4096, seed=2000)
    y64 = workloads.bf16_to_f32(x).astype(np.float64)
    _check_choice_against_brute_force(orc, x, y64, 1)
    # the data does separate the definition from the reciprocal shortcut
    q4 = orc.quantize(x, scale_rule=orc.SCALE_4, sf_layout=orc.SF_ROWMAJOR)
    t4 = np.float32(4.0) * np.float32(q4.tensor_scale)
    ab = _block_max(y64, 1).astype(np.float32)
    shortcut = orc.e4m3_rne_satfinite((ab * (np.float32(1.0) / t4)).astype(np.float32))
    assert (shortcut != q4.sf.reshape(1024, 256)).sum() > 1000


def test_four_over_six_never_worse_than_six(orc):
    x = _mixed_matrix(seed=22)
    R, C = x.shape
    y64 = workloads.bf16_to_f32(x).astype(np.float64)
    d46 = orc.dequantize(orc.quantize(x)).astype(np.float64)
    d6 = orc.dequantize(orc.quantize(x, scale_rule=orc.SCALE_6)).astype(np.float64)
    s46 = ((d46 - y64) ** 2).reshape(R, -1, 16).sum(-1)
    s6 = ((d6 - y64) ** 2).reshape(R, -1, 16).sum(-1)
    assert np.all(s46 <= s6 * (1 + 1e-3) + 1e-30)
    assert s46.sum() < s6.sum()


def test_dequantized_values_lie_on_grid_times_scale(orc):
    x = _mixed_matrix(seed=23)
    for kw in ({}, {"rounding": 1, "sr_seed": 9}, {"block_2d": True}, {"hadamard": True, "hadamard_seed": 3}):
        q = orc.quantize(x, sf_layout=orc.SF_ROWMAJOR, **kw)
        d = orc.dequantize(q).astype(np.float64)
        eff = np.repeat(orc.e4m3_decode(q.sf.reshape(q.rows, -1)).astype(np.float64) * q.tensor_scale, 16, 1)
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = np.where(eff > 0, np.abs(d) / eff, 0.0)
        on = np.min(np.abs(ratio[..., None] - GRID), axis=-1) <= 1e-6 * np.maximum(ratio, 1)
        assert on.all(), kw


def test_hand_built_block_prefers_four_and_ties_go_to_six(orc):
    x = np.zeros((1, 64), np.float32)
    x[0, 0] = 2688.0  # tensor amax -> s_t = 1
    x[0, 16:20] = [64.0, 48.0, 32.0, 16.0]  # = 16 * [4, 3, 2, 1]: exact with sf_4 = 16
    x[0, 32:48] = 0.0  # all-zero block: both scales 0, equal error -> 6
    x[0, 48] = 2688.0  # block max = amax: the 4-candidate saturates to 448 like the 6-candidate
    q = orc.quantize(workloads.bf16_bits(x), sf_layout=orc.SF_ROWMAJOR)
    assert q.tensor_scale == 1.0
    bits = int(q.choice[0, 0])
    assert bits & 2, "block 1 is exact under the 4-scale and must keep 4"
    assert not bits & 4 and not bits & 8 and not bits & 1
    assert q.sf[1] == orc.e4m3_rne_satfinite([16.0])[0]
    assert q.sf[2] == 0 and q.sf[3] == 0x7E and q.sf[0] == 0x7E
    d = orc.dequantize(q)
    assert np.array_equal(d[0, 16:20], x[0, 16:20])


def test_all_zero_tensor(orc):
    q = orc.quantize(np.zeros((16, 64), np.uint16))
    assert q.tensor_scale == 0.0
    assert not q.sf.any() and not q.codes.any() and not q.choice.any()


def test_supplied_amax_is_used(orc):
    x = _mixed_matrix(seed=24)
    q = orc.quantize(x, amax=1000.0)
    assert q.tensor_scale == np.float32(np.float32(1000.0) / np.float32(2688.0))
    assert not np.array_equal(q.sf, orc.quantize(x).sf)


def test_transposed_equals_quantizing_the_materialized_transpose(orc):
    x = _mixed_matrix(rows=48, cols=80, seed=25)
    xt = np.ascontiguousarray(x.T)
    for kw in ({}, {"hadamard": True, "hadamard_seed": 12}, {"scale_rule": orc.SCALE_6}):
        a = orc.quantize(x, transpose=True, **kw)
        b = orc.quantize(xt, **kw)
        assert a.rows == 80 and a.cols == 48
        assert np.array_equal(a.codes, b.codes) and np.array_equal(a.sf, b.sf)
        assert a.tensor_scale == b.tensor_scale and np.array_equal(a.choice, b.choice)


@pytest.mark.parametrize("rounding", [0, 1])
def test_2d_transposed_is_the_transpose(orc, rounding):
    x = _mixed_matrix(rows=48, cols=96, seed=26)
    a = orc.quantize(x, block_2d=True, rounding=rounding, sr_seed=5, sf_layout=orc.SF_ROWMAJOR)
    b = orc.quantize(x, block_2d=True, transpose=True, rounding=rounding, sr_seed=5, sf_layout=orc.SF_ROWMAJOR)
    ca = unpack_codes(a.codes, 96)
    cb = unpack_codes(b.codes, 48)
    assert np.array_equal(ca.T, cb)
    sa = a.sf.reshape(48, 6)
    sb = b.sf.reshape(96, 3)
    for i in range(3):
        for j in range(6):
            assert np.all(sa[16 * i: 16 * i + 16, j] == sa[16 * i, j])
            assert sb[16 * j, i] == sa[16 * i, j]


def test_2d_tile_uses_one_scale_and_beats_six_only(orc):
    x = _mixed_matrix(rows=64, cols=128, seed=27)
    y64 = workloads.bf16_to_f32(x).astype(np.float64)
    q = orc.quantize(x, block_2d=True, sf_layout=orc.SF_ROWMAJOR)
    q6 = orc.quantize(x, block_2d=True, scale_rule=orc.SCALE_6, sf_layout=orc.SF_ROWMAJOR)
    s = q.sf.reshape(64, 8)
    assert np.array_equal(s, np.repeat(s[::16], 16, axis=0))
    t = lambda d: ((d - y64) ** 2).reshape(4, 16, 8, 16).sum((1, 3))  # noqa: E731
    assert np.all(t(orc.dequantize(q)) <= t(orc.dequantize(q6)) * (1 + 1e-3) + 1e-30)


def test_sf_swizzle_offsets_by_hand(orc):
    # 128 rows x 4 scale columns per 512-byte tile; 32-row groups interleave at 4-byte
    # steps inside 16-byte rows; tiles row-major over (row tile, column tile).
    cases = [((0, 0, 8), 0), ((1, 0, 8), 16), ((31, 0, 8), 496), ((32, 0, 8), 4), ((33, 0, 8), 20),
             ((64, 0, 8), 8), ((96, 0, 8), 12), ((127, 3, 8), 511), ((0, 4, 8), 512),
             ((128, 0, 8), 1024), ((130, 5, 8), 1569), ((0, 1, 1), 1), ((129, 0, 1), 528)]
    for (r, c, nb), off in cases:
        assert orc.sf_offset(r, c, nb) == off, (r, c, nb)
    assert orc.sf_bytes(130, 9) == 256 * 12
    x = _mixed_matrix(rows=130 - 2, cols=144, seed=28)
    a = orc.quantize(x)
    b = orc.quantize(x, sf_layout=orc.SF_ROWMAJOR)
    assert np.array_equal(orc.sf_to_rowmajor(a.sf, a.rows, 9), b.sf.reshape(a.rows, 9))
    mask = np.ones(a.sf.size, bool)
    mask[[orc.sf_offset(r, c, 9) for r in range(a.rows) for c in range(9)]] = False
    assert not a.sf[mask].any(), "pad bytes must be zero"


@pytest.mark.parametrize("rows,nb", [(1, 1), (3, 3), (127, 4), (128, 5), (130, 33), (300, 9), (257, 128)])
def test_sf_to_rowmajor_is_the_offset_map(orc, rows, nb):
    """The tests' gather from a 128x4-tiled scale buffer (used for NVFP4 and for
    MXFP4's cols/32 scale columns alike) reads, for every (row, column), the
    byte the C oracle's offset names, and reaches every real byte once."""
    size = orc.sf_bytes(rows, nb)
    where = orc.sf_to_rowmajor(np.arange(size), rows, nb)
    want = np.array([[orc.sf_offset(r, c, nb) for c in range(nb)] for r in range(rows)])
    assert np.array_equal(where, want)
    assert np.unique(where).size == rows * nb and where.max() < size


def test_gemm_reference_closed_form(orc):
    K, M, N = 64, 3, 5
    A = np.full((M, K), 1.5, np.float32)
    W = np.tile(np.arange(1, N + 1, dtype=np.float32)[:, None], (1, K))
    W[:, ::2] *= -1
    out, bnd = orc.gemm_rows(A, W, [0, 2])
    assert np.array_equal(out, np.zeros((2, N)))
    assert np.array_equal(bnd, np.tile(1.5 * K * np.arange(1, N + 1), (2, 1)))
    rng = np.random.default_rng(1)
    A = rng.standard_normal((7, 96)).astype(np.float32)
    W = rng.standard_normal((11, 96)).astype(np.float32)
    out, _ = orc.gemm_rows(A, W, [1, 6])
    assert np.allclose(out, (A.astype(np.float64) @ W.T.astype(np.float64))[[1, 6]], rtol=1e-12, atol=1e-12)


def test_gemm_reference_matmul_matches_loop(orc):
    rng = np.random.default_rng(2)
    A = (rng.standard_normal((9, 320)) * 3).astype(np.float32)
    W = rng.standard_t(4, (13, 320)).astype(np.float32)
    rows = [0, 4, 8]
    o1, b1 = orc.gemm_rows(A, W, rows)
    o2, b2 = orc.gemm_rows_matmul(A, W, rows)
    assert np.allclose(o1, o2, rtol=1e-13, atol=1e-12 * b1.max())
    assert np.allclose(b1, b2, rtol=1e-13)


# ------------------------------------------------- the page's worked example


def test_page5_block_size_mae_reproduced(orc):
    torch = pytest.importorskip("torch")
    torch.manual_seed(0)
    x = torch.randn(4096)
    x[::512] *= 20
    for block, mae in read_golden("page5_mae.txt"):
        assert f"{orc.mae_nearest_grid(x.numpy(), int(block)):.4f}" == mae


def test_page5_mae_falls_as_blocks_shrink_on_own_generator(orc):
    x = workloads.normal(1, 4096, seed=31).reshape(-1)
    x[::512] *= 20
    m = [orc.mae_nearest_grid(x, b) for b in (4096, 32, 16)]
    assert m[0] > m[1] > m[2]


def test_outlier_matrix_four_over_six_lowers_error(orc):
    x = workloads.outlier_matrix()
    y = workloads.bf16_to_f32(x).astype(np.float64)
    d46 = orc.dequantize(orc.quantize(x)).astype(np.float64)
    d6 = orc.dequantize(orc.quantize(x, scale_rule=orc.SCALE_6)).astype(np.float64)
    assert np.abs(d46 - y).mean() < np.abs(d6 - y).mean()
    assert ((d46 - y) ** 2).sum() < ((d6 - y) ** 2).sum()


# ------------------------------------------------- quantized linear backward


def _grid_matrix(rng, rows, cols, sign_of_six=1.0):
    """Values on the E2M1 grid, with a 6 wherever (i + j) % 16 == 0, so every
    16-run along a row or a column (and every 16 x 16 tile) has amax 6."""
    g = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    v = rng.choice(g, (rows, cols)) * rng.choice([-1.0, 1.0], (rows, cols))
    i, j = np.indices((rows, cols))
    v[(i + j) % 16 == 0] = 6.0 * sign_of_six
    return v


@pytest.mark.parametrize("weight_2d", [False, True])
def test_linear_backward_on_grid_inputs_recovers_exact_products(orc, weight_2d):
    """Inputs already on the NVFP4 grid (block amax 6 in every orientation)
    quantize losslessly up to the FP32 rounding of eff = 448 * (6/2688), so
    the backward's operands must dequantize to dY, W^T, dY^T, X^T and its
    products to dY W and dY^T X.  A transposed or swapped operand fails."""
    rng = np.random.default_rng(31)
    M, N, K = 64, 128, 48
    dy, x, w = _grid_matrix(rng, M, N), _grid_matrix(rng, M, K, -1.0), _grid_matrix(rng, N, K)
    ops = orc.linear_backward_operands(workloads.bf16_bits(dy), workloads.bf16_bits(x), workloads.bf16_bits(w),
                                       grad_rounding=orc.ROUND_RNE, wgrad_hadamard=False, weight_2d=weight_2d)
    for q, ref in zip(ops, (dy, w.T, dy.T, x.T)):
        assert (q.rows, q.cols) == ref.shape
        assert np.allclose(orc.dequantize(q), ref, rtol=1e-6, atol=0)
    (dx, dxb), (dw, dwb) = orc.linear_backward_rows(ops, np.arange(M), np.arange(N))
    assert np.all(np.abs(dx - dy @ w) <= 1e-6 * dxb)
    assert np.all(np.abs(dw - dy.T @ x) <= 1e-6 * dwb)


def test_linear_backward_recipe_preserves_weight_gradient(orc):
    """With SR on dY and the RHT along M on both weight-gradient operands, the
    transform cancels in dY^T X: the reference stays within NVFP4 error of the
    exact product, while an RHT on one operand only would leave it unrelated."""
    rng = np.random.default_rng(32)
    M, N, K = 256, 64, 32
    dy = rng.laplace(0, 1e-3, (M, N))
    x = rng.standard_normal((M, K))
    dyb, xb, wb = workloads.bf16_bits(dy), workloads.bf16_bits(x), workloads.bf16_bits(rng.standard_normal((N, K)))
    dy, x = workloads.bf16_to_f32(dyb).astype(np.float64), workloads.bf16_to_f32(xb).astype(np.float64)
    exact = dy.T @ x
    ops = orc.linear_backward_operands(dyb, xb, wb, sr_seed=5, hadamard_seed=9)
    _, (dw, _) = orc.linear_backward_rows(ops, np.arange(0), np.arange(N))
    rel = np.linalg.norm(dw - exact) / np.linalg.norm(exact)
    assert rel < 0.3
    one_sided = orc.quantize(xb, transpose=True)  # X^T without the transform
    bad, _ = orc.gemm_rows(orc.dequantize(ops[2]), orc.dequantize(one_sided), np.arange(N))
    assert np.linalg.norm(bad - exact) / np.linalg.norm(exact) > 0.8


# ------------------------------------------------------------ MXFP4 (R12)


def test_e8m0_all_bytes(orc):
    for b in range(255):
        assert orc.e8m0_decode(b) == float(np.ldexp(np.float64(1.0), b - 127))
    assert math.isnan(orc.e8m0_decode(255))


def test_mx_exponent_against_brute_force(orc):
    """X6 = floor(log2 a) - 2, found here by searching X over the integers for
    the largest 2^(X+2) <= a in exact (Python float) arithmetic."""
    rng = np.random.default_rng(41)
    vals = list((rng.random(400) * 10.0 ** rng.uniform(-40, 38, 400)).astype(np.float32))
    vals += [np.float32(v) for v in (1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 6.5, 7.99, 8.0, 2.0 ** -126, 2.0 ** -140, 3e38)]
    for a in vals:
        a = float(a)
        if a <= 0:
            continue
        X = -200
        while 2.0 ** (X + 3) <= a:  # the largest X with 2^(X+2) <= a
            X += 1
        want6 = max(-127, min(127, X))
        assert orc.mx_exponent(a, 6) == want6, a
        assert orc.mx_exponent(a, 4) == max(-127, min(127, X + 1)), a


def _mx_blocks_fp64(orc, x_bits):
    """Per block: FP64 squared errors of both candidates, from the pinned
    E2M1 rounding and the exponents, summed directly in the input's units."""
    y = workloads.bf16_to_f32(x_bits).astype(np.float64).reshape(-1, 32)
    out = []
    for blk in y:
        a = np.abs(blk).max()
        if a == 0:
            out.append((0.0, 0.0))
            continue
        errs = []
        for m in (6, 4):
            X = orc.mx_exponent(float(a), m)
            q = (blk.astype(np.float32) * np.float32(2.0 ** -X)).astype(np.float32)
            g = np.array([orc.e2m1_decode(c) for c in orc.e2m1_rne(q)], np.float64)
            errs.append(float(((blk - g * 2.0 ** X) ** 2).sum()))
        out.append(tuple(errs))
    return out


def test_mx_choice_against_fp64_brute_force(orc):
    rng = np.random.default_rng(42)
    x = workloads.bf16_bits(rng.standard_t(3, (16, 128)).astype(np.float32) * 10.0 ** rng.uniform(-3, 3, (16, 1)))
    q = orc.quantize_mx(x)
    errs = _mx_blocks_fp64(orc, x)
    near = 0
    for (e6, e4), c in zip(errs, q.choice.reshape(-1)):
        if abs(e4 - e6) <= 1e-6 * max(e6, 1e-300):
            near += 1
            continue
        assert c == (1 if e4 < e6 else 0)
    assert near < len(errs) // 4
    assert 0 < q.choice.sum() < q.choice.size  # both candidates occur


def test_mx_grid_membership_and_no_worse_than_six(orc):
    x = workloads.gradients(32, 256, seed=43)
    q, q6 = orc.quantize_mx(x), orc.quantize_mx(x, scale_rule=1)
    d = orc.dequantize_mx(q)
    for r in range(q.rows):
        for c in range(q.cols):
            byte = q.codes[r, c // 2]
            code = (byte >> 4) if c & 1 else (byte & 15)
            X = int(q.scales[r, c // 32]) - 127
            assert d[r, c] == np.float32(orc.e2m1_decode(code) * 2.0 ** X)
    xf = workloads.bf16_to_f32(x).astype(np.float64)
    e46 = ((orc.dequantize_mx(q) - xf) ** 2).reshape(-1, 32).sum(1)
    e6 = ((orc.dequantize_mx(q6) - xf) ** 2).reshape(-1, 32).sum(1)
    assert np.all(e46 <= e6 * (1 + 1e-6))
    assert e46.sum() < e6.sum()


def test_mx_hand_built_blocks(orc):
    """A maximum of 7.5 saturates to 6 under the MX exponent (error 1.5) but
    rounds to 8 = 2 * 4 under the coarser one (error 0.5): 4 must win.  A block
    on the fine grid with maximum 6 is exact under the MX exponent: 6 wins and
    the block comes back unchanged."""
    a = np.zeros(32, np.float32)
    a[0] = 7.5
    b = np.array([6.0, 0.5, -1.5, 3.0] * 8, np.float32)
    q = orc.quantize_mx(workloads.bf16_bits(np.stack([a, b])))
    assert q.choice[0, 0] == 1 and q.scales[0, 0] == 127 + 1  # X4 = floor(log2 7.5) - 2 + 1 = 1
    assert q.choice[1, 0] == 0 and q.scales[1, 0] == 127 + 0  # X6 = floor(log2 6) - 2 = 0
    assert np.array_equal(orc.dequantize_mx(q)[1], b)
    z = orc.quantize_mx(np.zeros((1, 32), np.uint16))
    assert z.scales[0, 0] == 0 and not z.codes.any() and z.choice[0, 0] == 0


def test_mx_non_finite_blocks_get_the_nan_scale(orc):
    """R12: a block holding a NaN or an infinity gets the E8M0 NaN byte 0xFF
    (the OCP MX specification: a NaN scale makes its whole block NaN), zero
    codes and choice 0, and dequantizes to NaN; the other blocks of the row are
    quantized as if it were not there."""
    rng = np.random.default_rng(44)
    x = rng.standard_normal((3, 128)).astype(np.float32)
    x[0, 5] = np.inf
    x[1, 40] = -np.inf
    x[2, 70] = np.nan
    bits = workloads.bf16_bits(np.nan_to_num(x, nan=0.0, posinf=0.0, neginf=0.0))
    bits[0, 5], bits[1, 40], bits[2, 70] = 0x7F80, 0xFF80, 0x7FC0  # +inf, -inf, NaN
    q = orc.quantize_mx(bits)
    bad = {(0, 0), (1, 1), (2, 2)}
    for r in range(3):
        for b in range(4):
            if (r, b) in bad:
                assert q.scales[r, b] == 0xFF and q.choice[r, b] == 0
                assert not q.codes[r, 16 * b: 16 * b + 16].any()
            else:
                assert q.scales[r, b] != 0xFF
    clean = bits.copy()
    clean[0, 5] = clean[1, 40] = clean[2, 70] = 0
    qc = orc.quantize_mx(clean)
    for r in range(3):
        for b in range(4):
            if (r, b) not in bad:
                assert q.scales[r, b] == qc.scales[r, b]
                assert np.array_equal(q.codes[r, 16 * b: 16 * b + 16], qc.codes[r, 16 * b: 16 * b + 16])
    d = orc.dequantize_mx(q)
    for r, b in bad:
        assert np.isnan(d[r, 32 * b: 32 * b + 32]).all()
    assert np.isfinite(d[0, 32:]).all()


def test_candidate_scales_round_exact_ties_to_even(orc):
    """Blocks whose maximum makes a_b / (M s_t) land exactly on the midpoint of
    two E4M3 values (s_t = 7/16384; found with exact rational arithmetic):
    the candidate's scale byte must be the even neighbour (round to nearest
    even, on the exact quotient)."""
    from fos_testutil import e4m3_tie_blocks

    bits, ties = e4m3_tie_blocks()
    assert sum(1 for t in ties if t[1] == 4) > 100 and sum(1 for t in ties if t[1] == 6) >= 4
    for rule, M in ((orc.SCALE_4, 4), (orc.SCALE_6, 6)):
        q = orc.quantize(bits, scale_rule=rule, sf_layout=orc.SF_ROWMAJOR)
        assert q.tensor_scale == 7 / 16384
        sf = q.sf.reshape(bits.shape[0], 4)
        for r, (_, m, even) in enumerate(ties):
            if m == M:
                assert sf[r, 1] == even, (r, hex(sf[r, 1]), hex(even))
