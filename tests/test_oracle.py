"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these checks retypes the oracle's formula: each compares it with a
hand-worked fixture, a closed form, an invariant that uses another route
(the bsums), or a library routine applied to a special case (numpy integer
matmul, numpy's fp16 conversion, float64 einsum).
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import read_golden


def _block_from_golden(name):
    x = np.zeros(256, dtype=np.float32)
    q = np.zeros(256, dtype=np.int64)
    d = bsums = None
    for tok in read_golden(name):
        if tok[0] == "d":
            d = float(tok[1])
        elif tok[0] == "bsums":
            bsums = [int(v) for v in tok[1:]]
        else:
            i = int(tok[0])
            x[i] = np.float32(tok[1])
            q[i] = int(tok[2])
    return x, q, d, bsums


# ---------------------------------------------------------------- fp16 scales

def test_fp16_decode_all_patterns_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.fp16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


# ---------------------------------------------------------------- q8_K

@pytest.mark.parametrize("name", ["q8K_scale_one.txt", "q8K_scale_two.txt"])
def test_quantize_hand_worked_blocks(name):
    x, q, d, bsums = _block_from_golden(name)
    xq = oracle.quantize_q8K(x[None, :])
    assert xq.shape == (1, 1)
    assert xq["d"][0, 0] == np.float32(d)
    assert np.array_equal(xq["qs"][0, 0].astype(np.int64), q)
    assert list(xq["bsums"][0, 0]) == bsums


def test_quantize_zero_block_and_mixed_row():
    x = np.zeros((2, 512), dtype=np.float32)
    x[1, 256:] = np.linspace(-3, 3, 256, dtype=np.float32)
    xq = oracle.quantize_q8K(x)
    for t, b in [(0, 0), (0, 1), (1, 0)]:
        assert xq["d"][t, b] == 0.0
        assert not xq["qs"][t, b].any() and not xq["bsums"][t, b].any()
    assert xq["d"][1, 1] > 0


def test_quantize_integer_blocks_are_exact():
    """Every block with absmax exactly 127 has d = 1 and q = x (the lesson of
    the ternary post's "stuff that went wrong": force it in *every* block)."""
    rng = np.random.default_rng(1)
    x = rng.integers(-126, 127, size=(5, 1024)).astype(np.float32)
    for t in range(5):
        for b in range(4):
            pos = rng.integers(0, 256)
            x[t, 256 * b + pos] = 127.0 if rng.random() < 0.5 else -127.0
    xq = oracle.quantize_q8K(x)
    assert np.all(xq["d"] == 1.0)
    assert np.array_equal(xq["qs"].reshape(5, 1024).astype(np.float32), x)


def test_quantize_invariants_on_gaussian_with_outliers():
    s = synth.seeds(3)
    x = synth.activations(4, 2048, s["acts"], s["outliers"])
    xq = oracle.quantize_q8K(x)
    qs = xq["qs"].astype(np.int64)                       # [4][8][256]
    xb = x.reshape(4, 8, 256).astype(np.float64)
    d = xq["d"].astype(np.float64)
    amax = np.abs(xb).max(axis=2)
    # the largest magnitude maps to +-127 and nothing exceeds it
    assert np.all(np.abs(qs).max(axis=2) == 127)
    # d = amax/127 to within one f32 rounding
    assert np.all(np.abs(d * 127 - amax) <= amax * 2.0 ** -23)
    # round to nearest: |x - d q| <= d/2 up to the two roundings in 127/amax and d
    err = np.abs(xb - d[..., None] * qs)
    assert np.all(err <= 0.5 * d[..., None] * (1 + 1e-5) + 1e-30)
    # bsums are the sums of 16 consecutive q
    assert np.array_equal(xq["bsums"].astype(np.int64), qs.reshape(4, 8, 16, 16).sum(axis=3))


def test_quantize_sign_symmetry():
    """q8_K is symmetric: -x quantizes to -q with the same scale."""
    s = synth.seeds(0)
    x = synth.activations(2, 1024, s["acts"])
    a, b = oracle.quantize_q8K(x), oracle.quantize_q8K(-x)
    assert np.array_equal(a["d"], b["d"])
    assert np.array_equal(a["qs"].astype(np.int64), -b["qs"].astype(np.int64))


# ---------------------------------------------------------------- pq2_0 format

def test_pq2_0_hand_encoded_block():
    rows = read_golden("pq2_0_bits.txt")
    want = bytes(int(v, 16) for v in [r for r in rows if r[0] == "bytes"][0][1:])
    w = np.zeros(128, dtype=np.int64)
    for r in rows:
        if r[0] != "bytes":
            w[int(r[0])] = int(r[1])
    codes = (w + 1).astype(np.uint8)[None, :]
    scales = np.array([[1.0]], dtype=np.float16)
    packed = synth.pack_pq2_0(codes, scales)
    assert packed.tobytes() == want
    w_dec, sb = oracle.decode_pq2_0(np.frombuffer(want, dtype=np.uint8), 1, 128)
    assert np.array_equal(w_dec[0].astype(np.int64), w)
    assert sb[0, 0] == 0x3C00


def test_page_constants(golden):
    c = {r[0]: r[1] for r in golden("page_constants.txt")}
    assert int(c["pq2_0_block_bytes"]) == oracle.PQ2_BYTES
    assert float(c["bits_per_weight"]) == oracle.PQ2_BYTES * 8 / oracle.GROUP
    assert float(c["bytes_per_weight"]) == oracle.PQ2_BYTES / oracle.GROUP
    # the scaled bound: 16 * sum over a group of u*q at u = 2, q = 127
    codes = np.full((1, 256), 2, dtype=np.uint8)
    w = synth.pack_pq2_0(codes, np.ones((1, 2), dtype=np.float16))
    x = np.full((1, 256), 127.0, dtype=np.float32)
    xq = oracle.quantize_q8K(x)
    S = oracle.groupsums(w, xq, 1, 256)                   # sum (u-1) q = 128 * 127
    bs = xq["bsums"][0, 0].astype(np.int64)
    u_dot_q = int(S[0, 0, 0]) + int(bs[:8].sum())          # sum u q = sum (u-1) q + sum q
    assert 16 * u_dot_q == int(c["scaled_group_bound"])


# ---------------------------------------------------------------- repack layout

def test_tq_layout_single_codes():
    for row, k, byte, shift in [[int(v) for v in r] for r in read_golden("tq_layout_bits.txt")]:
        codes = np.ones((32, 128), dtype=np.uint8)          # w = 0 everywhere ...
        codes[row, k] = 2                                   # ... except one +1
        sc = np.zeros((32, 1), dtype=np.float16)
        sc[5, 0] = 1.0
        wtq = oracle.repack(synth.pack_pq2_0(codes, sc), 32, 128)
        assert wtq.size == 1088
        diff = np.nonzero(wtq[:1024] != 0x55)[0]
        assert list(diff) == [byte], (row, k, diff)
        assert (int(wtq[byte]) >> shift) & 3 == 2
        assert wtq[1024 + 10] == 0x00 and wtq[1024 + 11] == 0x3C   # row 5: fp16 1.0
        assert not np.any(np.delete(wtq[1024:], [10, 11]))


@pytest.mark.parametrize("rows,cols", [(32, 256), (100, 512), (1, 256), (65, 1024)])
def test_repack_roundtrip_on_random_bytes(rows, cols):
    """unrepack(repack(b)) == b for arbitrary bytes, code 3 included: the
    repack is a pure permutation of bits."""
    rng = np.random.default_rng(rows * 7 + cols)
    b = rng.integers(0, 256, size=rows * cols // 128 * 34, dtype=np.uint8)
    wtq = oracle.repack(b, rows, cols)
    assert wtq.size == -(-rows // 32) * (cols // 128) * 1088
    assert np.array_equal(oracle.unrepack(wtq, rows, cols), b)
    # the same multiset of codes (plus padding rows of code 1)
    pad = (-(-rows // 32) * 32 - rows) * cols
    cb = np.unpackbits(b.reshape(-1, 34)[:, 2:], bitorder="little").reshape(-1, 2)
    ct = np.unpackbits(wtq.reshape(-1, 1088)[:, :1024], bitorder="little").reshape(-1, 2)
    hist = lambda c: np.bincount(c[:, 0] + 2 * c[:, 1], minlength=4)
    assert np.array_equal(hist(ct) - np.array([0, pad, 0, 0]), hist(cb))


# ---------------------------------------------------------------- group sums

def _pack(w, scales=None):
    rows, cols = w.shape
    if scales is None:
        scales = np.ones((rows, cols // 128), dtype=np.float16)
    return synth.pack_pq2_0((w + 1).astype(np.uint8), scales)


def _q8K_exact(q_int):
    """A q8_K array with given integer values and d = 1 (absmax 127 forced)."""
    x = q_int.astype(np.float32).copy()
    ntok, cols = x.shape
    for t in range(ntok):
        for b in range(cols // 256):
            if np.abs(x[t, 256 * b:256 * (b + 1)]).max() != 127:
                x[t, 256 * b + 255] = 127.0
    xq = oracle.quantize_q8K(x)
    assert np.all(xq["d"] == 1.0)
    return xq, x


def test_groupsum_hand_worked_examples():
    q = np.full((1, 256), 127, dtype=np.int64)
    xq, _ = _q8K_exact(q)
    for wval, want in [(1, 16256), (-1, -16256), (0, 0)]:
        w = np.full((1, 256), wval, dtype=np.int64)
        S = oracle.groupsums(_pack(w), xq, 1, 256)
        assert list(S[0, 0]) == [want, want]
    # alternating +1/-1 against a constant activation cancels exactly
    w = np.tile(np.array([1, -1]), (1, 128))
    assert list(oracle.groupsums(_pack(w), xq, 1, 256)[0, 0]) == [0, 0]
    # w = +1 on even k only, q = k - 64 within group 0: sum over even k of (k - 64)
    qk = np.zeros((1, 256), dtype=np.int64)
    qk[0, :128] = np.arange(128) - 64
    xq2, x2 = _q8K_exact(qk)
    w = np.zeros((1, 256), dtype=np.int64)
    w[0, 0:128:2] = 1
    S = oracle.groupsums(_pack(w), xq2, 1, 256)
    assert S[0, 0, 0] == sum(k - 64 for k in range(0, 128, 2)) == -64
    assert S[0, 0, 1] == 0


def test_groupsum_equals_u_dot_minus_bsums():
    """sum (u-1) q = sum u q - sum y, with sum y over 128 values taken from the
    8 partial sums q8_K carries (ternary post, "the trick with 4 and 16")."""
    s = synth.seeds(2)
    rows, cols, ntok = 48, 1024, 3
    wpq = synth.pq2_0_weights(rows, cols, 2)
    x = synth.activations(ntok, cols, s["acts"])
    xq = oracle.quantize_q8K(x)
    S = oracle.groupsums(wpq, xq, rows, cols)
    u = synth.ternary_codes(rows, cols, s["weights"]).astype(np.int64)
    q = xq["qs"].reshape(ntok, cols).astype(np.int64)
    udq = np.einsum("rgk,tgk->trg", u.reshape(rows, cols // 128, 128), q.reshape(ntok, cols // 128, 128))
    ysum = xq["bsums"].astype(np.int64).reshape(ntok, cols // 128, 8).sum(axis=2)
    assert np.array_equal(S, udq - ysum[:, None, :])
    # the unscaled bound |isum| <= 128 * 127
    assert np.abs(S).max() <= 16256


def test_groupsum_matches_library_matmul_nonsquare():
    rng = np.random.default_rng(5)
    rows, cols, ntok = 7, 768, 5
    w = rng.integers(-1, 2, size=(rows, cols))
    q = rng.integers(-127, 128, size=(ntok, cols))
    xq, _ = _q8K_exact(q)
    qv = xq["qs"].reshape(ntok, cols).astype(np.int64)
    S = oracle.groupsums(_pack(w), xq, rows, cols)
    for g in range(cols // 128):
        sl = slice(128 * g, 128 * (g + 1))
        assert np.array_equal(S[:, :, g], qv[:, sl] @ w[:, sl].T)


# ---------------------------------------------------------------- matmul

def test_matmul_exact_integer_mode():
    """d_w = 1 and d_x = 1: y is exactly the integer product W x (the pages'
    integer oracle: batch widths 1-5, 7, 8; rows 4, 8, 12; inner 256-1024)."""
    rng = np.random.default_rng(11)
    for ntok in (1, 2, 3, 4, 5, 7, 8):
        for rows in (4, 8, 12):
            for cols in (256, 512, 1024):
                w = rng.integers(-1, 2, size=(rows, cols))
                q = rng.integers(-127, 128, size=(ntok, cols))
                xq, x = _q8K_exact(q)
                y, a = oracle.matmul(_pack(w), xq, rows, cols)
                want = x.astype(np.int64) @ w.T
                assert np.array_equal(y.astype(np.int64), want)
                S = oracle.groupsums(_pack(w), xq, rows, cols)
                assert np.array_equal(a, np.abs(S).sum(axis=2).astype(np.float64))


def test_matmul_extremes_and_constants():
    rows, cols = 4, 512
    for wv in (-1, 0, 1):
        for qv in (-127, 0, 127):
            w = np.full((rows, cols), wv)
            q = np.full((2, cols), qv)
            xq, x = _q8K_exact(q)
            y, _ = oracle.matmul(_pack(w), xq, rows, cols)
            assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ w.T)


def test_matmul_float_path_against_f64_brute_force():
    s = synth.seeds(3)
    rows, cols, ntok = 40, 2048, 6
    wpq = synth.pq2_0_weights(rows, cols, 3)
    x = synth.activations(ntok, cols, s["acts"], s["outliers"])
    xq = oracle.quantize_q8K(x)
    y, a = oracle.matmul(wpq, xq, rows, cols)
    w = synth.ternary_codes(rows, cols, s["weights"]).astype(np.float64) - 1
    dw = synth.group_scales(rows, cols, s["scales"]).astype(np.float64)
    wd = (w.reshape(rows, -1, 128) * dw[:, :, None]).reshape(rows, cols)
    xd = (xq["qs"].astype(np.float64) * xq["d"].astype(np.float64)[..., None]).reshape(ntok, cols)
    ref = np.einsum("tk,rk->tr", xd, wd)
    assert np.all(np.abs(y.astype(np.float64) - ref) <= 2.0 ** -24 * np.abs(ref) + 1e-12 * a)
    # scale by 2 on every weight scale doubles y exactly
    dw2 = (dw * 2).astype(np.float16)
    codes = synth.ternary_codes(rows, cols, s["weights"])
    y2, _ = oracle.matmul(synth.pack_pq2_0(codes, dw2), xq, rows, cols)
    assert np.array_equal(y2, 2 * y)


# ---------------------------------------------------------------- generator

def test_splitmix64_published_vector():
    """splitmix64 with seed 0: the reference outputs of Vigna's published code."""
    v = synth.splitmix64(0, 0, 3)
    assert [int(a) for a in v] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_generator_rows_are_addressable():
    full = synth.pq2_0_weights(64, 512, 1)
    part = synth.pq2_0_weights(8, 512, 1, row0=40)
    per_row = 512 // 128 * 34
    assert np.array_equal(full[40 * per_row:48 * per_row], part)
    u = synth.ternary_codes(300, 1024, 77)
    frac = np.bincount(u.ravel(), minlength=3) / u.size
    assert np.all(np.abs(frac - 1 / 3) < 0.01)
    sc = synth.group_scales(300, 1024, 78).astype(np.float32)
    assert sc.min() >= np.float16(0.005) and sc.max() <= np.float16(0.02)
