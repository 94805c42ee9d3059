"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every oracle function is checked here against something other than itself: a
closed form, a library routine (scipy's Sylvester Hadamard, numpy's integer
matmul), a published test vector, brute force on tiny inputs, or an invariant the
pages state.  Each test names the passage it pins.
"""
import itertools
import os

import numpy as np
import pytest
import scipy.linalg

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _matrix_of(fn, n):
    """Columns j = fn(e_j): the matrix of a linear row-map x -> fn(x) as x M."""
    eye = np.eye(n)
    return np.stack([fn(eye[i]) for i in range(n)])  # row i = e_i M


# --------------------------------------------------------------------------
# SplitMix64 / signs
# --------------------------------------------------------------------------

def test_splitmix64_published_vector():
    rows = _read_golden("splitmix64.txt")
    seed = int(rows[0][1])
    for idx, val in rows[1:]:
        assert oracle.splitmix64(seed, int(idx)) == int(val)


def test_signs_are_rademacher():
    s = oracle.signs(0x5EED, 1 << 16)
    assert set(np.unique(s).tolist()) == {-1, 1}
    # A fair +-1 sequence: mean within 5 sigma of 0, and both halves balanced.
    assert abs(s.mean()) < 5 / np.sqrt(s.size)
    # The sign is the top bit of the generator output, element by element.
    for i in (0, 1, 2, 1000, 65535):
        top = oracle.splitmix64(0x5EED, i) >> 63
        assert s[i] == (-1 if top else 1)


# --------------------------------------------------------------------------
# Hadamard transform (the H_n recursion of "Incoherence Processing via
# Randomized Hadamard Transforms")
# --------------------------------------------------------------------------

def test_hadamard_small_matrices_from_page_recursion():
    rows = _read_golden("hadamard_small.txt")
    i = 0
    while i < len(rows):
        n = int(rows[i][1])
        expect = np.array([[float(v) for v in rows[i + 1 + r]] for r in range(n)]) / np.sqrt(n)
        got = _matrix_of(lambda e: oracle.hadamard(e), n)
        np.testing.assert_allclose(got, expect, rtol=0, atol=1e-15)
        i += 1 + n


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64])
def test_hadamard_closed_form_and_orthogonality(n):
    h = _matrix_of(lambda e: oracle.hadamard(e), n)
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    pop = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    closed = (-1.0) ** pop / np.sqrt(n)
    np.testing.assert_allclose(h, closed, rtol=0, atol=1e-15)
    # Every entry is +-1/sqrt(n) and H H^T = I.
    np.testing.assert_allclose(np.abs(h), 1 / np.sqrt(n), rtol=1e-15)
    np.testing.assert_allclose(h @ h.T, np.eye(n), atol=1e-14)


@pytest.mark.parametrize("n", [2, 64, 1024, 4096])
def test_hadamard_equals_scipy_sylvester_matmul(n):
    rng = np.random.default_rng(n)
    x = rng.standard_normal((3, n))
    ref = x @ (scipy.linalg.hadamard(n).astype(np.float64) / np.sqrt(n))
    np.testing.assert_allclose(oracle.hadamard(x), ref, rtol=0, atol=1e-12 * np.abs(ref).max())


def test_hadamard_is_an_involution():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((4, 512))
    np.testing.assert_allclose(oracle.hadamard(oracle.hadamard(x)), x, atol=1e-13)


# --------------------------------------------------------------------------
# Randomized rotation R ("R = H_d diag(s)") and its invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("flags", [0, oracle.SIGNS_FIRST])
def test_rotation_matrix_closed_form(flags):
    n, seed = 32, 99
    s = oracle.signs(seed, n).astype(np.float64)
    h = scipy.linalg.hadamard(n) / np.sqrt(n)
    r = _matrix_of(lambda e: oracle.rotate(e[None], seed, flags)[0], n)
    expect = h @ np.diag(s) if flags == 0 else np.diag(s) @ h
    np.testing.assert_allclose(r, expect, atol=1e-15)
    np.testing.assert_allclose(r @ r.T, np.eye(n), atol=1e-14)


def test_rotation_forms_are_transposes():
    n, seed = 64, 5
    r0 = _matrix_of(lambda e: oracle.rotate(e[None], seed, 0)[0], n)
    r1 = _matrix_of(lambda e: oracle.rotate(e[None], seed, oracle.SIGNS_FIRST)[0], n)
    np.testing.assert_allclose(r0, r1.T, atol=1e-15)


@pytest.mark.parametrize("flags", [0, oracle.SIGNS_FIRST])
def test_rotation_preserves_norm_and_rms(flags):
    # "The Principle of Computational Invariance": ||xR||_2 = ||x||_2 and
    # therefore RMS(xR) = RMS(x), the RMSNorm denominator.
    rng = np.random.default_rng(11)
    x = rng.standard_normal((5, 4096)) * np.array([1, 10, 1e-3, 100, 1])[:, None]
    y = oracle.rotate(x, 0x5EED, flags)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    rms = lambda v: np.sqrt(np.mean(v * v, axis=1))
    np.testing.assert_allclose(rms(y), rms(x), rtol=1e-13)


@pytest.mark.parametrize("flags", [0, oracle.SIGNS_FIRST])
def test_computational_invariance_xw_equals_xr_rtw(flags):
    # "The Principle of Computational Invariance": Y = XW = (XR)(R^T W).
    # R^T W is formed column by column as the same row rotation applied to the
    # rows of W^T (the offline fold), so this also pins the fold's transpose and
    # sign side.
    rng = np.random.default_rng(3)
    d, k, b = 256, 40, 6
    x = rng.standard_normal((b, d))
    w = rng.standard_normal((d, k)) * 0.02
    xr = oracle.rotate(x, 0x5EED, flags)
    rtw = oracle.rotate(w.T, 0x5EED, flags).T
    np.testing.assert_allclose(xr @ rtw, x @ w, rtol=0, atol=1e-13 * np.abs(x @ w).max())


@pytest.mark.parametrize("d,attenuation,tol", [(int(a), float(b), float(c))
                                               for a, b, c in _read_golden("spike_attenuation.txt")])
@pytest.mark.parametrize("flags", [0, oracle.SIGNS_FIRST])
def test_single_spike_spreads_to_m_over_sqrt_d(d, attenuation, tol, flags):
    # "Incoherence Processing ...": x~_j = O(M/sqrt d); for one spike it is
    # exactly +-M/sqrt(d) in every coordinate.
    m = 100.0
    for pos in (0, 1, d // 3, d - 1):
        x = np.zeros((1, d))
        x[0, pos] = m
        y = oracle.rotate(x, 0x5EED, flags)[0]
        np.testing.assert_allclose(np.abs(y), m / np.sqrt(d), rtol=1e-13)
        assert abs(m / np.abs(y).max() - attenuation) <= tol + 1e-9


# --------------------------------------------------------------------------
# Quantizer and packing
# --------------------------------------------------------------------------

def _brute_force_code(r):
    """argmin_c |r - c| over the 16 INT4 codes, ties to the even code."""
    best = None
    for c in range(-8, 8):
        d = abs(r - c)
        if best is None or d < best[0] - 1e-300 or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def test_quant_matches_brute_force_and_invariants():
    rng = np.random.default_rng(21)
    y = rng.standard_normal((8, 256)) * rng.uniform(0.01, 100, size=(8, 1))
    codes, scales, ratio = oracle.quant_rows(y)
    for r in range(y.shape[0]):
        amax = np.abs(y[r]).max()
        assert scales[r] == pytest.approx(amax / 7, rel=1e-15)
        for j in range(0, 256, 7):
            assert codes[r, j] == _brute_force_code(y[r, j] / scales[r])
        # the absmax element maps to +-7; codes stay in [-7, 7]; error <= scale/2
        jm = np.argmax(np.abs(y[r]))
        assert codes[r, jm] == (7 if y[r, jm] > 0 else -7)
        assert codes[r].min() >= -7 and codes[r].max() <= 7
        assert np.all(np.abs(codes[r] * scales[r] - y[r]) <= scales[r] / 2 * (1 + 1e-12))


def test_quant_round_half_to_even_on_exact_ties():
    # absmax 7 -> scale 1 exactly, so y/scale = y and the ties are exact.
    y = np.array([[7.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, -6.5, 0.0]])
    codes, scales, _ = oracle.quant_rows(y)
    assert scales[0] == 1.0
    assert codes[0].tolist() == [7, 0, 2, 2, 0, -2, -2, 4, -6, 0]


def test_quant_degenerate_rows():
    codes, scales, _ = oracle.quant_rows(np.zeros((1, 16)))
    assert scales[0] == 0.0 and not codes.any()
    y = np.zeros((1, 16))
    y[0, 5] = -3e-7
    codes, scales, _ = oracle.quant_rows(y)
    assert codes[0, 5] == -7 and np.count_nonzero(codes) == 1


def test_pack_worked_example():
    rows = _read_golden("pack_example.txt")
    codes = np.array([int(v) for v in rows[0][1:]], dtype=np.int8)
    expect = np.array([int(v, 16) for v in rows[1][1:]], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.pack(codes[None])[0], expect)
    np.testing.assert_array_equal(oracle.unpack(expect[None], codes.size)[0], codes)


def test_pack_roundtrip_all_codes():
    codes = np.array(list(itertools.product(range(-8, 8), repeat=2)), dtype=np.int8).reshape(1, -1)
    packed = oracle.pack(codes)
    assert packed.shape == (1, codes.shape[1] // 2)
    # bit layout: low nibble = even element, two's complement
    lo = (packed[0] & 0xF).astype(np.int16)
    lo[lo >= 8] -= 16
    np.testing.assert_array_equal(lo, codes[0, 0::2])
    np.testing.assert_array_equal(oracle.unpack(packed, codes.shape[1]), codes)


def test_packed_size_is_a_quarter_of_16_bit():
    # "Why architecture matters here" (QuaRot page): four-bit values quarter the
    # bytes of sixteen-bit ones; the packed layout holds exactly n/2 bytes.
    x = np.random.default_rng(0).standard_normal((3, 128))
    out = oracle.fwht_quant(x, 1, oracle.SIGNS_FIRST)
    assert out["q"].nbytes * 4 == x.size * 2


# --------------------------------------------------------------------------
# Rotation + quantization pipeline, and the weight fold
# --------------------------------------------------------------------------

@pytest.mark.parametrize("flags", [0, oracle.SIGNS_FIRST])
def test_fwht_quant_is_rotate_then_quant_then_pack(flags):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 512))
    out = oracle.fwht_quant(x, 77, flags, want_y=True, want_ratio=True)
    # rotated rows: the explicit matrix product with scipy's Sylvester matrix
    s = oracle.signs(77, 512).astype(np.float64)
    h = scipy.linalg.hadamard(512) / np.sqrt(512)
    ref = (x @ h) * s if flags == 0 else (x * s) @ h
    np.testing.assert_allclose(out["y"], ref, atol=1e-12)
    codes = oracle.unpack(out["q"], 512)
    for r in range(6):
        sc = np.abs(ref[r]).max() / 7
        assert out["scales"][r] == np.float32(sc)
        for j in range(0, 512, 11):
            assert codes[r, j] == _brute_force_code(ref[r, j] / sc)


def test_rotation_reduces_int4_error_on_outlier_rows():
    # The pages' central claim ("a rotation turns a spiky, outlier-dominated
    # vector into a smooth one ... nearly lossless", QuaRot page, "Why
    # architecture matters here"): per-token INT4 error drops sharply after the
    # rotation on rows with 0.1%-style outlier channels.
    rng = np.random.default_rng(9)
    n = 4096
    x = rng.standard_normal((16, n))
    x[:, [10, 700, 2000, 4000]] *= 100
    def mse_after_quant(v):
        c, s, _ = oracle.quant_rows(v)
        return np.mean((c * s[:, None] - v) ** 2)
    plain = mse_after_quant(x)
    rot = oracle.rotate(x, 0x5EED, oracle.SIGNS_FIRST)
    rotated = mse_after_quant(rot)  # same norm, so the errors compare directly
    assert rotated < plain / 5  # measured about 8x on this seed


def test_weight_fold_then_quant_keeps_invariance_up_to_quant_error():
    # Offline fold W~ = R^T W ("Weight Absorption ...", 1. Offline Weight
    # Absorption), then per-output-channel INT4: the W4A4 product dequantized
    # approximates XW; with no quantization (fp64 rotated operands) it is exact.
    rng = np.random.default_rng(12)
    d, k, b = 1024, 32, 8
    x = rng.standard_normal((b, d))
    wt = rng.standard_normal((k, d)) * 0.02         # W^T, one output channel per row
    xa = oracle.fwht_quant(x, 5, oracle.SIGNS_FIRST, want_y=True)
    wf = oracle.fwht_quant(wt, 5, oracle.SIGNS_FIRST, want_y=True)
    exact = x @ wt.T
    np.testing.assert_allclose(xa["y"] @ wf["y"].T, exact, atol=1e-12)
    acc, y = oracle.w4a4_gemm(xa["q"], xa["scales"], wf["q"], wf["scales"], b, k, d)
    rel = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel < 0.25  # INT4 x INT4 on Gaussian data: roughly 15% relative error


# --------------------------------------------------------------------------
# W4A4 GEMM
# --------------------------------------------------------------------------

def _unpack_py(byte_row, k):
    """Independent pure-Python nibble decoding for the brute-force check."""
    out = []
    for b in byte_row:
        for v in (int(b) & 0xF, int(b) >> 4):
            out.append(v - 16 if v >= 8 else v)
    return out[:k]


def test_gemm_brute_force_tiny():
    rng = np.random.default_rng(31)
    M, N, K = 3, 5, 64
    aq = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    wq = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.uniform(0.1, 2, M).astype(np.float32)
    sw = rng.uniform(0.1, 2, N).astype(np.float32)
    acc, y = oracle.w4a4_gemm(aq, sa, wq, sw, M, N, K)
    for m in range(M):
        a = _unpack_py(aq[m], K)
        for n in range(N):
            w = _unpack_py(wq[n], K)
            s = sum(ai * wi for ai, wi in zip(a, w))
            assert acc[m, n] == s
            assert y[m, n] == s * float(sa[m]) * float(sw[n])


def test_gemm_matches_numpy_integer_matmul_and_entries():
    rng = np.random.default_rng(32)
    M, N, K = 17, 9, 256
    aq = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    wq = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.uniform(0.1, 2, M).astype(np.float32)
    sw = rng.uniform(0.1, 2, N).astype(np.float32)
    acc, y = oracle.w4a4_gemm(aq, sa, wq, sw, M, N, K)
    a = np.array([_unpack_py(r, K) for r in aq], dtype=np.int64)
    w = np.array([_unpack_py(r, K) for r in wq], dtype=np.int64)
    np.testing.assert_array_equal(acc, a @ w.T)
    ms = np.array([0, 16, 5, 3])
    cs = np.array([8, 0, 4, 4])
    e_acc, e_y = oracle.w4a4_gemm_entries(aq, sa, wq, sw, K, ms, cs)
    np.testing.assert_array_equal(e_acc, acc[ms, cs])
    np.testing.assert_array_equal(e_y, y[ms, cs])


def test_gemm_extreme_codes_fit_int32():
    K = 8192
    for byte, code in ((0x77, 7), (0x88, -8)):
        aq = np.full((1, K // 2), byte, np.uint8)
        acc, _ = oracle.w4a4_gemm(aq, np.ones(1, np.float32), aq, np.ones(1, np.float32), 1, 1, K)
        assert acc[0, 0] == code * code * K


# --------------------------------------------------------------------------
# KV cache write
# --------------------------------------------------------------------------

@pytest.mark.parametrize("flags", [0, oracle.SIGNS_FIRST])
def test_kv_is_per_head_rotation_then_quant(flags):
    rng = np.random.default_rng(41)
    T, H, D = 5, 3, 128
    k = rng.standard_normal((T, H, D))
    v = rng.standard_normal((T, H, D)) * 3
    out = oracle.kv_rotate_quant(k, v, 123, flags)
    s = oracle.signs(123, D).astype(np.float64)
    h = scipy.linalg.hadamard(D) / np.sqrt(D)
    for src, q, sc in ((k, out["kq"], out["ks"]), (v, out["vq"], out["vs"])):
        codes = oracle.unpack(q, D)
        for t in range(T):
            for hh in range(H):
                ref = (src[t, hh] @ h) * s if flags == 0 else (src[t, hh] * s) @ h
                scale = np.abs(ref).max() / 7
                assert sc[t, hh] == np.float32(scale)
                assert all(codes[t, hh, j] == _brute_force_code(ref[j] / scale)
                           for j in range(0, D, 9))


# --------------------------------------------------------------------------
# Attention read of the rotated INT4 cache ([QR] §End-to-end flow, "The KV
# cache"; §The architecture, the invariance box)
# --------------------------------------------------------------------------

def _rot_matrix(D, seed, flags):
    """R as an explicit matrix from scipy's Sylvester Hadamard: diag(s) H / sqrt(D)
    (signs first) or H diag(s) / sqrt(D)."""
    H = scipy.linalg.hadamard(D).astype(np.float64) / np.sqrt(D)
    S = np.diag(oracle.signs(seed, D).astype(np.float64))
    return S @ H if flags & 1 else H @ S


def _dequant_np(packed, scales, D):
    """Codes from the packed bytes by plain bit arithmetic (byte j: code 2j in the
    low nibble, 2j+1 in the high one, 4-bit two's complement), times the scale."""
    b = packed.astype(np.int64)
    nib = np.stack([b & 15, b >> 4], axis=-1).reshape(*packed.shape[:-1], D)
    codes = np.where(nib >= 8, nib - 16, nib).astype(np.float64)
    return codes * scales.astype(np.float64)[..., None]


def _attn_cache(T, H, D, seed_data, flags):
    rng = np.random.default_rng(seed_data)
    k = rng.standard_normal((T, H, D))
    v = rng.standard_normal((T, H, D))
    k[:, :, 3] *= 30.0
    return oracle.kv_rotate_quant(k, v, 321, flags)


@pytest.mark.parametrize("flags", [0, 1])
def test_attn_matches_explicit_matrices(flags):
    """Brute force with an explicit R: q~ = q R, scores on the dequantized rotated
    keys, numpy softmax, weighted rotated values, then o~ R^T."""
    T, H, D, M = 9, 3, 16, 2
    c = _attn_cache(T, H, D, 11, flags)
    q = np.random.default_rng(12).standard_normal((M, H, D))
    scale = 1.0 / np.sqrt(D)
    R = _rot_matrix(D, 321, flags)
    kh = _dequant_np(c["kq"], c["ks"], D)          # [T][H][D]
    vh = _dequant_np(c["vq"], c["vs"], D)
    ref_rot = np.empty((M, H, D))
    for m in range(M):
        for h in range(H):
            e = scale * (kh[:, h, :] @ (q[m, h] @ R))
            p = np.exp(e - e.max())
            p /= p.sum()
            ref_rot[m, h] = p @ vh[:, h, :]
    got_rot = oracle.attn_decode(q, c["kq"], c["ks"], c["vq"], c["vs"], 321, flags, scale, rotated_out=True)
    got = oracle.attn_decode(q, c["kq"], c["ks"], c["vq"], c["vs"], 321, flags, scale)
    np.testing.assert_allclose(got_rot, ref_rot, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got, ref_rot @ R.T, rtol=0, atol=1e-12)


@pytest.mark.parametrize("flags", [0, 1])
def test_attn_rotation_invariance(flags):
    """Scores through the rotated cache equal plain attention in the original
    basis on the cache taken back by R^T (R orthogonal): q~ . k^ = q . (k^ R^T)."""
    T, H, D = 17, 2, 32
    c = _attn_cache(T, H, D, 21, flags)
    q = np.random.default_rng(22).standard_normal((1, H, D)) * 2.0
    R = _rot_matrix(D, 321, flags)
    kb = _dequant_np(c["kq"], c["ks"], D) @ R.T     # original-basis keys
    vb = _dequant_np(c["vq"], c["vs"], D) @ R.T
    scale = 0.3
    got = oracle.attn_decode(q, c["kq"], c["ks"], c["vq"], c["vs"], 321, flags, scale)
    for h in range(H):
        e = scale * (kb[:, h, :] @ q[0, h])
        p = np.exp(e - e.max())
        p /= p.sum()
        np.testing.assert_allclose(got[0, h], p @ vb[:, h, :], rtol=0, atol=1e-12)


def test_attn_special_cases():
    """One cached token: the output is that token's value.  Identical keys, or a
    zero softmax scale: uniform weights, the mean of the values."""
    D, H = 8, 2
    c = _attn_cache(5, H, D, 31, 1)
    q = np.random.default_rng(32).standard_normal((1, H, D))
    vh = _dequant_np(c["vq"], c["vs"], D)
    one = oracle.attn_decode(q, c["kq"][:1], c["ks"][:1], c["vq"][:1], c["vs"][:1], 321, 1, 0.5, rotated_out=True)
    np.testing.assert_allclose(one[0], vh[0], rtol=0, atol=1e-15)
    zero = oracle.attn_decode(q, c["kq"], c["ks"], c["vq"], c["vs"], 321, 1, 0.0, rotated_out=True)
    np.testing.assert_allclose(zero[0], vh.mean(axis=0), rtol=0, atol=1e-14)
    kq_same = np.broadcast_to(c["kq"][:1], c["kq"].shape).copy()
    ks_same = np.broadcast_to(c["ks"][:1], c["ks"].shape).copy()
    same = oracle.attn_decode(q, kq_same, ks_same, c["vq"], c["vs"], 321, 1, 1.0, rotated_out=True)
    np.testing.assert_allclose(same[0], vh.mean(axis=0), rtol=0, atol=1e-14)


def test_attn_dominant_key_selects_its_value():
    """A key aligned with the rotated query at a large softmax scale takes all the
    weight (the others are below e^-50 relative)."""
    D, H, T, flags = 16, 1, 6, 1
    rng = np.random.default_rng(41)
    k = rng.standard_normal((T, H, D))
    v = rng.standard_normal((T, H, D))
    q = k[2:3].copy()                                  # query = key 2
    c = oracle.kv_rotate_quant(k, v, 321, flags)
    kh = _dequant_np(c["kq"], c["ks"], D)
    qr = q[0, 0] @ _rot_matrix(D, 321, flags)
    e = kh[:, 0, :] @ qr
    assert np.argmax(e) == 2
    scale = 60.0 / (e[2] - np.partition(e, -2)[-2])    # margin of 60 to the runner-up
    got = oracle.attn_decode(q, c["kq"], c["ks"], c["vq"], c["vs"], 321, flags, scale, rotated_out=True)
    vh = _dequant_np(c["vq"], c["vs"], D)
    np.testing.assert_allclose(got[0, 0], vh[2, 0], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Sizes that are not powers of two: n = m 2^k, R = diag(s)(H_m (x) H_{2^k})/sqrt(n)
# ([ROT] §The Computational Cost of Arbitrary Rotations, §SpinQuant: padding or
# products of Sylvester-compatible sizes)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("m", [12, 20, 28])
def test_paley_blocks_are_hadamard(m):
    """Entries +-1 and H H^T = m I exactly: the defining property of a Hadamard
    matrix, so H_m / sqrt(m) is orthogonal."""
    H = oracle.paley(m).astype(np.int64)
    assert set(np.unique(H)) == {-1, 1}
    np.testing.assert_array_equal(H @ H.T, m * np.eye(m, dtype=np.int64))
    if m in (12, 20):                      # Paley I: normalized first row, antisymmetric core
        assert np.all(H[0] == 1)
        core = H - np.eye(m, dtype=np.int64)
        np.testing.assert_array_equal(core, -core.T)


@pytest.mark.parametrize("m,b", [(12, 2), (12, 32), (20, 4), (20, 64), (28, 8), (28, 16)])
@pytest.mark.parametrize("flags", [0, 1])
def test_kron_rotation_matches_explicit_matrix(m, b, flags):
    """y = x R with R built by numpy's Kronecker product of H_m and scipy's
    Sylvester H_b (element a b + j of a row: segment a, offset j)."""
    n = m * b
    s = oracle.signs(77, n).astype(np.float64)
    K = np.kron(oracle.paley(m).astype(np.float64), scipy.linalg.hadamard(b).astype(np.float64)) / np.sqrt(n)
    R = np.diag(s) @ K if flags & 1 else K @ np.diag(s)
    x = np.random.default_rng(m + b).standard_normal((3, n))
    np.testing.assert_allclose(oracle.rotate(x, 77, flags), x @ R, rtol=0, atol=1e-12)


@pytest.mark.parametrize("n", [12 * 64, 20 * 128, 28 * 512])
def test_kron_rotation_norm_and_spike(n):
    """Orthogonal: norms kept.  Every entry of H_m (x) H_b is +-1, so a single spike
    of magnitude M lands as +-M/sqrt(n) on every coordinate."""
    x = np.random.default_rng(n).standard_normal((2, n))
    y = oracle.rotate(x, 5, 1)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    spike = np.zeros((1, n))
    spike[0, n // 3] = 250.0
    np.testing.assert_allclose(np.abs(oracle.rotate(spike, 5, 0)), 250.0 / np.sqrt(n), rtol=1e-12)


def test_kron_fwht_quant_is_rotate_then_quant_then_pack():
    n = 28 * 32
    x = np.random.default_rng(3).standard_normal((4, n)) * 3.0
    out = oracle.fwht_quant(x, 9, 1, want_y=True)
    y = oracle.rotate(x, 9, 1)
    np.testing.assert_allclose(out["y"], y, rtol=0, atol=0)
    codes, scales, _ = oracle.quant_rows(y)
    np.testing.assert_array_equal(out["q"], oracle.pack(codes))
    np.testing.assert_allclose(out["scales"], scales.astype(np.float32), rtol=0, atol=0)


# --------------------------------------------------------------------------
# W4A8 and per-group weight scales ([SQ] §The architecture: INT4 weights, INT8
# activations, per-channel or per-group scales; §End-to-end flow)
# --------------------------------------------------------------------------

def test_int8_quant_round_half_even_and_range():
    """scale = max|y|/127: the largest element maps to +-127; exact ties at .5
    round to even; every dequantized value lies within scale/2."""
    y = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -126.5, 3.0]])
    codes, scales, _ = oracle.quant_rows8(y)
    assert scales[0] == 1.0
    np.testing.assert_array_equal(codes[0], [127, 0, 2, 2, 0, -2, -126, 3])
    rng = np.random.default_rng(8)
    y = rng.standard_normal((5, 300)) * np.array([[1.0], [1e-3], [50.0], [7.0], [0.2]])
    codes, scales, _ = oracle.quant_rows8(y)
    assert np.all(np.abs(codes).max(axis=1) == 127)
    err = np.abs(codes * scales[:, None] - y)
    assert np.all(err <= scales[:, None] / 2 * (1 + 1e-12))
    zc, zs, _ = oracle.quant_rows8(np.zeros((1, 16)))
    assert zs[0] == 0.0 and not zc.any()


def test_fwht_quant8_is_rotate_then_int8():
    x = np.random.default_rng(9).standard_normal((4, 512)) * 4.0
    out = oracle.fwht_quant8(x, 3, 1)
    codes, scales, _ = oracle.quant_rows8(oracle.rotate(x, 3, 1))
    np.testing.assert_array_equal(out["q"], codes)
    np.testing.assert_array_equal(out["scales"], scales.astype(np.float32))


def test_group_quant_reduces_to_per_row_and_group_scales():
    """With one group per row the per-group fold is the per-row fold; with groups
    of 128 each group's scale is max|y_g|/7 of the rotated row."""
    x = np.random.default_rng(10).standard_normal((3, 1024))
    whole = oracle.fwht_quant_groups(x, 4, 1, 1024)
    row = oracle.fwht_quant(x, 4, 1)
    np.testing.assert_array_equal(whole["q"], row["q"])
    np.testing.assert_array_equal(whole["scales"][:, 0], row["scales"])
    g = oracle.fwht_quant_groups(x, 4, 1, 128)
    y = oracle.rotate(x, 4, 1).reshape(3, 8, 128)
    np.testing.assert_allclose(g["scales"], (np.abs(y).max(axis=2) / 7.0).astype(np.float32), rtol=0, atol=0)


@pytest.mark.parametrize("flags", [0, oracle.SIGNS_FIRST])
def test_group_quant_codes_and_scales_group_by_group(flags):
    """Per-group INT4 of the fold with groups of 128 inside rows of 1024: every
    code of every group equals the brute-force nearest code of y_g / (max|y_g|/7),
    with y = x R formed from scipy's explicit Sylvester matrix and the signs, and
    the packed bytes decoded by plain bit arithmetic.  The rotated rows are built
    with group magnitudes three orders apart (x = y R^T), so a code written at
    another group's offset, or a scale paired with the neighbouring group, fails."""
    n, group, seed = 1024, 128, 0x5EED
    ng = n // group
    rng = np.random.default_rng(44 + flags)
    mags = np.array([1e-3, 1.0, 30.0, 0.02, 5.0, 400.0, 0.5, 2e-2])
    y_target = rng.standard_normal((3, n)) * np.repeat(mags, group)[None, :]
    y_target[1] = y_target[1][::-1].copy()          # another magnitude order per row
    y_target[2] *= np.repeat(rng.permutation(mags), group)
    s = oracle.signs(seed, n).astype(np.float64)
    h = scipy.linalg.hadamard(n).astype(np.float64) / np.sqrt(n)
    r = np.diag(s) @ h if flags == oracle.SIGNS_FIRST else h @ np.diag(s)
    x = y_target @ r.T
    y = x @ r                                        # what the oracle should rotate x to
    out = oracle.fwht_quant_groups(x, seed, flags, group)
    assert out["q"].shape == (3, n // 2) and out["scales"].shape == (3, ng)
    codes = _unpack_np(out["q"], n)
    for row in range(3):
        for g in range(ng):
            yg = y[row, g * group:(g + 1) * group]
            sc = np.abs(yg).max() / 7.0
            assert out["scales"][row, g] == np.float32(sc)
            for j in range(group):
                rr = yg[j] / sc
                if abs(abs(rr - np.floor(rr)) - 0.5) < 1e-9:
                    continue                         # rounding-order tie: either code is right
                assert codes[row, g * group + j] == _brute_force_code(rr), (row, g, j)


def _unpack_np(packed, K):
    b = packed.astype(np.int64)
    nib = np.stack([b & 15, b >> 4], axis=-1).reshape(packed.shape[0], K)
    return np.where(nib >= 8, nib - 16, nib)


@pytest.mark.parametrize("group", [32, 128, 256])
def test_w4a8_gemm_brute_force(group):
    """Per group: numpy integer matmul of the INT8 codes with the INT4 codes
    (decoded here by plain bit arithmetic); y = sa * sum_g sw_g * acc_g."""
    M, N, K = 5, 7, 512
    rng = np.random.default_rng(group)
    qa = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    qw = rng.integers(0, 256, size=(N, K // 2)).astype(np.uint8)
    sa = rng.random(M).astype(np.float32) + 0.1
    sw = rng.random((N, K // group)).astype(np.float32) + 0.1
    w = _unpack_np(qw, K)
    a = qa.astype(np.int64)
    ng = K // group
    accg = np.stack([a[:, g * group:(g + 1) * group] @ w[:, g * group:(g + 1) * group].T for g in range(ng)])
    ref = sa.astype(np.float64)[:, None] * np.einsum("gmn,ng->mn", accg.astype(np.float64), sw.astype(np.float64))
    acc, y = oracle.w4a8_gemm(qa, sa, qw, sw, M, N, K, group)
    assert acc is None
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=0)
    swc = rng.random((N, 1)).astype(np.float32)
    acc, y = oracle.w4a8_gemm(qa, sa, qw, swc, M, N, K, K)
    np.testing.assert_array_equal(acc, a @ w.T)
