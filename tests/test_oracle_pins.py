"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against a closed form, an invariant, a
brute-force computation, a library routine on a special case, or a value fixed
by hand from the rules on the pages (fixtures under tests/golden/, each with its
citation).  A plausible mistake in the oracle (truncation instead of
ties-to-even, a /8 instead of /7, a transposed operand, a dropped LoRA term, a
wrong bias sign, fp16 scale rounding in the wrong direction) fails at least one.
"""
import os

import numpy as np
import pytest

import oracle
from synthetic import make_linear_case, random_codes

GOLD = os.path.join(os.path.dirname(__file__), "golden")
G = 64


def _f16(vals):
    return np.asarray(vals, np.float32).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------- fp16 routines
def test_f16_decode_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    ours = oracle.f16_to_f32_array(bits)
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(np.isinf(ours), np.isinf(ref))


def test_f16_roundtrip_exhaustive():
    for h in range(65536):
        e = (h >> 10) & 31
        if e == 31 and (h & 1023):
            continue  # NaN payloads are not preserved (canonical quiet NaN)
        assert oracle.f32_to_f16(oracle.f16_to_f32(h)) == h, hex(h)


def test_f16_encode_matches_numpy_rne():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(5000) * 1e-5).astype(np.float32),       # subnormal range
        (rng.standard_normal(2000) * 3e4).astype(np.float32),        # near overflow
    ])
    # exact midpoints between neighbouring fp16 values: ties must go to even
    h = np.arange(1, 0x7BFF, 97, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids, np.float32([65504, 65519.9, 65520, 6.1e-5, 0.0, -0.0])])
    ref = vals.astype(np.float16).view(np.uint16)
    ours = np.array([oracle.f32_to_f16(v) for v in vals], np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------- activation quantiser
def _read_ties():
    cases = []
    with open(os.path.join(GOLD, "act_quant_ties.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            gid, scale, xs, qs = [p.strip() for p in line.split("|")]
            cases.append((int(gid), np.float32(float(scale)),
                          [float(v) for v in xs.split()], [int(v) for v in qs.split()]))
    return cases


def test_act_quant_crafted_ties_golden():
    cases = _read_ties()
    X = np.zeros((1, G * len(cases)), np.float32)
    for gid, _, xs, _ in cases:
        X[0, gid * G: gid * G + len(xs)] = xs
    q, s = oracle.quantize_act(_f16(X))
    for gid, scale, xs, qs in cases:
        assert s[0, gid] == scale, (gid, s[0, gid], scale)
        exp = np.zeros(G, np.int8)
        exp[: len(qs)] = qs
        assert np.array_equal(q[0, gid * G:(gid + 1) * G], exp), gid


def test_act_quant_invariants():
    c = make_linear_case(96, 1024, 64, 32, seed=3)
    q, s = oracle.quantize_act(c.X)
    x = c.X.view(np.float16).astype(np.float64).reshape(96, 16, G)
    qq = q.astype(np.float64).reshape(96, 16, G)
    ss = s.astype(np.float64)[..., None]
    # reconstruction error within half a step (plus the rounding of x/s)
    assert np.all(np.abs(x - qq * ss) <= ss * (0.5 + 1e-6))
    # codes in [-7, 7]; the group's absmax element maps to +-7 with its sign
    assert q.min() >= -7 and q.max() <= 7
    am = np.abs(x).argmax(axis=2)
    top = np.take_along_axis(qq, am[..., None], axis=2)[..., 0]
    sign = np.sign(np.take_along_axis(x, am[..., None], axis=2)[..., 0])
    assert np.array_equal(top, 7 * sign)
    # scale is absmax/7 in fp32
    amax = np.abs(x).max(axis=2).astype(np.float32)
    assert np.array_equal(s, np.maximum(amax / np.float32(7), np.float32(1e-10)))


# -------------------------------------------------------------- weight quantiser
def test_weight_quant_closed_forms_golden():
    rows = []
    with open(os.path.join(GOLD, "weight_quant_closed_forms.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, amax, bits, val, code = [p.strip() for p in line.split("|")]
            rows.append((name, np.float32(float(amax)), int(bits, 16), float(val), int(code)))
    W = np.zeros((len(rows), G), np.float32)
    for i, (_, amax, _, _, _) in enumerate(rows):
        W[i, 5] = amax
        W[i, 9] = -amax * np.float32(0.5)
    q, s = oracle.quantize_weights(W)
    for i, (name, amax, bits, val, code) in enumerate(rows):
        assert int(s[i, 0]) == bits, name
        assert oracle.f16_to_f32(bits) == val, name
        assert q[i, 5] == code, name


def test_weight_quant_identity_closed_form():
    K = 256
    W = np.eye(K, dtype=np.float32)
    q, s = oracle.quantize_weights(W)
    for n in range(K):
        for g in range(K // G):
            if g == n // G:
                assert s[n, g] == 0x3092  # fp16(1/7) = 0.142822265625
            else:
                assert s[n, g] == 0x0400  # floor 2^-14
    assert np.array_equal(q, 7 * np.eye(K, dtype=np.int8))


def test_weight_quant_invariants():
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    q, s = oracle.quantize_weights(W)
    sv = s.view(np.float16).astype(np.float64)[..., None]
    w = W.astype(np.float64).reshape(64, 8, G)
    qq = q.astype(np.float64).reshape(64, 8, G)
    assert np.all(np.abs(w - qq * sv) <= sv * (0.5 + 1e-6))
    assert q.min() >= -8 and q.max() <= 7
    # fp16 scale = round-to-nearest of absmax/7 (numpy's RNE cast is the check)
    amax = np.abs(w).max(axis=2).astype(np.float32)
    exp = np.maximum(amax / np.float32(7), np.float32(2 ** -14)).astype(np.float16).view(np.uint16)
    assert np.array_equal(s, exp)


# ------------------------------------------------------------ integer partials
def test_group_partials_bruteforce_8x8x128():
    rng = np.random.default_rng(7)
    qA = random_codes(rng, (8, 128))
    qW = random_codes(rng, (8, 128))
    P = oracle.group_partials(qA, qW)
    for m in range(8):
        for n in range(8):
            for g in range(2):
                acc = 0
                for k in range(g * G, (g + 1) * G):
                    acc += int(qA[m, k]) * int(qW[n, k])
                assert P[m, n, g] == acc


def test_group_partials_extremes():
    qA = np.full((2, 128), -8, np.int8)
    qW = np.full((3, 128), -8, np.int8)
    assert np.all(oracle.group_partials(qA, qW) == 4096)
    alt = np.tile(np.array([7, -7], np.int8), 64)[None, :]
    assert np.all(oracle.group_partials(alt, np.full((1, 128), 5, np.int8)) == 0)
    # distinct rows/cols give distinct partials: a transposed operand would fail
    qA = np.zeros((2, 64), np.int8); qA[0, 0] = 1; qA[1, 1] = 1
    qW = np.zeros((3, 64), np.int8); qW[0, 0] = 2; qW[1, 1] = 3; qW[2, 0] = 5
    assert oracle.group_partials(qA, qW)[:, :, 0].tolist() == [[2, 0, 5], [0, 3, 0]]


# --------------------------------------------------------------- whole layer
def _dequant_reference(c, qA, sA, qW, sW, r=True):
    """Y from a dense fp64 matmul of the dequantised operands (the validation
    recipe of "INT4 Kernel Architecture, in depth", Failure modes)."""
    M, K = qA.shape
    xh = (qA.astype(np.float64).reshape(M, -1, G) * sA.astype(np.float64)[..., None]).reshape(M, K)
    N = qW.shape[0]
    wh = (qW.astype(np.float64).reshape(N, -1, G) * sW.view(np.float16).astype(np.float64)[..., None]).reshape(N, K)
    main = xh @ wh.T
    lora = 0.0
    if r and c.r:
        X = c.X.view(np.float16).astype(np.float64)
        lora = (X @ c.L_down.view(np.float16).astype(np.float64)) @ c.L_up.view(np.float16).astype(np.float64)
    cs = c.colscale.view(np.float16).astype(np.float64)
    b = c.bias.view(np.float16).astype(np.float64)
    return cs * (main + lora) + b


def test_linear_matches_dequantised_dense_reference():
    c = make_linear_case(40, 256, 48, 32, seed=11)
    ref = oracle.Reference(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    y = _dequant_reference(c, ref.qA, ref.sA, ref.qW, ref.sW)
    np.testing.assert_allclose(ref.Y, y, rtol=1e-12, atol=1e-12)


def test_linear_zero_input_gives_bias_exactly():
    c = make_linear_case(8, 128, 32, 32, seed=2)
    X0 = np.zeros_like(c.X)
    y = oracle.linear(X0, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    assert np.array_equal(y, np.broadcast_to(c.bias.view(np.float16).astype(np.float64), y.shape))


def test_linear_rank0_is_plain_grouped_gemm():
    c = make_linear_case(16, 192, 24, 0, seed=4)
    ref = oracle.Reference(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    y = _dequant_reference(c, ref.qA, ref.sA, ref.qW, ref.sW, r=False)
    np.testing.assert_allclose(ref.Y, y, rtol=1e-12, atol=1e-12)


def test_linear_zero_weights_is_textbook_lora():
    c = make_linear_case(12, 128, 40, 32, seed=6)
    W0 = np.zeros_like(c.W)
    y = oracle.linear(c.X, W0, c.L_down, c.L_up, c.colscale, c.bias)
    X = c.X.view(np.float16).astype(np.float64)
    lora = X @ c.L_down.view(np.float16).astype(np.float64) @ c.L_up.view(np.float16).astype(np.float64)
    exp = c.colscale.view(np.float16).astype(np.float64) * lora + c.bias.view(np.float16).astype(np.float64)
    np.testing.assert_allclose(y, exp, rtol=1e-12, atol=1e-13)


def test_linear_identity_weight_closed_form():
    K = N = 128
    c = make_linear_case(6, K, N, 0, seed=9)
    W = np.eye(N, K, dtype=np.float32)
    ref = oracle.Reference(c.X, W, c.L_down, c.L_up, c.colscale, c.bias)
    sw = 0.142822265625
    g = np.arange(N) // G
    main = 7 * sw * ref.sA.astype(np.float64)[:, g] * ref.qA.astype(np.float64)[:, np.arange(N)]
    exp = c.colscale.view(np.float16).astype(np.float64) * main + c.bias.view(np.float16).astype(np.float64)
    np.testing.assert_allclose(ref.Y, exp, rtol=1e-13, atol=1e-15)


def test_linear_sampled_matches_full():
    c = make_linear_case(20, 256, 36, 32, seed=12)
    full = oracle.linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, 20, 50)
    cols = rng.integers(0, 36, 50)
    s = oracle.linear_sampled(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias, rows, cols)
    assert np.array_equal(s, full[rows, cols])


# ---------------------------------------------------------------- stack glue
def test_f64_to_f16_matches_numpy_single_rounding():
    """The double -> binary16 encoder rounds once, to nearest even: numpy's
    float64 -> float16 cast does the same, over normals, subnormals, exact
    midpoints between binary16 neighbours and the overflow boundary."""
    rng = np.random.default_rng(5)
    vals = [rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000)]
    h = np.arange(0, 0x7c00, 7, dtype=np.uint16).view(np.float16).astype(np.float64)
    nxt = np.nextafter(h.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    mid = (h + nxt) / 2.0                            # exact midpoints: ties
    vals += [h, mid, -mid, np.nextafter(mid, 0.0), np.nextafter(mid, np.inf),
             np.array([65504.0, 65519.99, 65520.0, 1e-8, 2.0 ** -25, 3 * 2.0 ** -26, 0.0, -0.0])]
    v = np.concatenate(vals)
    got = oracle.f64_to_f16_array(v)
    want = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def _h(x):
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def test_rmsnorm_closed_forms():
    """Constant rows normalise to exactly 1 (or -1): c / sqrt(c^2 + 1e-6) is within
    2^-20 of 1 for |c| >= 1/8; a zero row stays zero; columns past K are ignored."""
    Y = np.zeros((4, 24), np.uint16)
    Y[0, :16] = _h(2.0)
    Y[1, :16] = _h(-0.125)
    Y[3, :16] = _h(3.0)
    Y[:, 16:] = _h(60000.0)                          # outside the K = 16 columns
    X = oracle.rmsnorm_f16(Y, 16)
    assert X.shape == (4, 16)
    assert np.all(X[0] == _h(1.0)) and np.all(X[1] == _h(-1.0)) and np.all(X[3] == _h(1.0))
    assert np.all(X[2] == 0)


def test_rmsnorm_invariants():
    """Odd in y (sign flip flips the output); scaling a row by a power of two
    (exact in fp16) changes only eps's share, so outputs move by at most one
    fp16 ulp, and rarely; output rows have mean square 1 up to the fp16 rounding."""
    rng = np.random.default_rng(6)
    y = rng.standard_normal((9, 256)).astype(np.float32)
    Y = _h(y)
    X = oracle.rmsnorm_f16(Y, 256)
    assert np.array_equal(oracle.rmsnorm_f16(_h(-y), 256), X ^ np.uint16(0x8000))
    X4 = oracle.rmsnorm_f16(_h(y * 4.0), 256)
    ulps = np.abs(X4.astype(np.int32) - X.astype(np.int32))
    assert ulps.max() <= 1 and (ulps > 0).mean() < 0.01
    xf = X.view(np.float16).astype(np.float64)
    assert np.all(np.abs((xf ** 2).mean(axis=1) - 1.0) < 2e-3)


# --------------------------------------------------------------------- W4A16
# "INT4 Kernel Architecture, in depth", "W4A16 versus W4A4": fp16 activations
# against the same dequantised INT4 weights.
def test_w4a16_one_hot_rows_read_single_weights():
    """Row m of X is e_{k_m}: y[m, n] = cs (qW[n, k] sW[n, k/64] + L_down[k] . L_up[:, n]) + bias
    -- one weight (and one LoRA row) per output, so a transposed or mis-grouped
    index shows up directly."""
    K, N, r = 256, 40, 16
    c = make_linear_case(6, K, N, r, seed=21)
    ks = np.array([0, 5, 63, 64, 130, 255])
    X = np.zeros((len(ks), K), np.float16)
    X[np.arange(len(ks)), ks] = 1.0
    y = oracle.w4a16_linear(X.view(np.uint16), c.W, c.L_down, c.L_up, c.colscale, c.bias)
    qW, sW = oracle.quantize_weights(c.W)
    Ld = c.L_down.view(np.float16).astype(np.float64)
    Lu = c.L_up.view(np.float16).astype(np.float64)
    cs = c.colscale.view(np.float16).astype(np.float64)
    b = c.bias.view(np.float16).astype(np.float64)
    for i, k in enumerate(ks):
        w = qW[:, k].astype(np.float64) * sW.view(np.float16)[:, k // G].astype(np.float64)
        np.testing.assert_allclose(y[i], cs * (w + Ld[k] @ Lu) + b, rtol=1e-14, atol=1e-14)


def test_w4a16_exact_homogeneity():
    """No LoRA, unit colscale, zero bias: scaling X by 2 scales y by 2 exactly."""
    c = make_linear_case(10, 192, 24, 0, seed=22)
    one = np.full(24, 0x3C00, np.uint16)
    zero = np.zeros(24, np.uint16)
    X2 = (c.X.view(np.float16) * np.float16(2)).view(np.uint16)
    y1 = oracle.w4a16_linear(c.X, c.W, None, None, one, zero)
    y2 = oracle.w4a16_linear(X2, c.W, None, None, one, zero)
    assert np.array_equal(y2, 2 * y1)


def test_w4a16_equals_w4a4_on_exactly_quantisable_inputs():
    """Activations that the W4A4 quantiser reproduces exactly (codes in [-7, 7]
    with a +-7 in every group, power-of-two scales) give the same layer through
    the integer-product path and through the W4A16 path."""
    M, K, N, r = 7, 256, 33, 16
    c = make_linear_case(M, K, N, r, seed=23)
    rng = np.random.default_rng(23)
    q = rng.integers(-7, 8, size=(M, K))
    q[:, ::G] = 7
    s = 2.0 ** rng.integers(-6, 2, size=(M, K // G))
    X = (q * np.repeat(s, G, axis=1)).astype(np.float16)
    assert np.array_equal(X.astype(np.float64), q * np.repeat(s, G, axis=1))
    qa, sa = oracle.quantize_act(X.view(np.uint16))
    assert np.array_equal(qa, q) and np.array_equal(sa.astype(np.float64), s)
    y4 = oracle.linear(X.view(np.uint16), c.W, c.L_down, c.L_up, c.colscale, c.bias)
    y16 = oracle.w4a16_linear(X.view(np.uint16), c.W, c.L_down, c.L_up, c.colscale, c.bias)
    np.testing.assert_allclose(y16, y4, rtol=1e-13, atol=1e-13)


def test_w4a16_matches_numpy_dequantised_matmul():
    c = make_linear_case(12, 320, 28, 32, seed=24)
    y = oracle.w4a16_linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    qW, sW = oracle.quantize_weights(c.W)
    wh = (qW.astype(np.float64).reshape(28, -1, G) * sW.view(np.float16).astype(np.float64)[..., None]).reshape(28, 320)
    X = c.X.view(np.float16).astype(np.float64)
    lora = X @ c.L_down.view(np.float16).astype(np.float64) @ c.L_up.view(np.float16).astype(np.float64)
    exp = c.colscale.view(np.float16).astype(np.float64) * (X @ wh.T + lora) + c.bias.view(np.float16).astype(np.float64)
    np.testing.assert_allclose(y, exp, rtol=1e-12, atol=1e-12)


# ---- asymmetric group-128 weights with a zero point ("INT4 Kernel
# Architecture, in depth", "How the weights are stored")
GA = 128


def _exact_asym_weights(rng, N, K):
    """Groups of integer multiples of s = 2^-e spanning exactly [-z s, (15 - z) s]:
    scale, zero point and codes are then exact, and dequantisation gives W back."""
    G = K // GA
    e = rng.integers(5, 9, size=(N, G))
    z = rng.integers(0, 16, size=(N, G))
    s = np.ldexp(1.0, -e)
    q = rng.integers(0, 16, size=(N, G, GA))
    q[:, :, 0], q[:, :, 1] = 0, 15  # both ends present: hi - lo = 15 s
    W = ((q - z[:, :, None]) * s[:, :, None]).reshape(N, K).astype(np.float32)
    return W, q.reshape(N, K), s, z


def test_asym_exact_groups_recover_codes_scale_zero_and_values():
    rng = np.random.default_rng(31)
    W, q, s, z = _exact_asym_weights(rng, 24, 512)
    qo, so, zo = oracle.quantize_weights_asym(W)
    assert np.array_equal(qo, q)
    assert np.array_equal(so.view(np.float16).astype(np.float64), s)
    assert np.array_equal(zo.view(np.float16).astype(np.float64), z)
    deq = (qo.reshape(24, -1, GA) - z[:, :, None]) * s[:, :, None]
    assert np.array_equal(deq.reshape(24, 512), W.astype(np.float64))


def test_asym_codes_range_and_half_step_bound():
    """Random groups (mixed signs, all-positive, all-negative): codes in 0..15,
    the group's minimum takes code 0, its maximum 14 or 15, and every value is
    within half a step of (q - zero) scale for the binary32 scale and zero."""
    rng = np.random.default_rng(32)
    N, K = 12, 1024
    W = rng.normal(0, 0.02, (N, K)).astype(np.float32)
    W[3] = np.abs(W[3]) + 1.0   # all positive: negative zero point
    W[4] = -np.abs(W[4]) - 0.5  # all negative: zero point above 15
    q, _, _ = oracle.quantize_weights_asym(W)
    assert q.min() >= 0 and q.max() <= 15
    g = W.reshape(N, -1, GA)
    qg = q.reshape(N, -1, GA)
    lo, hi = g.min(axis=2), g.max(axis=2)
    s32 = (np.maximum(hi - lo, np.float32(1e-8)) / np.float32(15)).astype(np.float32)
    z32 = np.rint(-lo / s32).astype(np.float32)
    n_i, g_i = np.indices(lo.shape)
    assert np.all(qg[n_i, g_i, g.argmin(axis=2)] == 0)
    assert np.all(np.isin(qg[n_i, g_i, g.argmax(axis=2)], (14, 15)))
    err = np.abs(g.astype(np.float64) - (qg - z32[:, :, None].astype(np.float64)) * s32[:, :, None])
    assert np.all(err <= 0.5001 * s32[:, :, None])


def test_w4a16_asym_on_exact_weights_equals_numpy_matmul():
    """With exactly representable weights the layer is the textbook
    colscale * (X W^T + X L_down L_up) + bias, in fp64 (numpy)."""
    rng = np.random.default_rng(33)
    M, N, K, r = 7, 40, 384, 16
    W, _, _, _ = _exact_asym_weights(rng, N, K)
    c = make_linear_case(M, K, N, r, seed=34)
    y = oracle.w4a16_asym_linear(c.X, W, c.L_down, c.L_up, c.colscale, c.bias)
    X = c.X.view(np.float16).astype(np.float64)
    Ld = c.L_down.view(np.float16).astype(np.float64)
    Lu = c.L_up.view(np.float16).astype(np.float64)
    ref = c.colscale.view(np.float16).astype(np.float64) * (X @ W.astype(np.float64).T + (X @ Ld) @ Lu) \
        + c.bias.view(np.float16).astype(np.float64)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_w4a16_asym_one_hot_rows_read_single_weights():
    """Row i of X is e_k: y = cs ((q[n,k] - zero[n,k/128]) scale[n,k/128] + L_down[k] . L_up[:, n]) + bias."""
    K, N, r = 512, 24, 16
    c = make_linear_case(4, K, N, r, seed=35)
    ks = np.array([0, 127, 128, 300, 511])
    X = np.zeros((len(ks), K), np.float16)
    X[np.arange(len(ks)), ks] = 1.0
    y = oracle.w4a16_asym_linear(X.view(np.uint16), c.W, c.L_down, c.L_up, c.colscale, c.bias)
    q, s, z = oracle.quantize_weights_asym(c.W)
    sf, zf = s.view(np.float16).astype(np.float64), z.view(np.float16).astype(np.float64)
    Ld = c.L_down.view(np.float16).astype(np.float64)
    Lu = c.L_up.view(np.float16).astype(np.float64)
    cs = c.colscale.view(np.float16).astype(np.float64)
    b = c.bias.view(np.float16).astype(np.float64)
    for i, k in enumerate(ks):
        w = (q[:, k] - zf[:, k // GA]) * sf[:, k // GA]
        np.testing.assert_allclose(y[i], cs * (w + Ld[k] @ Lu) + b, rtol=1e-14, atol=1e-14)


def test_asym_zero_point_of_zero_is_positive_zero():
    """A group whose minimum is 0 (either sign) gets zero point +0 (fp16 bits 0x0000)."""
    W = np.abs(np.random.default_rng(36).normal(0, 0.02, (2, 256))).astype(np.float32)
    W[0, 5] = 0.0
    W[1, 7] = -0.0
    W[:, 128:] += 0.05  # second group: minimum well above 0, negative zero point
    _, _, z = oracle.quantize_weights_asym(W)
    assert z[0, 0] == 0 and z[1, 0] == 0
    assert np.all(z[:, 1].view(np.float16) < 0)


# ---- SiLU(gate) * up on a fused gate|up output
def test_silu_mul_closed_forms_and_column_split():
    ln3 = np.log(3.0)
    Y = np.array([[0.0, ln3, 40.0, -40.0, 5.0, 2.0, 1.0, 1.0],
                  [1.0, 1.0, 1.0, 1.0, 0.0, ln3, 3.0, -2.0]])
    H = oracle.silu_mul(Y)
    assert H.shape == (2, 4)
    # row 0: gates (0, ln 3, 40, -40) times ups (5, 2, 1, 1)
    assert H[0, 0] == 0.0
    assert abs(H[0, 1] - 2 * 0.75 * ln3) < 1e-15
    assert abs(H[0, 2] - 40.0) < 1e-15             # silu(v) -> v for large v
    assert 0 > H[0, 3] > -40 * np.exp(-39.9)        # -> 0 from below for large -v
    # row 1: gates all 1 -> silu(1) = 1 / (1 + e^-1), times ups (0, ln 3, 3, -2)
    s1 = 1.0 / (1.0 + np.exp(-1.0))
    np.testing.assert_allclose(H[1], s1 * np.array([0.0, ln3, 3.0, -2.0]), rtol=1e-15)


def test_silu_mul_sampled_matches_full():
    c = make_linear_case(9, 128, 64, 16, seed=37)
    H = oracle.silu_mul_linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    rows, cols = np.array([0, 3, 8, 8]), np.array([0, 31, 5, 31])
    Hs = oracle.silu_mul_linear_sampled(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias, rows, cols)
    assert np.array_equal(Hs, H[rows, cols])


# ---- LoRA from the quantisation error ("W4A4 CUDA Kernel for Voice Clone", 2.1-2.2)
def planted_rank_case(N=96, K=256, rank=2, seed=41):
    """W = Q0 + D with Q0 = q0 s0 exactly quantisable (one element of each group at
    exactly 7 s0, the others |q0| <= 6) and D of rank `rank`, |D| <= 0.4 s0 and zero
    at the groups' first columns: the quantiser returns (q0, s0), so the error is D."""
    rng = np.random.default_rng(seed)
    G = K // 64
    s0 = np.ldexp(1.0, -rng.integers(6, 9, size=(N, G)))
    q0 = rng.integers(-6, 7, size=(N, K))
    q0[:, ::64] = 7
    u = rng.uniform(-1, 1, size=(N, rank))
    v = rng.uniform(-1, 1, size=(K, rank))
    v[::64] = 0.0
    D = u @ v.T
    smin = np.repeat(s0, 64, axis=1)
    D *= 0.4 * smin.min() / np.abs(D).max()
    W = (q0 * smin + D).astype(np.float32)
    return W, q0, s0, D


def test_svd_lora_recovers_a_planted_low_rank_error():
    W, q0, s0, D = planted_rank_case()
    best, errs = oracle.svd_lora(W, r=4, rounds=3)
    assert np.array_equal(best["codes"], q0)
    assert np.array_equal(oracle.f16_to_f32_array(best["scales"]).astype(np.float64), s0)
    L = (best["L_down"] @ best["L_up"]).T
    scale = np.linalg.norm(D)
    assert np.linalg.norm(L - D) <= 1e-6 * scale   # (fp32 rounding of W leaves ~1e-8)
    assert best["err"] <= 1e-5 * scale   # what is left is the fp32 rounding of W (~1e-7 here)


def test_svd_lora_full_rank_and_representable_weights():
    c = make_linear_case(1, 128, 32, 0, seed=42)
    best, _ = oracle.svd_lora(c.W, r=32, rounds=1)     # rank = min(N, K): no error left
    assert best["err"] <= 1e-12 * np.linalg.norm(c.W)
    W, q0, s0, _ = planted_rank_case(N=32, K=128, rank=1)
    Wq = (q0 * np.repeat(s0, 64, axis=1)).astype(np.float32)  # exactly representable
    best, errs = oracle.svd_lora(Wq, r=8, rounds=3)
    assert best["err"] == 0.0 and np.abs(best["L_up"]).max() == 0.0


def test_svd_lora_one_round_is_the_plain_quantiser_and_errors_fall():
    c = make_linear_case(1, 256, 64, 0, seed=43)
    best, errs = oracle.svd_lora(c.W, r=16, rounds=1)
    qW, sW = oracle.quantize_weights(c.W)
    assert np.array_equal(best["codes"], qW) and np.array_equal(best["scales"], sW)
    E = c.W.astype(np.float64) - oracle.dequantize_weights(qW, sW)
    # the rank-16 correction removes the 16 largest singular values' energy
    sv = np.linalg.svd(E, compute_uv=False)
    assert abs(best["err"] - np.sqrt((sv[16:] ** 2).sum())) <= 1e-9 * np.linalg.norm(E)
    best3, errs3 = oracle.svd_lora(c.W, r=16, rounds=3)
    assert errs3[0] == errs[0] and best3["err"] <= errs3[0]
    assert all(e2 < e1 for e1, e2 in zip(errs3[:-2], errs3[1:-1]))
