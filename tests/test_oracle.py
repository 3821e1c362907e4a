"""Pins for the CPU oracle: each test ties it to something other than itself
(brute force written differently, library routines on tiny inputs, closed
forms, hand-worked values, invariants of the mathematics, golden fixtures).
No GPU is needed."""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------- independent routes

def im2col_conv_numpy(x, w, bias, strides, pads, dilations, group, dtype=np.float64):
    """im2col + matrix product per group (the page's CPU-executor method in the
    "Kyanite" README, section "CPU executor"), written independently of the oracle."""
    N, C, H, W = x.shape
    K, Cg, R, S = w.shape
    sh, sw = strides
    pt, pl, pb, pr = pads
    dh, dw = dilations
    xp = np.zeros((N, C, H + pt + pb, W + pl + pr), dtype=dtype)
    xp[:, :, pt:pt + H, pl:pl + W] = x
    Ho = (H + pt + pb - dh * (R - 1) - 1) // sh + 1
    Wo = (W + pl + pr - dw * (S - 1) - 1) // sw + 1
    cols = np.empty((N, C, R, S, Ho, Wo), dtype=dtype)
    for r in range(R):
        for s in range(S):
            cols[:, :, r, s] = xp[:, :, r * dh: r * dh + sh * (Ho - 1) + 1: sh,
                                  s * dw: s * dw + sw * (Wo - 1) + 1: sw]
    Kg = K // group
    out = np.empty((N, K, Ho, Wo), dtype=dtype)
    for g in range(group):
        a = cols[:, g * Cg:(g + 1) * Cg].reshape(N, Cg * R * S, Ho * Wo)
        b = w[g * Kg:(g + 1) * Kg].reshape(Kg, Cg * R * S).astype(dtype)
        out[:, g * Kg:(g + 1) * Kg] = np.einsum("kj,njp->nkp", b, a).reshape(N, Kg, Ho, Wo)
    if bias is not None:
        out += np.asarray(bias, dtype=dtype).reshape(1, K, 1, 1)
    return out


def torch_conv_f64(x, w, bias, strides, pads, dilations, group):
    pt, pl, pb, pr = pads
    xt = torch.nn.functional.pad(torch.from_numpy(np.asarray(x, np.float64)), (pl, pr, pt, pb))
    b = None if bias is None else torch.from_numpy(np.asarray(bias, np.float64))
    return torch.nn.functional.conv2d(xt, torch.from_numpy(np.asarray(w, np.float64)), b,
                                      stride=strides, dilation=dilations, groups=group).numpy()


def random_cases(count, seed):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < count:
        N = int(rng.integers(1, 3))
        R, S = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        st = (int(rng.integers(1, 4)), int(rng.integers(1, 4)))
        dl = (int(rng.integers(1, 3)), int(rng.integers(1, 3)))
        pads = tuple(int(v) for v in rng.integers(0, 3, size=4))
        H, W = int(rng.integers(1, 8)), int(rng.integers(1, 8))
        kind = int(rng.integers(0, 3))
        if kind == 0:
            group = 1
            C, K = int(rng.integers(1, 9)), int(rng.integers(1, 9))
        elif kind == 1:
            group = 2
            C, K = 2 * int(rng.integers(1, 5)), 2 * int(rng.integers(1, 5))
        else:
            C = int(rng.integers(1, 9))
            group, K = C, C * int(rng.integers(1, 3))
        Ho = (H + pads[0] + pads[2] - dl[0] * (R - 1) - 1) // st[0] + 1
        Wo = (W + pads[1] + pads[3] - dl[1] * (S - 1) - 1) // st[1] + 1
        if Ho < 1 or Wo < 1:
            continue
        cases.append((N, C, H, W, K, R, S, st, pads, dl, group))
    return cases


# ------------------------------------------------------------------ brute force

@pytest.mark.parametrize("case", random_cases(80, 7))
def test_conv_matches_im2col_and_torch(case):
    N, C, H, W, K, R, S, st, pads, dl, group = case
    rng = np.random.default_rng(hash(case) & 0xFFFF)
    x = rng.standard_normal((N, C, H, W))
    w = rng.standard_normal((K, C // group, R, S))
    bias = rng.standard_normal(K) if rng.integers(0, 2) else None
    z = oracle.conv2d(x, w, bias, st, pads, dl, group)
    ref1 = im2col_conv_numpy(x, w, bias, st, pads, dl, group)
    ref2 = torch_conv_f64(x, w, bias, st, pads, dl, group)
    assert z.shape == ref1.shape == ref2.shape
    scale = max(1.0, float(np.abs(ref1).max()))
    assert np.abs(z - ref1).max() <= 1e-12 * scale
    assert np.abs(z - ref2).max() <= 1e-12 * scale
    # the point evaluator returns the same numbers
    pts = np.array(list(itertools.product(range(N), range(K), range(z.shape[2]),
                                          range(z.shape[3]))), dtype=np.int64)
    zp = oracle.conv2d_points(x, w, bias, st, pads, dl, group, pts)
    assert np.array_equal(zp, z.reshape(-1))


@pytest.mark.parametrize("case", random_cases(40, 11))
def test_int8_conv_matches_integer_im2col(case):
    N, C, H, W, K, R, S, st, pads, dl, group = case
    rng = np.random.default_rng(hash(case) & 0xFFFF)
    x = rng.integers(-128, 128, (N, C, H, W)).astype(np.int8)
    w = rng.integers(-128, 128, (K, C // group, R, S)).astype(np.int8)
    acc = oracle.conv2d_s8(x, w, st, pads, dl, group)
    ref = im2col_conv_numpy(x.astype(np.int64), w.astype(np.int64), None, st, pads, dl, group,
                            dtype=np.int64)
    assert acc.dtype == np.int64 and np.array_equal(acc, ref)
    pts = np.array(list(itertools.product(range(N), range(K), range(acc.shape[2]),
                                          range(acc.shape[3]))), dtype=np.int64)
    assert np.array_equal(oracle.conv2d_s8_points(x, w, st, pads, dl, group, pts),
                          acc.reshape(-1))


def test_rejects_bad_arguments():
    x = np.zeros((1, 4, 5, 5))
    with pytest.raises(ValueError):
        oracle.conv2d(x, np.zeros((2, 3, 3, 3)))               # C/group mismatch
    with pytest.raises(ValueError):
        oracle.conv2d(x, np.zeros((2, 4, 7, 7)))               # window larger than input
    with pytest.raises(ValueError):
        oracle.conv2d_points(x, np.zeros((2, 4, 3, 3)), None, (1, 1), (0, 0, 0, 0), (1, 1), 1,
                             np.array([[0, 2, 0, 0]]))          # k out of range


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("C,H,W,R,S,st,pads,dl", [
    (16, 9, 9, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1)),
    (3, 12, 12, 7, 7, (2, 2), (3, 3, 3, 3), (1, 1)),
    (5, 10, 8, 3, 2, (2, 1), (2, 0, 1, 1), (2, 1)),
    (64, 6, 6, 1, 1, (1, 1), (0, 0, 0, 0), (1, 1)),
])
def test_all_ones_counts_valid_taps(C, H, W, R, S, st, pads, dl):
    """All-ones x and W: each output is C times the number of taps that land
    inside the image; C*R*S in the interior."""
    K = 3
    z = oracle.conv2d(np.ones((1, C, H, W)), np.ones((K, C, R, S)), None, st, pads, dl, 1)
    Ho, Wo = z.shape[2:]
    for oh in range(Ho):
        nr = sum(0 <= oh * st[0] - pads[0] + r * dl[0] < H for r in range(R))
        for ow in range(Wo):
            ns = sum(0 <= ow * st[1] - pads[1] + s * dl[1] < W for s in range(S))
            assert np.all(z[0, :, oh, ow] == C * nr * ns)
    if R == 3 and H >= 3:
        assert z[0, 0, 1, 1] == C * R * S


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split(None, 1)
            out.setdefault(key, []).append(vals[0] if vals else "")
    return out


def test_golden_allones_matmul_64():
    g = _read_golden("allones_1x1_c64.txt")
    N, C, H, W, K, R, S, sh, sw, pt, pl, pb, pr, dh, dw, group = map(int, g["shape"][0].split())
    z = oracle.conv2d(np.ones((N, C, H, W)), np.ones((K, C // group, R, S)), None, (sh, sw),
                      (pt, pl, pb, pr), (dh, dw), group)
    assert z.size == int(g["expected_count"][0])
    assert np.all(z == float(g["expected_all"][0]))


def test_golden_handworked():
    g = _read_golden("handworked_2x2.txt")
    x = np.array([float(v) for v in g["x"][0].split()]).reshape(1, 1, 3, 3)
    w = np.array([float(v) for v in g["w"][0].split()]).reshape(1, 1, 2, 2)
    assert len(g["case"]) == 5
    for case in g["case"]:
        attrs, shape, vals = case.split("|")
        sh, sw, pt, pl, pb, pr, dh, dw = map(int, attrs.split())
        ho, wo = map(int, shape.split())
        want = np.array([float(v) for v in vals.split()]).reshape(1, 1, ho, wo)
        z = oracle.conv2d(x, w, None, (sh, sw), (pt, pl, pb, pr), (dh, dw), 1)
        assert np.array_equal(z, want), case
        xi = x.astype(np.int8)
        wi = w.astype(np.int8)
        assert np.array_equal(oracle.conv2d_s8(xi, wi, (sh, sw), (pt, pl, pb, pr), (dh, dw), 1),
                              want.astype(np.int64))


def test_golden_relu6():
    g = _read_golden("relu6_clamp.txt")
    u = np.array([float(v) for v in g["u"][0].split()])
    assert np.array_equal(oracle.activation(u, oracle.ACT_RELU),
                          np.array([float(v) for v in g["relu"][0].split()]))
    assert np.array_equal(oracle.activation(u, oracle.ACT_RELU6),
                          np.array([float(v) for v in g["relu6"][0].split()]))
    assert np.array_equal(oracle.activation(u, oracle.ACT_NONE), u)
    assert np.array_equal(oracle.activation(u, oracle.ACT_CLIP, -1.0, 2.0),
                          np.clip(u, -1.0, 2.0))


def test_1x1_conv_is_matmul():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 24, 5, 7))
    w = rng.standard_normal((40, 24, 1, 1))
    z = oracle.conv2d(x, w)
    for n in range(2):
        ref = w[:, :, 0, 0] @ x[n].reshape(24, -1)
        assert np.allclose(z[n].reshape(40, -1), ref, rtol=1e-13, atol=1e-13)


def test_identity_kernel_returns_input():
    rng = np.random.default_rng(4)
    C = 6
    x = rng.standard_normal((2, C, 9, 5))
    w = np.zeros((C, C, 3, 3))
    for c in range(C):
        w[c, c, 1, 1] = 1.0
    assert np.array_equal(oracle.conv2d(x, w, None, (1, 1), (1, 1, 1, 1)), x)


def test_depthwise_is_per_channel_conv():
    rng = np.random.default_rng(5)
    C = 5
    x = rng.standard_normal((2, C, 8, 8))
    w = rng.standard_normal((C, 1, 3, 3))
    z = oracle.conv2d(x, w, None, (2, 2), (1, 1, 1, 1), (1, 1), C)
    for c in range(C):
        zc = oracle.conv2d(x[:, c:c + 1], w[c:c + 1], None, (2, 2), (1, 1, 1, 1), (1, 1), 1)
        assert np.array_equal(z[:, c:c + 1], zc)


def test_stride_is_subsampled_unit_stride():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((1, 4, 11, 10))
    w = rng.standard_normal((3, 4, 3, 3))
    z1 = oracle.conv2d(x, w, None, (1, 1), (1, 1, 1, 1))
    z2 = oracle.conv2d(x, w, None, (2, 2), (1, 1, 1, 1))
    assert np.array_equal(z2, z1[:, :, ::2, ::2])


def test_dilation_is_zero_dilated_kernel():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((1, 3, 12, 12))
    w = rng.standard_normal((4, 3, 3, 3))
    wd = np.zeros((4, 3, 5, 5))
    wd[:, :, ::2, ::2] = w
    assert np.allclose(oracle.conv2d(x, w, None, (1, 1), (2, 2, 2, 2), (2, 2)),
                       oracle.conv2d(x, wd, None, (1, 1), (2, 2, 2, 2), (1, 1)),
                       rtol=0, atol=1e-12)


# ------------------------------------------------------------ BN and auto_pad

def test_bn_fold_invariant():
    """conv(s*W) + (s*bias + t) == BN(conv(W) + bias), s = gamma/sqrt(var+eps),
    t = beta - mean*s: the fold of the "tensorforge" page (W' = scale*W,
    bias = shift), checked in unrounded float64."""
    rng = np.random.default_rng(8)
    K, C = 8, 5
    x = rng.standard_normal((2, C, 7, 7))
    w = rng.standard_normal((K, C, 3, 3))
    bias = rng.standard_normal(K)
    gamma, beta = rng.uniform(0.5, 1.5, K), rng.normal(0, 0.1, K)
    mean, var = rng.normal(0, 0.1, K), rng.uniform(0.5, 1.5, K)
    eps = 1e-5
    s = gamma / np.sqrt(var + eps)
    t = beta - mean * s
    lhs = oracle.conv2d(x, w * s[:, None, None, None], s * bias + t, (1, 1), (1, 1, 1, 1))
    rhs = oracle.batchnorm(oracle.conv2d(x, w, bias, (1, 1), (1, 1, 1, 1)), gamma, beta, mean,
                           var, eps)
    assert np.abs(lhs - rhs).max() <= 1e-12 * np.abs(rhs).max()
    # identity BN: gamma=1, beta=0, mean=0, var=1-eps
    z = oracle.conv2d(x, w, bias, (1, 1), (1, 1, 1, 1))
    ident = oracle.batchnorm(z, np.ones(K), np.zeros(K), np.zeros(K), np.full(K, 1 - eps), eps)
    assert np.abs(ident - z).max() <= 1e-15 * np.abs(z).max()
    # point form agrees with the tensor form
    chan = np.broadcast_to(np.arange(K).reshape(1, K, 1, 1), z.shape).reshape(-1)
    assert np.array_equal(oracle.batchnorm(z.reshape(-1), gamma, beta, mean, var, eps, chan),
                          oracle.batchnorm(z, gamma, beta, mean, var, eps).reshape(-1))


def test_bn_hand_value():
    # (z - mean)/sqrt(var + eps)*gamma + beta with var + eps = 4: (5 - 1)/2*3 + 0.5 = 6.5
    out = oracle.batchnorm(np.full((1, 1, 1, 1), 5.0), [3.0], [0.5], [1.0], [4.0 - 1e-5], 1e-5)
    assert abs(out.item() - 6.5) < 1e-12


@pytest.mark.parametrize("n_in,k,s,d,upper,lower", [
    (5, 3, 2, 1, (1, 1), (1, 1)),
    (4, 3, 2, 1, (0, 1), (1, 0)),
    (7, 1, 2, 1, (0, 0), (0, 0)),
    (6, 3, 1, 2, (2, 2), (2, 2)),
    (224, 7, 2, 1, (2, 3), (3, 2)),
])
def test_auto_pad(n_in, k, s, d, upper, lower):
    pu = oracle.resolve_pads(n_in, n_in, k, k, (s, s), (d, d), auto_pad="SAME_UPPER")
    pl = oracle.resolve_pads(n_in, n_in, k, k, (s, s), (d, d), auto_pad="SAME_LOWER")
    assert (pu[0], pu[2]) == upper and (pl[0], pl[2]) == lower
    for p in (pu, pl):
        assert oracle.out_hw(n_in, n_in, k, k, (s, s), p, (d, d)) == (-(-n_in // s),) * 2
    assert oracle.resolve_pads(n_in, n_in, k, k, (s, s), (d, d), (1, 2, 3, 4), "VALID") == (0,) * 4
    assert oracle.resolve_pads(n_in, n_in, k, k, (s, s), (d, d), (1, 2, 3, 4)) == (1, 2, 3, 4)


def test_same_upper_matches_torch_same():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((1, 2, 6, 9))
    w = rng.standard_normal((3, 2, 4, 2))
    p = oracle.resolve_pads(6, 9, 4, 2, auto_pad="SAME_UPPER")
    ref = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(w),
                                     padding="same").numpy()
    assert np.allclose(oracle.conv2d(x, w, None, (1, 1), p), ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------------- requant

def test_requant_hand_cases():
    K = 1
    b = np.zeros(K, np.int32)
    m = np.full(K, 1 << 30, np.int32)       # M / 2^31 = 0.5
    sh = np.full(K, 31, np.int32)
    v = np.array([3, -3, 1, -1, 2, -2, 0])
    ch = np.zeros_like(v)
    # 1.5 -> 2, -1.5 -> -1, 0.5 -> 1, -0.5 -> 0 (ties toward +inf)
    assert oracle.requant_s8(v, ch, b, m, sh).tolist() == [2, -1, 1, 0, 1, -1, 0]
    # saturation at the int8 range
    assert oracle.requant_s8(np.array([400, -400, 255, -257]), np.zeros(4, np.int64), b, m,
                             sh).tolist() == [127, -128, 127, -128]
    # ReLU clamps at the output zero point; bias is added before scaling
    zp = 5
    assert oracle.requant_s8(np.array([-20, 0, 20]), np.zeros(3, np.int64), b, m, sh, zp,
                             relu=True).tolist() == [5, 5, 15]
    assert oracle.requant_s8(np.array([-20, 0, 20]), np.zeros(3, np.int64), b, m, sh, zp,
                             relu=False).tolist() == [-5, 5, 15]
    assert oracle.requant_s8(np.array([1]), np.zeros(1, np.int64), np.array([9], np.int32), m,
                             sh).tolist() == [5]
    # per-channel parameters select by channel
    acc = np.arange(2 * 3 * 2 * 2, dtype=np.int64).reshape(2, 3, 2, 2) * 10
    mm = np.array([1 << 30, 1 << 29, 3 << 28], np.int32)
    ss = np.full(3, 31, np.int32)
    out = oracle.requant_s8(acc, None, np.zeros(3, np.int32), mm, ss)
    for k in range(3):
        ref = oracle.requant_s8(acc[:, k], np.zeros_like(acc[:, k]), np.zeros(1, np.int32),
                                mm[k:k + 1], ss[k:k + 1])
        assert np.array_equal(out[:, k], ref)


def test_requant_matches_exact_rational_rounding():
    """Python integers: round-half-up of v*M/2^sh is floor((2vM + 2^sh) / 2^(sh+1))."""
    rng = np.random.default_rng(10)
    K = 64
    mult = rng.integers(1 << 30, (1 << 31) - 1, K).astype(np.int32)
    shift = rng.integers(20, 50, K).astype(np.int32)
    bias = rng.integers(-(1 << 16), 1 << 16, K).astype(np.int32)
    acc = rng.integers(-(1 << 27), 1 << 27, 5000)
    chan = rng.integers(0, K, 5000)
    for zp, relu in ((0, True), (-7, False), (12, True)):
        out = oracle.requant_s8(acc, chan, bias, mult, shift, zp, relu)
        for a, k, o in zip(acc.tolist(), chan.tolist(), out.tolist()):
            v = a + int(bias[k])
            M, s = int(mult[k]), int(shift[k])
            q = (2 * v * M + (1 << s)) // (1 << (s + 1)) + zp
            lo = max(zp, -128) if relu else -128
            assert o == min(max(q, lo), 127)
    with pytest.raises(ValueError):
        oracle.requant_s8(np.array([1]), np.zeros(1, np.int64), np.zeros(1, np.int32),
                          np.zeros(1, np.int32), np.full(1, 31, np.int32))


# ----------------------------------------------------------- tolerance sanity

def test_fp32_accumulation_meets_tolerance():
    """A plain float32 running sum over the largest reduction of the workloads
    (C=512, 3x3: 4608 terms) stays inside |d| <= 1e-3 + 1e-3|ref| of the float64
    result, so the tolerance is attainable by fp32 accumulation."""
    g = torch.Generator().manual_seed(11)
    C, K = 512, 8
    x = torch.randn(1, C, 7, 7, generator=g).to(torch.bfloat16).double().numpy()
    w = (torch.randn(K, C, 3, 3, generator=g) * math.sqrt(2.0 / (C * 9))
         ).to(torch.bfloat16).double().numpy()
    ref = oracle.conv2d(x, w, None, (1, 1), (1, 1, 1, 1))
    f32 = oracle.conv2d_f32acc(x, w, None, (1, 1), (1, 1, 1, 1))
    ok, worst, _ = oracle.tolerance_ok(f32, ref)
    assert ok and worst < 0.1, worst


def test_tolerance_helper_flags_a_planted_error():
    ref = np.linspace(-3, 3, 101)
    y = ref.copy()
    assert oracle.tolerance_ok(y, ref)[0]
    y[17] += 2e-3 + 1e-3 * abs(ref[17])
    ok, worst, idx = oracle.tolerance_ok(y, ref)
    assert not ok and idx == 17 and worst > 1.0


# ----------------------------------------------------------- residual stage

def test_residual_with_identity_kernel_is_shifted_input():
    """Closed form: an identity 3x3 kernel (pad 1) returns x, so with a residual r and ReLU the
    whole pipeline must give max(x + r, 0) exactly."""
    rng = np.random.default_rng(40)
    C = 5
    x = rng.standard_normal((2, C, 7, 6))
    r = rng.standard_normal((2, C, 7, 6))
    w = np.zeros((C, C, 3, 3))
    for c in range(C):
        w[c, c, 1, 1] = 1.0
    y = oracle.conv_bn_act(x, w, None, None, oracle.ACT_RELU, pads=(1, 1, 1, 1), residual=r)
    assert np.array_equal(y, np.maximum(x + r, 0.0))


def test_residual_joins_after_bn_and_before_the_clamp():
    """A residual equal to minus the BN output leaves a zero pre-activation: every activation
    then gives 0 (Clip gives its lower bound), whatever the conv and BN values."""
    rng = np.random.default_rng(41)
    x = rng.standard_normal((1, 4, 6, 6))
    w = rng.standard_normal((3, 4, 3, 3))
    bn = (rng.uniform(0.5, 1.5, 3), rng.normal(0, 0.1, 3), rng.normal(0, 0.1, 3), rng.uniform(0.5, 1.5, 3))
    u = oracle.batchnorm(oracle.conv2d(x, w, None, (1, 1), (1, 1, 1, 1)), *bn)
    for act in (oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_RELU6):
        y = oracle.conv_bn_act(x, w, None, bn, act, pads=(1, 1, 1, 1), residual=-u)
        assert np.max(np.abs(y)) < 1e-12
    y = oracle.conv_bn_act(x, w, None, bn, oracle.ACT_CLIP, 0.25, 2.0, pads=(1, 1, 1, 1), residual=-u)
    assert np.allclose(y, 0.25, atol=1e-12)


def test_residual_pipeline_matches_torch_on_tiny_cases():
    """Library route: torch conv2d (float64) + batch_norm (inference) + residual + ReLU6."""
    rng = np.random.default_rng(42)
    for trial in range(6):
        N, C, K, H, W = 2, int(rng.integers(1, 6)), int(rng.integers(1, 6)), 6, 5
        x = rng.standard_normal((N, C, H, W))
        w = rng.standard_normal((K, C, 3, 3))
        b = rng.standard_normal(K)
        bn = (rng.uniform(0.5, 1.5, K), rng.normal(0, 0.1, K), rng.normal(0, 0.1, K), rng.uniform(0.5, 1.5, K))
        stride = (1 + trial % 2, 1)
        z = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b), stride, 1)
        z = torch.nn.functional.batch_norm(z, torch.from_numpy(bn[2]), torch.from_numpy(bn[3]),
                                           torch.from_numpy(bn[0]), torch.from_numpy(bn[1]), False, 0.0, 1e-5)
        r = rng.standard_normal(tuple(z.shape))
        ref = torch.clamp(z + torch.from_numpy(r), 0.0, 6.0).numpy()
        y = oracle.conv_bn_act(x, w, b, bn, oracle.ACT_RELU6, strides=stride, pads=(1, 1, 1, 1), residual=r)
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
        pts = np.array([[n, k, i, j] for n in range(N) for k in range(K) for i in range(z.shape[2])
                        for j in range(z.shape[3])][::7], dtype=np.int64)
        yp = oracle.conv_bn_act_points(x, w, b, bn, oracle.ACT_RELU6, stride, (1, 1, 1, 1), (1, 1), 1, pts,
                                       residual=r)
        assert np.allclose(yp, ref[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------- QLinearConv (zero points)

def _windows(xp, R, S, sh, sw, Ho, Wo):
    """im2col of an already padded NCHW input: [N][C][R][S][Ho][Wo]."""
    N, C = xp.shape[:2]
    out = np.empty((N, C, R, S, Ho, Wo), dtype=xp.dtype)
    for r in range(R):
        for s in range(S):
            out[:, :, r, s] = xp[:, :, r: r + sh * (Ho - 1) + 1: sh, s: s + sw * (Wo - 1) + 1: sw]
    return out


@pytest.mark.parametrize("case", range(8))
def test_qlinear_sums_match_the_zero_point_identity(case):
    """The page's expansion sum (a - az)(b - bz) = sum ab - az sum b - bz sum a + n az bz, taken over
    every tap of the zero-point-padded input (n = C*R*S), against the oracle's direct sums."""
    rng = np.random.default_rng(50 + case)
    N, C, K, H, W = 2, int(rng.integers(1, 5)), int(rng.integers(1, 5)), 6, 7
    R = S = 3
    st = (1 + case % 2, 1 + (case // 2) % 2)
    pads = (1, 1, 1, 1) if case % 3 else (0, 1, 2, 0)
    xu = case % 2 == 0                                 # uint8 or int8 activations
    x = (rng.integers(0, 256, (N, C, H, W)).astype(np.uint8) if xu
         else rng.integers(-128, 128, (N, C, H, W)).astype(np.int8))
    w = rng.integers(-127, 128, (K, C, R, S)).astype(np.int8)
    zx = int(rng.integers(0, 256)) if xu else int(rng.integers(-128, 128))
    zw = rng.integers(-20, 21, K)
    bias = rng.integers(-5000, 5000, K).astype(np.int32)
    acc = oracle.qlinear_conv_acc(x, zx, w, zw, bias, st, pads)
    pt, pl, pb, pr = pads
    xp = np.full((N, C, H + pt + pb, W + pl + pr), zx, dtype=np.int64)
    xp[:, :, pt:pt + H, pl:pl + W] = x
    Ho, Wo = acc.shape[2:]
    cols = _windows(xp, R, S, st[0], st[1], Ho, Wo).reshape(N, C * R * S, Ho, Wo)
    wf = w.reshape(K, -1).astype(np.int64)
    n = C * R * S
    sum_ab = np.einsum("kj,njhw->nkhw", wf, cols)
    sum_a = cols.sum(axis=1)[:, None]                 # over the input taps, per output position
    sum_b = wf.sum(axis=1)[None, :, None, None]
    zwk = zw.reshape(1, K, 1, 1)
    ident = sum_ab - zx * sum_b - zwk * sum_a + n * zx * zwk + bias.reshape(1, K, 1, 1)
    assert np.array_equal(acc, ident)


def test_qlinear_without_zero_points_is_the_int8_sum():
    rng = np.random.default_rng(60)
    x = rng.integers(-128, 128, (2, 5, 7, 6)).astype(np.int8)
    w = rng.integers(-127, 128, (4, 5, 3, 3)).astype(np.int8)
    acc = oracle.qlinear_conv_acc(x, 0, w, 0, None, (2, 1), (1, 0, 1, 2))
    assert np.array_equal(acc, oracle.conv2d_s8(x, w, (2, 1), (1, 0, 1, 2)))


def test_qlinear_input_at_its_zero_point_leaves_the_bias():
    """x == x_zp everywhere: every corrected product is 0, so y = saturate(rint(B*m) + y_zp)."""
    rng = np.random.default_rng(61)
    zx = 117
    x = np.full((1, 3, 5, 5), zx, dtype=np.uint8)
    w = rng.integers(-127, 128, (6, 3, 3, 3)).astype(np.int8)
    bias = np.array([-400, -3, 0, 7, 250, 90000], dtype=np.int32)
    acc = oracle.qlinear_conv_acc(x, zx, w, rng.integers(-3, 4, 6), bias, (1, 1), (1, 1, 1, 1))
    assert np.array_equal(acc, np.broadcast_to(bias.reshape(1, 6, 1, 1), acc.shape))
    y = oracle.qlinear_requant(acc, 0.25, 0.5, 1.0, 100)          # m = 1/8, y_zp = 100
    # -400/8 = -50 -> 50; -3/8 -> -0 -> 100; 0 -> 100; 7/8 -> 1 -> 101; 250/8 = 31.25 -> 131;
    # 90000/8 = 11250 -> saturates at 255
    assert y[0, :, 0, 0].tolist() == [50, 100, 100, 101, 131, 255]


def test_qlinear_requant_rounds_half_to_even_and_saturates():
    acc = np.array([1, 3, 5, -1, -3, 7, 1000, -1000], dtype=np.int64).reshape(1, 8, 1, 1)
    y = oracle.qlinear_requant(acc, 0.5, 1.0, 1.0, 0, np.int8)     # m = 0.5
    assert y.reshape(-1).tolist() == [0, 2, 2, 0, -2, 4, 127, -128]
    y = oracle.qlinear_requant(acc, 0.5, 1.0, 1.0, 3, np.uint8)
    assert y.reshape(-1).tolist() == [3, 5, 5, 3, 1, 7, 255, 0]
    # per-channel weight scales: channel k scales by k + 1
    acc = np.full((1, 3, 1, 1), 10, dtype=np.int64)
    y = oracle.qlinear_requant(acc, 0.5, np.array([1.0, 2.0, 3.0], np.float32), 2.0, 0, np.int8)
    assert y.reshape(-1).tolist() == [2, 5, 8]                      # 2.5 -> 2, 5, 7.5 -> 8


def test_qlinear_refuses_zero_points_outside_their_types():
    """ONNX QLinearConv: x_zero_point has x's type, w_zero_point w's type, y's type is
    y_zero_point's type; a zero point outside that type's range is refused, not wrapped."""
    x = np.zeros((1, 2, 4, 4), np.int8)
    w = np.zeros((3, 2, 3, 3), np.int8)
    with pytest.raises(ValueError, match="x_zero_point"):
        oracle.qlinear_conv_acc(x, 200, w, 0)
    with pytest.raises(ValueError, match="w_zero_point"):
        oracle.qlinear_conv_acc(x, 0, w, np.array([0, 130, 0]))
    with pytest.raises(ValueError, match="w_zero_point"):
        oracle.qlinear_conv_acc(x, 0, w.astype(np.uint8), -1)
    acc = np.zeros((1, 3, 2, 2), np.int64)
    with pytest.raises(ValueError, match="y_zero_point"):
        oracle.qlinear_requant(acc, 1.0, 1.0, 1.0, -3, np.uint8)
    with pytest.raises(ValueError, match="y_zero_point"):
        oracle.qlinear_requant(acc, 1.0, 1.0, 1.0, 128, np.int8)
    with pytest.raises(ValueError, match="uint8 or int8"):
        oracle.qlinear_requant(acc, 1.0, 1.0, 1.0, 0, np.int16)


def test_qlinear_requant_takes_float32_steps():
    """The multiplier is one float32 rounding of the float64 quotient, and the product is a
    float32 product: sums above 2^24 first round to float32 (ties to even), so neighbouring
    integers can land on the same code; a float64 product would separate them."""
    m = oracle.qlinear_multiplier(0.1, np.array([0.3], np.float32), 0.7, 1)
    ref = np.float32(np.float64(np.float32(0.1)) * np.float64(np.float32(0.3)) / np.float64(np.float32(0.7)))
    assert m.dtype == np.float32 and m[0] == ref
    # acc = 7*2^22 - 1 is a float32 tie that rounds to 7*2^22 (even), so with m = 2^-23 the float32
    # product is exactly 3.5 -> 4 (half to even); the float64 product 3.5 - 2^-23 would give 3
    acc = np.array([7 * (1 << 22) - 1, 7 * (1 << 22) + 1], dtype=np.int64).reshape(1, 2, 1, 1)
    y = oracle.qlinear_requant(acc, 1.0, np.array([2.0 ** -23, 2.0 ** -23], np.float32), 1.0, 0, np.int8)
    assert y.reshape(-1).tolist() == [4, 4]
    y = oracle.qlinear_requant(acc, 1.0, np.array([2.0 ** -2, 2.0 ** -2], np.float32), 1.0, 0, np.int8)
    assert y.reshape(-1).tolist() == [127, 127]         # saturation
    # 5 * 0.1f: float32(0.1) * 5 = 0.50000000745 in float64 but exactly 0.5 in float32 -> 0 (even)
    acc = np.array([5], dtype=np.int64).reshape(1, 1, 1, 1)
    y = oracle.qlinear_requant(acc, 0.1, np.array([1.0], np.float32), 1.0, 0, np.int8)
    assert y.reshape(-1).tolist() == [0]


def test_qlinear_relu_keeps_the_codes_of_non_negative_real_values():
    """A fused Relu in the quantized domain: dequantized, the result is max(dequantized y, 0)."""
    rng = np.random.default_rng(62)
    acc = rng.integers(-40000, 40000, (2, 4, 3, 3)).astype(np.int64)
    for y_dtype, zp in ((np.uint8, 120), (np.int8, -7)):
        y = oracle.qlinear_requant(acc, 0.02, np.array([0.004, 0.003, 0.005, 0.002], np.float32), 0.3, zp, y_dtype)
        yr = oracle.qlinear_requant(acc, 0.02, np.array([0.004, 0.003, 0.005, 0.002], np.float32), 0.3, zp, y_dtype,
                                    relu=True)
        real = (y.astype(np.int64) - zp) * 0.3
        real_r = (yr.astype(np.int64) - zp) * 0.3
        assert np.array_equal(real_r, np.maximum(real, 0.0))
        assert (yr < zp).sum() == 0 and (y < zp).any()


# ----------------------------------------------------------- pre-activation prologue

def test_round_bf16_matches_the_library_conversion_and_ties_go_to_even():
    """Against torch's float32 -> bfloat16 conversion (a library routine, round to nearest even),
    on random values over many binades and on exact ties."""
    rng = np.random.default_rng(70)
    a = (rng.standard_normal(200000) * np.exp2(rng.integers(-30, 30, 200000))).astype(np.float32)
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(a), ref)
    # ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> 1 (even); 1 + 3*2^-8 -> 1 + 2^-6 (even)
    t = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2 + 2.0 ** -7], np.float32)
    assert oracle.round_bf16(t).tolist() == [1.0, 1 + 2.0 ** -6, -1.0, 2.0]


def test_preactivation_closed_forms():
    rng = np.random.default_rng(71)
    x = oracle.round_bf16(rng.standard_normal((2, 5, 4, 3)))
    one, zero = np.ones(5), np.zeros(5)
    # identity affine, no activation: x itself (already bf16)
    assert np.array_equal(oracle.preactivation(x, one, zero, oracle.ACT_NONE), x)
    # ReLU zeroes exactly the negative inputs
    u = oracle.preactivation(x, one, zero, oracle.ACT_RELU)
    assert np.array_equal(u, np.maximum(x, 0.0))
    # a per-channel affine: channel c scaled by 2^c (exact in bf16), shifted by 0
    s = np.exp2(np.arange(5.0))
    u = oracle.preactivation(x, s, zero, oracle.ACT_NONE)
    assert np.array_equal(u, x * s.reshape(1, 5, 1, 1))


def test_preactivation_pads_after_the_activation():
    """The conv's zero padding is applied to u: with shift = 1 and ReLU every real input maps to
    max(x + 1, 0) but padded taps still contribute 0.  Checked against torch on the padded u."""
    rng = np.random.default_rng(72)
    x = oracle.round_bf16(rng.standard_normal((1, 3, 5, 5)))
    w = rng.standard_normal((4, 3, 3, 3))
    pre = (np.ones(3), np.ones(3), oracle.ACT_RELU)
    y = oracle.conv_bn_act(x, w, pads=(1, 1, 1, 1), pre=pre)
    u = oracle.round_bf16(np.maximum(x + 1.0, 0.0))
    ref = torch.nn.functional.conv2d(torch.from_numpy(u), torch.from_numpy(w), padding=1).numpy()
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # padding x with zeros first and activating after would add relu(0 + 1) = 1 on the border
    xp = np.pad(x, ((0, 0), (0, 0), (1, 1), (1, 1)))
    wrong = torch.nn.functional.conv2d(torch.from_numpy(oracle.round_bf16(np.maximum(xp + 1.0, 0.0))),
                                       torch.from_numpy(w)).numpy()
    assert not np.allclose(y[..., 0, 0], wrong[..., 0, 0])


# ----------------------------------------------------------- MobileNetV2 inverted residual

@pytest.mark.parametrize("cin,ch,cout,stride,res,expand", [(8, 48, 8, 1, True, True), (8, 48, 12, 2, False, True),
                                                           (16, 16, 8, 1, False, False)])
def test_inverted_residual_matches_torch(cin, ch, cout, stride, res, expand):
    """The block against torch's conv2d / batch_norm / hardtanh(0, 6) on CPU in float64."""
    rng = np.random.default_rng(80 + cin + ch + stride)
    x = rng.standard_normal((2, cin, 9, 9))
    we = rng.standard_normal((ch, cin, 1, 1)) if expand else None
    wd = rng.standard_normal((ch, 1, 3, 3))
    wp = rng.standard_normal((cout, ch, 1, 1))

    def bn(k):
        return (rng.uniform(0.5, 1.5, k), rng.normal(0, 0.1, k), rng.normal(0, 0.1, k), rng.uniform(0.5, 1.5, k))

    be, bd, bp = bn(ch), bn(ch), bn(cout)
    y = oracle.inverted_residual(x, we, be, wd, bd, wp, bp, stride, res)
    F = torch.nn.functional
    T = torch.from_numpy

    def tbn(z, p):
        return F.batch_norm(z, T(p[2]), T(p[3]), T(p[0]), T(p[1]), False, 0.0, 1e-5)

    h = T(x)
    if expand:
        h = F.hardtanh(tbn(F.conv2d(h, T(we)), be), 0.0, 6.0)
    h = F.hardtanh(tbn(F.conv2d(h, T(wd), stride=stride, padding=1, groups=ch), bd), 0.0, 6.0)
    ref = tbn(F.conv2d(h, T(wp)), bp)
    if res:
        ref = ref + T(x)
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
