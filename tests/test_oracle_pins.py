"""Pins of the fp64 oracle against things other than itself.

Every check below ties the oracle to a fact fixed by the mathematics or by a
library routine: closed forms of special cases (hand-derived values in
tests/golden/closed_forms.json), torch's SDPA / softmax in fp64, a
statistical property of Gaussian noise logits, exact-algebra invariants
(streamed == definition, split-merge == single pass), and a brute-force
re-evaluation on tiny inputs.  Source: "ATMA: Length-Invariant Language
Modeling via Polar Attention and Gated-Delta Compression Memory", §2.1
(three channels), §2.2 (fused kernel: streaming accumulators with squared
correction factors), §3 (training length 2K).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import DEFAULT_CONSTS, oracle_decode, oracle_fwd, oracle_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")
LN_T0 = math.log(2048.0)


def golden(name):
    with open(GOLDEN) as f:
        cases = {c["name"]: c for c in json.load(f)["cases"]}
    return cases[name]


def rnd(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


def unit(x, axis=-1):
    return x / np.linalg.norm(x, axis=axis, keepdims=True)


# ----------------------------------------------------------- n_eff (§2.1.2)

def test_neff_uniform_logits_equals_n():
    """q = 0 gives equal logits, p_j = 1/n, inverse Simpson index = n."""
    T, d = 300, 8
    q = np.zeros((1, 1, T, d))
    k, v = rnd((1, 1, T, d), 1), rnd((1, 1, T, d), 2)
    out, neff, conf = oracle_fwd(q, k, v, np.zeros_like(q), np.zeros((1, d)))
    n = np.arange(1, T + 1)
    np.testing.assert_allclose(neff[0, 0], n, rtol=1e-12)
    g = golden("uniform_row_neff")
    _, ne, _ = oracle_rows(np.zeros((g["n"], 4)), rnd((g["n"], 4), 3),
                           rnd((g["n"], 4), 4), np.zeros((g["n"], 4)),
                           np.zeros(4), [g["n"] - 1])
    assert ne[0] == pytest.approx(eval(g["expr"]), rel=1e-12)


def test_neff_one_hot_is_one():
    """One key aligned at logit ~50 above the rest: n_eff -> 1."""
    T, d = 64, 16
    q, k, v = rnd((T, d), 5), rnd((T, d), 6), rnd((T, d), 7)
    i, j = 50, 17
    k[j] = 50.0 * q[i] / np.linalg.norm(q[i])
    k[j] *= 4.0  # logit ~ 4*50*|q|/sqrt(d) >> noise
    out, ne, conf = oracle_rows(q, k, v, np.zeros((T, d)), np.zeros(d), [i])
    assert abs(ne[0] - 1.0) < 1e-6
    # direction collapses onto v_j (one-hot closed form)
    np.testing.assert_allclose(out[0], unit(v[j]), atol=1e-9)


def test_neff_bounds_random():
    """1 <= n_eff <= n for every row of random inputs (several scales)."""
    for seed, scale in ((8, 1.0), (9, 3.0), (10, 0.1)):
        T, d = 200, 16
        q = rnd((1, 2, T, d), seed, scale)
        k, v = rnd((1, 2, T, d), seed + 100), rnd((1, 2, T, d), seed + 200)
        _, neff, _ = oracle_fwd(q, k, v, np.zeros_like(q), np.zeros((2, d)))
        n = np.arange(1, T + 1)
        assert np.all(neff >= 1 - 1e-12)
        assert np.all(neff <= n + 1e-9)


def test_neff_matches_torch_softmax():
    """n_eff = 1 / sum(softmax^2) with torch's fp64 softmax; for n <= 2048
    the temperature is neutral, so the logits are plain SDPA logits."""
    T, d = 256, 64
    q, k, v = rnd((1, 2, T, d), 11), rnd((1, 2, T, d), 12), rnd((1, 2, T, d), 13)
    _, neff, _ = oracle_fwd(q, k, v, np.zeros_like(q), np.zeros((2, d)))
    qt, kt = torch.from_numpy(q), torch.from_numpy(k)
    logits = qt @ kt.transpose(-1, -2) / math.sqrt(d)
    mask = torch.ones(T, T, dtype=torch.bool).triu(1)
    p = torch.softmax(logits.masked_fill(mask, float("-inf")), dim=-1)
    ref = 1.0 / (p * p).sum(-1)
    np.testing.assert_allclose(neff, ref.numpy(), rtol=1e-11)


# ------------------------------------------------------ direction (§2.1.1)

def test_direction_matches_sdpa_within_training_length():
    """For n <= 2048 the direction is normalize(causal SDPA) (torch, fp64)."""
    T, d = 256, 64
    q, k, v = rnd((1, 2, T, d), 14), rnd((1, 2, T, d), 15), rnd((1, 2, T, d), 16)
    out, _, _ = oracle_fwd(q, k, v, np.zeros_like(q), np.zeros((2, d)))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        is_causal=True).numpy()
    np.testing.assert_allclose(out, unit(ref), atol=1e-11)
    np.testing.assert_allclose(np.linalg.norm(out, axis=-1), 1.0, atol=1e-12)


def test_direction_uniform_is_mean_of_values():
    """q = 0: u_i = normalize(mean of v_0..v_i)."""
    T, d = 50, 8
    v = rnd((T, d), 17)
    out, _, _ = oracle_rows(np.zeros((T, d)), rnd((T, d), 18), v,
                            np.zeros((T, d)), np.zeros(d), list(range(T)))
    ref = unit(np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None])
    np.testing.assert_allclose(out, ref, atol=1e-12)


def test_direction_zero_values_guarded():
    """All-zero values: a = 0, the eps guard gives u = 0 (no NaN)."""
    T, d = 20, 8
    w = rnd((1, d), 19)
    mem = rnd((1, 1, T, d), 20)
    out, neff, _ = oracle_fwd(rnd((1, 1, T, d), 21), rnd((1, 1, T, d), 22),
                              np.zeros((1, 1, T, d)), mem, w)
    assert np.all(np.isfinite(out))
    # out - mem is parallel to w (u vanished)
    r = out[0, 0] - mem[0, 0]
    cosang = np.abs(r @ w[0]) / (np.linalg.norm(r, axis=1) * np.linalg.norm(w[0]) + 1e-300)
    assert np.all((np.linalg.norm(r, axis=1) < 1e-15) | (cosang > 1 - 1e-12))


@pytest.mark.parametrize("c,expect", [(1e-7, 0.1), (1e-5, 1.0), (1e-6 / 3, 1.0 / 3)])
def test_direction_guard_closed_form_constant_values(c, expect):
    """q = 0 and every value v_j = c e_0: a = c e_0 at every row whatever n,
    so the unit-sphere projection with guard eps = 1e-6 gives
    u = c / max(c, eps) e_0 -- 0.1 e_0 for c = 1e-7, e_0 for c = 1e-5.  The
    normaliser l = n grows along the rows, so a guard taken on the
    unnormalised accumulator |acc| = n c instead of |a| = c gives n-dependent
    answers and fails here."""
    T, d = 50, 8
    v = np.zeros((T, d))
    v[:, 0] = c
    out, _, _ = oracle_rows(np.zeros((T, d)), rnd((T, d), 23), v, np.zeros((T, d)),
                            np.zeros(d), list(range(T)))
    ref = np.zeros((T, d))
    ref[:, 0] = expect
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-15)
    # the same through the decode (definition and split-merge forms)
    for ns in (0, 3):
        od, _, _ = oracle_decode(np.zeros((1, 1, d)), rnd((1, 1, T, d), 24), v[None, None],
                                 np.zeros((1, 1, d)), np.zeros((1, d)), nsplit=ns, tile=7)
        np.testing.assert_allclose(od[0, 0], ref[0], rtol=1e-12, atol=1e-15)


def test_direction_guard_straddles_eps_along_rows():
    """q = 0 and values of scale 1e-6: a_i is the running mean of v_0..v_i,
    whose norm falls through eps = 1e-6 as i grows, so rows on both sides
    of the guard appear: u_i = a_i / |a_i| above it and a_i / eps below."""
    T, d = 400, 16
    v = rnd((T, d), 25, scale=1e-6)
    out, _, _ = oracle_rows(np.zeros((T, d)), rnd((T, d), 26), v, np.zeros((T, d)),
                            np.zeros(d), list(range(T)))
    a = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    an = np.linalg.norm(a, axis=1)
    assert (an > 2e-6).any() and (an < 0.5e-6).any()  # both sides present
    ref = a / np.maximum(an, 1e-6)[:, None]
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-15)
    # a guard of another size moves the rows below it
    out3, _, _ = oracle_rows(np.zeros((T, d)), rnd((T, d), 26), v, np.zeros((T, d)),
                             np.zeros(d), list(range(T)), consts={"eps": 1e-5})
    np.testing.assert_allclose(out3, a / np.maximum(an, 1e-5)[:, None], rtol=1e-10, atol=1e-15)


# ---------------------------------------------------- temperature (§2.1.1)

@pytest.mark.parametrize("name", ["temperature_at_4096", "temperature_at_8192",
                                  "temperature_below_T0"])
def test_temperature_recovered_from_two_key_row(name):
    """A row whose mass sits on two keys with raw logit gap 1 and orthogonal
    values: u_0/u_1 = p_0/p_1 = exp(tau * 1), so tau = ln(u_0/u_1)."""
    g = golden(name)
    n, d = g["n"], 4
    T = n + 777  # later rows exist: the temperature must follow the row's n
    q = np.zeros((T, d))
    q[n - 1] = [2.0, 0.0, 0.0, 0.0]           # |q| / sqrt(d) = 1
    k = np.tile([-50.0, 0.0, 0.0, 0.0], (T, 1))  # far below: weight ~e^-50
    k[0] = [1.0, 0.0, 0.0, 0.0]                 # raw logit 1
    k[1] = [0.0, 0.0, 0.0, 0.0]                 # raw logit 0
    v = np.tile([0.0, 0.0, 1.0, 0.0], (T, 1))
    v[0] = [1.0, 0.0, 0.0, 0.0]
    v[1] = [0.0, 1.0, 0.0, 0.0]
    out, ne, _ = oracle_rows(q, k, v, np.zeros((T, d)), np.zeros(d), [n - 1])
    tau = math.log(out[0, 0] / out[0, 1])
    assert tau == pytest.approx(eval(g["expr"]), rel=1e-9)
    # two-point participation ratio (p0 + p1)^2 / (p0^2 + p1^2)
    r = math.exp(-tau)
    assert ne[0] == pytest.approx((1 + r) ** 2 / (1 + r * r), rel=1e-6)


def test_temperature_sharpens_beyond_training_length():
    """Beyond 2K keys the same logit pattern gets a smaller n_eff."""
    d = 16
    n_small, n_big = 1500, 6000
    k = rnd((n_big, d), 23)
    q = np.zeros((n_big, d))
    q[n_small - 1] = q[n_big - 1] = rnd(d, 24)
    v = rnd((n_big, d), 25)
    # same keys for both rows up to n_small; n_big row sees more keys, so
    # compare against SDPA with the neutral scale over the same n_big keys
    _, ne, _ = oracle_rows(q, k, v, np.zeros((n_big, d)), np.zeros(d), [n_big - 1])
    logits = torch.from_numpy(k) @ torch.from_numpy(q[n_big - 1]) / math.sqrt(d)
    p = torch.softmax(logits, 0)
    assert ne[0] < float(1.0 / (p * p).sum())


# ----------------------------------------------- null floor / gate (§2.1.1)

@pytest.mark.parametrize("n,tau,key_std,sigma_k", [
    (2000, 1.0, 1.0, 1.0),
    (4096, 12 / 11, 1.0, 1.0),
    (2000, 1.0, 2.0, 2.0),
])
def test_null_floor_is_expected_noise_maximum(n, tau, key_std, sigma_k):
    """With keys iid N(0, key_std^2) the logits are noise with std
    sigma = tau*key_std*|q|/sqrt(d).  Recover b = logsumexp - logit(conf) and
    check b = sigma_emp * sqrt(2 ln n), sigma_emp the measured logit std."""
    d = 64
    ratios = []
    for r in range(6):
        q = rnd((n, d), 100 + r)
        k = rnd((n, d), 200 + r, key_std)
        v = rnd((n, d), 300 + r)
        consts = dict(DEFAULT_CONSTS, sigma_k=sigma_k)
        _, _, conf = oracle_rows(q, k, v, np.zeros((n, d)), np.zeros(d),
                                 [n - 1], consts=consts)
        s = tau * (k @ q[n - 1]) / math.sqrt(d)
        lse = float(torch.logsumexp(torch.from_numpy(s), 0))
        c = conf[0]
        b = lse - math.log(c / (1 - c))
        ratios.append(b / (s.std() * math.sqrt(2 * math.log(n))))
    assert np.mean(ratios) == pytest.approx(1.0, abs=0.03)


def test_null_floor_misspecified_key_scale():
    """Keys twice as wide as the null model assumes: the floor is half the
    measured noise maximum (sigma uses sigma_k, not the data)."""
    n, d = 2000, 64
    ratios = []
    for r in range(6):
        q, k = rnd((n, d), 400 + r), rnd((n, d), 500 + r, 2.0)
        _, _, conf = oracle_rows(q, k, rnd((n, d), 600 + r), np.zeros((n, d)),
                                 np.zeros(d), [n - 1])
        s = (k @ q[n - 1]) / math.sqrt(d)
        lse = float(torch.logsumexp(torch.from_numpy(s), 0))
        b = lse - math.log(conf[0] / (1 - conf[0]))
        ratios.append(b / (s.std() * math.sqrt(2 * math.log(n))))
    assert np.mean(ratios) == pytest.approx(0.5, abs=0.02)


def _exact_expected_max(n):
    """E[max of n iid N(0,1)] = integral of x * n phi(x) Phi(x)^(n-1) dx,
    by numerical quadrature (scipy)."""
    from scipy import integrate, special
    f = lambda x: x * n * math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi) * \
        math.exp((n - 1) * special.log_ndtr(x))  # noqa: E731
    val, _ = integrate.quad(f, -12.0, 12.0, limit=400, points=[0.0, 2.0, 3.0, 4.0])
    return val


@pytest.mark.parametrize("n", [1000, 2000])
def test_second_order_floor_matches_exact_expected_maximum(n):
    """floor_order 2 (second-order extreme-value floor): b/sigma is the
    expected maximum of n iid N(0,1) within 1.5 % (numerical integral); the
    leading order sqrt(2 ln n) is more than 8 % above it."""
    d = 16
    q = np.zeros((n, d))
    q[n - 1, 0] = 8.0                      # |q| / sqrt(d) = 2, tau = 1 (n <= 2048)
    k, v = rnd((n, d), 700), rnd((n, d), 701)
    sigma = 2.0
    s = (k @ q[n - 1]) / math.sqrt(d)
    lse = float(torch.logsumexp(torch.from_numpy(s), 0))
    exact = _exact_expected_max(n)
    ratio = {}
    for order in (1, 2):
        consts = dict(DEFAULT_CONSTS, floor_order=order)
        _, _, conf = oracle_rows(q, k, v, np.zeros((n, d)), np.zeros(d), [n - 1],
                                 consts=consts)
        b = lse - math.log(conf[0] / (1 - conf[0]))
        ratio[order] = b / sigma / exact
    assert ratio[2] == pytest.approx(1.0, abs=0.015)
    assert ratio[1] > 1.08


def test_second_order_floor_single_key_is_zero():
    d = 8
    q, k, v = rnd((3, d), 702), rnd((3, d), 703), rnd((3, d), 704)
    consts = dict(DEFAULT_CONSTS, floor_order=2)
    _, _, conf = oracle_rows(q, k, v, np.zeros((3, d)), np.zeros(d), [0], consts=consts)
    s00 = q[0] @ k[0] / math.sqrt(d)
    assert conf[0] == pytest.approx(1 / (1 + math.exp(-s00)), rel=1e-12)


def test_conf_uniform_and_row_zero_closed_forms():
    g = golden("uniform_row_conf")
    n = g["n"]
    _, _, conf = oracle_rows(np.zeros((n, 8)), rnd((n, 8), 26), rnd((n, 8), 27),
                             np.zeros((n, 8)), np.zeros(8), [n - 1, 0, 9])
    assert conf[0] == pytest.approx(eval(g["expr"]), rel=1e-12)
    assert conf[2] == pytest.approx(10 / 11, rel=1e-12)
    # row 0: b = 0 and conf = sigmoid(s_00)
    T, d = 4, 8
    q, k, v = rnd((T, d), 28), rnd((T, d), 29), rnd((T, d), 30)
    out, ne, conf = oracle_rows(q, k, v, np.zeros((T, d)), rnd(d, 31), [0])
    s00 = q[0] @ k[0] / math.sqrt(d)
    assert conf[0] == pytest.approx(1 / (1 + math.exp(-s00)), rel=1e-12)
    assert ne[0] == pytest.approx(1.0, abs=1e-15)
    # count(n_eff = 1) = 0, so out_0 = v_0/|v_0| + mem (mem = 0 here)
    np.testing.assert_allclose(out[0], unit(v[0]), atol=1e-14)


def test_needle_raises_confidence_and_lowers_neff():
    """A planted key aligned with the query lifts the gate above the same row
    without it, and concentrates the distribution (§2.1: the floor keeps
    background noise from drowning the signal)."""
    T, d = 1024, 64
    q, k, v = rnd((T, d), 32), rnd((T, d), 33), rnd((T, d), 34)
    rows = [100, 400, 700, 1023]
    k2 = k.copy()
    for idx, i in enumerate(rows):
        j = (37 * idx + 11) % (i + 1)
        k2[j] = 4.0 * q[i] / np.linalg.norm(q[i])
    _, ne0, c0 = oracle_rows(q, k, v, np.zeros((T, d)), np.zeros(d), rows)
    _, ne1, c1 = oracle_rows(q, k2, v, np.zeros((T, d)), np.zeros(d), rows)
    assert np.all(c1 > c0)
    assert np.all(ne1 < ne0)


# ------------------------------------------------------- count (§2.1.2)

def test_count_closed_form_bounded_monotone_saturating():
    """q = 0 rows, w = e_0: count = (out - u)[0] with u the closed-form mean
    direction; count(n=2048) = 2048/2049*tanh(1); bounded, monotone."""
    d = 2
    rows = [0, 1, 9, 99, 2047, 4095, 30000]
    T = rows[-1] + 1
    v = rnd((T, d), 35)
    w = np.array([1.0, 0.0])
    out, ne, conf = oracle_rows(np.zeros((T, d)), rnd((T, d), 36), v,
                                np.zeros((T, d)), w, rows)
    u = unit(np.cumsum(v, axis=0)[rows])
    count = (out - u)[:, 0]
    assert np.all(np.abs((out - u)[:, 1]) < 1e-13)
    g = golden("uniform_row_count_at_T0")
    assert count[rows.index(2047)] == pytest.approx(g["value"], rel=1e-10)
    assert count[0] == 0.0 or abs(count[0]) < 1e-15
    assert np.all(np.diff(count) > 0)
    assert np.all(count < 1.0) and np.all(count >= 0.0)


def test_count_monotone_in_neff_at_fixed_conf():
    """At a fixed gate, tanh(ln n_eff / kappa) rises with n_eff: rows of
    growing n_eff with the same conf give growing count.  Read from out with
    w = e_0 and u removed via the w = 0 run."""
    d, T = 8, 512
    q, k, v = rnd((T, d), 37, 0.5), rnd((T, d), 38), rnd((T, d), 39)
    rows = list(range(10, T, 25))
    w = np.zeros(d)
    w[0] = 1.0
    o1, ne, cf = oracle_rows(q, k, v, np.zeros((T, d)), w, rows)
    o0, _, _ = oracle_rows(q, k, v, np.zeros((T, d)), np.zeros(d), rows)
    count = (o1 - o0)[:, 0]
    g = count / cf  # remove the gate
    order = np.argsort(ne)
    assert np.all(np.diff(g[order]) >= -1e-12)
    assert np.all(g < 1.0)


# ---------------------------------------------- memory / head (§2.1.3, §2.1)

def test_memory_stream_is_additive():
    T, d = 64, 16
    q, k, v = rnd((1, 2, T, d), 40), rnd((1, 2, T, d), 41), rnd((1, 2, T, d), 42)
    w, mem = rnd((2, d), 43), rnd((1, 2, T, d), 44)
    o1, n1, c1 = oracle_fwd(q, k, v, mem, w)
    o0, n0, c0 = oracle_fwd(q, k, v, np.zeros_like(mem), w)
    np.testing.assert_allclose(o1 - o0, mem, atol=1e-14)
    np.testing.assert_array_equal(n1, n0)


def test_count_uses_own_head_weight():
    """q = 0 rows of three heads with distinct w: out - u - mem = count*w[h]."""
    H, T, d = 3, 40, 4
    q = np.zeros((1, H, T, d))
    k, v = rnd((1, H, T, d), 45), rnd((1, H, T, d), 46)
    w, mem = rnd((H, d), 47), rnd((1, H, T, d), 48)
    out, _, _ = oracle_fwd(q, k, v, mem, w)
    n = np.arange(1, T + 1)
    count = n / (n + 1) * np.tanh(np.log(n) / LN_T0)  # closed form at q = 0
    for h in range(H):
        u = unit(np.cumsum(v[0, h], axis=0))
        np.testing.assert_allclose(out[0, h] - u - mem[0, h],
                                   count[:, None] * w[h][None, :], atol=1e-13)


# -------------------------------------- streamed / split algebra (§2.2)

@pytest.mark.parametrize("tile", [1, 3, 7, 16, 64])
def test_streamed_equals_definition(tile):
    T, d = 64, 8
    q, k, v = rnd((1, 2, T, d), 49, 2.0), rnd((1, 2, T, d), 50), rnd((1, 2, T, d), 51)
    w, mem = rnd((2, d), 52), rnd((1, 2, T, d), 53)
    a = oracle_fwd(q, k, v, mem, w, mode="definition")
    b = oracle_fwd(q, k, v, mem, w, mode="streamed", tile=tile)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)


def test_streamed_equals_definition_beyond_training_length():
    T, d = 2300, 4
    q, k, v = rnd((T, d), 54, 2.0), rnd((T, d), 55), rnd((T, d), 56)
    rows = [0, 2046, 2047, 2048, 2299]
    a = oracle_rows(q, k, v, np.zeros((T, d)), rnd(d, 57), rows)
    b = oracle_rows(q, k, v, np.zeros((T, d)), rnd(d, 57), rows, mode="streamed",
                    tile=128)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("nsplit,tile", [(1, 64), (2, 5), (7, 16), (16, 1), (40, 3)])
def test_split_merge_equals_single_pass(nsplit, tile):
    B, H, Tkv, d = 2, 2, 33, 8
    q = rnd((B, H, d), 58, 2.0)
    k, v = rnd((B, H, Tkv, d), 59), rnd((B, H, Tkv, d), 60)
    mem, w = rnd((B, H, d), 61), rnd((H, d), 62)
    a = oracle_decode(q, k, v, mem, w, nsplit=0)
    b = oracle_decode(q, k, v, mem, w, nsplit=nsplit, tile=tile)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)


def test_decode_equals_last_prefill_row():
    B, H, T, d = 1, 2, 300, 16
    q, k, v = rnd((B, H, T, d), 63), rnd((B, H, T, d), 64), rnd((B, H, T, d), 65)
    mem, w = rnd((B, H, T, d), 66), rnd((H, d), 67)
    o, n, c = oracle_fwd(q, k, v, mem, w)
    od, nd, cd = oracle_decode(q[:, :, -1], k, v, mem[:, :, -1], w, nsplit=3)
    np.testing.assert_allclose(od, o[:, :, -1], atol=1e-12)
    np.testing.assert_allclose(nd, n[:, :, -1], rtol=1e-12)
    np.testing.assert_allclose(cd, c[:, :, -1], rtol=1e-12)


# ------------------------------------------------ brute force, tiny inputs

def _brute_row(q, K, V, mem, w, i, d):
    """Re-evaluation of one row with Python floats, key by key."""
    n = i + 1
    tau = max(1.0, math.log(n) / LN_T0)
    s = [tau * sum(q[i][x] * K[j][x] for x in range(d)) / math.sqrt(d)
         for j in range(n)]
    Z = sum(math.exp(t) for t in s)
    p = [math.exp(t) / Z for t in s]
    neff = 1.0 / sum(t * t for t in p)
    a = [sum(p[j] * V[j][x] for j in range(n)) for x in range(d)]
    an = math.sqrt(sum(t * t for t in a))
    u = [t / max(an, 1e-6) for t in a]
    qn = math.sqrt(sum(t * t for t in q[i]))
    b = tau * qn / math.sqrt(d) * math.sqrt(2 * math.log(n))
    conf = 1.0 / (1.0 + math.exp(-(math.log(Z) - b)))
    count = conf * math.tanh(math.log(neff) / LN_T0)
    return [u[x] + count * w[x] + mem[i][x] for x in range(d)], neff, conf


def test_brute_force_tiny():
    T, d = 6, 3
    q, k, v = rnd((T, d), 68, 1.5), rnd((T, d), 69), rnd((T, d), 70)
    mem, w = rnd((T, d), 71), rnd(d, 72)
    out, ne, cf = oracle_rows(q, k, v, mem, w, list(range(T)))
    for i in range(T):
        o, n_, c_ = _brute_row(q.tolist(), k.tolist(), v.tolist(), mem.tolist(),
                               w.tolist(), i, d)
        np.testing.assert_allclose(out[i], o, atol=1e-13)
        assert ne[i] == pytest.approx(n_, rel=1e-13)
        assert cf[i] == pytest.approx(c_, rel=1e-13)


# ----------------------------------------------- paged, grouped decode (NEXT)

def _paged(B, Hq, Hkv, T, d, P, seed, ragged=True):
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.custom_paged(B=B, Hq=Hq, Hkv=Hkv, T=T, d=d, page=P, dtype="f32",
                             seed=seed, ragged=ragged)
    return inputs.make_paged_decode(wl, "cpu")


def test_paged_decode_identity_layout_equals_contiguous_decode():
    """With pages laid out in order and one query head per KV head, the
    paged decode is the contiguous decode of the same cache."""
    from oracle import oracle_decode_paged
    B, H, T, d, P = 2, 3, 100, 8, 16
    x = _paged(B, H, H, T, d, P, 800, ragged=False)
    npg = (T + P - 1) // P
    table = np.arange(B * npg).reshape(B, npg).astype(np.int32)
    k = rnd((B, H, npg * P, d), 801)
    v = rnd((B, H, npg * P, d), 802)
    # pages[b * npg + p, h, r] = k[b, h, p * P + r]
    kp = k.reshape(B, H, npg, P, d).transpose(0, 2, 1, 3, 4).reshape(B * npg, H, P, d)
    vp = v.reshape(B, H, npg, P, d).transpose(0, 2, 1, 3, 4).reshape(B * npg, H, P, d)
    lens = np.full(B, T)
    a = oracle_decode_paged(x["q"], kp, vp, table, lens, x["mem"], x["w_count"])
    b = oracle_decode(x["q"], k[:, :, :T], v[:, :, :T], x["mem"], x["w_count"])
    for u, w in zip(a, b):
        np.testing.assert_allclose(u, w, rtol=1e-13, atol=1e-13)


def test_paged_decode_page_permutation_invariance():
    """Moving physical pages (and the table with them) changes nothing."""
    from oracle import oracle_decode_paged
    x = _paged(3, 4, 2, 90, 8, 16, 803)
    kp = x["k_pages"].double().numpy()
    vp = x["v_pages"].double().numpy()
    perm = np.random.default_rng(804).permutation(kp.shape[0])
    inv = np.argsort(perm)
    table = x["block_table"].numpy()
    a = oracle_decode_paged(x["q"], kp, vp, table, x["seq_lens"], x["mem"], x["w_count"])
    b = oracle_decode_paged(x["q"], kp[perm], vp[perm], inv[table], x["seq_lens"],
                            x["mem"], x["w_count"])
    for u, w in zip(a, b):
        np.testing.assert_array_equal(u, w)


def test_paged_decode_grouped_heads_share_kv():
    """Query heads of one group read the same keys: identical queries in a
    group give identical results; n = seq_len per sequence (a one-token
    sequence has n_eff = 1)."""
    from oracle import oracle_decode_paged
    x = _paged(3, 8, 2, 70, 8, 16, 805)
    q = x["q"].clone()
    q[:, 1] = q[:, 0]          # heads 0 and 1 share kv head 0 (G = 4)
    w = torch.zeros_like(x["w_count"])
    mem = torch.zeros_like(x["mem"])
    out, ne, cf = oracle_decode_paged(q, x["k_pages"], x["v_pages"], x["block_table"],
                                      x["seq_lens"], mem, w)
    np.testing.assert_array_equal(out[:, 0], out[:, 1])
    lens = x["seq_lens"].numpy()
    one = np.where(lens == 1)[0]
    assert len(one) == 1
    np.testing.assert_allclose(ne[one[0]], 1.0, rtol=0, atol=1e-15)
    assert np.all(ne <= lens[:, None] + 1e-9)


# ------------------------------------------- gated-delta memory step (NEXT)

def test_memory_step_delta_write_closed_form():
    """alpha = beta = 1: the step writes v at k^ exactly (S k^ = v), keeps
    what S held on the orthogonal complement of k^, and reads mem = S q^."""
    from oracle import oracle_memory_step
    d = 16
    S0 = rnd((1, 1, d, d), 900)
    q, k, v = rnd((1, 1, 1, d), 901), rnd((1, 1, 1, d), 902), rnd((1, 1, 1, d), 903)
    one = np.ones((1, 1, 1))
    S1, mem = oracle_memory_step(S0, q, k, v, one, one)
    kh = k[0, 0, 0] / np.linalg.norm(k[0, 0, 0])
    np.testing.assert_allclose(S1[0, 0] @ kh, v[0, 0, 0], atol=1e-12)
    x = rnd(d, 904)
    x -= (x @ kh) * kh                      # orthogonal to k^
    np.testing.assert_allclose(S1[0, 0] @ x, S0[0, 0] @ x, atol=1e-12)
    qh = q[0, 0, 0] / np.linalg.norm(q[0, 0, 0])
    np.testing.assert_allclose(mem[0, 0, 0], S1[0, 0] @ qh, atol=1e-12)


def test_memory_step_gate_and_empty_state_closed_forms():
    from oracle import oracle_memory_step
    d = 8
    S0 = rnd((1, 1, d, d), 905)
    q, k, v = rnd((1, 1, 1, d), 906), rnd((1, 1, 1, d), 907), rnd((1, 1, 1, d), 908)
    a = np.full((1, 1, 1), 0.7)
    S1, _ = oracle_memory_step(S0, q, k, v, a, np.zeros((1, 1, 1)))
    np.testing.assert_allclose(S1, 0.7 * S0, atol=1e-14)        # beta = 0: pure decay
    b = np.full((1, 1, 1), 0.3)
    S2, mem = oracle_memory_step(np.zeros((1, 1, d, d)), q, k, v, a, b)
    kh = k[0, 0, 0] / np.linalg.norm(k[0, 0, 0])
    qh = q[0, 0, 0] / np.linalg.norm(q[0, 0, 0])
    np.testing.assert_allclose(S2[0, 0], 0.3 * np.outer(v[0, 0, 0], kh), atol=1e-14)
    np.testing.assert_allclose(mem[0, 0, 0], 0.3 * (kh @ qh) * v[0, 0, 0], atol=1e-14)


def test_memory_step_is_stable_for_any_key_scale():
    """With values zero the state never grows, whatever the key scale and the
    gates in [0, 1]: the L2 normalisation keeps the transition's eigenvalues
    in [0, 1] (the pages' stability argument)."""
    from oracle import oracle_memory_step
    d, T = 8, 40
    S = rnd((1, 1, d, d), 909)
    k = rnd((1, 1, T, d), 910, 30.0)        # large keys
    q = rnd((1, 1, T, d), 911)
    g = np.random.default_rng(912)
    alpha, beta = g.uniform(0.5, 1, (1, 1, T)), g.uniform(0, 1, (1, 1, T))
    beta[0, 0, ::3] = 1.0
    S_end, _ = oracle_memory_step(S, q, k, np.zeros((1, 1, T, d)), alpha, beta)
    norms = [np.linalg.norm(S[0, 0], 2)]
    St = S
    for t in range(T):
        St, _ = oracle_memory_step(St, q[:, :, t:t + 1], k[:, :, t:t + 1],
                                   np.zeros((1, 1, 1, d)), alpha[:, :, t:t + 1],
                                   beta[:, :, t:t + 1])
        norms.append(np.linalg.norm(St[0, 0], 2))
    assert np.all(np.diff(norms) <= 1e-12)
    np.testing.assert_allclose(St, S_end, atol=1e-12)  # T steps = one call of T


def test_memory_step_matches_rank_one_form():
    """Brute re-evaluation: S a(I - b k^k^T) + b v k^T equals
    a S + (b v - a b (S k^)) k^T (the in-place row form)."""
    from oracle import oracle_memory_step
    d = 12
    S0 = rnd((2, 1, d, d), 913)
    q, k, v = rnd((2, 1, 1, d), 914), rnd((2, 1, 1, d), 915), rnd((2, 1, 1, d), 916)
    a = np.array([0.9, 0.4]).reshape(2, 1, 1)
    b = np.array([0.2, 1.0]).reshape(2, 1, 1)
    S1, _ = oracle_memory_step(S0, q, k, v, a, b)
    for i in range(2):
        kh = k[i, 0, 0] / np.linalg.norm(k[i, 0, 0])
        u = S0[i, 0] @ kh
        ref = a[i, 0, 0] * S0[i, 0] + np.outer(b[i, 0, 0] * v[i, 0, 0] - a[i, 0, 0] * b[i, 0, 0] * u, kh)
        np.testing.assert_allclose(S1[i, 0], ref, atol=1e-12)


# ------------------------------------------------------- backward (NEXT)

@pytest.mark.parametrize("floor_order", [1, 2])
def test_backward_matches_finite_differences_of_the_c_oracle(floor_order):
    """The backward oracle (dense torch restatement + autograd) against
    central differences of the plain-C forward oracle, coordinate by
    coordinate, for q, k, v, w and mem, rows on both sides of the 2K
    temperature knee excluded for speed (tau = 1 here; tau > 1 below)."""
    from oracle import oracle_bwd
    B, H, T, d = 1, 2, 12, 8
    q, k, v = rnd((B, H, T, d), 1000, 1.5), rnd((B, H, T, d), 1001), rnd((B, H, T, d), 1002)
    mem, w, g = rnd((B, H, T, d), 1003), rnd((H, d), 1004, 0.3), rnd((B, H, T, d), 1005)
    consts = dict(DEFAULT_CONSTS, floor_order=floor_order)
    grads = oracle_bwd(q, k, v, mem, w, g, consts)

    def loss(**kw):
        x = dict(q=q, k=k, v=v, mem=mem, w=w)
        x.update(kw)
        out, _, _ = oracle_fwd(x["q"], x["k"], x["v"], x["mem"], x["w"], consts=consts,
                               nthreads=1)
        return float((out * g).sum())

    rng = np.random.default_rng(1006)
    h = 1e-6
    for name, arr, gname in (("q", q, "dq"), ("k", k, "dk"), ("v", v, "dv"),
                             ("w", w, "dw"), ("mem", mem, "dmem")):
        for _ in range(6):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            xp, xm = arr.copy(), arr.copy()
            xp[idx] += h
            xm[idx] -= h
            fd = (loss(**{name: xp}) - loss(**{name: xm})) / (2 * h)
            assert grads[gname][idx] == pytest.approx(fd, rel=1e-5, abs=1e-7), (name, idx)


def test_backward_beyond_training_length_finite_differences():
    """Same check on rows past 2048 keys (tau > 1), a few rows only."""
    from oracle import oracle_bwd
    T, d = 2060, 4
    q, k, v = rnd((1, 1, T, d), 1010), rnd((1, 1, T, d), 1011), rnd((1, 1, T, d), 1012)
    mem, w = np.zeros((1, 1, T, d)), rnd((1, d), 1013, 0.3)
    g = np.zeros((1, 1, T, d))
    g[0, 0, -3:] = rnd((3, d), 1014)          # loss on the last rows only
    grads = oracle_bwd(q, k, v, mem, w, g)

    def loss(qq):
        out, _, _ = oracle_rows(qq[0, 0], k[0, 0], v[0, 0], mem[0, 0], w[0],
                                [T - 3, T - 2, T - 1])
        return float((out * g[0, 0, -3:]).sum())

    h = 1e-6
    for i in (T - 1, T - 2):
        for x in range(d):
            qp, qm = q.copy(), q.copy()
            qp[0, 0, i, x] += h
            qm[0, 0, i, x] -= h
            fd = (loss(qp) - loss(qm)) / (2 * h)
            assert grads["dq"][0, 0, i, x] == pytest.approx(fd, rel=1e-5, abs=1e-7)


def test_backward_closed_forms():
    """d out / d mem is the identity; d/dw sums count * dout over rows."""
    from oracle import oracle_bwd
    B, H, T, d = 1, 2, 9, 4
    q = np.zeros((B, H, T, d))
    q[..., 0] = 1e-3                                   # near-uniform rows
    k, v = rnd((B, H, T, d), 1020), rnd((B, H, T, d), 1021)
    w, g = rnd((H, d), 1022), rnd((B, H, T, d), 1023)
    grads = oracle_bwd(q, k, v, np.zeros_like(q), w, g)
    np.testing.assert_array_equal(grads["dmem"], g)
    _, neff, conf = oracle_fwd(q, k, v, np.zeros_like(q), w)
    count = conf * np.tanh(np.log(neff) / math.log(2048.0))
    np.testing.assert_allclose(grads["dw"], np.einsum("bht,bhtd->hd", count, g), rtol=1e-10)


# --------------------------------------------------------------- row stats
def test_row_stats_closed_form_zero_query():
    """q = 0: every logit is 0, so lse = ln n and a is the running mean of v."""
    from oracle import oracle_row_stats
    rng = np.random.default_rng(81)
    T, d = 40, 16
    q = np.zeros((1, 1, T, d))
    k = rng.standard_normal((1, 1, T, d))
    v = rng.standard_normal((1, 1, T, d))
    st = oracle_row_stats(q, k, v)
    n = np.arange(1, T + 1)
    np.testing.assert_allclose(st["lse"][0, 0], np.log(n), rtol=0, atol=1e-13)
    mean = np.cumsum(v[0, 0], axis=0) / n[:, None]
    np.testing.assert_allclose(st["anorm"][0, 0], np.linalg.norm(mean, axis=-1), rtol=1e-12)


def test_row_stats_lse_agrees_with_the_c_oracle_gate():
    """conf = sigmoid(lse - b) in the C oracle (an independent implementation):
    b + logit(conf) recovers the same logsumexp."""
    from oracle import oracle_fwd, oracle_row_stats
    rng = np.random.default_rng(82)
    B, H, T, d = 1, 2, 96, 32
    q, k, v, mem = (rng.standard_normal((B, H, T, d)) for _ in range(4))
    w = rng.standard_normal((H, d)) * 0.1
    _, _, conf = oracle_fwd(q, k, v, mem, w)
    st = oracle_row_stats(q, k, v)
    n = np.arange(1, T + 1, dtype=np.float64)
    sigma = np.linalg.norm(q, axis=-1) / math.sqrt(d)          # tau = 1 below 2048 keys
    b = sigma * np.sqrt(2.0 * np.log(n))
    ok = (conf > 1e-6) & (conf < 1 - 1e-6)
    assert ok.mean() > 0.9
    lse_c = b + np.log(conf) - np.log1p(-conf)
    np.testing.assert_allclose(st["lse"][ok], lse_c[ok], rtol=0, atol=1e-8)


def test_row_stats_anorm_matches_sdpa():
    """Below the 2K training length tau = 1, so a is causal SDPA's output."""
    import torch
    from oracle import oracle_row_stats
    rng = np.random.default_rng(83)
    q, k, v = (rng.standard_normal((2, 2, 70, 24)) for _ in range(3))
    st = oracle_row_stats(q, k, v)
    a = torch.nn.functional.scaled_dot_product_attention(
        torch.as_tensor(q), torch.as_tensor(k), torch.as_tensor(v), is_causal=True).numpy()
    np.testing.assert_allclose(st["anorm"], np.linalg.norm(a, axis=-1), rtol=1e-11)


@pytest.mark.parametrize("floor_order", [1, 2])
def test_sampled_backward_equals_the_dense_oracle(floor_order):
    """The blockwise, per-output form used at full lengths reproduces the
    dense autograd oracle (itself pinned by finite differences) at every row
    and key, including rows beyond the 2K training length and a block size
    that does not divide T."""
    from oracle import oracle_bwd, oracle_bwd_sampled
    rng = np.random.default_rng(91)
    B, H, T, d = 1, 2, 2300, 16
    q, k, v, mem, g = (rng.standard_normal((B, H, T, d)) for _ in range(5))
    q[0, 1, 7] = 0.0  # a row with |q| = 0 (no floor gradient)
    w = rng.standard_normal((H, d)) * 0.2
    c = {"floor_order": floor_order}
    ref = oracle_bwd(q, k, v, mem, w, g, consts=c)
    rows = [0, 1, 7, 500, 2047, 2048, 2299]
    keys = [0, 3, 1000, 2200, 2299]
    for h in range(H):
        got = oracle_bwd_sampled(q[0, h], k[0, h], v[0, h], w[h], g[0, h], rows, keys,
                                 consts=c, block=333)
        np.testing.assert_allclose(got["dq"], ref["dq"][0, h, rows], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(got["dk"], ref["dk"][0, h, keys], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(got["dv"], ref["dv"][0, h, keys], rtol=1e-9, atol=1e-11)
        dw_h = (got["count"][:, None] * g[0, h]).sum(axis=0)
        np.testing.assert_allclose(dw_h, ref["dw"][h], rtol=1e-9)
