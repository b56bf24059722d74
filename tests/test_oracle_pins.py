"""Pins of the fp64 CPU oracle to things other than itself (no GPU needed).

Each test fixes the oracle against something the pages or the mathematics
determine independently of its code:
  * IEEE-754 binary16 rounding, exhaustively, against NumPy's float64->float16
    conversion (a direct, correctly rounded conversion);
  * the update written as dense matrices, S' = (I - beta khat khat^T) diag(alpha) S
    + beta khat v^T, in NumPy fp64 and in 50-digit mpmath, with alpha taken from
    the identity exp(-softplus(a)) = 1 / (1 + e^a) rather than the oracle's form;
  * closed forms: identity step, full forget, delta-rule recall, basis key, reset;
  * the norm bound of ROCm/ATOM pull request 2945 (Limitations);
  * the per-slot state sizes printed by pull request 2130 (Memory).
Shapes with K != V are used so that a transposed operand cannot pass.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from kda_linear_attention_gated_gb300 import workloads

EPS = 1e-6
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

pytestmark = pytest.mark.usefixtures("oracle_mod")


# ---------------------------------------------------------------------------
# independent restatements used as pins
# ---------------------------------------------------------------------------
def dense_step(S, q, k, v, a, b):
    """One token as dense fp64 matrix algebra.  S: [K, V]."""
    K = S.shape[0]
    kh = k / np.sqrt(k @ k + EPS)
    qh = q / np.sqrt(q @ q + EPS)
    beta = 1.0 / (1.0 + np.exp(-b))
    with np.errstate(over="ignore"):
        alpha = 1.0 / (1.0 + np.exp(a))
    S1 = (np.eye(K) - beta * np.outer(kh, kh)) @ np.diag(alpha) @ S + beta * np.outer(kh, v)
    return S1, S1.T @ qh / math.sqrt(K)


def f32_ulps(x32, y64):
    """|x - y| in units of the fp32 spacing at y."""
    y64 = np.asarray(y64, np.float64)
    sp = np.spacing(np.abs(y64).astype(np.float32)).astype(np.float64)
    return np.abs(np.asarray(x32, np.float64) - y64) / sp


# ---------------------------------------------------------------------------
# fp16 rounding
# ---------------------------------------------------------------------------
def test_f16_widen_round_trip_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    wide = oracle_mod.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(wide), nan)
    assert np.array_equal(wide[~nan], ref[~nan])
    back = oracle_mod.f64_to_f16_rne(wide[~nan])
    assert np.array_equal(back, bits[~nan])          # -0.0 included


def test_f16_rne_midpoints_and_neighbours(oracle_mod):
    # every pair of adjacent finite fp16 values of one sign, their exact midpoint
    # (representable in fp64) and the fp64 values one ulp either side of it
    pos = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (pos[:-1] + pos[1:]) / 2
    # the midpoint between the largest finite value and 2^16 (rounds to inf)
    mids = np.concatenate([mids, [65520.0]])
    cand = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf),
                           [65519.99, 65536.0, 1e9, 2.0**-25, 2.0**-26, 3 * 2.0**-26]])
    cand = np.concatenate([cand, -cand])
    got = oracle_mod.f64_to_f16_rne(cand)
    ref = cand.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_f16_specials(oracle_mod):
    got = oracle_mod.f64_to_f16_rne(np.array([np.inf, -np.inf, np.nan, 0.0, -0.0]))
    assert got[0] == 0x7C00 and got[1] == 0xFC00
    assert (got[2] & 0x7C00) == 0x7C00 and (got[2] & 0x3FF) != 0
    assert got[3] == 0 and got[4] == 0x8000


# ---------------------------------------------------------------------------
# brute force
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("K,V,HV,T,seed", [(5, 3, 2, 4, 0), (3, 7, 1, 6, 1), (16, 16, 2, 8, 2),
                                           (8, 24, 3, 3, 3)])
def test_verify_matches_dense_brute_force(oracle_mod, K, V, HV, T, seed):
    rng = np.random.default_rng(seed)
    n, ns = 2, 2 + 2 * T
    pool = (rng.standard_normal((ns, HV, K, V)) * 0.1).astype(np.float32)
    init = np.array([0, 1], np.int32)
    snap = np.arange(2, 2 + n * T, dtype=np.int32).reshape(n, T)
    q, k, a = (rng.standard_normal((n, T, HV, K)) for _ in range(3))
    v = rng.standard_normal((n, T, HV, V))
    b = rng.standard_normal((n, T, HV))
    pool0 = pool.copy()
    o = oracle_mod.spec_verify(pool, init, snap, q, k, v, a, b)
    for r in range(n):
        for h in range(HV):
            S = pool0[init[r], h].astype(np.float64)
            for t in range(T):
                S, ob = dense_step(S, q[r, t, h], k[r, t, h], v[r, t, h], a[r, t, h], b[r, t, h])
                np.testing.assert_allclose(o[r, t, h], ob, rtol=1e-12, atol=1e-13)
                assert f32_ulps(pool[snap[r, t], h], S).max() <= 0.5000001
    # the init slots are only read
    assert np.array_equal(pool[init], pool0[init])


def test_tiny_decode_chain_matches_dense(oracle_mod):
    """Config 'tiny': 8 sequential decode calls on a 1-slot fp32 pool (state
    rounded to fp32 between calls, as a stored state is)."""
    tiny = workloads.make_tiny(seed=0)
    pool = tiny["pool"].numpy().copy()
    S = pool[0].astype(np.float64)
    for t in range(8):
        f = lambda x: x[t].double().numpy()  # noqa: E731
        o = oracle_mod.decode_step(pool, tiny["slot"], f(tiny["q"]), f(tiny["k"]), f(tiny["v"]),
                                   f(tiny["a"]), f(tiny["b"]))
        for h in range(2):
            Sh, ob = dense_step(S[h], f(tiny["q"])[0, h], f(tiny["k"])[0, h], f(tiny["v"])[0, h],
                                f(tiny["a"])[0, h], f(tiny["b"])[0, h])
            np.testing.assert_allclose(o[0, h], ob, rtol=1e-12, atol=1e-13)
            assert f32_ulps(pool[0, h], Sh).max() <= 0.5000001
        S = pool[0].astype(np.float64)


def test_tiny_against_mpmath_50_digits(oracle_mod):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    tiny = workloads.make_tiny(seed=0)
    T, HV, K, V = 8, 2, 16, 16
    pool = np.zeros((1 + T, HV, K, V), np.float32)
    pool[0] = tiny["pool"].numpy()[0]
    g = {n: tiny[n].double().numpy()[:, 0] for n in ("q", "k", "v", "a", "b")}  # [T, HV, ...]
    o = oracle_mod.spec_verify(pool, np.array([0], np.int32),
                               np.arange(1, 1 + T, dtype=np.int32)[None],
                               *(g[n][None] for n in ("q", "k", "v", "a", "b")))
    for h in range(HV):
        S = mp.matrix([[mp.mpf(float(x)) for x in row] for row in pool[0, h]])
        for t in range(T):
            q, k, v, a = ([mp.mpf(float(x)) for x in g[n][t, h]] for n in ("q", "k", "v", "a"))
            b = mp.mpf(float(g["b"][t, h]))
            kn = mp.sqrt(sum(x * x for x in k) + mp.mpf("1e-6"))
            qn = mp.sqrt(sum(x * x for x in q) + mp.mpf("1e-6"))
            kh = [x / kn for x in k]
            qh = [x / qn for x in q]
            beta = 1 / (1 + mp.exp(-b))
            alpha = [mp.exp(-mp.log(1 + mp.exp(x))) for x in a]
            for i in range(K):
                for j in range(V):
                    S[i, j] *= alpha[i]
            u = [sum(S[i, j] * kh[i] for i in range(K)) for j in range(V)]
            for i in range(K):
                for j in range(V):
                    S[i, j] += beta * kh[i] * (v[j] - u[j])
            for j in range(V):
                oj = sum(S[i, j] * qh[i] for i in range(K)) / mp.sqrt(K)
                assert abs(float(oj) - o[0, t, h, j]) <= 1e-13 * max(1.0, abs(float(oj)))


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
def _rand_step(rng, n=3, HV=2, K=16, V=8):
    return dict(q=rng.standard_normal((n, HV, K)), k=rng.standard_normal((n, HV, K)),
                v=rng.standard_normal((n, HV, V)), a=rng.standard_normal((n, HV, K)),
                b=rng.standard_normal((n, HV)))


@pytest.mark.parametrize("state_dtype", [np.float32, np.float16])
def test_identity_step_leaves_pool_bit_identical(oracle_mod, state_dtype):
    """alpha = 1 (a = -inf) and beta = 0 (b = -inf): the update is the identity,
    so the widen -> store round trip must return the pool's exact bits (an fp32
    pool is unchanged by the fp16 machinery: ROCm/ATOM pull request 2945, Summary)."""
    rng = np.random.default_rng(5)
    x = _rand_step(rng)
    x["a"][:] = -np.inf
    x["b"][:] = -np.inf
    pool = (rng.standard_normal((4, 2, 16, 8)) * 0.1).astype(state_dtype)
    before = pool.copy()
    slots = np.array([2, 0, 3], np.int32)
    o = oracle_mod.decode_step(pool, slots, **x)
    assert pool.tobytes() == before.tobytes()
    for r, s in enumerate(slots):
        for h in range(2):
            qh = x["q"][r, h] / np.sqrt(x["q"][r, h] @ x["q"][r, h] + EPS)
            np.testing.assert_allclose(o[r, h], before[s, h].astype(np.float64).T @ qh / 4.0,
                                       rtol=1e-12, atol=1e-14)


def test_full_forget_closed_form(oracle_mod):
    """alpha = 0 (a = +inf): S' = beta khat v^T and o = beta (qhat.khat) v / sqrt(K)."""
    rng = np.random.default_rng(6)
    x = _rand_step(rng)
    x["a"][:] = np.inf
    pool = (rng.standard_normal((3, 2, 16, 8)) * 0.1).astype(np.float32)
    slots = np.array([1, 2, 0], np.int32)
    o = oracle_mod.decode_step(pool, slots, **x)
    for r, s in enumerate(slots):
        for h in range(2):
            k, q, v = x["k"][r, h], x["q"][r, h], x["v"][r, h]
            kh, qh = k / np.sqrt(k @ k + EPS), q / np.sqrt(q @ q + EPS)
            beta = 1 / (1 + np.exp(-x["b"][r, h]))
            assert f32_ulps(pool[s, h], beta * np.outer(kh, v)).max() <= 0.5000001
            np.testing.assert_allclose(o[r, h], beta * (qh @ kh) * v / 4.0, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("b_val", [None, np.inf])
def test_delta_rule_recall(oracle_mod, b_val):
    """With q = k the read-out is S'^T khat / sqrt(K) = (u + beta |khat|^2 (v - u)) / sqrt(K),
    u = (diag(alpha) S)^T khat; with beta = 1 the state recalls v for k (up to |khat|^2)."""
    rng = np.random.default_rng(7)
    x = _rand_step(rng)
    x["q"] = x["k"].copy()
    if b_val is not None:
        x["b"][:] = b_val
    pool = (rng.standard_normal((3, 2, 16, 8)) * 0.1).astype(np.float32)
    before = pool.copy()
    slots = np.array([0, 1, 2], np.int32)
    o = oracle_mod.decode_step(pool, slots, **x)
    for r, s in enumerate(slots):
        for h in range(2):
            k, v = x["k"][r, h], x["v"][r, h]
            kk = k @ k
            kh = k / np.sqrt(kk + EPS)
            alpha = 1 / (1 + np.exp(x["a"][r, h]))
            beta = 1 / (1 + np.exp(-x["b"][r, h]))
            u = (alpha[:, None] * before[s, h].astype(np.float64)).T @ kh
            kap = kk / (kk + EPS)
            np.testing.assert_allclose(o[r, h] * 4.0, u + beta * kap * (v - u), rtol=1e-12, atol=1e-14)
            if b_val is not None:
                np.testing.assert_allclose(o[r, h] * 4.0, v, rtol=1e-6, atol=1e-6)


def test_basis_key_touches_one_row(oracle_mod):
    """k = c e_i: rows r != i only decay; row i becomes (1 - beta s^2) alpha_i S_i + beta s v,
    s = c / sqrt(c^2 + eps)."""
    rng = np.random.default_rng(8)
    x = _rand_step(rng, n=1, HV=1, K=16, V=8)
    i, c = 5, 2.5
    x["k"][:] = 0.0
    x["k"][0, 0, i] = c
    pool = (rng.standard_normal((1, 1, 16, 8)) * 0.1).astype(np.float32)
    S = pool[0, 0].astype(np.float64)
    oracle_mod.decode_step(pool, np.array([0], np.int32), **x)
    alpha = 1 / (1 + np.exp(x["a"][0, 0]))
    beta = 1 / (1 + np.exp(-x["b"][0, 0]))
    s = c / math.sqrt(c * c + EPS)
    want = alpha[:, None] * S
    want[i] = (1 - beta * s * s) * alpha[i] * S[i] + beta * s * x["v"][0, 0]
    assert f32_ulps(pool[0, 0], want).max() <= 0.5000001


def test_zero_key_gives_no_nan(oracle_mod):
    rng = np.random.default_rng(9)
    x = _rand_step(rng, n=1, HV=1)
    x["k"][:] = 0.0
    pool = (rng.standard_normal((1, 1, 16, 8)) * 0.1).astype(np.float32)
    S = pool[0, 0].astype(np.float64)
    o = oracle_mod.decode_step(pool, np.array([0], np.int32), **x)
    alpha = 1 / (1 + np.exp(x["a"][0, 0]))
    assert np.isfinite(o).all()
    assert f32_ulps(pool[0, 0], alpha[:, None] * S).max() <= 0.5000001


def test_reset_equals_zero_state(oracle_mod):
    rng = np.random.default_rng(10)
    x = _rand_step(rng)
    p1 = (rng.standard_normal((3, 2, 16, 8)) * 0.1).astype(np.float16)
    p2 = p1.copy()
    p2[1] = 0
    slots = np.array([0, 1, 2], np.int32)
    o1 = oracle_mod.decode_step(p1, slots, reset=np.array([0, 1, 0], np.uint8), **x)
    o2 = oracle_mod.decode_step(p2, slots, **x)
    assert p1.tobytes() == p2.tobytes()
    assert np.array_equal(o1, o2)


def test_out_of_range_slot_is_refused(oracle_mod):
    rng = np.random.default_rng(11)
    x = _rand_step(rng, n=1)
    pool = np.zeros((2, 2, 16, 8), np.float32)
    with pytest.raises(ValueError):
        oracle_mod.decode_step(pool, np.array([2], np.int32), **x)


# ---------------------------------------------------------------------------
# the norm bound (ROCm/ATOM pull request 2945, Limitations)
# ---------------------------------------------------------------------------
def test_norm_bound_every_token(oracle_mod):
    """|S'[:, j]|^2 <= |S[:, j]|^2 + v_j^2 for every token and column, on the tiny
    workload and on a larger random one with extreme gates."""
    rng = np.random.default_rng(12)
    cases = [workloads.make_tiny(seed=0)]
    for case in cases:
        T, HV = 8, 2
        pool = np.zeros((1 + T, HV, 16, 16), np.float32)
        pool[0] = case["pool"].numpy()[0]
        g = {n: case[n].double().numpy()[:, 0][None] for n in ("q", "k", "v", "a", "b")}
        oracle_mod.spec_verify(pool, np.array([0], np.int32),
                               np.arange(1, 1 + T, dtype=np.int32)[None], *(g[n] for n in "qkvab"))
        prev = pool[0].astype(np.float64)
        for t in range(T):
            cur = pool[1 + t].astype(np.float64)
            lhs = (cur ** 2).sum(axis=1)                    # [HV, V]
            rhs = (prev ** 2).sum(axis=1) + g["v"][0, t] ** 2
            assert (lhs <= rhs * (1 + 1e-6) + 1e-12).all()
            prev = cur
    # extreme gates: beta near 1, alpha near 1
    K, V, T = 32, 16, 6
    pool = np.zeros((1 + T, 1, K, V), np.float32)
    pool[0] = rng.standard_normal((1, K, V)) * 3
    q, k = rng.standard_normal((1, T, 1, K)), rng.standard_normal((1, T, 1, K))
    v = rng.standard_normal((1, T, 1, V)) * 4
    a = np.full((1, T, 1, K), -30.0)
    b = np.full((1, T, 1), 30.0)
    oracle_mod.spec_verify(pool, np.array([0], np.int32), np.arange(1, 1 + T, dtype=np.int32)[None],
                           q, k, v, a, b)
    prev = pool[0].astype(np.float64)
    for t in range(T):
        cur = pool[1 + t].astype(np.float64)
        assert ((cur ** 2).sum(axis=1) <= ((prev ** 2).sum(axis=1) + v[0, t] ** 2) * (1 + 1e-6)).all()
        prev = cur


def test_verify_equals_chained_decode_fp32(oracle_mod):
    """T verify tokens == T decode calls, up to the fp32 rounding the decode chain adds."""
    d = workloads.make_verify(n=2, t=4, hv=2, k=16, v=16, num_slots=16,
                              state_dtype=torch.float32, seed=4)
    pool_v = d.pool.numpy().copy()
    pool_d = d.pool.numpy().copy()
    ov = oracle_mod.spec_verify(pool_v, d.init_slot, d.snap_slot, d.q, d.k, d.v, d.a, d.b)
    for t in range(4):
        od = oracle_mod.decode_step(pool_d, d.init_slot, d.q[:, t], d.k[:, t], d.v[:, t],
                                    d.a[:, t], d.b[:, t])
        np.testing.assert_allclose(od, ov[:, t], rtol=1e-5, atol=1e-6)
        for r in range(2):
            np.testing.assert_allclose(pool_d[d.init_slot[r]], pool_v[d.snap_slot[r, t]],
                                       rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------------------
# the pages' printed state sizes
# ---------------------------------------------------------------------------
def test_state_bytes_match_printed_memory_table():
    g = json.load(open(os.path.join(GOLDEN, "state_memory_pr2130.json")))
    hv, k, v = g["state_shape"]
    per_layer = {"fp32": hv * k * v * 4, "fp16": hv * k * v * 2}
    kda_half = g["layers"] * (per_layer["fp32"] - per_layer["fp16"])
    printed = g["state_per_slot_MB"]["fp32"] - g["state_per_slot_MB"]["fp16"]
    assert round(kda_half / 1e6, 2) == pytest.approx(printed, abs=1e-9)
    # 68 layers (the other count the pages give) does not reproduce the table
    assert round(68 * (per_layer["fp32"] - per_layer["fp16"]) / 1e6, 2) != pytest.approx(printed)
    for dt in ("fp32", "fp16"):
        assert round(g["state_per_slot_MB"][dt] * 1e6 * 64 / 2**30, 2) == g["state_pool_64_slots_GB"][dt]


# ---------------------------------------------------------------------------
# The general step (accepted-length speculative decode, packed variable-length
# requests, padding, grouped q/k heads, learned gate scale): each feature is
# pinned to the plain forms above or to a closed form.
# ---------------------------------------------------------------------------
def _pool64(pool):
    return pool.numpy().copy() if pool.dtype == torch.float32 else pool.view(torch.int16).numpy().view(np.uint16).copy()


def _general(inp, **over):
    pool = _pool64(inp.pool)
    kw = dict(cu_seqlens=inp.cu_seqlens, accepted=inp.accepted, reset=inp.reset, a_log=inp.a_log,
              dt_bias=inp.dt_bias, in_place=inp.in_place)
    kw.update(over)
    o = oracle.step(pool, inp.slot_table, inp.q, inp.k, inp.v, inp.a, inp.b, **kw)
    return pool, o


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_general_step_is_verify_from_the_accepted_column(state_dtype):
    inp = workloads.make_general(n=5, t=4, num_cols=6, hv=3, k=16, v=32, num_slots=40,
                                 state_dtype=state_dtype, seed=21, reset_p=0.3)
    pool, o = _general(inp)
    n, t = 5, 4
    ref = _pool64(inp.pool)
    init = inp.slot_table[torch.arange(n), inp.accepted.long() - 1]
    o_ref = oracle.spec_verify(ref, init, inp.slot_table[:, :t], inp.q.reshape(n, t, 3, 16),
                               inp.k.reshape(n, t, 3, 16), inp.v.reshape(n, t, 3, 32),
                               inp.a.reshape(n, t, 3, 16), inp.b.reshape(n, t, 3), reset=inp.reset)
    assert np.array_equal(pool, ref)
    assert np.array_equal(o.reshape(n, t, 3, 32), o_ref)


@pytest.mark.parametrize("h_qk", [1, 2])
def test_grouped_heads_equal_repeated_q_and_k(h_qk):
    inp = workloads.make_general(n=3, t=3, hv=4, h_qk=h_qk, k=16, v=16, num_slots=20,
                                 state_dtype=torch.float32, seed=22)
    pool, o = _general(inp)
    rep = 4 // h_qk
    pool2, o2 = _general(inp, accepted=inp.accepted)  # same call, to show it is deterministic
    q = inp.q.repeat_interleave(rep, dim=1)
    k = inp.k.repeat_interleave(rep, dim=1)
    ref = _pool64(inp.pool)
    o_ref = oracle.step(ref, inp.slot_table, q, k, inp.v, inp.a, inp.b, accepted=inp.accepted)
    assert np.array_equal(pool, ref) and np.array_equal(o, o_ref)
    assert np.array_equal(pool2, pool) and np.array_equal(o2, o)
    # a wrong head map (h % H instead of h / (HV / H)) would differ
    q_bad = inp.q.repeat(1, rep, 1)
    if h_qk > 1:
        o_bad = oracle.step(_pool64(inp.pool), inp.slot_table, q_bad, inp.k.repeat(1, rep, 1), inp.v, inp.a,
                            inp.b, accepted=inp.accepted)
        assert not np.allclose(o_bad, o)


def test_gate_scale_closed_forms():
    """exp(-s softplus(a + d)) = (1 + e^(a+d))^(-s).  s = 1, d = 0 is the plain
    gate to the bit; s = 2 equals the plain gate at a' = log((1 + e^(a+d))^2 - 1)."""
    inp = workloads.make_general(n=3, t=2, hv=2, k=16, v=16, num_slots=12, state_dtype=torch.float32,
                                 seed=23)
    zero_log, zero_bias = torch.zeros(2), torch.zeros(2, 16)
    p1, o1 = _general(inp, a_log=zero_log, dt_bias=zero_bias)
    p0, o0 = _general(inp)
    assert np.array_equal(p1, p0) and np.array_equal(o1, o0)
    d = torch.linspace(-1.0, 1.0, 32, dtype=torch.float64).reshape(2, 16)
    p2, o2 = _general(inp, a_log=torch.full((2,), np.log(2.0), dtype=torch.float64), dt_bias=d)
    x = inp.a.double() + d[None]
    a_eq = torch.log(torch.square(1.0 + torch.exp(x)) - 1.0)
    ref = _pool64(inp.pool)
    o_ref = oracle.step(ref, inp.slot_table, inp.q, inp.k, inp.v, a_eq, inp.b, accepted=inp.accepted)
    np.testing.assert_allclose(o2, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(p2, ref, rtol=0, atol=2e-7)  # fp32 pool: at most an ulp of rounding apart


def test_varlen_equals_each_request_alone():
    lens = [3, 0, 1, 5, 2]
    inp = workloads.make_general(n=5, t_lens=lens, num_cols=6, hv=2, k=16, v=16, num_slots=40,
                                 state_dtype=torch.float16, seed=24, reset_p=0.4)
    pool, o = _general(inp)
    ref = _pool64(inp.pool)
    cu = inp.cu_seqlens.long()
    for r, tr in enumerate(lens):
        if tr == 0:
            continue
        sl = slice(int(cu[r]), int(cu[r + 1]))
        init = inp.slot_table[r:r + 1, int(inp.accepted[r]) - 1]
        o_r = oracle.spec_verify(ref, init, inp.slot_table[r:r + 1, :tr], inp.q[sl][None], inp.k[sl][None],
                                 inp.v[sl][None], inp.a[sl][None], inp.b[sl][None],
                                 reset=None if inp.reset is None else inp.reset[r:r + 1])
        assert np.array_equal(o[sl], o_r[0])
    assert np.array_equal(pool, ref)


def test_padding_request_touches_nothing():
    inp = workloads.make_general(n=6, t=3, hv=2, k=16, v=16, num_slots=30, state_dtype=torch.float32,
                                 seed=25, pad_p=0.5)
    pad = (inp.slot_table < 0).all(dim=1)
    assert 0 < int(pad.sum()) < 6
    before = _pool64(inp.pool)
    pool, o = _general(inp)
    o = o.reshape(6, 3, 2, 16)
    assert (o[pad.numpy()] == 0).all() and (o[~pad.numpy()] != 0).any()
    # the padded requests' inputs do not matter
    q2 = inp.q.clone().reshape(6, 3, 2, 16)
    q2[pad] = 7.0
    ref = _pool64(inp.pool)
    o_ref = oracle.step(ref, inp.slot_table, q2.reshape(18, 2, 16), inp.k, inp.v, inp.a, inp.b,
                        accepted=inp.accepted)
    assert np.array_equal(pool, ref) and np.array_equal(o.reshape(18, 2, 16), o_ref)
    # slots of padded rows are all -1, so nothing outside the real rows' slots changed
    real = inp.slot_table[~pad].reshape(-1)
    real = real[real >= 0].long().numpy()
    untouched = np.setdiff1d(np.arange(30), real)
    assert np.array_equal(pool[untouched], before[untouched])


def test_dropped_snapshot_is_not_stored():
    inp = workloads.make_general(n=4, t=4, hv=2, k=16, v=16, num_slots=24, state_dtype=torch.float16,
                                 seed=26)
    full_pool, full_o = _general(inp)
    table = inp.slot_table.clone()
    c0 = inp.accepted.long() - 1
    # drop one snapshot column that is not the initial one, per request
    drop_col = (c0 + 1) % 4
    dropped = table[torch.arange(4), drop_col].clone()
    table[torch.arange(4), drop_col] = -1
    pool = _pool64(inp.pool)
    o = oracle.step(pool, table, inp.q, inp.k, inp.v, inp.a, inp.b, accepted=inp.accepted)
    assert np.array_equal(o, full_o)  # the recurrence does not depend on what is kept
    before = _pool64(inp.pool)
    for r in range(4):
        s = int(dropped[r])
        assert np.array_equal(pool[s], before[s])          # not stored
        assert not np.array_equal(full_pool[s], before[s])  # the full run stored it
    keep = np.setdiff1d(np.arange(24), dropped.numpy())
    assert np.array_equal(pool[keep], full_pool[keep])


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_in_place_step_is_decode_on_the_accepted_slot(state_dtype):
    inp = workloads.make_general(n=6, num_cols=3, hv=2, k=16, v=32, num_slots=30, state_dtype=state_dtype,
                                 seed=27, in_place=True, reset_p=0.3)
    pool, o = _general(inp)
    ref = _pool64(inp.pool)
    slots = inp.slot_table[torch.arange(6), inp.accepted.long() - 1]
    o_ref = oracle.decode_step(ref, slots, inp.q, inp.k, inp.v, inp.a, inp.b, reset=inp.reset)
    assert np.array_equal(pool, ref) and np.array_equal(o, o_ref)


def test_general_layout_errors():
    inp = workloads.make_general(n=2, t=2, num_cols=2, hv=2, k=16, v=16, num_slots=10,
                                 state_dtype=torch.float32, seed=28)
    with pytest.raises(ValueError):
        _general(inp, accepted=torch.tensor([3, 1], dtype=torch.int32))   # column 2 of 2
    with pytest.raises(ValueError):
        _general(inp, accepted=torch.tensor([0, 1], dtype=torch.int32))   # column -1
    bad = inp.slot_table.clone()
    bad[0, 1] = 10
    with pytest.raises(ValueError):
        oracle.step(_pool64(inp.pool), bad, inp.q, inp.k, inp.v, inp.a, inp.b, accepted=inp.accepted)
