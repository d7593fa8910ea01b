"""Pins for the CPU oracle: each test checks it against something other than
itself -- a closed form, a special case with a known answer, a library
routine, or an equivalence between two independently written code paths --
chosen so that a dropped term, a wrong sign, a transposed operand or a wrong
index makes at least one of them fail.

The rule being pinned is the standard gated delta rule (the decode rule of the
fused sigmoid-gating delta-rule kernel named in the vLLM PR #52191 summary,
section 实现拆解 items 3-4) and the ReplaySSM checkpoint + input-buffer mode
(AREX ReplaySSM article, section "缓存输入而非状态").
"""
import math

import numpy as np
import pytest
import torch

import oracle
from hybrid_ssm_gated_gb300 import workload as wl

EPS = 1e-6  # l2norm epsilon of the rule


# ----------------------------------------------------------------- formats


def _special_f32():
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 70000.0, 6.0e-8, 5.96e-8, 2.98e-8,
            1e-40, -1e-45, 3.3895313892515355e38, 3.4e38, float("inf"), float("-inf")]
    # exact ties for bf16: 1 + 2^-8 (halfway between 1 and 1 + 2^-7) and its odd neighbour
    vals += [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11]
    return np.array(vals, dtype=np.float32)


def _random_f32(n=1 << 18, seed=0):
    r = np.random.default_rng(seed)
    mant = r.uniform(1.0, 2.0, n)
    expo = r.integers(-140, 128, n)
    sign = r.choice([-1.0, 1.0], n)
    x = (sign * mant * np.exp2(expo.astype(np.float64))).astype(np.float32)
    return np.concatenate([x, _special_f32()])


def test_round_bf16_matches_torch():
    x = _random_f32()
    ours = oracle.round_to(x.astype(np.float64), "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_f16_matches_torch():
    x = _random_f32(seed=1)
    x = x[np.abs(x) < 1e6]  # keep most values in or near the binary16 range
    x = np.concatenate([x, _special_f32()])
    ours = oracle.round_to(x.astype(np.float64), "f16")
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours.view(np.uint16), ref)


def test_round_f32_matches_numpy():
    r = np.random.default_rng(2)
    x = r.standard_normal(1 << 16) * np.exp2(r.integers(-140, 120, 1 << 16))
    ours = oracle.round_to(x, "f32")
    assert np.array_equal(ours, x.astype(np.float32))


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_load_every_bit_pattern(dt):
    bits = np.arange(1 << 16, dtype=np.uint16)
    tt = torch.bfloat16 if dt == "bf16" else torch.float16
    ref = torch.from_numpy(bits.view(np.int16)).view(tt).to(torch.float64).numpy()
    arr = bits if dt == "bf16" else bits.view(np.float16)
    ours = oracle.load(arr, dt)
    finite = np.isfinite(ref) | np.isinf(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.all(np.isnan(ours[~finite]))


# ----------------------------------------------------------------- gating


def test_gating_closed_forms():
    # softplus(0) = ln 2, so alpha = 2^-exp(A_log): A_log = 0 -> 1/2, A_log = ln 3 -> 1/8
    al, be = oracle.gating(0.0, 0.25, -0.25, 0.0)
    assert al == pytest.approx(0.5, rel=1e-15) and be == 0.5
    al, _ = oracle.gating(math.log(3.0), 0.0, 0.0, 0.0)
    assert al == pytest.approx(0.125, rel=1e-14)
    # sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4
    assert oracle.gating(0.0, 0.0, 0.0, math.log(3.0))[1] == pytest.approx(0.75, rel=1e-15)
    assert oracle.gating(0.0, 0.0, 0.0, -math.log(3.0))[1] == pytest.approx(0.25, rel=1e-15)
    # limits: beta(+inf) = 1, beta(-inf) = 0, alpha(a=+inf) = 0, alpha(A_log=-inf) = 1
    assert oracle.gating(0.0, 0.0, 0.0, math.inf)[1] == 1.0
    assert oracle.gating(0.0, 0.0, 0.0, -math.inf)[1] == 0.0
    assert oracle.gating(0.0, 0.0, math.inf, 0.0)[0] == 0.0
    assert oracle.gating(-math.inf, 0.3, 1.7, 0.0)[0] == 1.0
    # below the cut-over softplus is ln(1 + e^x), however large x: ln 15 -> ln 16, ln(2^26 - 1) -> 26 ln 2
    assert oracle.gating(0.0, 0.0, math.log(15.0), 0.0)[0] == pytest.approx(1 / 16, rel=1e-14)
    assert oracle.gating(0.0, 0.0, math.log(2.0 ** 26 - 1), 0.0)[0] == pytest.approx(2.0 ** -26, rel=1e-12)
    # above the softplus cut-over the argument passes through: exp(A_log)=1/25, x=25 -> e^-1
    al, _ = oracle.gating(math.log(1 / 25), 5.0, 20.0, 0.0)
    assert al == pytest.approx(math.exp(-1.0), rel=1e-14)
    # far below it softplus(x) ~ e^x: alpha ~ exp(-e^A * e^x)
    al, _ = oracle.gating(1.0, 0.0, -30.0, 0.0)
    assert al == pytest.approx(math.exp(-math.e * math.exp(-30.0)), rel=1e-15)
    # decay is monotone: larger a -> smaller alpha
    alphas = [oracle.gating(0.7, 0.1, x, 0.0)[0] for x in np.linspace(-5, 5, 21)]
    assert all(x > y for x, y in zip(alphas, alphas[1:]))


def test_l2norm_direction_and_scale():
    r = np.random.default_rng(3)
    x = r.standard_normal(128) * 10
    y = oracle.l2norm(x)
    assert np.linalg.norm(y) == pytest.approx(1.0, abs=1e-8)
    assert np.allclose(y * np.linalg.norm(x), x, rtol=1e-8)
    assert np.allclose(oracle.l2norm(7.5 * x), y, rtol=1e-9)
    e = np.zeros(16)
    e[3] = 1.0
    assert oracle.l2norm(e, 0.25)[3] == pytest.approx(0.25 / math.sqrt(1 + EPS), rel=1e-15)
    assert oracle.l2norm(np.zeros(8)).tolist() == [0.0] * 8


# ----------------------------------------------------------------- decode


def _basis(n, i):
    e = np.zeros(n)
    e[i] = 1.0
    return e


def _batch(B, Hk, Hv, dk, dv, seed):
    r = np.random.default_rng(seed)
    return dict(q=r.standard_normal((B, Hk, dk)), k=r.standard_normal((B, Hk, dk)),
                v=r.standard_normal((B, Hv, dv)), a=r.standard_normal((B, Hv)),
                b=r.standard_normal((B, Hv)))


def test_pure_decay_closed_form():
    """beta = 0 (b = -inf) leaves only the decay: S_t = 2^-t S_0 when alpha = 1/2
    (A_log = 0, a = -dt_bias), and the readout of q = e_m is column m of S_t."""
    B, Hk, Hv, dk, dv = 2, 1, 2, 8, 4
    r = np.random.default_rng(4)
    pool = r.standard_normal((3, Hv, dv, dk))
    pool0 = pool.copy()
    slots = np.array([2, 0], dtype=np.int32)
    dt_bias = np.array([0.5, -0.75], dtype=np.float32)
    A_log = np.zeros(Hv, dtype=np.float32)
    for t in range(1, 6):
        m = (3 * t) % dk
        q = np.broadcast_to(_basis(dk, m), (B, Hk, dk)).astype(np.float32)
        k = r.standard_normal((B, Hk, dk)).astype(np.float32)
        v = r.standard_normal((B, Hv, dv)).astype(np.float32)
        a = np.broadcast_to(-dt_bias, (B, Hv)).astype(np.float32)
        b = np.full((B, Hv), -np.inf, dtype=np.float32)
        out, bad = oracle.decode_step(pool, "f64", slots, q, k, v, a, b, "f32", A_log, dt_bias)
        assert bad == 0
        scale = 2.0 ** -t
        for bi, s in enumerate(slots):
            assert np.allclose(pool[s], scale * pool0[s], rtol=1e-14, atol=0)
            expect = scale * pool0[s][:, :, m] / math.sqrt(1 + EPS) / math.sqrt(dk)
            assert np.allclose(out[bi], expect, rtol=1e-12, atol=1e-300)
    assert np.array_equal(pool[1], pool0[1])  # a slot nobody uses stays untouched


def test_exact_retrieval_orthogonal_keys():
    """alpha = 1, beta = 1, S_0 = 0: writing value v under key e_i and reading
    with q = e_i returns v / ((1 + eps) sqrt(dk))."""
    dk, dv = 8, 6
    S = np.zeros((dv, dk))
    r = np.random.default_rng(5)
    keys = [3, 0, 7, 5]
    vals = [r.standard_normal(dv) for _ in keys]
    for t, (i, v) in enumerate(zip(keys, vals)):
        for s in range(t + 1):  # read every key written so far, including this step's
            S_try = S.copy()
            out = oracle.decode_head(S_try, "f64", _basis(dk, keys[s]), _basis(dk, i), v, "f64", 1.0, 1.0)
            expect = vals[s] / ((1 + EPS) * math.sqrt(dk))
            assert np.allclose(out, expect, rtol=1e-12, atol=1e-15)
        oracle.decode_head(S, "f64", _basis(dk, i), _basis(dk, i), v, "f64", 1.0, 1.0)
    # overwriting key 3 replaces its value (up to the eps of the normalisation)
    v_new = r.standard_normal(dv)
    out = oracle.decode_head(S, "f64", _basis(dk, 3), _basis(dk, 3), v_new, "f64", 1.0, 1.0)
    assert np.allclose(out * math.sqrt(dk), v_new, rtol=1e-5, atol=1e-5)


def test_delta_rule_overwrite_with_decay():
    """beta = 1 and any alpha: the updated state maps the (unit) key exactly to v,
    because the correction subtracts the *decayed* prediction alpha S^T k."""
    dk, dv = 16, 12
    r = np.random.default_rng(6)
    for alpha in (1.0, 0.8, 0.3, 1e-3):
        S = r.standard_normal((dv, dk))
        k = r.standard_normal(dk)
        v = r.standard_normal(dv)
        oracle.decode_head(S, "f64", r.standard_normal(dk), k, v, "f64", alpha, 1.0)
        kn = k / np.linalg.norm(k)
        assert np.allclose(S @ kn, v, rtol=0, atol=1e-5 * (1 + np.abs(v).max()))


def test_scalar_recurrence_geometric_series():
    """dk = dv = 1, k = q = 1, constant gates: s_t = r s_{t-1} + c is a
    geometric series with r = alpha (1 - beta/(1+eps)), c = beta v / sqrt(1+eps)."""
    alpha, beta, v, s0 = 0.9, 0.35, 2.5, -1.25
    S = np.array([[s0]])
    kh = 1.0 / math.sqrt(1 + EPS)
    rr = alpha * (1 - beta * kh * kh)
    cc = beta * v * kh
    for n in range(1, 40):
        out = oracle.decode_head(S, "f64", [1.0], [1.0], [v], "f64", alpha, beta)
        s_n = rr ** n * s0 + cc * (1 - rr ** n) / (1 - rr)
        assert S[0, 0] == pytest.approx(s_n, rel=1e-12)
        assert out[0] == pytest.approx(s_n * kh, rel=1e-12)


def test_matrix_form_tiny():
    """Brute force in matrix form: S' = alpha (I - beta k k^T) S + beta k v^T,
    o = S'^T q, with S dk x dv (the storage holds S^T)."""
    dk, dv = 5, 3
    r = np.random.default_rng(7)
    for trial in range(20):
        St = r.standard_normal((dv, dk))
        q, k, v = r.standard_normal(dk), r.standard_normal(dk), r.standard_normal(dv)
        alpha, beta = r.uniform(0.05, 1.0), r.uniform(0.0, 1.0)
        S = St.T.copy()
        kn = k / math.sqrt(k @ k + EPS)
        qn = q / math.sqrt(q @ q + EPS) / math.sqrt(dk)
        S_new = alpha * (np.eye(dk) - beta * np.outer(kn, kn)) @ S + beta * np.outer(kn, v)
        out = oracle.decode_head(St, "f64", q, k, v, "f64", alpha, beta)
        assert np.allclose(St.T, S_new, rtol=1e-12, atol=1e-14)
        assert np.allclose(out, S_new.T @ qn, rtol=1e-12, atol=1e-14)


def test_gqa_equals_mha_with_repeated_key_heads():
    """Value head h reads key head h // (Hv/Hk): GQA with keys [k0, k1] equals
    MHA with keys [k0, k0, k1, k1]."""
    B, Hk, Hv, dk, dv = 3, 2, 4, 8, 8
    x = _batch(B, Hk, Hv, dk, dv, 8)
    A_log = np.linspace(0.1, 1.9, Hv).astype(np.float32)
    dt_bias = np.linspace(-0.9, 0.9, Hv).astype(np.float32)
    pool = np.random.default_rng(9).standard_normal((B, Hv, dv, dk)).astype(np.float32)
    slots = np.arange(B, dtype=np.int32)
    p1, p2 = pool.copy(), pool.copy()
    o1, _ = oracle.decode_step(p1, "f32", slots, x["q"], x["k"], x["v"], x["a"], x["b"], "f64", A_log, dt_bias)
    rep = lambda t: np.repeat(t, Hv // Hk, axis=1)
    o2, _ = oracle.decode_step(p2, "f32", slots, rep(x["q"]), rep(x["k"]), x["v"], x["a"], x["b"], "f64",
                               A_log, dt_bias)
    assert np.array_equal(o1, o2) and np.array_equal(p1, p2)
    # and the mapping is not h % Hk: swapping the key heads changes heads 0 and 1
    p3 = pool.copy()
    o3, _ = oracle.decode_step(p3, "f32", slots, x["q"][:, ::-1].copy(), x["k"][:, ::-1].copy(), x["v"],
                               x["a"], x["b"], "f64", A_log, dt_bias)
    assert not np.allclose(o3[:, 0], o1[:, 0])


def test_slots_padding_and_out_of_range():
    B, Hk, Hv, dk, dv = 4, 1, 2, 4, 4
    x = _batch(B, Hk, Hv, dk, dv, 10)
    pool = np.random.default_rng(11).standard_normal((2, Hv, dv, dk)).astype(np.float32)
    pool0 = pool.copy()
    slots = np.array([-1, 2, 1, -3], dtype=np.int32)
    out, bad = oracle.decode_step(pool, "f32", slots, x["q"], x["k"], x["v"], x["a"], x["b"], "f64",
                                  np.zeros(Hv, np.float32), np.zeros(Hv, np.float32))
    assert bad == Hv  # the out-of-range sequence, counted per (sequence, head) unit; padding is not an error
    assert np.all(out[0] == 0) and np.all(out[1] == 0) and np.any(out[2] != 0) and np.all(out[3] == 0)
    assert np.array_equal(pool[0], pool0[0]) and not np.array_equal(pool[1], pool0[1])


@pytest.mark.parametrize("sdt", ["bf16", "f16", "f32"])
def test_narrow_state_rounds_once_at_write_back(sdt):
    """The stored state is the rounded fp64 result; the output comes from the
    unrounded state (it matches the fp64-state run exactly)."""
    dk, dv = 16, 8
    r = np.random.default_rng(12)
    S_narrow = oracle.round_to(r.standard_normal((dv, dk)) * 0.1, sdt)
    S_wide = oracle.load(S_narrow, sdt).copy()
    q, k, v = r.standard_normal(dk), r.standard_normal(dk), r.standard_normal(dv)
    o1 = oracle.decode_head(S_narrow, sdt, q, k, v, "f64", 0.7, 0.4)
    o2 = oracle.decode_head(S_wide, "f64", q, k, v, "f64", 0.7, 0.4)
    assert np.array_equal(o1, o2)
    assert np.array_equal(S_narrow.view(np.uint8), oracle.round_to(S_wide, sdt).view(np.uint8))


def test_batch_step_matches_per_head_calls():
    """The batched driver (slots, gating, GQA offsets, threads) equals per-head calls."""
    B, Hk, Hv, dk, dv = 4, 2, 4, 16, 8
    x = _batch(B, Hk, Hv, dk, dv, 13)
    A_log, dt_bias = np.float32([0.1, 0.5, 1.0, 1.9]), np.float32([-0.5, 0.0, 0.5, 0.9])
    pool = np.random.default_rng(14).standard_normal((6, Hv, dv, dk)).astype(np.float32)
    slots = np.array([4, 0, 5, 2], dtype=np.int32)
    p1 = pool.copy()
    o1, _ = oracle.decode_step(p1, "f32", slots, x["q"], x["k"], x["v"], x["a"], x["b"], "f64", A_log,
                               dt_bias, nthreads=3)
    for bi in range(B):
        for h in range(Hv):
            kh = h // (Hv // Hk)
            al, be = oracle.gating(A_log[h], dt_bias[h], x["a"][bi, h], x["b"][bi, h])
            S = pool[slots[bi], h].copy()
            o = oracle.decode_head(S, "f32", x["q"][bi, kh], x["k"][bi, kh], x["v"][bi, h], "f64", al, be)
            assert np.array_equal(o, o1[bi, h])
            assert np.array_equal(S, p1[slots[bi], h])


# ----------------------------------------------------------------- ReplaySSM


def _tokens(n, dk, dv, seed, T=1):
    r = np.random.default_rng(seed)
    return [dict(q=r.standard_normal((T, dk)), k=r.standard_normal((T, dk)), v=r.standard_normal((T, dv)),
                 a=r.standard_normal(T), b=r.standard_normal(T)) for _ in range(n)]


def _decode_run(S, toks, A_log, dt_bias, sdt="f64"):
    outs = []
    for t in toks:
        for j in range(t["q"].shape[0]):
            al, be = oracle.gating(A_log, dt_bias, t["a"][j], t["b"][j])
            outs.append(oracle.decode_head(S, sdt, t["q"][j], t["k"][j], t["v"][j], "f64", al, be))
    return np.array(outs)


def test_replay_equals_per_step_updates_fp64():
    """With an unrounded checkpoint, L replay steps plus folds are the same
    computation as per-step decode updates."""
    dk, dv, L = 8, 6, 4
    r = np.random.default_rng(15)
    S0 = r.standard_normal((dv, dk)) * 0.1
    toks = _tokens(3 * L + 1, dk, dv, 16)
    head = oracle.ReplayHead(S0, "f64", "f64", L)
    outs = np.array([head.window(**t, A_log=0.4, dt_bias=0.2)[0] for t in toks])
    S = S0.copy()
    ref = _decode_run(S, toks, 0.4, 0.2)
    assert np.allclose(outs, ref, rtol=1e-11, atol=1e-13)
    head.flush(force=True)
    assert np.allclose(head.S0, S, rtol=1e-11, atol=1e-13)
    assert head.count == 0 and head.pos == len(toks) and head.ckpt_pos == len(toks)


@pytest.mark.parametrize("sdt", ["bf16", "f16", "f32"])
def test_replay_rounds_only_at_folds(sdt):
    """A narrow checkpoint is rounded only when the buffer is folded: the first
    L outputs are exact fp64 evolutions of S0; the fold at step L+1 stores
    round(S_L) and the run continues from it."""
    dk, dv, L = 8, 8, 4
    r = np.random.default_rng(17)
    S0 = oracle.round_to(r.standard_normal((dv, dk)) * 0.1, sdt)
    toks = _tokens(2 * L + 2, dk, dv, 18)
    head = oracle.ReplayHead(S0, sdt, "f64", L)
    outs = np.array([head.window(**t, A_log=0.3, dt_bias=-0.1)[0] for t in toks])
    S = oracle.load(S0, sdt).copy()
    ref1 = _decode_run(S, toks[:L], 0.3, -0.1)
    S = oracle.load(oracle.round_to(S, sdt), sdt).copy()  # fold 1 (at token L+1)
    ref2 = _decode_run(S, toks[L:2 * L], 0.3, -0.1)
    S = oracle.load(oracle.round_to(S, sdt), sdt).copy()  # fold 2 (at token 2L+1)
    ref3 = _decode_run(S, toks[2 * L:], 0.3, -0.1)
    assert np.allclose(outs, np.concatenate([ref1, ref2, ref3]), rtol=1e-11, atol=1e-13)
    assert head.ckpt_pos == 2 * L and head.count == 2


def test_window_equals_sequential_steps():
    """Output j of a T-token window reads the state after window tokens <= j."""
    dk, dv, L, T = 8, 4, 8, 4
    r = np.random.default_rng(19)
    S0 = r.standard_normal((dv, dk)) * 0.1
    pre = _tokens(3, dk, dv, 20)
    win = _tokens(1, dk, dv, 21, T=T)[0]
    h1 = oracle.ReplayHead(S0, "f64", "f64", L)
    h2 = oracle.ReplayHead(S0, "f64", "f64", L)
    for t in pre:
        h1.window(**t, A_log=1.0, dt_bias=0.0)
        h2.window(**t, A_log=1.0, dt_bias=0.0)
    o_win = h1.window(**win, A_log=1.0, dt_bias=0.0)
    o_seq = np.array([h2.window(q=win["q"][j:j + 1], k=win["k"][j:j + 1], v=win["v"][j:j + 1],
                                a=win["a"][j:j + 1], b=win["b"][j:j + 1], A_log=1.0, dt_bias=0.0)[0]
                      for j in range(T)])
    assert np.allclose(o_win, o_seq, rtol=1e-12, atol=1e-14)
    assert h1.pos == h2.pos == 3 + T


@pytest.mark.parametrize("acc", [0, 1, 2, 3])
def test_rollback_equals_run_on_kept_tokens(acc):
    """After a T=4 window with `acc` accepted drafts and a rollback, the next
    output equals a run that only ever saw the 1 + acc kept tokens."""
    dk, dv, L, T = 8, 6, 8, 4
    r = np.random.default_rng(22)
    S0 = r.standard_normal((dv, dk)) * 0.1
    pre = _tokens(2, dk, dv, 23)
    win = _tokens(1, dk, dv, 24, T=T)[0]
    nxt = _tokens(1, dk, dv, 25)[0]
    h = oracle.ReplayHead(S0, "f64", "f64", L)
    for t in pre:
        h.window(**t, A_log=0.5, dt_bias=0.5)
    h.window(**win, A_log=0.5, dt_bias=0.5)
    h.rollback(T, acc)
    assert h.count == 2 + 1 + acc and h.pos == 3 + acc
    o = h.window(**nxt, A_log=0.5, dt_bias=0.5)[0]
    kept = {k: v[: 1 + acc] for k, v in win.items()}
    S = S0.copy()
    ref = _decode_run(S, pre + [kept, nxt], 0.5, 0.5)[-1]
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-14)


def test_fold_rule_and_pointer_bookkeeping():
    """Fold exactly when an append would overflow the L-entry buffer; rollback
    only moves the pointer back."""
    dk, dv, L = 4, 4, 4
    h = oracle.ReplayHead(np.zeros((dv, dk)), "f64", "f64", L, pos=10)
    one = _tokens(1, dk, dv, 26)[0]
    for i in range(3):
        h.window(**one, A_log=0.0, dt_bias=0.0)
    assert (h.count, h.pos, h.ckpt_pos) == (3, 13, 10)
    two = _tokens(1, dk, dv, 27, T=2)[0]
    h.window(**two, A_log=0.0, dt_bias=0.0)  # 3 + 2 > 4: fold first
    assert (h.count, h.pos, h.ckpt_pos) == (2, 15, 13)
    h.rollback(2, 0)
    assert (h.count, h.pos, h.ckpt_pos) == (1, 14, 13)
    h.window(**two, A_log=0.0, dt_bias=0.0)
    h.window(**one, A_log=0.0, dt_bias=0.0)
    assert (h.count, h.pos, h.ckpt_pos) == (4, 17, 13)  # full, not folded yet
    h.flush(force=False)  # a full buffer folds even without force
    assert (h.count, h.pos, h.ckpt_pos) == (0, 17, 17)
    h.window(**one, A_log=0.0, dt_bias=0.0)
    h.flush(force=False)  # not full: nothing happens
    assert (h.count, h.ckpt_pos) == (1, 17)
    h.flush(force=True)
    assert (h.count, h.ckpt_pos) == (0, 18)
    with pytest.raises(ValueError):
        h.rollback(4, 4)  # accepted must be < T
    h.window(**one, A_log=0.0, dt_bias=0.0)
    with pytest.raises(ValueError):
        h.rollback(3, 0)  # two tokens back would pass the checkpoint, whose entries are folded away
    assert (h.count, h.pos, h.ckpt_pos) == (1, 19, 18)
    with pytest.raises(ValueError):
        h.window(**_tokens(1, dk, dv, 28, T=5)[0], A_log=0.0, dt_bias=0.0)  # T > L


def test_replay_buffer_holds_raw_inputs():
    """Only state-building inputs are buffered: raw k and v bits as given, and
    the gates; q is never stored."""
    dk, dv, L = 8, 8, 4
    w = wl.Workload("t", B=1, Hk=1, Hv=1, dk=dk, dv=dv, steps=1, in_dtype="bf16", T=3)
    x = wl.step_inputs(w, 0)
    h = oracle.ReplayHead(np.zeros((dv, dk)), "f64", "bf16", L)
    h.window(q=x["q"][0, :, 0], k=x["k"][0, :, 0], v=x["v"][0, :, 0], a=wl.values(x["a"][0, :, 0], "bf16"),
             b=wl.values(x["b"][0, :, 0], "bf16"), A_log=0.2, dt_bias=0.1)
    assert np.array_equal(h.ek[:3], x["k"][0, :, 0]) and np.array_equal(h.ev[:3], x["v"][0, :, 0])
    for j in range(3):
        al, be = oracle.gating(0.2, 0.1, wl.values(x["a"][0, j, 0], "bf16"), wl.values(x["b"][0, j, 0], "bf16"))
        assert h.ea[j] == al and h.eb[j] == be


def test_tiny_workload_regression_fixture():
    """The oracle still produces the stored outputs of the tiny workload
    (fixture written by tests/golden/make_tiny_golden.py from the oracle)."""
    import json
    import os

    from tests.golden.make_tiny_golden import compute

    with open(os.path.join(os.path.dirname(__file__), "golden", "tiny_decode.json")) as f:
        doc = json.load(f)
    outs, pool = compute()
    # libm's exp/log1p may differ by an ulp between machines: compare to 1e-12
    close = lambda x, y: np.allclose(x, np.array(y), rtol=1e-12, atol=1e-15)
    assert close(outs[0, 0, 0], doc["out_step0_b0_h0"])
    assert close(outs[7, 1, 3], doc["out_step7_b1_h3"])
    assert close(pool[1, 2, 5].astype(np.float64), doc["final_state_slot1_h2_col5"])
    assert close(np.abs(outs).sum(), doc["sum_abs_out"])
