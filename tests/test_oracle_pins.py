"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks one oracle function against a hand-derived golden value, a
brute-force loop on tiny inputs, a closed form, an invariant, or a library
routine that the oracle does not use. A plausible mistake (a dropped term, a
wrong sign or index, a transposed operand) fails at least one of them; the
mutation test at the end plants such mistakes and checks that they are caught.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as oracle
import moe_synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


# ---------------------------------------------------------------- routing

def test_route_softmax_golden():
    c = GOLD["route_softmax"]
    l = np.array(c["logits"], np.float32)
    r = oracle.route(None, np.zeros((4, 1)), np.array(c["bias"], np.float32), c["k"],
                     "softmax", True, 1.0, logits32=l)
    assert r["idx"].tolist() == c["idx"]
    np.testing.assert_allclose(r["gate"], c["gate"], rtol=0, atol=1e-7)
    assert r["cnt"].tolist() == c["cnt"]
    assert r["off"].tolist() == c["off"]
    assert r["perm"].tolist() == c["perm"]
    assert r["inv"].tolist() == c["inv"]


def test_route_sigmoid_golden():
    c = GOLD["route_sigmoid"]
    l = np.array(c["logits"], np.float32)
    r = oracle.route(None, np.zeros((4, 1)), np.array(c["bias"], np.float32), c["k"],
                     "sigmoid", True, c["scale"], logits32=l)
    assert r["idx"].tolist() == c["idx"]
    np.testing.assert_allclose(r["gate"], c["gate"], rtol=0, atol=1e-7)


def _brute_topk(key_row, k):
    """Pick the largest remaining key k times; the lowest index wins a tie."""
    left = list(range(len(key_row)))
    out = []
    for _ in range(k):
        best = left[0]
        for e in left[1:]:
            if key_row[e] > key_row[best]:
                best = e
        out.append(best)
        left.remove(best)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_select_experts_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 17, 9, 3
    l = (rng.integers(-3, 4, size=(T, E)) * 0.5).astype(np.float32)   # many exact ties
    b = (rng.integers(-1, 2, size=E) * 0.5).astype(np.float32)
    idx = oracle.select_experts(l, b, k)
    key = l + b
    for t in range(T):
        assert idx[t].tolist() == _brute_topk([float(v) for v in key[t]], k)


def test_bias_steers_selection_only():
    l = np.array([[1.0, 0.0, -1.0]], np.float32)
    b = np.array([0.0, 0.0, 5.0], np.float32)
    r = oracle.route(None, np.zeros((3, 1)), b, 2, "softmax", True, 1.0, logits32=l)
    assert r["idx"].tolist() == [[2, 0]]
    e = [math.exp(-1.0), math.exp(1.0)]
    np.testing.assert_allclose(r["gate"][0], [e[0] / sum(e), e[1] / sum(e)], rtol=1e-12)


def test_softmax_gates_brute_force():
    rng = np.random.default_rng(3)
    T, E, k = 5, 7, 3
    l = rng.standard_normal((T, E))
    idx = oracle.select_experts(l.astype(np.float32), np.zeros(E, np.float32), k)
    g_r = oracle.gates_softmax(l, idx, renorm=True)
    g_a = oracle.gates_softmax(l, idx, renorm=False)
    for t in range(T):
        sel = [math.exp(l[t, e]) for e in idx[t]]
        full = sum(math.exp(v) for v in l[t])
        for j, e in enumerate(idx[t]):
            assert abs(g_r[t, j] - sel[j] / sum(sel)) < 1e-14
            assert abs(g_a[t, j] - math.exp(l[t, e]) / full) < 1e-14
    np.testing.assert_allclose(g_r.sum(1), 1.0, rtol=1e-14)


def test_sigmoid_gates_brute_force():
    rng = np.random.default_rng(4)
    T, E, k, lam = 4, 6, 2, 2.5
    l = rng.standard_normal((T, E)) * 3
    idx = oracle.select_experts(l.astype(np.float32), np.zeros(E, np.float32), k)
    g = oracle.gates_sigmoid(l, idx, lam, renorm=True)
    for t in range(T):
        s = [1.0 / (1.0 + math.exp(-l[t, e])) for e in idx[t]]
        for j in range(k):
            assert abs(g[t, j] - lam * s[j] / sum(s)) < 1e-13
    np.testing.assert_allclose(g.sum(1), lam, rtol=1e-14)


# ------------------------------------------------------------ permutation

@pytest.mark.parametrize("seed", range(5))
def test_permutation_brute_force_and_invariants(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 13, 6, 3
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    cnt = oracle.expert_counts(idx, E)
    off = oracle.expert_offsets(cnt)
    perm, inv = oracle.stable_permutation(idx)
    # brute force: walk experts in order, then assignments in order
    flat = idx.ravel().tolist()
    want = [a for e in range(E) for a in range(T * k) if flat[a] == e]
    assert perm.tolist() == want
    assert [flat.count(e) for e in range(E)] == cnt.tolist()
    assert cnt.sum() == T * k                       # dropless
    assert np.all(np.diff(off) >= 0) and off[0] == 0 and off[-1] == T * k
    for p in range(T * k):
        assert inv[perm[p]] == p
        e = flat[perm[p]]
        assert off[e] <= p < off[e + 1]
    for t in range(T):
        assert len(set(idx[t].tolist())) == k       # k distinct experts per token
    X = rng.standard_normal((T, 5))
    Xs = oracle.permute_rows(X, perm, k)
    back = oracle.unpermute_rows(Xs, inv)
    assert np.array_equal(back, X[np.arange(T * k) // k])   # bit-exact identity


# ----------------------------------------------------------------- FFN

def _ffn_loops(x, Wg, Wu, Wd):
    """SwiGLU by explicit loops (brute force)."""
    T, d = len(x), len(x[0])
    f = len(Wg)
    out = []
    for t in range(T):
        h = []
        for i in range(f):
            u = sum(x[t][c] * Wg[i][c] for c in range(d))
            v = sum(x[t][c] * Wu[i][c] for c in range(d))
            h.append(u / (1.0 + math.exp(-u)) * v)
        out.append([sum(h[i] * Wd[c][i] for i in range(f)) for c in range(d)])
    return np.array(out)


def test_expert_ffn_brute_force():
    rng = np.random.default_rng(5)
    T, d, f = 3, 6, 4
    x, Wg, Wu, Wd = (rng.standard_normal(s) for s in ((T, d), (f, d), (f, d), (d, f)))
    _, _, _, o = oracle.expert_ffn(x, Wg, Wu, Wd)
    np.testing.assert_allclose(o, _ffn_loops(x.tolist(), Wg.tolist(), Wu.tolist(), Wd.tolist()),
                               rtol=1e-12, atol=1e-14)


def test_ffn_golden_forward_backward():
    c = GOLD["ffn_single_expert"]
    x = np.array(c["x"])
    args = (x, np.zeros((1, 2)), np.zeros(1, np.float32), np.array(c["Wg"]), np.array(c["Wu"]),
            np.array(c["Wd"]))
    kw = dict(k=1, router="softmax", renorm=True, scale=1.0)
    y = oracle.forward(*args, **kw)["y"]
    np.testing.assert_allclose(y, c["y"], rtol=1e-15)
    g = oracle.backward(*args, np.array(c["dy"]), **kw)
    for n in ("dx", "dWg", "dWu", "dWd"):
        np.testing.assert_allclose(g[n], c[n], rtol=1e-14, err_msg=n)
    assert np.all(g["dWr"] == 0)


def _layer(seed, T=8, d=6, E=4, f=5, S=0, wr=1.0):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((T, d)), Wr=wr * rng.standard_normal((E, d)),
                b=np.zeros(E, np.float32), Wg=rng.standard_normal((E + S, f, d)) / 2,
                Wu=rng.standard_normal((E + S, f, d)) / 2, Wd=rng.standard_normal((E + S, d, f)) / 2)


def test_single_expert_equals_one_ffn_exactly():
    L = _layer(6, E=1)
    y = oracle.forward(L["x"], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"], 1, "softmax", True, 1.0)["y"]
    want = _ffn_loops(L["x"].tolist(), L["Wg"][0].tolist(), L["Wu"][0].tolist(), L["Wd"][0].tolist())
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-14)


def test_k_equals_E_identical_experts_uniform_gates_is_dense_ffn():
    L = _layer(7, E=5)
    Wg = np.repeat(L["Wg"][:1], 5, 0)
    Wu = np.repeat(L["Wu"][:1], 5, 0)
    Wd = np.repeat(L["Wd"][:1], 5, 0)
    Wr = np.zeros_like(L["Wr"])                    # all logits 0: softmax gates 1/E
    y = oracle.forward(L["x"], Wr, L["b"], Wg, Wu, Wd, 5, "softmax", True, 1.0)["y"]
    want = _ffn_loops(L["x"].tolist(), Wg[0].tolist(), Wu[0].tolist(), Wd[0].tolist())
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-13)


def test_forward_brute_force_with_shared_expert():
    L = _layer(8, S=1)
    k, lam = 2, 2.5
    r = oracle.forward(L["x"], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"], k, "sigmoid", True, lam,
                       n_shared=1)
    E = L["Wr"].shape[0]
    for t in range(L["x"].shape[0]):
        xl = [L["x"][t].tolist()]
        l = [sum(L["x"][t][c] * L["Wr"][e][c] for c in range(6)) for e in range(E)]
        sel = _brute_topk(l, k)
        s = [1 / (1 + math.exp(-l[e])) for e in sel]
        want = _ffn_loops(xl, L["Wg"][E].tolist(), L["Wu"][E].tolist(), L["Wd"][E].tolist())[0]
        for j, e in enumerate(sel):
            want = want + lam * s[j] / sum(s) * _ffn_loops(xl, L["Wg"][e].tolist(), L["Wu"][e].tolist(),
                                                           L["Wd"][e].tolist())[0]
        np.testing.assert_allclose(r["y"][t], want, rtol=1e-12, atol=1e-13)


def test_ffn_matches_torch_float64():
    """The expert FFN is a textbook SwiGLU: cross-check with torch's own ops in float64."""
    L = _layer(9)
    _, _, _, o = oracle.expert_ffn(L["x"], L["Wg"][0], L["Wu"][0], L["Wd"][0])
    X, Wg, Wu, Wd = (torch.from_numpy(a) for a in (L["x"], L["Wg"][0], L["Wu"][0], L["Wd"][0]))
    want = torch.nn.functional.linear(torch.nn.functional.silu(X @ Wg.T) * (X @ Wu.T), Wd)
    np.testing.assert_allclose(o, want.numpy(), rtol=1e-12, atol=1e-14)


def test_token_permutation_equivariance_and_duplicates():
    L = _layer(10, S=1)
    x = L["x"].copy()
    x[5] = x[2]
    kw = dict(k=2, router="softmax", renorm=True, scale=1.0, n_shared=1)
    y = oracle.forward(x, L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"], **kw)["y"]
    assert np.array_equal(y[5], y[2])
    p = np.random.default_rng(0).permutation(x.shape[0])
    y2 = oracle.forward(x[p], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"], **kw)["y"]
    np.testing.assert_allclose(y2, y[p], rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("mx", [False, True])
def test_token_subset_rows_equal_full_batch(mx):
    """y and dx rows of a few tokens, evaluated alone (only the experts they reach), match the rows
    of the whole batch: every operand of a token's y and dx (x, dY, h, du, dv; MXFP8 blocks along
    each row) belongs to that token. Full-size GPU checks sample tokens on this basis."""
    L = _layer(12, T=96, d=64, E=6, f=64, S=1, wr=0.5)
    kw = dict(k=2, router="sigmoid", renorm=True, scale=2.5, n_shared=1, mx=mx)
    dy = np.random.default_rng(13).standard_normal(L["x"].shape)
    args = (L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"])
    full_y = oracle.forward(L["x"], *args, **kw)["y"]
    full = oracle.backward(L["x"], *args, dy, **kw)
    toks = np.array([3, 50, 95])
    reached = sorted(set(full["idx"][toks].ravel().tolist()) | {6})
    sub_y = oracle.forward(L["x"][toks], *args, **kw)["y"]
    sub = oracle.backward(L["x"][toks], *args, dy[toks], experts=reached, **kw)
    # equal up to the summation order of the library matmul over a different number of rows
    np.testing.assert_allclose(sub_y, full_y[toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(sub["dx"], full["dx"][toks], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------- backward

def _selection_margin(x, Wr, b, k):
    key = oracle.selection_keys(oracle.router_logits(x, Wr).astype(np.float32), b)
    s = -np.sort(-key, axis=1)
    return float(np.min(s[:, k - 1] - s[:, k])) if key.shape[1] > k else np.inf


@pytest.mark.parametrize("router,renorm,S", [("softmax", True, 0), ("softmax", False, 1),
                                             ("sigmoid", True, 1), ("sigmoid", False, 0)])
def test_backward_matches_central_differences(router, renorm, S):
    L = _layer(11 + S, T=5, d=4, E=4, f=3, S=S)
    k, lam = 2, (2.5 if router == "sigmoid" else 1.0)
    dy = np.random.default_rng(99).standard_normal(L["x"].shape)
    assert _selection_margin(L["x"], L["Wr"], L["b"], k) > 1e-3
    kw = dict(k=k, router=router, renorm=renorm, scale=lam, n_shared=S)
    g = oracle.backward(L["x"], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"], dy, **kw)
    names = {"x": "dx", "Wr": "dWr", "Wg": "dWg", "Wu": "dWu", "Wd": "dWd"}
    h = 1e-6
    for name, gname in names.items():
        P = L[name]
        fd = np.zeros_like(P)
        for ix in itertools.product(*(range(n) for n in P.shape)):
            old = P[ix]
            P[ix] = old + h
            lp = oracle.loss(L["x"], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"], dy, **kw)
            P[ix] = old - h
            lm = oracle.loss(L["x"], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"], dy, **kw)
            P[ix] = old
            fd[ix] = (lp - lm) / (2 * h)
        err = np.linalg.norm(g[gname] - fd) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-6, (name, err)


def test_backward_linear_in_dy():
    L = _layer(13, S=1)
    kw = dict(k=2, router="sigmoid", renorm=True, scale=2.5, n_shared=1)
    rng = np.random.default_rng(1)
    d1, d2 = rng.standard_normal(L["x"].shape), rng.standard_normal(L["x"].shape)
    args = (L["x"], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"])
    g1 = oracle.backward(*args, d1, **kw)
    g2 = oracle.backward(*args, d2, **kw)
    g3 = oracle.backward(*args, 2 * d1 - 3 * d2, **kw)
    for n in ("dx", "dWr", "dWg", "dWu", "dWd"):
        np.testing.assert_allclose(g3[n], 2 * g1[n] - 3 * g2[n], rtol=1e-10, atol=1e-12)


# -------------------------------------------------------- chunking, ring

def test_chunked_equals_unchunked():
    L = _layer(14, T=11, S=1)
    dy = np.random.default_rng(2).standard_normal(L["x"].shape)
    kw = dict(k=2, router="sigmoid", renorm=True, scale=2.5, n_shared=1)
    args = (L["x"], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"], dy)
    c = oracle.chunked_forward_backward(*args, chunk=4, **kw)
    y = oracle.forward(*args[:6], **kw)["y"]
    g = oracle.backward(*args, **kw)
    np.testing.assert_allclose(c["y"], y, rtol=1e-13, atol=1e-14)
    for n in ("dx", "dWr", "dWg", "dWu", "dWd"):
        np.testing.assert_allclose(c[n], g[n], rtol=1e-12, atol=1e-13)
    assert oracle.chunk_bounds(8192, 2368) == [(0, 2368), (2368, 4736), (4736, 7104), (7104, 8192)]


@pytest.mark.parametrize("n,R", [(4, 1), (4, 2), (4, 3), (4, 4), (4, 9), (7, 3)])
def test_ring_schedule_matches_slot_simulation(n, R):
    ev = oracle.ring_schedule(n, R)
    slot = {}
    for phase, c, s, rec in ev:
        if phase == "fwd":
            slot[s] = c
        else:
            assert rec == (slot.get(s) != c)
            slot[s] = c
    assert sum(e[3] for e in ev) == max(0, n - R)
    assert [e[1] for e in ev if e[0] == "bwd"] == list(reversed(range(n)))


# ------------------------------------------------------------------- MX

def test_e4m3_decode_golden():
    c = GOLD["e4m3_decode"]
    got = oracle.e4m3_decode(np.array(c["codes"], np.uint8))
    for g, w in zip(got, c["values"]):
        assert g == w and math.copysign(1, g) == math.copysign(1, w)
    assert math.isnan(oracle.e4m3_decode(np.array([0x7F], np.uint8))[0])


def test_mx_blocks_golden():
    for case in GOLD["mx_blocks"]["cases"]:
        blk = np.full(32, case["fill"])
        blk[:len(case["head"])] = case["head"]
        codes, scales = oracle.mx_quantize(blk[None, :], axis=1)
        assert int(scales[0, 0]) == case["scale"], case["why"]
        n = len(case["head"])
        assert codes[0, :n].tolist() == case["codes_head"], case["why"]
        assert all(int(c) == case["fill_code"] for c in codes[0, n:])


def test_e4m3_matches_torch_cast_in_range():
    """In range, E4M3 rounding is the library's float8_e4m3fn cast (ties to even)."""
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1, 30, 200)])
    v = v[np.abs(v) <= 448]
    v = np.concatenate([v, oracle.e4m3_decode(np.arange(256, dtype=np.uint8))])
    v = v[~np.isnan(v)]
    mid = (oracle.e4m3_decode(np.arange(1, 126, dtype=np.uint8)) +
           oracle.e4m3_decode(np.arange(2, 127, dtype=np.uint8))) / 2      # exact halfway points
    v = np.concatenate([v, mid, -mid])
    want = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn)
    got_codes = oracle.e4m3_encode(oracle.e4m3_round(v.astype(np.float32).astype(np.float64)))
    assert np.array_equal(got_codes, want.view(torch.uint8).numpy())


def test_mx_roundtrip_exact_for_representable_and_bounded_error():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 256, size=(3, 64)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38                 # no NaN
    vals = oracle.e4m3_decode(codes) * 2.0 ** 5
    vals[:, ::32] = np.sign(vals[:, ::32] + 0.5) * 448 * 2.0 ** 5 / 1.75 * 1.75  # amax sets X = 5
    c2, s2 = oracle.mx_quantize(vals, axis=1)
    assert np.array_equal(oracle.mx_dequantize(c2, s2, axis=1), vals)
    a = rng.standard_normal((4, 96)) * 3
    q = oracle.mx_fake_quant(a, axis=1)
    blk_max = np.repeat(np.abs(a).reshape(4, 3, 32).max(-1), 32, axis=1)
    assert np.all(np.abs(q - a) <= blk_max * 2.0 ** -3 + 1e-300)      # half a quantum of the top binade, x2


def test_mx_quantize_axis0_is_transpose_of_axis1():
    a = np.random.default_rng(2).standard_normal((64, 40))
    c0, s0 = oracle.mx_quantize(a, axis=0)
    c1, s1 = oracle.mx_quantize(a.T, axis=1)
    assert np.array_equal(c0, c1.T) and np.array_equal(s0, s1.T)


# ------------------------------------------------------- input generator

def test_zipf_targets_feasible():
    for T, k, E, s in ((2048, 6, 64, 1.0), (8192, 8, 256, 1.2)):
        t = moe_synth.zipf_targets(T, k, E, s)
        assert abs(sum(t) - T * k) < 1e-6 and max(t) <= T + 1e-9
        assert all(t[i] >= t[i + 1] - 1e-9 for i in range(E - 1))


# --------------------------------------------------------- mutation check

def test_planted_mistakes_are_caught(monkeypatch):
    """Plant plausible mistakes in the oracle (on the CPU) and check a pin fails for each."""
    c = GOLD["ffn_single_expert"]
    args = (np.array(c["x"]), np.zeros((1, 2)), np.zeros(1, np.float32), np.array(c["Wg"]),
            np.array(c["Wu"]), np.array(c["Wd"]))
    kw = dict(k=1, router="softmax", renorm=True, scale=1.0)

    def golden_ok():
        g = oracle.backward(*args, np.array(c["dy"]), **kw)
        y = oracle.forward(*args, **kw)["y"]
        return (np.allclose(y, c["y"], rtol=1e-12) and
                all(np.allclose(g[n], c[n], rtol=1e-12) for n in ("dx", "dWg", "dWu", "dWd")))

    assert golden_ok()
    good_grad = oracle.silu_grad
    monkeypatch.setattr(oracle, "silu_grad", lambda z: oracle.sigmoid(z))   # dropped term
    assert not golden_ok()
    monkeypatch.setattr(oracle, "silu_grad", good_grad)
    good_ffn = oracle.expert_ffn

    def swapped(xr, Wg_e, Wu_e, Wd_e):                                       # gate/up swapped
        return good_ffn(xr, Wu_e, Wg_e, Wd_e)
    monkeypatch.setattr(oracle, "expert_ffn", swapped)
    assert not golden_ok()
    monkeypatch.setattr(oracle, "expert_ffn", good_ffn)
    cr = GOLD["route_softmax"]
    good_sel = oracle.select_experts
    monkeypatch.setattr(oracle, "select_experts",
                        lambda l, b, k: np.argsort(-(np.asarray(l, np.float32) + b), axis=1)[:, ::-1][:, :k]
                        .astype(np.int32))                                   # wrong order
    r = oracle.route(None, np.zeros((4, 1)), np.array(cr["bias"], np.float32), 2, "softmax", True, 1.0,
                     logits32=np.array(cr["logits"], np.float32))
    assert r["idx"].tolist() != cr["idx"]
    monkeypatch.setattr(oracle, "select_experts", good_sel)


# ------------------------------------------------------------ MX layer math

def _mx_layer(seed=20, T=9, d=64, f=96, E=3):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((T, d)), Wr=rng.standard_normal((E, d)), b=np.zeros(E, np.float32),
                Wg=rng.standard_normal((E + 1, f, d)) / 8, Wu=rng.standard_normal((E + 1, f, d)) / 8,
                Wd=rng.standard_normal((E + 1, d, f)) / 8, dy=rng.standard_normal((T, d)))


MXKW = dict(k=2, router="sigmoid", renorm=True, scale=2.5, n_shared=1)


def test_mx_paths_reduce_to_exact_with_identity_quantisers(monkeypatch):
    L = _mx_layer()
    args = (L["x"], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"])
    y = oracle.forward(*args, **MXKW)["y"]
    g = oracle.backward(*args, L["dy"], **MXKW)
    monkeypatch.setattr(oracle, "mx_fake_quant", lambda a, axis=-1: np.asarray(a, np.float64))
    ym = oracle.forward(*args, mx=True, **MXKW)["y"]
    gm = oracle.backward(*args, L["dy"], mx=True, **MXKW)
    np.testing.assert_allclose(ym, y, rtol=1e-12, atol=1e-12)
    for n in ("dx", "dWg", "dWu", "dWd", "dWr"):
        np.testing.assert_allclose(gm[n], g[n], rtol=1e-11, atol=1e-12, err_msg=n)


def test_mx_quantisation_axes(monkeypatch):
    """Each operand is quantised along its GEMM's K (d != f, so a transposed operand shows)."""
    L = _mx_layer(T=9, d=64, f=96)
    calls = []
    real = oracle.mx_fake_quant

    def spy(a, axis=-1):
        a = np.asarray(a, np.float64)
        calls.append((a.shape, axis % a.ndim))
        return real(a, axis)
    monkeypatch.setattr(oracle, "mx_fake_quant", spy)
    args = (L["x"], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"])
    oracle.forward(*args, mx=True, **MXKW)
    fwd = set(calls)
    assert ((9, 64), 1) in fwd                      # x along d
    assert ((96, 64), 1) in fwd                     # Wg, Wu [f, d] along d
    assert ((64, 96), 1) in fwd                     # Wd [d, f] along f
    assert all(s[1] == 96 and ax == 1 for s, ax in fwd if s[0] not in (9, 96, 64))   # h rows along f
    calls.clear()
    oracle.backward(*args, L["dy"], mx=True, **MXKW)
    bwd = set(calls)
    assert ((64, 96), 0) in bwd                     # Wd along d (its axis 0) for dy . Wd
    assert ((96, 64), 0) in bwd                     # Wg, Wu along f (axis 0) for du . Wg
    assert ((96, 64), 1) in bwd                     # and along d in the recomputed forward
    token_calls = [(s, ax) for s, ax in bwd if ax == 0 and s[0] % 32 == 0 and s not in ((64, 96), (96, 64))]
    assert token_calls and all(s[1] in (64, 96) for s, _ in token_calls)   # token-axis blocks, zero padded


def test_token_axis_quantiser_brute_force():
    rng = np.random.default_rng(3)
    a = rng.standard_normal((45, 7)) * np.exp(rng.standard_normal((45, 7)))
    q = oracle.mx_fake_quant_tokens(a)
    assert q.shape == a.shape
    for c in range(7):
        for b0 in (0, 32):
            blk = a[b0:b0 + 32, c]
            full = np.zeros(32)
            full[:len(blk)] = blk
            want = oracle.mx_fake_quant(full[None, :], axis=1)[0][:len(blk)]
            assert np.array_equal(q[b0:b0 + 32, c], want)


def test_backward_expert_filter_matches_full_backward():
    L = _mx_layer(T=11)
    args = (L["x"], L["Wr"], L["b"], L["Wg"], L["Wu"], L["Wd"], L["dy"])
    for mx in (False, True):
        full = oracle.backward(*args, mx=mx, **MXKW)
        part = oracle.backward(*args, mx=mx, experts=[1, 3], **MXKW)      # expert 3 is the shared one
        assert set(part["dWg"]) == {1, 3}
        for e in (1, 3):
            for n in ("dWg", "dWu", "dWd"):
                np.testing.assert_array_equal(part[n][e], full[n][e])


# ------------------------------------------------------------ the checkers

def test_rel_frobenius_hand_cases():
    # ||(0, 1)|| / ||(3, 4)|| = 1 / 5
    assert oracle.rel_frobenius([[3.0, 5.0]], [[3.0, 4.0]]) == pytest.approx(0.2, abs=1e-15)
    # every element counts, squared: diff (-3, 0, 0, 1) against ref norm 5 -> sqrt(10) / 5
    assert oracle.rel_frobenius([[0.0, 0.0], [0.0, 5.0]], [[3.0, 0.0], [0.0, 4.0]]) == \
        pytest.approx(math.sqrt(10) / 5, abs=1e-15)
    # relative to the reference, not to the argument: swapping them changes the value
    assert oracle.rel_frobenius([[3.0, 4.0]], [[3.0, 5.0]]) == pytest.approx(1 / math.sqrt(34), abs=1e-15)
    # a sign flip is an error of twice the norm
    assert oracle.rel_frobenius([[-1.0, -2.0]], [[1.0, 2.0]]) == pytest.approx(2.0, abs=1e-15)
    assert oracle.rel_frobenius(np.zeros((2, 3)), np.zeros((2, 3))) == 0.0


def test_routing_check_margins_and_exceptions():
    from routing_checks import key_margins, routing_exceptions
    # keys of token 0: 3, 2, 1.5, 0 (k = 2: gaps among the 3 largest are 1 and 0.5); token 1 has a tie
    logits = np.array([[3.0, 2.0, 1.5, 0.0], [1.0, 1.0, 0.0, -1.0]], np.float32)
    bias = np.zeros(4, np.float32)
    assert key_margins(logits, bias, 2).tolist() == [0.5, 0.0]
    # the bias enters the keys: +1 on expert 3 makes token 0's keys 3, 2, 1.5, 1 -> gaps 1, 0.5
    assert key_margins(logits, np.array([0, 0, 0, 1], np.float32), 2).tolist() == [0.5, 0.0]
    # routing_exceptions computes the oracle's logits from x and Wr: with Wr = I the logits are x
    x = logits.astype(np.float64)
    Wr = np.eye(4)
    ok = routing_exceptions(np.array([[0, 1], [0, 1]]), logits, x, Wr, bias, 2)
    assert ok["exceptions"] == 0 and ok["near_ties"] == 1 and ok["logit_err"] == 0.0
    # a wrong expert on the well-separated token is an exception; on the tied token it is not
    bad = routing_exceptions(np.array([[0, 2], [1, 0]]), logits, x, Wr, bias, 2)
    assert bad["exceptions"] == 1 and bad["near_tie_disagreements"] == 1
    # a large measured logit error turns token 0 into a near-tie as well (4 x 0.2 > 0.5)
    noisy = routing_exceptions(np.array([[0, 2], [0, 1]]), logits + np.float32(0.2), x, Wr, bias, 2)
    assert noisy["near_ties"] == 2 and noisy["exceptions"] == 0
