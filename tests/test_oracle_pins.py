"""Pins for the fp64 oracle: each test checks it against something other than
itself -- a second algorithm, an invariant of the delta rule, a closed form, a
library routine, or finite differences.  CPU only."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

RNG = np.random.default_rng(1234)


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _core_inputs(rng, T, hk, hv, dk, dv, g_scale=0.3):
    qh = _unit_rows(rng.standard_normal((T, hk, dk))) * dk ** -0.5
    kh = _unit_rows(rng.standard_normal((T, hk, dk)))
    v = rng.standard_normal((T, hv, dv))
    g = -rng.uniform(0.0, g_scale, size=(T, hv))
    beta = rng.uniform(0.05, 0.95, size=(T, hv))
    return qh, kh, v, g, beta


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# --------------------------------------------------------------- pin 1: chunked form
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
@pytest.mark.parametrize("chunk", [4, 16, 64])
def test_chunked_form_matches_recurrence(T, chunk):
    rng = np.random.default_rng(T * 100 + chunk)
    hk, hv, dk, dv = 1, 2, 8, 8
    qh, kh, v, g, beta = _core_inputs(rng, T, hk, hv, dk, dv)
    cu = np.array([0, T], dtype=np.int32)
    S0 = rng.standard_normal((1, hv, dv, dk))
    o1, s1 = oracle.delta_rule(qh, kh, v, g, beta, cu, S0)
    o2, s2 = oracle.chunked_delta_rule(qh, kh, v, g, beta, cu, S0, chunk)
    assert _rel(o2, o1) < 1e-12
    assert _rel(s2, s1) < 1e-12


@pytest.mark.parametrize("chunk", [4, 16, 64])
def test_chunked_form_matches_recurrence_varlen(chunk):
    rng = np.random.default_rng(7 + chunk)
    hk, hv, dk, dv = 2, 6, 8, 4
    cu = np.array([0, 37, 37, 137, 200, 201], dtype=np.int32)  # includes an empty sequence
    T = int(cu[-1])
    qh, kh, v, g, beta = _core_inputs(rng, T, hk, hv, dk, dv, g_scale=2.0)
    S0 = rng.standard_normal((len(cu) - 1, hv, dv, dk))
    o1, s1 = oracle.delta_rule(qh, kh, v, g, beta, cu, S0)
    o2, s2 = oracle.chunked_delta_rule(qh, kh, v, g, beta, cu, S0, chunk)
    assert _rel(o2, o1) < 1e-12
    assert _rel(s2, s1) < 1e-12
    # the empty sequence passes its state through unchanged
    np.testing.assert_array_equal(s1[1], S0[1])


# --------------------------------------------------------------- pin 2: memory invariant
@pytest.mark.parametrize("n", [1, 5, 16])
def test_delta_rule_memory_invariant(n):
    """g = 0, beta = 1, orthonormal keys, S0 = 0: the state stores v_i at k_i."""
    rng = np.random.default_rng(n)
    dk, dv = 16, 8
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :n].T.copy()                      # n orthonormal rows
    vals = rng.standard_normal((n, dv))
    kh = keys.reshape(n, 1, dk)
    qh = rng.standard_normal((n, 1, dk))
    v = vals.reshape(n, 1, dv)
    g = np.zeros((n, 1))
    beta = np.ones((n, 1))
    cu = np.array([0, n], dtype=np.int32)
    _, S = oracle.delta_rule(qh, kh, v, g, beta, cu)
    recalled = S[0, 0] @ keys.T                    # [dv, n]
    np.testing.assert_allclose(recalled.T, vals, rtol=0, atol=1e-12)


def test_delta_rule_overwrites_same_key():
    """beta = 1, g = 0: writing the same key twice keeps only the last value."""
    dk, dv = 8, 4
    rng = np.random.default_rng(3)
    k = _unit_rows(rng.standard_normal(dk))
    v1, v2 = rng.standard_normal(dv), rng.standard_normal(dv)
    kh = np.stack([k, k]).reshape(2, 1, dk)
    v = np.stack([v1, v2]).reshape(2, 1, dv)
    _, S = oracle.delta_rule(kh, kh, v, np.zeros((2, 1)), np.ones((2, 1)),
                             np.array([0, 2], dtype=np.int32))
    np.testing.assert_allclose(S[0, 0] @ k, v2, atol=1e-13)


# --------------------------------------------------------------- pin 3: pure decay
def test_pure_decay():
    rng = np.random.default_rng(5)
    T, hk, hv, dk, dv = 50, 1, 3, 8, 8
    qh, kh, v, g, _ = _core_inputs(rng, T, hk, hv, dk, dv, g_scale=0.5)
    beta = np.zeros((T, hv))
    S0 = rng.standard_normal((1, hv, dv, dk))
    cu = np.array([0, T], dtype=np.int32)
    o, S = oracle.delta_rule(qh, kh, v, g, beta, cu, S0)
    for h in range(hv):
        gam = np.cumsum(g[:, h])
        np.testing.assert_allclose(S[0, h], S0[0, h] * np.exp(gam[-1]), rtol=1e-13, atol=0)
        want = np.exp(gam)[:, None] * (qh[:, 0] @ S0[0, h].T)
        np.testing.assert_allclose(o[:, h], want, rtol=1e-12, atol=1e-300)


# --------------------------------------------------------------- closed forms
def test_single_token_closed_form():
    """T = 1 from S0 = 0: S = beta v k^T and o = beta (k . q) v."""
    rng = np.random.default_rng(9)
    qh, kh, v, g, beta = _core_inputs(rng, 1, 1, 2, 8, 8)
    o, S = oracle.delta_rule(qh, kh, v, g, beta, np.array([0, 1], dtype=np.int32))
    for h in range(2):
        np.testing.assert_allclose(S[0, h], beta[0, h] * np.outer(v[0, h], kh[0, 0]), atol=1e-15)
        np.testing.assert_allclose(o[0, h], beta[0, h] * (kh[0, 0] @ qh[0, 0]) * v[0, h],
                                   atol=1e-15)


def test_gates_against_library():
    rng = np.random.default_rng(11)
    a, b = rng.standard_normal((40, 3)) * 4, rng.standard_normal((40, 3)) * 4
    A_log = np.log(rng.uniform(1, 16, size=3))
    dt_bias = rng.standard_normal(3)
    g, beta = oracle.gates(a, b, A_log, dt_bias)
    ta = torch.from_numpy(a)
    want_g = -torch.exp(torch.from_numpy(A_log)) * F.softplus(ta + torch.from_numpy(dt_bias))
    np.testing.assert_allclose(g, want_g.numpy(), rtol=1e-14)
    np.testing.assert_allclose(beta, torch.sigmoid(torch.from_numpy(b)).numpy(), rtol=1e-14)


def test_conv_against_library():
    """Causal depthwise conv = torch grouped conv1d with left padding K-1,
    restarted per sequence; with a conv cache = the cache prepended."""
    rng = np.random.default_rng(13)
    C, K = 6, 4
    cu = np.array([0, 2, 9, 30], dtype=np.int32)
    x = rng.standard_normal((30, C))
    w = rng.uniform(-0.5, 0.5, size=(C, K))
    cs = rng.standard_normal((3, C, K - 1))
    for cache in (None, cs):
        pre, out, cso = oracle.conv_silu(x, w, cu, cache)
        wt = torch.from_numpy(w)[:, None, :]
        for n in range(3):
            s, e = cu[n], cu[n + 1]
            seq = torch.from_numpy(x[s:e].T)[None]                     # [1, C, L]
            if cache is None:
                ref = F.conv1d(seq, wt, padding=K - 1, groups=C)[0, :, : e - s]
                hist = np.concatenate([np.zeros((C, K - 1)), x[s:e].T], axis=1)
            else:
                full = torch.cat([torch.from_numpy(cache[n])[None], seq], dim=2)
                ref = F.conv1d(full, wt, groups=C)[0]
                hist = np.concatenate([cache[n], x[s:e].T], axis=1)
            np.testing.assert_allclose(pre[s:e], ref.T.numpy(), rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(out[s:e], F.silu(ref.T).numpy(), rtol=1e-13, atol=1e-14)
            np.testing.assert_array_equal(cso[n], hist[:, -(K - 1):])


@pytest.mark.parametrize("gate,fn", [("silu", F.silu), ("sigmoid", torch.sigmoid)])
def test_gated_norm_against_library(gate, fn):
    rng = np.random.default_rng(17)
    o = rng.standard_normal((20, 3, 16))
    z = rng.standard_normal((20, 3, 16))
    w = rng.normal(0, 0.02, size=16)
    y, rstd = oracle.gated_rmsnorm(o, z, w, 1e-6, gate)
    to = torch.from_numpy(o)
    ref = F.rms_norm(to, (16,), weight=1 + torch.from_numpy(w), eps=1e-6) * fn(
        torch.from_numpy(z))
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-14)
    # the backward against torch autograd of the same library expression
    dy = rng.standard_normal(o.shape)
    to.requires_grad_(True)
    tz = torch.from_numpy(z).requires_grad_(True)
    tw = torch.from_numpy(w).requires_grad_(True)
    (F.rms_norm(to, (16,), weight=1 + tw, eps=1e-6) * fn(tz) * torch.from_numpy(dy)).sum().backward()
    do, dz, dw = oracle.gated_rmsnorm_bwd(o, z, w, dy, 1e-6, gate)
    np.testing.assert_allclose(do, to.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dz, tz.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dw, tw.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_l2norm_against_library():
    """x / sqrt(|x|^2 + eps) vs torch's normalize (x / |x|): relative gap <= eps/(2|x|^2)."""
    rng = np.random.default_rng(19)
    x = rng.standard_normal((30, 4, 32))
    out = oracle.l2norm(x, 1e-6, 32 ** -0.5)
    ref = F.normalize(torch.from_numpy(x), dim=-1).numpy() * 32 ** -0.5
    bound = 1e-6 / (2 * np.min(np.sum(x * x, -1))) + 1e-14
    assert np.max(np.abs(out - ref) / np.abs(ref)) <= bound


# --------------------------------------------------------------- structural extras
def _layer(rng, lens, hk, hv, d, K=4, dt_bias=0.0, cache=False, s0=False):
    T = sum(lens)
    C = 2 * hk * d + hv * d
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = len(lens)
    return dict(
        x=rng.standard_normal((T, C)), conv_w=rng.uniform(-0.5, 0.5, size=(C, K)),
        a=rng.standard_normal((T, hv)), b=rng.standard_normal((T, hv)),
        A_log=np.log(rng.uniform(1, 16, size=hv)), dt_bias=np.full(hv, dt_bias),
        z=rng.standard_normal((T, hv, d)), norm_w=rng.normal(0, 0.02, size=d), cu=cu,
        hk=hk, hv=hv, dk=d, dv=d,
        S0=rng.standard_normal((N, hv, d, d)) * 0.3 if s0 else None,
        conv_state=rng.standard_normal((N, C, K - 1)) if cache else None)


def test_varlen_equals_separate_runs():
    rng = np.random.default_rng(21)
    lens = [5, 70, 1, 33]
    p = _layer(rng, lens, 1, 2, 8, dt_bias=-4.0, cache=True, s0=True)
    f = oracle.forward(**p)
    cu = p["cu"]
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        q = dict(p, x=p["x"][s:e], a=p["a"][s:e], b=p["b"][s:e], z=p["z"][s:e],
                 cu=np.array([0, e - s], dtype=np.int32), S0=p["S0"][n:n + 1],
                 conv_state=p["conv_state"][n:n + 1])
        fn = oracle.forward(**q)
        np.testing.assert_array_equal(fn["y"], f["y"][s:e])
        np.testing.assert_array_equal(fn["S_final"][0], f["S_final"][n])
        np.testing.assert_array_equal(fn["conv_state_out"][0], f["conv_state_out"][n])


@pytest.mark.parametrize("split", [1, 2, 3, 17, 64, 99])
def test_split_with_handoff_equals_one_run(split):
    rng = np.random.default_rng(23 + split)
    p = _layer(rng, [100], 1, 3, 8, dt_bias=-5.0)
    f = oracle.forward(**p)
    first = dict(p, x=p["x"][:split], a=p["a"][:split], b=p["b"][:split], z=p["z"][:split],
                 cu=np.array([0, split], dtype=np.int32))
    f1 = oracle.forward(**first)
    second = dict(p, x=p["x"][split:], a=p["a"][split:], b=p["b"][split:], z=p["z"][split:],
                  cu=np.array([0, 100 - split], dtype=np.int32), S0=f1["S_final"],
                  conv_state=f1["conv_state_out"])
    f2 = oracle.forward(**second)
    np.testing.assert_allclose(np.concatenate([f1["y"], f2["y"]]), f["y"], rtol=1e-12,
                               atol=1e-13)
    np.testing.assert_allclose(f2["S_final"], f["S_final"], rtol=1e-12, atol=1e-13)


def test_gva_equals_explicit_repetition():
    rng = np.random.default_rng(29)
    T, dk, dv = 40, 8, 8
    qh, kh, v, g, beta = _core_inputs(rng, T, 2, 6, dk, dv)
    cu = np.array([0, 17, 40], dtype=np.int32)
    o, S = oracle.delta_rule(qh, kh, v, g, beta, cu)
    rep = lambda a: np.repeat(a, 3, axis=1)      # v-head h -> k-head h // 3
    o2, S2 = oracle.delta_rule(rep(qh), rep(kh), v, g, beta, cu)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(S, S2)


def test_decode_equals_last_step():
    rng = np.random.default_rng(31)
    p = _layer(rng, [30, 12], 1, 2, 8, dt_bias=-3.0)
    f = oracle.forward(**p)
    cu = p["cu"]
    # run all but the last token of each sequence, then one decode step each
    lens = np.diff(cu)
    head = [np.arange(cu[n], cu[n + 1] - 1) for n in range(2)]
    idx = np.concatenate(head)
    q = dict(p, x=p["x"][idx], a=p["a"][idx], b=p["b"][idx], z=p["z"][idx],
             cu=np.concatenate([[0], np.cumsum(lens - 1)]).astype(np.int32))
    fh = oracle.forward(**q)
    last = cu[1:] - 1
    y, o, S, cs = oracle.decode_step(p["x"][last], p["conv_w"], fh["conv_state_out"],
                                     p["a"][last], p["b"][last], p["A_log"], p["dt_bias"],
                                     p["z"][last], p["norm_w"], fh["S_final"], 1, 2, 8, 8)
    np.testing.assert_allclose(y, f["y"][last], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, f["S_final"], rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(cs, f["conv_state_out"])


def test_group_major_layout_keeps_each_group_contiguous():
    """Group-major x holds each k-head group's q, k and v heads as one contiguous
    block of (2 + G) d channels: that block alone, as an H_k = 1 problem (where
    the flat and group-major orders coincide), gives exactly the group's part of
    the whole problem -- outputs, final state, conv cache and every gradient."""
    rng = np.random.default_rng(61)
    hk, hv, d, G = 3, 6, 4, 2
    p = _layer(rng, [19, 8], hk, hv, d, dt_bias=-3.0, cache=True, s0=True)
    f = oracle.forward(**p, layout="group")
    dy = rng.standard_normal(f["y"].shape)
    dcso = rng.standard_normal(f["conv_state_out"].shape)
    r = oracle.backward(**p, dy=dy, layout="group", dconv_state_out=dcso)
    w = (2 + G) * d
    for kh in range(hk):
        ch, hs = slice(kh * w, (kh + 1) * w), slice(kh * G, (kh + 1) * G)
        q = dict(p, x=p["x"][:, ch], conv_w=p["conv_w"][ch], a=p["a"][:, hs], b=p["b"][:, hs],
                 A_log=p["A_log"][hs], dt_bias=p["dt_bias"][hs], z=p["z"][:, hs], hk=1, hv=G,
                 S0=p["S0"][:, hs], conv_state=p["conv_state"][:, ch])
        fg = oracle.forward(**q)
        np.testing.assert_allclose(fg["y"], f["y"][:, hs], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(fg["S_final"], f["S_final"][:, hs], rtol=1e-12, atol=1e-13)
        np.testing.assert_array_equal(fg["conv_state_out"], f["conv_state_out"][:, ch])
        rg = oracle.backward(**q, dy=dy[:, hs], dconv_state_out=dcso[:, ch])
        for k in ("dx", "dconv_state"):
            np.testing.assert_allclose(rg[k], r[k][:, ch], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(rg["dconv_w"], r["dconv_w"][ch], rtol=1e-11, atol=1e-12)
        for k in ("da", "db", "dz"):
            np.testing.assert_allclose(rg[k], r[k][:, hs], rtol=1e-11, atol=1e-12)
    # with a single group the two orders are the same order
    assert (oracle.group_major_order(1, 3, 4, 4) == np.arange(5 * 4)).all()


# --------------------------------------------------------------- pin 4: finite differences
def _loss(p, dy, dSf, dcso=None):
    f = oracle.forward(**p)
    L = float(np.sum(f["y"] * dy) + np.sum(f["S_final"] * dSf))
    if dcso is not None:
        L += float(np.sum(f["conv_state_out"] * dcso))
    return L


GRAD_OF = {"x": "dx", "conv_w": "dconv_w", "a": "da", "b": "db", "A_log": "dA_log",
           "dt_bias": "ddt_bias", "z": "dz", "norm_w": "dnorm_w", "S0": "dS0",
           "conv_state": "dconv_state"}


@pytest.mark.parametrize("d,hk,hv,dt_bias", [(4, 1, 2, -2.0), (8, 1, 2, 0.0), (8, 2, 4, -4.0)])
def test_backward_finite_differences(d, hk, hv, dt_bias):
    """Central differences (step 1e-6, fp64) along a random direction for every
    input agree with the hand-written reverse mode to 1e-6 relative."""
    rng = np.random.default_rng(37 + d + hv)
    p = _layer(rng, [23, 17], hk, hv, d, dt_bias=dt_bias, cache=True, s0=True)
    f = oracle.forward(**p)
    dy = rng.standard_normal(f["y"].shape)
    dSf = rng.standard_normal(f["S_final"].shape)
    gr = oracle.backward(**{k: v for k, v in p.items()}, dy=dy, dS_final=dSf)
    eps = 1e-6
    for name, gname in GRAD_OF.items():
        R = rng.standard_normal(np.shape(p[name]))
        pp = dict(p, **{name: p[name] + eps * R})
        pm = dict(p, **{name: p[name] - eps * R})
        fd = (_loss(pp, dy, dSf) - _loss(pm, dy, dSf)) / (2 * eps)
        an = float(np.sum(gr[gname] * R))
        assert abs(fd - an) <= 1e-6 * max(abs(an), 1e-3), (name, fd, an)


@pytest.mark.parametrize("gate,layout,lens", [("sigmoid", "flat", [23, 17]),
                                              ("silu", "group", [23, 2, 0, 9]),
                                              ("sigmoid", "group", [1, 30])])
def test_backward_finite_differences_variants(gate, layout, lens):
    """The same central differences for the sigmoid output gate, the group-major
    channel layout, and a loss that also weighs conv_state_out (the gradient a
    split sequence hands back), with sequences shorter than the conv window."""
    rng = np.random.default_rng(53 + len(lens))
    p = _layer(rng, lens, 2, 4, 4, dt_bias=-2.0, cache=True, s0=True)
    p.update(gate=gate, layout=layout)
    f = oracle.forward(**p)
    dy = rng.standard_normal(f["y"].shape)
    dSf = rng.standard_normal(f["S_final"].shape)
    dcso = rng.standard_normal(f["conv_state_out"].shape)
    gr = oracle.backward(**p, dy=dy, dS_final=dSf, dconv_state_out=dcso)
    eps = 1e-6
    for name, gname in GRAD_OF.items():
        R = rng.standard_normal(np.shape(p[name]))
        pp = dict(p, **{name: p[name] + eps * R})
        pm = dict(p, **{name: p[name] - eps * R})
        fd = (_loss(pp, dy, dSf, dcso) - _loss(pm, dy, dSf, dcso)) / (2 * eps)
        an = float(np.sum(gr[gname] * R))
        assert abs(fd - an) <= 1e-6 * max(abs(an), 1e-3), (name, fd, an)


def test_core_backward_finite_differences():
    """Same check on the delta-rule stage alone (q^, k^, v, g, beta, S0)."""
    rng = np.random.default_rng(41)
    T, hk, hv, dk, dv = 30, 1, 2, 6, 5
    qh, kh, v, g, beta = _core_inputs(rng, T, hk, hv, dk, dv, g_scale=0.4)
    cu = np.array([0, 11, 30], dtype=np.int32)
    S0 = rng.standard_normal((2, hv, dv, dk))
    do = rng.standard_normal((T, hv, dv))
    dSf = rng.standard_normal((2, hv, dv, dk))
    args = dict(qh=qh, kh=kh, v=v, g=g, beta=beta, S0=S0)

    def L(a):
        o, S = oracle.delta_rule(a["qh"], a["kh"], a["v"], a["g"], a["beta"], cu, a["S0"])
        return float(np.sum(o * do) + np.sum(S * dSf))

    dq, dkk, dvv, dg, dbeta, dS0 = oracle.delta_rule_bwd(qh, kh, v, g, beta, cu, do, S0, dSf)
    grads = dict(qh=dq, kh=dkk, v=dvv, g=dg, beta=dbeta, S0=dS0)
    for name in args:
        R = rng.standard_normal(args[name].shape)
        eps = 1e-6
        fd = (L(dict(args, **{name: args[name] + eps * R}))
              - L(dict(args, **{name: args[name] - eps * R}))) / (2 * eps)
        an = float(np.sum(grads[name] * R))
        assert abs(fd - an) <= 1e-6 * max(abs(an), 1e-3), (name, fd, an)


def test_backward_matches_autograd_elementwise():
    """Element-wise check of the reverse mode on a tiny case: torch autograd
    differentiates a plain fp64 torch transcription of the forward."""
    rng = np.random.default_rng(43)
    d, hk, hv = 4, 1, 2
    p = _layer(rng, [9, 6], hk, hv, d, dt_bias=-1.0, cache=True, s0=True)
    f = oracle.forward(**p)
    dy = rng.standard_normal(f["y"].shape)
    gr = oracle.backward(**p, dy=dy)
    t = {k: torch.tensor(p[k], requires_grad=True) for k in GRAD_OF}
    cu = p["cu"]
    K = 4
    ys = []
    for n in range(2):
        s, e = int(cu[n]), int(cu[n + 1])
        seq = torch.cat([t["conv_state"][n], t["x"][s:e].T], dim=1)[None]
        xc = F.silu(F.conv1d(seq, t["conv_w"][:, None, :], groups=seq.shape[1])[0].T)
        q = xc[:, :hk * d].reshape(-1, hk, d)
        k = xc[:, hk * d:2 * hk * d].reshape(-1, hk, d)
        v = xc[:, 2 * hk * d:].reshape(-1, hv, d)
        q = q / torch.sqrt((q * q).sum(-1, keepdim=True) + 1e-6) * d ** -0.5
        k = k / torch.sqrt((k * k).sum(-1, keepdim=True) + 1e-6)
        g = -torch.exp(t["A_log"]) * F.softplus(t["a"][s:e] + t["dt_bias"])
        beta = torch.sigmoid(t["b"][s:e])
        outs = []
        for h in range(hv):
            S = t["S0"][n, h]
            oh = []
            for i in range(e - s):
                kk = k[i, h // (hv // hk)]
                S = torch.exp(g[i, h]) * S
                S = S + beta[i, h] * torch.outer(v[i, h] - S @ kk, kk)
                oh.append(S @ q[i, h // (hv // hk)])
            outs.append(torch.stack(oh))
        o = torch.stack(outs, dim=1)
        zz = t["z"][s:e]
        y = o * torch.rsqrt((o * o).mean(-1, keepdim=True) + 1e-6) * (1 + t["norm_w"]) * F.silu(zz)
        ys.append(y)
    y = torch.cat(ys)
    (y * torch.from_numpy(dy)).sum().backward()
    for name, gname in GRAD_OF.items():
        np.testing.assert_allclose(gr[gname], t[name].grad.numpy(), rtol=1e-10, atol=1e-12,
                                   err_msg=name)
