"""Pins of the fp64 oracle to things other than itself (CPU only).

- torch.nn.LSTMCell / GRUCell / RNNCell in float64 (independent library
  implementations of the textbook cells), forward and autograd backward;
- hand-worked single steps (tests/golden/hand_steps.json);
- central finite differences of every gradient for all four cells;
- sLSTM: the unstabilised closed form, the stabiliser invariants and the
  shift invariance of the stabiliser;
- sequence-level invariants (chunked continuation, batch permutation, T=0).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_steps.json")
FNS = ["lstm", "gru", "elman", "slstm", "slstm_logsig"]


def rand_problem(fn, B, T, N, D, seed, rscale=1.0):
    rng = np.random.default_rng(seed)
    G, S = oracle.GATES[fn], oracle.STATES[fn]
    Wx = rng.normal(size=(B, T, G, N, D))
    R = rng.normal(size=(G, N, D, D)) * rscale / math.sqrt(D)
    b = rng.normal(size=(G, N, D))
    s0 = rng.normal(size=(S, B, 1, N, D))
    if fn.startswith("slstm"):
        s0[2] = np.abs(s0[2]) + 0.5  # normaliser must be positive
        s0[3] = rng.normal(size=s0[3].shape) * 0.5
    return Wx, R, b, s0


# ---------------------------------------------------------------- golden steps
@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_steps(case):
    fn, D = case["fn"], case["D"]
    G, S = oracle.GATES[fn], oracle.STATES[fn]
    Wx = np.array(case["Wx"], dtype=np.float64).reshape(1, 1, G, 1, D)
    R = np.array(case["R"], dtype=np.float64).reshape(G, 1, D, D)
    b = np.array(case["b"], dtype=np.float64).reshape(G, 1, D)
    s0 = np.array(case["s0"], dtype=np.float64).reshape(S, 1, 1, 1, D)
    states, last = oracle.fwd(fn, Wx, R, b, s0)
    exp = np.array(case["expect"], dtype=np.float64).reshape(S, D)
    np.testing.assert_allclose(states[:, 0, 0, 0, :], exp, rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(last[:, 0, 0], states[:, 0, -1])


# ------------------------------------------------------------ torch.nn cells
def _torch_cell(fn, D, G, R, b, n):
    kw = dict(dtype=torch.float64)
    if fn == "lstm":
        cell = torch.nn.LSTMCell(G * D, D, **kw)
    elif fn == "gru":
        cell = torch.nn.GRUCell(G * D, D, **kw)
    else:
        cell = torch.nn.RNNCell(G * D, D, nonlinearity="tanh", **kw)
    with torch.no_grad():
        cell.weight_ih.copy_(torch.eye(G * D, dtype=torch.float64))
        cell.bias_ih.zero_()
        # torch computes W_hh @ h; row (g, j), column i  <->  R[g, n, i, j]
        cell.weight_hh.copy_(torch.from_numpy(R[:, n].transpose(0, 2, 1).reshape(G * D, D)))
        cell.bias_hh.copy_(torch.from_numpy(b[:, n].reshape(G * D)))
    return cell


@pytest.mark.parametrize("fn", ["lstm", "gru", "elman"])
@pytest.mark.parametrize("shape", [(3, 5, 2, 4), (2, 7, 1, 5)])
def test_against_torch_cells(fn, shape):
    B, T, N, D = shape
    G, S = oracle.GATES[fn], oracle.STATES[fn]
    Wx, R, b, s0 = rand_problem(fn, B, T, N, D, seed=11 + D, rscale=1.5)
    rng = np.random.default_rng(5)
    dst = rng.normal(size=(S, B, T, N, D))
    dl = rng.normal(size=(S, B, 1, N, D))
    states, last = oracle.fwd(fn, Wx, R, b, s0)
    dWx, dR, db, ds0 = oracle.bwd(fn, Wx, R, b, s0, dst, dl)

    for n in range(N):
        cell = _torch_cell(fn, D, G, R, b, n)
        x = torch.from_numpy(Wx[:, :, :, n, :].reshape(B, T, G * D).copy()).requires_grad_(True)
        h = torch.from_numpy(s0[0, :, 0, n, :].copy()).requires_grad_(True)
        c0 = c = torch.from_numpy(s0[1, :, 0, n, :].copy()).requires_grad_(True) if fn == "lstm" else None
        h0 = h
        outs_h, outs_c = [], []
        for t in range(T):
            if fn == "lstm":
                h, c = cell(x[:, t], (h, c))
                outs_c.append(c)
            else:
                h = cell(x[:, t], h)
            outs_h.append(h)
        Hs = torch.stack(outs_h, 1)  # [B,T,D]
        np.testing.assert_allclose(states[0, :, :, n, :], Hs.detach().numpy(), rtol=1e-12, atol=1e-13)
        loss = (Hs * torch.from_numpy(dst[0, :, :, n, :])).sum() + (h * torch.from_numpy(dl[0, :, 0, n, :])).sum()
        if fn == "lstm":
            Cs = torch.stack(outs_c, 1)
            np.testing.assert_allclose(states[1, :, :, n, :], Cs.detach().numpy(), rtol=1e-12, atol=1e-13)
            loss = loss + (Cs * torch.from_numpy(dst[1, :, :, n, :])).sum() + (c * torch.from_numpy(dl[1, :, 0, n, :])).sum()
        loss.backward()
        np.testing.assert_allclose(dWx[:, :, :, n, :].reshape(B, T, G * D), x.grad.numpy(), rtol=1e-10, atol=1e-12)
        tdR = cell.weight_hh.grad.numpy().reshape(G, D, D).transpose(0, 2, 1)
        np.testing.assert_allclose(dR[:, n], tdR, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(db[:, n], cell.bias_hh.grad.numpy().reshape(G, D), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(ds0[0, :, 0, n, :], h0.grad.numpy(), rtol=1e-10, atol=1e-12)
        if fn == "lstm":
            np.testing.assert_allclose(ds0[1, :, 0, n, :], c0.grad.numpy(), rtol=1e-10, atol=1e-12)


# ------------------------------------------------------- finite differences
def _loss(fn, Wx, R, b, s0, W1, W2):
    st, last = oracle.fwd(fn, Wx, R, b, s0)
    return float((st * W1).sum() + (last * W2).sum())


@pytest.mark.parametrize("fn", FNS)
def test_finite_differences(fn):
    B, T, N, D = 2, 4, 2, 3
    Wx, R, b, s0 = rand_problem(fn, B, T, N, D, seed=3, rscale=1.2)
    rng = np.random.default_rng(9)
    S = oracle.STATES[fn]
    W1 = rng.normal(size=(S, B, T, N, D))
    W2 = rng.normal(size=(S, B, 1, N, D))
    grads = oracle.bwd(fn, Wx, R, b, s0, W1, W2)
    eps = 1e-6
    for name, arr, g in zip(["Wx", "R", "b", "s0"], [Wx, R, b, s0], grads):
        fd = np.zeros_like(arr)
        flat, fflat = arr.reshape(-1), fd.reshape(-1)
        for k in range(flat.size):
            keep = flat[k]
            flat[k] = keep + eps
            lp = _loss(fn, Wx, R, b, s0, W1, W2)
            flat[k] = keep - eps
            lm = _loss(fn, Wx, R, b, s0, W1, W2)
            flat[k] = keep
            fflat[k] = (lp - lm) / (2 * eps)
        scale = max(1.0, np.abs(fd).max())
        np.testing.assert_allclose(g, fd, rtol=0, atol=2e-7 * scale, err_msg=f"{fn} d{name}")


# ------------------------------------------------------------------- sLSTM
def _preacts(Wx, R, b, h_prev):
    """a[b,t,g,n,j] = Wx + h_{t-1} . R[g,n] + b, via numpy einsum."""
    return Wx + np.einsum("btni,gnij->btgnj", h_prev, R) + b[None, None]


def _forget(fn, af):
    """The forget gate f (not its log): e^{a_f} for slstm, sigmoid(a_f) for
    slstm_logsig, written directly rather than through the log."""
    return np.exp(af) if fn == "slstm" else 1.0 / (1.0 + np.exp(-af))


@pytest.mark.parametrize("fn", ["slstm", "slstm_logsig"])
def test_slstm_unstabilised_closed_form(fn):
    """Stabilised states times exp(m) equal the plain recurrence
    c~ = f c~ + e^{a_i} tanh(a_z), n~ = f n~ + e^{a_i}; h = sig(a_o) c~/n~,
    with f = e^{a_f} (slstm) or sigmoid(a_f) (slstm_logsig)."""
    B, T, N, D = 2, 12, 2, 3
    Wx, R, b, s0 = rand_problem(fn, B, T, N, D, seed=21)
    st, _ = oracle.fwd(fn, Wx, R, b, s0)
    h_prev = np.concatenate([s0[0], st[0, :, :-1]], axis=1)
    a = _preacts(Wx, R, b, h_prev)
    ct = s0[1, :, 0] * np.exp(s0[3, :, 0])
    nt = s0[2, :, 0] * np.exp(s0[3, :, 0])
    for t in range(T):
        ai, af, az, ao = (a[:, t, g] for g in range(4))
        ct = _forget(fn, af) * ct + np.exp(ai) * np.tanh(az)
        nt = _forget(fn, af) * nt + np.exp(ai)
        h = ct / nt / (1 + np.exp(-ao))
        np.testing.assert_allclose(st[0, :, t], h, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(st[1, :, t] * np.exp(st[3, :, t]), ct, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(st[2, :, t] * np.exp(st[3, :, t]), nt, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("fn", ["slstm", "slstm_logsig"])
def test_slstm_stabiliser_invariants(fn):
    B, T, N, D = 3, 40, 2, 4
    Wx, R, b, s0 = rand_problem(fn, B, T, N, D, seed=8, rscale=2.0)
    Wx *= 3.0  # large gate values: the unstabilised form would overflow soon
    s0[2] = 1.0
    s0[3] = 0.0
    st, _ = oracle.fwd(fn, Wx, R, b, s0)
    assert np.all(np.isfinite(st))
    h_prev = np.concatenate([s0[0], st[0, :, :-1]], axis=1)
    m_prev = np.concatenate([s0[3], st[3, :, :-1]], axis=1)
    a = _preacts(Wx, R, b, h_prev)
    ig = np.exp(a[:, :, 0] - st[3])
    fg = _forget(fn, a[:, :, 1]) * np.exp(m_prev - st[3])
    # a is recomputed here in another summation order: allow rounding only
    assert np.all(ig <= 1.0 + 1e-12) and np.all(fg <= 1.0 + 1e-12)
    np.testing.assert_allclose(np.maximum(ig, fg), 1.0, rtol=0, atol=1e-12)
    assert np.all(st[2] >= 1.0 - 1e-12)  # n_t >= 1 when n_0 = 1
    # |c/n| <= max(|c0/n0|, 1): c/n is a convex combination of c0/n0 and tanh values
    bound = np.maximum(np.abs(s0[1] / s0[2]), 1.0)
    assert np.all(np.abs(st[1] / st[2]) <= bound + 1e-12)


@pytest.mark.parametrize("fn", ["slstm", "slstm_logsig"])
def test_slstm_shift_invariance(fn):
    B, T, N, D = 2, 10, 1, 3
    Wx, R, b, s0 = rand_problem(fn, B, T, N, D, seed=13)
    st, _ = oracle.fwd(fn, Wx, R, b, s0)
    k = 0.7
    s1 = s0.copy()
    s1[3] += k
    s1[1] *= math.exp(-k)
    s1[2] *= math.exp(-k)
    st2, _ = oracle.fwd(fn, Wx, R, b, s1)
    np.testing.assert_allclose(st2[0], st[0], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------- sequences
def test_lstm_gru_elman_bounds():
    for fn in ["lstm", "elman", "gru"]:
        Wx, R, b, s0 = rand_problem(fn, 2, 30, 2, 4, seed=2, rscale=2.0)
        s0[0] = np.clip(s0[0], -0.99, 0.99)
        st, _ = oracle.fwd(fn, Wx * 3, R, b, s0)
        if fn in ("lstm", "elman"):
            assert np.all(np.abs(st[0]) < 1.0)
        if fn == "gru":
            assert np.all(np.abs(st[0]) <= np.maximum(np.abs(s0[0]).max(), 1.0) + 1e-12)
        if fn == "lstm":
            t = np.arange(1, 31)[None, :, None, None]
            assert np.all(np.abs(st[1]) <= np.abs(s0[1]) + t + 1e-12)


@pytest.mark.parametrize("fn", FNS)
def test_chunked_continuation(fn):
    B, T, N, D = 2, 9, 2, 3
    Wx, R, b, s0 = rand_problem(fn, B, T, N, D, seed=4)
    st, last = oracle.fwd(fn, Wx, R, b, s0)
    st1, l1 = oracle.fwd(fn, Wx[:, :4], R, b, s0)
    st2, l2 = oracle.fwd(fn, Wx[:, 4:], R, b, l1)
    np.testing.assert_allclose(np.concatenate([st1, st2], axis=2), st, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l2, last, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("fn", FNS)
def test_batch_permutation(fn):
    B, T, N, D = 4, 5, 2, 3
    Wx, R, b, s0 = rand_problem(fn, B, T, N, D, seed=6)
    perm = np.array([2, 0, 3, 1])
    st, _ = oracle.fwd(fn, Wx, R, b, s0)
    stp, _ = oracle.fwd(fn, Wx[perm], R, b, s0[:, perm])
    np.testing.assert_allclose(stp, st[:, perm], rtol=1e-14, atol=0)


@pytest.mark.parametrize("fn", FNS)
def test_zero_length_and_zero_initial(fn):
    G, S = oracle.GATES[fn], oracle.STATES[fn]
    Wx, R, b, s0 = rand_problem(fn, 2, 0, 1, 3, seed=1)
    st, last = oracle.fwd(fn, Wx, R, b, s0)
    assert st.shape == (S, 2, 0, 1, 3)
    np.testing.assert_array_equal(last, s0)
    dl = np.random.default_rng(0).normal(size=s0.shape)
    dWx, dR, db, ds0 = oracle.bwd(fn, Wx, R, b, s0, None, dl)
    np.testing.assert_array_equal(ds0, dl)
    assert not dR.any() and not db.any()
    # states0 = None means zeros
    Wx, R, b, _ = rand_problem(fn, 2, 3, 1, 3, seed=1)
    a, _ = oracle.fwd(fn, Wx, R, b, None)
    z, _ = oracle.fwd(fn, Wx, R, b, np.zeros((S, 2, 1, 1, 3)))
    np.testing.assert_array_equal(a, z)


def test_threads_do_not_change_results():
    Wx, R, b, s0 = rand_problem("lstm", 3, 6, 2, 4, seed=31)
    d = np.random.default_rng(1).normal(size=(2, 3, 6, 2, 4))
    a = oracle.bwd("lstm", Wx, R, b, s0, d, nthreads=1)
    c = oracle.bwd("lstm", Wx, R, b, s0, d, nthreads=4)
    for x, y in zip(a, c):
        np.testing.assert_allclose(x, y, rtol=1e-13, atol=1e-14)


# --------------------------------------------------- bfloat16 operand mode
def _bf16(x):
    """binary32 then bfloat16 (round to nearest even), by torch's conversions."""
    return x.float().bfloat16().double()


class _Bf16OperandBranch(torch.autograd.Function):
    """The recurrent branch y = bf16(h) @ W + b with bfloat16 operands and exact
    accumulation. Its backward takes bfloat16 operands too:
    dh = bf16(dy) @ W^T, dW = bf16(h)^T bf16(dy), db = sum bf16(dy)."""

    @staticmethod
    def forward(ctx, h, W, b):
        hb = _bf16(h)
        ctx.save_for_backward(hb, W)
        return hb @ W + b

    @staticmethod
    def backward(ctx, dy):
        hb, W = ctx.saved_tensors
        dyb = _bf16(dy)
        return dyb @ W.T, hb.T @ dyb, dyb.sum(0)


def _torch_cell_step(fn, x, branch, sp, D):
    """One step of each cell written with torch operations, for autograd.
    x: the input pre-activations [B, G*D]; branch: the recurrent branch
    h.R + b [B, G*D]; sp: the previous states (list of [B, D]). GRU applies
    the reset gate to the whole recurrent branch of n (bias included); sLSTM
    takes the max of the stabiliser with torch.where, so a tie sends the whole
    derivative to the forget branch."""
    if fn == "lstm":
        a = x + branch
        i, f, g, o = a.split(D, dim=1)
        c = torch.sigmoid(f) * sp[1] + torch.sigmoid(i) * torch.tanh(g)
        return [torch.sigmoid(o) * torch.tanh(c), c]
    if fn == "gru":
        xr, xz, xn = x.split(D, dim=1)
        qr, qz, qn = branch.split(D, dim=1)
        r, z = torch.sigmoid(xr + qr), torch.sigmoid(xz + qz)
        nn_ = torch.tanh(xn + r * qn)
        return [(1 - z) * nn_ + z * sp[0]]
    if fn == "elman":
        return [torch.tanh(x + branch)]
    ai, af, az, ao = (x + branch).split(D, dim=1)
    lf = af if fn == "slstm" else torch.nn.functional.logsigmoid(af)
    mp = sp[3]
    m = torch.where(lf + mp >= ai, lf + mp, ai)
    ig, fg = torch.exp(ai - m), torch.exp(lf + mp - m)
    c = fg * sp[1] + ig * torch.tanh(az)
    n = fg * sp[2] + ig
    return [torch.sigmoid(ao) * c / n, c, n, m]


@pytest.mark.parametrize("fn", FNS)
def test_bf16_operand_mode_against_torch_autograd(fn):
    """The oracle's bfloat16 mode equals torch autograd of the same cell with a
    bfloat16-operand recurrent matmul (cell and derivatives by torch). For GRU
    the operand of the backward contraction is the gradient reaching the
    recurrent branch, r * dn_pre for gate n, not dWx_n = dn_pre: autograd
    delivers exactly that to the branch, so a rounding applied to the wrong
    quantity fails here."""
    B, T, N, D = 3, 8, 1, 6
    G, S = oracle.GATES[fn], oracle.STATES[fn]
    Wx, R, b, s0 = rand_problem(fn, B, T, N, D, seed=17, rscale=1.5)
    rng = np.random.default_rng(2)
    dst = rng.normal(size=(S, B, T, N, D))
    dl = rng.normal(size=(S, B, 1, N, D))
    states, last = oracle.fwd(fn, Wx, R, b, s0, round_bf16=True)
    dWx, dR, db, ds0 = oracle.bwd(fn, Wx, R, b, s0, dst, dl, round_bf16=True)
    plain, _ = oracle.fwd(fn, Wx, R, b, s0)
    assert np.abs(plain - states).max() > 1e-6  # the mode changes the result
    pdWx, pdR, _, _ = oracle.bwd(fn, Wx, R, b, s0, dst, dl)
    assert np.abs(pdR - dR).max() > 1e-6

    x = torch.from_numpy(Wx[:, :, :, 0, :].copy()).requires_grad_(True)        # [B,T,G,D]
    W = torch.from_numpy(R[:, 0].transpose(1, 0, 2).reshape(D, G * D).copy()).requires_grad_(True)
    bb = torch.from_numpy(b[:, 0].reshape(G * D).copy()).requires_grad_(True)
    init = [torch.from_numpy(s0[s, :, 0, 0].copy()).requires_grad_(True) for s in range(S)]
    sp = list(init)
    seq = [[] for _ in range(S)]
    for t in range(T):
        branch = _Bf16OperandBranch.apply(sp[0], W, bb)
        sp = _torch_cell_step(fn, x[:, t].reshape(B, G * D), branch, sp, D)
        for s in range(S):
            seq[s].append(sp[s])
    loss = 0.0
    for s in range(S):
        Hs = torch.stack(seq[s], 1)  # [B,T,D]
        np.testing.assert_allclose(states[s, :, :, 0], Hs.detach().numpy(), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(last[s, :, 0, 0], sp[s].detach().numpy(), rtol=1e-12, atol=1e-13)
        loss = loss + (Hs * torch.from_numpy(dst[s, :, :, 0])).sum() + (sp[s] * torch.from_numpy(dl[s, :, 0, 0])).sum()
    loss.backward()
    np.testing.assert_allclose(dWx[:, :, :, 0], x.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dR[:, 0], W.grad.numpy().reshape(D, G, D).transpose(1, 0, 2),
                               rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(db[:, 0], bb.grad.numpy().reshape(G, D), rtol=1e-10, atol=1e-12)
    for s in range(S):
        np.testing.assert_allclose(ds0[s, :, 0, 0], init[s].grad.numpy(), rtol=1e-10, atol=1e-12)


# ------------------------------------------------------- input projection oracle
def test_projection_matches_torch_linear_and_autograd():
    """The projection oracle against torch.nn.functional.linear in float64 and
    its autograd gradients (a library routine, not a retyped formula)."""
    from oracle import projection
    g = torch.Generator().manual_seed(11)
    x = torch.randn(37, 24, generator=g, dtype=torch.float64, requires_grad=True)
    W = torch.randn(40, 24, generator=g, dtype=torch.float64, requires_grad=True)
    bias = torch.randn(40, generator=g, dtype=torch.float64, requires_grad=True)
    dy = torch.randn(37, 40, generator=g, dtype=torch.float64)
    y = torch.nn.functional.linear(x, W, bias)
    y.backward(dy)
    np.testing.assert_allclose(projection.fwd(x, W, bias), y.detach().numpy(), rtol=1e-12, atol=1e-12)
    dx, dW, db = projection.bwd(x, W, dy)
    np.testing.assert_allclose(dx, x.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dW, W.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(db, bias.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_projection_then_scan_is_torch_lstm_with_input_weights():
    """Projection followed by the scan oracle equals torch.nn.LSTM with
    input_size = I: weight_ih = W_x, bias_ih = projection bias, weight_hh =
    the stacked R[g]^T blocks, bias_hh = b (one head)."""
    from oracle import oracle, projection
    B, T, I, D = 3, 7, 5, 4
    g = torch.Generator().manual_seed(12)
    x = torch.randn(B, T, I, generator=g, dtype=torch.float64)
    W = torch.randn(4 * D, I, generator=g, dtype=torch.float64)
    bias_x = torch.randn(4 * D, generator=g, dtype=torch.float64)
    R = torch.randn(4, 1, D, D, generator=g, dtype=torch.float64) / 2
    b = torch.randn(4, 1, D, generator=g, dtype=torch.float64)
    s0 = torch.randn(2, B, 1, 1, D, generator=g, dtype=torch.float64)
    Wx = projection.fwd(x.reshape(B * T, I), W, bias_x).reshape(B, T, 4, 1, D)
    st, _ = oracle.fwd("lstm", Wx, R.numpy(), b.numpy(), s0.numpy())
    lstm = torch.nn.LSTM(I, D, batch_first=True).double()
    with torch.no_grad():
        lstm.weight_ih_l0.copy_(W)
        lstm.bias_ih_l0.copy_(bias_x)
        lstm.weight_hh_l0.copy_(torch.cat([R[k, 0].t() for k in range(4)], dim=0))
        lstm.bias_hh_l0.copy_(b[:, 0].reshape(-1))
        out, _ = lstm(x, (s0[0, :, 0, 0][None], s0[1, :, 0, 0][None]))
    np.testing.assert_allclose(st[0, :, :, 0, :], out.numpy(), rtol=1e-10, atol=1e-12)


def test_stack_oracle_matches_two_layer_torch_lstm():
    """The chained oracle (projection then scan, per layer, and its backward
    through both layers) against torch.nn.LSTM(num_layers=2) in float64:
    outputs and every gradient by autograd."""
    from oracle import stack
    B, T, I, D = 2, 6, 5, 4
    g = torch.Generator().manual_seed(21)
    x = torch.randn(B, T, I, generator=g, dtype=torch.float64, requires_grad=True)
    layers, torch_w = [], []
    for l in range(2):
        Il = I if l == 0 else D
        W = torch.randn(4 * D, Il, generator=g, dtype=torch.float64)
        bx = torch.randn(4 * D, generator=g, dtype=torch.float64)
        R = torch.randn(4, 1, D, D, generator=g, dtype=torch.float64) / 2
        b = torch.randn(4, 1, D, generator=g, dtype=torch.float64)
        s0 = torch.randn(2, B, 1, 1, D, generator=g, dtype=torch.float64)
        layers.append(dict(W_x=W.numpy(), bias_x=bx.numpy(), R=R.numpy(), b=b.numpy(), states=s0.numpy()))
        torch_w.append((W, bx, R, b, s0))
    lstm = torch.nn.LSTM(I, D, num_layers=2, batch_first=True).double()
    with torch.no_grad():
        for l, (W, bx, R, b, s0) in enumerate(torch_w):
            getattr(lstm, f"weight_ih_l{l}").copy_(W)
            getattr(lstm, f"bias_ih_l{l}").copy_(bx)
            getattr(lstm, f"weight_hh_l{l}").copy_(torch.cat([R[k, 0].t() for k in range(4)], dim=0))
            getattr(lstm, f"bias_hh_l{l}").copy_(b[:, 0].reshape(-1))
    h0 = torch.stack([w[4][0, :, 0, 0] for w in torch_w]).clone().requires_grad_(True)
    c0 = torch.stack([w[4][1, :, 0, 0] for w in torch_w]).clone().requires_grad_(True)
    out, _ = lstm(x, (h0, c0))
    dh = torch.randn(B, T, D, generator=g, dtype=torch.float64)
    out.backward(dh)
    h, _, _ = stack.fwd("lstm", x.detach().numpy(), layers)
    np.testing.assert_allclose(h, out.detach().numpy(), rtol=1e-10, atol=1e-12)
    dx, grads = stack.bwd("lstm", x.detach().numpy(), layers, dh.numpy())
    np.testing.assert_allclose(dx, x.grad.numpy(), rtol=1e-9, atol=1e-11)
    for l in range(2):
        gw = grads[l]
        np.testing.assert_allclose(gw["W_x"], getattr(lstm, f"weight_ih_l{l}").grad.numpy(), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(gw["bias_x"], getattr(lstm, f"bias_ih_l{l}").grad.numpy(), rtol=1e-9, atol=1e-11)
        whh = getattr(lstm, f"weight_hh_l{l}").grad.numpy()  # rows (g, j), columns i  = dR[g][i][j]^T
        dR_t = np.concatenate([gw["R"][k, 0].T for k in range(4)], axis=0)
        np.testing.assert_allclose(dR_t, whh, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(gw["b"][:, 0].reshape(-1), getattr(lstm, f"bias_hh_l{l}").grad.numpy(),
                                   rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(gw["states"][0, :, 0, 0], h0.grad[l].numpy(), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(gw["states"][1, :, 0, 0], c0.grad[l].numpy(), rtol=1e-9, atol=1e-11)
