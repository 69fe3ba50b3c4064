"""Pins of the oracle's routing, permutation, combine, repack and grouped GEMMs
against brute force on small inputs, round-trip identities and finite
differences of the whole forward."""
import numpy as np
import pytest

from oracle import moe_oracle as O


def _brute_route(idx, expert_begin, E, align):
    T, k = idx.shape
    counts = [0] * E
    rank = {}
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j]) - expert_begin
            if 0 <= e < E:
                rank[(t, j)] = counts[e]
                counts[e] += 1
    offs = [0]
    for e in range(E):
        offs.append(offs[-1] + (counts[e] + align - 1) // align * align)
    row_of = []
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j]) - expert_begin
            row_of.append(offs[e] + rank[(t, j)] if 0 <= e < E else -1)
    return counts, offs, row_of


@pytest.mark.parametrize("T,k,E,eb,nexp", [(37, 2, 4, 0, 4), (50, 3, 5, 2, 9), (8, 1, 3, 0, 3), (64, 4, 2, 1, 8)])
def test_route_matches_brute_force(T, k, E, eb, nexp):
    rng = np.random.default_rng(T * 31 + k)
    idx = np.stack([rng.permutation(nexp)[:k] for _ in range(T)])
    rt = O.route(idx, eb, E)
    counts, offs, row_of = _brute_route(idx, eb, E, O.ALIGN)
    assert list(rt.counts) == counts
    assert list(rt.offsets) == offs
    assert list(rt.row_of) == row_of
    # tok_of / slot_of are the inverse map, -1 on pad rows
    for i, r in enumerate(row_of):
        if r >= 0:
            assert rt.tok_of[r] == i // k and rt.slot_of[r] == i
    assert (rt.tok_of >= 0).sum() == sum(counts)


@pytest.mark.parametrize("T,k,E,eb,nexp", [(37, 2, 4, 0, 4), (50, 3, 5, 2, 9), (64, 4, 2, 1, 8)])
def test_permute_probs_brute_force(T, k, E, eb, nexp):
    """prob_perm walks the assignments in (t, j) order with the brute-force
    routing: the row of (t, j) holds p[t, j]; every other row (pad rows,
    rows of no kept assignment) holds 0.  Probabilities are distinct, so a
    slot/token mix-up or a transposed index cannot pass."""
    rng = np.random.default_rng(T * 7 + k)
    idx = np.stack([rng.permutation(nexp)[:k] for _ in range(T)])
    p = rng.permutation(T * k).reshape(T, k) / (T * k) + 0.5
    rt = O.route(idx, eb, E)
    _, offs, row_of = _brute_route(idx, eb, E, O.ALIGN)
    got = O.permute_probs(p, rt)
    assert got.shape == (offs[-1],)
    ref = np.zeros(offs[-1])
    for t in range(T):
        for j in range(k):
            r = row_of[t * k + j]
            if r >= 0:
                ref[r] = p[t, j]
    assert np.array_equal(got, ref)


def test_route_empty_expert_and_all_on_one():
    idx = np.zeros((40, 1), dtype=np.int64) + 2      # every token on expert 2
    rt = O.route(idx, 0, 4)
    assert list(rt.counts) == [0, 0, 40, 0]
    assert list(rt.offsets) == [0, 0, 0, 64, 64]
    assert list(rt.row_of) == list(range(40))


def test_permute_unpermute_identity():
    rng = np.random.default_rng(11)
    T, H, E = 45, 16, 5
    x = rng.normal(size=(T, H))
    idx = rng.integers(0, E, size=(T, 1))
    rt = O.route(idx, 0, E)
    xp = O.permute(x, rt)
    assert np.all(xp[rt.tok_of < 0] == 0)
    out = O.unpermute_combine(xp, rt.row_of, np.ones((T, 1)))
    assert np.array_equal(out, x)


def test_combine_weighted_sum_brute_force():
    rng = np.random.default_rng(12)
    T, H, k, E = 20, 6, 3, 4
    idx = np.stack([rng.permutation(6)[:k] for _ in range(T)])   # some experts not local
    p = rng.random((T, k))
    rt = O.route(idx, 0, E)
    y = rng.normal(size=(rt.R_pad, H))
    out = O.unpermute_combine(y, rt.row_of, p)
    for t in range(T):
        ref = np.zeros(H)
        for j in range(k):
            e = idx[t, j]
            if e < E:
                ref += p[t, j] * y[rt.row_of[t * k + j]]
        assert np.allclose(out[t], ref, rtol=0, atol=1e-14)


def test_repack_hand_order_and_bijection():
    # F = 4, G = 2: packed rows = in0 in1 gate0 gate1 in2 in3 gate2 gate3
    assert list(O.packed_to_logical(4, 2)) == [0, 1, 4, 5, 2, 3, 6, 7]
    W = np.arange(2 * 128 * 3).reshape(2, 128, 3)
    Wp = O.repack_fc1(W, 32)
    assert np.array_equal(O.unpack_fc1(Wp, 32), W)
    assert np.array_equal(Wp[1, 32], W[1, 64])       # first gate row of block 0
    assert np.array_equal(Wp[1, 64], W[1, 32])       # second input block


def test_grouped_gemm_triple_loop_two_experts():
    rng = np.random.default_rng(13)
    T, H, N = 10, 4, 3
    idx = rng.integers(0, 2, size=(T, 1))
    rt = O.route(idx, 0, 2)
    A = O.permute(rng.normal(size=(T, H)), rt)
    B = rng.normal(size=(2, N, H))
    C = O.grouped_gemm_rows(A, B, rt)
    for r in range(rt.R_pad):
        e = rt.expert_of_row[r]
        for n in range(N):
            ref = 0.0
            if rt.tok_of[r] >= 0:
                for h in range(H):
                    ref += A[r, h] * B[e, n, h]
            assert abs(C[r, n] - ref) < 1e-12


def _toy(act=O.ACT_SWIGLU, seed=14):
    rng = np.random.default_rng(seed)
    T, H, F, E, G = 9, 5, 4, 2, 2
    idx = rng.integers(0, E, size=(T, 1))
    rt = O.route(idx, 0, E)
    x = rng.normal(size=(T, H))
    W1 = rng.normal(size=(E, 2 * F, H)) * 0.5
    b1 = rng.normal(size=(E, 2 * F)) * 0.1
    W2 = rng.normal(size=(E, F, H)) * 0.5
    dY = rng.normal(size=(rt.R_pad, H))
    return rng, rt, x, W1, b1, W2, dY, F, G


@pytest.mark.parametrize("act", [O.ACT_SWIGLU, O.ACT_GEGLU, O.ACT_SREGLU])
def test_fc1_and_dglu_against_finite_differences(act):
    """L = sum(dY * (act(x W1^T + b1) @ W2_e)) over real rows.  dglu_bwd must be
    dL/dpre in packed order (so W2's orientation, the packing and the
    activation derivative are all checked at once)."""
    rng, rt, x, W1, b1, W2, dY, F, G = _toy(act)
    prm = O.ActParams(act)
    xp = O.permute(x, rt)
    W1p = O.repack_fc1(W1, G)
    b1p = O.repack_fc1(b1[..., None], G)[..., 0]
    fo = O.fc1_glu_fwd(xp, W1p, b1p, rt, prm, G)
    # recompute pre in float64 (fo.pre_bf16 is rounded)
    pre = O.grouped_gemm_rows(xp, W1p, rt)
    for e in range(rt.E):
        r0, n = rt.offsets[e], rt.counts[e]
        pre[r0:r0 + n] += b1p[e]
    pre[rt.tok_of < 0] = 0

    def loss(P):
        u, g = O.unpack_glu_cols(P, G)
        y = O.act_fwd(u, g, prm)
        y[rt.tok_of < 0] = 0
        return float(np.sum(dY * O.grouped_gemm_rows(y, np.transpose(W2, (0, 2, 1)), rt)))

    d = O.dglu_bwd(dY, W2, pre, rt, prm, G).astype(np.float64)
    h = 1e-6
    for r in np.nonzero(rt.tok_of >= 0)[0][:5]:
        for c in range(2 * F):
            P1, P2 = pre.copy(), pre.copy()
            P1[r, c] += h
            P2[r, c] -= h
            fd = (loss(P1) - loss(P2)) / (2 * h)
            assert abs(d[r, c] - fd) <= 1e-4 * max(1.0, abs(fd)), (r, c, d[r, c], fd)
    # forward: the activation of the unrounded pre-activation
    u, g = O.unpack_glu_cols(pre, G)
    ref = O.act_fwd(u, g, prm)
    ref[rt.tok_of < 0] = 0
    assert np.allclose(fo.y, ref.astype(np.float32))
    assert np.all(fo.pre_bf16[rt.tok_of < 0] == 0)


def test_wgrad_triple_loop():
    rng = np.random.default_rng(15)
    T, H, M = 12, 3, 4
    idx = rng.integers(0, 3, size=(T, 1))
    rt = O.route(idx, 0, 3)
    A = O.permute(rng.normal(size=(T, M)), rt).T
    B = O.permute(rng.normal(size=(T, H)), rt).T
    D = O.grouped_wgrad(A, B, rt)
    for e in range(3):
        for m in range(M):
            for n in range(H):
                ref = sum(A[m, r] * B[n, r] for r in range(rt.R_pad) if rt.expert_of_row[r] == e)
                assert abs(D[e, m, n] - ref) < 1e-12


@pytest.mark.parametrize("act", [O.ACT_SWIGLU, O.ACT_GEGLU])
def test_feature_scaling_gradients_against_finite_differences(act):
    """Feature scaling: a = p * act(pre) per row, L = sum(dY * (a @ W2_e)).
    dglu_bwd(row_scale=p) must be dL/dpre and dglu_row_prob_grad must be
    dL/dp; the forward with row_scale must be p * act(pre); rows_to_slots
    maps a row value to every (token, slot) routed there."""
    rng, rt, x, W1, b1, W2, dY, F, G = _toy(act, seed=21)
    prm = O.ActParams(act)
    xp = O.permute(x, rt)
    W1p = O.repack_fc1(W1, G)
    pre = O.grouped_gemm_rows(xp, W1p, rt)
    pre[rt.tok_of < 0] = 0
    p = rng.uniform(0.1, 1.0, size=rt.R_pad)
    p[rt.tok_of < 0] = 0

    def loss(P, pp):
        u, g = O.unpack_glu_cols(P, G)
        y = O.act_fwd(u, g, prm) * pp[:, None]
        y[rt.tok_of < 0] = 0
        return float(np.sum(dY * O.grouped_gemm_rows(y, np.transpose(W2, (0, 2, 1)), rt)))

    dp = O.dglu_row_prob_grad(dY, W2, pre, rt, prm, G)
    d = O.dglu_bwd(dY, W2, pre, rt, prm, G, row_scale=p).astype(np.float64)
    h = 1e-6
    for r in np.nonzero(rt.tok_of >= 0)[0]:
        e = np.zeros_like(p); e[r] = h
        fd = (loss(pre, p + e) - loss(pre, p - e)) / (2 * h)
        assert abs(dp[r] - fd) <= 1e-6 * max(1.0, abs(fd)), (r, dp[r], fd)
    for r in np.nonzero(rt.tok_of >= 0)[0][:3]:
        for c in range(2 * F):
            P1, P2 = pre.copy(), pre.copy()
            P1[r, c] += h
            P2[r, c] -= h
            fd = (loss(P1, p) - loss(P2, p)) / (2 * h)
            assert abs(d[r, c] - fd) <= 1e-4 * max(1.0, abs(fd)), (r, c)
    assert np.all(dp[rt.tok_of < 0] == 0)
    fo = O.fc1_glu_fwd(xp, W1p, None, rt, prm, G, row_scale=p)
    u, g = O.unpack_glu_cols(pre, G)
    assert np.allclose(fo.y, (O.act_fwd(u, g, prm) * p[:, None]).astype(np.float32), rtol=1e-6, atol=1e-7)
    slots = O.rows_to_slots(dp, rt.row_of, rt.row_of.size, 1)
    for i, r in enumerate(rt.row_of):
        assert slots[i, 0] == (dp[r] if r >= 0 else 0.0)


@pytest.mark.parametrize("oss", [False, True])
def test_fc1_bias_grad_against_finite_differences(oss):
    """dL/db1p[e, c] for L = sum(dY * (act(x W1p^T + b1p_e) @ W2_e)): central
    differences in one bias entry at a time against fc1_bias_grad of
    dglu_bwd's dFC1 (plain SwiGLU, and the GPT-OSS form with the gate clamp,
    alpha and the +1 offset, whose bias the gradient is for)."""
    rng, rt, x, W1, b1, W2, dY, F, G = _toy(O.ACT_SWIGLU, seed=21)
    prm = (O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0) if oss
           else O.ActParams(O.ACT_SWIGLU))
    xp = O.permute(x, rt)
    W1p = O.repack_fc1(W1 * (4.0 if oss else 1.0), G)   # reach past the +-7 clamp for some rows
    b1p = O.repack_fc1(b1[..., None], G)[..., 0]
    W2t = np.transpose(W2, (0, 2, 1))

    def pre_of(b):
        pre = O.grouped_gemm_rows(xp, W1p, rt)
        for e in range(rt.E):
            r0, n = rt.offsets[e], rt.counts[e]
            pre[r0:r0 + n] += b[e]
        pre[rt.tok_of < 0] = 0
        return pre

    def loss(b):
        u, g = O.unpack_glu_cols(pre_of(b), G)
        y = O.act_fwd(u, g, prm)
        y[rt.tok_of < 0] = 0
        return float(np.sum(dY * O.grouped_gemm_rows(y, W2t, rt)))

    pre = pre_of(b1p)
    if oss:
        _, g = O.unpack_glu_cols(pre, G)
        assert (np.abs(g[rt.tok_of >= 0]) > 7).any()
    db = O.fc1_bias_grad(O.dglu_bwd(dY, W2, pre, rt, prm, G), rt)
    assert db.shape == b1p.shape
    h = 1e-6
    for e in range(rt.E):
        for c in range(2 * F):
            bp, bm = b1p.copy(), b1p.copy()
            bp[e, c] += h
            bm[e, c] -= h
            fd = (loss(bp) - loss(bm)) / (2 * h)
            assert abs(db[e, c] - fd) <= 1e-4 * max(1.0, abs(fd)), (e, c, db[e, c], fd)


def test_grouped_gemm_quant_closed_form():
    """GroupGemm + Quantize on operands whose product is a constant per expert
    (A = 1, B_e = c_e / K): every row-wise block of expert e holds c_e, so its
    codes and scale are the hand-worked MXFP8 values of c_e (1.0 -> scale 0x77
    code 0x78; 448 -> 0x7F / 0x7E; 0.75 -> 0x76 / 0x7C), pad rows give scale 0
    and code 0, and the column-wise copy of a block of 32 equal rows is the
    same code."""
    K, N = 64, 64
    idx = np.repeat(np.arange(3), [40, 3, 33])[:, None]
    rt = O.route(idx, 0, 3)
    c = np.array([1.0, 448.0, 0.75])
    A = np.ones((rt.R_pad, K))
    A[rt.tok_of < 0] = 0
    B = np.stack([np.full((N, K), ce / K) for ce in c])
    y = O.grouped_gemm_quant_fwd(A, B, rt)
    assert y.dtype == np.float32
    q, s = O.mx_quantize_rows(y)
    qc, sc = O.mx_quantize_cols(y)
    expect = {0: (0x77, 0x78), 1: (0x7F, 0x7E), 2: (0x76, 0x7C)}
    for e, (sb, code) in expect.items():
        r0, n = int(rt.offsets[e]), int(rt.counts[e])
        assert np.all(s[r0:r0 + n] == sb) and np.all(q[r0:r0 + n] == code)
        assert np.all(s[r0 + n:int(rt.offsets[e + 1])] == 0) and np.all(q[r0 + n:int(rt.offsets[e + 1])] == 0)
    # expert 0 rows 0..31 are all real: its first column block is 32 copies of 1.0
    assert np.all(sc[:, 0] == 0x77) and np.all(qc[:, :32] == 0x78)
