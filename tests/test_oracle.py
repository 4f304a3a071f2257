"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself: a hand-worked
example, brute-force loops written from a different formulation, a closed form, an
invariant, or a library routine (torch float64 SDPA / autograd)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------------ all-to-all
def test_a2a_hand_worked_example():
    P, S, H, G, D = 2, 4, 2, 2, 1
    qkv = np.array([[[10 * s + c] for c in range(H + 2 * G)] for s in range(S)], np.float64)
    q, k, v = O.seq_to_head(qkv, P, H, G)
    tensors = {"q": q, "k": k, "v": v}
    seq = O.head_to_seq(q, P)
    n = 0
    for name, r, s, h, val in _read_golden("a2a_P2_S4_H2_G2_D1.txt"):
        r, s, h, val = int(r), int(s), int(h), float(val)
        if name == "seq":
            assert seq[r, s, h, 0] == val
        else:
            assert tensors[name][r, s, h, 0] == val
        n += 1
    assert n == 32


@pytest.mark.parametrize("P,S,H,G,D", [(2, 6, 4, 2, 3), (3, 6, 6, 3, 2), (1, 5, 2, 1, 2),
                                       (4, 8, 8, 4, 1)])
def test_a2a_matches_elementwise_index_formula(P, S, H, G, D):
    """Brute force from the element formula out[r2][s][h2][d] = in[s][r2*H/P + h2][d]."""
    x = _rng(1).standard_normal((S, H + 2 * G, D))
    q, k, v = O.seq_to_head(x, P, H, G)
    hq, hk = H // P, G // P
    for r2 in range(P):
        for s in range(S):
            for d in range(D):
                for h2 in range(hq):
                    assert q[r2, s, h2, d] == x[s, r2 * hq + h2, d]
                for h2 in range(hk):
                    assert k[r2, s, h2, d] == x[s, H + r2 * hk + h2, d]
                    assert v[r2, s, h2, d] == x[s, H + G + r2 * hk + h2, d]
    seq = O.head_to_seq(q, P)
    n = S // P
    for r in range(P):
        for t in range(n):
            for h in range(H):
                for d in range(D):
                    assert seq[r, t, h, d] == q[h // hq, r * n + t, h % hq, d]


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_a2a_round_trip_is_identity(P):
    S, H, G, D = 64, 8, 8, 4
    x = synthetic.bf16_to_f64(synthetic.normal_bf16(0, 5, (S, H + 2 * G, D)))
    q, k, v = O.seq_to_head(x, P, H, G)
    for part, lo, hi in ((q, 0, H), (k, H, H + G), (v, H + G, H + 2 * G)):
        back = O.head_to_seq(part, P).reshape(S, hi - lo, D)
        assert np.array_equal(back, x[:, lo:hi])


def test_a2a_single_rank_is_plain_split():
    x = _rng(2).standard_normal((10, 6, 3))
    q, k, v = O.seq_to_head(x, 1, 2, 2)
    assert np.array_equal(q[0], x[:, :2]) and np.array_equal(k[0], x[:, 2:4])
    assert np.array_equal(v[0], x[:, 4:])


def test_a2a_volume_counts_cross_rank_blocks():
    """Closed form of the per-rank volume equals the bytes of the blocks whose sender and
    receiver differ, and scales as hidden * S / P."""
    for P, S, H, G, D in [(2, 8, 4, 2, 4), (4, 64, 8, 4, 8), (8, 1024, 32, 8, 128)]:
        n = S // P
        cross_s2h = sum(n * ((H + 2 * G) // P) * D * 2 for r in range(P) for r2 in range(P)
                        if r2 != r)
        cross_h2s = sum(n * (H // P) * D * 2 for r in range(P) for r2 in range(P) if r2 != r)
        s2h, h2s = O.a2a_volume_bytes(S, P, H, G, D)
        assert s2h * P == cross_s2h and h2s * P == cross_h2s
    a = sum(O.a2a_volume_bytes(4096, 8, 32, 8, 128))
    assert sum(O.a2a_volume_bytes(8192, 8, 32, 8, 128)) == 2 * a


# ------------------------------------------------------------------------ projection
@pytest.mark.parametrize("T,K,C", [(5, 4, 6), (4, 4, 4)])   # square: a transposed w keeps its shape
def test_projection_brute_force_and_identity(T, K, C):
    x = _rng(3).standard_normal((T, K))
    w = _rng(4).standard_normal((C, K))
    y = O.qkv_projection(x, w)
    for s in range(T):
        for c in range(C):
            assert abs(y[s, c] - sum(x[s, j] * w[c, j] for j in range(K))) < 1e-12
    eye = np.eye(K)
    assert np.array_equal(O.qkv_projection(eye, w), w.T)


# ------------------------------------------------------------------------------ RoPE
def test_rope_matches_complex_rotation():
    """Rotate-half RoPE is multiplication of z_i = x_i + 1j * x_{i+D/2} by
    exp(1j * p * theta^(-2i/D))."""
    D, theta = 8, 10000.0
    x = _rng(5).standard_normal((7, 3, D))
    pos = np.array([0, 1, 2, 5, 100, 4096, 1048575])
    y = O.apply_rope(x, pos, theta)
    z = x[..., :D // 2] + 1j * x[..., D // 2:]
    freq = np.array([theta ** (-2.0 * i / D) for i in range(D // 2)])
    zr = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    assert np.allclose(y[..., :D // 2], zr.real, rtol=0, atol=1e-12)
    assert np.allclose(y[..., D // 2:], zr.imag, rtol=0, atol=1e-12)


def test_rope_invariants():
    D, theta = 16, 500000.0
    x = _rng(6).standard_normal((4, 2, D))
    assert np.allclose(O.apply_rope(x, np.zeros(4), theta), x, rtol=0, atol=0)
    y = O.apply_rope(x, np.array([3, 77, 1000, 131071]), theta)
    pair = lambda a: a[..., :D // 2] ** 2 + a[..., D // 2:] ** 2
    assert np.allclose(pair(y), pair(x), rtol=1e-12, atol=1e-12)
    # the lowest pair turns by exactly p radians
    p = 3.0
    yy = O.apply_rope(x[:1], np.array([p]), theta)
    ang = math.atan2(yy[0, 0, D // 2], yy[0, 0, 0]) - math.atan2(x[0, 0, D // 2], x[0, 0, 0])
    assert abs(math.remainder(ang - p, 2 * math.pi)) < 1e-12
    # scores of rotated q, k depend only on the position difference
    q = _rng(7).standard_normal((1, 1, D))
    k = _rng(8).standard_normal((1, 1, D))
    s1 = np.sum(O.apply_rope(q, [10], theta) * O.apply_rope(k, [3], theta))
    s2 = np.sum(O.apply_rope(q, [1007], theta) * O.apply_rope(k, [1000], theta))
    assert abs(s1 - s2) < 1e-10


# ------------------------------------------------------------------------- attention
def test_attention_hand_worked_example():
    g = {r[0]: [float(t) for t in r[1:]] for r in _read_golden("attention_S3_D1.txt")}
    q = np.array(g["q"]).reshape(3, 1, 1)
    k = np.array(g["k"]).reshape(3, 1, 1)
    v = np.array(g["v"]).reshape(3, 1, 1)
    o, lse = O.causal_attention(q, k, v)
    assert np.allclose(o[:, 0, 0], g["o"], rtol=0, atol=1e-14)
    assert np.allclose(lse[0], g["lse"], rtol=0, atol=1e-14)


def _brute_attention(q, k, v, scale):
    S, H, D = q.shape
    G = k.shape[1]
    o = np.zeros_like(q)
    lse = np.zeros((H, S))
    for h in range(H):
        g = h // (H // G)
        for i in range(S):
            sc = [scale * sum(q[i, h, d] * k[j, g, d] for d in range(D)) for j in range(i + 1)]
            m = max(sc)
            e = [math.exp(s - m) for s in sc]
            tot = sum(e)
            for d in range(D):
                o[i, h, d] = sum(e[j] * v[j, g, d] for j in range(i + 1)) / tot
            lse[h, i] = m + math.log(tot)
    return o, lse


@pytest.mark.parametrize("S,H,G,D", [(1, 1, 1, 1), (5, 2, 2, 3), (8, 4, 2, 4), (7, 6, 2, 2)])
def test_attention_brute_force(S, H, G, D):
    r = _rng(9)
    q, k, v = (r.standard_normal((S, n, D)) for n in (H, G, G))
    o, lse = O.causal_attention(q, k, v)
    ob, lb = _brute_attention(q, k, v, 1 / math.sqrt(D))
    assert np.allclose(o, ob, rtol=0, atol=1e-12) and np.allclose(lse, lb, rtol=0, atol=1e-12)


def test_attention_closed_forms():
    S, H, G, D = 40, 4, 2, 8
    r = _rng(10)
    k, v = r.standard_normal((S, G, D)), r.standard_normal((S, G, D))
    o, lse = O.causal_attention(np.zeros((S, H, D)), k, v)
    for h in range(H):
        g = h // 2
        prefix_mean = np.cumsum(v[:, g], axis=0) / np.arange(1, S + 1)[:, None]
        assert np.allclose(o[:, h], prefix_mean, rtol=0, atol=1e-13)
        assert np.allclose(lse[h], np.log(np.arange(1, S + 1)), rtol=0, atol=1e-13)
    q = r.standard_normal((S, H, D))
    o, lse = O.causal_attention(q, k, np.ones((S, G, D)))
    assert np.allclose(o, 1.0, rtol=0, atol=1e-13)          # weights of a row sum to one
    o, lse = O.causal_attention(q, k, v)
    for h in range(H):                                       # row 0 sees only key 0
        assert np.array_equal(o[0, h], v[0, h // 2])
        assert abs(lse[h, 0] - q[0, h] @ k[0, h // 2] / math.sqrt(D)) < 1e-13


def test_attention_shift_invariance():
    """Adding u to every key adds the per-row constant q_i.u*scale: o unchanged, lse shifts."""
    S, H, G, D = 33, 2, 1, 4
    r = _rng(11)
    q, k, v = r.standard_normal((S, H, D)), r.standard_normal((S, G, D)), r.standard_normal((S, G, D))
    u = 3.0 * r.standard_normal(D)
    o1, l1 = O.causal_attention(q, k, v)
    o2, l2 = O.causal_attention(q, k + u, v)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12)
    shift = (q @ u).T / math.sqrt(D)
    assert np.allclose(l2 - l1, shift, rtol=0, atol=1e-12)


@pytest.mark.parametrize("S,H,G,D", [(256, 4, 2, 16), (100, 3, 3, 8), (64, 8, 1, 32)])
def test_attention_matches_torch_sdpa_float64(S, H, G, D):
    r = _rng(12)
    q, k, v = r.standard_normal((S, H, D)), r.standard_normal((S, G, D)), r.standard_normal((S, G, D))
    o, lse = O.causal_attention(q, k, v)
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(H // G, dim=0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(H // G, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    assert np.allclose(o, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    sc = (tq @ tk.transpose(1, 2)) / math.sqrt(D)
    sc = sc.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    assert np.allclose(lse, torch.logsumexp(sc, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_sharded_equals_unsharded_exactly():
    """Heads are independent, and the all-to-alls only move data: the Ulysses result is
    bit-for-bit the unsharded attention."""
    S, H, G, D, P = 96, 8, 4, 8, 4
    x = synthetic.bf16_to_f64(synthetic.normal_bf16(0, 5, (S, H + 2 * G, D)))
    q, k, v = O.seq_to_head(x, P, H, G)
    o_head, lse_head = O.ulysses_attention(q, k, v)
    o_seq = O.head_to_seq(o_head, P).reshape(S, H, D)
    o_ref, lse_ref = O.causal_attention(x[:, :H], x[:, H:H + G], x[:, H + G:])
    assert np.array_equal(o_seq, o_ref)
    assert np.array_equal(lse_head.reshape(H, S), lse_ref)


def test_sampled_rows_equal_full_rows():
    S, H, G, D = 300, 4, 2, 8
    r = _rng(13)
    q, k, v = r.standard_normal((S, H, D)), r.standard_normal((S, G, D)), r.standard_normal((S, G, D))
    rows = synthetic.sample_rows(S, 3, 20)
    o, lse = O.causal_attention(q, k, v)
    os_, ls = O.causal_attention_rows(q, k, v, rows)
    assert np.allclose(os_, o[rows], rtol=0, atol=1e-13)
    assert np.allclose(ls, lse[:, rows], rtol=0, atol=1e-13)


# -------------------------------------------------------------------------- backward
def _torch_attention(q, k, v, H, G):
    S, _, D = q.shape
    tq = q.permute(1, 0, 2)
    tk = k.permute(1, 0, 2).repeat_interleave(H // G, dim=0)
    tv = v.permute(1, 0, 2).repeat_interleave(H // G, dim=0)
    sc = (tq @ tk.transpose(1, 2)) / math.sqrt(D)
    sc = sc.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    return (torch.softmax(sc, dim=-1) @ tv).permute(1, 0, 2)


@pytest.mark.parametrize("S,H,G,D", [(32, 4, 2, 8), (17, 2, 1, 4), (48, 3, 3, 16)])
def test_backward_matches_torch_autograd(S, H, G, D):
    r = _rng(14)
    q, k, v, do = (r.standard_normal((S, n, D)) for n in (H, G, G, H))
    dq, dk, dv = O.causal_attention_bwd(q, k, v, do)
    tq, tk, tv = (torch.from_numpy(a).clone().requires_grad_(True) for a in (q, k, v))
    (_torch_attention(tq, tk, tv, H, G) * torch.from_numpy(do)).sum().backward()
    for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.allclose(mine, ref.numpy(), rtol=0, atol=1e-11)


def test_backward_finite_differences():
    S, H, G, D = 8, 2, 1, 4
    r = _rng(15)
    q, k, v, do = (r.standard_normal((S, n, D)) for n in (H, G, G, H))
    dq, dk, dv = O.causal_attention_bwd(q, k, v, do)

    def loss(qq, kk, vv):
        return float(np.sum(O.causal_attention(qq, kk, vv)[0] * do))

    eps = 1e-6
    for arr, grad, idx in ((q, dq, (5, 1, 2)), (q, dq, (0, 0, 0)), (k, dk, (3, 0, 1)),
                           (k, dk, (7, 0, 3)), (v, dv, (2, 0, 0)), (v, dv, (6, 0, 2))):
        args = [q.copy(), k.copy(), v.copy()]
        which = 0 if arr is q else 1 if arr is k else 2
        args[which][idx] += eps
        up = loss(*args)
        args[which][idx] -= 2 * eps
        dn = loss(*args)
        fd = (up - dn) / (2 * eps)
        assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd))


def test_backward_invariants_and_sampling():
    S, H, G, D = 200, 4, 2, 8
    r = _rng(16)
    q, k, v, do = (r.standard_normal((S, n, D)) for n in (H, G, G, H))
    dq, dk, dv = O.causal_attention_bwd(q, k, v, do)
    # softmax is invariant to a per-row shift, so the key gradients sum to zero
    assert np.allclose(dk.sum(axis=0), 0.0, rtol=0, atol=1e-11)
    # the last key is seen only by the last row; with that row's query zero its weights
    # are uniform, so dv[S-1] = (sum over the group of dO[S-1]) / S
    q0 = q.copy()
    q0[-1] = 0.0
    _, _, dv0 = O.causal_attention_bwd(q0, k, v, do)
    assert np.allclose(dv0[-1, 0], (do[-1, 0] + do[-1, 1]) / S, rtol=0, atol=1e-13)
    rows = synthetic.sample_rows(S, 4, 12)
    dqs, dks, dvs = O.causal_attention_bwd_rows(q, k, v, do, rows, S - 37)
    assert np.allclose(dqs, dq[rows], rtol=0, atol=1e-12)
    assert np.allclose(dks, dk[S - 37:], rtol=0, atol=1e-12)
    assert np.allclose(dvs, dv[S - 37:], rtol=0, atol=1e-12)


# ------------------------------------------------------------------------ whole block
def test_block_forward_equals_unsharded_pipeline():
    S, hidden, H, G, D, P, theta = 64, 32, 8, 4, 8, 4, 10000.0
    x = synthetic.bf16_to_f64(synthetic.normal_bf16(0, 0, (S, hidden)))
    w = synthetic.bf16_to_f64(synthetic.normal_bf16(0, 1, ((H + 2 * G) * D, hidden), std=0.02))
    o_seq, lse, _ = O.ulysses_block_forward(x, w, P, H, G, D, theta)
    y = (x @ w.T).reshape(S, H + 2 * G, D)
    pos = np.arange(S)
    qr = O.apply_rope(y[:, :H], pos, theta)
    kr = O.apply_rope(y[:, H:H + G], pos, theta)
    o, l = O.causal_attention(qr, kr, y[:, H + G:])
    assert np.allclose(o_seq.reshape(S, H, D), o, rtol=0, atol=1e-12)
    assert np.allclose(lse.reshape(H, S), l, rtol=0, atol=1e-12)


def test_generator_is_deterministic_and_normal():
    a = synthetic.normal_bf16(0, 0, (1 << 16,))
    b = synthetic.normal_bf16(0, 0, (1 << 16,))
    c = synthetic.normal_bf16(0, 0, (1000,), offset=500)
    assert np.array_equal(a, b) and np.array_equal(a[500:1500], c)
    x = synthetic.bf16_to_f64(a)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    w = synthetic.bf16_to_f64(synthetic.normal_bf16(0, 1, (1 << 16,), std=0.02))
    assert abs(w.std() - 0.02) < 0.001


# ------------------------------------------------- backward of projection and RoPE
def test_rope_backward_inverts_and_matches_autograd():
    D, theta = 16, 500000.0
    r = _rng(20)
    x = r.standard_normal((9, 3, D))
    pos = np.array([0, 1, 5, 77, 1000, 4095, 65535, 131071, 1 << 20])
    assert np.allclose(O.rope_backward(O.apply_rope(x, pos, theta), pos, theta), x,
                       rtol=0, atol=1e-12)
    g = r.standard_normal(x.shape)
    half = D // 2
    tx = torch.from_numpy(x).clone().requires_grad_(True)
    phi = torch.from_numpy(O.rope_angles(pos, D, theta))[:, None, :]
    lo, hi = tx[..., :half], tx[..., half:]
    y = torch.cat([lo * torch.cos(phi) - hi * torch.sin(phi), hi * torch.cos(phi) + lo * torch.sin(phi)], -1)
    (y * torch.from_numpy(g)).sum().backward()
    assert np.allclose(O.rope_backward(g, pos, theta), tx.grad.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("T,K,C", [(5, 4, 6), (4, 4, 4)])   # square: transposes keep their shape
def test_projection_backward_brute_force(T, K, C):
    r = _rng(21)
    x, w, dy = r.standard_normal((T, K)), r.standard_normal((C, K)), r.standard_normal((T, C))
    dx, dw = O.qkv_projection_backward(x, w, dy)
    for s in range(T):
        for k in range(K):
            assert abs(dx[s, k] - sum(dy[s, c] * w[c, k] for c in range(C))) < 1e-12
    for c in range(C):
        for k in range(K):
            assert abs(dw[c, k] - sum(dy[s, c] * x[s, k] for s in range(T))) < 1e-12


def test_block_backward_matches_torch_autograd():
    """The whole block's training gradients against torch float64 autograd of the same
    forward written in torch (projection, RoPE, unsharded causal GQA attention)."""
    S, hidden, H, G, D, P, theta = 32, 16, 4, 2, 8, 2, 10000.0
    r = _rng(22)
    x, w = r.standard_normal((S, hidden)), 0.3 * r.standard_normal(((H + 2 * G) * D, hidden))
    do = r.standard_normal((S, H * D))
    dx, dw, _ = O.ulysses_block_backward(x, w, do, P, H, G, D, theta)
    tx, tw = (torch.from_numpy(a).clone().requires_grad_(True) for a in (x, w))
    y = (tx @ tw.T).reshape(S, H + 2 * G, D)
    half = D // 2
    phi = torch.from_numpy(O.rope_angles(np.arange(S), D, theta))[:, None, :]

    def rope(t):
        lo, hi = t[..., :half], t[..., half:]
        return torch.cat([lo * torch.cos(phi) - hi * torch.sin(phi), hi * torch.cos(phi) + lo * torch.sin(phi)], -1)

    q, k, v = rope(y[:, :H]), rope(y[:, H:H + G]), y[:, H + G:]
    o = _torch_attention(q, k, v, H, G)
    (o.reshape(S, H * D) * torch.from_numpy(do)).sum().backward()
    assert np.allclose(dx, tx.grad.numpy(), rtol=0, atol=1e-10)
    assert np.allclose(dw, tw.grad.numpy(), rtol=0, atol=1e-10)


@pytest.mark.parametrize("T,H,D,hidden", [(5, 3, 2, 4), (4, 2, 2, 4)])   # square wo: H * D = hidden
def test_output_projection_brute_force(T, H, D, hidden):
    """y[t][j] = sum over heads h and dims d of o[t][h][d] wo[j][h*D + d], written as loops;
    the backward the same way (do[t][h][d] = sum_j dy[t][j] wo[j][h*D+d],
    dwo[j][h*D+d] = sum_t dy[t][j] o[t][h][d])."""
    r = _rng(31)
    o, wo, dy = r.standard_normal((T, H, D)), r.standard_normal((hidden, H * D)), \
        r.standard_normal((T, hidden))
    y = O.output_projection(o, wo)
    do, dwo = O.output_projection_backward(o, wo, dy)
    for t in range(T):
        for j in range(hidden):
            ref = sum(o[t, h, d] * wo[j, h * D + d] for h in range(H) for d in range(D))
            assert abs(y[t, j] - ref) < 1e-12
    for t in range(T):
        for h in range(H):
            for d in range(D):
                ref = sum(dy[t, j] * wo[j, h * D + d] for j in range(hidden))
                assert abs(do[t, h * D + d] - ref) < 1e-12
    for j in range(hidden):
        for h in range(H):
            for d in range(D):
                ref = sum(dy[t, j] * o[t, h, d] for t in range(T))
                assert abs(dwo[j, h * D + d] - ref) < 1e-12


def test_layer_sharded_output_projection_equals_unsharded():
    """Per-rank projection of the restored shards equals one projection of the whole
    sequence, and head->seq followed by it equals summing each rank's head group of the
    head layout (the arithmetic is the same, only the order of the data differs)."""
    S, hidden, H, G, D, P = 16, 8, 4, 2, 4, 2
    r = _rng(32)
    x, w = r.standard_normal((S, hidden)), 0.3 * r.standard_normal(((H + 2 * G) * D, hidden))
    wo = r.standard_normal((hidden, H * D))
    y, _, o_seq = O.ulysses_layer_forward(x, w, wo, P, H, G, D)
    assert np.allclose(y, O.output_projection(o_seq.reshape(S, H, D), wo), rtol=0, atol=1e-12)
    _, _, (_, _, _, _, o_head) = O.ulysses_block_forward(x, w, P, H, G, D)
    hp = H // P
    y2 = sum(o_head[r2].reshape(S, hp * D) @ wo[:, r2 * hp * D:(r2 + 1) * hp * D].T
             for r2 in range(P))
    assert np.allclose(y, y2, rtol=0, atol=1e-12)


def test_layer_backward_matches_torch_autograd():
    """Whole block with the output projection: dx, dw, dwo and dO against torch float64
    autograd of an independent torch restatement."""
    S, hidden, H, G, D, P, theta = 32, 16, 4, 2, 8, 2, 10000.0
    r = _rng(33)
    x, w = r.standard_normal((S, hidden)), 0.3 * r.standard_normal(((H + 2 * G) * D, hidden))
    wo = 0.3 * r.standard_normal((hidden, H * D))
    dy = r.standard_normal((S, hidden))
    dx, dw, dwo, do_seq = O.ulysses_layer_backward(x, w, wo, dy, P, H, G, D, theta)
    tx, tw, two = (torch.from_numpy(a).clone().requires_grad_(True) for a in (x, w, wo))
    y = (tx @ tw.T).reshape(S, H + 2 * G, D)
    half = D // 2
    phi = torch.from_numpy(O.rope_angles(np.arange(S), D, theta))[:, None, :]

    def rope(t):
        lo, hi = t[..., :half], t[..., half:]
        return torch.cat([lo * torch.cos(phi) - hi * torch.sin(phi),
                          hi * torch.cos(phi) + lo * torch.sin(phi)], -1)

    q, k, v = rope(y[:, :H]), rope(y[:, H:H + G]), y[:, H + G:]
    o = _torch_attention(q, k, v, H, G)
    o.retain_grad()
    out = o.reshape(S, H * D) @ two.T
    (out * torch.from_numpy(dy)).sum().backward()
    assert np.allclose(dx, tx.grad.numpy(), rtol=0, atol=1e-10)
    assert np.allclose(dw, tw.grad.numpy(), rtol=0, atol=1e-10)
    assert np.allclose(dwo, two.grad.numpy(), rtol=0, atol=1e-10)
    assert np.allclose(do_seq, o.grad.numpy().reshape(S, H, D), rtol=0, atol=1e-10)


@pytest.mark.parametrize("S,P,H,G,D", [(16, 4, 2, 2, 4), (24, 3, 4, 2, 8), (8, 1, 2, 1, 4),
                                       (32, 8, 8, 8, 4)])
def test_ring_attention_equals_unsharded_causal_attention(S, P, H, G, D):
    """The ring's online merge over shards reaches exactly the plain per-row softmax of the
    whole sequence (up to rounding), and its lse too."""
    r = _rng(41)
    q, k, v = (r.standard_normal((S, n, D)) for n in (H, G, G))
    o, lse, sent = O.ring_attention(q.reshape(P, S // P, H, D), k.reshape(P, S // P, G, D),
                                    v.reshape(P, S // P, G, D))
    ro, rl = O.causal_attention(q, k, v)
    assert np.allclose(o.reshape(S, H, D), ro, rtol=0, atol=1e-12)
    assert np.allclose(lse.transpose(1, 0, 2).reshape(H, S), rl, rtol=0, atol=1e-12)
    assert sent == O.ring_volume_bytes(S, P, G, D)


def test_ring_versus_ulysses_volume():
    """Per-rank bytes: ring (P-1)(S/P)2G D against Ulysses' two all-to-alls
    (S/P)(2H+2G)D (P-1)/P, so ring / Ulysses = P G / (H + G): P/2 for multi-head attention
    (G = H), P/5 under 4:1 GQA (1.6 at P = 8 for the 8B head shape)."""
    S, P, D = 131072, 8, 128
    for H, G, ratio in ((32, 32, P / 2), (32, 8, P / 5)):
        ring = O.ring_volume_bytes(S, P, G, D)
        uly = sum(O.a2a_volume_bytes(S, P, H, G, D))
        assert ring == (P - 1) * (S // P) * 2 * G * D * 2
        assert abs(ring / uly - ratio) < 1e-12
