"""The GPU tests' error bounds, checked on the CPU against the arithmetic they come from.

A bound must admit a correct kernel and still catch a wrong one. So for each bound a numpy
simulation applies to the fp64 definition exactly the roundings the kernels declare, and must
stay inside the bound with margin. Where a plausible coarser rounding exists (bf16 where the
kernel keeps fp16), the simulation with that rounding must leave the bound."""
import numpy as np
import pytest

import oracle as O
import synthetic
from oracle import ulysses_oracle as OU
from tolerances import assert_rel, bf16_ulp, peaked_bounds


def _bf16(a):
    return synthetic.bf16_to_f64(synthetic.f32_to_bf16(np.asarray(a, np.float32)))


def _f16(a):
    return np.asarray(a, np.float16).astype(np.float64)


# ------------------------------------------------------------- peaked-softmax bounds
def _peaked_rank0(S=1024, P=4, H=8, G=4, D=128, std=3.0):
    """Rank 0's inputs of the GPU tests' peaked case (same generator keys)."""
    f = lambda bits: synthetic.bf16_to_f64(bits)[0]
    q = f(synthetic.normal_bf16(0, synthetic.TENSOR_Q, (P, S, H // P, D), std=std))
    k = f(synthetic.normal_bf16(0, synthetic.TENSOR_K, (P, S, G // P, D), std=std))
    v = f(synthetic.normal_bf16(0, synthetic.TENSOR_V, (P, S, G // P, D), std=std))
    do = f(synthetic.normal_bf16(synthetic.SEED_DO, 0, (P, S, H // P, D)))
    return q, k, v, do


def _floor_log2(m):
    return int(np.frexp(m)[1]) - 1


def _bwd_exponents(q, k, v, do, scale):
    """The backward's per-call power-of-two exponents, restated from the kernels' rule:
    2^kp scale in [2^7, 2^8); q' = 2^eq q and k' = 2^-eq k with eq = floor((E(max|k|) -
    E(max|q|)) / 2); max|v'| in [2^-1, 2^0); edo the largest exponent with
    2^kp scale D max|dO'| max|v'| < 2^14 and max|dO'| < 2^15; every exponent within
    [-60, 60] (kp within [-30, 30])."""
    D = q.shape[-1]
    clamp = lambda e, lim=60: int(min(max(e, -lim), lim))   # noqa: E731
    kp = clamp(8 - int(np.frexp(scale)[1]), 30)
    mq, mk, mv, mdo = (float(np.abs(t).max()) for t in (q, k, v, do))
    eq = clamp((_floor_log2(mk) - _floor_log2(mq)) // 2) if mq > 0 and mk > 0 else 0
    ek = -eq
    ev = clamp(-1 - _floor_log2(mv)) if mv > 0 else 0
    edo = 0
    if mdo > 0:
        edo = 14 - _floor_log2(mdo)
        if mv > 0:
            edo = min(edo, 13 - _floor_log2(2.0 ** kp * scale * D * mdo * mv * 2.0 ** ev))
        edo = clamp(edo)
    return kp, eq, ek, ev, edo


def _simulate(q, k, v, do, p_store, ds_store):
    """The kernels' roundings on the fp64 definition:
    - forward: unnormalised P (relative to the row max) stored as bf16 for P V; the row sum
      from the unrounded P;
    - backward: O held as bf16 plus its bf16 residual for the row term D; P_s = scale * P
      unrounded; dS = P_s (dP - D) from the unrounded P_s.  Both are stored scaled by the
      call's powers of two (P' = 2^kp P_s, dS' = 2^(kp+edo+ev) dS): dS' with `ds_store` for
      dQ and dK, P' with `p_store` for dV, and the stored values scaled back exactly.  The
      scaled fp16 copies of q, k, v, dO are exact (normal fp16 holds every bf16 value);
    - every output rounded once to bf16."""
    S, hl, D = q.shape
    gl = k.shape[1]
    grp, scale = hl // gl, 1.0 / np.sqrt(D)
    kp, _, _, ev, edo = _bwd_exponents(q, k, v, do, scale)
    f_p, f_ds = 2.0 ** kp, 2.0 ** (kp + edo + ev)
    o, lse = O.causal_attention(q, k, v)
    o_hi = _bf16(o)
    o_lo = _bf16(o - o_hi)
    mask = np.tril(np.ones((S, S), bool))
    o_sim, dq = np.zeros_like(q), np.zeros_like(q)
    dk, dv = np.zeros_like(k), np.zeros_like(v)
    for h in range(hl):
        g = h // grp
        s = np.where(mask, scale * q[:, h] @ k[:, g].T, -np.inf)
        pu = np.exp(s - s.max(axis=1, keepdims=True))
        o_sim[:, h] = (_bf16(pu) @ v[:, g]) / pu.sum(axis=1)[:, None]
        d_row = np.sum(do[:, h] * (o_hi[:, h] + o_lo[:, h]), axis=1)
        ps = np.where(mask, scale * np.exp(s - lse[h][:, None]), 0.0)
        ds = ds_store(f_ds * ps * (do[:, h] @ v[:, g].T - d_row[:, None])) / f_ds
        dq[:, h] = ds @ k[:, g]
        dk[:, g] += ds.T @ q[:, h]
        dv[:, g] += (p_store(f_p * ps).T @ do[:, h]) / (f_p * scale)
    return tuple(_bf16(t) for t in (o_sim, dq, dk, dv))


def _ratios(sim, ref, bounds):
    """Worst error over bound per output, the bound widened by one bf16 ulp as in the tests."""
    return [float((np.abs(s - r) / (b + bf16_ulp(r))).max()) for s, r, b in zip(sim, ref, bounds)]


@pytest.fixture(scope="module")
def peaked():
    q, k, v, do = _peaked_rank0()
    o, _ = O.causal_attention(q, k, v)
    dq, dk, dv = O.causal_attention_bwd(q, k, v, do)
    return (q, k, v, do), (o, dq, dk, dv), peaked_bounds(q, k, v, do, 8, 4)


def test_peaked_bounds_admit_the_kernels_roundings(peaked):
    inputs, ref, bounds = peaked
    ratios = _ratios(_simulate(*inputs, _f16, _f16), ref, bounds)
    assert max(ratios) <= 0.9, dict(zip(("o", "dq", "dk", "dv"), ratios))


def test_peaked_bounds_catch_bf16_ds(peaked):
    inputs, ref, bounds = peaked
    _, rq, rk, _ = _ratios(_simulate(*inputs, _f16, _bf16), ref, bounds)
    assert rq >= 1.5 and rk >= 1.5, (rq, rk)


def test_peaked_bounds_catch_bf16_p_for_dv(peaked):
    inputs, ref, bounds = peaked
    rv = _ratios(_simulate(*inputs, _bf16, _f16), ref, bounds)[3]
    assert rv >= 1.5, rv


# ------------------------------------------------------- whole-step gradient tolerance
@pytest.mark.parametrize("S,P,hidden,H,G,D,theta", [(1024, 4, 512, 8, 8, 64, 0.0),
                                                    (2048, 8, 4096, 32, 8, 128, 500000.0)])
def test_training_step_tolerance_leaves_room_beyond_bf16_storage(S, P, hidden, H, G, D, theta):
    """The whole-step gradients (dqkv, dx, dW) are held to max|err| <= 2e-2 max|ref| and a
    normwise error <= 1.5e-2 against the unrounded fp64 pipeline.  Storing every
    intermediate as bf16 (projection output, RoPE'd q/k, dQ/dK/dV, the gradient after the
    RoPE backward, dx), with everything else exact, must use at most half of that, leaving
    the other half to the kernels' internal roundings (which the stage bounds cover)."""
    x = synthetic.bf16_to_f64(synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, hidden)))
    w = synthetic.bf16_to_f64(synthetic.normal_bf16(0, synthetic.TENSOR_W, ((H + 2 * G) * D, hidden),
                                                    std=0.02))
    do = synthetic.bf16_to_f64(synthetic.normal_bf16(synthetic.SEED_DO, 0, (S, H, D)))
    rdx, rdw, rdqkv = O.ulysses_block_backward(x, w, do, P, H, G, D, theta)
    qkv = _bf16(O.qkv_projection(x, w)).reshape(S, H + 2 * G, D)
    pos = np.arange(S)
    if theta:
        qkv = np.concatenate([_bf16(O.apply_rope(qkv[:, :H + G], pos, theta)), qkv[:, H + G:]],
                             axis=1)
    q, k, v = O.seq_to_head(qkv, P, H, G)
    do_head = OU._seq_to_head_one(do, P)
    grads = [O.causal_attention_bwd(q[r], k[r], v[r], do_head[r]) for r in range(P)]
    dq, dk, dv = (np.stack([_bf16(g[i]) for g in grads]) for i in range(3))
    g = O.head_to_seq_qkv(dq, dk, dv, P)
    if theta:
        g = np.concatenate([_bf16(O.rope_backward(g[:, :H + G], pos, theta)), g[:, H + G:]],
                           axis=1)
    g = _bf16(g)
    dx, dw = O.qkv_projection_backward(x, w, g.reshape(S, -1))
    for name, got, ref in (("dqkv", g, rdqkv), ("dx", _bf16(dx), rdx), ("dw", dw, rdw)):
        assert_rel(got, ref, name, rel_max=1e-2, rel_norm=7.5e-3)


@pytest.mark.parametrize("S,P,hidden,H,G,D,theta", [(1024, 4, 512, 8, 8, 64, 0.0),
                                                    (2048, 8, 4096, 32, 8, 128, 500000.0)])
def test_layer_tolerance_leaves_room_beyond_bf16_storage(S, P, hidden, H, G, D, theta):
    """The whole-layer test holds y, dWo (and dx, dW, covered above) to the same tolerance.
    Storing the attention output, y and dO as bf16, with everything else exact, must use at
    most half of it."""
    x = synthetic.bf16_to_f64(synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, hidden)))
    w = synthetic.bf16_to_f64(synthetic.normal_bf16(0, synthetic.TENSOR_W, ((H + 2 * G) * D, hidden),
                                                    std=0.02))
    wo = synthetic.bf16_to_f64(synthetic.normal_bf16(0, synthetic.TENSOR_WO, (hidden, H * D), std=0.02))
    dy = synthetic.bf16_to_f64(synthetic.normal_bf16(synthetic.SEED_DO, synthetic.TENSOR_WO, (S, hidden)))
    o_seq, _, _ = O.ulysses_block_forward(x, w, P, H, G, D, theta)
    o = o_seq.reshape(S, H, D)
    ry = O.output_projection(o, wo)
    rdo, rdwo = O.output_projection_backward(o, wo, dy)
    o16 = _bf16(o)
    y = _bf16(O.output_projection(o16, wo))
    do, dwo = O.output_projection_backward(o16, wo, dy)
    for name, got, ref in (("y", y, ry), ("dO", _bf16(do), rdo), ("dWo", dwo, rdwo)):
        assert_rel(got, ref, name, rel_max=1e-2, rel_norm=7.5e-3)


# ------------------------------------------------------------------------------ RoPE
ROPE_L = 1024   # the split of a position into s = sh * ROPE_L + sl used by the table


def _rope_fp32(x, pos, theta, D):
    """The permute kernel's RoPE: (cos, sin)(s w_i) rebuilt in fp32 by angle addition from a
    two-level table of fp32 values computed in fp64 (hi: sh * ROPE_L * w_i, lo: sl * w_i),
    then the pair rotation in fp32 (numpy rounds each product, so this is slightly coarser
    than the kernel's fused multiply-adds) and one bf16 rounding."""
    f32 = np.float32
    w = theta ** (-2.0 * np.arange(D // 2) / D)
    sh, sl = pos // ROPE_L, pos % ROPE_L
    a, b = np.outer(sh * ROPE_L, w), np.outer(sl, w)
    a_c, a_s = np.cos(a).astype(f32), np.sin(a).astype(f32)
    b_c, b_s = np.cos(b).astype(f32), np.sin(b).astype(f32)
    cs = a_c * b_c - a_s * b_s
    sn = a_s * b_c + a_c * b_s
    lo, hi = x[..., :D // 2].astype(f32), x[..., D // 2:].astype(f32)
    cs, sn = cs[:, None, :], sn[:, None, :]
    return _bf16(np.concatenate([lo * cs - hi * sn, hi * cs + lo * sn], axis=-1)), (cs, sn, w)


def _rope_positions():
    rng = np.random.default_rng(5)
    far = rng.integers(0, 1 << 20, 2048)
    return np.unique(np.concatenate([np.arange(64), far, [(1 << 20) - 1]]))


def test_rope_bound_admits_the_two_level_table():
    """The GPU test holds RoPE to one bf16 ulp (at the exact value) + 1e-5 against the fp64
    rotation of the same bf16 input, at positions up to 2^20."""
    D, theta = 128, 500000.0
    pos = _rope_positions()
    x = synthetic.bf16_to_f64(synthetic.normal_bf16(0, synthetic.TENSOR_QKV, (pos.size, 4, D), std=1.28))
    got, (cs, sn, w) = _rope_fp32(x, pos, theta, D)
    ang = np.outer(pos, w)
    assert np.abs(cs[:, 0] - np.cos(ang)).max() < 1e-6 and np.abs(sn[:, 0] - np.sin(ang)).max() < 1e-6
    ref = O.apply_rope(x, pos, theta)
    err = np.abs(got - ref)
    assert np.all(err <= bf16_ulp(ref) + 1e-5), (err / (bf16_ulp(ref) + 1e-5)).max()


def test_rope_bound_catches_an_fp32_angle():
    """Forming the angle s * w_i itself in fp32 (instead of the fp64 table) loses it at
    large positions: the bound catches that."""
    D, theta = 128, 500000.0
    pos = _rope_positions()
    x = synthetic.bf16_to_f64(synthetic.normal_bf16(0, synthetic.TENSOR_QKV, (pos.size, 4, D), std=1.28))
    f32 = np.float32
    w = (theta ** (-2.0 * np.arange(D // 2) / D)).astype(f32)
    ang = pos.astype(f32)[:, None] * w[None, :]
    cs, sn = np.cos(ang).astype(f32)[:, None, :], np.sin(ang).astype(f32)[:, None, :]
    lo, hi = x[..., :D // 2].astype(f32), x[..., D // 2:].astype(f32)
    got = _bf16(np.concatenate([lo * cs - hi * sn, hi * cs + lo * sn], axis=-1))
    ref = O.apply_rope(x, pos, theta)
    assert np.any(np.abs(got - ref) > bf16_ulp(ref) + 1e-5)


# ------------------------------------------------------------- the fixed target bound
def test_fixed_bound_leaves_margin_at_the_8b_head_shape():
    """Outside the peaked case the GPU tests hold attention to max|err| <= max(2e-2, one bf16
    ulp) and mean|err| <= 2e-3 (the target's bound).  At the 8B head shape (S=2048, P=8,
    rank 0: 4 query heads on one KV head, q/k/v std 1.28) the kernels' roundings use about
    half of the max bound and a tenth of the mean bound."""
    S, P, H, G, D, std = 2048, 8, 32, 8, 128, 1.28
    f = lambda bits: synthetic.bf16_to_f64(bits)[0]
    q = f(synthetic.normal_bf16(0, synthetic.TENSOR_Q, (P, S, H // P, D), std=std))
    k = f(synthetic.normal_bf16(0, synthetic.TENSOR_K, (P, S, G // P, D), std=std))
    v = f(synthetic.normal_bf16(0, synthetic.TENSOR_V, (P, S, G // P, D), std=std))
    do = f(synthetic.normal_bf16(synthetic.SEED_DO, 0, (P, S, H // P, D)))
    o, _ = O.causal_attention(q, k, v)
    ref = (o,) + O.causal_attention_bwd(q, k, v, do)
    for name, got, r in zip(("o", "dq", "dk", "dv"), _simulate(q, k, v, do, _f16, _f16), ref):
        e = np.abs(got - r)
        assert (e / np.maximum(2e-2, bf16_ulp(r))).max() <= 0.6 and e.mean() <= 0.25 * 2e-3, name
