"""GPU parity of every step of the Ulysses block against the fp64 CPU oracle, at sizes the
oracle finishes in seconds (several tiles plus ragged tails).  Calls go through the C ABI
(ctypes binding); inputs come from the seeded generator on the host."""
import math

import numpy as np
import pytest
import torch

import long_context_sequence_gb300 as U
import oracle as O
import synthetic
from tolerances import assert_within as _assert_within, peaked_bounds as _peaked_bounds
from gpu_helpers import (assert_close, assert_close_f32, bf16_ulp_distance, dev_bf16, empty_bf16,
                         host_bits, host_f64)

pytestmark = pytest.mark.gpu


def _plan(S, P, H, G, D, hidden=64, theta=0.0, **kw):
    return U.ulysses_plan(U.make_config(S, P, hidden, H, G, D, rope_theta=theta, **kw))


def _ok(plan):
    st = U.ulysses_sync_status(plan)
    assert st == U.ULY_OK, U.ulysses_last_error()


PERMUTE_CASES = [(1024, 4, 8, 8, 64), (2048, 8, 32, 8, 128), (1000, 4, 8, 4, 128),
                 (8, 8, 8, 8, 64), (24, 1, 4, 2, 64), (4096, 2, 4, 2, 128),
                 (4096, 16, 32, 16, 128),   # 16 ranks, one KV head each
                 (2048, 4, 32, 4, 128)]     # GQA 8:1


@pytest.mark.parametrize("S,P,H,G,D", PERMUTE_CASES)
def test_permutes_bit_exact(S, P, H, G, D):
    plan = _plan(S, P, H, G, D)
    x = synthetic.normal_bf16(0, synthetic.TENSOR_QKV, (S, H + 2 * G, D))
    xg = dev_bf16(x)
    q, k, v = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, G // P, D)), empty_bf16((P, S, G // P, D))
    U.ulysses_seq_to_head(plan, xg, q, k, v)
    oq, ok, ov = O.seq_to_head(x, P, H, G)
    _ok(plan)
    assert np.array_equal(host_bits(q), oq)
    assert np.array_equal(host_bits(k), ok)
    assert np.array_equal(host_bits(v), ov)
    # head -> seq restores the sequence sharding (query part and KV part)
    back_q = empty_bf16((P, S // P, H, D))
    back_k = empty_bf16((P, S // P, G, D))
    U.ulysses_head_to_seq(plan, q, H, back_q)
    U.ulysses_head_to_seq(plan, k, G, back_k)
    _ok(plan)
    assert np.array_equal(host_bits(back_q), O.head_to_seq(oq, P))
    assert np.array_equal(host_bits(back_q).reshape(S, H, D), x[:, :H])
    assert np.array_equal(host_bits(back_k).reshape(S, G, D), x[:, H:H + G])
    # seq -> head of a single tensor (the path of dO)
    q2 = empty_bf16((P, S, H // P, D))
    U.ulysses_seq_to_head_heads(plan, back_q, H, q2)
    _ok(plan)
    assert np.array_equal(host_bits(q2), oq)
    expect = S * (H + 2 * G) * D * 4 + 2 * S * H * D * 4 + S * G * D * 4
    assert U.ulysses_bytes_moved(plan) == expect


def test_seq_to_head_fp32_input_rounds_to_nearest_even():
    S, P, H, G, D = 512, 4, 8, 4, 64
    plan = _plan(S, P, H, G, D)
    x = synthetic.normal_f64(0, synthetic.TENSOR_QKV, (S, H + 2 * G, D)).astype(np.float32)
    q, k, v = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, G // P, D)), empty_bf16((P, S, G // P, D))
    U.ulysses_seq_to_head(plan, torch.from_numpy(x).cuda(), q, k, v)
    _ok(plan)
    oq, ok, ov = O.seq_to_head(synthetic.f32_to_bf16(x), P, H, G)
    assert np.array_equal(host_bits(q), oq) and np.array_equal(host_bits(k), ok)
    assert np.array_equal(host_bits(v), ov)


@pytest.mark.parametrize("S,P,H,G,D,theta", [(2048, 8, 32, 8, 128, 500000.0),
                                             (3000, 4, 8, 4, 64, 10000.0)])
def test_seq_to_head_rope_within_one_ulp(S, P, H, G, D, theta):
    plan = _plan(S, P, H, G, D, theta=theta)
    x = synthetic.normal_bf16(0, synthetic.TENSOR_QKV, (S, H + 2 * G, D), std=1.28)
    q, k, v = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, G // P, D)), empty_bf16((P, S, G // P, D))
    U.ulysses_seq_to_head(plan, dev_bf16(x), q, k, v, apply_rope=True)
    _ok(plan)
    xf = synthetic.bf16_to_f64(x)
    pos = np.arange(S)
    rot = np.concatenate([O.apply_rope(xf[:, :H + G], pos, theta), xf[:, H + G:]], axis=1)
    oq, ok, ov = O.seq_to_head(rot, P, H, G)
    for got, ref in ((q, oq), (k, ok)):
        # fp32 rotation then one bf16 rounding: within one bf16 ulp of the exact value
        # (ulp taken at the exact value's magnitude) plus the fp32 rotation error
        err = np.abs(host_f64(got) - ref)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
        bound = ulp + 1e-5
        assert np.all(err <= bound), "RoPE error %.3g ulp" % (err / ulp).max()
    assert np.array_equal(host_bits(v), O.seq_to_head(x, P, H, G)[2])   # v untouched


@pytest.mark.parametrize("S,hidden,C", [(1024, 512, 1536), (1000, 200, 640), (2048, 4096, 6144),
                                        (130, 64, 256)])
def test_qkv_projection(S, hidden, C):
    D = 64
    n_heads = C // D
    G = n_heads // 6 if n_heads % 6 == 0 else 1
    H = n_heads - 2 * G
    plan = _plan(S, 1, H, G, D, hidden=hidden)
    x = synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, hidden))
    w = synthetic.normal_bf16(0, synthetic.TENSOR_W, (C, hidden), std=0.02)
    out = empty_bf16((S, C))
    U.ulysses_qkv_proj(plan, dev_bf16(x), dev_bf16(w), out)
    _ok(plan)
    ref = O.qkv_projection(synthetic.bf16_to_f64(x), synthetic.bf16_to_f64(w))
    got = host_f64(out)
    assert_close(got, ref, "qkv")
    # each value is the fp32 sum rounded once to bf16: within one bf16 rounding step
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-4)


def _attn_inputs(S, P, H, G, D, std):
    q = synthetic.normal_bf16(0, synthetic.TENSOR_Q, (P, S, H // P, D), std=std)
    k = synthetic.normal_bf16(0, synthetic.TENSOR_K, (P, S, G // P, D), std=std)
    v = synthetic.normal_bf16(0, synthetic.TENSOR_V, (P, S, G // P, D), std=std)
    return q, k, v


ATTN_CASES = [  # S, P, H, G, D, std of q/k/v
    (1024, 4, 8, 8, 64, 0.45),       # tiny block shape (hidden 512, W std 0.02)
    (2048, 8, 32, 8, 128, 1.28),     # Llama-3.1-8B head shape (hidden 4096, W std 0.02)
    (1000, 4, 8, 4, 128, 1.0),       # ragged tail, GQA 2:1
    (384, 2, 4, 2, 64, 1.0),         # odd number of 128-row tiles
    (130, 1, 2, 1, 128, 1.0),        # one rank, tail of 2 rows
    (1002, 2, 4, 2, 64, 1.0),        # two ranks, S % 4 = 2 (the dQ accumulator pads rows)
    (8, 8, 8, 8, 64, 1.0),           # one token per rank
    (4096, 16, 32, 16, 128, 1.0),    # 16 ranks: two query heads and one KV head per rank
    (2048, 4, 32, 4, 128, 1.28),     # GQA 8:1
    (1024, 4, 8, 4, 128, 3.0),       # peaked softmax: logits with std ~9
]


PEAKED = 3.0   # q/k std at which the logits' std is ~9: a sharply peaked softmax


@pytest.mark.parametrize("S,P,H,G,D,std", ATTN_CASES)
def test_attention_forward(S, P, H, G, D, std):
    plan = _plan(S, P, H, G, D)
    q, k, v = _attn_inputs(S, P, H, G, D, std)
    o = empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    U.ulysses_attn_fwd(plan, dev_bf16(q), dev_bf16(k), dev_bf16(v), o, lse)
    _ok(plan)
    ro, rl = O.ulysses_attention(*(synthetic.bf16_to_f64(a) for a in (q, k, v)))
    if std >= PEAKED:
        qf, kf, vf = (synthetic.bf16_to_f64(a) for a in (q, k, v))
        dof = np.zeros_like(qf)
        for r in range(P):
            bo = _peaked_bounds(qf[r], kf[r], vf[r], dof[r], H, G)[0]
            _assert_within(host_f64(o)[r], ro[r], bo, "o[rank %d]" % r)
    else:
        assert_close(host_f64(o), ro, "o")
    assert_close_f32(host_f64(lse), rl, "lse")
    # row 0 of every head is exactly V[0] of its KV head
    vo = synthetic.bf16_to_f64(v)
    grp = H // G
    for h in range(H // P):
        assert np.array_equal(host_f64(o)[:, 0, h], vo[:, 0, h // grp])


@pytest.mark.parametrize("S,P,H,G,D,std", ATTN_CASES)
def test_attention_backward(S, P, H, G, D, std):
    plan = _plan(S, P, H, G, D)
    q, k, v = _attn_inputs(S, P, H, G, D, std)
    do = synthetic.normal_bf16(synthetic.SEED_DO, 0, (P, S, H // P, D))
    qg, kg, vg, dog = (dev_bf16(a) for a in (q, k, v, do))
    o, o_lo = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    if std >= PEAKED:
        # The backward forms D = dO . O from the O it is given.  In the peaked regime the
        # forward's own O error (bf16 P, tested above) would flow through D, so here the
        # backward gets the exact forward state: O as bf16 plus its bf16 residual, and lse.
        ro, rl = O.ulysses_attention(*(synthetic.bf16_to_f64(a) for a in (q, k, v)))
        hi = synthetic.f32_to_bf16(ro.astype(np.float32))
        lo = synthetic.f32_to_bf16((ro - synthetic.bf16_to_f64(hi)).astype(np.float32))
        o.copy_(dev_bf16(hi))
        o_lo.copy_(dev_bf16(lo))
        lse.copy_(torch.from_numpy(rl.astype(np.float32)).cuda())
    else:
        U.ulysses_attn_fwd(plan, qg, kg, vg, o, lse, o_lo=o_lo)
    ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)   # contents on entry must not matter
    dq, dk, dv = empty_bf16(q.shape), empty_bf16(k.shape), empty_bf16(v.shape)
    U.ulysses_attn_bwd(plan, qg, kg, vg, o, lse, dog, dq, dk, dv, ws, o_lo=o_lo)
    _ok(plan)
    qf, kf, vf, dof = (synthetic.bf16_to_f64(a) for a in (q, k, v, do))
    for r in range(P):
        rdq, rdk, rdv = O.causal_attention_bwd(qf[r], kf[r], vf[r], dof[r])
        if std >= PEAKED:
            _, bq, bk, bv = _peaked_bounds(qf[r], kf[r], vf[r], dof[r], H, G)
            _assert_within(host_f64(dq)[r], rdq, bq, "dq[rank %d]" % r)
            _assert_within(host_f64(dk)[r], rdk, bk, "dk[rank %d]" % r)
            _assert_within(host_f64(dv)[r], rdv, bv, "dv[rank %d]" % r)
            continue
        assert_close(host_f64(dq)[r], rdq, "dq[rank %d]" % r)
        assert_close(host_f64(dk)[r], rdk, "dk[rank %d]" % r)
        assert_close(host_f64(dv)[r], rdv, "dv[rank %d]" % r)


def test_block_forward_end_to_end_tiny():
    """The tiny block (S=1024, P=4, hidden 512, 8/8 heads, D=64) from X and W_qkv to the
    sequence-sharded output, against the oracle's unrounded fp64 pipeline."""
    S, P, hidden, H, G, D = 1024, 4, 512, 8, 8, 64
    plan = _plan(S, P, H, G, D, hidden=hidden)
    x = synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, hidden))
    w = synthetic.normal_bf16(0, synthetic.TENSOR_W, ((H + 2 * G) * D, hidden), std=0.02)
    qkv = empty_bf16((P, S // P, H + 2 * G, D))
    q, k, v = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, G // P, D)), empty_bf16((P, S, G // P, D))
    o = empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    o_seq = empty_bf16((P, S // P, H, D))
    U.ulysses_qkv_proj(plan, dev_bf16(x), dev_bf16(w), qkv)
    U.ulysses_seq_to_head(plan, qkv, q, k, v)
    U.ulysses_attn_fwd(plan, q, k, v, o, lse)
    U.ulysses_head_to_seq(plan, o, H, o_seq)
    _ok(plan)
    ro, rl, _ = O.ulysses_block_forward(synthetic.bf16_to_f64(x), synthetic.bf16_to_f64(w),
                                        P, H, G, D)
    assert_close(host_f64(o_seq), ro, "o_seq")
    assert_close_f32(host_f64(lse), rl, "lse")


def test_block_forward_end_to_end_rope_8b_shape():
    """8B-shaped block with RoPE (theta 500000) at S=2048, P=8, end to end."""
    S, P, hidden, H, G, D, theta = 2048, 8, 4096, 32, 8, 128, 500000.0
    plan = _plan(S, P, H, G, D, hidden=hidden, theta=theta)
    x = synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, hidden))
    w = synthetic.normal_bf16(0, synthetic.TENSOR_W, ((H + 2 * G) * D, hidden), std=0.02)
    qkv = empty_bf16((P, S // P, H + 2 * G, D))
    q, k, v = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, G // P, D)), empty_bf16((P, S, G // P, D))
    o = empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    o_seq = empty_bf16((P, S // P, H, D))
    U.ulysses_qkv_proj(plan, dev_bf16(x), dev_bf16(w), qkv)
    U.ulysses_seq_to_head(plan, qkv, q, k, v, apply_rope=True)
    U.ulysses_attn_fwd(plan, q, k, v, o, lse)
    U.ulysses_head_to_seq(plan, o, H, o_seq)
    _ok(plan)
    ro, rl, _ = O.ulysses_block_forward(synthetic.bf16_to_f64(x), synthetic.bf16_to_f64(w),
                                        P, H, G, D, theta)
    # Against the unrounded fp64 pipeline the bf16 storage of q/k/v (relative 2^-9) moves
    # the logits of this 8B-scale block (std ~1.6) by up to ~1e-2, so the end-to-end
    # bound is 5e-2 max / 2e-3 mean; each stage alone meets 2e-2 (tests above).
    assert_close(host_f64(o_seq), ro, "o_seq", max_abs=5e-2)
    assert_close_f32(host_f64(lse), rl, "lse", max_abs=5e-2)


def test_empty_sequence_is_a_no_op():
    plan = _plan(0, 4, 8, 8, 64)
    z = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    U.ulysses_seq_to_head(plan, z, z, z, z)
    U.ulysses_attn_fwd(plan, z, z, z, z, torch.empty(0, device="cuda"))
    U.ulysses_head_to_seq(plan, z, 8, z)
    _ok(plan)


def test_misaligned_pointer_is_rejected_before_launch():
    S, P, H, G, D = 256, 2, 4, 2, 64
    plan = _plan(S, P, H, G, D)
    buf = torch.zeros(P * S * (H // P) * D + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(U.UlyssesError) as ei:
        U.ulysses_attn_fwd(plan, buf.data_ptr() + 2, buf.data_ptr(), buf.data_ptr(),
                           buf.data_ptr(), buf.data_ptr())
    assert ei.value.status == U.ULY_ERR_INVALID_ARG
    _ok(plan)


def test_forward_rounding_residual_and_backward_without_it():
    """o + o_lo reproduces the fp32 output to ~16 bits; the backward also runs without
    o_lo (row terms from the bf16 o alone) and still meets the bound on the tiny shape."""
    S, P, H, G, D = 1024, 4, 8, 8, 64
    plan = _plan(S, P, H, G, D)
    q, k, v = _attn_inputs(S, P, H, G, D, 0.45)
    do = synthetic.normal_bf16(synthetic.SEED_DO, 0, (P, S, H // P, D))
    qg, kg, vg, dog = (dev_bf16(a) for a in (q, k, v, do))
    o, o_lo = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    U.ulysses_attn_fwd(plan, qg, kg, vg, o, lse, o_lo=o_lo)
    ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    dq, dk, dv = empty_bf16(q.shape), empty_bf16(k.shape), empty_bf16(v.shape)
    U.ulysses_attn_bwd(plan, qg, kg, vg, o, lse, dog, dq, dk, dv, ws)
    _ok(plan)
    qf, kf, vf, dof = (synthetic.bf16_to_f64(a) for a in (q, k, v, do))
    ro, _ = O.ulysses_attention(qf, kf, vf)
    hi, lo = host_f64(o), host_f64(o_lo)
    assert np.all(np.abs(lo) <= np.abs(hi) * 2.0 ** -8 * 1.01 + 1e-30)   # about half a bf16 ulp
    assert np.abs(hi + lo - ro).max() < np.abs(hi - ro).max()     # closer than o alone
    assert np.abs(hi + lo - ro).max() < 2e-3
    for r in range(P):
        rdq, rdk, rdv = O.causal_attention_bwd(qf[r], kf[r], vf[r], dof[r])
        assert_close(host_f64(dq)[r], rdq, "dq[rank %d] without o_lo" % r)
        assert_close(host_f64(dk)[r], rdk, "dk[rank %d] without o_lo" % r)
        assert_close(host_f64(dv)[r], rdv, "dv[rank %d] without o_lo" % r)
