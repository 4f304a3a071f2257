"""GPU parity of the block's training-step completion against the fp64 oracle: the
gradient head->seq all-to-all (with and without the RoPE backward), the QKV projection
backward (dx, dw), the whole block's gradients from dO to dx and dw, and the output
projection fused with the head->seq all-to-all (forward and backward, and the whole layer
from x to y and from dy to dx, dw, dwo).  Calls go through
the C ABI (ctypes binding); inputs come from the seeded generator on the host."""
import numpy as np
import pytest
import torch

import long_context_sequence_gb300 as U
import oracle as O
import synthetic
from tolerances import assert_rel as _assert_rel
from gpu_helpers import assert_close, dev_bf16, empty_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu


def _plan(S, P, H, G, D, hidden=64, theta=0.0):
    return U.ulysses_plan(U.make_config(S, P, hidden, H, G, D, rope_theta=theta))


def _ok(plan):
    st = U.ulysses_sync_status(plan)
    assert st == U.ULY_OK, U.ulysses_last_error()


def _grads(S, P, H, G, D):
    dq = synthetic.normal_bf16(synthetic.SEED_DO, synthetic.TENSOR_Q, (P, S, H // P, D))
    dk = synthetic.normal_bf16(synthetic.SEED_DO, synthetic.TENSOR_K, (P, S, G // P, D))
    dv = synthetic.normal_bf16(synthetic.SEED_DO, synthetic.TENSOR_V, (P, S, G // P, D))
    return dq, dk, dv


GRAD_PERMUTE_CASES = [(1024, 4, 8, 8, 64), (2048, 8, 32, 8, 128), (1000, 4, 8, 4, 128),
                      (8, 8, 8, 8, 64), (24, 1, 4, 2, 64)]


@pytest.mark.parametrize("S,P,H,G,D", GRAD_PERMUTE_CASES)
def test_gradient_head_to_seq_bit_exact_and_inverse(S, P, H, G, D):
    plan = _plan(S, P, H, G, D)
    dq, dk, dv = _grads(S, P, H, G, D)
    out = empty_bf16((P, S // P, H + 2 * G, D))
    U.ulysses_head_to_seq_qkv(plan, dev_bf16(dq), dev_bf16(dk), dev_bf16(dv), out)
    _ok(plan)
    got = host_bits(out).reshape(S, H + 2 * G, D)
    assert np.array_equal(got, O.head_to_seq_qkv(dq, dk, dv, P))
    # seq->head of the result gives the three inputs back
    q2, k2, v2 = empty_bf16(dq.shape), empty_bf16(dk.shape), empty_bf16(dv.shape)
    U.ulysses_seq_to_head(plan, out, q2, k2, v2)
    _ok(plan)
    for a, b in ((q2, dq), (k2, dk), (v2, dv)):
        assert np.array_equal(host_bits(a), b)


@pytest.mark.parametrize("S,P,H,G,D,theta", [(2048, 8, 32, 8, 128, 500000.0),
                                             (1000, 4, 8, 4, 64, 10000.0)])
def test_gradient_head_to_seq_rope_backward(S, P, H, G, D, theta):
    """q and k parts turned back by their angles within one bf16 rounding (+1e-5 for the
    fp32 angle), v bit for bit."""
    plan = _plan(S, P, H, G, D, theta=theta)
    dq, dk, dv = _grads(S, P, H, G, D)
    out = empty_bf16((P, S // P, H + 2 * G, D))
    U.ulysses_head_to_seq_qkv(plan, dev_bf16(dq), dev_bf16(dk), dev_bf16(dv), out,
                              apply_rope=True)
    _ok(plan)
    got = host_f64(out).reshape(S, H + 2 * G, D)
    plain = synthetic.bf16_to_f64(O.head_to_seq_qkv(dq, dk, dv, P))
    ref = O.rope_backward(plain[:, :H + G], np.arange(S), theta)
    err = np.abs(got[:, :H + G] - ref)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    assert np.all(err <= ulp + 1e-5), "RoPE backward error %.3g ulp" % (err / ulp).max()
    assert np.array_equal(host_bits(out).reshape(S, H + 2 * G, D)[:, H + G:],
                          O.head_to_seq_qkv(dq, dk, dv, P)[:, H + G:])
    # forward then backward rotation is the identity (up to the two roundings)
    fwd = O.apply_rope(ref, np.arange(S), theta)
    assert np.abs(fwd - plain[:, :H + G]).max() < 1e-9


@pytest.mark.parametrize("S,hidden,C", [(1024, 512, 1536), (1000, 200, 640), (2048, 4096, 6144),
                                        (130, 64, 256), (4096, 256, 384)])
def test_qkv_projection_backward(S, hidden, C):
    D = 64
    n_heads = C // D
    G = n_heads // 6 if n_heads % 6 == 0 else 1
    H = n_heads - 2 * G
    plan = _plan(S, 1, H, G, D, hidden=hidden)
    x = synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, hidden))
    w = synthetic.normal_bf16(0, synthetic.TENSOR_W, (C, hidden), std=0.02)
    dy = synthetic.normal_bf16(synthetic.SEED_DO, synthetic.TENSOR_QKV, (S, C))
    dx = empty_bf16((S, hidden))
    dw = torch.empty((C, hidden), dtype=torch.float32, device="cuda")
    U.ulysses_qkv_proj_bwd(plan, dev_bf16(x), dev_bf16(w), dev_bf16(dy), dx, dw)
    _ok(plan)
    xf, wf, dyf = (synthetic.bf16_to_f64(a) for a in (x, w, dy))
    rdx, rdw = O.qkv_projection_backward(xf, wf, dyf)
    gdx, gdw = host_f64(dx), host_f64(dw)
    # dx: the fp32 sum rounded once to bf16
    assert np.all(np.abs(gdx - rdx) <= np.abs(rdx) * 2.0 ** -8 + 1e-4)
    # dw: fp32 sum over the S tokens; bounded by K u sum |dy||x| with u = 2^-24 and K <= 2^12
    absdot = np.abs(dyf).T @ np.abs(xf)
    bound = absdot * 2.0 ** -12 + 1e-6
    assert np.all(np.abs(gdw - rdw) <= bound), (np.abs(gdw - rdw) / bound).max()
    # either output alone
    dx2 = empty_bf16((S, hidden))
    U.ulysses_qkv_proj_bwd(plan, dev_bf16(x), dev_bf16(w), dev_bf16(dy), dx2, None)
    dw2 = torch.empty((C, hidden), dtype=torch.float32, device="cuda")
    U.ulysses_qkv_proj_bwd(plan, dev_bf16(x), dev_bf16(w), dev_bf16(dy), None, dw2)
    _ok(plan)
    assert torch.equal(dx2, dx) and torch.equal(dw2, dw)


def _training_step(S, P, hidden, H, G, D, theta):
    plan = _plan(S, P, H, G, D, hidden=hidden, theta=theta)
    C = (H + 2 * G) * D
    x = synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, hidden))
    w = synthetic.normal_bf16(0, synthetic.TENSOR_W, (C, hidden), std=0.02)
    do_seq = synthetic.normal_bf16(synthetic.SEED_DO, 0, (S, H, D))
    xg, wg = dev_bf16(x), dev_bf16(w)
    qkv = empty_bf16((P, S // P, H + 2 * G, D))
    q, k, v = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, G // P, D)), empty_bf16((P, S, G // P, D))
    o, o_lo = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    do = empty_bf16((P, S, H // P, D))
    dq, dk, dv = empty_bf16(q.shape), empty_bf16(k.shape), empty_bf16(v.shape)
    dqkv = empty_bf16((P, S // P, H + 2 * G, D))
    dx = empty_bf16((S, hidden))
    dw = torch.empty((C, hidden), dtype=torch.float32, device="cuda")
    ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    rope = theta > 0
    U.ulysses_qkv_proj(plan, xg, wg, qkv)
    U.ulysses_seq_to_head(plan, qkv, q, k, v, apply_rope=rope)
    U.ulysses_attn_fwd(plan, q, k, v, o, lse, o_lo=o_lo)
    U.ulysses_seq_to_head_heads(plan, dev_bf16(do_seq), H, do)
    U.ulysses_attn_bwd(plan, q, k, v, o, lse, do, dq, dk, dv, ws, o_lo=o_lo)
    U.ulysses_head_to_seq_qkv(plan, dq, dk, dv, dqkv, apply_rope=rope)
    U.ulysses_qkv_proj_bwd(plan, xg, wg, dqkv, dx, dw)
    _ok(plan)
    rdx, rdw, rdqkv = O.ulysses_block_backward(
        synthetic.bf16_to_f64(x), synthetic.bf16_to_f64(w), synthetic.bf16_to_f64(do_seq),
        P, H, G, D, theta)
    _assert_rel(host_f64(dqkv).reshape(S, H + 2 * G, D), rdqkv, "dqkv")
    _assert_rel(host_f64(dx), rdx, "dx")
    _assert_rel(host_f64(dw), rdw, "dw")


def test_training_step_end_to_end_tiny():
    """Tiny block (S=1024, P=4, hidden 512, 8/8 heads, D=64): dO -> dx, dw."""
    _training_step(1024, 4, 512, 8, 8, 64, 0.0)


def test_training_step_end_to_end_rope_8b_shape():
    """8B-shaped block with RoPE (theta 500000) at S=2048, P=8: dO -> dx, dw."""
    _training_step(2048, 8, 4096, 32, 8, 128, 500000.0)


def test_training_step_empty_sequence():
    plan = _plan(0, 4, 8, 8, 64)
    z = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    U.ulysses_head_to_seq_qkv(plan, z, z, z, z)
    U.ulysses_qkv_proj_bwd(plan, z, z, z, z, torch.empty(0, device="cuda"))
    _ok(plan)


# ----------------------------------------------------- output projection (fused head->seq)
O_PROJ_CASES = [  # S, P, H, D, hidden
    (1024, 4, 8, 64, 512),       # tiny block
    (2048, 8, 32, 128, 4096),    # Llama-3.1-8B shape
    (1000, 4, 8, 128, 200),      # ragged S and hidden
    (384, 2, 6, 64, 384),        # H*D = 384: the last N tile runs past the head layout
    (130, 1, 2, 128, 64),        # one rank
]


def _o_proj_inputs(S, P, H, D, hidden):
    o = synthetic.normal_bf16(0, synthetic.TENSOR_Q, (P, S, H // P, D))
    wo = synthetic.normal_bf16(0, synthetic.TENSOR_WO, (hidden, H * D), std=0.02)
    dy = synthetic.normal_bf16(synthetic.SEED_DO, synthetic.TENSOR_WO, (S, hidden))
    return o, wo, dy


@pytest.mark.parametrize("S,P,H,D,hidden", O_PROJ_CASES)
def test_o_proj_reads_the_head_layout(S, P, H, D, hidden):
    plan = _plan(S, P, H, P, D, hidden=hidden)
    o, wo, _ = _o_proj_inputs(S, P, H, D, hidden)
    y = empty_bf16((S, hidden))
    U.ulysses_o_proj(plan, dev_bf16(o), dev_bf16(wo), y)
    _ok(plan)
    o_seq = synthetic.bf16_to_f64(O.head_to_seq(o, P)).reshape(S, H, D)
    ref = O.output_projection(o_seq, synthetic.bf16_to_f64(wo))
    got = host_f64(y)
    assert_close(got, ref, "y")
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-4)


@pytest.mark.parametrize("S,P,H,D,hidden", O_PROJ_CASES)
def test_o_proj_backward_writes_the_head_layout(S, P, H, D, hidden):
    plan = _plan(S, P, H, P, D, hidden=hidden)
    o, wo, dy = _o_proj_inputs(S, P, H, D, hidden)
    do = empty_bf16((P, S, H // P, D))
    dwo = torch.empty((hidden, H * D), dtype=torch.float32, device="cuda")
    U.ulysses_o_proj_bwd(plan, dev_bf16(o), dev_bf16(wo), dev_bf16(dy), do, dwo)
    _ok(plan)
    of = synthetic.bf16_to_f64(O.head_to_seq(o, P)).reshape(S, H, D)
    wof, dyf = synthetic.bf16_to_f64(wo), synthetic.bf16_to_f64(dy)
    rdo, rdwo = O.output_projection_backward(of, wof, dyf)
    # head layout: rank r2 holds heads r2*H/P .. of every token
    rdo_head = rdo.reshape(S, P, H // P, D).transpose(1, 0, 2, 3)
    gdo = host_f64(do)
    assert np.all(np.abs(gdo - rdo_head) <= np.abs(rdo_head) * 2.0 ** -8 + 1e-4)
    absdot = np.abs(dyf).T @ np.abs(of.reshape(S, H * D))
    bound = absdot * 2.0 ** -12 + 1e-6
    assert np.all(np.abs(host_f64(dwo) - rdwo) <= bound)
    # either output alone
    do2 = empty_bf16((P, S, H // P, D))
    U.ulysses_o_proj_bwd(plan, dev_bf16(o), dev_bf16(wo), dev_bf16(dy), do2, None)
    dwo2 = torch.empty((hidden, H * D), dtype=torch.float32, device="cuda")
    U.ulysses_o_proj_bwd(plan, dev_bf16(o), dev_bf16(wo), dev_bf16(dy), None, dwo2)
    _ok(plan)
    assert torch.equal(do2, do) and torch.equal(dwo2, dwo)


def _layer_step(S, P, hidden, H, G, D, theta):
    """Whole block with the fused output projection, forward and training gradients."""
    plan = _plan(S, P, H, G, D, hidden=hidden, theta=theta)
    C = (H + 2 * G) * D
    x = synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, hidden))
    w = synthetic.normal_bf16(0, synthetic.TENSOR_W, (C, hidden), std=0.02)
    wo = synthetic.normal_bf16(0, synthetic.TENSOR_WO, (hidden, H * D), std=0.02)
    dy = synthetic.normal_bf16(synthetic.SEED_DO, synthetic.TENSOR_WO, (S, hidden))
    xg, wg, wog = dev_bf16(x), dev_bf16(w), dev_bf16(wo)
    qkv = empty_bf16((P, S // P, H + 2 * G, D))
    q, k, v = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, G // P, D)), empty_bf16((P, S, G // P, D))
    o, o_lo = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    y = empty_bf16((S, hidden))
    do = empty_bf16((P, S, H // P, D))
    dwo = torch.empty((hidden, H * D), dtype=torch.float32, device="cuda")
    dq, dk, dv = empty_bf16(q.shape), empty_bf16(k.shape), empty_bf16(v.shape)
    dqkv = empty_bf16((P, S // P, H + 2 * G, D))
    dx = empty_bf16((S, hidden))
    dw = torch.empty((C, hidden), dtype=torch.float32, device="cuda")
    ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    rope = theta > 0
    U.ulysses_qkv_proj(plan, xg, wg, qkv)
    U.ulysses_seq_to_head(plan, qkv, q, k, v, apply_rope=rope)
    U.ulysses_attn_fwd(plan, q, k, v, o, lse, o_lo=o_lo)
    U.ulysses_o_proj(plan, o, wog, y)
    U.ulysses_o_proj_bwd(plan, o, wog, dev_bf16(dy), do, dwo)
    U.ulysses_attn_bwd(plan, q, k, v, o, lse, do, dq, dk, dv, ws, o_lo=o_lo)
    U.ulysses_head_to_seq_qkv(plan, dq, dk, dv, dqkv, apply_rope=rope)
    U.ulysses_qkv_proj_bwd(plan, xg, wg, dqkv, dx, dw)
    _ok(plan)
    xf, wf, wof, dyf = (synthetic.bf16_to_f64(a) for a in (x, w, wo, dy))
    ry, _, _ = O.ulysses_layer_forward(xf, wf, wof, P, H, G, D, theta)
    rdx, rdw, rdwo, _ = O.ulysses_layer_backward(xf, wf, wof, dyf, P, H, G, D, theta)
    _assert_rel(host_f64(y), ry, "y")
    _assert_rel(host_f64(dwo), rdwo, "dwo")
    _assert_rel(host_f64(dx), rdx, "dx")
    _assert_rel(host_f64(dw), rdw, "dw")


def test_layer_end_to_end_tiny():
    """Tiny block with the output projection (hidden 512): x -> y and dy -> dx, dw, dwo."""
    _layer_step(1024, 4, 512, 8, 8, 64, 0.0)


def test_layer_end_to_end_rope_8b_shape():
    """8B-shaped block with RoPE and the output projection at S=2048, P=8."""
    _layer_step(2048, 8, 4096, 32, 8, 128, 500000.0)
