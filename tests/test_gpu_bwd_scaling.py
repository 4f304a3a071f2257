"""The attention backward at the magnitudes of a real training step.

The training step the pages describe ("Ulysses Sequence Parallelism: Training with
Million-Token Contexts", para 1) feeds the backward the gradient of a token-averaged loss,
whose entries are typically 1e-5 .. 1e-8, far below fp16's normal range (2^-14), and bf16
activations may exceed fp16's 65504.  The backward therefore scales each fp16 operand by a
power of two chosen per call.  Checked here, through the C ABI:
  - dO ~ N(0, 1e-6^2) and N(0, 1e-8^2) at the Llama-3.1-8B head shape, against the oracle
    with the 2e-2 / 2e-3 bounds applied to the gradients divided by sigma_dO (the bounds
    are then scale-invariant: a kernel that lost the small gradients fails them);
  - scaling q, k, v and dO by powers of two (q above 65504, k below fp16's normal range)
    scales dV and dK by exactly the implied factors, bit for bit, and dQ within rounding;
  - a zero dO gives zero gradients;
  - an input beyond the exponents' range is reported (ULY_ERR_RANGE), not silently clipped,
    and the plan works again once the status has been read."""
import numpy as np
import pytest
import torch

import long_context_sequence_gb300 as U
import oracle as O
import synthetic
from gpu_helpers import assert_close, bf16_ulp, dev_bf16, empty_bf16, host_f64

pytestmark = pytest.mark.gpu

S, P, H, G, D, STD = 2048, 8, 32, 8, 128, 1.28   # 8B head shape at S=2048


def _inputs(std_do=1.0):
    q = synthetic.normal_bf16(0, synthetic.TENSOR_Q, (P, S, H // P, D), std=STD)
    k = synthetic.normal_bf16(0, synthetic.TENSOR_K, (P, S, G // P, D), std=STD)
    v = synthetic.normal_bf16(0, synthetic.TENSOR_V, (P, S, G // P, D), std=STD)
    do = synthetic.normal_bf16(synthetic.SEED_DO, 0, (P, S, H // P, D), std=std_do)
    return q, k, v, do


def _scaled_bits(bits, e):
    """bf16 values times 2^e (exact while they stay normal)."""
    return synthetic.f32_to_bf16((synthetic.bf16_to_f64(bits) * 2.0 ** e).astype(np.float32))


def _fwd_bwd(plan, q, k, v, do):
    qg, kg, vg, dog = (dev_bf16(a) for a in (q, k, v, do))
    o, o_lo = empty_bf16(q.shape), empty_bf16(q.shape)
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    U.ulysses_attn_fwd(plan, qg, kg, vg, o, lse, o_lo=o_lo)
    ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    ws.fill_(0x5A)   # contents on entry must not matter
    dq, dk, dv = empty_bf16(q.shape), empty_bf16(k.shape), empty_bf16(v.shape)
    U.ulysses_attn_bwd(plan, qg, kg, vg, o, lse, dog, dq, dk, dv, ws, o_lo=o_lo)
    st = U.ulysses_sync_status(plan)
    assert st == U.ULY_OK, U.ulysses_last_error()
    return (o, o_lo, lse), (host_f64(dq), host_f64(dk), host_f64(dv))


@pytest.mark.parametrize("sigma", [1e-6, 1e-8])
def test_backward_small_upstream_gradients(sigma):
    plan = U.ulysses_plan(U.make_config(S, P, 64, H, G, D))
    q, k, v, do = _inputs(std_do=sigma)
    _, (dq, dk, dv) = _fwd_bwd(plan, q, k, v, do)
    qf, kf, vf, dof = (synthetic.bf16_to_f64(a) for a in (q, k, v, do))
    for r in range(P):
        rdq, rdk, rdv = O.causal_attention_bwd(qf[r], kf[r], vf[r], dof[r])
        for name, got, ref in (("dq", dq[r], rdq), ("dk", dk[r], rdk), ("dv", dv[r], rdv)):
            assert np.abs(ref).max() > 0
            assert_close(got / sigma, ref / sigma, "%s[rank %d] / sigma_dO (%g)" % (name, r, sigma))


def test_power_of_two_scaling_is_exact():
    """q * 2^16 (entries up to ~4e5, above fp16's 65504), k * 2^-16 (~2e-5, below fp16's
    normal range), v * 2^17, dO * 2^-20 (~1e-6).  The logits are unchanged, so the forward
    is the base case's scaled exactly (o by 2^17, lse equal), and the backward, whose fp16
    operands are normalised per call, must give dV * 2^-20 and dK * 2^13 bit for bit and dQ
    * 2^-19 up to its atomic summation order."""
    plan = U.ulysses_plan(U.make_config(S, P, 64, H, G, D))
    q, k, v, do = _inputs()
    a, b, c = 16, 17, -20
    qs, ks, vs, dos = _scaled_bits(q, a), _scaled_bits(k, -a), _scaled_bits(v, b), _scaled_bits(do, c)
    assert synthetic.bf16_to_f64(qs).max() > 65504 and np.abs(synthetic.bf16_to_f64(ks)).max() < 2.0 ** -10
    (o0, lo0, l0), (dq0, dk0, dv0) = _fwd_bwd(plan, q, k, v, do)
    (o1, lo1, l1), (dq1, dk1, dv1) = _fwd_bwd(plan, qs, ks, vs, dos)
    assert np.array_equal(host_f64(o1), host_f64(o0) * 2.0 ** b)
    assert np.array_equal(host_f64(lo1), host_f64(lo0) * 2.0 ** b)
    assert torch.equal(l1, l0)
    assert np.array_equal(dv1, dv0 * 2.0 ** c)
    assert np.array_equal(dk1, dk0 * 2.0 ** (a + b + c))
    # dQ's fp32 atomic additions (one per 128-key block) run in no fixed order.  Reordering
    # them changes the sum by the fp32 rounding of the partial sums, at most about
    # (S / 128) * 2^-24 * max|partial| <= 2^-20 max|dQ| here; where the sum cancels that
    # exceeds the bf16 spacing of the small result.  So: one bf16 step, or 2^-16 max|dQ|.
    d = np.abs(dq1 * 2.0 ** -(b + c - a) - dq0)
    bound = np.maximum(bf16_ulp(dq0), 2.0 ** -16 * np.abs(dq0).max())
    assert np.all(d <= bound) and d.mean() < 1e-4, (d.max(), d.mean(), (d / bound).max())
    # and the scaled case against the oracle, scaled back
    qf, kf, vf, dof = (synthetic.bf16_to_f64(t) for t in (qs, ks, vs, dos))
    for r in (0, P - 1):
        rdq, rdk, rdv = O.causal_attention_bwd(qf[r], kf[r], vf[r], dof[r])
        assert_close(dq1[r] * 2.0 ** -(b + c - a), rdq * 2.0 ** -(b + c - a), "dq[rank %d]" % r)
        assert_close(dk1[r] * 2.0 ** -(a + b + c), rdk * 2.0 ** -(a + b + c), "dk[rank %d]" % r)
        assert_close(dv1[r] * 2.0 ** -c, rdv * 2.0 ** -c, "dv[rank %d]" % r)


def test_zero_upstream_gradient_gives_zero_gradients():
    plan = U.ulysses_plan(U.make_config(S, P, 64, H, G, D))
    q, k, v, do = _inputs()
    _, grads = _fwd_bwd(plan, q, k, v, np.zeros_like(do))
    for g in grads:
        assert np.all(g == 0)


def test_input_beyond_the_exponent_range_is_reported():
    """q * 2^80 cannot be normalised within the exponents' range (|e| <= 60): its fp16 copy
    would saturate, and the call says so through the status word instead of returning
    clipped gradients.  Reading the status clears it and the plan works again."""
    Ss, Ps, Hs, Gs = 512, 2, 4, 2
    plan = U.ulysses_plan(U.make_config(Ss, Ps, 64, Hs, Gs, D))
    q = synthetic.normal_bf16(0, synthetic.TENSOR_Q, (Ps, Ss, Hs // Ps, D))
    k = synthetic.normal_bf16(0, synthetic.TENSOR_K, (Ps, Ss, Gs // Ps, D))
    v = synthetic.normal_bf16(0, synthetic.TENSOR_V, (Ps, Ss, Gs // Ps, D))
    do = synthetic.normal_bf16(synthetic.SEED_DO, 0, (Ps, Ss, Hs // Ps, D))
    qg, kg, vg, dog = (dev_bf16(t) for t in (q, k, v, do))
    o, lse = empty_bf16(q.shape), torch.empty((Ps, Hs // Ps, Ss), dtype=torch.float32, device="cuda")
    U.ulysses_attn_fwd(plan, qg, kg, vg, o, lse)
    assert U.ulysses_sync_status(plan) == U.ULY_OK
    ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    dq, dk, dv = empty_bf16(q.shape), empty_bf16(k.shape), empty_bf16(v.shape)
    huge = dev_bf16(_scaled_bits(q, 80))
    U.ulysses_attn_bwd(plan, huge, kg, vg, o, lse, dog, dq, dk, dv, ws)
    assert U.ulysses_sync_status(plan) == U.ULY_ERR_RANGE
    assert "range" in U.ulysses_last_error()
    assert U.ulysses_sync_status(plan) == U.ULY_OK
    U.ulysses_attn_bwd(plan, qg, kg, vg, o, lse, dog, dq, dk, dv, ws)
    assert U.ulysses_sync_status(plan) == U.ULY_OK
    qf, kf, vf, dof = (synthetic.bf16_to_f64(t) for t in (q, k, v, do))
    for r in range(Ps):
        rdq, rdk, rdv = O.causal_attention_bwd(qf[r], kf[r], vf[r], dof[r])
        assert_close(host_f64(dq)[r], rdq, "dq after a reported range error")
        assert_close(host_f64(dk)[r], rdk, "dk after a reported range error")
        assert_close(host_f64(dv)[r], rdv, "dv after a reported range error")
