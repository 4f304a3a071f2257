"""Failure detection without a GPU fault: a plan flag makes the forward (or backward)
kernel's MMA issuer withhold one completion signal, so the element-wise warps' bounded
waits run out.
The kernel must end on its own, report ULY_ERR_TIMEOUT through the plan's status word,
and leave the CUDA context usable for the next plan."""
import numpy as np
import pytest
import torch

import long_context_sequence_gb300 as U
import oracle as O
import synthetic
from gpu_helpers import assert_close, assert_close_f32, dev_bf16, empty_bf16, host_f64

pytestmark = pytest.mark.gpu


def _fwd(plan, S, P, H, G, D):
    q = synthetic.normal_bf16(0, synthetic.TENSOR_Q, (P, S, H // P, D))
    k = synthetic.normal_bf16(0, synthetic.TENSOR_K, (P, S, G // P, D))
    v = synthetic.normal_bf16(0, synthetic.TENSOR_V, (P, S, G // P, D))
    o = empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    U.ulysses_attn_fwd(plan, dev_bf16(q), dev_bf16(k), dev_bf16(v), o, lse)
    return (q, k, v), o, lse


def test_stalled_wait_times_out_and_context_survives():
    S, P, H, G, D = 2048, 2, 4, 2, 128
    bad = U.ulysses_plan(U.make_config(S, P, 64, H, G, D, flags=U.ULY_FLAG_INJECT_STALL,
                                       wait_timeout_ms=100))
    _fwd(bad, S, P, H, G, D)
    assert U.ulysses_sync_status(bad) == U.ULY_ERR_TIMEOUT
    assert "ran past" in U.ulysses_last_error()
    assert U.ulysses_sync_status(bad) == U.ULY_OK       # reading the status cleared it
    bad.close()
    good = U.ulysses_plan(U.make_config(S, P, 64, H, G, D))
    (q, k, v), o, lse = _fwd(good, S, P, H, G, D)
    assert U.ulysses_sync_status(good) == U.ULY_OK
    ro, rl = O.ulysses_attention(*(synthetic.bf16_to_f64(a) for a in (q, k, v)))
    assert_close(host_f64(o), ro, "o after a timed-out launch")
    assert_close_f32(host_f64(lse), rl, "lse after a timed-out launch")


def test_stalled_backward_times_out_and_context_survives():
    """The backward's S^T issuer withholds its first commit in block 0: every wait in the
    kernel is bounded, so the call ends, reports ULY_ERR_TIMEOUT, and a fresh plan then
    gives oracle-correct gradients."""
    S, P, H, G, D = 1024, 2, 4, 2, 128
    good = U.ulysses_plan(U.make_config(S, P, 64, H, G, D))
    q = synthetic.normal_bf16(0, synthetic.TENSOR_Q, (P, S, H // P, D))
    k = synthetic.normal_bf16(0, synthetic.TENSOR_K, (P, S, G // P, D))
    v = synthetic.normal_bf16(0, synthetic.TENSOR_V, (P, S, G // P, D))
    do = synthetic.normal_bf16(synthetic.SEED_DO, 0, (P, S, H // P, D))
    qg, kg, vg, dog = (dev_bf16(a) for a in (q, k, v, do))
    o, o_lo = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    U.ulysses_attn_fwd(good, qg, kg, vg, o, lse, o_lo=o_lo)
    assert U.ulysses_sync_status(good) == U.ULY_OK

    def bwd(plan):
        ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
        dq, dk, dv = empty_bf16(q.shape), empty_bf16(k.shape), empty_bf16(v.shape)
        U.ulysses_attn_bwd(plan, qg, kg, vg, o, lse, dog, dq, dk, dv, ws, o_lo=o_lo)
        return dq, dk, dv

    bad = U.ulysses_plan(U.make_config(S, P, 64, H, G, D, flags=U.ULY_FLAG_INJECT_STALL,
                                       wait_timeout_ms=100))
    bwd(bad)
    assert U.ulysses_sync_status(bad) == U.ULY_ERR_TIMEOUT
    bad.close()
    dq, dk, dv = bwd(good)
    assert U.ulysses_sync_status(good) == U.ULY_OK
    qf, kf, vf, dof = (synthetic.bf16_to_f64(a) for a in (q, k, v, do))
    for r in range(P):
        rdq, rdk, rdv = O.causal_attention_bwd(qf[r], kf[r], vf[r], dof[r])
        assert_close(host_f64(dq)[r], rdq, "dq after a timed-out backward")
        assert_close(host_f64(dk)[r], rdk, "dk after a timed-out backward")
        assert_close(host_f64(dv)[r], rdv, "dv after a timed-out backward")


def test_unread_error_status_makes_later_calls_abort_until_read():
    """The plan's status word is sticky: after a timed-out call, a second call on the same
    plan, made before ulysses_sync_status, gives up at its first wait that does not complete
    at once (so it ends long before the wait limit) and the error is still reported; once
    the status has been read (and cleared), the next call waits the full limit again."""
    import time
    S, P, H, G, D = 2048, 2, 4, 2, 128
    limit_ms = 300
    bad = U.ulysses_plan(U.make_config(S, P, 64, H, G, D, flags=U.ULY_FLAG_INJECT_STALL,
                                       wait_timeout_ms=limit_ms))

    q, k, v = (dev_bf16(synthetic.normal_bf16(0, t, (P, S, n // P, D)))
               for t, n in ((synthetic.TENSOR_Q, H), (synthetic.TENSOR_K, G), (synthetic.TENSOR_V, G)))
    o = empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")

    def timed_call():
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        U.ulysses_attn_fwd(bad, q, k, v, o, lse)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) * 1e3

    first = timed_call()
    assert first >= 0.9 * limit_ms
    second = timed_call()                     # status not read in between
    assert second < 0.5 * limit_ms, second
    assert U.ulysses_sync_status(bad) == U.ULY_ERR_TIMEOUT
    third = timed_call()                      # status read: the stall is waited out again
    assert third >= 0.9 * limit_ms
    assert U.ulysses_sync_status(bad) == U.ULY_ERR_TIMEOUT
