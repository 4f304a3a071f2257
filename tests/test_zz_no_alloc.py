"""The allocation-free backward (ulysses_attn_bwd_noalloc), called through the C ABI.

It exists for callers that cannot allocate device memory when they call the backward
(their HBM already belongs to their own pool or caching allocator, the path must not
synchronise on cudaMalloc, or a plain C caller has no device allocator); it runs the same
kernels as ulysses_attn_bwd on a fixed scratch array inside the library.  Checked on two
calls in a row (the shared scratch must carry nothing over): dK and dV equal the
workspace path's bit for bit (no atomics there), dQ agrees within its atomic summation
order, all three match the oracle, and the device's free memory does not move across the
calls.  Also the size limit.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import long_context_sequence_gb300 as U
import oracle as O
import synthetic
from gpu_helpers import assert_close, bf16_ulp, dev_bf16, empty_bf16, host_f64

pytestmark = pytest.mark.gpu


def test_noalloc_backward_matches_workspace_backward_twice():
    S, P, H, G, D = 1024, 4, 8, 4, 128
    plan = U.ulysses_plan(U.make_config(S, P, 64, H, G, D))
    q = synthetic.normal_bf16(0, synthetic.TENSOR_Q, (P, S, H // P, D))
    k = synthetic.normal_bf16(0, synthetic.TENSOR_K, (P, S, G // P, D))
    v = synthetic.normal_bf16(0, synthetic.TENSOR_V, (P, S, G // P, D))
    qg, kg, vg = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    o, o_lo = empty_bf16(qg.shape), empty_bf16(qg.shape)
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    U.ulysses_attn_fwd(plan, qg, kg, vg, o, lse, o_lo=o_lo)
    ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    qf, kf, vf = (synthetic.bf16_to_f64(a) for a in (q, k, v))
    for call, seed in enumerate((1, 7)):
        do = synthetic.normal_bf16(seed, 0, (P, S, H // P, D))
        dog = dev_bf16(do)
        ref = [empty_bf16(qg.shape), empty_bf16(kg.shape), empty_bf16(vg.shape)]
        got = [empty_bf16(qg.shape), empty_bf16(kg.shape), empty_bf16(vg.shape)]
        U.ulysses_attn_bwd(plan, qg, kg, vg, o, lse, dog, *ref, ws, o_lo=o_lo)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        U.ulysses_attn_bwd_noalloc(plan, qg, kg, vg, o, lse, dog, *got, o_lo=o_lo)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before, "call %d allocated" % (call + 1)
        assert U.ulysses_sync_status(plan) == U.ULY_OK, U.ulysses_last_error()
        dq, dk, dv = (host_f64(t) for t in got)
        rq, rk, rv = (host_f64(t) for t in ref)
        assert np.array_equal(dk, rk), "dk differs from the workspace path (call %d)" % (call + 1)
        assert np.array_equal(dv, rv), "dv differs from the workspace path (call %d)" % (call + 1)
        assert np.all(np.abs(dq - rq) <= bf16_ulp(rq)), "dq (call %d)" % (call + 1)
        dof = synthetic.bf16_to_f64(do)
        for r in range(P):
            odq, odk, odv = O.causal_attention_bwd(qf[r], kf[r], vf[r], dof[r])
            assert_close(dq[r], odq, "dq[rank %d] (call %d)" % (r, call + 1))
            assert_close(dk[r], odk, "dk[rank %d] (call %d)" % (r, call + 1))
            assert_close(dv[r], odv, "dv[rank %d] (call %d)" % (r, call + 1))


def test_noalloc_backward_rejects_plans_above_its_scratch():
    S, P, H, G, D = 65536, 8, 32, 8, 128        # needs ~1 GB of scratch
    plan = U.ulysses_plan(U.make_config(S, P, 64, H, G, D))
    assert U.ulysses_workspace_bytes(plan) > 64 << 20
    z = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(U.UlyssesError) as ei:
        U.ulysses_attn_bwd_noalloc(plan, z, z, z, z, torch.zeros(4, device="cuda"), z, z, z, z)
    assert ei.value.status == U.ULY_ERR_UNSUPPORTED
    assert "scratch" in U.ulysses_last_error()
    assert U.ulysses_sync_status(plan) == U.ULY_OK
