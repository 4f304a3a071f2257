"""The allocation-free backward (ulysses_attn_bwd_noalloc), called through the C ABI.

It exists for callers that cannot allocate device memory when they call the backward
(their HBM already belongs to their own pool, or the path must not synchronise on
cudaMalloc); it runs the same kernels on a fixed scratch array inside the library.
Checked against ulysses_attn_bwd with a caller workspace, within the parity tolerance,
on two calls in a row (the shared scratch must not carry anything over), plus the size
limit.  This file is collected last on purpose."""
import pytest
import torch

import long_context_sequence_gb300 as U
import synthetic
from gpu_helpers import assert_close, dev_bf16, empty_bf16, host_f64

pytestmark = pytest.mark.gpu


def test_noalloc_backward_matches_workspace_backward_twice():
    S, P, H, G, D = 1024, 4, 8, 4, 128
    plan = U.ulysses_plan(U.make_config(S, P, 64, H, G, D))
    q = dev_bf16(synthetic.normal_bf16(0, synthetic.TENSOR_Q, (P, S, H // P, D)))
    k = dev_bf16(synthetic.normal_bf16(0, synthetic.TENSOR_K, (P, S, G // P, D)))
    v = dev_bf16(synthetic.normal_bf16(0, synthetic.TENSOR_V, (P, S, G // P, D)))
    o, o_lo = empty_bf16(q.shape), empty_bf16(q.shape)
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    U.ulysses_attn_fwd(plan, q, k, v, o, lse, o_lo=o_lo)
    ws = torch.empty(U.ulysses_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((1, 7)):
        do = dev_bf16(synthetic.normal_bf16(seed, 0, (P, S, H // P, D)))
        ref = [empty_bf16(q.shape), empty_bf16(k.shape), empty_bf16(v.shape)]
        got = [empty_bf16(q.shape), empty_bf16(k.shape), empty_bf16(v.shape)]
        U.ulysses_attn_bwd(plan, q, k, v, o, lse, do, *ref, ws, o_lo=o_lo)
        U.ulysses_attn_bwd_noalloc(plan, q, k, v, o, lse, do, *got, o_lo=o_lo)
        assert U.ulysses_sync_status(plan) == U.ULY_OK, U.ulysses_last_error()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert_close(host_f64(g), host_f64(r), "%s (call %d)" % (name, call + 1))


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
