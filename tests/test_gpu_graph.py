"""The whole layer's training step is capturable in a CUDA graph: every call is asynchronous
on the caller's stream, builds its tensor maps on the host and neither allocates nor
synchronises.  A captured step, replayed on new inputs, gives what eager calls give."""
import numpy as np
import pytest
import torch

import long_context_sequence_gb300 as U
import synthetic
from gpu_helpers import dev_bf16, empty_bf16, host_f64

pytestmark = pytest.mark.gpu


def test_training_step_replays_from_a_cuda_graph():
    S, P, hidden, H, G, D, theta = 1024, 4, 512, 8, 8, 64, 10000.0
    C = (H + 2 * G) * D
    plan = U.ulysses_plan(U.make_config(S, P, hidden, H, G, D, rope_theta=theta))
    x = dev_bf16(synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, hidden)))
    w = dev_bf16(synthetic.normal_bf16(0, synthetic.TENSOR_W, (C, hidden), std=0.02))
    wo = dev_bf16(synthetic.normal_bf16(0, synthetic.TENSOR_WO, (hidden, H * D), std=0.02))
    dy = dev_bf16(synthetic.normal_bf16(synthetic.SEED_DO, synthetic.TENSOR_WO, (S, hidden)))
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

    def step():
        U.ulysses_qkv_proj(plan, x, w, qkv)
        U.ulysses_seq_to_head(plan, qkv, q, k, v, apply_rope=True)
        U.ulysses_attn_fwd(plan, q, k, v, o, lse, o_lo=o_lo)
        U.ulysses_o_proj(plan, o, wo, y)
        U.ulysses_o_proj_bwd(plan, o, wo, dy, do, dwo)
        U.ulysses_attn_bwd(plan, q, k, v, o, lse, do, dq, dk, dv, ws, o_lo=o_lo)
        U.ulysses_head_to_seq_qkv(plan, dq, dk, dv, dqkv, apply_rope=True)
        U.ulysses_qkv_proj_bwd(plan, x, w, dqkv, dx, dw)

    def outputs():
        return [t.clone() for t in (y, dwo, dx, dw)]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                     # eager, also sets the kernels' attributes
    torch.cuda.current_stream().wait_stream(side)
    assert U.ulysses_sync_status(plan) == U.ULY_OK, U.ulysses_last_error()
    eager = outputs()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    assert U.ulysses_sync_status(plan) == U.ULY_OK, U.ulysses_last_error()
    replayed = outputs()

    # new inputs into the captured buffers: the replay must follow them
    x.copy_(dev_bf16(synthetic.normal_bf16(7, synthetic.TENSOR_X, (S, hidden))))
    graph.replay()
    torch.cuda.synchronize()
    replayed_new = outputs()
    with torch.cuda.stream(side):
        step()
    torch.cuda.synchronize()
    assert U.ulysses_sync_status(plan) == U.ULY_OK, U.ulysses_last_error()
    eager_new = outputs()

    for a, b, name in zip(replayed + replayed_new, eager + eager_new,
                          ["y", "dwo", "dx", "dw"] * 2):
        ga, gb = host_f64(a), host_f64(b)
        if name == "y":
            assert np.array_equal(ga, gb), name            # no reductions on this path
        else:
            # dQ is summed with atomics, so the order of its fp32 additions may differ
            scale = np.abs(gb).max()
            assert np.abs(ga - gb).max() <= 1e-2 * scale, name
    assert not np.array_equal(host_f64(replayed[0]), host_f64(replayed_new[0]))
