"""GPU parity of ring attention on the virtual ranks (the comparator of the Ulysses-trick
page, para 3) against the fp64 oracle's unsharded causal attention: the ring's merged output
and lse, its exchange bytes, and agreement with the Ulysses path on the same inputs."""
import numpy as np
import pytest
import torch

import long_context_sequence_gb300 as U
import oracle as O
import synthetic
from gpu_helpers import assert_close, assert_close_f32, dev_bf16, empty_bf16, host_f64

pytestmark = pytest.mark.gpu


def _ok(plan):
    st = U.ulysses_sync_status(plan)
    assert st == U.ULY_OK, U.ulysses_last_error()


def _inputs(S, P, H, G, D, std):
    n = S // P
    q = synthetic.normal_bf16(0, synthetic.TENSOR_Q, (P, n, H, D), std=std)
    k = synthetic.normal_bf16(0, synthetic.TENSOR_K, (P, n, G, D), std=std)
    v = synthetic.normal_bf16(0, synthetic.TENSOR_V, (P, n, G, D), std=std)
    return q, k, v


def _ring(S, P, H, G, D, q, k, v):
    plan = U.ulysses_plan(U.make_config(S, P, 64, H, G, D))
    n = S // P
    o = empty_bf16((P, n, H, D))
    lse = torch.empty((P, H, n), dtype=torch.float32, device="cuda")
    ws = torch.empty(U.ulysses_ring_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)   # contents on entry must not matter
    before = U.ulysses_bytes_moved(plan)
    U.ulysses_ring_attn_fwd(plan, dev_bf16(q), dev_bf16(k), dev_bf16(v), o, lse, ws)
    _ok(plan)
    moved = U.ulysses_bytes_moved(plan) - before
    return plan, o, lse, moved


RING_CASES = [  # S, P, H, G, D, std
    (1024, 4, 8, 8, 64, 0.45),       # tiny block shape
    (2048, 8, 32, 8, 128, 1.28),     # Llama-3.1-8B head shape
    (1000, 4, 8, 4, 128, 1.0),       # shard of 250 rows: ragged tiles in every step
    (384, 2, 4, 2, 64, 1.0),
    (8, 8, 8, 8, 64, 1.0),           # one token per rank
    (130, 1, 2, 1, 128, 1.0),        # one rank: the diagonal step only
    (4096, 16, 32, 16, 128, 1.0),    # 16 ranks, 15 shard rotations
    (2048, 4, 32, 4, 128, 1.28),     # GQA 8:1
]


@pytest.mark.parametrize("S,P,H,G,D,std", RING_CASES)
def test_ring_attention_equals_causal_attention(S, P, H, G, D, std):
    q, k, v = _inputs(S, P, H, G, D, std)
    plan, o, lse, moved = _ring(S, P, H, G, D, q, k, v)
    n = S // P
    ro, rl = O.causal_attention(*(synthetic.bf16_to_f64(a).reshape(S, -1, D) for a in (q, k, v)))
    assert_close(host_f64(o).reshape(S, H, D), ro, "o")
    assert_close_f32(host_f64(lse).transpose(1, 0, 2).reshape(H, S), rl, "lse")
    # the exchange: every rank forwards its K and V shard P - 1 times (read + write bytes)
    assert moved == (P - 1) * P * n * G * D * 2 * 2 * 2
    assert moved == P * 2 * 2 * O.ring_volume_bytes(S, P, G, D) // 2


def test_ring_matches_the_ulysses_path_on_the_same_tokens():
    """8B head shape at S=2048, P=8: Ulysses (seq->head, attention, head->seq) and ring
    attention give the same output from the same q, k, v shards."""
    S, P, H, G, D = 2048, 8, 32, 8, 128
    q, k, v = _inputs(S, P, H, G, D, 1.28)
    _, o_ring, lse_ring, _ = _ring(S, P, H, G, D, q, k, v)
    plan = U.ulysses_plan(U.make_config(S, P, 64, H, G, D))
    n = S // P
    qkv = np.concatenate([q, k, v], axis=2)                     # [P][n][H + 2G][D]
    qh, kh, vh = empty_bf16((P, S, H // P, D)), empty_bf16((P, S, G // P, D)), empty_bf16((P, S, G // P, D))
    U.ulysses_seq_to_head(plan, dev_bf16(qkv), qh, kh, vh)
    o = empty_bf16((P, S, H // P, D))
    lse = torch.empty((P, H // P, S), dtype=torch.float32, device="cuda")
    U.ulysses_attn_fwd(plan, qh, kh, vh, o, lse)
    o_seq = empty_bf16((P, n, H, D))
    U.ulysses_head_to_seq(plan, o, H, o_seq)
    _ok(plan)
    # both within their bound of the exact result, so within twice it of each other
    assert_close(host_f64(o_ring), host_f64(o_seq), "ring vs ulysses", max_abs=4e-2, mean_abs=4e-3)
    lse_u = host_f64(lse).reshape(H, S)      # [P][H/P][S] is head-major already
    lse_r = host_f64(lse_ring).transpose(1, 0, 2).reshape(H, S)
    assert np.abs(lse_u - lse_r).max() < 1e-3


def test_ring_sampled_rows_8b_shape_32k():
    """S=32768, P=8: seed-sampled query rows of every rank against the oracle's per-row
    definition over the full causal prefix."""
    S, P, H, G, D = 32768, 8, 32, 8, 128
    n = S // P
    q, k, v = _inputs(S, P, H, G, D, 1.28)
    _, o, lse, _ = _ring(S, P, H, G, D, q, k, v)
    rows = synthetic.sample_rows(S, P, 48)
    qf, kf, vf = (synthetic.bf16_to_f64(a).reshape(S, -1, D) for a in (q, k, v))
    ro, rl = O.causal_attention_rows(qf, kf, vf, rows)
    o_h = host_f64(o).reshape(S, H, D)
    lse_h = host_f64(lse).transpose(1, 0, 2).reshape(H, S)
    assert_close(o_h[rows], ro, "o")
    assert_close_f32(lse_h[:, rows], rl, "lse")


def test_ring_empty_sequence_is_a_no_op():
    plan = U.ulysses_plan(U.make_config(0, 4, 64, 8, 8, 64))
    z = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    U.ulysses_ring_attn_fwd(plan, z, z, z, z, torch.empty(0, device="cuda"), z)
    _ok(plan)
