"""Every library call of the block's training step on one small case, with every output
(and workspace) placed between NaN-filled guard bands: out-of-bounds evidence where
compute-sanitizer is not available.  Used by tests/test_gpu_debug_build.py in-process
(release library) and as a child process with ULY_LIBRARY=debug (the bounds-checking debug
build, whose kernels also count every out-of-range index they compute).

Run as a script: python tests/canary_block.py S P hidden H G D theta  -> prints "CANARY OK"."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import long_context_sequence_gb300 as U  # noqa: E402
import oracle as O  # noqa: E402
import synthetic  # noqa: E402

GUARD = 4096                                    # bytes of guard band on each side
PATTERN = {torch.bfloat16: 0x7FA5, torch.float32: 0x7FA5A5A5, torch.uint8: 0xA5}
BITS = {torch.bfloat16: torch.int16, torch.float32: torch.int32, torch.uint8: torch.uint8}


class Guarded:
    """A tensor of `shape` inside a buffer with GUARD bytes of a NaN pattern on each side."""

    def __init__(self, shape, dtype=torch.bfloat16):
        self.dtype = dtype
        esz = torch.empty(0, dtype=dtype).element_size()
        self.pad = GUARD // esz
        n = int(np.prod(shape)) if len(shape) else 1
        self.buf = torch.empty(self.pad * 2 + n, dtype=dtype, device="cuda")
        bits = self.buf.view(BITS[dtype])
        pat = PATTERN[dtype]
        if dtype == torch.bfloat16:
            pat = pat - (1 << 16) if pat >= 1 << 15 else pat
        bits.fill_(pat)
        self.t = self.buf[self.pad:self.pad + n].view(shape)

    def intact(self):
        bits = self.buf.view(BITS[self.dtype])
        pat = bits[0].item()
        return bool((bits[:self.pad] == pat).all() and (bits[-self.pad:] == pat).all())


def run(S, P, hidden, H, G, D, theta):
    """All calls once; returns the list of guarded outputs whose guard bands changed, the
    status of the plan(s) and the worst |error| of o_seq against the oracle."""
    plan = U.ulysses_plan(U.make_config(S, P, hidden, H, G, D, rope_theta=theta))
    sh = plan.shapes()
    rope = theta > 0
    dev = lambda a: synthetic.to_torch_bf16(a).cuda()   # noqa: E731
    x = synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, hidden))
    w = synthetic.normal_bf16(0, synthetic.TENSOR_W, ((H + 2 * G) * D, hidden), std=0.02)
    wo = synthetic.normal_bf16(0, synthetic.TENSOR_WO, (hidden, H * D), std=0.02)
    dy = synthetic.normal_bf16(synthetic.SEED_DO, synthetic.TENSOR_WO, (S, hidden))
    xg, wg, wog, dyg = dev(x), dev(w), dev(wo), dev(dy)
    out = {}

    def g(name, shape, dtype=torch.bfloat16):
        out[name] = Guarded(shape, dtype)
        return out[name].t

    qkv = g("qkv", sh["qkv"])
    q, k, v = g("q", sh["q"]), g("k", sh["k"]), g("v", sh["v"])
    o, o_lo = g("o", sh["o"]), g("o_lo", sh["o"])
    lse = g("lse", sh["lse"], torch.float32)
    o_seq = g("o_seq", sh["o_seq"])
    o2 = g("o2", sh["o"])
    y = g("y", (S, hidden))
    do_head = g("do_head", sh["o"])
    dwo = g("dwo", (hidden, H * D), torch.float32)
    ws = g("ws", (U.ulysses_workspace_bytes(plan),), torch.uint8)
    dq, dk, dv = g("dq", sh["q"]), g("dk", sh["k"]), g("dv", sh["v"])
    dqkv = g("dqkv", sh["qkv"])
    dx, dw = g("dx", (S, hidden)), g("dw", sh["w"], torch.float32)
    U.ulysses_qkv_proj(plan, xg, wg, qkv)
    U.ulysses_seq_to_head(plan, qkv, q, k, v, apply_rope=rope)
    U.ulysses_attn_fwd(plan, q, k, v, o, lse, o_lo=o_lo)
    U.ulysses_head_to_seq(plan, o, H, o_seq)
    U.ulysses_seq_to_head_heads(plan, o_seq, H, o2)
    U.ulysses_o_proj(plan, o, wog, y)
    U.ulysses_o_proj_bwd(plan, o, wog, dyg, do_head, dwo)
    U.ulysses_attn_bwd(plan, q, k, v, o, lse, do_head, dq, dk, dv, ws, o_lo=o_lo)
    U.ulysses_head_to_seq_qkv(plan, dq, dk, dv, dqkv, apply_rope=rope)
    U.ulysses_qkv_proj_bwd(plan, xg, wg, dqkv, dx, dw)
    rws = g("ring_ws", (U.ulysses_ring_workspace_bytes(plan),), torch.uint8)
    o_ring, lse_ring = g("o_ring", sh["o_seq"]), g("lse_ring", (P, H, S // P), torch.float32)
    U.ulysses_ring_attn_fwd(plan, o_seq, o_seq[:, :, :G].contiguous(),
                            o_seq[:, :, :G].contiguous(), o_ring, lse_ring, rws)
    statuses = [U.ulysses_sync_status(plan)]
    msgs = [U.ulysses_last_error()]
    # one real rank's pack and unpack calls
    rank = P - 1
    rp = U.ulysses_plan_rank(U.make_config(S, P, hidden, H, G, D, rope_theta=theta), rank)
    rs = rp.shapes()
    sq, sk, sv = g("send_q", rs["q"]), g("send_k", rs["k"]), g("send_v", rs["v"])
    U.ulysses_a2a_pack_qkv(rp, qkv[rank], sq, sk, sv, apply_rope=rope)   # the rank's shard
    sdo = g("send_do", rs["o"])
    U.ulysses_a2a_pack_heads(rp, o_seq[rank], H, sdo)
    ol = g("o_local", rs["o_seq"])
    U.ulysses_a2a_unpack_heads(rp, sdo, H, ol)
    gl = g("dqkv_local", rs["qkv"])
    U.ulysses_a2a_unpack_qkv(rp, sq, sk, sv, gl, apply_rope=rope)
    statuses.append(U.ulysses_sync_status(rp))
    msgs.append(U.ulysses_last_error())
    torch.cuda.synchronize()
    broken = sorted(name for name, t in out.items() if not t.intact())
    ro, _, _ = O.ulysses_block_forward(synthetic.bf16_to_f64(x), synthetic.bf16_to_f64(w), P, H, G,
                                       D, theta)
    err = float(np.abs(synthetic.bf16_to_f64(synthetic.torch_bf16_to_bits(o_seq)) - ro).max())
    return broken, statuses, err, " | ".join(m for m in msgs if m)


if __name__ == "__main__":
    S, P, hidden, H, G, D = (int(a) for a in sys.argv[1:7])
    theta = float(sys.argv[7])
    broken, statuses, err, msg = run(S, P, hidden, H, G, D, theta)
    print("library:", U.LIB_PATH)
    print("broken guard bands:", broken, "statuses:", statuses, "o_seq max|err|: %.3g" % err, msg)
    if broken or any(s != U.ULY_OK for s in statuses) or not err < 5e-2:
        sys.exit(1)
    print("CANARY OK")
