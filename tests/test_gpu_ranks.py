"""The multi-GPU Ulysses data plane on one GPU, through the C ABI.

"Snowflake's Ulysses trick trains transformers on million-token contexts across GPUs",
para 2: every rank projects its own token shard, an all-to-all leaves it the full sequence
for its head group, it runs attention on that group, and an all-to-all restores the shard.
Here all P ranks of a group run one after another on one GPU, each through its own rank
plan (ulysses_plan_rank) and only its own buffers; the all-to-all between them is done by
copying each send block to the receiving rank's buffer, as the library's block table
(ulysses_a2a_table) lays them out.  The rank path must reproduce the single-GPU virtual-rank
path bit for bit (pack, attention forward, unpack, output projection, gradient unpack with
the RoPE backward) and its attention gradients must match the oracle.  One more test runs
the library's own NCCL exchange in a one-rank group."""
import numpy as np
import pytest
import torch

import long_context_sequence_gb300 as U
import oracle as O
import synthetic
from gpu_helpers import assert_close, dev_bf16, empty_bf16, host_f64

pytestmark = pytest.mark.gpu

S, P, HID, H, G, D, THETA = 2048, 4, 512, 8, 4, 128, 500000.0
N = S // P


def _cfg(P_=P):
    return U.make_config(S, P_, HID, H, G, D, rope_theta=THETA)


def _exchange(sends, to_head, n_heads):
    """The all-to-all among the emulated ranks: rank r's receive block p is rank p's send
    block r, at the offsets of the block table."""
    recvs = [torch.empty_like(s) for s in sends]
    for r in range(P):
        tab = U.ulysses_a2a_table(_cfg(), r, to_head, n_heads)
        for b in tab:
            p = b["peer"]
            src_tab = U.ulysses_a2a_table(_cfg(), p, to_head, n_heads)[r]
            assert src_tab["count"] == b["count"]
            dst = recvs[r].view(-1)[b["recv_offset"]:b["recv_offset"] + b["count"]]
            dst.copy_(sends[p].view(-1)[src_tab["send_offset"]:src_tab["send_offset"] + b["count"]])
    return recvs


@pytest.fixture(scope="module")
def block():
    x = synthetic.normal_bf16(0, synthetic.TENSOR_X, (S, HID))
    w = synthetic.normal_bf16(0, synthetic.TENSOR_W, ((H + 2 * G) * D, HID), std=0.02)
    wo = synthetic.normal_bf16(0, synthetic.TENSOR_WO, (HID, H * D), std=0.02)
    do = synthetic.normal_bf16(synthetic.SEED_DO, 0, (S, H, D))
    return tuple(dev_bf16(a) for a in (x, w, wo, do)) + (synthetic.bf16_to_f64(do),)


def test_rank_plans_reproduce_the_virtual_path(block):
    x, w, wo, do_seq, do_f = block
    virt = U.ulysses_plan(_cfg())
    sh = virt.shapes()
    # the single-GPU virtual-rank path
    qkv = empty_bf16(sh["qkv"])
    q, k, v = empty_bf16(sh["q"]), empty_bf16(sh["k"]), empty_bf16(sh["v"])
    o, o_lo = empty_bf16(sh["o"]), empty_bf16(sh["o"])
    lse = torch.empty(sh["lse"], dtype=torch.float32, device="cuda")
    o_seq, y = empty_bf16(sh["o_seq"]), empty_bf16((S, HID))
    U.ulysses_qkv_proj(virt, x, w, qkv)
    U.ulysses_seq_to_head(virt, qkv, q, k, v, apply_rope=True)
    U.ulysses_attn_fwd(virt, q, k, v, o, lse, o_lo=o_lo)
    U.ulysses_head_to_seq(virt, o, H, o_seq)
    U.ulysses_o_proj(virt, o, wo, y)
    assert U.ulysses_sync_status(virt) == U.ULY_OK, U.ulysses_last_error()

    plans = [U.ulysses_plan_rank(_cfg(), r) for r in range(P)]
    rs = plans[0].shapes()
    assert rs["q"] == (P, N, H // P, D) and rs["qkv"] == (N, H + 2 * G, D)
    # 1. local projection of every shard, then the send buffers
    send = {n: [] for n in "qkv"}
    for r, pl in enumerate(plans):
        ql = empty_bf16(rs["qkv"])
        U.ulysses_qkv_proj(pl, x[r * N:(r + 1) * N], w, ql)
        assert torch.equal(ql.view(N, -1), qkv.view(S, -1)[r * N:(r + 1) * N])
        sq, sk, sv = empty_bf16(rs["q"]), empty_bf16(rs["k"]), empty_bf16(rs["v"])
        U.ulysses_a2a_pack_qkv(pl, ql, sq, sk, sv, apply_rope=True)
        # block p of rank r's send buffer = rank p's head group over rank r's tokens
        for p in range(P):
            assert torch.equal(sq[p], q[p, r * N:(r + 1) * N])
            assert torch.equal(sk[p], k[p, r * N:(r + 1) * N])
            assert torch.equal(sv[p], v[p, r * N:(r + 1) * N])
        send["q"].append(sq)
        send["k"].append(sk)
        send["v"].append(sv)
    # 2. seq -> head exchange: what a rank receives is, in token order, its head layout
    rq = _exchange(send["q"], True, H)
    rk = _exchange(send["k"], True, G)
    rv = _exchange(send["v"], True, G)
    outs = []
    for r, pl in enumerate(plans):
        assert torch.equal(rq[r].view(S, -1), q[r].view(S, -1))
        assert torch.equal(rk[r].view(S, -1), k[r].view(S, -1))
        # 3. attention of the rank's head group over all S tokens
        orr, olr = empty_bf16(rs["o"]), empty_bf16(rs["o"])
        lr = torch.empty(rs["lse"], dtype=torch.float32, device="cuda")
        U.ulysses_attn_fwd(pl, rq[r], rk[r], rv[r], orr, lr, o_lo=olr)
        assert U.ulysses_sync_status(pl) == U.ULY_OK, U.ulysses_last_error()
        assert torch.equal(orr.view(S, -1), o[r].view(S, -1))
        assert torch.equal(olr.view(S, -1), o_lo[r].view(S, -1))
        assert torch.equal(lr, lse[r])
        outs.append(orr)
    # 4. head -> seq exchange of o (sent as it stands), unpack, and the output projection
    #    straight from the receive buffer
    ro = _exchange(outs, False, H)
    for r, pl in enumerate(plans):
        ol = empty_bf16(rs["o_seq"])
        U.ulysses_a2a_unpack_heads(pl, ro[r], H, ol)
        assert torch.equal(ol, o_seq.view(S, H, D)[r * N:(r + 1) * N])
        yl = empty_bf16((N, HID))
        U.ulysses_o_proj(pl, ro[r], wo, yl)
        assert torch.equal(yl, y[r * N:(r + 1) * N])
        assert U.ulysses_sync_status(pl) == U.ULY_OK, U.ulysses_last_error()
    # 5. the volume each rank sent to the others, as the pages count it (para 3)
    s2h, h2s = U.ulysses_a2a_volume(_cfg())
    blocks = [U.ulysses_a2a_table(_cfg(), 0, True, n) for n in (H, G, G)] + \
        [U.ulysses_a2a_table(_cfg(), 0, False, H)]
    assert sum(b["count"] * 2 for t in blocks for b in t if b["peer"] != 0) == s2h + h2s


def test_rank_backward_and_gradient_unpack(block):
    """dO's pack and exchange, the attention backward per rank against the oracle, and the
    gradient exchange with the RoPE backward, bit for bit against the virtual path's
    gradient permute of the same gradients."""
    x, w, wo, do_seq, do_f = block
    virt = U.ulysses_plan(_cfg())
    sh = virt.shapes()
    qkv = empty_bf16(sh["qkv"])
    q, k, v = empty_bf16(sh["q"]), empty_bf16(sh["k"]), empty_bf16(sh["v"])
    U.ulysses_qkv_proj(virt, x, w, qkv)
    U.ulysses_seq_to_head(virt, qkv, q, k, v, apply_rope=True)
    plans = [U.ulysses_plan_rank(_cfg(), r) for r in range(P)]
    rs = plans[0].shapes()
    sends = []
    for r, pl in enumerate(plans):
        sd = empty_bf16(rs["o"])
        U.ulysses_a2a_pack_heads(pl, do_seq[r * N:(r + 1) * N], H, sd)
        sends.append(sd)
    rdo = _exchange(sends, True, H)
    qf, kf, vf = host_f64(q), host_f64(k), host_f64(v)
    gq, gk, gv = [], [], []
    for r, pl in enumerate(plans):
        orr = empty_bf16(rs["o"])
        lr = torch.empty(rs["lse"], dtype=torch.float32, device="cuda")
        olr = empty_bf16(rs["o"])
        U.ulysses_attn_fwd(pl, q[r], k[r], v[r], orr, lr, o_lo=olr)
        ws = torch.empty(U.ulysses_workspace_bytes(pl), dtype=torch.uint8, device="cuda")
        dq, dk, dv = empty_bf16(rs["q"]), empty_bf16(rs["k"]), empty_bf16(rs["v"])
        U.ulysses_attn_bwd(pl, q[r], k[r], v[r], orr, lr, rdo[r], dq, dk, dv, ws, o_lo=olr)
        assert U.ulysses_sync_status(pl) == U.ULY_OK, U.ulysses_last_error()
        # the received dO is, in token order, this rank's heads of dO
        dof = host_f64(rdo[r]).reshape(S, H // P, D)
        assert np.array_equal(dof, do_f[:, r * (H // P):(r + 1) * (H // P)])
        rdq, rdk, rdv = O.causal_attention_bwd(qf[r], kf[r], vf[r], dof)
        assert_close(host_f64(dq).reshape(S, -1, D), rdq, "dq[rank %d]" % r)
        assert_close(host_f64(dk).reshape(S, -1, D), rdk, "dk[rank %d]" % r)
        assert_close(host_f64(dv).reshape(S, -1, D), rdv, "dv[rank %d]" % r)
        gq.append(dq)
        gk.append(dk)
        gv.append(dv)
    # the gradients go back (sent as they stand) and are unpacked with the RoPE backward
    xq, xk, xv = _exchange(gq, False, H), _exchange(gk, False, G), _exchange(gv, False, G)
    ref = empty_bf16(sh["qkv"])
    U.ulysses_head_to_seq_qkv(virt, torch.stack([t.view(S, -1, D) for t in gq]),
                              torch.stack([t.view(S, -1, D) for t in gk]),
                              torch.stack([t.view(S, -1, D) for t in gv]), ref, apply_rope=True)
    for r, pl in enumerate(plans):
        got = empty_bf16(rs["qkv"])
        U.ulysses_a2a_unpack_qkv(pl, xq[r], xk[r], xv[r], got, apply_rope=True)
        assert torch.equal(got.view(N, -1), ref.view(S, -1)[r * N:(r + 1) * N])
    assert U.ulysses_sync_status(virt) == U.ULY_OK, U.ulysses_last_error()


def test_rank_plan_rejects_the_single_gpu_permutes():
    pl = U.ulysses_plan_rank(_cfg(), 1)
    z = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(U.UlyssesError) as ei:
        U.ulysses_seq_to_head(pl, z, z, z, z)
    assert ei.value.status == U.ULY_ERR_INVALID_ARG and "rank plan" in str(ei.value)
    virt = U.ulysses_plan(_cfg())
    with pytest.raises(U.UlyssesError) as ei:
        U.ulysses_a2a_pack_heads(virt, z, H, z)
    assert ei.value.status == U.ULY_ERR_INVALID_ARG
    with pytest.raises(U.UlyssesError):
        U.ulysses_plan_rank(_cfg(), P)


def test_nccl_exchange_in_a_one_rank_group(block):
    """The library's own exchange (one NCCL group of sends and receives) in a group of one
    rank: every block goes to the rank itself, so the whole P=1 rank path must reproduce the
    virtual P=1 path bit for bit.  A communicator of the wrong size is refused."""
    x, w, wo, do_seq, do_f = block
    try:
        uid = U.ulysses_nccl_unique_id()
    except U.UlyssesError as e:
        if e.status == U.ULY_ERR_UNSUPPORTED:
            pytest.skip("NCCL is not loadable here: %s" % e)
        raise
    comm = U.ulysses_nccl_comm_init(1, 0, uid)
    try:
        cfg1 = _cfg(1)
        virt = U.ulysses_plan(cfg1)
        pl = U.ulysses_plan_rank(cfg1, 0)
        sh, rs = virt.shapes(), pl.shapes()
        qkv = empty_bf16(sh["qkv"])
        q, k, v = empty_bf16(sh["q"]), empty_bf16(sh["k"]), empty_bf16(sh["v"])
        o, lse = empty_bf16(sh["o"]), torch.empty(sh["lse"], dtype=torch.float32, device="cuda")
        o_seq = empty_bf16(sh["o_seq"])
        U.ulysses_qkv_proj(virt, x, w, qkv)
        U.ulysses_seq_to_head(virt, qkv, q, k, v, apply_rope=True)
        U.ulysses_attn_fwd(virt, q, k, v, o, lse)
        U.ulysses_head_to_seq(virt, o, H, o_seq)
        ql = empty_bf16(rs["qkv"])
        U.ulysses_qkv_proj(pl, x, w, ql)
        sq, sk, sv = empty_bf16(rs["q"]), empty_bf16(rs["k"]), empty_bf16(rs["v"])
        U.ulysses_a2a_pack_qkv(pl, ql, sq, sk, sv, apply_rope=True)
        rq, rk, rv = torch.empty_like(sq), torch.empty_like(sk), torch.empty_like(sv)
        before = U.ulysses_bytes_moved(pl)
        U.ulysses_a2a_exchange(pl, comm, [sq, sk, sv], [rq, rk, rv])
        assert U.ulysses_bytes_moved(pl) == before      # nothing leaves a one-rank group
        orr, lr = empty_bf16(rs["o"]), torch.empty(rs["lse"], dtype=torch.float32, device="cuda")
        U.ulysses_attn_fwd(pl, rq, rk, rv, orr, lr)
        ro = torch.empty_like(orr)
        U.ulysses_a2a_exchange(pl, comm, [orr], [ro])
        ol = empty_bf16(rs["o_seq"])
        U.ulysses_a2a_unpack_heads(pl, ro, H, ol)
        torch.cuda.synchronize()
        assert U.ulysses_sync_status(pl) == U.ULY_OK, U.ulysses_last_error()
        assert torch.equal(rq.view(S, -1), q.view(S, -1))
        assert torch.equal(ol, o_seq.view(S, H, D))
        assert torch.equal(lr, lse[0])
        # a plan of two ranks cannot use a communicator of one
        pl2 = U.ulysses_plan_rank(_cfg(2), 0)
        with pytest.raises(U.UlyssesError) as ei:
            U.ulysses_a2a_exchange(pl2, comm, [sq], [rq])
        assert ei.value.status == U.ULY_ERR_INVALID_ARG and "communicator" in str(ei.value)
    finally:
        U.ulysses_nccl_comm_destroy(comm)


@pytest.mark.parametrize("theta", [0.0, THETA])
def test_rank_pack_of_fp32_projection_output(theta):
    """An fp32 projection output packed by a rank plan (rounded to bf16 on the way, RoPE at
    the shard's global positions when theta > 0) equals the virtual path's seq->head of the
    same fp32 tensor, block for block, bit for bit."""
    cfg = U.make_config(S, P, HID, H, G, D, rope_theta=theta)
    virt = U.ulysses_plan(cfg)
    sh = virt.shapes()
    x = synthetic.normal_f64(0, synthetic.TENSOR_QKV, (S, H + 2 * G, D), std=1.28).astype(np.float32)
    xg = torch.from_numpy(x).cuda()
    q, k, v = empty_bf16(sh["q"]), empty_bf16(sh["k"]), empty_bf16(sh["v"])
    U.ulysses_seq_to_head(virt, xg, q, k, v, apply_rope=theta > 0)
    for r in range(P):
        pl = U.ulysses_plan_rank(cfg, r)
        rs = pl.shapes()
        sq, sk, sv = empty_bf16(rs["q"]), empty_bf16(rs["k"]), empty_bf16(rs["v"])
        U.ulysses_a2a_pack_qkv(pl, xg[r * N:(r + 1) * N].contiguous(), sq, sk, sv,
                               apply_rope=theta > 0)
        assert U.ulysses_sync_status(pl) == U.ULY_OK, U.ulysses_last_error()
        for p in range(P):
            assert torch.equal(sq[p], q[p, r * N:(r + 1) * N])
            assert torch.equal(sk[p], k[p, r * N:(r + 1) * N])
            assert torch.equal(sv[p], v[p, r * N:(r + 1) * N])
