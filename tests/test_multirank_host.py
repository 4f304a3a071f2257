"""The multi-GPU Ulysses data plane on CPU: one process per rank over gloo (world size 2
and 4), each rank holding only its own token shard.

"Snowflake's Ulysses trick trains transformers on million-token contexts across GPUs",
para 2: after the local projection an all-to-all leaves every rank the full sequence for
its head group, and a second all-to-all restores the sequence sharding.  Each rank packs its
send buffer by the library's block table (ulysses_a2a_table, host only), the ranks exchange
the buffers with a real all-to-all (gloo's all_to_all_single), and what each rank receives
must equal, bit for bit, its share of the oracle's seq->head and head->seq.  Also: the bytes
each rank sends to the other ranks equal the per-rank volume of para 3
(ulysses_a2a_volume), and the benchmark's job timing takes the slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _guarded(target, rank, world, port, out, *args):
    """Runs one rank; a failure is reported through the queue instead of a hang."""
    try:
        target(rank, world, port, out, *args)
    except BaseException as e:   # noqa: B902 (report every failure of the child)
        import traceback
        out.put((rank, "error", traceback.format_exc()))
        raise SystemExit(1) from e


def _run(target, world, *args):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_guarded, args=(target, r, world, port, q) + args)
             for r in range(world)]
    for p in procs:
        p.start()
    res = []
    for _ in procs:
        item = q.get(timeout=120)
        assert item[1] != "error", "rank %d failed:\n%s" % (item[0], item[2])
        res.append(item)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


def _init(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _timing_worker(rank, world, port, out):
    _init(rank, world, port)
    import bench
    local_ms = [40.0, 55.0][rank]
    ms = bench.reduce_max_ms(local_ms, world, dist)
    tf = bench.job_tflops(1e12, world, ms)
    out.put((rank, ms, tf))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_uses_the_slowest_rank():
    for rank, ms, tf in _run(_timing_worker, 2):
        assert ms == 55.0
        assert tf == pytest.approx(2 * 1e12 / 0.055 / 1e12)


def _exchange(send: np.ndarray) -> np.ndarray:
    """The all-to-all over gloo: block p of `send` goes to rank p (equal blocks).  The bf16
    bit patterns travel as pairs in 32-bit words (gloo has no 16-bit integers)."""
    t = torch.from_numpy(send.view(np.int32).copy())
    r = torch.empty_like(t)
    dist.all_to_all_single(r, t)
    return r.numpy().view(np.uint16)


def _pack(x_local: np.ndarray, blocks, D) -> np.ndarray:
    """Send buffer of one tensor from the table: block p = the shard's rows of the heads
    [send_head_begin, +n_heads), laid out [n_tokens][n_heads][D] at send_offset."""
    send = np.empty(sum(b["count"] for b in blocks), np.uint16)
    for b in blocks:
        h0, nh = b["send_head_begin"], b["n_heads"]
        send[b["send_offset"]:b["send_offset"] + b["count"]] = x_local[:, h0:h0 + nh].reshape(-1)
    return send


def _a2a_worker(rank, world, port, out, S, H, G, D):
    _init(rank, world, port)
    import long_context_sequence_gb300 as U
    import oracle as O
    import synthetic
    P = world
    n = S // P
    cfg = U.make_config(S, P, 64, H, G, D)
    qkv = synthetic.normal_bf16(0, synthetic.TENSOR_QKV, (S, H + 2 * G, D))   # every rank draws it
    local = qkv[rank * n:(rank + 1) * n]                                        # but keeps its shard
    want_q, want_k, want_v = O.seq_to_head(qkv, P, H, G)
    sent = 0
    got = {}
    # seq -> head, one exchange per tensor (q: heads [0, H), k: [H, H+G), v: [H+G, H+2G))
    for name, lo, nh in (("q", 0, H), ("k", H, G), ("v", H + G, G)):
        blocks = U.ulysses_a2a_table(cfg, rank, True, nh)
        assert [b["peer"] for b in blocks] == list(range(P))
        assert all(b["send_token_begin"] == rank * n and b["n_tokens"] == n for b in blocks)
        recv = _exchange(_pack(local[:, lo:lo + nh], blocks, D))
        # the received blocks, in block order, are the head layout [S][nh/P][D]
        for b in blocks:
            assert b["recv_head_begin"] == rank * (nh // P)
            assert b["recv_token_begin"] == b["peer"] * n
        got[name] = recv.reshape(S, nh // P, D)
        sent += sum(b["count"] * 2 for b in blocks if b["peer"] != rank)
    ok_s2h = (np.array_equal(got["q"], want_q[rank]) and np.array_equal(got["k"], want_k[rank])
              and np.array_equal(got["v"], want_v[rank]))
    # head -> seq of a head-layout tensor (the attention output's path): the query part
    blocks = U.ulysses_a2a_table(cfg, rank, False, H)
    o_head = got["q"]
    send = np.empty(o_head.size, np.uint16)
    for b in blocks:      # block p: p's tokens of my heads, which o_head holds in token order
        t0 = b["send_token_begin"]
        send[b["send_offset"]:b["send_offset"] + b["count"]] = o_head[t0:t0 + n].reshape(-1)
    assert np.array_equal(send, o_head.reshape(-1))       # o is its own send buffer
    recv = _exchange(send)
    o_local = np.empty((n, H, D), np.uint16)
    for b in blocks:
        h0, nh = b["recv_head_begin"], b["n_heads"]
        assert b["recv_token_begin"] == rank * n
        o_local[:, h0:h0 + nh] = recv[b["recv_offset"]:b["recv_offset"] + b["count"]].reshape(n, nh, D)
    sent += sum(b["count"] * 2 for b in blocks if b["peer"] != rank)
    want_o = O.head_to_seq(want_q, P)[rank]
    ok_h2s = np.array_equal(o_local, want_o) and np.array_equal(o_local, local[:, :H])
    vol = sum(U.ulysses_a2a_volume(cfg))
    out.put((rank, bool(ok_s2h), bool(ok_h2s), sent, vol))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,S,H,G,D", [(2, 256, 8, 4, 64), (4, 512, 32, 8, 128)])
def test_all_to_alls_across_ranks_match_the_oracle(world, S, H, G, D):
    for rank, ok_s2h, ok_h2s, sent, vol in _run(_a2a_worker, world, S, H, G, D):
        assert ok_s2h, "rank %d: seq->head differs from the oracle" % rank
        assert ok_h2s, "rank %d: head->seq differs from the oracle" % rank
        assert sent == vol, (rank, sent, vol)
