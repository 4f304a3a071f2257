"""Plain, slow CPU oracle for the Ulysses sequence-parallel attention block.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU-baseline
leg may import this module.  The GPU library never calls it and shares no code with it.

Everything is float64 numpy.  Library primitives (matmul, exp, log) serve as steps; there
is no blocking, fusion or reordering beyond chunking independent query rows to bound
memory.

Sources are the web pages on the method, cited by title and paragraph:
  [UT]  "Snowflake's Ulysses trick trains transformers on million-token contexts across
        GPUs" (inblix): para 2 (local QKV projection, seq->head all-to-all, independent
        heads with FlashAttention, inverse all-to-all), para 3 (two all-to-alls per layer,
        volume O(hidden x seq_len / P)).
  [USP] "Ulysses Sequence Parallelism: Training with Million-Token Contexts" (neubench
        copy of the Hugging Face post): para 3 (quadratic attention, FlashAttention tiling
        never materialises the full matrix), para 5 (the second all-to-all reverses the
        redistribution), para 7 (heads are partitioned across GPUs), para 8 (the input is
        split along the sequence dimension).
Points the pages leave open are read as follows (the plainest reading):
  * shards are contiguous: rank r holds tokens [r*S/P, (r+1)*S/P);
  * head groups are contiguous: rank r gets query heads [r*H/P, (r+1)*H/P) and KV heads
    [r*G/P, (r+1)*G/P); query head h uses KV head h // (H/G) (grouped-query attention);
  * attention is causal (key j visible to query i iff j <= i), scale 1/sqrt(D),
    logsumexp in natural log;
  * RoPE is the rotate-half form: for pair (i, i + D/2) at position p the pair is rotated
    by angle p * theta^(-2i/D), positions are global token indices;
  * the projection weight has nn.Linear layout [(H + 2G) * D][hidden], columns ordered
    q heads, then k heads, then v heads;
  * the block ends with the output projection of the restored shard, weight wo in
    nn.Linear layout [hidden][H * D], input columns ordered head-major (h * D + d);
  * the training step's loss is L = sum(output * upstream gradient); its gradients follow
    the forward steps in reverse (RoPE backward = rotation by the negative angle).

Pins (tests/test_oracle.py): brute-force loops on tiny inputs, a hand-worked attention
example and a hand-written all-to-all index table under tests/golden/, closed forms
(Q = 0 gives prefix means and lse = ln(i+1)), invariants (round trip, sharded equals
unsharded, norm-preserving RoPE, softmax shift invariance, sum of dK is zero, ring attention
equals unsharded attention), torch float64 SDPA and autograd, and central finite differences.
"""
from __future__ import annotations

import math

import numpy as np

ROW_CHUNK = 256          # query rows handled per matmul (independent rows; memory bound)


# --------------------------------------------------------------------------- projection
def qkv_projection(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Local QKV projection y[s][c] = sum_k x[s][k] * w[c][k]   [UT para 2].

    x: [T][hidden], w: [C][hidden] (C = (H + 2G) * D).  Returns [T][C] float64."""
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64).T


# --------------------------------------------------------------------------------- RoPE
def rope_angles(positions: np.ndarray, head_dim: int, theta: float) -> np.ndarray:
    """phi[p][i] = p * theta^(-2 i / D) for i < D/2 (float64)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    return np.asarray(positions, np.float64)[:, None] * inv_freq[None, :]


def apply_rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE of x [T][n_heads][D] at the given global positions [T]."""
    x = np.asarray(x, np.float64)
    half = x.shape[-1] // 2
    phi = rope_angles(positions, x.shape[-1], theta)[:, None, :]
    c, s = np.cos(phi), np.sin(phi)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


# ------------------------------------------------------------------------- all-to-alls
def shard_sequence(x: np.ndarray, P: int) -> list:
    """Contiguous sequence shards: rank r holds rows [r*S/P, (r+1)*S/P)   [USP para 8]."""
    n = x.shape[0] // P
    return [x[r * n:(r + 1) * n] for r in range(P)]


def seq_to_head(qkv_seq: np.ndarray, P: int, H: int, G: int):
    """seq->head all-to-all   [UT para 2].

    qkv_seq: [S][H + 2G][D] where rank r holds tokens [r*S/P, (r+1)*S/P).
    Returns q [P][S][H/P][D], k [P][S][G/P][D], v [P][S][G/P][D]: after the exchange
    rank r2 holds every token for its head group.  Written as the exchange itself:
    every sender rank r ships to every receiver rank r2 its tokens' slice of r2's heads.
    """
    S, _, D = qkv_seq.shape
    n, hq, hk = S // P, H // P, G // P
    q = np.empty((P, S, hq, D), qkv_seq.dtype)
    k = np.empty((P, S, hk, D), qkv_seq.dtype)
    v = np.empty((P, S, hk, D), qkv_seq.dtype)
    shards = shard_sequence(qkv_seq, P)
    for r in range(P):                      # sender: owns tokens [r*n, (r+1)*n)
        local = shards[r]
        for r2 in range(P):                 # receiver: owns head group r2
            q[r2, r * n:(r + 1) * n] = local[:, r2 * hq:(r2 + 1) * hq]
            k[r2, r * n:(r + 1) * n] = local[:, H + r2 * hk:H + (r2 + 1) * hk]
            v[r2, r * n:(r + 1) * n] = local[:, H + G + r2 * hk:H + G + (r2 + 1) * hk]
    return q, k, v


def head_to_seq(x_head: np.ndarray, P: int) -> np.ndarray:
    """head->seq all-to-all, the inverse redistribution   [USP para 5; UT para 2].

    x_head: [P][S][n/P][D] (rank r2 holds head group r2 for every token).
    Returns [P][S/P][n][D]: rank r holds its own tokens for every head."""
    _, S, hl, D = x_head.shape
    n = S // P
    out = np.empty((P, n, hl * P, D), x_head.dtype)
    for r2 in range(P):                     # sender: owns head group r2
        for r in range(P):                  # receiver: owns tokens [r*n, (r+1)*n)
            out[r, :, r2 * hl:(r2 + 1) * hl] = x_head[r2, r * n:(r + 1) * n]
    return out


# ------------------------------------------------------------------- attention forward
def _kv_head(h: int, H: int, G: int) -> int:
    return h // (H // G)


def causal_attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows,
                          scale: float | None = None):
    """Causal multi-head (grouped-query) attention for the given query rows.

    q: [S][H][D], k, v: [S][G][D] (float64 or convertible).  For each head h (KV head
    g = h // (H/G)) and query row i, with scores s_j = scale * q_i . k_j over j <= i:
        m = max_j s_j,  p_j = exp(s_j - m),  l = sum_j p_j,
        o_i = sum_j p_j v_j / l,  lse_i = m + ln l.
    Returns o [len(rows)][H][D] and lse [H][len(rows)].
    Heads are computed one at a time, so each head's numbers do not depend on which
    other heads are present   [UT para 2: attention heads are independent]."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    rows = np.asarray(rows, np.int64)
    S, H, D = q.shape
    G = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = np.zeros((rows.size, H, D))
    lse = np.zeros((H, rows.size))
    for h in range(H):
        g = _kv_head(h, H, G)
        kh = np.ascontiguousarray(k[:, g])
        vh = np.ascontiguousarray(v[:, g])
        for c0 in range(0, rows.size, ROW_CHUNK):
            rc = rows[c0:c0 + ROW_CHUNK]
            jmax = int(rc.max()) + 1
            qc = np.ascontiguousarray(q[rc, h])
            s = scale * (qc @ kh[:jmax].T)                           # [rows][keys]
            s[np.arange(jmax)[None, :] > rc[:, None]] = -np.inf     # causal: j <= i
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            l = p.sum(axis=1, keepdims=True)
            o[c0:c0 + rc.size, h] = (p @ vh[:jmax]) / l
            lse[h, c0:c0 + rc.size] = (m + np.log(l))[:, 0]
    return o, lse


def causal_attention(q, k, v, scale=None):
    """All rows of causal_attention_rows: o [S][H][D], lse [H][S]."""
    return causal_attention_rows(q, k, v, np.arange(np.asarray(q).shape[0]), scale)


def ulysses_attention(q_head, k_head, v_head, scale=None):
    """Per-rank attention on head groups: q_head [P][S][H/P][D], k/v [P][S][G/P][D].

    Each virtual rank attends over the full sequence with its own heads only   [UT para 2].
    Returns o_head [P][S][H/P][D] and lse [P][H/P][S]."""
    P = q_head.shape[0]
    outs, lses = [], []
    for r in range(P):
        o, lse = causal_attention(q_head[r], k_head[r], v_head[r], scale)
        outs.append(o)
        lses.append(lse)
    return np.stack(outs), np.stack(lses)


# ------------------------------------------------------------------ attention backward
def causal_attention_bwd_rows(q, k, v, do, dq_rows, key_lo: int, scale=None):
    """Gradients of L = sum(O * dO) for causal attention, restricted for sampling.

    Returns dq for the query rows dq_rows ([len][H][D]) and dk, dv for keys
    [key_lo, S) ([S - key_lo][G][D]); key_lo = 0 and dq_rows = all rows give the full
    gradients.  With P_ij = exp(s_ij - lse_i) for j <= i:
        D_i   = dO_i . o_i
        dP_ij = dO_i . v_j
        dS_ij = P_ij (dP_ij - D_i)
        dq_i  = scale * sum_j dS_ij k_j
        dk_j  = scale * sum_{h in group} sum_i dS_ij q_i
        dv_j  = sum_{h in group} sum_i P_ij dO_i
    Only rows i >= key_lo reach keys j >= key_lo (causality), so those rows plus
    dq_rows are the only rows recomputed."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    S, H, D = q.shape
    G = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq_rows = np.asarray(dq_rows, np.int64)
    rows = np.union1d(dq_rows, np.arange(key_lo, S, dtype=np.int64))
    o, lse = causal_attention_rows(q, k, v, rows, scale)
    want_dq = np.isin(rows, dq_rows)
    dq_pos = {int(r): i for i, r in enumerate(dq_rows)}
    dq = np.zeros((dq_rows.size, H, D))
    dk = np.zeros((S - key_lo, G, D))
    dv = np.zeros((S - key_lo, G, D))
    for h in range(H):
        g = _kv_head(h, H, G)
        kh = np.ascontiguousarray(k[:, g])
        vh = np.ascontiguousarray(v[:, g])
        for c0 in range(0, rows.size, ROW_CHUNK):
            sel = slice(c0, c0 + ROW_CHUNK)
            rc = rows[sel]
            jmax = int(rc.max()) + 1
            qc = np.ascontiguousarray(q[rc, h])
            doc = np.ascontiguousarray(do[rc, h])
            s = scale * (qc @ kh[:jmax].T)
            mask = np.arange(jmax)[None, :] > rc[:, None]
            p = np.exp(s - lse[h, sel][:, None])
            p[mask] = 0.0
            dp = doc @ vh[:jmax].T
            delta = np.sum(doc * o[sel, h], axis=1, keepdims=True)
            ds = p * (dp - delta)
            wq = want_dq[sel]
            if wq.any():
                dqc = scale * (ds[wq] @ kh[:jmax])
                for row, val in zip(rc[wq], dqc):
                    dq[dq_pos[int(row)], h] = val
            tail = rc >= key_lo
            if tail.any() and jmax > key_lo:
                dk[:jmax - key_lo, g] += scale * (ds[tail][:, key_lo:].T @ qc[tail])
                dv[:jmax - key_lo, g] += p[tail][:, key_lo:].T @ doc[tail]
    return dq, dk, dv


def causal_attention_bwd(q, k, v, do, scale=None):
    """Full gradients (dq [S][H][D], dk, dv [S][G][D]) of L = sum(O * dO)."""
    S = np.asarray(q).shape[0]
    return causal_attention_bwd_rows(q, k, v, do, np.arange(S), 0, scale)


# ------------------------------------------------------------------------ whole block
def ulysses_block_forward(x, w, P: int, H: int, G: int, D: int, theta: float = 0.0,
                          scale=None):
    """One Ulysses attention block, step by step   [UT para 2; USP paras 5, 7, 8].

    x: [S][hidden], w: [(H + 2G) * D][hidden].
      1. shard the sequence into P contiguous shards;
      2. each rank projects its tokens to q, k, v (and applies RoPE at global positions
         when theta > 0);
      3. seq->head all-to-all;
      4. each rank runs causal attention on its head group over the full sequence;
      5. head->seq all-to-all.
    Returns o_seq [P][S/P][H][D], lse [P][H/P][S] and the intermediate head tensors."""
    x = np.asarray(x, np.float64)
    S = x.shape[0]
    n = S // P
    local = []
    for r, xr in enumerate(shard_sequence(x, P)):
        y = qkv_projection(xr, w).reshape(n, H + 2 * G, D)
        if theta:
            pos = np.arange(r * n, (r + 1) * n)
            y = np.concatenate([apply_rope(y[:, :H + G], pos, theta), y[:, H + G:]], axis=1)
        local.append(y)
    qkv_seq = np.concatenate(local, axis=0)
    q, k, v = seq_to_head(qkv_seq, P, H, G)
    o_head, lse = ulysses_attention(q, k, v, scale)
    return head_to_seq(o_head, P), lse, (qkv_seq, q, k, v, o_head)


def a2a_volume_bytes(S: int, P: int, H: int, G: int, D: int, elem_bytes: int = 2):
    """Bytes one rank sends to the other ranks in one block's two all-to-alls.

    seq->head: the rank's S/P tokens of every head except its own group's;
    head->seq: its S tokens of its H/P output heads except its own token range.
    Both are (P-1)/P of a shard: (S/P) * (H + 2G) * D and (S/P) * H * D elements
    times (P-1)/P, i.e. O(hidden * S / P)   [UT para 3]."""
    n = S // P
    s2h = n * (H + 2 * G) * D * elem_bytes * (P - 1) // P
    h2s = n * H * D * elem_bytes * (P - 1) // P
    return s2h, h2s


# ------------------------------------------------------- rest of the block's backward
def rope_backward(g: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Gradient through rotate-half RoPE: each pair (i, i + D/2) was turned by the angle
    p * theta^(-2i/D); the gradient turns back by the same angle (the transpose of a
    rotation).  g: [T][n_heads][D]."""
    g = np.asarray(g, np.float64)
    half = g.shape[-1] // 2
    phi = rope_angles(positions, g.shape[-1], theta)[:, None, :]
    c, s = np.cos(phi), np.sin(phi)
    lo, hi = g[..., :half], g[..., half:]
    return np.concatenate([lo * c + hi * s, hi * c - lo * s], axis=-1)


def qkv_projection_backward(x: np.ndarray, w: np.ndarray, dy: np.ndarray):
    """Gradients of y = x w^T: dx = dy w ([T][hidden]), dw = dy^T x ([C][hidden])."""
    dy = np.asarray(dy, np.float64)
    return dy @ np.asarray(w, np.float64), dy.T @ np.asarray(x, np.float64)


def head_to_seq_qkv(dq_head, dk_head, dv_head, P: int) -> np.ndarray:
    """The three head-layout gradients back to the projection layout [S][H + 2G][D]:
    the inverse of seq_to_head, written as the same rank-to-rank exchange."""
    S = dq_head.shape[1]
    parts = [head_to_seq(t, P).reshape(S, -1, t.shape[-1]) for t in (dq_head, dk_head, dv_head)]
    return np.concatenate(parts, axis=1)


def ulysses_block_backward(x, w, do_seq, P: int, H: int, G: int, D: int, theta: float = 0.0,
                           scale=None):
    """Training step of one Ulysses block: gradients dx [S][hidden] and dw [C][hidden] of
    L = sum(o_seq * do_seq), following the forward's steps in reverse:
      dO seq->head; per-rank attention backward; head->seq of dq, dk, dv; RoPE backward
      at global positions; projection backward.
    Returns dx, dw and the intermediate dqkv_seq [S][H + 2G][D]."""
    x = np.asarray(x, np.float64)
    S = x.shape[0]
    _, _, (qkv_seq, q, k, v, _) = ulysses_block_forward(x, w, P, H, G, D, theta, scale)
    do_seq = np.asarray(do_seq, np.float64).reshape(S, H, D)
    do_head = np.stack([head for head in _seq_to_head_one(do_seq, P)])
    dq, dk, dv = [], [], []
    for r in range(P):
        a, b, c = causal_attention_bwd(q[r], k[r], v[r], do_head[r], scale)
        dq.append(a)
        dk.append(b)
        dv.append(c)
    dqkv = head_to_seq_qkv(np.stack(dq), np.stack(dk), np.stack(dv), P)
    if theta:
        pos = np.arange(S)
        dqkv = np.concatenate([rope_backward(dqkv[:, :H + G], pos, theta), dqkv[:, H + G:]],
                              axis=1)
    dx, dw = qkv_projection_backward(x, w, dqkv.reshape(S, -1))
    return dx, dw, dqkv


def _seq_to_head_one(x_seq: np.ndarray, P: int):
    """seq->head of one tensor [S][n][D] -> [P][S][n/P][D] (rank-to-rank exchange)."""
    S, n, D = x_seq.shape
    per, hl = S // P, n // P
    out = np.empty((P, S, hl, D), x_seq.dtype)
    for r in range(P):
        for r2 in range(P):
            out[r2, r * per:(r + 1) * per] = x_seq[r * per:(r + 1) * per, r2 * hl:(r2 + 1) * hl]
    return out


# ------------------------------------------------------------------ output projection
# After the second all-to-all restores the sequence sharding [UT para 2], the attention
# block ends, as every transformer attention block does, with its output projection
# y = o wo^T, o the rank's shard [S/P][H * D] and wo the nn.Linear weight [hidden][H * D].
def output_projection(o_seq: np.ndarray, wo: np.ndarray) -> np.ndarray:
    """y[t][j] = sum_c o[t][c] wo[j][c] with c = h * D + d; o_seq: [..][H][D] tokens."""
    o = np.asarray(o_seq, np.float64)
    o = o.reshape(-1, o.shape[-2] * o.shape[-1])
    return o @ np.asarray(wo, np.float64).T


def output_projection_backward(o_seq: np.ndarray, wo: np.ndarray, dy: np.ndarray):
    """Gradients of y = o wo^T: do = dy wo ([T][H * D]) and dwo = dy^T o ([hidden][H * D])."""
    o = np.asarray(o_seq, np.float64)
    o = o.reshape(-1, o.shape[-2] * o.shape[-1])
    dy = np.asarray(dy, np.float64)
    return dy @ np.asarray(wo, np.float64), dy.T @ o


def ulysses_layer_forward(x, w, wo, P: int, H: int, G: int, D: int, theta: float = 0.0,
                          scale=None):
    """The whole attention block: ulysses_block_forward, then each rank's output projection
    of its restored shard.  Returns y [S][hidden], lse and o_seq [P][S/P][H][D]."""
    o_seq, lse, _ = ulysses_block_forward(x, w, P, H, G, D, theta, scale)
    y = np.concatenate([output_projection(o_seq[r], wo) for r in range(P)], axis=0)
    return y, lse, o_seq


def ulysses_layer_backward(x, w, wo, dy, P: int, H: int, G: int, D: int, theta: float = 0.0,
                           scale=None):
    """Gradients of L = sum(y * dy) for the whole block: the output projection's backward
    per rank gives dO in the sequence layout and dwo (summed over all ranks' tokens), then
    ulysses_block_backward.  Returns dx, dw, dwo and dO_seq [S][H][D]."""
    o_seq, _, _ = ulysses_block_forward(x, w, P, H, G, D, theta, scale)
    S = np.asarray(x).shape[0]
    do_seq, dwo = output_projection_backward(o_seq.reshape(S, H, D), wo, dy)
    dx, dw, _ = ulysses_block_backward(x, w, do_seq, P, H, G, D, theta, scale)
    return dx, dw, dwo, do_seq.reshape(S, H, D)


# --------------------------------------------------------------- ring attention (comparator)
# The pages set Ulysses against ring attention, whose per-GPU communication is O(hidden * S)
# against Ulysses' O(hidden * S / P) [UT para 3].  Ring attention keeps the sequence sharding
# throughout: rank r holds its queries and, in step t = 0 .. P-1, the K/V shard
# (r - t) mod P; after each step every rank passes the shard it holds to rank r + 1.
def ring_attention(q_seq, k_seq, v_seq, scale=None):
    """Ring attention on P ranks, causal by global token position, GQA.

    q_seq [P][S/P][H][D]; k_seq, v_seq [P][S/P][G][D] (rank r starts with shard r).  Each
    rank keeps a running row max m, sum l and accumulator acc over the shards it has seen
    (rows of a step with no visible key leave the state unchanged) and divides by l at the
    end.  Returns o_seq [P][S/P][H][D], lse [P][H][S/P] and the bytes each rank sent
    (it forwards its K/V shard P - 1 times, bf16)."""
    q = np.asarray(q_seq, np.float64)
    k = np.asarray(k_seq, np.float64)
    v = np.asarray(v_seq, np.float64)
    P, n, H, D = q.shape
    G = k.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    m = np.full((P, H, n), -np.inf)
    l = np.zeros((P, H, n))
    acc = np.zeros((P, H, n, D))
    held_k, held_v = [k[r] for r in range(P)], [v[r] for r in range(P)]
    held_id = list(range(P))
    sent = 0
    for t in range(P):
        for r in range(P):
            j = held_id[r]
            rows = r * n + np.arange(n)
            keys = j * n + np.arange(n)
            visible = keys[None, :] <= rows[:, None]            # [row][key]
            if not visible.any():
                continue
            for h in range(H):
                g = _kv_head(h, H, G)
                s = scale * (q[r, :, h, :] @ held_k[r][:, g, :].T)
                s = np.where(visible, s, -np.inf)
                m_step = s.max(axis=1)
                m_new = np.maximum(m[r, h], m_step)
                keep = np.where(np.isfinite(m_new), np.exp(m[r, h] - m_new), 0.0)
                p = np.where(visible, np.exp(s - m_new[:, None]), 0.0)
                acc[r, h] = acc[r, h] * keep[:, None] + p @ held_v[r][:, g, :]
                l[r, h] = l[r, h] * keep + p.sum(axis=1)
                m[r, h] = m_new
        if t < P - 1:   # every rank passes the shard it holds to the next rank
            held_k = [held_k[(r - 1) % P] for r in range(P)]
            held_v = [held_v[(r - 1) % P] for r in range(P)]
            held_id = [held_id[(r - 1) % P] for r in range(P)]
            sent += n * 2 * G * D * 2
    o = (acc / l[..., None]).transpose(0, 2, 1, 3)             # [P][n][H][D]
    lse = m + np.log(l)
    return o, lse, sent


def ring_volume_bytes(S: int, P: int, G: int, D: int, elem_bytes: int = 2):
    """Bytes one rank sends in ring attention's forward: its K/V shard, forwarded P - 1
    times, (P - 1) * (S/P) * 2G * D elements."""
    return (P - 1) * (S // P) * 2 * G * D * elem_bytes
