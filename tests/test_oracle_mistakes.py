"""Planted mistakes: every plausible slip in the oracle makes some pin of test_oracle.py fail.

Each case edits one snippet of one oracle function's own source, on the CPU:
- a flipped sign;
- a wrong or swapped index;
- a dropped term or scale;
- a transposed operand;
- an off-by-one mask;
- a wrong convention.

The edited function is re-executed with the oracle module's globals and patched in for the
duration of the test. Then every pin of test_oracle.py runs, with all its parameter sets,
and at least one must fail. This shows that the pins constrain the oracle, rather than
merely agreeing with it."""
import __future__
import inspect

import numpy as np
import pytest

import oracle
import test_oracle as pins
from oracle import ulysses_oracle as U

# (case, oracle function, snippet, replacement)
MISTAKES = [
    # all-to-alls
    ("a2a q from the sender's head group", "seq_to_head",
     "q[r2, r * n:(r + 1) * n] = local[:, r2 * hq:(r2 + 1) * hq]",
     "q[r2, r * n:(r + 1) * n] = local[:, r * hq:(r + 1) * hq]"),
    ("a2a k read from the q columns", "seq_to_head",
     "local[:, H + r2 * hk:H + (r2 + 1) * hk]", "local[:, r2 * hk:(r2 + 1) * hk]"),
    ("a2a v read from the k columns", "seq_to_head",
     "local[:, H + G + r2 * hk:H + G + (r2 + 1) * hk]", "local[:, H + r2 * hk:H + (r2 + 1) * hk]"),
    ("head->seq with sender and receiver swapped", "head_to_seq",
     "x_head[r2, r * n:(r + 1) * n]", "x_head[r, r2 * n:(r2 + 1) * n]"),
    ("a2a volume without one of k, v", "a2a_volume_bytes",
     "n * (H + 2 * G) * D", "n * (H + G) * D"),
    # projection
    ("projection with w not transposed", "qkv_projection",
     "@ np.asarray(w, np.float64).T", "@ np.asarray(w, np.float64)"),
    # RoPE
    ("RoPE turning the wrong way", "apply_rope",
     "[lo * c - hi * s, hi * c + lo * s]", "[lo * c + hi * s, hi * c - lo * s]"),
    ("RoPE frequency exponent -i/D", "rope_angles",
     "theta ** (-2.0 * i / head_dim)", "theta ** (-1.0 * i / head_dim)"),
    ("RoPE on interleaved pairs", "apply_rope",
     "lo, hi = x[..., :half], x[..., half:]", "lo, hi = x[..., 0::2], x[..., 1::2]"),
    ("RoPE at shard-local positions", "ulysses_block_forward",
     "pos = np.arange(r * n, (r + 1) * n)", "pos = np.arange(0, n)"),
    ("RoPE applied to v as well", "ulysses_block_forward",
     "[apply_rope(y[:, :H + G], pos, theta), y[:, H + G:]]",
     "[apply_rope(y[:, :H + 2 * G], pos, theta), y[:, H + 2 * G:]]"),
    ("RoPE backward turning forward again", "rope_backward",
     "[lo * c + hi * s, hi * c - lo * s]", "[lo * c - hi * s, hi * c + lo * s]"),
    # attention forward
    ("causal mask letting in one future key", "causal_attention_rows",
     "s[np.arange(jmax)[None, :] > rc[:, None]] = -np.inf",
     "s[np.arange(jmax)[None, :] > rc[:, None] + 1] = -np.inf"),
    ("causal mask hiding the diagonal", "causal_attention_rows",
     "s[np.arange(jmax)[None, :] > rc[:, None]] = -np.inf",
     "s[np.arange(jmax)[None, :] >= rc[:, None]] = -np.inf"),
    ("softmax scale dropped", "causal_attention_rows",
     "s = scale * (qc @ kh[:jmax].T)", "s = (qc @ kh[:jmax].T)"),
    ("softmax not normalised", "causal_attention_rows",
     "(p @ vh[:jmax]) / l", "(p @ vh[:jmax])"),
    ("logsumexp in base 2", "causal_attention_rows",
     "(m + np.log(l))[:, 0]", "(m + np.log2(l))[:, 0]"),
    ("GQA: query head h on KV head h mod G", "_kv_head",
     "return h // (H // G)", "return h % G"),
    # attention backward
    ("backward without the D term", "causal_attention_bwd_rows",
     "ds = p * (dp - delta)", "ds = p * dp"),
    ("backward dq without the scale", "causal_attention_bwd_rows",
     "dqc = scale * (ds[wq] @ kh[:jmax])", "dqc = (ds[wq] @ kh[:jmax])"),
    ("backward dv from dS instead of P", "causal_attention_bwd_rows",
     "+= p[tail][:, key_lo:].T @ doc[tail]", "+= ds[tail][:, key_lo:].T @ doc[tail]"),
    ("backward dk against dO instead of q", "causal_attention_bwd_rows",
     "(ds[tail][:, key_lo:].T @ qc[tail])", "(ds[tail][:, key_lo:].T @ doc[tail])"),
    ("backward mask hiding the diagonal", "causal_attention_bwd_rows",
     "mask = np.arange(jmax)[None, :] > rc[:, None]",
     "mask = np.arange(jmax)[None, :] >= rc[:, None]"),
    # rest of the training step
    ("projection backward dw transposed", "qkv_projection_backward",
     "dy.T @ np.asarray(x, np.float64)", "np.asarray(x, np.float64).T @ dy"),
    ("projection backward dx against w transposed", "qkv_projection_backward",
     "dy @ np.asarray(w, np.float64)", "dy @ np.asarray(w, np.float64).T"),
    ("output projection with wo not transposed", "output_projection",
     "o @ np.asarray(wo, np.float64).T", "o @ np.asarray(wo, np.float64)"),
    ("output projection backward dwo transposed", "output_projection_backward",
     "dy.T @ o", "o.T @ dy"),
    # ring attention
    ("ring passes K one way and V the other", "ring_attention",
     "held_k = [held_k[(r - 1) % P] for r in range(P)]",
     "held_k = [held_k[(r + 1) % P] for r in range(P)]"),
    ("ring accumulator not rescaled", "ring_attention",
     "acc[r, h] = acc[r, h] * keep[:, None] + p @ held_v[r][:, g, :]",
     "acc[r, h] = acc[r, h] + p @ held_v[r][:, g, :]"),
    ("ring volume without V", "ring_volume_bytes",
     "(P - 1) * (S // P) * 2 * G * D * elem_bytes", "(P - 1) * (S // P) * G * D * elem_bytes"),
]


def _pin_calls():
    """Every pin of test_oracle.py with every parameter set: (label, function, args)."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        sets = [()]
        for mark in getattr(fn, "pytestmark", []):
            if mark.name == "parametrize":
                sets = [v if isinstance(v, tuple) else (v,) for v in mark.args[1]]
        calls += [("%s%s" % (name, list(args) if args else ""), fn, args) for args in sets]
    return calls


def _plant(monkeypatch, fname, snippet, replacement):
    """Replace `snippet` in the source of oracle function `fname` and patch the result in."""
    src = inspect.getsource(getattr(U, fname))
    assert src.count(snippet) == 1, "snippet not found once in %s" % fname
    code = compile(src.replace(snippet, replacement), U.__file__, "exec",
                   flags=__future__.annotations.compiler_flag, dont_inherit=True)
    local = {}
    exec(code, U.__dict__, local)
    monkeypatch.setattr(U, fname, local[fname])
    if fname in vars(oracle):
        monkeypatch.setattr(oracle, fname, local[fname])


def _failing_pins():
    """Labels of the pins that fail (an assertion or any other error) on the oracle as patched."""
    failed = []
    with np.errstate(all="ignore"):   # a planted mistake may produce NaN or inf
        for label, fn, args in _pin_calls():
            try:
                fn(*args)
            except Exception:
                failed.append(label)
    return failed


def test_pins_pass_on_the_oracle_as_written():
    assert _failing_pins() == []


@pytest.mark.parametrize("case,fname,snippet,replacement", MISTAKES, ids=[m[0] for m in MISTAKES])
def test_planted_mistake_fails_a_pin(monkeypatch, case, fname, snippet, replacement):
    _plant(monkeypatch, fname, snippet, replacement)
    assert _failing_pins(), "no pin catches: " + case
