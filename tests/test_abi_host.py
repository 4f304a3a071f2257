"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports every symbol
that include/ulysses.h declares, validates configs and reports the all-to-all volume."""
import os
import re

import pytest

import long_context_sequence_gb300 as U
import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build_library()
    return U.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "ulysses.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ulysses_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 13
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(names) == sorted(U.EXPORTED)


def test_config_validation_errors(lib):
    good = dict(seq_len=1024, P=4, hidden=512, n_q_heads=8, n_kv_heads=8, head_dim=64)
    cases = [
        (dict(n_kv_heads=6), U.ULY_ERR_INVALID_ARG),        # H % G
        (dict(n_q_heads=6, n_kv_heads=6), U.ULY_ERR_INVALID_ARG),   # H % P
        (dict(n_q_heads=8, n_kv_heads=2), U.ULY_ERR_UNSUPPORTED),   # G % P: replication
        (dict(head_dim=96), U.ULY_ERR_UNSUPPORTED),
        (dict(hidden=100), U.ULY_ERR_INVALID_ARG),
        (dict(seq_len=1022), U.ULY_ERR_INVALID_ARG),          # S % P
        (dict(P=0), U.ULY_ERR_INVALID_ARG),
        (dict(seq_len=-4), U.ULY_ERR_INVALID_ARG),
    ]
    for over, status in cases:
        cfg = U.make_config(**{**good, **over})
        with pytest.raises(U.UlyssesError) as ei:
            U.ulysses_a2a_volume(cfg)
        assert ei.value.status == status, (over, ei.value)
    cfg = U.make_config(**good)
    cfg.batch = 2
    with pytest.raises(U.UlyssesError) as ei:
        U.ulysses_a2a_volume(cfg)
    assert ei.value.status == U.ULY_ERR_UNSUPPORTED
    cfg = U.make_config(**good)
    cfg.causal = 0
    with pytest.raises(U.UlyssesError):
        U.ulysses_a2a_volume(cfg)
    cfg = U.make_config(**good, flags=0x80)
    with pytest.raises(U.UlyssesError):
        U.ulysses_a2a_volume(cfg)


@pytest.mark.parametrize("S,P,H,G,D", [(1024, 4, 8, 8, 64), (32768, 8, 32, 8, 128),
                                       (131072, 8, 32, 8, 128), (4096, 1, 8, 8, 128)])
def test_a2a_volume_matches_oracle_closed_form(lib, S, P, H, G, D):
    got = U.ulysses_a2a_volume(U.make_config(S, P, 4096, H, G, D))
    assert got == O.a2a_volume_bytes(S, P, H, G, D)


def test_null_plan_is_rejected(lib):
    class Fake:
        handle = None
    with pytest.raises(U.UlyssesError) as ei:
        U.ulysses_attn_fwd(Fake(), 0, 0, 0, 0, 0, stream=0)
    assert ei.value.status == U.ULY_ERR_INVALID_ARG
    assert "plan" in U.ulysses_last_error()


@pytest.mark.parametrize("S,P,H,G,D", [(131072, 8, 32, 8, 128), (1024, 4, 8, 8, 64), (8, 1, 2, 1, 64)])
def test_ring_volume_matches_oracle_closed_form(lib, S, P, H, G, D):
    assert U.ulysses_ring_volume(U.make_config(S, P, 4096, H, G, D)) == \
        O.ring_volume_bytes(S, P, G, D)


def test_missing_library_fails_loudly(tmp_path):
    """Without libulysses.so every entry point raises: there is no CPU or PyTorch fallback
    behind the binding.  (A fresh interpreter, so that this session's loaded library is not
    reused.)"""
    import subprocess
    import sys
    code = (
        "import functools\n"
        "import long_context_sequence_gb300 as U\n"
        "U.load_library = functools.partial(U.load_library, %r)\n"
        "failures = 0\n"
        "for call in (lambda: U.ulysses_plan(U.make_config(1024, 4, 512, 8, 8, 64)),\n"
        "             lambda: U.ulysses_last_error(),\n"
        "             lambda: U.ulysses_a2a_volume(U.make_config(1024, 4, 512, 8, 8, 64))):\n"
        "    try:\n"
        "        call()\n"
        "    except ImportError as e:\n"
        "        assert 'not built' in str(e)\n"
        "        failures += 1\n"
        "print(failures)\n"
    ) % str(tmp_path / "missing.so")
    env = dict(os.environ, PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         cwd=ROOT, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "3"


def test_a2a_table_host_only(lib):
    """The block table of a rank (no GPU): P equal contiguous blocks, block-major in both
    buffers; seq->head sends the rank's tokens of every peer's heads, head->seq the inverse."""
    cfg = U.make_config(seq_len=4096, P=8, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128)
    n = 4096 // 8
    for rank in (0, 3, 7):
        t = U.ulysses_a2a_table(cfg, rank, True, 32)
        assert [b["peer"] for b in t] == list(range(8))
        assert all(b["count"] == n * 4 * 128 and b["send_offset"] == b["peer"] * b["count"] ==
                   b["recv_offset"] for b in t)
        assert all(b["send_token_begin"] == rank * n and b["send_head_begin"] == 4 * b["peer"] and
                   b["recv_token_begin"] == b["peer"] * n and b["recv_head_begin"] == 4 * rank
                   for b in t)
        back = U.ulysses_a2a_table(cfg, rank, False, 8)
        assert all(b["send_token_begin"] == b["peer"] * n and b["send_head_begin"] == rank and
                   b["recv_token_begin"] == rank * n and b["recv_head_begin"] == b["peer"]
                   for b in back)
    for bad in (dict(rank=8, to_head=True, n_heads=32), dict(rank=-1, to_head=True, n_heads=32),
                dict(rank=0, to_head=False, n_heads=16)):
        with pytest.raises(U.UlyssesError) as ei:
            U.ulysses_a2a_table(cfg, **bad)
        assert ei.value.status == U.ULY_ERR_INVALID_ARG
