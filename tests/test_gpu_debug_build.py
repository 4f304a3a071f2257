"""Out-of-bounds evidence without compute-sanitizer.

Every output and workspace of the block's calls (projection, both all-to-alls, attention
forward and backward, the gradient permute with the RoPE backward, the projection and
output-projection backwards, ring attention, and one real rank's pack and unpack calls) sits
between NaN-filled guard bands; after the calls the bands must be untouched.  The release
library runs in this process; the debug build (libulysses_debug.so, built with ULY_DEBUG:
every kernel checks every global index it computes against its buffer's extent and counts
the misses, which ulysses_sync_status reports as ULY_ERR_BOUNDS) runs in a child process on
the same cases.  The cases are the tiny block and ragged shapes."""
import os
import subprocess
import sys

import pytest

import canary_block

pytestmark = pytest.mark.gpu

CASES = [  # S, P, hidden, H, G, D, theta
    (1024, 4, 512, 8, 8, 64, 0.0),           # the tiny block
    (1000, 4, 200, 8, 4, 128, 500000.0),     # ragged tail, GQA, RoPE
    (130, 1, 64, 2, 1, 128, 10000.0),        # one rank, a tail of 2 rows
    (24, 8, 64, 8, 8, 64, 0.0),              # three tokens per rank
]


@pytest.mark.parametrize("case", CASES)
def test_release_library_writes_nothing_outside_its_outputs(case):
    broken, statuses, err, msg = canary_block.run(*case)
    assert not broken, "guard bands changed: %s" % broken
    assert all(s == 0 for s in statuses), (statuses, msg)
    assert err < 5e-2


@pytest.mark.parametrize("case", CASES)
def test_debug_build_finds_no_out_of_bounds_index(case):
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, ULY_LIBRARY="debug")
    res = subprocess.run([sys.executable, os.path.join(here, "canary_block.py"), *map(str, case)],
                         capture_output=True, text=True, env=env, timeout=600)
    assert res.returncode == 0 and "CANARY OK" in res.stdout, res.stdout + res.stderr
    assert "libulysses_debug.so" in res.stdout
