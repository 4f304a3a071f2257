"""Helpers shared by the GPU parity tests: device transfer of the seeded inputs and the
tolerance checks.  Attention outputs and gradients must satisfy max |err| <= 2e-2 and
mean |err| <= 2e-3 against the fp64 oracle; permutations must match bit for bit."""
import numpy as np
import torch

import synthetic
from tolerances import bf16_ulp  # noqa: F401  (also used by the tests through here)

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return synthetic.to_torch_bf16(bits).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return synthetic.torch_bf16_to_bits(t)


def host_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return synthetic.bf16_to_f64(host_bits(t))
    return t.detach().cpu().double().numpy()


def empty_bf16(shape):
    return torch.empty(shape, dtype=torch.bfloat16, device="cuda")


def assert_close(got, ref, name, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    """max |err| <= max_abs and mean |err| <= mean_abs.  A bf16 output of magnitude >= 4
    cannot be closer than half its ulp (>= 0.0156, 0.031 at >= 8) to the fp64 value, so
    per element the bound is max(max_abs, one bf16 ulp of the reference value)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s has non-finite values" % name
    d = np.abs(got - ref)
    if d.size == 0:
        return
    bound = np.maximum(max_abs, bf16_ulp(ref))
    excess = d / bound
    worst = np.unravel_index(np.argmax(excess), d.shape)
    msg = "%s: max|err| %.3g (bound there %.3g) at %s (got %.5g ref %.5g), mean|err| %.3g, " \
          "max|ref| %.3g" % (name, d[worst], bound[worst], worst, got[worst], ref[worst],
                             d.mean(), np.abs(ref).max())
    assert excess.max() <= 1.0 and d.mean() <= mean_abs, msg


def assert_close_f32(got, ref, name, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    """The same bounds for an fp32 output (the logsumexp): flat, with no widening by a bf16
    ulp, since an fp32 value carries 24 significant bits."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s has non-finite values" % name
    d = np.abs(got - ref)
    if d.size == 0:
        return
    worst = np.unravel_index(np.argmax(d), d.shape)
    msg = "%s: max|err| %.3g at %s (got %.7g ref %.7g), mean|err| %.3g, max|ref| %.3g" % (
        name, d[worst], worst, got[worst], ref[worst], d.mean(), np.abs(ref).max())
    assert d.max() <= max_abs and d.mean() <= mean_abs, msg
    return float(d.max())


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in units in the last place between bf16 bit patterns (same-sign ordering)."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(key(a_bits) - key(b_bits))
