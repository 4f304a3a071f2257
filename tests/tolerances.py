"""Error bounds the GPU parity tests hold the kernels to (numpy only, no GPU needed).

They live apart from the GPU tests so that CPU tests can check the derivations themselves:
that the bounds admit the kernels' declared roundings, and that coarser roundings exceed them."""
import numpy as np


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at the magnitude of x (normal range)."""
    return 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126))) - 7)


def peaked_bounds(q, k, v, do, H, G):
    """Per-element error bounds of one rank's attention from its arithmetic, for the peaked
    regime, where the magnitudes outgrow the absolute 2e-2 / 2e-3 bounds.  Built from the
    fp64 quantities of the definition (P, dP, D, dS):
      O:   P V with bf16 P (relative 2^-9 per weight) and fp32 sums: 2^-8 sum_j P_ij |v_j|;
      dV:  fp16 P (2^-12) and fp32 sums:                     2^-11 sum_i P_ij |dO_i|;
      dK:  fp16 dS (2^-12) and fp32 sums:            2^-11 scale sum_i |dS_ij| |q_i|;
      dQ:  likewise                                   2^-11 scale sum_j |dS_ij| |k_j|;
    and, through dS_ij = P_ij (dP_ij - D_i), the row term D_i = dO_i . O_i formed from O held
    as bf16 plus its bf16 residual (relative 2^-16, fp32 dot): |dD_i| <= 2^-15 sum |dO_i O_i|,
    adding scale |dD_i| sum_j P_ij |k_j| to dQ and scale sum_i P_ij |dD_i| |q_i| to dK;
    and fp16's subnormal floor: the stored scale*P and scale*dS below 2^-14 round to a
    2^-24 grid, an absolute 2^-25 each, adding 2^-25 sum over visible keys |k_j| to dQ,
    2^-25 sum over visible queries |q_i| to dK and 2^-25 / scale sum |dO_i| to dV;
    each plus one bf16 ulp of the value for the output's own rounding (in the check)."""
    S, hl, D = q.shape
    gl = k.shape[1]
    grp = hl // gl
    scale = 1.0 / np.sqrt(D)
    bo, bq = np.zeros_like(q), np.zeros_like(q)
    bk, bv = np.zeros_like(k), np.zeros_like(v)
    mask = np.tril(np.ones((S, S), bool))
    for h in range(hl):
        g = h // grp
        s = np.where(mask, scale * q[:, h] @ k[:, g].T, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        o = p @ v[:, g]
        dp = do[:, h] @ v[:, g].T
        ds = np.where(mask, p * (dp - np.sum(do[:, h] * o, axis=1, keepdims=True)), 0.0)
        dd = 2.0 ** -15 * np.sum(np.abs(do[:, h] * o), axis=1)          # |error of D_i|
        bo[:, h] = 2.0 ** -8 * (p @ np.abs(v[:, g]))
        bq[:, h] = 2.0 ** -11 * scale * (np.abs(ds) @ np.abs(k[:, g])) + \
            scale * dd[:, None] * (p @ np.abs(k[:, g]))
        bk[:, g] += 2.0 ** -11 * scale * (np.abs(ds).T @ np.abs(q[:, h])) + \
            scale * (p * dd[:, None]).T @ np.abs(q[:, h])
        bv[:, g] += 2.0 ** -11 * (p.T @ np.abs(do[:, h]))
        m = mask.astype(np.float64)
        bq[:, h] += 2.0 ** -25 * (m @ np.abs(k[:, g]))
        bk[:, g] += 2.0 ** -25 * (m.T @ np.abs(q[:, h]))
        bv[:, g] += 2.0 ** -25 / scale * (m.T @ np.abs(do[:, h]))
    return bo, bq, bk, bv


def assert_within(got, ref, bound, name):
    err = np.abs(np.asarray(got, np.float64) - ref)
    lim = bound + bf16_ulp(ref)
    worst = np.unravel_index(np.argmax(err / lim), err.shape)
    assert np.all(err <= lim), "%s: err %.3g > bound %.3g at %s" % (name, err[worst], lim[worst], worst)


def assert_rel(got, ref, name, rel_max=2e-2, rel_norm=1.5e-2):
    """End-to-end gradients against the unrounded fp64 pipeline, scaled to the gradient's
    magnitude: dw is a sum over all S tokens (|dw| reaches ~100 on the 8B shape), so an
    absolute bound does not fit it.  Storage of every intermediate in bf16 alone gives
    max|err|/max|ref| ~ 6e-3 and a normwise error ~ 6e-3 on the 8B shape."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape and np.all(np.isfinite(got)), name
    d = np.abs(got - ref)
    m = np.abs(ref).max()
    rn = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert d.max() <= rel_max * m and rn <= rel_norm, \
        "%s: max|err| %.3g (max|ref| %.3g), normwise %.3g" % (name, d.max(), m, rn)
