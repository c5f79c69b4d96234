"""Coefficients of the residual weight's polynomial in the CUDA kernels.

The kernels form 1 - 2^delta for delta in [-1/2, 0] as delta * p(delta), with
p a degree-4 polynomial fitted to (1 - 2^delta) / delta by the Remez exchange
algorithm on relative error (the minimax fit; Remez, 1934).  This script
recomputes OMC1..OMC5 of specverify.cu, the maximum relative error of the fit
in fp64, and that of the kernels' fp32 evaluation (Horner with fused
multiply-adds, coefficients rounded to fp32), against -expm1(delta ln 2).

    python fit_one_minus_exp2.py
"""
import numpy as np

LO, HI, DEG = -0.5, 0.0, 4
LN2 = np.log(2.0)


def target(d):
    """(1 - 2^d) / d, with its limit -ln 2 at d = 0."""
    d = np.asarray(d, dtype=np.float64)
    out = np.full_like(d, -LN2)
    nz = d != 0.0
    out[nz] = -np.expm1(d[nz] * LN2) / d[nz]
    return out


def remez(deg, grid, iters=40):
    """Minimax polynomial (increasing powers) of `target` on `grid`, relative error."""
    m = deg + 2
    ref = (np.cos(np.pi * np.arange(m) / (m - 1))[::-1] + 1) / 2 * (HI - LO) + LO
    gg = target(grid)
    for _ in range(iters):
        a = np.zeros((m, m))
        a[:, :deg + 1] = np.vander(ref, deg + 1, increasing=True)
        a[:, deg + 1] = (-1.0) ** np.arange(m) * target(ref)
        c = np.linalg.solve(a, target(ref))[:deg + 1]
        err = np.vander(grid, deg + 1, increasing=True) @ c / gg - 1
        cut = np.flatnonzero(np.diff(np.sign(err)) != 0) + 1
        bounds = np.concatenate([[0], cut, [len(grid)]])
        ext = np.array([b0 + np.argmax(np.abs(err[b0:b1])) for b0, b1 in zip(bounds[:-1], bounds[1:])])
        while len(ext) > m:  # keep m alternating extrema: drop the smaller end
            ext = ext[1:] if abs(err[ext[0]]) < abs(err[ext[-1]]) else ext[:-1]
        if len(ext) == m:
            ref = grid[ext]
    return c, np.abs(err).max()


def fp32_eval_error(c, grid):
    """Maximum relative error of delta * p(delta) evaluated as the kernels do in fp32."""
    c32 = np.asarray(c, dtype=np.float32)
    d = grid.astype(np.float32)
    d = d[d < 0]
    p = np.full_like(d, c32[-1])
    for cj in c32[-2::-1]:  # fused multiply-add: one rounding per step
        p = (p.astype(np.float64) * d.astype(np.float64) + np.float64(cj)).astype(np.float32)
    f = (p.astype(np.float64) * d.astype(np.float64)).astype(np.float32)
    exact = -np.expm1(d.astype(np.float64) * LN2)
    return np.abs(f.astype(np.float64) / exact - 1).max()


def main():
    grid = np.linspace(LO, HI, 400001)
    c, e = remez(DEG, grid)
    print(f"minimax relative error of p on [{LO}, {HI}]: {e:.3g}")
    print(f"fp32 evaluation, maximum relative error: {fp32_eval_error(c, grid):.3g}")
    for j, v in enumerate(c, 1):
        print(f"OMC{j} = {v:.17g}")


if __name__ == "__main__":
    main()
