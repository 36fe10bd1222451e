"""Comparison helpers shared by the GPU tests (no method arithmetic here)."""
import numpy as np

# Output tolerances: bf16 inputs vs the fp64 oracle (max-abs, mean-abs), and
# the fp32 workload.
TOL_BF16 = (2e-2, 1e-2)
TOL_F32 = (1e-5, 1e-5)
# lse_out on the bf16 tensor-core path: the softmax weights are rounded to bf16
# (an 8-bit significand, unit roundoff u = 2^-8) before they are summed, so
# with every weight off by a relative |d| <= u the sum l is off by at most a
# factor (1 +- u) and ln(l) by at most -ln(1 - u) = 3.91e-3 (max-abs; 4e-3
# with the fp32 noise of the scores and the merge).  The rounding errors are
# unbiased, so over heads whose sums mix many weights the mean stays far
# below that (about u / sqrt(3 n) for n comparable terms): mean-abs 5e-4.
TOL_LSE_BF16 = (4e-3, 5e-4)
TOL_LSE_F32 = (1e-5, 1e-5)
# Top-K: two index sets may differ only in elements whose oracle score lies
# within this relative distance of the K-th oracle score.
TOPK_REL = 1e-6


def tol_for(cfg):
    return TOL_F32 if cfg.dtype == "f32" else TOL_BF16


def assert_close(got, ref, tol, what=""):
    err = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert err.max() <= tol[0] and err.mean() <= tol[1], \
        f"{what}: max-abs {err.max():.3e} (tol {tol[0]}), mean-abs {err.mean():.3e} (tol {tol[1]})"
    return float(err.max()), float(err.mean())


def assert_topk_sets(gpu_idx, gpu_cnt, ref, scores_of, K, what=""):
    """gpu_idx [nq,K], gpu_cnt [nq] against oracle results `ref` (decode() dict).

    Counts must match exactly; index lists must be ascending and -1 padded;
    sets must be identical except for elements whose oracle score is within
    TOPK_REL of the K-th oracle score (scores_of(q) returns the fp64 oracle
    scores of query q).  Returns the number of queries with a tolerated swap.
    """
    swaps = 0
    for q in range(gpu_idx.shape[0]):
        c = int(ref["cnt"][q])
        assert int(gpu_cnt[q]) == c, f"{what} q{q}: count {int(gpu_cnt[q])} != {c}"
        gi = gpu_idx[q]
        assert (gi[c:] == -1).all(), f"{what} q{q}: padding not -1"
        assert (np.diff(gi[:c]) > 0).all(), f"{what} q{q}: not ascending / duplicates"
        g, o = set(gi[:c].tolist()), set(ref["topk_idx"][q, :c].tolist())
        if g == o:
            continue
        sc = scores_of(q)
        kth = min(sc[list(o)])
        for x in g ^ o:
            assert 0 <= x < len(sc), f"{what} q{q}: index {x} out of range"
            lim = TOPK_REL * max(abs(sc[x]), abs(kth))
            assert abs(sc[x] - kth) <= lim, \
                f"{what} q{q}: set differs at {x}: score {sc[x]!r} vs K-th {kth!r}"
        swaps += 1
    return swaps
