"""Shared helpers of the GPU parity tests (comparison and row sampling)."""

import numpy as np

# Tolerances against the float64 oracle (same seeded inputs on both sides):
# bf16 inputs with float32 accumulation: max-abs 2e-2 and mean-abs 2e-3, on
# the output and on the lse; float32 inputs: 1e-4 on both.
TOL = {"bf16": (2e-2, 2e-3), "f32": (1e-4, 1e-4)}


def errors(got, want):
    """(max-abs, mean-abs) error over the finite entries of ``want``; the
    -inf entries of ``want`` must be -inf in ``got`` too."""
    g = got.detach().to("cpu").double().numpy() if hasattr(got, "detach") else np.asarray(got)
    w = np.asarray(want, dtype=np.float64)
    assert g.shape == w.shape, (g.shape, w.shape)
    ninf = np.isneginf(w)
    if ninf.any():
        assert np.array_equal(np.isneginf(g), ninf), "-inf pattern differs"
    fin = ~ninf
    if not fin.any():
        return 0.0, 0.0
    d = np.abs(g[fin] - w[fin])
    assert np.all(np.isfinite(d)), "non-finite values in the result"
    return float(d.max()), float(d.mean())


def assert_close(got, want, kind, what=""):
    mx, mean = errors(got, want)
    tmax, tmean = TOL[kind]
    assert mx <= tmax and mean <= tmean, (
        f"{what}: max-abs {mx:.3e} (tol {tmax}), mean-abs {mean:.3e} (tol {tmean})")
    return mx, mean


def sample_rows(S, seg_len, n_random, seed):
    """Every segment boundary row (first and last of each segment) plus
    ``n_random`` seeded random rows; sorted, unique."""
    rows = set()
    for s in range(0, S, seg_len):
        rows.add(s)
        rows.add(min(S - 1, s + seg_len - 1))
    rows.update(np.random.default_rng(seed).integers(0, S, n_random).tolist())
    rows.add(S - 1)
    return np.array(sorted(rows), dtype=np.int64)


def decode_visit_log(log, B, H, n_qt, stride):
    """int32 log -> nested lists [b][h][query tile] of 4-tuples."""
    a = log.detach().to("cpu").numpy().reshape(B, H, n_qt, stride)
    res = []
    for b in range(B):
        hb = []
        for h in range(H):
            tiles = []
            for q in range(n_qt):
                n = int(a[b, h, q, 0])
                e = a[b, h, q, 1:1 + 4 * n].reshape(n, 4)
                tiles.append([tuple(int(x) for x in row) for row in e])
            hb.append(tiles)
        res.append(hb)
    return res
