"""Shared helpers for the GPU parity tests (tolerance, row sampling, comparison)."""
import numpy as np
import torch

# |O - O_ref| <= ATOL + RTOL * |O_ref| element-wise, |lse - lse_ref| <= LSE_ATOL.
ATOL = 4e-3
RTOL = 8e-3
LSE_ATOL = 1e-3


def check_out(got, ref, what=""):
    """got: bf16/fp32 tensor or array; ref: float64 array of the same shape."""
    if isinstance(got, torch.Tensor):
        got = got.detach().float().cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst excess {np.max(err - bound):.3g}; first at {idx.tolist()} "
                             f"(got {got[tuple(idx[0])]}, ref {ref[tuple(idx[0])]})")
    return float(err.max()) if err.size else 0.0


def check_lse(got, ref, what=""):
    if isinstance(got, torch.Tensor):
        got = got.detach().cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: lse shape {got.shape} vs {ref.shape}"
    inf_ref = np.isneginf(ref)
    assert (np.isneginf(got) == inf_ref).all(), f"{what}: -inf pattern of lse differs"
    fin = ~inf_ref
    err = np.abs(got[fin] - ref[fin])
    if err.size and err.max() > LSE_ATOL:
        raise AssertionError(f"{what}: lse error {err.max():.3g} > {LSE_ATOL}")
    return float(err.max()) if err.size else 0.0


def sample_rows(B, Hq, Sq, G, n_random=48, seed=0):
    """Rows (b, h, i) covering tile edges, the ragged tail, head-group edges and random picks."""
    rng = np.random.default_rng(seed)
    i_set = {0, 1, 31, 32, 63, 64, 127, 128, 129, 255, 256, Sq // 2, Sq - 129, Sq - 128, Sq - 2, Sq - 1}
    i_set = sorted(i for i in i_set if 0 <= i < Sq)
    h_set = sorted({0, G - 1, min(G, Hq - 1), Hq // 2, Hq - 1})
    b_set = sorted({0, B - 1})
    rows = [(b, h, i) for b in b_set for h in h_set for i in i_set]
    for _ in range(n_random):
        rows.append((int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(Sq))))
    return np.array(sorted(set(rows)), dtype=np.int64)


def gather_rows(out, lse, rows, layout):
    """Pick rows (b, h, i) out of a [B,S,H,d] / [B,H,S,d] output and a [B,H,S] lse."""
    b = torch.as_tensor(rows[:, 0])
    h = torch.as_tensor(rows[:, 1])
    i = torch.as_tensor(rows[:, 2])
    o = out.cpu()
    o_rows = o[b, i, h] if layout == "bshd" else o[b, h, i]
    l_rows = lse.cpu()[b, h, i]
    return o_rows, l_rows
