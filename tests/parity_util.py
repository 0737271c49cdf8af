"""Shared helpers of the GPU parity tests: tolerance checks against the float64 oracle.

Tolerances (bf16 inputs, fp32 accumulation):
  * outputs: max |O_gpu - O_oracle| <= 1e-2.  Outputs the library rounds to bf16 (the merged
    output of bf16 inputs, round to nearest even) additionally get the rounding bound of that
    format, half an ulp <= 2^-8 |O| per element (8 significant bits): with few visible keys O is
    close to a single N(0,1) value row and |O| reaches ~4.5, where rounding alone is ~0.018;
  * the probabilities P enter the tensor-core PV product as bf16 (its operands are bf16), so an
    output element of a partial carries up to 2^-8 sum_j p_j |v_j| / l of rounding besides: a
    check given o_abs (the oracle's partial attention of |V|, that weighted sum) adds
    2^-8 o_abs.  It matters when one or two keys dominate a partial and their |v| is large;
  * LSE: |LSE_gpu - LSE_oracle| <= 1e-3 |LSE_oracle| + 1e-5.  The absolute floor covers rows
    whose LSE is near 0: fp32 dot products of 128 bf16 products of unit scale carry ~1e-6
    absolute error, far inside 1e-5;
  * an empty partial must be empty (-inf) on both sides: that set is decided by integers
    (positions, chunk bounds, round-robin ranks), so it is compared exactly.
"""
import numpy as np
import torch

ATOL_O = 1e-2
RTOL_LSE = 1e-3
ATOL_LSE = 1e-5
BF16_HALF_ULP_REL = 2.0 ** -8


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def check_partials(out, lse, O_ref, L_ref, rows=None, what="", o_abs=None):
    """out [P, R, H, d], lse [P, R, H] (GPU, full) vs oracle [P, R', H, d] on rows (or all);
    o_abs (same shape as O_ref): the oracle's partials of |V|, for the bound of P's bf16
    rounding."""
    if rows is not None:
        idx = torch.as_tensor(rows, device=lse.device, dtype=torch.long)
        out = out.index_select(1, idx)
        lse = lse.index_select(1, idx)
    lse = to_np(lse)
    out = to_np(out)
    fin_ref = np.isfinite(L_ref)
    fin = np.isfinite(lse)
    assert not np.isnan(lse).any(), f"{what}: NaN in lse"
    assert np.array_equal(fin, fin_ref), f"{what}: empty-partial sets differ " \
        f"({int((fin != fin_ref).sum())} entries)"
    dl = np.abs(lse[fin] - L_ref[fin])
    tol = RTOL_LSE * np.abs(L_ref[fin]) + ATOL_LSE
    assert (dl <= tol).all(), f"{what}: lse max err {dl.max():.3e} (worst ratio {(dl / tol).max():.2f})"
    do = np.abs(out[fin] - O_ref[fin])
    assert np.isfinite(out[fin]).all(), f"{what}: non-finite output"
    tol_o = ATOL_O + (BF16_HALF_ULP_REL * o_abs[fin] if o_abs is not None else 0.0)
    assert (do <= tol_o).all(), f"{what}: out max err {do.max(initial=0):.3e} " \
        f"(worst ratio {(do / tol_o).max(initial=0):.2f})"
    return float(do.max(initial=0)), float(dl.max(initial=0))


def check_merged(out, lse, O_ref, L_ref, what="", o_abs=None):
    """Merged output vs the oracle; o_abs: the oracle's merged attention of |V| (the bound of
    P's bf16 rounding, see the module docstring)."""
    rounded = out.dtype == torch.bfloat16
    out = to_np(out)
    do = np.abs(out - O_ref)
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    tol = ATOL_O + (BF16_HALF_ULP_REL * np.abs(O_ref) if rounded else 0.0)
    if o_abs is not None:
        tol = tol + BF16_HALF_ULP_REL * o_abs
    assert (do <= tol).all(), f"{what}: merged out max err {do.max():.3e} " \
        f"(worst ratio {(do / tol).max():.2f})"
    if lse is not None:
        lse = to_np(lse)
        fin = np.isfinite(L_ref)
        assert np.array_equal(np.isfinite(lse), fin)
        dl = np.abs(lse[fin] - L_ref[fin])
        assert (dl <= RTOL_LSE * np.abs(L_ref[fin]) + ATOL_LSE).all(), \
            f"{what}: merged lse max err {dl.max():.3e}"
    return float(do.max(initial=0))


def check_same_rounded(a, b, what=""):
    """Two bf16 outputs of the same exact attention computed along different paths: each is
    within the f32 error of the truth before rounding, and the two roundings may land one ulp
    apart (<= 2^-7 |x|)."""
    a, b = to_np(a), to_np(b)
    tol = ATOL_O + 2 * BF16_HALF_ULP_REL * np.abs(b)
    d = np.abs(a - b)
    assert (d <= tol).all(), f"{what}: max diff {d.max():.3e} (worst ratio {(d / tol).max():.2f})"
