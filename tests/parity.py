"""Parity rules between the CUDA path and the fp64 oracle.

Selection: the GPU's set must equal the oracle's, except for blocks whose fp64
score lies within 1e-4 relative of the oracle's k-th score; a swap outside that
band is still accepted (and counted separately) when the two scores differ by less
than the fp32 dot-product error bound, because fp32 accumulation cannot order them.
Callers assert how many such fp32-bound swaps they accept (zero unless stated).

Attention (graded on the GPU's own selection): max |out - ref| <= 2e-2 and mean
|out - ref| <= 2e-3 (the stated absolute rule), and also ||out - ref|| / ||ref|| <= 8e-3.
The absolute rule alone cannot fail on the N(0,1)/sqrt(256) inputs: their outputs are
about 1e-3, so an all-zero output would pass it. A correct bf16 output sits at a relative
error of about 1.7e-3 (one rounding to 8 significant bits); dropping one selected block
moves it by 2e-2 or more and dropping one token by about 1e-2 to 2e-2, on both the
stated and the sharp distribution (tests/test_parity_rules.py plants both mistakes in
the oracle and checks that these rules reject them). The lse must agree to 2.5e-4:
one dropped token of 2052 near-uniform ones moves it by 4.9e-4.
"""

import numpy as np
import torch

import oracle as O
from oracle import qsa_oracle as OQ

SEL_BAND = 1e-4
ATT_MAX_ABS = 2e-2
ATT_MEAN_ABS = 2e-3
ATT_REL = 8e-3
LSE_ABS = 2.5e-4


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit array (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def check_selection(gpu_blocks, gpu_count, q_idx_bits, pooled_bits, nb, k=O.BLOCK_TOPK, scores=None, bound=None):
    """Compare one row's GPU selection with the oracle's. Returns counts of
    (exempt swaps within the band, swaps accepted only under the fp32 bound).
    ``scores`` / ``bound`` override the bf16 scores (for FP8 keys)."""
    if scores is None:
        scores = O.score_blocks(q_idx_bits, pooled_bits[:nb])
        bound = None
    want = O.select_blocks(scores, k)
    kk = min(k, nb)
    assert gpu_count == kk, (gpu_count, kk)
    got = np.asarray(gpu_blocks[:kk], dtype=np.int64)
    assert np.all(np.diff(got) > 0), "selection not strictly ascending"
    assert got.size == 0 or (got[0] >= 0 and got[-1] < nb)
    assert np.all(np.asarray(gpu_blocks[kk:]) == -1)
    diff = np.setxor1d(got, want)
    if diff.size == 0:
        return 0, 0
    kth = O.kth_score(scores, k)
    if bound is None:
        bound = O.score_error_bound(q_idx_bits, pooled_bits[:nb])
    kth_bound = bound[OQ._rank_order(scores)[kk - 1]]
    gap = np.abs(scores[diff] - kth)
    in_band = gap <= SEL_BAND * abs(kth)
    in_fp32 = ~in_band & (gap <= bound[diff] + kth_bound)
    assert np.all(in_band | in_fp32), (diff[~(in_band | in_fp32)], gap[~(in_band | in_fp32)], kth)
    return int(in_band.sum()), int(in_fp32.sum())


def check_attention(gpu_out, ref_out, max_abs=ATT_MAX_ABS, mean_abs=ATT_MEAN_ABS, rel=ATT_REL):
    """gpu_out: bf16 tensor or float array; ref_out: float64 array of the same shape.
    Returns (max abs error, mean abs error, relative norm error)."""
    g = gpu_out.float().cpu().numpy().astype(np.float64) if isinstance(gpu_out, torch.Tensor) else gpu_out
    g = np.asarray(g, dtype=np.float64)
    err = np.abs(g - ref_out)
    assert np.all(np.isfinite(g))
    assert err.max() <= max_abs, err.max()
    assert err.mean() <= mean_abs, err.mean()
    ref_norm = np.linalg.norm(ref_out)
    r = float(np.linalg.norm(g - ref_out) / max(ref_norm, 1e-300))
    # the relative rule applies whenever the reference is not negligibly small (1e-6 rms)
    if ref_norm > 1e-6 * np.sqrt(ref_out.size):
        assert r <= rel, f"relative error {r:.3e} > {rel:.1e}"
    return float(err.max()), float(err.mean()), r


def check_lse(gpu_lse, ref_lse, tol=LSE_ABS):
    """fp32 lse of the GPU against the oracle's fp64 lse."""
    g = np.asarray(gpu_lse, dtype=np.float64)
    d = float(np.max(np.abs(g - ref_lse))) if g.size else 0.0
    assert d <= tol, f"lse differs by {d:.3e} > {tol:.1e}"
    return d
