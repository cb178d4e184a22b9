"""Parity rules between the CUDA path and the fp64 oracle.

Selection: the GPU's set must equal the oracle's, except for blocks whose fp64
score lies within 1e-4 relative of the oracle's k-th score; a swap outside that
band is still accepted (and counted separately) when the two scores differ by less
than the fp32 dot-product error bound, because fp32 accumulation cannot order them.
Attention (graded on the GPU's own selection): max |out - ref| <= 2e-2 and mean
|out - ref| <= 2e-3.
"""

import numpy as np
import torch

import oracle as O

SEL_BAND = 1e-4
ATT_MAX_ABS = 2e-2
ATT_MEAN_ABS = 2e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit array (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def check_selection(gpu_blocks, gpu_count, q_idx_bits, pooled_bits, nb, k=O.BLOCK_TOPK):
    """Compare one row's GPU selection with the oracle's. Returns counts of
    (exempt swaps within the band, swaps within the fp32 bound)."""
    scores = O.score_blocks(q_idx_bits, pooled_bits[:nb])
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
    bound = O.score_error_bound(q_idx_bits, pooled_bits[:nb])
    kth_bound = bound[O._rank_order(scores)[kk - 1]]
    gap = np.abs(scores[diff] - kth)
    in_band = gap <= SEL_BAND * abs(kth)
    in_fp32 = ~in_band & (gap <= bound[diff] + kth_bound)
    assert np.all(in_band | in_fp32), (diff[~(in_band | in_fp32)], gap[~(in_band | in_fp32)], kth)
    return int(in_band.sum()), int(in_fp32.sum())


def check_attention(gpu_out, ref_out, max_abs=ATT_MAX_ABS, mean_abs=ATT_MEAN_ABS):
    """gpu_out: bf16 tensor or float array; ref_out: float64 array of the same shape."""
    g = gpu_out.float().cpu().numpy().astype(np.float64) if isinstance(gpu_out, torch.Tensor) else gpu_out
    err = np.abs(g - ref_out)
    assert np.all(np.isfinite(g))
    assert err.max() <= max_abs, err.max()
    assert err.mean() <= mean_abs, err.mean()
    return float(err.max()), float(err.mean()), float(np.linalg.norm(g - ref_out) / max(np.linalg.norm(ref_out), 1e-300))
