"""Comparison rules between the CUDA library and the CPU oracle.

- Index sets (stage-1 keep, channel set i1, block set i2) must be identical,
  except items whose oracle score lies within REL_TIE (relative) of the oracle's
  k-th score: those are exempt from the symmetric difference.  Channel sums are
  exact on both sides (fp64 in the oracle; fp32 with an error-free check, else
  fp64, in the kernel), so i1 is compared with no exemption.
- Stage-1 keep sets are compared with the same band only: the kernels rank
  log2 of each key's score, so scores far below the fp32 range still rank as
  in the oracle.
- Attention outputs: max-abs difference <= ATOL_OUT against the oracle's output
  for the same selected blocks (bf16 inputs, fp32 accumulation on the GPU).
"""
import numpy as np

from two_stage_kv_gb300.synth import bf16_bits_to_f64

REL_TIE = 1e-4
ATOL_OUT = 2e-3


def t2bits(t):
    """bf16 torch tensor (any device) -> numpy uint16 bits."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def t2f64(t):
    return bf16_bits_to_f64(t2bits(t))


def check_topk(gpu_idx, scores, k, what="", rel=REL_TIE):
    """Returns the number of tie-exempt differences; asserts everything else."""
    from oracle import kth_value, topk_lowest_index
    gpu_idx = np.asarray(gpu_idx, dtype=np.int64)
    scores = np.asarray(scores, dtype=np.float64)
    k = min(k, scores.shape[0])
    assert gpu_idx.shape[0] == k, f"{what}: {gpu_idx.shape[0]} indices, expected {k}"
    if k == 0:
        return 0
    assert np.all(np.diff(gpu_idx) > 0), f"{what}: indices not strictly ascending"
    assert gpu_idx.min() >= 0 and gpu_idx.max() < scores.shape[0], f"{what}: index out of range"
    ref = topk_lowest_index(scores, k)
    if np.array_equal(gpu_idx, ref):
        return 0
    kth = kth_value(scores, k)
    diff = np.setxor1d(gpu_idx, ref)
    exempt = np.abs(scores[diff] - kth) <= rel * abs(kth)
    assert np.all(exempt), (f"{what}: non-exempt differences at {diff[~exempt][:10]} "
                            f"(scores {scores[diff[~exempt][:10]]}, k-th {kth})")
    return int(diff.size)


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))
