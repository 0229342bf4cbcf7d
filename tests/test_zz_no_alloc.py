"""GPU test of rkv_snap_evict_noalloc, the stage-1 entry point for callers that
cannot allocate device memory (an engine whose pool owns all device memory, a
plugin hook that must not call cudaMalloc).  It must give the same keep set, compacted caches and pooled scores
as rkv_snap_evict with a caller-allocated workspace, on consecutive calls that
reuse the library's fixed scratch, and reject shapes whose scratch would not
fit.  Collected last so a failure here comes after every other test ran.
"""
import math

import numpy as np
import pytest
import torch

from two_stage_kv_gb300 import rkv
from two_stage_kv_gb300.synth import small_random

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bf16(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)


def _case(seed, B, Hq, Hkv, S, W, P, B1):
    D = 128
    cap = S + 3
    k = _bf16(small_random(seed, (B, Hkv, cap, D)))
    v = _bf16(small_random(seed + 1, (B, Hkv, cap, D)))
    q = _bf16(small_random(seed + 2, (B, Hq, W, D)))
    return (B, Hq, Hkv, D), q, k, v, cap


def _run(noalloc, dims, q, k, v, cap, S, W, P, B1):
    B, Hq, Hkv, D = dims
    keep = torch.full((B, Hkv, B1), -1, dtype=torch.int32, device=DEV)
    ko = torch.zeros((B, Hkv, B1, D), dtype=torch.bfloat16, device=DEV)
    vo = torch.zeros_like(ko)
    pooled = torch.zeros((B, Hkv, S - W), dtype=torch.float32, device=DEV)
    scale = 1 / math.sqrt(D)
    if noalloc:
        rkv.rkv_snap_evict_noalloc(dims, q, W, k, v, cap, S, P, 0, B1, scale, keep, B1, ko, vo, B1, pooled)
    else:
        nbytes = rkv.rkv_snap_evict_workspace(dims, S, W)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        rkv.rkv_snap_evict(dims, q, W, k, v, cap, S, P, 0, B1, scale, keep, B1, ko, vo, B1, pooled, ws, nbytes)
    torch.cuda.synchronize()
    return keep, ko, vo, pooled


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [(71, 2, 32, 8, 6000, 32, 63, 900), (72, 1, 64, 8, 9001, 32, 63, 1300)]
    for seed, B, Hq, Hkv, S, W, P, B1 in cases:       # two calls in a row share the scratch
        dims, q, k, v, cap = _case(seed, B, Hq, Hkv, S, W, P, B1)
        ref = _run(False, dims, q, k, v, cap, S, W, P, B1)
        got = _run(True, dims, q, k, v, cap, S, W, P, B1)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
        assert (got[0] >= 0).all()


def test_noalloc_rejects_oversized_scratch():
    # 16 rows of a 32K prompt need about 34 MiB of scratch.  Every tensor is a
    # real allocation of the full shape, so the call would stay in bounds even
    # if the size check did not come first.
    B, Hq, Hkv, D, S, W, B1 = 16, 32, 8, 128, 32768, 32, 4000
    dims = (B, Hq, Hkv, D)
    assert rkv.rkv_snap_evict_workspace(dims, S, W) > 32 << 20
    q = torch.zeros((B, Hq, W, D), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((B, Hkv, S, D), dtype=torch.bfloat16, device=DEV)
    v = torch.zeros_like(k)
    keep = torch.zeros((B, Hkv, B1), dtype=torch.int32, device=DEV)
    ko = torch.zeros((B, Hkv, B1, D), dtype=torch.bfloat16, device=DEV)
    vo = torch.zeros_like(ko)
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_snap_evict_noalloc(dims, q, W, k, v, S, S, 63, 0, B1, 0.1, keep, B1, ko, vo, B1, None)
    assert e.value.status == 3 and "fixed scratch" in str(e.value)
    torch.cuda.synchronize()
