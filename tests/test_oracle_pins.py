"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test ties an oracle function to something other than itself: a value
printed on the pages (tests/golden), a library routine that computes the same
special case (torch SDPA, max_pool1d, topk, amax), a mathematical invariant
(the Kmax/Kmin bound), or an independent pure-Python brute force.  The
mutation tests at the end plant a plausible mistake in the oracle and check
that a pin catches it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import brute_ref
import oracle
from oracle import rocketkv_oracle as ro

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# Budget split: worked example and clamp printed on the pages
# ---------------------------------------------------------------------------


def test_split_worked_example():
    g = _gold("split_worked_example.json")
    c = g["c"]
    r = oracle.split_factor(c)
    assert round(r, 2) == g["r"]
    s1, s2 = oracle.stage_factors(c, r)
    assert round(s1, 1) == g["stage1_factor"]
    assert round(s2, 1) == g["stage2_factor"]
    page, head = oracle.hsa_internal_split(c, r)
    assert page == g["page_size"]
    assert round(head, 1) == g["head_factor"]
    # the two stages multiply back to the total
    assert math.isclose(s1 * s2, c, rel_tol=1e-12)
    assert math.isclose(page * head, s2, rel_tol=1e-12)


def test_split_clamp():
    for case in _gold("split_clamp.json")["cases"]:
        assert math.isclose(oracle.split_factor(case["c"]), case["r"], abs_tol=1e-12)
    # monotone between the clamps
    cs = [2.0 ** e for e in np.linspace(0, 14, 57)]
    rs = [oracle.split_factor(c) for c in cs]
    assert all(b >= a for a, b in zip(rs, rs[1:]))


def test_budget_split_counts():
    # B1 is the stage-1 keep count: S / c**r tokens, c = S/t.
    r, B1, k2 = oracle.budget_split(32768, 1024, 16)
    assert r == 0.5 and B1 == math.floor(32768 / math.sqrt(32)) and k2 == 32
    # t/2 tokens for step 3: k2 * blk never exceeds t/2
    for S, t, blk in [(4096, 256, 16), (109000, 256, 16), (32768, 2048, 32), (5000, 100, 7)]:
        r, B1, k2 = oracle.budget_split(S, t, blk)
        assert k2 * blk <= max(t // 2, blk)
        assert 33 <= B1 <= S
    # budget above the prompt: nothing evicted
    assert oracle.budget_split(100, 1000, 16)[1] == 100


def test_kv_cache_size():
    for case in _gold("kv_cache_size.json")["cases"]:
        b = oracle.kv_cache_bytes(case["layers"], case["kv_heads"], case["head_dim"], case["seq"],
                                  case["bytes"], case["batch"])
        v = b / case["unit_divisor"]
        p = case["printed"] / (case["unit_divisor"] if case["printed"] > 1e5 else 1)
        if case["compare"] == "floor":
            assert math.floor(v) == round(p)
        else:
            assert round(v, case["printed_digits"]) == round(p, case["printed_digits"])


def test_table1_rows_and_derivation():
    g = _gold("table1_storage.json")
    for row in g["rows_at_c"]:
        st, tr = oracle.table1_storage_traffic(row["c"], oracle.split_factor(row["c"]))[row["method"]]
        assert math.isclose(st, row["storage"]) and math.isclose(tr, row["traffic"])
    # text beside Table 1: after stage 1 the relative storage is 1/c**r, and Kmax
    # and Kmin each add 1/c**((1-r)/2) of that; traffic is 1/c for all methods.
    for c in [4.0, 16.0, 64.0, 425.78]:
        r = oracle.split_factor(c)
        rk, rkt = oracle.table1_storage_traffic(c, r)["RocketKV"]
        mt, mtt = oracle.table1_storage_traffic(c, r)["RocketKV-MT"]
        assert math.isclose(rk, (1 / c ** r) * (1 + 2 / c ** ((1 - r) / 2)))
        assert math.isclose(mt - rk, 1 - 1 / c ** r)
        assert rkt == mtt == 1 / c


# ---------------------------------------------------------------------------
# Top-k ordering (reading R5)
# ---------------------------------------------------------------------------


def test_topk_ties_lowest_index():
    v = np.array([3.0, 1.0, 3.0, 2.0, 3.0])
    assert oracle.topk_lowest_index(v, 2).tolist() == [0, 2]
    assert oracle.topk_lowest_index(v, 4).tolist() == [0, 2, 3, 4]
    assert oracle.topk_lowest_index(v, 9).tolist() == [0, 1, 2, 3, 4]
    assert oracle.topk_lowest_index(np.array([-0.0, 0.0, -1.0]), 1).tolist() == [0]


def test_topk_matches_library_on_distinct_values():
    x = _rng(1).standard_normal(1000)
    for k in [1, 7, 100, 999]:
        ref = torch.topk(torch.from_numpy(x), k).indices.sort().values.numpy()
        assert oracle.topk_lowest_index(x, k).tolist() == ref.tolist()


# ---------------------------------------------------------------------------
# Stage 1 against library routines
# ---------------------------------------------------------------------------


def _sdpa_probs(Q, K, pos):
    """Attention probabilities from torch SDPA: with V = identity the output is P."""
    S = K.shape[0]
    mask = torch.arange(S)[None, :] <= torch.as_tensor(pos)[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None, None], torch.from_numpy(K)[None, None],
        torch.eye(S, dtype=torch.float64)[None, None], attn_mask=mask[None, None])
    return out[0, 0].numpy()


def test_snap_scores_vs_sdpa():
    G, W, D, S = 3, 5, 8, 40
    r = _rng(2)
    q = r.standard_normal((G, W, D))
    K = r.standard_normal((S, D))
    scale = 1 / math.sqrt(D)
    pos = np.tile(np.arange(S - W, S), G)
    P = _sdpa_probs(q.reshape(G * W, D), K, pos)
    ref = P[:, : S - W].sum(axis=0)
    np.testing.assert_allclose(oracle.snap_scores(q, K, scale), ref, rtol=1e-12, atol=1e-15)


def test_max_pool_vs_library():
    x = _rng(3).standard_normal(300)
    for P in [1, 3, 7, 63, 301]:
        ref = torch.nn.functional.max_pool1d(torch.from_numpy(x)[None, None], P, stride=1,
                                             padding=P // 2)[0, 0].numpy()
        assert np.array_equal(oracle.max_pool(x, P), ref)
        assert np.array_equal(oracle.max_pool_fast(x, P), ref)


def test_stage1_degenerate_plain_topk():
    # G = 1, W = 1, pool kernel 1: the single softmax row is monotone in q.k,
    # so the kept prefix is the top-(B1-1) of q.k.
    D, S, B1 = 8, 200, 41
    r = _rng(4)
    q = r.standard_normal((1, 1, D))
    K = r.standard_normal((S, D))
    keep, _ = oracle.snap_keep(q, K, B1, 1, 1, 1 / math.sqrt(D))
    qk = K[: S - 1] @ q[0, 0]
    ref = np.sort(torch.topk(torch.from_numpy(qk), B1 - 1).indices.numpy())
    assert keep.tolist() == ref.tolist() + [S - 1]


def test_stage1_keep_all_cases():
    r = _rng(5)
    q = r.standard_normal((2, 4, 8))
    K = r.standard_normal((30, 8))
    assert oracle.snap_keep(q, K, 30, 4, 7, 0.3)[0].tolist() == list(range(30))
    assert oracle.snap_keep(q, K[:3], 3, 4, 7, 0.3)[0].tolist() == [0, 1, 2]


def test_stage1_window_and_sinks_kept():
    r = _rng(6)
    G, W, D, S = 2, 4, 8, 64
    q = r.standard_normal((G, W, D))
    K = r.standard_normal((S, D))
    keep, _ = oracle.snap_keep(q, K, 20, W, 7, 0.35, n_sink=3)
    assert keep[:3].tolist() == [0, 1, 2]
    assert keep[-W:].tolist() == list(range(S - W, S))
    assert len(keep) == 20 and np.all(np.diff(keep) > 0)


# ---------------------------------------------------------------------------
# KT cache against library reductions
# ---------------------------------------------------------------------------


def test_kt_vs_amax_amin():
    r = _rng(7)
    for n, blk in [(64, 16), (70, 16), (1, 16), (33, 32), (5, 1)]:
        K = r.standard_normal((n + 9, 8))
        kmax, kmin = oracle.build_kt(K, n, blk)
        nblk = -(-n // blk)
        pad = np.full((nblk * blk, 8), np.nan)
        pad[:n] = K[:n]
        t = torch.from_numpy(pad).reshape(nblk, blk, 8)
        ref_max = torch.nan_to_num(t, nan=-np.inf).amax(dim=1).T.numpy()
        ref_min = torch.nan_to_num(t, nan=np.inf).amin(dim=1).T.numpy()
        assert np.array_equal(kmax, ref_max) and np.array_equal(kmin, ref_min)


def test_kt_append_equals_rebuild():
    r = _rng(8)
    blk, D = 16, 8
    K = r.standard_normal((100, D))
    n0 = 37
    kmax, kmin = oracle.build_kt(K, n0, blk)
    for n in range(n0, 100):
        kmax, kmin = oracle.kt_append(kmax, kmin, n, K[n], blk)
        rmax, rmin = oracle.build_kt(K, n + 1, blk)
        assert np.array_equal(kmax[:, : rmax.shape[1]], rmax) and np.array_equal(kmin[:, : rmin.shape[1]], rmin)


# ---------------------------------------------------------------------------
# HSA special cases (Algorithm 1)
# ---------------------------------------------------------------------------


def _sdpa(qg, K, V, scale, tokens=None):
    n = K.shape[0]
    mask = torch.zeros(qg.shape[0], n, dtype=torch.bool)
    mask[:, tokens if tokens is not None else slice(None)] = True
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qg)[None, None], torch.from_numpy(K)[None, None], torch.from_numpy(V)[None, None],
        attn_mask=mask[None, None], scale=scale)[0, 0].numpy()


def test_exact_topk_special_case():
    # k1 = D and blk = 1: every block is one key and Kmax = Kmin = k, so the
    # block score is exactly qbar . k and HSA is Exact-TopK attention.
    r = _rng(9)
    G, D, n, k2 = 4, 16, 300, 20
    qg = r.standard_normal((G, D))
    K = r.standard_normal((n, D))
    V = r.standard_normal((n, D))
    kmax, kmin = oracle.build_kt(K, n, 1)
    res = oracle.hsa_decode(qg, K, V, n, kmax, kmin, 1, D, k2, 0.25)
    qk = K @ qg.sum(axis=0)
    ref_sel = np.sort(torch.topk(torch.from_numpy(qk), k2).indices.numpy())
    assert res["i2"].tolist() == ref_sel.tolist()
    np.testing.assert_allclose(res["y"], _sdpa(qg, K, V, 0.25, ref_sel), rtol=1e-12, atol=1e-12)


def test_full_attention_special_case():
    r = _rng(10)
    G, D, n, blk = 4, 16, 203, 16
    qg = r.standard_normal((G, D))
    K = r.standard_normal((n, D))
    V = r.standard_normal((n, D))
    kmax, kmin = oracle.build_kt(K, n, blk)
    res = oracle.hsa_decode(qg, K, V, n, kmax, kmin, blk, 5, 1000, 0.3)
    assert res["i2"].tolist() == list(range(-(-n // blk)))
    np.testing.assert_allclose(res["y"], _sdpa(qg, K, V, 0.3), rtol=1e-12, atol=1e-12)


def check_bound(qg, K, n, blk, k1, res):
    """Block score >= (kept-channel part of) qbar . k for every key in the block."""
    qbar = qg.sum(axis=0)
    i1 = res["i1"]
    for b in range(res["s"].shape[0]):
        rows = K[b * blk: min(n, (b + 1) * blk)]
        part = rows[:, i1] @ qbar[i1]
        if not np.all(res["s"][b] >= part - 1e-9 * (1 + np.abs(part))):
            return False
    return True


def test_bound_invariant():
    r = _rng(11)
    for G, D, n, blk, k1 in [(4, 16, 100, 16, 4), (1, 8, 37, 5, 8), (8, 32, 64, 32, 31)]:
        qg = r.standard_normal((G, D))
        K = r.standard_normal((n, D))
        kmax, kmin = oracle.build_kt(K, n, blk)
        res = oracle.hsa_decode(qg, K, K, n, kmax, kmin, blk, k1, 3, 0.2)
        assert check_bound(qg, K, n, blk, k1, res)
        if k1 == D:   # all channels: the bound covers the full dot product
            full = (K[:n] @ qg.sum(axis=0))
            per_blk = np.array([full[b * blk:(b + 1) * blk].max() for b in range(res["s"].shape[0])])
            assert np.all(res["s"] >= per_blk - 1e-9)


def test_permutation_invariance_within_group():
    r = _rng(12)
    G, D, n, blk = 4, 16, 90, 8
    qg = r.standard_normal((G, D))
    K = r.standard_normal((n, D))
    V = r.standard_normal((n, D))
    kmax, kmin = oracle.build_kt(K, n, blk)
    a = oracle.hsa_decode(qg, K, V, n, kmax, kmin, blk, 6, 3, 0.3)
    perm = [2, 0, 3, 1]
    b = oracle.hsa_decode(qg[perm], K, V, n, kmax, kmin, blk, 6, 3, 0.3)
    assert a["i1"].tolist() == b["i1"].tolist() and a["i2"].tolist() == b["i2"].tolist()
    np.testing.assert_allclose(a["y"][perm], b["y"], rtol=1e-12)


def test_sign_at_zero_takes_kmax():
    D = 4
    qg = np.array([[1.0, 2.0, -3.0, 1.0], [-1.0, 1.0, 1.0, 1.0]])    # qbar = [0, 3, -2, 2]
    K = np.array([[5.0, 0.0, 1.0, 0.0], [-5.0, 0.0, -1.0, 0.0]])
    kmax, kmin = oracle.build_kt(K, 2, 2)
    i1, qbar = oracle.hsa_channels(qg, 4)
    s = oracle.hsa_block_scores(qbar, i1, kmax, kmin)
    # channel 0 contributes qbar_0 * Kmax = 0 either way; channel 2 (qbar<0) uses Kmin = -1
    assert s.tolist() == [0.0 * 5 + 3 * 0 + (-2) * (-1) + 2 * 0]


def test_block_score_is_box_maximum_by_corners():
    # The score of a block is the largest value of sum_{c in i1} qbar_c x_c over
    # the box Kmin <= x <= Kmax.  A linear form over a box peaks at a corner, so
    # enumerating all 2^k1 corners gives the score with no per-channel argument.
    r = _rng(13)
    for G, D, n, blk, k1 in [(4, 12, 70, 8, 6), (2, 8, 33, 4, 8), (3, 10, 20, 20, 5)]:
        qg = r.standard_normal((G, D))
        qg[:, 0] = 0.0                                          # one zero group sum
        K = r.standard_normal((n, D))
        kmax, kmin = oracle.build_kt(K, n, blk)
        i1, qbar = oracle.hsa_channels(qg, k1)
        s = oracle.hsa_block_scores(qbar, i1, kmax, kmin)
        for b in range(s.shape[0]):
            best = -np.inf
            for corner in range(1 << k1):
                x = [kmax[c, b] if (corner >> u) & 1 else kmin[c, b] for u, c in enumerate(i1)]
                best = max(best, float(np.dot(qbar[i1], x)))
            assert abs(s[b] - best) <= 1e-12 * (1 + abs(best))


# ---------------------------------------------------------------------------
# Multi-turn identity
# ---------------------------------------------------------------------------


def test_mt_identity():
    r = _rng(13)
    G, D, full, blk = 4, 16, 400, 16
    Kf = r.standard_normal((full, D))
    Vf = r.standard_normal((full, D))
    idx = np.sort(r.choice(full, 150, replace=False))
    qg = r.standard_normal((G, D))
    n = idx.size
    kmax, kmin = oracle.build_kt_mt(Kf, idx, n, blk)
    a = oracle.hsa_decode_mt(qg, Kf, Vf, idx, n, kmax, kmin, blk, 8, 4, 0.25)
    kc, vc = Kf[idx], Vf[idx]
    k2max, k2min = oracle.build_kt(kc, n, blk)
    b = oracle.hsa_decode(qg, kc, vc, n, k2max, k2min, blk, 8, 4, 0.25)
    assert np.array_equal(kmax, k2max)
    assert a["i2"].tolist() == b["i2"].tolist()
    assert np.array_equal(a["y"], b["y"])


# ---------------------------------------------------------------------------
# Multi-turn over the blocks of the full cache (the other reading)
# ---------------------------------------------------------------------------


def _masked_case(seed, n, n_prompt, blk, D=8, G=2, dens=0.3):
    r = _rng(seed)
    K = r.standard_normal((n, D))
    V = r.standard_normal((n, D))
    qg = r.standard_normal((G, D))
    keep = np.sort(r.choice(n_prompt, max(1, int(dens * n_prompt)), replace=False))
    cand = oracle.candidate_rows(keep, n_prompt, n)
    return qg, K, V, keep, cand


@pytest.mark.parametrize("seed,n,n_prompt,blk,k1,k2", [
    (40, 37, 30, 4, 3, 2), (41, 50, 50, 5, 8, 3), (42, 23, 17, 1, 8, 4),
    (43, 64, 40, 8, 2, 30), (44, 45, 44, 3, 5, 1),
])
def test_mt_masked_vs_brute_force(seed, n, n_prompt, blk, k1, k2):
    qg, K, V, keep, cand = _masked_case(seed, n, n_prompt, blk)
    kmax, kmin, has = oracle.build_kt_masked(K, n, cand, blk)
    res = oracle.hsa_decode_mt_masked(qg, K, V, n, cand, kmax, kmin, has, blk, k1, k2, 0.3)
    y, i1, i2 = brute_ref.hsa_masked(qg.tolist(), K.tolist(), V.tolist(), n, cand.tolist(), blk, k1, k2, 0.3)
    assert res["i1"].tolist() == i1
    assert res["i2"].tolist() == i2
    np.testing.assert_allclose(res["y"], np.array(y), rtol=1e-12, atol=1e-12)


def test_mt_masked_candidates():
    # kept prompt rows plus every row decoded after the prompt
    cand = oracle.candidate_rows(np.array([0, 3, 7, 9]), 8, 12)
    assert np.flatnonzero(cand).tolist() == [0, 3, 7, 8, 9, 10, 11]


def test_mt_masked_full_attention_when_k2_covers():
    qg, K, V, keep, cand = _masked_case(45, 90, 70, 8, D=16, G=4)
    kmax, kmin, has = oracle.build_kt_masked(K, 90, cand, 8)
    res = oracle.hsa_decode_mt_masked(qg, K, V, 90, cand, kmax, kmin, has, 8, 4, 1000, 0.25)
    np.testing.assert_allclose(res["y"], _sdpa(qg, K, V, 0.25, np.flatnonzero(cand)), rtol=1e-12, atol=1e-12)


def test_mt_masked_bounds_skip_other_rows():
    qg, K, V, keep, cand = _masked_case(46, 80, 64, 8)
    K[~cand] = 1e3 * np.sign(_rng(47).standard_normal(K[~cand].shape))   # never a bound
    kmax, kmin, has = oracle.build_kt_masked(K, 80, cand, 8)
    ref_max = torch.from_numpy(np.where(cand[:, None], K, -np.inf)).reshape(10, 8, -1).amax(dim=1).numpy().T
    ref_min = torch.from_numpy(np.where(cand[:, None], K, np.inf)).reshape(10, 8, -1).amin(dim=1).numpy().T
    ref_has = cand.reshape(10, 8).any(axis=1)
    assert has.tolist() == ref_has.tolist()
    assert np.array_equal(kmax[:, has], ref_max[:, has]) and np.array_equal(kmin[:, has], ref_min[:, has])
    assert np.all(np.abs(kmax[:, has]) < 1e3)


def test_mt_masked_tail_always_chosen():
    qg, K, V, keep, cand = _masked_case(48, 100, 90, 8, D=16, G=4)
    K[96:] = -5.0 * qg.sum(axis=0)          # the newest block scores lowest of all
    kmax, kmin, has = oracle.build_kt_masked(K, 100, cand, 8)
    res = oracle.hsa_decode_mt_masked(qg, K, V, 100, cand, kmax, kmin, has, 8, 16, 2, 0.25)
    assert 12 in res["i2"].tolist()
    finite = res["s"][np.isfinite(res["s"])]
    assert res["s"][12] == np.inf and len(finite) == has.sum() - 1


def test_mt_masked_other_rows_do_not_matter():
    qg, K, V, keep, cand = _masked_case(49, 70, 60, 4)
    kmax, kmin, has = oracle.build_kt_masked(K, 70, cand, 4)
    a = oracle.hsa_decode_mt_masked(qg, K, V, 70, cand, kmax, kmin, has, 4, 4, 5, 0.3)
    r = _rng(50)
    K2, V2 = K.copy(), V.copy()
    K2[~cand] = r.standard_normal(K2[~cand].shape) * 10
    V2[~cand] = r.standard_normal(V2[~cand].shape) * 10
    kmax2, kmin2, has2 = oracle.build_kt_masked(K2, 70, cand, 4)
    b = oracle.hsa_decode_mt_masked(qg, K2, V2, 70, cand, kmax2, kmin2, has2, 4, 4, 5, 0.3)
    assert a["i2"].tolist() == b["i2"].tolist()
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-12, atol=1e-12)


def test_mt_masked_matches_candidate_reading_on_whole_blocks():
    # Candidate sets made of whole blocks, decoded rows from a block boundary,
    # and a newest block that is chosen anyway: both multi-turn readings form
    # the same blocks, pick the same ones and attend the same rows.
    r = _rng(51)
    G, D, blk, n_prompt, n = 4, 16, 8, 160, 180
    K = r.standard_normal((n, D))
    V = r.standard_normal((n, D))
    qg = r.standard_normal((G, D))
    K[176:] = 3.0 * np.sign(qg.sum(axis=0))
    kept_blocks = np.sort(r.choice(n_prompt // blk, 7, replace=False))
    keep = (kept_blocks[:, None] * blk + np.arange(blk)).reshape(-1)
    cand = oracle.candidate_rows(keep, n_prompt, n)
    kmax, kmin, has = oracle.build_kt_masked(K, n, cand, blk)
    a = oracle.hsa_decode_mt_masked(qg, K, V, n, cand, kmax, kmin, has, blk, 6, 4, 0.25)
    idx = np.flatnonzero(cand)
    km10, kn10 = oracle.build_kt_mt(K, idx, idx.size, blk)
    b = oracle.hsa_decode_mt(qg, K, V, idx, idx.size, km10, kn10, blk, 6, 4, 0.25)
    phys = np.flatnonzero(has)                   # compacted block i <-> physical block phys[i]
    assert phys[b["i2"]].tolist() == a["i2"].tolist()
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-12, atol=1e-12)


def test_kt_append_masked_equals_rebuild():
    qg, K, V, keep, cand = _masked_case(52, 75, 61, 6)
    kmax, kmin, has = oracle.build_kt_masked(K, 61, cand, 6)
    for n in range(61, 75):
        kmax, kmin, has = oracle.kt_append_masked(kmax, kmin, has, n, K[n], 6)
    rmax, rmin, rhas = oracle.build_kt_masked(K, 75, cand, 6)
    assert has.tolist() == rhas.tolist()
    assert np.array_equal(kmax, rmax) and np.array_equal(kmin, rmin)


# ---------------------------------------------------------------------------
# FP8 (e4m3) storage
# ---------------------------------------------------------------------------


def _torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_closed_forms_and_library():
    c = np.arange(256, dtype=np.uint8)
    d = oracle.e4m3_decode(c)
    assert d[0x38] == 1.0 and d[0xB8] == -1.0 and d[0x7E] == 448.0 and d[0x01] == 2.0 ** -9
    assert d[0x08] == 2.0 ** -6 and d[0x07] == 7 * 2.0 ** -9 and d[0x3C] == 1.5
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF]) and np.isfinite(np.delete(d, [0x7F, 0xFF])).all()
    lib = torch.from_numpy(c).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.nan_to_num(d, nan=7e7), np.nan_to_num(lib.astype(np.float64), nan=7e7))


def test_e4m3_encode_vs_library_including_ties():
    pos = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (pos[1:] + pos[:-1]) / 2
    x = np.concatenate([_rng(60).uniform(-464, 464, 20000), mids, -mids, pos, -pos, [464.0, -464.0]])
    assert np.array_equal(oracle.e4m3_encode(x), _torch_e4m3(x))


def test_e4m3_saturation_nan_and_round_trip():
    assert oracle.e4m3_encode(np.array([1000.0, -1e9, np.nan, 449.0]).astype(np.float64)).tolist() == \
        [0x7E, 0xFE, 0x7F, 0x7E]
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(finite)), finite)


def test_fp8_quantize_vs_library():
    X = _rng(61).standard_normal((64, 16)) * 8
    for sc in (1.0, 0.0625, 0.37):
        ref = _torch_e4m3(torch.from_numpy(X.astype(np.float32)).div(np.float32(sc)).numpy())
        assert np.array_equal(oracle.fp8_quantize(X, sc), ref)


def test_hsa_fp8_full_attention_and_dequantized_identity():
    r = _rng(62)
    G, D, n, blk = 4, 16, 150, 16
    qg = r.standard_normal((G, D))
    Kc = oracle.fp8_quantize(r.standard_normal((n, D)) * 3, 0.25)
    Vc = oracle.fp8_quantize(r.standard_normal((n, D)), 0.125)
    kmax, kmin = oracle.build_kt_fp8(Kc, n, blk)
    Kd, Vd = oracle.e4m3_decode(Kc) * 0.25, oracle.e4m3_decode(Vc) * 0.125
    full = oracle.hsa_decode_fp8(qg, Kc, Vc, n, kmax, kmin, 0.25, 0.125, blk, 6, 1000, 0.3)
    np.testing.assert_allclose(full["y"], _sdpa(qg, Kd, Vd, 0.3), rtol=1e-12, atol=1e-12)
    # a power-of-two K scale scales every score exactly: the same choices as the
    # bf16 path on the dequantized cache
    a = oracle.hsa_decode_fp8(qg, Kc, Vc, n, kmax, kmin, 0.25, 0.125, blk, 6, 3, 0.3)
    dmax, dmin = oracle.build_kt(Kd, n, blk)
    b = oracle.hsa_decode(qg, Kd, Vd, n, dmax, dmin, blk, 6, 3, 0.3)
    assert a["i1"].tolist() == b["i1"].tolist() and a["i2"].tolist() == b["i2"].tolist()
    np.testing.assert_allclose(a["s"] * 0.25, b["s"], rtol=1e-12)
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Brute force of the whole pipeline on tiny inputs
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("seed,G,W,D,S,B1,P,blk,k1,k2,sink", [
    (20, 2, 4, 8, 48, 20, 7, 4, 3, 2, 0),
    (21, 1, 3, 4, 40, 12, 5, 3, 2, 3, 2),
    (22, 3, 2, 8, 64, 30, 63, 5, 8, 4, 0),
])
def test_pipeline_vs_brute_force(seed, G, W, D, S, B1, P, blk, k1, k2, sink):
    r = _rng(seed)
    q_obs = r.standard_normal((G, W, D))
    K = r.standard_normal((S, D))
    V = r.standard_normal((S, D))
    T = 3
    qs = r.standard_normal((T, G, D))
    kn = r.standard_normal((T, D))
    vn = r.standard_normal((T, D))
    scale = 1 / math.sqrt(D)
    keep, pooled, steps = oracle.pipeline_group(q_obs, K, V, qs, kn, vn, B1, W, P, blk, k1, k2, scale, sink)

    bkeep, bpooled = brute_ref.snap_keep(q_obs.tolist(), K.tolist(), B1, W, P, scale, sink)
    assert keep.tolist() == bkeep
    np.testing.assert_allclose(pooled, bpooled, rtol=1e-12)
    Kc = [K[i].tolist() for i in bkeep]
    Vc = [V[i].tolist() for i in bkeep]
    for t in range(T):
        Kc.append(kn[t].tolist())
        Vc.append(vn[t].tolist())
        n = len(Kc)
        kmax, kmin = brute_ref.kt(Kc, n, blk)
        y, i1, i2, s = brute_ref.hsa(qs[t].tolist(), Kc, Vc, n, kmax, kmin, blk, k1, k2, scale)
        assert steps[t]["i1"].tolist() == i1
        assert steps[t]["i2"].tolist() == i2
        np.testing.assert_allclose(steps[t]["s"], s, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(steps[t]["y"], y, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# Mutation tests: a planted mistake in the oracle must fail a pin
# ---------------------------------------------------------------------------


def test_mutation_sign_flip_fails_bound(monkeypatch):
    def wrong(qbar, i1, kmax, kmin):
        g = qbar[i1]
        return g @ np.where((g < 0)[:, None], kmax[i1, :], kmin[i1, :])
    monkeypatch.setattr(ro, "hsa_block_scores", wrong)
    r = _rng(30)
    qg = r.standard_normal((4, 16))
    K = r.standard_normal((64, 16))
    kmax, kmin = ro.build_kt(K, 64, 16)
    res = ro.hsa_decode(qg, K, K, 64, kmax, kmin, 16, 16, 2, 0.2)
    assert not check_bound(qg, K, 64, 16, 16, res)


def test_mutation_window_denominator_fails_sdpa(monkeypatch):
    # dropping the window keys from the softmax denominator must be caught
    def wrong(q_obs_group, K, scale):
        G, W, D = q_obs_group.shape
        S = K.shape[0]
        lg = (q_obs_group.reshape(G * W, D) @ K[: S - W].T) * scale
        p = np.exp(lg - lg.max(axis=1, keepdims=True))
        return (p / p.sum(axis=1, keepdims=True)).sum(axis=0)
    r = _rng(31)
    q = r.standard_normal((2, 4, 8))
    K = r.standard_normal((30, 8))
    pos = np.tile(np.arange(26, 30), 2)
    ref = _sdpa_probs(q.reshape(8, 8), K, pos)[:, :26].sum(axis=0)
    assert not np.allclose(wrong(q, K, 1 / math.sqrt(8)), ref, rtol=1e-6)


def test_mutation_unforced_tail_fails_brute_force(monkeypatch):
    # forgetting to force the newest block in must be caught by the brute force
    def wrong(q_group, Kfull, Vfull, n, cand, kmax, kmin, has, blk, k1, k2, scale):
        nblk = (n + blk - 1) // blk
        i1, qbar = ro.hsa_channels(q_group, k1)
        s = np.where(has[:nblk], ro.hsa_block_scores(qbar, i1, kmax[:, :nblk], kmin[:, :nblk]), -np.inf)
        return {"i1": i1, "i2": ro.topk_lowest_index(s, k2), "s": s}
    monkeypatch.setattr(ro, "hsa_decode_mt_masked", wrong)
    qg, K, V, keep, cand = _masked_case(53, 100, 90, 8, D=16, G=4)
    K[96:] = -5.0 * qg.sum(axis=0)
    kmax, kmin, has = ro.build_kt_masked(K, 100, cand, 8)
    res = ro.hsa_decode_mt_masked(qg, K, V, 100, cand, kmax, kmin, has, 8, 16, 2, 0.25)
    _, _, i2 = brute_ref.hsa_masked(qg.tolist(), K.tolist(), V.tolist(), 100, cand.tolist(), 8, 16, 2, 0.25)
    assert res["i2"].tolist() != i2


def test_mutation_round_half_away_fails_library():
    # rounding ties away from zero instead of to the even code must be caught
    pos = ro.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (pos[1:] + pos[:-1]) / 2
    hi = np.searchsorted(pos, mids)
    wrong = hi.astype(np.uint8)                     # every tie goes up
    assert not np.array_equal(wrong, _torch_e4m3(mids))
    assert np.array_equal(ro.e4m3_encode(mids), _torch_e4m3(mids))


def test_mutation_transposed_kt_fails_library():
    K = _rng(32).standard_normal((32, 8))
    kmax, _ = ro.build_kt(K, 32, 16)
    ref = torch.from_numpy(K).reshape(2, 16, 8).amax(dim=1).numpy()     # [nblk, D]
    assert not np.array_equal(kmax.reshape(2, 8), ref)   # wrong layout reading
    assert np.array_equal(kmax, ref.T)
