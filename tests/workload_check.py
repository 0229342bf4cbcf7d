"""Oracle check of one (batch row, KV head) pair of a single-turn workload run.

The GPU run records, for every pair, its stage-1 keep list and pooled scores,
its KT cache after compaction and after the last step, and at every decode
step its channel set, block set and fp32 outputs.  `check_pair` regenerates
that pair's seeded inputs (the same generator the GPU run used) and checks
each stage against the CPU oracle, on the GPU's own upstream results so that
one tie-exempt difference does not cascade:

  stage 1   pooled scores within 1e-4 (relative), keep set under the tie rule,
            the window rows kept;
  KT        bit-exact after compaction and after every append;
  decode    channel set exact, block set under the tie rule, outputs within
            2e-3 of the oracle's attention over the same blocks.

It needs no GPU and imports no torch, so full-size runs can spread the pairs
over host processes (`check_pairs`, a spawn pool: nothing is forked from a
process that holds a CUDA context).
"""
from __future__ import annotations

import math
import multiprocessing as mp
import os

import numpy as np

import oracle
from parity_util import ATOL_OUT, check_topk, max_abs
from two_stage_kv_gb300 import synth
from two_stage_kv_gb300.synth import bf16_bits_to_f64 as f64


def _needle_hits(wl, needles, keep, sel_at_step):
    """Per needle: 1 when its token survives stage 1 (keep) and its block is among
    the blocks chosen at the step whose query looks for it."""
    hits = []
    for i, p in enumerate(needles):
        pos = np.searchsorted(keep, p)
        ok = pos < len(keep) and keep[pos] == p
        hits.append(int(ok and (pos // wl.blk) in set(np.asarray(sel_at_step(synth.needle_step(wl, i))).tolist())))
    return hits


def check_pair(task):
    """Checks one pair; returns {"worst", "exempt", "hits", "hits_oracle"}.
    Raises AssertionError (naming the pair and stage) on any violation."""
    wl, layer, b, h = task["wl"], task["layer"], task["b"], task["h"]
    G, D, blk, k1, k2, B1 = wl.G, wl.D, wl.blk, wl.k1, task["k2"], task["B1"]
    scale = 1 / math.sqrt(D)
    qd = synth.q_decode(wl, layer)
    kb, vb = synth.kv_slice(wl, layer, b, h, qd)
    qo = f64(synth.q_obs(wl, layer, qd)[b, h * G:(h + 1) * G])
    kn, vn = synth.kv_new(wl, layer)
    K, V = f64(kb), f64(vb)
    tag = f"layer {layer} pair ({b},{h})"

    # stage 1
    ref_keep, pooled = oracle.snap_keep(qo, K, B1, wl.W, wl.P, scale)
    pg = task["pooled"].astype(np.float64)
    rel = np.max(np.abs(pg - pooled) / np.maximum(np.abs(pooled), 1e-30))
    assert rel < 1e-4, f"{tag}: pooled scores differ by {rel} (relative)"
    got = task["keep"].astype(np.int64)
    assert got[-wl.W:].tolist() == list(range(wl.S - wl.W, wl.S)), f"{tag}: window rows not kept"
    exempt = check_topk(got[:B1 - wl.W], pooled, B1 - wl.W, f"{tag} keep")

    # KT after compaction, on the GPU's keep list
    n_all = B1 + wl.steps
    Kc = np.zeros((n_all, D))
    Vc = np.zeros((n_all, D))
    Kc[:B1], Vc[:B1] = K[got], V[got]
    kmax, kmin = oracle.build_kt(Kc[:B1], B1, blk)
    kt0 = f64(task["kt0"])
    assert np.array_equal(kt0[0, :, :kmax.shape[1]], kmax) and np.array_equal(kt0[1, :, :kmin.shape[1]], kmin), \
        f"{tag}: KT after compaction"

    # decode steps (each appends its token, then attends every candidate)
    worst = 0.0
    ref_sel = []
    n = B1
    for s in range(wl.steps):
        Kc[n], Vc[n] = f64(kn[s, b, h]), f64(vn[s, b, h])
        kmax, kmin = oracle.kt_append(kmax, kmin, n, Kc[n], blk)
        qg = f64(qd[s, b, h * G:(h + 1) * G])
        res = oracle.hsa_decode(qg, Kc, Vc, n + 1, kmax, kmin, blk, k1, k2, scale)
        ref_sel.append(res["i2"])
        assert task["sc"][s].tolist() == res["i1"].tolist(), f"{tag} step {s}: channel set"
        k2e = min(k2, res["s"].shape[0])
        sb = task["sb"][s, :k2e]
        exempt += check_topk(sb, res["s"], k2, f"{tag} step {s} blocks")
        y = res["y"] if np.array_equal(sb, res["i2"]) else \
            oracle.attention_over_blocks(qg, Kc, Vc, n + 1, sb, blk, scale)
        worst = max(worst, max_abs(task["out"][s], y))
        n += 1
    assert worst <= ATOL_OUT, f"{tag}: outputs differ by {worst}"
    ktf = f64(task["kt_final"])
    nb = kmax.shape[1]
    assert np.array_equal(ktf[0, :, :nb], kmax) and np.array_equal(ktf[1, :, :nb], kmin), f"{tag}: final KT"

    hits = hits_o = []
    if wl.n_needles:
        needles = synth.needle_positions(wl, layer, b)
        hits = _needle_hits(wl, needles, got, lambda s: task["sb"][s])
        hits_o = _needle_hits(wl, needles, ref_keep, lambda s: ref_sel[s])
    return {"worst": worst, "exempt": exempt, "hits": hits, "hits_oracle": hits_o}


def check_pairs(tasks, procs=None):
    """check_pair over every task: in this process for a few tasks, otherwise over
    single-threaded spawn workers (one per host core, at most len(tasks))."""
    procs = procs or min(len(tasks), os.cpu_count() or 1)
    if procs <= 1 or len(tasks) <= 2:
        return [check_pair(t) for t in tasks]
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        with mp.get_context("spawn").Pool(procs) as pool:
            return pool.map(check_pair, tasks, chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
