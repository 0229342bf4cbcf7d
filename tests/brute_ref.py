"""Pure-Python brute force of the whole two-stage path, for tiny inputs only.

Written independently of the numpy oracle (plain lists, math.exp, full
sorts) so that a slip in either one shows up as a disagreement.  Follows the
same pages ("RocketKV: Accelerating Long-Context LLM Inference via Two-Stage
KV Cache Compression", method details: SnapKV stage, HSA Algorithm 1,
RocketKV-MT) and the same readings of them.
"""
import math


def _dot(a, b):
    return sum(x * y for x, y in zip(a, b))


def full_sort_topk(vals, k):
    """k largest by full sort on (-value, index); ascending indices."""
    order = sorted(range(len(vals)), key=lambda i: (-vals[i], i))
    return sorted(order[:k])


def snap_keep(q_obs, K, B1, W, P, scale, n_sink=0):
    """q_obs[g][w][d], K[j][d] lists.  Returns (keep, pooled)."""
    S = len(K)
    if B1 >= S or S - W <= 0:
        return list(range(S)), []
    score = [0.0] * (S - W)
    for g in range(len(q_obs)):
        for w in range(W):
            last = S - W + w
            logits = [_dot(q_obs[g][w], K[j]) * scale for j in range(last + 1)]
            m = max(logits)
            e = [math.exp(x - m) for x in logits]
            tot = sum(e)
            for j in range(S - W):
                score[j] += e[j] / tot
    half = P // 2
    pooled = []
    for j in range(S - W):
        lo, hi = max(0, j - half), min(S - W - 1, j + half)
        pooled.append(max(score[lo:hi + 1]))
    n_top = B1 - W - n_sink
    cand = pooled[n_sink:]
    top = [i + n_sink for i in full_sort_topk(cand, n_top)]
    return list(range(n_sink)) + top + list(range(S - W, S)), pooled


def kt(Kc, n, blk):
    D = len(Kc[0])
    nblk = (n + blk - 1) // blk
    kmax = [[0.0] * nblk for _ in range(D)]
    kmin = [[0.0] * nblk for _ in range(D)]
    for b in range(nblk):
        rows = Kc[b * blk:min(n, (b + 1) * blk)]
        for c in range(D):
            col = [r[c] for r in rows]
            kmax[c][b] = max(col)
            kmin[c][b] = min(col)
    return kmax, kmin


def hsa(qg, Kc, Vc, n, kmax, kmin, blk, k1, k2, scale):
    """qg[g][d].  Returns (y[g][d], i1, i2, s)."""
    G, D = len(qg), len(qg[0])
    a = [sum(abs(qg[g][c]) for g in range(G)) for c in range(D)]
    i1 = full_sort_topk(a, k1)
    nblk = (n + blk - 1) // blk
    s = []
    for b in range(nblk):
        tot = 0.0
        for c in i1:
            qs = sum(qg[g][c] for g in range(G))
            tot += qs * (kmax[c][b] if qs >= 0 else kmin[c][b])
        s.append(tot)
    i2 = full_sort_topk(s, k2)
    toks = [b * blk + i for b in i2 for i in range(blk) if b * blk + i < n]
    y = []
    for g in range(G):
        logits = [_dot(qg[g], Kc[j]) * scale for j in toks]
        m = max(logits)
        e = [math.exp(x - m) for x in logits]
        tot = sum(e)
        y.append([sum(e[t] * Vc[toks[t]][d] for t in range(len(toks))) / tot for d in range(D)])
    return y, i1, i2, s


def hsa_masked(qg, K, V, n, cand, blk, k1, k2, scale):
    """RocketKV-MT over fixed blocks of the full cache (the other multi-turn
    reading): bounds over candidate rows only, blocks without a candidate
    last, the newest row's block first, attention over the candidate rows of
    the chosen blocks.  Returns (y, i1, i2)."""
    G, D = len(qg), len(qg[0])
    a = [sum(abs(qg[g][c]) for g in range(G)) for c in range(D)]
    i1 = full_sort_topk(a, k1)
    nblk = (n + blk - 1) // blk
    s = []
    for b in range(nblk):
        rows = [r for r in range(b * blk, min(n, (b + 1) * blk)) if cand[r]]
        if not rows:
            s.append(-math.inf)
            continue
        tot = 0.0
        for c in i1:
            qs = sum(qg[g][c] for g in range(G))
            col = [K[r][c] for r in rows]
            tot += qs * (max(col) if qs >= 0 else min(col))
        s.append(tot)
    tail = (n - 1) // blk
    if s[tail] != -math.inf:
        s[tail] = math.inf
    i2 = full_sort_topk(s, k2)
    toks = [b * blk + i for b in i2 for i in range(blk) if b * blk + i < n and cand[b * blk + i]]
    y = []
    for g in range(G):
        logits = [_dot(qg[g], K[j]) * scale for j in toks]
        m = max(logits)
        e = [math.exp(x - m) for x in logits]
        tot = sum(e)
        y.append([sum(e[t] * V[toks[t]][d] for t in range(len(toks))) / tot for d in range(D)])
    return y, i1, i2
