"""Host-side model of the router's arithmetic (CPU only).

`route_topk_kernel` splits the choices over a cluster of C CTAs (16, or 8
where 16 cannot be resident) and each CTA's chunk over 32 warps; pass 1
counts experts per warp segment, the per-warp prefixes and the other CTAs'
chunk counts give every warp its first row in each group, and pass 2 walks
each segment 32 choices at a time, ranking equal experts by lane.  This
model restates that partition and ranking and checks, for both cluster
sizes and awkward sizes (fewer choices than warps, sizes that leave empty
chunks and segments, ragged tails), that it gives the oracle's stable
routing and that every position lies in [0, routed rows).
"""
import numpy as np
import pytest

from oracle import dispatch as D

WARPS = 32


def _model(ids, E, C):
    ids = np.asarray(ids, np.int64).reshape(-1)
    n = ids.size
    per_cta = (n + C - 1) // C
    segs = []                                  # (cta, warp, s0, s1)
    for c in range(C):
        c0, c1 = min(n, c * per_cta), min(n, c * per_cta + per_cta)
        per = (c1 - c0 + WARPS - 1) // WARPS
        for w in range(WARPS):
            s0 = min(c1, c0 + w * per)
            s1 = min(c1, s0 + per)
            segs.append((c, w, s0, s1))
    hist = np.zeros((C, WARPS, E), np.int64)  # pass 1
    for c, w, s0, s1 in segs:
        for i in range(s0, s1):
            if 0 <= ids[i] < E:
                hist[c, w, ids[i]] += 1
    warp_prefix = np.cumsum(hist, axis=1) - hist          # exclusive over warps
    cnt = hist.sum(axis=1)                                # chunk counts [C, E]
    before = np.cumsum(cnt, axis=0) - cnt                 # earlier CTAs' counts
    tot = cnt.sum(axis=0)
    ro = np.concatenate([[0], np.cumsum(tot)])
    first = ro[:-1][None, None, :] + before[:, None, :] + warp_prefix
    src = np.full(n, -7, np.int64)
    dst = np.full(n, -9, np.int64)
    for c, w, s0, s1 in segs:                             # pass 2
        h = first[c, w].copy()
        for b in range(s0, s1, 32):
            lanes = [(i, ids[i]) for i in range(b, min(b + 32, s1))]
            for lane, (i, e) in enumerate(lanes):
                if not 0 <= e < E:
                    dst[i] = -1
                    continue
                rank = sum(1 for _, e2 in lanes[:lane] if e2 == e)
                pos = h[e] + rank
                assert 0 <= pos < ro[-1]
                src[pos] = i
                dst[i] = pos
            for e in {e for _, e in lanes if 0 <= e < E}:
                h[e] += sum(1 for _, e2 in lanes if e2 == e)
    return ro, src[:ro[-1]], dst


@pytest.mark.parametrize("C", [16, 8])
@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (3, 2, 3), (7, 3, 5), (40, 8, 64), (129, 2, 8),
                                   (300, 4, 33), (1000, 1, 2)])
def test_router_partition_and_ranks_give_the_stable_routing(C, T, k, E):
    rng = np.random.default_rng(T * 31 + k)
    ids = np.stack([rng.choice(E, min(k, E), replace=False) for _ in range(T)]).astype(np.int64)
    if T > 10:
        ids[3, 0] = -1                                    # dropped choices
        ids[T - 2, -1] = E
    ro, src, dst = _model(ids, E, C)
    ro_ref, _, src_ref, _ = D.route_topk(ids, E)
    assert np.array_equal(ro, ro_ref.astype(np.int64))
    assert np.array_equal(src, src_ref.astype(np.int64))
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    assert np.all(dst[~valid] == -1)
    assert np.array_equal(src[dst[valid]], np.nonzero(valid)[0])   # dst inverts src
