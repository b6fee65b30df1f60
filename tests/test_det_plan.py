"""CPU checks of the deterministic backward's plan (which unit adds to which dQ
tile when), read back through attn_bwd_det_plan from the same code the kernels
run ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
Asymmetric Hardware Scaling", abstract and Figures 7-8: a fixed order of the
key tiles' additions makes dQ bit-reproducible).

What must hold for the tickets never to deadlock and for the sums to be fixed:
- every dQ tile's additions carry ranks 0 .. m-1, once each (m = the key
  tiles that see it);
- every unit visits each of its query tiles exactly once;
- with the units taken in rounds of n_ctas co-resident CTAs (the persistent
  kernel) or launched in unit order, always some addition can go ahead until
  all are done (simulated below without timing);
- the rotated walk puts a round's units of one head on distinct query tiles
  at every step, and a tile's predecessor in that round sigma steps earlier.
No GPU is used.
"""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def A():
    from exact_attention_77_gb300 import build

    build.build()
    import exact_attention_77_gb300 as A

    return A


def _walk(first, n, rotated, i_lo=0):
    out, i = [], first
    for _ in range(n - i_lo):
        out.append(i)
        i = (i - 1 if i > 0 else n - 1) if rotated else i - 1
    return out


def _rounds(n_units, G):
    """Persistent CTAs: CTA b takes unit r G + b (r even) or r G + G-1-b (r odd)."""
    seq = [[] for _ in range(G)]
    for r in range((n_units + G - 1) // G):
        for b in range(G):
            u = r * G + ((G - 1 - b) if (r & 1) else b)
            if u < n_units:
                seq[b].append(u)
    return seq


def _progresses(plan, n, G, causal, rotated):
    """Untimed run: each CTA works through its units' additions in walk order;
    an addition goes ahead when its tile's ticket equals its rank.  True when
    all finish (no set of CTAs waits on each other forever)."""
    head, key, first, rank = plan["head"], plan["key_tile"], plan["first_tile"], plan["rank"]
    seqs = _rounds(len(head), G)
    work = []
    for seq in seqs:
        w = []
        for u in seq:
            for i in _walk(int(first[u]), n, rotated, int(key[u]) if causal else 0):
                w.append((int(head[u]), i, int(rank[u, i])))
        work.append(w)
    ticket = {}
    pos = [0] * G
    total = sum(len(w) for w in work)
    done = 0
    while done < total:
        moved = False
        for b in range(G):
            while pos[b] < len(work[b]):
                h, i, r = work[b][pos[b]]
                if ticket.get((h, i), 0) != r:
                    break
                ticket[(h, i)] = r + 1
                pos[b] += 1
                done += 1
                moved = True
        if not moved:
            return False
    return True


CASES = [
    # n_heads, n_tiles, n_ctas, group, desc
    (16, 128, 152, 8, 0),
    (16, 128, 152, 16, 0),
    (16, 128, 152, 4, 1),
    (64, 32, 152, 8, 0),
    (64, 32, 152, 16, 1),
    (256, 8, 152, 256, 0),
    (3, 5, 7, 2, 0),  # a smaller last group, ragged rounds
    (2, 3, 4, 1, 1),
    (1, 1, 152, 1, 0),
]


@pytest.mark.parametrize("n_heads,n,G,group,desc", CASES)
@pytest.mark.parametrize("rotated", [0, 1])
def test_ranks_walks_and_progress(A, n_heads, n, G, group, desc, rotated):
    plan = A.attn_bwd_det_plan(n_heads, n, G, group, desc, 0, rotated)
    head, key, first, rank = plan["head"], plan["key_tile"], plan["first_tile"], plan["rank"]
    n_units = n_heads * n
    # every (head, key tile) unit exactly once
    assert sorted(zip(head.tolist(), key.tolist())) == [(h, j) for h in range(n_heads) for j in range(n)]
    # each unit visits every query tile once
    for u in range(n_units):
        assert sorted(_walk(int(first[u]), n, rotated)) == list(range(n))
    # each dQ tile's additions are ranked 0 .. n-1
    for h in range(n_heads):
        us = np.nonzero(head == h)[0]
        for i in range(n):
            assert sorted(rank[us, i].tolist()) == list(range(n))
    assert _progresses(plan, n, G, False, rotated)


@pytest.mark.parametrize("n_heads,n,G,group,desc", CASES)
def test_rotated_round_spreads_a_head_over_tiles(A, n_heads, n, G, group, desc):
    plan = A.attn_bwd_det_plan(n_heads, n, G, group, desc, 0, 1)
    head, first, rank = plan["head"], plan["first_tile"], plan["rank"]
    n_units = n_heads * n
    for r0 in range(0, n_units, G):
        units = range(r0, min(r0 + G, n_units))
        for h in set(int(head[u]) for u in units):
            mine = [u for u in units if head[u] == h]
            walks = [_walk(int(first[u]), n, True) for u in mine]
            for s in range(n):
                assert len({w[s] for w in walks}) == len(walks)  # distinct tiles at each step
            # within the round a tile's additions go in visiting order
            for i in range(n):
                order = sorted(mine, key=lambda u: _walk(int(first[u]), n, True).index(i))
                ranks = [int(rank[u, i]) for u in order]
                assert ranks == sorted(ranks) and ranks == list(range(ranks[0], ranks[0] + len(ranks)))


def test_rotated_without_shared_rounds_is_the_plain_plan(A):
    # one unit of a head per round: no rotation (the plain walk and ranks)
    a = A.attn_bwd_det_plan(256, 8, 152, 256, 0, 0, 1)
    b = A.attn_bwd_det_plan(256, 8, 152, 256, 0, 0, 0)
    for k in ("head", "key_tile", "first_tile", "rank"):
        assert np.array_equal(a[k], b[k])


@pytest.mark.parametrize("n_heads,n,G,group,desc", [(16, 32, 152, 16, 0), (16, 32, 152, 16, 1), (4, 9, 5, 2, 1)])
def test_causal_plan(A, n_heads, n, G, group, desc):
    plan = A.attn_bwd_det_plan(n_heads, n, G, group, desc, 1, 0)
    head, key, rank = plan["head"], plan["key_tile"], plan["rank"]
    for h in range(n_heads):
        us = np.nonzero(head == h)[0]
        for i in range(n):
            vis = [u for u in us if key[u] <= i]
            assert all(rank[u, i] == -1 for u in us if key[u] > i)
            assert sorted(rank[vis, i].tolist()) == list(range(i + 1))
    assert _progresses(plan, n, G, True, False)


def test_plan_argument_errors(A):
    lib = A.get_lib()
    z = np.zeros(64, np.int32)
    p = z.ctypes.data
    assert lib.attn_bwd_det_plan(0, 4, 4, 1, 0, 0, 0, p, p, p, p) == A.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_det_plan(2, 4, 4, 1, 2, 0, 0, p, p, p, p) == A.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_det_plan(2, 4, 4, 1, 0, 1, 1, p, p, p, p) == A.ATTN_ERR_INVALID_ARG  # rotated is non-causal
    assert lib.attn_bwd_det_plan(2, 4, 4, 1, 0, 0, 0, None, p, p, p) == A.ATTN_ERR_INVALID_ARG
