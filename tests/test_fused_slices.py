"""Host restatement of the fused decode step's bookkeeping (no GPU).

The fused step (IDX_FUSED_SELECT) gives scorer CTA c the slice
[P c / G, P (c + 1) / G) of the (request, page) order; every CTA writes a
local top 16 per (request, row) of its slice to candidate slot b + c, adds
its page count to the request's counter, and the CTA whose addition
completes the count merges the candidates of CTAs cta_of(first page) ..
cta_of(last page), skipping empty slices.  Requests without pages are
written by CTA b mod G.  These checks walk the same arithmetic on the host,
for shapes with empty slices, one request over every CTA, and thousands of
requests per slice, and confirm that

  * cta_of(u) is the CTA whose slice holds position u;
  * the request lists built a round at a time cover each slice exactly;
  * (request, CTA) pairs that share pages have distinct slots b + c, all
    below num_reqs + 512 (the workspace's slot count);
  * every request with pages is won by exactly one CTA, whose merge range
    holds exactly the CTAs that wrote its candidates;
  * every request is written exactly once;

and that the merge of two descending candidate lists by rank counting is
the top 16 of their union, so folding the parts' local top 16s gives the
row's top 16.
"""

import numpy as np
import pytest

MAX_GRID = 512
CHUNK_REQS = 128


def cta_of(u, P, G):
    return ((u + 1) * G - 1) // P


def p0(c, P, G):
    return P * c // G


def simulate(npages, G):
    B = len(npages)
    P = int(sum(npages))
    off = np.concatenate([[0], np.cumsum(npages)])
    counters = np.zeros(B, dtype=np.int64)
    slots = {}
    wins = {}
    written = np.zeros(B, dtype=np.int64)
    for c in range(G):  # zero-page requests
        for b in range(c, B, G):
            if npages[b] == 0:
                written[b] += 1
    for c in range(G):
        lo_p, hi_p = p0(c, P, G), p0(c + 1, P, G)
        count = hi_p - lo_p
        if count == 0:
            continue
        # (b0, j0): the request holding position lo_p
        b0 = int(np.searchsorted(off, lo_p, side="right") - 1)
        while npages[b0] == 0:
            b0 += 1
        j0 = lo_p - off[b0]
        assert 0 <= j0 < npages[b0]
        b, lo, rem, o = b0, j0, count, lo_p - j0
        covered = 0
        while True:
            reqs = []
            while rem > 0 and len(reqs) < CHUNK_REQS and b < B:
                n = npages[b]
                take = min(n - lo, rem)
                if take > 0:
                    reqs.append((b, lo, lo + take, o, n))
                    rem -= take
                o += n
                b += 1
                lo = 0
            if not reqs:
                break
            for (rb, rlo, rhi, roff, rn) in reqs:
                assert roff == off[rb]
                # every page of the list lies in this slice
                assert lo_p <= roff + rlo and roff + rhi <= hi_p
                covered += rhi - rlo
                slot = rb + c
                assert slot < B + MAX_GRID
                assert slot not in slots, "two (request, CTA) pairs share a candidate slot"
                slots[slot] = (rb, c)
            for (rb, rlo, rhi, roff, rn) in reqs:
                before = counters[rb]
                counters[rb] += rhi - rlo
                if before + (rhi - rlo) == rn:
                    assert rb not in wins
                    wins[rb] = c
                    counters[rb] = 0
        assert covered == count
    for b in range(B):
        if npages[b] == 0:
            continue
        assert b in wins, "a request nobody merged"
        assert counters[b] == 0
        written[b] += 1
        cf, cl = cta_of(off[b], P, G), cta_of(off[b] + npages[b] - 1, P, G)
        merged = [c for c in range(cf, cl + 1) if p0(c + 1, P, G) > p0(c, P, G)]
        wrote = sorted(c for (rb, c) in slots.values() if rb == b)
        assert merged == wrote
    assert (written == 1).all()
    return P


@pytest.mark.parametrize("seed", range(6))
def test_cta_of_finds_the_slice(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        G = int(rng.integers(1, 200))
        P = int(rng.integers(1, 5000))
        u = rng.integers(0, P, size=50)
        c = cta_of(u, P, G)
        assert ((p0(c, P, G) <= u) & (u < p0(c + 1, P, G))).all()
        assert (c < G).all()


@pytest.mark.parametrize("case", ["ragged", "fewer_pages_than_ctas", "one_request", "zero_page_mix",
                                  "many_small", "long_context"])
def test_slices_lists_slots_and_merges(case):
    rng = np.random.default_rng(7)
    G = 152
    if case == "ragged":
        npages = rng.integers(64, 1313, size=64)
    elif case == "fewer_pages_than_ctas":
        npages = np.array([23, 29, 31])
    elif case == "one_request":
        npages = np.array([3906])
    elif case == "zero_page_mix":
        npages = np.array([0, 0, 7, 0, 15, 16, 17, 0, 31, 0, 1, 0])
    elif case == "many_small":
        npages = np.where(np.arange(20_000) % 500 == 0, rng.integers(150, 234, size=20_000), 1)
    else:
        npages = np.full(16, 3906)
    simulate([int(x) for x in npages], G)
    simulate([int(x) for x in npages], 7)


def test_no_pages_at_all():
    simulate([0, 0, 0, 0], 152)


def merge16(run, lst):
    """Host restatement of the merge the fused step's last CTA uses: the top
    16 of two descending lists of 16 distinct nonzero keys (0 padding); a
    key's place is its index in its own list plus the larger keys of the
    other list."""
    top = [0] * 16
    for own, other in ((run, lst), (lst, run)):
        for idx, x in enumerate(own):
            if x == 0:
                continue
            rank = idx + sum(1 for y in other if y > x)
            if rank < 16:
                top[rank] = x
    return top


@pytest.mark.parametrize("seed", range(4))
def test_merge_of_sorted_lists_is_the_union_top16(seed):
    rng = np.random.default_rng(100 + seed)
    for _ in range(2000):
        keys = rng.choice(np.arange(1, 200, dtype=np.int64), size=int(rng.integers(0, 33)), replace=False)
        split = int(rng.integers(0, len(keys) + 1))
        a = sorted(keys[:split].tolist(), reverse=True)[:16]
        b = sorted(keys[split:].tolist(), reverse=True)[:16]
        pad = lambda v: v + [0] * (16 - len(v))
        want = pad(sorted(a + b, reverse=True)[:16])
        assert merge16(pad(a), pad(b)) == want
    # folding the lists of several parts gives the top 16 of their union,
    # which is the top 16 of the row when each part holds its own top 16
    for _ in range(300):
        row = rng.permutation(np.arange(1, 400, dtype=np.int64))[: int(rng.integers(1, 300))]
        cuts = np.sort(rng.integers(0, len(row) + 1, size=int(rng.integers(0, 6))))
        parts = np.split(row, cuts)
        run = None
        for p in parts:
            loc = sorted(p.tolist(), reverse=True)[:16]
            loc = loc + [0] * (16 - len(loc))
            run = loc if run is None else merge16(run, loc)
        want = sorted(row.tolist(), reverse=True)[:16]
        assert run == want + [0] * (16 - len(want))
