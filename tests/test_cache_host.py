"""Host-side cache bookkeeping in libphs.so: refcounted page allocator with
copy on write, radix prefix tree over whole pages, window-safe match length.
Checked against plain Python models on random operation sequences (index
work: exact equality).  CPU only."""
import numpy as np
import pytest

import paged_hybrid_sliding_gb300 as phs

P = 16


# ------------------------------------------------------------- allocator --
def test_allocator_matches_model():
    rng = np.random.default_rng(0)
    N = 64
    a = phs.PageAllocator(N)
    rc = np.zeros(N, np.int64)
    live = []
    for step in range(3000):
        op = rng.integers(0, 4)
        if op == 0:
            n = int(rng.integers(0, 6))
            if n > (rc == 0).sum():
                with pytest.raises(phs.PhsError) as e:
                    a.alloc(n)
                assert e.value.code == -11
                continue
            pages = a.alloc(n)
            assert np.all(rc[pages] == 0) and len(set(pages.tolist())) == n
            rc[pages] = 1
            live.extend(pages.tolist())
        elif op == 1 and live:
            p = [live[i] for i in rng.integers(0, len(live), size=int(rng.integers(1, 4)))]
            a.incref(p)
            for x in p:
                rc[x] += 1
            live.extend(p)
        elif op == 2 and live:
            i = int(rng.integers(0, len(live)))
            p = live.pop(i)
            a.decref([p])
            rc[p] -= 1
        elif op == 3 and live:
            p = live[int(rng.integers(0, len(live)))]
            if rc[p] > 1 and (rc == 0).sum() == 0:
                continue
            q = a.cow(p)
            if rc[p] == 1:
                assert q == p
            else:
                assert rc[q] == 0 and q != p
                rc[p] -= 1
                rc[q] = 1
                live.remove(p)
                live.append(q)
        assert a.free_count() == (rc == 0).sum()
    assert np.array_equal(a.refcounts(), rc)


def test_allocator_rejects_dead_pages_atomically():
    a = phs.PageAllocator(8)
    p = a.alloc(2)
    with pytest.raises(phs.PhsError):
        a.incref([p[0], 7])          # 7 was never allocated
    assert np.array_equal(a.refcounts()[p], [1, 1])   # nothing changed
    a.decref(p)
    with pytest.raises(phs.PhsError):
        a.decref(p)


# ----------------------------------------------------------------- radix --
class RadixModel:
    """Whole-page prefixes -> page id; the first insert of a prefix wins."""

    def __init__(self):
        self.page_of = {}

    def insert(self, tokens, pages):
        for k in range(len(tokens) // P):
            key = tuple(tokens[:(k + 1) * P])
            self.page_of.setdefault(key, int(pages[k]))

    def match(self, tokens):
        out = []
        for k in range(len(tokens) // P):
            key = tuple(tokens[:(k + 1) * P])
            if key not in self.page_of:
                break
            out.append(self.page_of[key])
        return out


def _random_sequences(rng, n, vocab=5):
    # sequences sharing prefixes: branch off a random earlier sequence
    seqs = []
    for i in range(n):
        L = int(rng.integers(P, 12 * P))
        if seqs and rng.random() < 0.8:
            base = seqs[int(rng.integers(0, len(seqs)))]
            cut = int(rng.integers(0, len(base) + 1))
            s = list(base[:cut]) + list(rng.integers(0, vocab, size=max(0, L - cut)))
        else:
            s = list(rng.integers(0, vocab, size=L))
        seqs.append(s)
    return seqs


@pytest.mark.parametrize("seed", range(4))
def test_radix_match_and_insert_match_model(seed):
    rng = np.random.default_rng(seed)
    a = phs.PageAllocator(4096)
    t = phs.RadixTree(a, P)
    model = RadixModel()
    held = []  # pages referenced by "requests" (from match and fresh allocations)
    for s in _random_sequences(rng, 60):
        got = t.match(s)
        want = model.match(s)
        assert got.tolist() == want
        held.extend(got.tolist())
        fresh = a.alloc(len(s) // P - len(got))
        held.extend(fresh.tolist())
        pages = np.concatenate([got, fresh]).astype(np.int32)
        t.insert(s, pages)
        model.insert(s, pages)
    # refcounts: one per request reference + one per cached page
    rc = np.zeros(4096, np.int64)
    for p in held:
        rc[p] += 1
    for p in set(model.page_of.values()):
        rc[p] += 1
    assert np.array_equal(a.refcounts(), rc)
    assert t.cached_pages() == len(model.page_of)
    # finishing every request leaves only the tree's references; evicting
    # everything frees them all
    a.decref(held)
    freed = t.evict(10 ** 6)
    assert freed == len(model.page_of)
    assert a.free_count() == 4096 and t.cached_pages() == 0


def test_radix_split_keeps_both_branches():
    a = phs.PageAllocator(32)
    t = phs.RadixTree(a, P)
    A = list(range(64))
    B = list(range(32)) + [99] * 32
    pa = a.alloc(4)
    t.insert(A, pa)
    got = t.match(B)                   # shares the first two pages
    assert got.tolist() == pa[:2].tolist()
    pb = np.concatenate([got, a.alloc(2)])
    t.insert(B, pb)
    assert t.match(A).tolist() == pa.tolist()
    assert t.match(B).tolist() == pb.tolist()
    assert t.cached_pages() == 6


def test_radix_evicts_lru_and_spares_pages_in_use():
    a = phs.PageAllocator(16)
    t = phs.RadixTree(a, P)
    seqs = [[i] * 32 for i in range(3)]
    pages = [a.alloc(2) for _ in seqs]
    for s, p in zip(seqs, pages):
        t.insert(s, p)
        a.decref(p)                    # the inserting request finished
    in_use = t.match(seqs[0])          # a live request on sequence 0
    a.decref(t.match(seqs[2]))         # a request on 2 came and went
    freed = t.evict(2)                 # LRU evictable leaf: sequence 1
    assert freed == 2
    rc = a.refcounts()
    assert np.all(rc[pages[1]] == 0) and np.all(rc[in_use] >= 2)
    freed = t.evict(100)               # sequence 2 goes too; 0 is in use
    assert t.cached_pages() == 2 and np.all(a.refcounts()[in_use] >= 2)


# ----------------------------------------------------------- window-safe --
def _window_safe_brute(valid, L, W, align):
    best = 0
    for l in range(1, L + 1):
        if l % align == 0 and all(valid[t] for t in range(max(0, l - W), l)):
            best = l
    return best


@pytest.mark.parametrize("seed", range(6))
def test_window_safe_len_brute_force(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        L = int(rng.integers(0, 90))
        W = int(rng.integers(1, 40))
        align = int(rng.choice([1, 4, 16]))
        valid = (rng.random(L) < rng.choice([0.5, 0.9, 0.99])).astype(np.uint8)
        assert phs.window_safe_len(valid, L, W, align) == _window_safe_brute(valid, L, W, align)


def test_radix_window_safe_match():
    # a finished request keeps the SWA KV of its last W tokens (saved as
    # segment pages): a new request sharing its prefix may only resume where
    # a whole window is covered, and gets that window's segment pages
    a = phs.PageAllocator(64)
    sa = phs.PageAllocator(16)
    t = phs.RadixTree(a, P, swa_alloc=sa)
    W = 32
    s = list(range(160))               # 10 pages
    seg = sa.alloc(2)
    t.insert(s, a.alloc(10), swa_pages=[-1] * 8 + seg.tolist())
    full = t.match(s)
    assert len(full) == 10
    safe, sw = t.match_window_safe(s, W)
    assert len(safe) == 10 and sw.tolist() == seg.tolist()
    safe, sw = t.match_window_safe(s[:150], W)   # tail [112,144) has no SWA KV
    assert len(safe) == 0 and len(sw) == 0
    # a second finished request maps more pages
    seg2 = sa.alloc(2)
    t.insert(s[:128], np.arange(8, dtype=np.int32), swa_pages=[-1] * 6 + seg2.tolist())
    safe, sw = t.match_window_safe(s[:150], W)
    assert len(safe) * P == 144        # [96,160) mapped now: [112,144) is covered
    assert sw.tolist() == [seg2[1], seg[0]]
    safe, sw = t.match_window_safe(s[:120], W)
    assert len(safe) == 0 and len(sw) == 0      # [80,112) is not
    assert t.match_window_safe(s[:16], 64)[0].tolist() == []   # page 0 has no SWA KV
    # every returned segment page carries a reference for the caller (on
    # top of the saving requests' own and the tree's)
    rc = sa.refcounts()
    assert rc[seg[1]] == 3 and rc[seg2[1]] == 3 and rc[seg[0]] == 4 and rc[seg2[0]] == 2


class HybridModel(RadixModel):
    """Adds, per cached page, the SWA segment page (the first one given)."""

    def __init__(self):
        super().__init__()
        self.swa_of = {}

    def insert(self, tokens, pages, swa):
        super().insert(tokens, pages)
        for k in range(len(tokens) // P):
            key = tuple(tokens[:(k + 1) * P])
            if swa[k] >= 0 and self.swa_of.get(key, -1) < 0:
                self.swa_of[key] = int(swa[k])

    def match_window_safe(self, tokens, W):
        pages = self.match(tokens)
        swa = [self.swa_of.get(tuple(tokens[:(k + 1) * P]), -1) for k in range(len(pages))]
        best = 0
        for L in range(P, len(pages) * P + 1, P):
            lo = L - min(L, W)
            if all(swa[j] >= 0 for j in range(lo // P, L // P)):
                best = L
        lo = best - min(best, W)
        return pages[:best // P], swa[lo // P:best // P]


@pytest.mark.parametrize("seed", range(3))
def test_radix_swa_mapping_matches_model(seed):
    rng = np.random.default_rng(100 + seed)
    W = 48
    a = phs.PageAllocator(4096)
    sa = phs.PageAllocator(2048)
    t = phs.RadixTree(a, P, swa_alloc=sa)
    model = HybridModel()
    held, held_swa = [], []
    for s in _random_sequences(rng, 60):
        got, gsw = t.match_window_safe(s, W)
        want, wsw = model.match_window_safe(s, W)
        assert got.tolist() == want and gsw.tolist() == wsw
        held.extend(got.tolist())
        held_swa.extend(gsw.tolist())
        npg = len(s) // P
        fresh = a.alloc(npg - len(got))
        held.extend(fresh.tolist())
        pages = np.concatenate([got, fresh]).astype(np.int32)
        # the finished request saved the segment pages of its last window
        # (whole pages only; some requests saved none)
        swa = np.full(npg, -1, np.int32)
        if rng.random() < 0.8 and npg:
            k = min(npg, W // P)
            swa[npg - k:] = sa.alloc(k)
            held_swa.extend(swa[npg - k:].tolist())
        t.insert(s, pages, swa_pages=swa)
        model.insert(s, pages, swa)
    rc = np.zeros(2048, np.int64)
    for p in held_swa:
        rc[p] += 1
    for p in set(model.swa_of.values()):
        rc[p] += 1
    assert np.array_equal(sa.refcounts(), rc)
    # requests finished: evicting everything releases the SWA pages too
    a.decref(held)
    sa.decref(held_swa)
    t.evict(10 ** 6)
    assert a.free_count() == 4096 and sa.free_count() == 2048


def test_radix_swa_mapping_argument_errors():
    a = phs.PageAllocator(8)
    t = phs.RadixTree(a, P)            # no SWA allocator
    with pytest.raises(phs.PhsError):
        t.insert(list(range(16)), a.alloc(1), swa_pages=[3])
    with pytest.raises(ValueError):
        phs.RadixTree(a, P, swa_alloc=a)
    sa = phs.PageAllocator(4)
    t2 = phs.RadixTree(a, P, swa_alloc=sa)
    with pytest.raises(phs.PhsError) as e:   # the window must be whole pages
        t2.match_window_safe(list(range(32)), 40)
    assert e.value.code == -7


def test_tree_keeps_its_allocators_alive():
    # the caller may let go of the allocators before the tree: the tree's
    # references keep them alive until it is destroyed
    a, sa = phs.PageAllocator(8), phs.PageAllocator(4)
    t = phs.RadixTree(a, P, swa_alloc=sa)
    s = list(range(32))
    t.insert(s, a.alloc(2), swa_pages=[-1, int(sa.alloc(1)[0])])
    a.close()
    sa.close()
    assert len(t.match(s)) == 2
    pages, seg = t.match_window_safe(s, 16)
    assert len(pages) == 2 and len(seg) == 1
    t.close()
