"""Host bookkeeping of prefix sharing (no GPU): page reference counts and
the token-keyed index of whole-page prefixes (Vosti abstract: a paged,
prefix-sharing KV cache with KV tied to its logical token prefix)."""
import pytest

from deterministic_invariant_bf16_gb300.engine import PageAllocator, PrefixIndex


def test_shared_pages_return_after_the_last_owner():
    a = PageAllocator(8, seed=3)
    p = a.take(3)
    assert len(a.free) == 5
    a.share(p[:2])
    a.give_back(p)               # first owner: only the unshared page frees
    assert len(a.free) == 6 and p[2] in a.free and p[0] not in a.free
    a.give_back(p[:2])           # second owner
    assert len(a.free) == 8
    with pytest.raises(RuntimeError):
        a.give_back([p[0]])      # not in use any more
    with pytest.raises(RuntimeError):
        a.share([p[0]])
    with pytest.raises(RuntimeError):
        a.take(9)


def test_prefix_index_whole_pages_only():
    ix = PrefixIndex()
    toks = list(range(100, 150))                 # 50 tokens: 3 whole pages
    ix.add(4, toks)
    assert ix.lookup(toks) == (4, 48)
    assert ix.lookup(toks[:47]) == (4, 32)       # 2 whole pages of the query
    assert ix.lookup(toks[:15]) == (None, 0)     # less than a page
    other = toks[:20] + [7] * 30                 # diverges inside page 2
    assert ix.lookup(other) == (4, 16)
    assert ix.lookup([1] + toks[1:]) == (None, 0)
    ix.add(5, toks + list(range(30)))            # longer owner of the same
    assert ix.lookup(toks) == (4, 48)            # first owner kept
    assert ix.lookup(toks + list(range(30)))[1] == 80
    ix.drop(4)
    assert ix.lookup(toks) == (5, 48)
