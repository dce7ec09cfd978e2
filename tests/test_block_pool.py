"""The host page allocator with prefix caching (psw_block_pool_*, C++ in
libpsw) against a plain-Python model of "Gemma 4 model architecture
analysis" sections 6.2 and 6.6 (oracle/block_pool.py).

The model itself is pinned first: its FNV-1a against the hash's published
test vectors, and its behaviour against the pages' semantics (pages shared
by requests with a common prefix, reference counts, least-recently-freed
reuse, freed pages still hit until reused). Then the native pool must give
the model's exact answers (ids, hits, counts, errors) on long random
sequences of operations."""
import numpy as np
import pytest

from oracle import block_pool as model
from paged_sliding_window_gb300 import binding, build


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return binding.load()


# ---------------------------------------------------------------- model pins
def test_model_fnv1a_published_vectors():
    # FNV-1a 64-bit test vectors of the hash's published definition
    assert model.fnv1a64(b"") == 0xCBF29CE484222325
    assert model.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert model.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_model_prefix_sharing_semantics():
    """Two requests with a common 48-token prefix: the second shares the
    first three pages (reference count 2) and computes only the rest."""
    m = model.BlockPoolModel(16)
    a = list(range(1000, 1078))           # 78 tokens
    b = a[:48] + list(range(5000, 5020))  # 68 tokens, 48 in common
    rc, row_a, cached_a = m.admit(a, 8)
    assert rc == 0 and cached_a == 0 and row_a[:5] == [0, 1, 2, 3, 4] and row_a[5:] == [-1] * 3
    assert m.commit(a, row_a) == 0       # four full pages named
    rc, row_b, cached_b = m.admit(b, 8)
    assert rc == 0 and cached_b == 48 and row_b[:3] == row_a[:3]
    assert [m.ref[x] for x in row_a[:3]] == [2, 2, 2] and m.ref[row_a[3]] == 1
    assert row_b[3:5] == [5, 6]           # the rest comes from the free queue
    # the page holding a prompt's last token is never taken from the cache
    rc, row_c, cached_c = m.admit(a[:32], 8)
    assert cached_c == 16 and row_c[0] == row_a[0] and row_c[1] != row_a[1]


def test_model_lru_reuse_and_freed_pages_still_hit():
    m = model.BlockPoolModel(4)
    toks = list(range(32))
    rc, row, _ = m.admit(toks + [99], 4)   # pages 0, 1, 2
    m.commit(toks + [99], row)
    assert m.release(row[:3][::-1]) == 0   # freed back to front: 2, 1, 0 join the queue
    assert m.free == [3, 2, 1, 0]
    rc, row2, cached = m.admit(toks + [7], 4)  # hits pages 0 and 1 although they are free
    assert cached == 32 and row2 == [0, 1, 3, -1] and m.free == [2]  # the head (3) was reused
    # allocating the last free page evicts nothing cached; exhausting the pool fails cleanly
    assert m.allocate(2)[0] == model.ENOBLOCKS and m.free == [2]


def test_model_release_checks_before_changing_anything():
    m = model.BlockPoolModel(4)
    _, ids = m.allocate(2)
    assert m.release([ids[0], ids[0]]) == model.EBLOCK  # held once, released twice
    assert m.ref[ids[0]] == 1 and m.release([7]) == model.EBLOCK


# ---------------------------------------------------------------- native pool
def test_native_hash_matches_model():
    rng = np.random.default_rng(5)
    parent = 0
    for _ in range(50):
        toks = rng.integers(-2 ** 31, 2 ** 31, size=16).tolist()
        h = binding.block_hash(parent, toks)
        assert h == model.block_hash(parent, toks)
        parent = h


def test_native_pool_scenario():
    p = binding.BlockPool(16)
    a = list(range(1000, 1078))
    b = a[:48] + list(range(5000, 5020))
    rc, row_a, ca = p.admit(a, 8)
    assert rc == 0 and ca == 0 and row_a[:5] == [0, 1, 2, 3, 4]
    assert p.commit(a, row_a) == 0
    rc, row_b, cb = p.admit(b, 8)
    assert cb == 48 and row_b[:3] == row_a[:3] and [p.ref_count(x) for x in row_a[:3]] == [2] * 3
    assert p.release([row_a[0], row_a[0], row_a[0]]) == -20  # held twice, not three times
    assert p.ref_count(row_a[0]) == 2
    assert p.allocate(100)[0] == -19 and p.num_free() == 16 - 7


@pytest.mark.parametrize("prefix_cache", [True, False])
def test_native_pool_matches_model_on_random_operations(prefix_cache):
    rng = np.random.default_rng(11 + prefix_cache)
    n_blocks = 48
    p, m = binding.BlockPool(n_blocks, prefix_cache), model.BlockPoolModel(n_blocks, prefix_cache)
    prompts = [rng.integers(0, 50, size=int(rng.integers(1, 200))).tolist() for _ in range(6)]
    live = []  # (tokens, row)
    for step in range(3000):
        op = rng.integers(0, 4)
        if op == 0 or not live:  # admit a prompt, often sharing a prefix with another
            base = prompts[int(rng.integers(0, len(prompts)))]
            cut = int(rng.integers(0, len(base) + 1))
            toks = base[:cut] + rng.integers(0, 50, size=int(rng.integers(1, 40))).tolist()
            got, want = p.admit(toks, 16), m.admit(toks, 16)
            assert got == tuple(want) if want[1] is not None else got[0] == want[0], step
            if got[0] == 0:
                live.append((toks, got[1]))
                if rng.random() < 0.7:
                    assert p.commit(toks, got[1]) == m.commit(toks, got[1])
        elif op == 1:  # release a request, back to front
            toks, row = live.pop(int(rng.integers(0, len(live))))
            ids = [x for x in row if x >= 0][::-1]
            assert p.release(ids) == m.release(ids), step
        elif op == 2:  # raw allocation and its release
            n = int(rng.integers(0, 6))
            got, want = p.allocate(n), m.allocate(n)
            assert got[0] == want[0] and got[1] == want[1], step
            if got[0] == 0 and got[1]:
                assert p.release(got[1]) == m.release(want[1]) == 0
        else:  # a bad release: nothing may change
            bad = [int(rng.integers(0, n_blocks))] * 3
            assert p.release(bad) == m.release(bad), step
        assert p.num_free() == m.num_free(), step
        for blk in range(0, n_blocks, 7):
            assert p.ref_count(blk) == m.ref[blk], (step, blk)
