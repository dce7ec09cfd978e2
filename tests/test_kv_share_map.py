"""The KV-sharing map and layer types of a hybrid stack (psw_kv_share_map,
host arithmetic through the C ABI) against the topologies printed on the
pages and the interleaving rule of InfiniLM PR 581 (Gemma-3 item 2)."""
import json
import os

import pytest

from paged_sliding_window_gb300 import binding, build

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return binding.load()


def test_interleaving_rule_5_to_1():
    """(i + 1) % pattern == 0 -> full: pattern 6 gives five sliding layers then
    one full layer, repeated."""
    full, target = binding.kv_share_map(12, 6)
    assert full == [False] * 5 + [True] + [False] * 5 + [True]
    assert target == list(range(12))


def test_gemma4_e2b_topology_matches_the_page():
    g = json.load(open(os.path.join(GOLDEN, "kv_share_e2b.json")))
    n, owners = g["n_layers"], g["owners"]
    full, target = binding.kv_share_map(n, 5, n - owners)
    assert target[:owners] == list(range(owners))
    assert {str(i): target[i] for i in range(owners, n)} == g["shared_targets"]
    for layer, kind in g["source_layer_types"].items():
        assert full[int(layer)] == (kind == "full")
    readers = {s: sum(1 for t in target[owners:] if t == int(s)) for s in g["readers_per_source"]}
    assert readers == g["readers_per_source"]
    # each shared layer reads a layer of its own type
    assert all(full[i] == full[target[i]] for i in range(n))
    # 15 caches instead of 35
    assert len(set(target)) == owners


def test_gemma3n_e2b_topology_matches_the_page():
    g = json.load(open(os.path.join(GOLDEN, "kv_share_gemma3n_e2b.json")))
    lo, hi = g["shared_layers"]
    n = g["n_layers"]
    _, target = binding.kv_share_map(n, 5, hi - lo + 1)
    assert sorted(set(target[lo:hi + 1])) == g["source_layers"]
    assert target[:lo] == list(range(lo))


def test_share_map_rejects_bad_stacks():
    lib = binding.load()
    for args in ((0, 5, 0), (10, 0, 0), (10, 5, 10), (10, 5, -1), (10, 5, 9)):
        assert lib.psw_kv_share_map(*args, None, None) == -18, args
