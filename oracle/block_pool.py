"""Plain-Python model of the page allocator with prefix caching.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only the tests use it; it
shares no code with the library's C++ pool and never imports the package.

It follows "Gemma 4 model architecture analysis" (vLLM-Kunlun), section 6.2
(each page is {block_id, ref_cnt, block_hash}; unreferenced pages wait in a
free queue in least-recently-freed order) and section 6.6 (prefix caching:
a full page is named by the hash of its tokens chained with the previous
page's, and ``get_cached_block`` on a hit touches the page and raises its
reference count). Everything is the most direct Python: a list for the free
queue (popped from the front, appended at the back, removed from the middle
on a hit), a dict from hash to block id.

The page hash is FNV-1a over 64 bits, from its published definition: start
at the offset basis 14695981039346656037; for every byte, xor it in, then
multiply by the prime 1099511628211 modulo 2^64. A page's bytes are its
parent hash (8 bytes, little-endian) followed by its tokens (4 bytes each,
little-endian two's complement).
"""
from __future__ import annotations

BLOCK_SIZE = 16
FNV_OFFSET = 14695981039346656037
FNV_PRIME = 1099511628211
MASK64 = (1 << 64) - 1

OK, ENULL, ECAPACITY, ENOBLOCKS, EBLOCK = 0, -1, -11, -19, -20


def fnv1a64(data: bytes, h: int = FNV_OFFSET) -> int:
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(parent: int, tokens) -> int:
    data = int(parent).to_bytes(8, "little")
    for t in tokens:
        data += (int(t) & 0xFFFFFFFF).to_bytes(4, "little")
    return fnv1a64(data)


class BlockPoolModel:
    def __init__(self, num_blocks: int, prefix_cache: bool = True):
        self.ref = [0] * num_blocks
        self.hash_of = [None] * num_blocks
        self.free = list(range(num_blocks))  # front = least recently freed
        self.cached = {}
        self.prefix_cache = prefix_cache

    def num_free(self) -> int:
        return len(self.free)

    def allocate(self, n: int):
        if n > len(self.free):
            return ENOBLOCKS, []
        ids = []
        for _ in range(n):
            b = self.free.pop(0)
            if self.hash_of[b] is not None:  # reused page: its old name goes
                if self.cached.get(self.hash_of[b]) == b:
                    del self.cached[self.hash_of[b]]
                self.hash_of[b] = None
            self.ref[b] = 1
            ids.append(b)
        return OK, ids

    def release(self, ids) -> int:
        need = {}
        for b in ids:
            if not 0 <= b < len(self.ref):
                return EBLOCK
            need[b] = need.get(b, 0) + 1
            if need[b] > self.ref[b]:
                return EBLOCK
        for b in ids:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        return OK

    def get_cached(self, h: int) -> int:
        if not self.prefix_cache or h not in self.cached:
            return -1
        b = self.cached[h]
        if self.ref[b] == 0:
            self.free.remove(b)
        self.ref[b] += 1
        return b

    def cache(self, b: int, h: int) -> int:
        if not 0 <= b < len(self.ref) or self.ref[b] <= 0:
            return EBLOCK
        if not self.prefix_cache or h in self.cached:
            return OK
        if self.hash_of[b] is not None and self.cached.get(self.hash_of[b]) == b:
            del self.cached[self.hash_of[b]]
        self.hash_of[b] = h
        self.cached[h] = b
        return OK

    def admit(self, tokens, max_blocks: int):
        """Returns (status, table_row, n_cached_tokens)."""
        n = len(tokens)
        need = (n + BLOCK_SIZE - 1) // BLOCK_SIZE
        if need > max_blocks:
            return ECAPACITY, None, 0
        full = (n - 1) // BLOCK_SIZE if n > 0 else 0
        row, parent = [], 0
        for i in range(full):
            h = block_hash(parent, tokens[i * BLOCK_SIZE:(i + 1) * BLOCK_SIZE])
            b = self.get_cached(h)
            if b < 0:
                break
            row.append(b)
            parent = h
        rc, ids = self.allocate(need - len(row))
        if rc != OK:
            self.release(row)
            return rc, None, 0
        row += ids
        return OK, row + [-1] * (max_blocks - need), (len(row) - len(ids)) * BLOCK_SIZE

    def commit(self, tokens, row) -> int:
        parent = 0
        for i in range(len(tokens) // BLOCK_SIZE):
            h = block_hash(parent, tokens[i * BLOCK_SIZE:(i + 1) * BLOCK_SIZE])
            rc = self.cache(row[i], h)
            if rc != OK:
                return rc
            parent = h
        return OK
