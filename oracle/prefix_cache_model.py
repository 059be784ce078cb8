"""Plain Python model of the block allocator with its prefix cache.

TEST INFRASTRUCTURE ONLY (part of the oracle; see oracle/__init__.py).  It
states the policy in the simplest terms so that the C++ allocator can be
checked against it operation by operation:

* "micro-vLLM" wiki, execution chain: the KVCacheManager allocates and
  releases blocks and keeps the prefix cache;
* "从零手写 vLLM 核心：mini-vllm 项目深度解析" §2: blocks are shared by
  reference and handed out on demand; a request that does not fit is refused
  whole (admission control); §工程启示: KV rollback.

Policy: a block is free, cached (count 0, registered hash) or live.  New
blocks come from the free blocks, lowest id first among never-used ones and
most recently freed first after that (a stack), then from cached blocks,
least recently released first.
"""
from __future__ import annotations

BLOCK = 16


class ModelError(Exception):
    def __init__(self, code):
        super().__init__(code)
        self.code = code  # 1 invalid, 3 no blocks, 4 bad block id


class PrefixCacheModel:
    def __init__(self, num_blocks: int):
        self.n = num_blocks
        self.free = list(range(num_blocks - 1, -1, -1))  # stack, top at the end
        self.refs = [0] * num_blocks
        self.hash_of = {}      # block -> hash
        self.by_hash = {}      # hash -> block
        self.cached = []       # count-0 registered blocks, oldest first

    def _live(self, b):
        return 0 <= b < self.n and self.refs[b] > 0

    def _take(self):
        if self.free:
            b = self.free.pop()
        else:
            b = self.cached.pop(0)
            self._unregister(b)
        self.refs[b] = 1
        return b

    def _unregister(self, b):
        h = self.hash_of.pop(b, None)
        if h is not None and self.by_hash.get(h) == b:
            del self.by_hash[h]

    def _drop(self, b):
        self.refs[b] -= 1
        if self.refs[b] == 0:
            if b in self.hash_of:
                self.cached.append(b)
            else:
                self.free.append(b)

    def num_free(self):
        return len(self.free) + len(self.cached)

    def alloc(self, k):
        if k > self.num_free():
            raise ModelError(3)
        return [self._take() for _ in range(k)]

    def share(self, ids):
        if not all(self._live(b) for b in ids):
            raise ModelError(4)
        for b in ids:
            self.refs[b] += 1

    def _check_droppable(self, ids):
        """Every id live and named at most as often as it is referenced."""
        if not all(self._live(b) for b in ids):
            raise ModelError(4)
        for b in set(ids):
            if ids.count(b) > self.refs[b]:
                raise ModelError(4)

    def free_ids(self, ids):
        self._check_droppable(ids)
        for b in ids:
            self._drop(b)

    def insert(self, b, h):
        if not self._live(b):
            raise ModelError(4)
        if b in self.hash_of:
            if self.hash_of[b] != h:
                raise ModelError(1)
            return
        if h in self.by_hash:
            return
        self.by_hash[h] = b
        self.hash_of[b] = h

    def lookup(self, hashes):
        out = []
        for h in hashes:
            b = self.by_hash.get(h)
            if b is None:
                break
            if self.refs[b] == 0:
                self.cached.remove(b)
            self.refs[b] += 1
            out.append(b)
        return out

    def cow(self, b):
        if not self._live(b):
            raise ModelError(4)
        if self.refs[b] == 1:
            self._unregister(b)
            return b, False
        if not self.num_free():
            raise ModelError(3)
        nb = self._take()
        self.refs[b] -= 1
        return nb, True

    def rollback(self, table, new_len):
        keep = -(-new_len // BLOCK)
        if keep > len(table):
            raise ModelError(1)
        self._check_droppable(list(table[keep:]))
        for b in table[keep:]:
            self._drop(b)
        if keep and new_len % BLOCK and self.refs[table[keep - 1]] == 1:
            self._unregister(table[keep - 1])
        return table[:keep]
