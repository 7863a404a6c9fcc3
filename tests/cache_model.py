"""Plain-Python model of the cache manager's policies, for the tests only.

Written from the policy rules (position-agnostic: one copy of a document serves
any offset; position-aware: one copy per (document, offset); prefix caching: a
copy serves only the same preceding segments), with exact tuple keys where the
library hashes the prefix, a list as the free stack and an OrderedDict as the
LRU order. It also records which (identity, block index) every block id was
last filled with, so a test can check that a hit never hands out blocks that
were since reused for something else.
"""
from collections import OrderedDict

BLOCK = 16
AGNOSTIC, AWARE, PREFIX = 0, 1, 2


def nblocks(n):
    return (n + BLOCK - 1) // BLOCK


class _Entry:
    def __init__(self, key, doc, offset, tokens, blocks):
        self.key, self.doc, self.offset, self.tokens, self.blocks = key, doc, offset, tokens, blocks
        self.pins, self.in_map = 0, True


class CacheModel:
    def __init__(self, num_blocks, policy):
        self.policy = policy
        self.free = list(range(num_blocks - 1, -1, -1))  # pop() hands out the lowest id first
        self.map = {}
        self.lru = OrderedDict()  # id(entry) -> entry, least recently used first
        self.tickets = {}
        self.next_ticket = 1
        self.st = dict(hit_blocks=0, miss_blocks=0, evicted_blocks=0, rejected=0, resident_blocks=0,
                       peak_resident_blocks=0)

    def _key(self, doc, offset, prefix):
        if self.policy == AGNOSTIC:
            return doc
        if self.policy == AWARE:
            return (doc, offset)
        return prefix

    def _serves(self, e, doc, ln, offset):
        if self.policy == PREFIX:
            return e.tokens == ln
        return e.doc == doc and e.tokens >= ln and (self.policy == AGNOSTIC or e.offset == offset)

    def _free_blocks(self, e):
        self.free.extend(e.blocks)
        self.st["resident_blocks"] -= len(e.blocks)
        self.st["evicted_blocks"] += len(e.blocks)
        e.blocks = []

    def _evict(self, e):
        self._free_blocks(e)
        del self.lru[id(e)]
        del self.map[e.key]

    def _unpin(self, e):
        e.pins -= 1
        if e.pins == 0 and not e.in_map:
            self._free_blocks(e)

    def admit(self, segs, pos0=0):
        """Returns (ticket, [block ids per segment], [hit flags]) or None when refused."""
        plan, new_keys, new_blocks, pinned = [], {}, 0, []
        offset, prefix = pos0, (pos0,)
        for i, (doc, ln) in enumerate(segs):
            prefix = prefix + ((doc, ln),)
            k = self._key(doc, offset, prefix)
            hit, first = None, -1
            j = new_keys.get(k)
            if self.policy != PREFIX and j is not None and ln <= segs[j][1] and doc == segs[j][0]:
                first = j
            else:
                e = self.map.get(k)
                if e is not None and self._serves(e, doc, ln, offset):
                    hit = e
                    e.pins += 1
                    pinned.append(e)
                else:
                    new_keys[k] = i
                    new_blocks += nblocks(ln)
            plan.append((k, offset, hit, first))
            offset += ln
        if len(self.free) < new_blocks:
            avail = len(self.free) + sum(len(e.blocks) for e in self.lru.values() if e.pins == 0)
            if avail < new_blocks:
                for e in pinned:
                    self._unpin(e)
                self.st["rejected"] += 1
                return None
        for e in list(self.lru.values()):
            if len(self.free) >= new_blocks:
                break
            if e.pins == 0:
                self._evict(e)
        made = [None] * len(segs)
        for i, (k, off, hit, first) in enumerate(plan):
            if hit is not None or first >= 0:
                continue
            old = self.map.get(k)
            if old is not None:
                if old.pins == 0:
                    self._evict(old)
                else:
                    old.in_map = False
                    del self.lru[id(old)]
                    del self.map[k]
            doc, ln = segs[i]
            e = _Entry(k, doc, off, ln, [self.free.pop() for _ in range(nblocks(ln))])
            self.st["resident_blocks"] += len(e.blocks)
            self.st["peak_resident_blocks"] = max(self.st["peak_resident_blocks"], self.st["resident_blocks"])
            self.lru[id(e)] = e
            self.map[k] = e
            e.pins = 1
            pinned.append(e)
            made[i] = e
        out, flags = [], []
        for i, (k, off, hit, first) in enumerate(plan):
            e = hit if hit is not None else (made[first] if first >= 0 else made[i])
            if first >= 0:
                e.pins += 1
                pinned.append(e)
            nb = nblocks(segs[i][1])
            out.append(list(e.blocks[:nb]))
            is_hit = hit is not None or first >= 0
            flags.append(int(is_hit))
            self.st["hit_blocks" if is_hit else "miss_blocks"] += nb
            if e.in_map:
                self.lru.move_to_end(id(e))
        t = self.next_ticket
        self.next_ticket += 1
        self.tickets[t] = pinned
        return t, out, flags

    def release(self, t):
        for e in self.tickets.pop(t):
            self._unpin(e)


def simulate(policy, num_blocks, requests, pos0=None, concurrency=1):
    m = CacheModel(num_blocks, policy)
    live = []
    for r, segs in enumerate(requests):
        a = m.admit(segs, pos0[r] if pos0 is not None else 0)
        live.append(a[0] if a else 0)
        if len(live) >= concurrency:
            j = len(live) - concurrency
            if live[j]:
                m.release(live[j])
            live[j] = 0
    for t in live:
        if t:
            m.release(t)
    return m.st
