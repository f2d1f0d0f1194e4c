"""Block pool, block tables, fork and copy-on-write (test infrastructure).

Plain Python restatement of the paging scheme on the pages:

* fixed-size physical blocks (16 tokens by default) in one flat pool, and a
  per-sequence table mapping logical block i (tokens 16i .. 16i+15) to a
  physical block id -- "The 8GB VRAM Breakthrough", §3 "How
  Logical-to-Physical Block Tables Work"; "PagedAttention aplica memória
  virtual ao cache KV de LLMs", section "A analogia com memória virtual";
* the pool itself: a stack of free block ids and one reference count per
  block; rent pops a free id, sharing increments the count, giving back
  decrements it and pushes the id once it reaches zero -- "A Ideia de 60
  Anos Que Domou a Memória da GPU", section "o código: a diferença entre
  reservar e mapear".  That listing never sets the count on rent; here a
  rented block starts at one owner (otherwise its first give-back would go
  negative);
* a sequence takes a new block only when its current one is full --
  same page, section "a ideia roubada";
* prefix sharing: a fork points the child's table at the parent's blocks
  and raises their counts; a write into a *partially filled* shared block
  first clones that block (copy-on-write) -- "The 8GB VRAM Breakthrough",
  §3 "Copy-on-Write (CoW) Prefix Sharing"; "A Ideia de 60 Anos...", section
  "o bônus que paga o ingresso: compartilhar".

Appends are all-or-nothing: when the pool cannot supply every block an
append needs, nothing changes and ``OutOfBlocks`` is raised.
"""


class OutOfBlocks(Exception):
    pass


class DoubleFree(Exception):
    pass


class BadSequence(Exception):
    pass


class BlockPool:
    """Free stack + per-block reference counts."""

    def __init__(self, num_blocks, free_order=None):
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        assert sorted(order) == list(range(num_blocks)), "free_order must be a permutation"
        self.num_blocks = num_blocks
        # The stack top is the list's end; reversing makes the first pop
        # return free_order[0], the next free_order[1], and so on.
        self.free = list(reversed(order))
        self.ref = [0] * num_blocks

    def num_free(self):
        return len(self.free)

    def alloc(self):
        if not self.free:
            raise OutOfBlocks()
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def incref(self, b):
        if self.ref[b] <= 0:
            raise DoubleFree(b)
        self.ref[b] += 1

    def decref(self, b):
        if self.ref[b] <= 0:
            raise DoubleFree(b)
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)


class KVCacheManager:
    """Sequences, their block tables and token slots over one ``BlockPool``.

    ``slot = physical_block * block_size + offset_in_block``.
    Sequence ids are handed out as 0, 1, 2, ... in creation order.
    """

    def __init__(self, num_blocks, block_size=16, free_order=None):
        self.pool = BlockPool(num_blocks, free_order)
        self.block_size = block_size
        self.tables = {}
        self.lens = {}
        self._next_id = 0

    # -- sequences -------------------------------------------------------
    def create(self):
        sid = self._next_id
        self._next_id += 1
        self.tables[sid] = []
        self.lens[sid] = 0
        return sid

    def _check(self, sid):
        if sid not in self.tables:
            raise BadSequence(sid)

    def fork(self, parent):
        """Child shares every block of the parent (counts go up by one)."""
        self._check(parent)
        child = self.create()
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.pool.incref(b)
        return child

    def free(self, sid):
        """Give back every block, in logical order."""
        self._check(sid)
        for b in self.tables[sid]:
            self.pool.decref(b)
        del self.tables[sid]
        del self.lens[sid]

    def append(self, sid, n_tokens):
        """Reserve slots for ``n_tokens`` new tokens of sequence ``sid``.

        Returns ``(slots, copies)``: one slot per new token, and the list of
        ``(src, dst)`` block copies the caller must perform before writing
        (at most one: the clone of a shared, partially filled tail block).
        """
        self._check(sid)
        bs = self.block_size
        table = self.tables[sid]
        length = self.lens[sid]
        if n_tokens <= 0:
            return [], []
        cow = length % bs != 0 and self.pool.ref[table[-1]] > 1
        blocks_after = -(-(length + n_tokens) // bs)
        need = (blocks_after - len(table)) + (1 if cow else 0)
        if need > self.pool.num_free():
            raise OutOfBlocks()
        copies = []
        if cow:
            src = table[-1]
            dst = self.pool.alloc()
            self.pool.decref(src)
            table[-1] = dst
            copies.append((src, dst))
        slots = []
        for _ in range(n_tokens):
            if length % bs == 0:
                table.append(self.pool.alloc())
            slots.append(table[length // bs] * bs + length % bs)
            length += 1
        self.lens[sid] = length
        return slots, copies

    # -- views -----------------------------------------------------------
    def length(self, sid):
        self._check(sid)
        return self.lens[sid]

    def table(self, sid):
        self._check(sid)
        return list(self.tables[sid])

    def block_tables(self, sids, max_blocks):
        """Row-major ``[len(sids), max_blocks]`` table, unused entries -1."""
        rows, lens = [], []
        for sid in sids:
            t = self.table(sid)
            if len(t) > max_blocks:
                raise ValueError("sequence needs more than max_blocks blocks")
            rows.append(t + [-1] * (max_blocks - len(t)))
            lens.append(self.lens[sid])
        return rows, lens

    def unique_blocks(self, sids):
        """Distinct physical blocks referenced by the given sequences."""
        s = set()
        for sid in sids:
            s.update(self.tables[sid])
        return len(s)


class PrefixCache:
    """Global cache of computed full blocks over one ``KVCacheManager``.

    "Capítulo 8 — Gerenciamento de KV Cache de Próxima Geração", §8.3: the
    prompt is cut into block-sized chunks; a chunk whose block is already in
    the cache is mapped into the new request's table and its prefill
    skipped; otherwise the prefill runs and the resulting block is
    registered.  A chunk's identity here is the whole token prefix up to and
    including it (the tuple of token ids itself, so equal chunks after
    different prefixes are different entries and nothing can collide).  The
    cache holds one reference on each entry's block.  Eviction (the pages
    give no policy): least recently used first, among entries no other
    entry extends and whose block no sequence holds.
    """

    def __init__(self, manager):
        self.m = manager
        self.entries = {}    # prefix tuple -> [block, last_use]
        self.clock = 0
        self.lookups = 0
        self.hit_blocks = 0
        self._order = {}     # prefix tuple -> creation index (tie-break)
        self._created = 0

    def register(self, sid, tokens):
        """Registers the full blocks of ``sid`` holding ``tokens``; returns
        the number of entries added."""
        bs = self.m.block_size
        tokens = [int(t) for t in tokens]
        if len(tokens) > self.m.length(sid):
            raise ValueError("more tokens than the sequence holds")
        table = self.m.table(sid)
        added = 0
        for i in range(len(tokens) // bs):
            key = tuple(tokens[:(i + 1) * bs])
            if key in self.entries:
                continue
            self.clock += 1
            self.entries[key] = [table[i], self.clock]
            self._order[key] = self._created
            self._created += 1
            self.m.pool.incref(table[i])
            added += 1
        return added

    def match(self, tokens):
        """New sequence whose table is the longest cached chain of full
        blocks matching ``tokens``; returns ``(sid, matched_tokens)``."""
        bs = self.m.block_size
        tokens = [int(t) for t in tokens]
        self.clock += 1
        blocks = []
        for i in range(len(tokens) // bs):
            key = tuple(tokens[:(i + 1) * bs])
            if key not in self.entries:
                break
            self.entries[key][1] = self.clock
            blocks.append(self.entries[key][0])
        sid = self.m.create()
        for b in blocks:
            self.m.pool.incref(b)
        self.m.tables[sid] = blocks
        self.m.lens[sid] = len(blocks) * bs
        self.lookups += 1
        self.hit_blocks += len(blocks)
        return sid, len(blocks) * bs

    def _is_leaf(self, key):
        bs = self.m.block_size
        return not any(len(k) == len(key) + bs and k[:len(key)] == key for k in self.entries)

    def evict(self, n_blocks):
        """Drops up to ``n_blocks`` entries; returns how many were dropped."""
        freed = 0
        while freed < n_blocks:
            cands = [k for k, (b, _) in self.entries.items()
                     if self.m.pool.ref[b] == 1 and self._is_leaf(k)]
            if not cands:
                break
            victim = min(cands, key=lambda k: (self.entries[k][1], self._order[k]))
            b = self.entries.pop(victim)[0]
            del self._order[victim]
            self.m.pool.decref(b)
            freed += 1
        return freed

    def clear(self):
        """Drops every entry, releasing the blocks in registration order."""
        for b, _ in self.entries.values():
            self.m.pool.decref(b)
        self.entries.clear()
        self._order.clear()
