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
