"""Host model of a reference-counted block pool with copy-on-write (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Written from the behaviour that [vLLM-TGI] "Inside vLLM and TGI: Paging,
Versioned Schedulers and Operations", section "Exact CPU block manager and
copy-on-write", specifies, and from the sharing paragraph of [VM-LLM] "vLLM
and PagedAttention: Virtual Memory for LLM Serving":

* the pool is a uniform set of blocks of width b with a free list;
* admitting a request takes ceil(len / b) blocks at once, or fails with
  MemoryError and takes nothing;
* forking copies the parent's table and adds one reference to each block;
* appending writes into the last block when it has room and nobody else
  holds it; when the last block is full a fresh block is taken; when it is
  partial and shared, a fresh block is taken, the shared block's contents
  are copied into it, the old block loses one reference and the table is
  repointed (copy-on-write); if a fresh block is needed and none is free the
  append fails with MemoryError and changes nothing;
* releasing drops one reference from every block of the table; a block
  whose count reaches zero returns to the free list;
* invariants: each block's count equals the number of table entries naming
  it, the free list has no duplicates and is exactly the set of blocks with
  count zero, every block but the last of a table is full, and the last
  holds between 1 and b entries.

Free-list order is a policy the pages leave open (one page pops from the
end, the other from the front).  This model fixes one order so that a second
implementation can be compared entry by entry: blocks are taken from the
front of the list, the initial list is the caller's ``free_order`` (default
0..N-1), and a freed block is put back at the front, so the most recently
freed block is reused first.

Each block stores the token payloads written into it, so ``read`` returns a
sequence's tokens in logical order through its table, as the worked example
of [vLLM-TGI] does.
"""

from collections import Counter, deque, namedtuple

from .paging import blocks_needed

AppendResult = namedtuple("AppendResult", "slot copy grew")
AppendResult.__doc__ = """Outcome of one append.

slot  flat physical slot (block * b + offset) the token was written to
copy  (src, dst) block pair that must be copied before the write, or None
grew  True when the table gained an entry because its last block was full
"""


class BlockPool:
    """Reference-counted pool of ``num_blocks`` blocks of ``width`` slots."""

    def __init__(self, num_blocks, width, free_order=None, auto_verify=True):
        if not isinstance(num_blocks, int) or not isinstance(width, int):
            raise ValueError("pool size and block width must be integers")
        if num_blocks < 1 or width < 1:
            raise ValueError("pool size and block width must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of 0..num_blocks-1")
        self.width = width
        self.num_blocks = num_blocks
        self.refcount = [0] * num_blocks
        self.payload = [[] for _ in range(num_blocks)]
        self.free = deque(order)
        self.tables = {}
        # Large pools may skip the O(N) invariant check after every operation
        # and call verify() once at the end instead.
        self.auto_verify = auto_verify

    # -- block-level helpers ------------------------------------------------
    def _take(self):
        blk = self.free.popleft()
        assert self.refcount[blk] == 0
        self.refcount[blk] = 1
        self.payload[blk] = []
        return blk

    def _unref(self, blk):
        self.refcount[blk] -= 1
        if self.refcount[blk] == 0:
            self.payload[blk] = []
            self.free.appendleft(blk)

    # -- sequence operations -----------------------------------------------
    def admit(self, name, tokens):
        """Create a sequence holding ``tokens``; atomic on failure."""
        tokens = list(tokens)
        if name in self.tables or not tokens:
            raise ValueError("sequence exists or has no tokens")
        need = blocks_needed(len(tokens), self.width)
        if need > len(self.free):
            raise MemoryError("pool cannot hold %d more blocks" % need)
        table = []
        for i in range(need):
            blk = self._take()
            self.payload[blk] = tokens[i * self.width:(i + 1) * self.width]
            table.append(blk)
        self.tables[name] = table
        self._check()
        return list(table)

    def fork(self, parent, child):
        """Give ``child`` a copy of ``parent``'s table, sharing every block."""
        if child in self.tables:
            raise ValueError("sequence exists")
        table = list(self.tables[parent])
        for blk in table:
            self.refcount[blk] += 1
        self.tables[child] = table
        self._check()

    def append(self, name, token):
        """Append one token; returns an :data:`AppendResult`."""
        table = self.tables[name]
        last = table[-1]
        fill = len(self.payload[last])
        grow = fill == self.width
        cow = (not grow) and self.refcount[last] > 1
        if (grow or cow) and not self.free:
            raise MemoryError("no free block for growth or copy-on-write")
        pair = None
        if grow:
            table.append(self._take())
        elif cow:
            fresh = self._take()
            self.payload[fresh] = list(self.payload[last])
            self._unref(last)
            table[-1] = fresh
            pair = (last, fresh)
        tail = table[-1]
        slot = tail * self.width + len(self.payload[tail])
        self.payload[tail].append(token)
        self._check()
        return AppendResult(slot, pair, grow)

    def release(self, name):
        for blk in self.tables.pop(name):
            self._unref(blk)
        self._check()

    # -- queries -----------------------------------------------------------
    def read(self, name):
        """Tokens of ``name`` in logical order, read through its table."""
        return [tok for blk in self.tables[name] for tok in self.payload[blk]]

    def length(self, name):
        return sum(len(self.payload[blk]) for blk in self.tables[name])

    def table(self, name):
        return list(self.tables[name])

    def num_free(self):
        return len(self.free)

    def _check(self):
        if self.auto_verify:
            self.verify()

    def verify(self):
        """Check the structural invariants; raises AssertionError if broken."""
        held = Counter(blk for tbl in self.tables.values() for blk in tbl)
        for blk in range(self.num_blocks):
            assert self.refcount[blk] == held.get(blk, 0), "refcount of block %d" % blk
        assert len(set(self.free)) == len(self.free), "duplicate free entry"
        assert set(self.free) == {b for b in range(self.num_blocks) if self.refcount[b] == 0}
        for tbl in self.tables.values():
            for blk in tbl[:-1]:
                assert len(self.payload[blk]) == self.width, "non-last block not full"
            assert 1 <= len(self.payload[tbl[-1]]) <= self.width, "last block fill"
