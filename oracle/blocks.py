"""Host model of a shared block pool with copy-on-write (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it must do comes from [vLLM-TGI] "Inside vLLM and TGI: Paging,
Versioned Schedulers and Operations", section "Exact CPU block manager and
copy-on-write", and the sharing paragraph of [VM-LLM] "vLLM and
PagedAttention: Virtual Memory for LLM Serving": a request is admitted with
all the blocks its tokens need or not at all; a fork shares every block of
its parent; an append that finds its last block full takes a new one, and
one that finds its last block partly filled and shared first moves onto a
private copy of it; a block returns to the free list when no table names it.

How this model keeps that state is its own, and is chosen to be easy to
check rather than fast:

* Physical memory is one flat list of ``num_blocks * width`` slots, indexed
  like the device pool's rows: slot = block * width + offset.  A slot holds
  the token last written there, or nothing.
* A sequence is only a ``length`` and a ``table``.  Its tokens are never
  stored per sequence: reading it gathers slot ``translate(t)`` for every
  position t < length, the paged read itself.
* Everything else is derived when asked for: how many tables name a block
  (its reference count), how full a sequence's last block is
  (``length - (len(table) - 1) * width``), and which blocks are free.
* The one piece of policy that is not derived is the order of the free
  list, which the pages leave open (one pops from the end, the other from
  the front).  It is kept so that a second implementation can be compared
  entry by entry: fresh blocks come from the front; the initial order is the
  caller's ``free_order`` (default 0..N-1); blocks that lose their last
  holder go back to the front in table order, so the last block of a
  released table is reused first.

``verify`` recomputes what the rules imply from scratch instead of
trusting any counter: the free list is exactly the unheld blocks, each table
has ceil(length / width) distinct entries, and a block named by several
tables sits at the same logical index in each with the same number of
valid positions (a write into a shared block without a copy breaks that).
"""

from collections import Counter, deque, namedtuple

from .paging import blocks_needed, translate

AppendResult = namedtuple("AppendResult", "slot copy grew")
AppendResult.__doc__ = """Outcome of one append.

slot  flat physical slot (block * width + offset) the token was written to
copy  (src, dst) block pair that must be copied before the write, or None
grew  True when the table gained an entry because its last block was full
"""

_EMPTY = object()   # a slot nothing has been written to since its block was taken


class BlockPool:
    """``num_blocks`` physical blocks of ``width`` slots shared by sequences."""

    def __init__(self, num_blocks, width, free_order=None, auto_verify=True):
        if not isinstance(num_blocks, int) or not isinstance(width, int):
            raise ValueError("pool size and block width must be integers")
        if num_blocks < 1 or width < 1:
            raise ValueError("pool size and block width must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.width = width
        self.slots = [_EMPTY] * (num_blocks * width)
        self.lengths = {}
        self.tables = {}
        self.free = deque(order)
        # Large pools may skip the full recomputation after every operation
        # and call verify() once at the end instead.
        self.auto_verify = auto_verify

    # -- derived quantities --------------------------------------------------
    def refcounts(self):
        """List over blocks: how many table entries name each block."""
        counts = [0] * self.num_blocks
        for table in self.tables.values():
            for blk in table:
                counts[blk] += 1
        return counts

    def holders_of_tail(self, blk):
        """How many tables end in ``blk``.  A partly filled block can only be
        the last entry of any table naming it, so for such a block this is
        its reference count."""
        return sum(1 for table in self.tables.values() if table[-1] == blk)

    def tail_fill(self, name):
        """Valid positions in the last block of ``name`` (1 .. width)."""
        return self.lengths[name] - (len(self.tables[name]) - 1) * self.width

    def block_contents(self, blk):
        """Tokens written into physical block ``blk`` since it was taken."""
        row = self.slots[blk * self.width:(blk + 1) * self.width]
        return [tok for tok in row if tok is not _EMPTY]

    # -- physical memory -------------------------------------------------------
    def _fresh_blocks(self, count):
        """Take ``count`` blocks from the front of the free list, blanked."""
        got = [self.free.popleft() for _ in range(count)]
        for blk in got:
            self.slots[blk * self.width:(blk + 1) * self.width] = [_EMPTY] * self.width
        return got

    def _duplicate(self, src, dst):
        """Physical block copy: every slot of ``src`` into ``dst``."""
        w = self.width
        self.slots[dst * w:(dst + 1) * w] = self.slots[src * w:(src + 1) * w]

    def _store(self, name, token):
        """Write ``token`` at position ``length`` of ``name`` through its
        table and extend the sequence by one; returns the slot."""
        slot = translate(self.lengths[name], self.width, self.tables[name])[3]
        self.slots[slot] = token
        self.lengths[name] += 1
        return slot

    # -- sequence operations -----------------------------------------------------
    def admit(self, name, tokens):
        """Create a sequence holding ``tokens``; on failure nothing changes."""
        tokens = list(tokens)
        if name in self.tables:
            raise ValueError("sequence %r exists" % (name,))
        if not tokens:
            raise ValueError("a sequence needs at least one token")
        need = blocks_needed(len(tokens), self.width)
        if need > len(self.free):
            raise MemoryError("%d blocks needed, %d free" % (need, len(self.free)))
        self.tables[name] = self._fresh_blocks(need)
        self.lengths[name] = 0
        for tok in tokens:
            self._store(name, tok)
        self._after()
        return list(self.tables[name])

    def fork(self, parent, child):
        """``child`` starts as ``parent``: same length, same blocks."""
        if child in self.tables:
            raise ValueError("sequence %r exists" % (child,))
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        self._after()

    def append(self, name, token):
        """Add one token at the end of ``name``; returns an AppendResult.

        The position's block is decided first: a new block when the last
        one is full, a private copy when the last one is partly filled and
        other tables also end in it, else the last block itself.  When a
        block is needed and none is free, MemoryError and no change."""
        table = self.tables[name]
        tail = table[-1]
        full = self.tail_fill(name) == self.width
        shared = not full and self.holders_of_tail(tail) > 1
        if (full or shared) and not self.free:
            raise MemoryError("no free block for %s" % ("growth" if full else "a copy"))
        pair = None
        if full:
            table.extend(self._fresh_blocks(1))
        elif shared:
            (mine,) = self._fresh_blocks(1)
            self._duplicate(tail, mine)
            table[-1] = mine
            pair = (tail, mine)
        slot = self._store(name, token)
        self._after()
        return AppendResult(slot, pair, full)

    def release(self, name):
        """Drop ``name``; blocks no other table names become free."""
        table = self.tables.pop(name)
        del self.lengths[name]
        still_held = {blk for other in self.tables.values() for blk in other}
        for blk in table:
            if blk not in still_held:
                self.free.appendleft(blk)
        self._after()

    # -- queries ----------------------------------------------------------------
    def read(self, name):
        """Tokens of ``name`` in logical order, gathered through its table."""
        table = self.tables[name]
        return [self.slots[translate(t, self.width, table)[3]] for t in range(self.lengths[name])]

    def length(self, name):
        return self.lengths[name]

    def table(self, name):
        return list(self.tables[name])

    def num_free(self):
        return len(self.free)

    def _after(self):
        if self.auto_verify:
            self.verify()

    def verify(self):
        """Recompute the pool's invariants; AssertionError if one fails."""
        w = self.width
        named = Counter(blk for table in self.tables.values() for blk in table)
        assert len(self.free) == len(set(self.free)), "a block is listed free twice"
        assert set(self.free) == set(range(self.num_blocks)) - set(named), \
            "free list differs from the blocks no table names"
        where = {}
        for name, table in self.tables.items():
            length = self.lengths[name]
            assert length >= 1, "sequence %r is empty" % (name,)
            assert len(table) == blocks_needed(length, w), "table of %r has a wrong size" % (name,)
            assert len(set(table)) == len(table), "table of %r names a block twice" % (name,)
            for j, blk in enumerate(table):
                valid = min(w, length - j * w)
                seen = where.setdefault(blk, (j, valid))
                assert seen == (j, valid), \
                    "block %d is shared with a different index or fill" % blk
