"""Host block manager model (test infrastructure only).

Follows the block manager of [KV-CB] section 三 (the Rust core modules):
fixed 16-token blocks, a per-request block table mapping logical to physical
block ids, a pool of free physical block ids, and a reference count per block
for shared prefixes; plus copy-on-write for shared blocks ([LLM-INF] 2.2,
[KV-CB] 4.2).  The sketch on the page is prior art, not a specification; the
readings taken where it is incomplete or wrong:

* free list discipline is FIFO: allocation takes from the front, release
  appends to the back, a table is released in logical order;
* allocation is all-or-nothing: when too few blocks are free the state is
  left unchanged and an out-of-memory error is raised;
* release decrements the refcount and returns the block to the free list only
  when it reaches 0 (the page's version drops shared blocks on the floor);
* append returns the slot (block * 16 + row), not the block id;
* fork(parent, child) gives the child the parent's table, refcount + 1 on
  every block (the page documents sharing but has no call for it);
* append into a partially filled block whose refcount is > 1 first moves the
  sequence to a fresh block and reports the (src, dst) pair to copy;
* block payloads are never zeroed (unwritten rows are never read).
"""
from collections import deque

BLOCK_SIZE = 16


class AllocError(Exception):
    pass


class OutOfBlocks(AllocError):
    pass


class UnknownSeq(AllocError):
    pass


class InvalidOp(AllocError):
    pass


def blocks_for(n_tokens):
    """ceil(n / 16): blocks needed for n tokens ([KV-CB] 三, allocate)."""
    return (n_tokens + BLOCK_SIZE - 1) // BLOCK_SIZE


class BlockAllocator:
    def __init__(self, num_blocks, free_order=None):
        if num_blocks <= 0:
            raise InvalidOp("num_blocks must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise InvalidOp("free_order must be a permutation of the pool")
        self.total = num_blocks
        self.free = deque(order)
        self.refcount = [0] * num_blocks
        self.tables = {}
        self.ntokens = {}

    # -- queries -------------------------------------------------------------
    def table(self, seq):
        if seq not in self.tables:
            raise UnknownSeq(seq)
        return list(self.tables[seq]), self.ntokens[seq]

    def utilization(self):
        """(total - free) / total ([KV-CB] 三, utilisation)."""
        return (self.total - len(self.free)) / self.total

    # -- mutations -----------------------------------------------------------
    def _take(self):
        blk = self.free.popleft()
        self.refcount[blk] = 1
        return blk

    def alloc_seq(self, seq, n_tokens):
        if seq in self.tables:
            raise InvalidOp("sequence already exists")
        if n_tokens < 0:
            raise InvalidOp("negative token count")
        need = blocks_for(n_tokens)
        if need > len(self.free):
            raise OutOfBlocks(f"need {need} blocks, {len(self.free)} free")
        self.tables[seq] = [self._take() for _ in range(need)]
        self.ntokens[seq] = n_tokens

    def _append_need(self, seq, rc):
        """Blocks one append of seq would take, given refcounts rc (mutated)."""
        tab, n = self.tables[seq], self.ntokens[seq]
        if n < len(tab) * BLOCK_SIZE:
            last = tab[-1]
            if rc[last] > 1:
                rc[last] -= 1
                return 1
            return 0
        return 1

    def append_slot(self, seq):
        """Reserve the next token's slot -> (slot, cow_src, cow_dst)."""
        if seq not in self.tables:
            raise UnknownSeq(seq)
        if self._append_need(seq, list(self.refcount)) > len(self.free):
            raise OutOfBlocks("no free block for append")
        tab, n = self.tables[seq], self.ntokens[seq]
        src = dst = -1
        if n < len(tab) * BLOCK_SIZE:
            last = tab[-1]
            if self.refcount[last] > 1:
                src, dst = last, self._take()
                self.refcount[src] -= 1
                tab[-1] = dst
        else:
            tab.append(self._take())
        slot = tab[n // BLOCK_SIZE] * BLOCK_SIZE + n % BLOCK_SIZE
        self.ntokens[seq] = n + 1
        return slot, src, dst

    def append_slots(self, seqs):
        """All-or-nothing batch append -> list of (slot, cow_src, cow_dst)."""
        if len(set(seqs)) != len(seqs):
            raise InvalidOp("duplicate sequence in a batch append")
        for s in seqs:
            if s not in self.tables:
                raise UnknownSeq(s)
        rc = list(self.refcount)
        need = sum(self._append_need(s, rc) for s in seqs)
        if need > len(self.free):
            raise OutOfBlocks(f"batch append needs {need} blocks, {len(self.free)} free")
        return [self.append_slot(s) for s in seqs]

    def append_tokens(self, seq, n):
        """n successive appends, all or nothing -> (slots, (cow_src, cow_dst))."""
        if seq not in self.tables:
            raise UnknownSeq(seq)
        tab, ntok = self.tables[seq], self.ntokens[seq]
        rc = list(self.refcount)
        need = 0
        cap = len(tab) * BLOCK_SIZE
        if n > 0 and ntok < cap:
            need += self._append_need(seq, rc)
        if ntok + n > cap:
            need += blocks_for(ntok + n - cap)
        if need > len(self.free):
            raise OutOfBlocks(f"append of {n} tokens needs {need} blocks")
        slots, cow = [], (-1, -1)
        for _ in range(n):
            slot, src, dst = self.append_slot(seq)
            slots.append(slot)
            if src >= 0:
                cow = (src, dst)
        return slots, cow

    def fork_seqs(self, parents, children):
        """Forks in order, all or nothing."""
        made = set()
        for p, c in zip(parents, children):
            if p not in self.tables and p not in made:
                raise UnknownSeq(p)
            if c in self.tables or c in made:
                raise InvalidOp("child exists")
            made.add(c)
        for p, c in zip(parents, children):
            self.fork(p, c)

    def free_seqs(self, seqs):
        """Releases in order, all or nothing."""
        if len(set(seqs)) != len(seqs):
            raise InvalidOp("duplicate sequence")
        for s in seqs:
            if s not in self.tables:
                raise UnknownSeq(s)
        for s in seqs:
            self.free_seq(s)

    def reselect(self, seqs, parent_idx):
        """Sequence seqs[i] takes over seqs[parent_idx[i]]'s table: fork every
        parent into a temporary sequence, release the old ones in order, then
        rename.  All or nothing."""
        if len(set(seqs)) != len(seqs):
            raise InvalidOp("duplicate sequence")
        for s in seqs:
            if s not in self.tables:
                raise UnknownSeq(s)
        if any(not 0 <= p < len(seqs) for p in parent_idx):
            raise InvalidOp("parent index out of range")
        tmp = [("reselect", i) for i in range(len(seqs))]
        for i, p in enumerate(parent_idx):
            self.fork(seqs[p], tmp[i])
        for s in seqs:
            self.free_seq(s)
        for i, s in enumerate(seqs):
            self.tables[s] = self.tables.pop(tmp[i])
            self.ntokens[s] = self.ntokens.pop(tmp[i])

    def fork(self, parent, child):
        if parent not in self.tables:
            raise UnknownSeq(parent)
        if child in self.tables:
            raise InvalidOp("child already exists")
        self.tables[child] = list(self.tables[parent])
        self.ntokens[child] = self.ntokens[parent]
        for blk in self.tables[child]:
            self.refcount[blk] += 1

    def free_seq(self, seq):
        if seq not in self.tables:
            raise UnknownSeq(seq)
        for blk in self.tables.pop(seq):
            self.refcount[blk] -= 1
            if self.refcount[blk] == 0:
                self.free.append(blk)
        del self.ntokens[seq]

    # -- invariants (checked by the tests after every operation) -------------
    def check_invariants(self):
        referenced = set()
        count = [0] * self.total
        for seq, tab in self.tables.items():
            assert len(tab) == blocks_for(self.ntokens[seq]), "table length != ceil(n/16)"
            for blk in tab:
                count[blk] += 1
                referenced.add(blk)
        assert count == self.refcount, "refcount != number of tables holding the block"
        assert len(set(self.free)) == len(self.free), "duplicate in free list"
        assert all(self.refcount[b] == 0 for b in self.free), "free block still referenced"
        assert len(self.free) + len(referenced) == self.total, "blocks lost or double counted"
