"""Pure-Python model of the paged KV block allocator (oracle, test-only).

Behaviour, and where it comes from:

* The KV memory is a pool of fixed-size physical blocks of ``block_size``
  tokens; any free block anywhere can be used ("Visual walkthrough", Step 7;
  "How LLM Inference Serving Works", section "PagedAttention: Virtual Memory
  for the KV Cache").
* Each sequence owns a block table mapping its logical blocks, in order, to
  physical blocks.  A new physical block is taken only when a token is
  appended and the current block is full (position % block_size == 0) --
  "Putting It Together: The Life of a Request in vLLM".
* Sharing: several tables may point at the same physical blocks; each block
  carries a reference count, and a block is copied only when a branch needs to
  write into it (copy-on-write) -- section "Sharing comes for free"; "Visual
  walkthrough", Step 8 (shared prefix).  Forking a sequence copies its table
  and adds one reference to every block; appending into a partly filled last
  block whose count is above one first moves the writer onto a fresh block and
  reports the (source, destination) pair so the caller can copy the block's
  contents.
* When a request ends its blocks' counts drop, and a block whose count reaches
  zero is free again ("Putting It Together").
* When no block is free the request cannot grow; the engine then preempts
  ("When memory runs out anyway").  Here that is an ``OutOfBlocks`` error that
  leaves the allocator exactly as it was.

Readings of what the pages leave open: the free list is first-in first-out,
seeded with the caller's order (default 0..num_blocks-1); blocks freed by a
sequence are appended at its tail in the sequence's logical block order; the
slot of position ``pos`` is table[pos // bs] * bs + pos % bs.
"""
import hashlib
from collections import OrderedDict, deque


class InvalidArg(ValueError):
    """Unknown or duplicate sequence id, or a malformed argument."""


class OutOfBlocks(RuntimeError):
    """The pool has too few free blocks for the request; nothing was changed."""


class BlockAllocatorModel:
    def __init__(self, num_blocks, block_size, initial_free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise InvalidArg("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if initial_free_order is None \
            else [int(x) for x in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise InvalidArg("initial_free_order must be a permutation of the pool")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = deque(order)
        self.ref = [0] * num_blocks
        self.tables = {}
        self.lens = {}

    # -- sequences ---------------------------------------------------------
    def add_seq(self, seq):
        if seq in self.tables:
            raise InvalidArg(f"sequence {seq} exists")
        self.tables[seq] = []
        self.lens[seq] = 0

    def _check(self, seq):
        if seq not in self.tables:
            raise InvalidArg(f"unknown sequence {seq}")

    def _needs_block(self, seq):
        """1 if the next append takes a block (fresh block or copy-on-write)."""
        pos = self.lens[seq]
        if pos % self.block_size == 0:
            return 1
        return 1 if self.ref[self.tables[seq][-1]] > 1 else 0

    def _available(self):
        return len(self.free)

    def _take(self):
        blk = self.free.popleft()
        self.ref[blk] = 1
        return blk

    def _release(self, blk):
        self.ref[blk] -= 1
        if self.ref[blk] == 0:
            self.free.append(blk)

    def _append(self, seq):
        table = self.tables[seq]
        pos = self.lens[seq]
        cow = (-1, -1)
        if pos % self.block_size == 0:
            table.append(self._take())
        elif self.ref[table[-1]] > 1:
            src = table[-1]
            dst = self._take()
            self.ref[src] -= 1
            table[-1] = dst
            cow = (src, dst)
        self.lens[seq] = pos + 1
        slot = table[pos // self.block_size] * self.block_size + pos % self.block_size
        return slot, cow[0], cow[1]

    def append_slot(self, seq):
        """Append one token; returns (slot, cow_src, cow_dst) with -1 for no copy."""
        self._check(seq)
        if self._needs_block(seq) > self._available():
            raise OutOfBlocks("no free block")
        return self._append(seq)

    def append_slots(self, seqs):
        """Append one token to each of ``seqs`` (distinct), all or nothing.

        Returns a list of (slot, cow_src, cow_dst), one per sequence in order.
        """
        seqs = list(seqs)
        if len(set(seqs)) != len(seqs):
            raise InvalidArg("a sequence appears twice in one batch")
        for s in seqs:
            self._check(s)
        need = sum(self._needs_block(s) for s in seqs)
        if need > self._available():
            raise OutOfBlocks("not enough free blocks for the batch")
        return [self._append(s) for s in seqs]

    def reserve(self, seq, num_tokens):
        """Append ``num_tokens`` tokens to one sequence, all or nothing.

        Returns (cow_src, cow_dst) of the copy the first append needed, or
        (-1, -1).
        """
        self._check(seq)
        if num_tokens < 0:
            raise InvalidArg("negative token count")
        if num_tokens == 0:
            return (-1, -1)
        pos = self.lens[seq]
        bs = self.block_size
        fresh = -(-(pos + num_tokens) // bs) - (-(-pos // bs))
        cow = 1 if (pos % bs != 0 and self.ref[self.tables[seq][-1]] > 1) else 0
        if fresh + cow > self._available():
            raise OutOfBlocks("not enough free blocks")
        first = self._append(seq)
        for _ in range(num_tokens - 1):
            self._append(seq)
        return (first[1], first[2])

    def fork(self, parent, child):
        """``child`` starts as a copy of ``parent``, sharing all its blocks."""
        self._check(parent)
        if child in self.tables:
            raise InvalidArg(f"sequence {child} exists")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for blk in self.tables[child]:
            self.ref[blk] += 1

    def free_seq(self, seq):
        """Drop the sequence; blocks whose count reaches zero go to the free tail."""
        self._check(seq)
        for blk in self.tables[seq]:
            self._release(blk)
        del self.tables[seq]
        del self.lens[seq]

    # -- queries -----------------------------------------------------------
    def block_table(self, seq):
        self._check(seq)
        return list(self.tables[seq])

    def seq_len(self, seq):
        self._check(seq)
        return self.lens[seq]

    def refcount(self, blk):
        return self.ref[blk]

    def num_free(self):
        return len(self.free)

    def free_list(self):
        return list(self.free)

    def tail_waste(self, seq):
        """Empty slots in the sequence's last block (Visual walkthrough, Step 7)."""
        self._check(seq)
        return len(self.tables[seq]) * self.block_size - self.lens[seq]


class PrefixCachingAllocatorModel(BlockAllocatorModel):
    """The allocator with automatic prefix caching ("How LLM Inference Serving
    Works", section "Prefix Caching and Chunked Prefill"; "Putting It
    Together": counts drop at the end of a request and the blocks become
    cached-but-evictable).

    * Each full block of a prompt is named by a hash of the tokens in the
      block and of all tokens before it: name_i = H(name_{i-1}, tokens_i).
      The pages do not fix H; the reading used is SHA-256 over the parent's
      32-byte name followed by the block's tokens as little-endian int32, the
      first block's parent being 32 zero bytes or, with a per-request
      cache_salt, SHA-256(salt) ("mixed into the first block's hash").
    * A new prompt reuses the blocks of its longest cached prefix; a block
      matches only if the whole prefix up to it is identical.
    * A named block nobody references is kept, cached-but-evictable, in LRU
      order; fresh blocks come from the free list first, then by evicting the
      least recently used cached block (its name is dropped).
    * Only prompt blocks are named.  A name already held by another block
      keeps that block.
    """

    def __init__(self, num_blocks, block_size, initial_free_order=None):
        super().__init__(num_blocks, block_size, initial_free_order)
        self.by_name = {}
        self.name_of = {}
        self.evictable = OrderedDict()   # least recently used first

    @staticmethod
    def root_name(salt=b""):
        return hashlib.sha256(bytes(salt)).digest() if salt else bytes(32)

    @staticmethod
    def block_name(parent, tokens):
        body = b"".join(int(t).to_bytes(4, "little", signed=True) for t in tokens)
        return hashlib.sha256(bytes(parent) + body).digest()

    def _available(self):
        return len(self.free) + len(self.evictable)

    def _take(self):
        if self.free:
            blk = self.free.popleft()
        else:
            blk, _ = self.evictable.popitem(last=False)
            del self.by_name[self.name_of.pop(blk)]
        self.ref[blk] = 1
        return blk

    def _release(self, blk):
        self.ref[blk] -= 1
        if self.ref[blk] == 0:
            if blk in self.name_of:
                self.evictable[blk] = True
            else:
                self.free.append(blk)

    def add_seq_prompt(self, seq, tokens, salt=b""):
        """Registers ``seq`` with its prompt; returns the number of cached tokens."""
        if seq in self.tables:
            raise InvalidArg(f"sequence {seq} exists")
        tokens = [int(t) for t in tokens]
        bs = self.block_size
        names, parent = [], self.root_name(salt)
        for i in range(len(tokens) // bs):
            parent = self.block_name(parent, tokens[i * bs:(i + 1) * bs])
            names.append(parent)
        hits = 0
        while hits < len(names) and names[hits] in self.by_name:
            hits += 1
        hit_blocks = [self.by_name[n] for n in names[:hits]]
        unreferenced = sum(1 for b in hit_blocks if self.ref[b] == 0)
        need = -(-len(tokens) // bs) - hits
        if need > self._available() - unreferenced:
            raise OutOfBlocks("not enough free or evictable blocks for the prompt")
        self.tables[seq] = []
        for b in hit_blocks:
            if self.ref[b] == 0:
                del self.evictable[b]
            self.ref[b] += 1
            self.tables[seq].append(b)
        self.lens[seq] = hits * bs
        for _ in range(len(tokens) - hits * bs):
            self._append(seq)
        for i in range(hits, len(names)):
            if names[i] in self.by_name:
                continue
            blk = self.tables[seq][i]
            self.by_name[names[i]] = blk
            self.name_of[blk] = names[i]
        return hits * bs

    def evictable_list(self):
        return list(self.evictable)
