"""Host block manager: free list, reference counts, block tables, copy-on-write.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It produces the
addressing (slots, block tables, copy pairs) that the pin tests feed to the
attention oracle; it stores no K/V itself.

Follows [KVS] "19.2 KV Cache 系统化管理":
* §19.2.3 block pool: every block starts free; allocating takes a block off
  the END of the free list and gives it reference count 1; running out is an
  error; releasing decrements the count and returns the block at zero.
* §19.2.3 block table: logical block = tokens so far // block size, slot =
  tokens so far % block size; a new logical block allocates a physical one;
  releasing a request releases every block it maps.
* §19.2.2 Fig 19-8 copy-on-write: a sequence about to write into a block
  whose reference count is above 1 allocates a new block, copies the old
  contents, remaps its table entry and drops one reference on the old block;
  [OS] "LLM 推理引擎的内存管理与调度…" §四 describes the same with shared tail
  blocks and parallel sampling.
"""


class BlockExhausted(RuntimeError):
    """No free physical block is left (the pages' pool raises here too)."""


class BlockPool:
    def __init__(self, num_blocks):
        self.num_blocks = num_blocks
        self.ref_counts = [0] * num_blocks
        self.free_list = list(range(num_blocks))

    def allocate(self):
        if not self.free_list:
            raise BlockExhausted("no free physical block")
        blk = self.free_list.pop()
        self.ref_counts[blk] = 1
        return blk

    def share(self, blk):
        assert self.ref_counts[blk] > 0
        self.ref_counts[blk] += 1

    def release(self, blk):
        assert self.ref_counts[blk] > 0
        self.ref_counts[blk] -= 1
        if self.ref_counts[blk] == 0:
            self.free_list.append(blk)


class BlockTable:
    """One request's logical -> physical block mapping and token count."""

    def __init__(self, pool, block_size):
        self.pool = pool
        self.block_size = block_size
        self.mapping = []
        self.num_filled = 0
        self.copies = []      # (src, dst) pairs this table asked for (CoW)

    def append_slot(self):
        """Reserve the slot of the next token and return its flat slot id
        (physical block * block_size + offset).  Allocates a block when the
        token starts a new logical block; copies-on-write when it lands in a
        block that other tables still share."""
        lb, off = divmod(self.num_filled, self.block_size)
        if lb == len(self.mapping):
            self.mapping.append(self.pool.allocate())
        elif self.pool.ref_counts[self.mapping[lb]] > 1:
            old = self.mapping[lb]
            new = self.pool.allocate()
            self.copies.append((old, new))
            self.mapping[lb] = new
            self.pool.release(old)
        self.num_filled += 1
        return self.mapping[lb] * self.block_size + off

    def fork(self):
        """A new table sharing every block of this one (parallel sampling)."""
        child = BlockTable(self.pool, self.block_size)
        child.mapping = list(self.mapping)
        child.num_filled = self.num_filled
        for blk in self.mapping:
            self.pool.share(blk)
        return child

    def release_all(self):
        for blk in self.mapping:
            self.pool.release(blk)
        self.mapping = []
        self.num_filled = 0
