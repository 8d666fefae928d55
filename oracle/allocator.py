"""Reference block allocator -- TEST INFRASTRUCTURE ONLY.

A plain Python statement of the KV block bookkeeping the pages describe, used
to check the library's native allocator step by step.  It shares no code with
the library.

Rules and their sources:
  * A sequence of len tokens holds exactly ceil(len / B) blocks; nothing is
    reserved ahead ("How PagedAttention changed LLM serving throughput",
    "How PagedAttention fixes it"; "PagedAttention and vLLM, annotated" §3).
  * A new physical block is taken only when the last one is full ("vLLM &
    PagedAttention" §V, steps 1-3).
  * Every physical block carries a reference count; fork shares all of a
    sequence's blocks; a write into a shared (count > 1) last block first
    copies it to a fresh block, repoints the writer and decrements the old
    count, so the last writer writes in place ("vLLM & PagedAttention" §VII,
    Fig. 8; "PagedAttention and vLLM, annotated" §4.4).  Full shared blocks
    are never copied.
  * Freeing a sequence decrements each of its blocks; a block whose count
    reaches zero returns to the pool ("vLLM & PagedAttention" §VII, Fig. 9).
  * fork, append and free are the three sequence primitives ("vLLM &
    PagedAttention" §X).
  * Beam search ("vLLM & PagedAttention" §VII and Fig. 9): one step turns
    the current candidates into the next set.  Every new candidate names its
    parent; the parent's first child continues the parent's sequence, each
    further child forks it; every new candidate then appends its token (a
    write into a shared partly filled block copies that one block); parents
    nobody chose are pruned last, and blocks only they held return to the
    pool.  All or nothing.
  * Swapping ("vLLM & PagedAttention" §VIII and Fig. 4): the blocks of an
    evicted sequence group move to a second (CPU) allocator and back.  A
    group leaves all together or not at all; sequences that share blocks go
    together, so a group must hold every reference to its blocks.  Sharing
    survives the move: each distinct block gets one block in the other pool,
    with the same reference count.

Where the pages are silent (which free block is handed out next), this reads:
the pool hands blocks out in a given initial order; freed blocks are pushed
back in the freed sequence's logical order and are handed out again last-in,
first-out.  An allocation that cannot be met changes nothing.
"""
from __future__ import annotations


class AllocatorOOM(Exception):
    """The pool has too few free blocks; the allocator state is unchanged."""


def blocks_needed(length: int, block_size: int) -> int:
    """ceil(length / block_size): the blocks a sequence of `length` tokens holds."""
    return -(-length // block_size)


class RefAllocator:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad allocator size")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the pool")
        self.B = block_size
        self.num_blocks = num_blocks
        self.ref = [0] * num_blocks
        self._free = list(reversed(order))          # pop() hands out order[0] first
        self._seqs: dict[int, dict] = {}
        self._next_id = 0

    # -- queries -----------------------------------------------------------
    def num_free(self) -> int:
        return len(self._free)

    def block_ref(self, block: int) -> int:
        return self.ref[block]

    def block_table(self, seq: int) -> list[int]:
        return list(self._seqs[seq]["blocks"])

    def seq_len(self, seq: int) -> int:
        return self._seqs[seq]["len"]

    def free_list(self) -> list[int]:
        """Free blocks in the order they would be handed out."""
        return list(reversed(self._free))

    # -- primitives --------------------------------------------------------
    def _pop(self) -> int:
        b = self._free.pop()
        self.ref[b] = 1
        return b

    def seq_new(self, length: int) -> int:
        n = blocks_needed(length, self.B)
        if n > len(self._free):
            raise AllocatorOOM(f"need {n} blocks, {len(self._free)} free")
        blocks = [self._pop() for _ in range(n)]
        sid = self._next_id
        self._next_id += 1
        self._seqs[sid] = {"blocks": blocks, "len": length}
        return sid

    def fork(self, seq: int) -> int:
        parent = self._seqs[seq]
        for b in parent["blocks"]:
            self.ref[b] += 1
        sid = self._next_id
        self._next_id += 1
        self._seqs[sid] = {"blocks": list(parent["blocks"]), "len": parent["len"]}
        return sid

    def append(self, seq: int):
        """Add one token.  Returns (slot, cow) where cow is (src, dst) when the
        shared last block had to be copied first, else None."""
        st = self._seqs[seq]
        pos = st["len"]
        cow = None
        if pos % self.B == 0:                       # last block full, or none yet
            if not self._free:
                raise AllocatorOOM("no free block for a new logical block")
            st["blocks"].append(self._pop())
        else:
            last = st["blocks"][-1]
            if self.ref[last] > 1:                  # shared: copy on write
                if not self._free:
                    raise AllocatorOOM("no free block for copy-on-write")
                fresh = self._pop()
                self.ref[last] -= 1
                st["blocks"][-1] = fresh
                cow = (last, fresh)
        st["len"] = pos + 1
        slot = st["blocks"][pos // self.B] * self.B + pos % self.B
        return slot, cow

    def free(self, seq: int) -> None:
        st = self._seqs.pop(seq)
        for b in st["blocks"]:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self._free.append(b)

    # -- beam search ---------------------------------------------------------
    def beam_step(self, beams, parents):
        """One beam-search step: new candidate i continues beams[parents[i]].
        Returns (new beam ids, slots of their new tokens, copy-on-write
        pairs); raises AllocatorOOM with nothing changed."""
        beams = [int(b) for b in beams]
        parents = [int(p) for p in parents]
        if len(set(beams)) != len(beams) or any(b not in self._seqs for b in beams):
            raise ValueError("unknown or repeated beam")
        if any(p < 0 or p >= len(beams) for p in parents):
            raise ValueError("parent index out of range")
        snapshot = (list(self.ref), list(self._free), self._next_id,
                    {k: {"blocks": list(v["blocks"]), "len": v["len"]} for k, v in self._seqs.items()})
        taken = [False] * len(beams)
        new = []
        for p in parents:
            if not taken[p]:
                taken[p] = True
                new.append(beams[p])
            else:
                new.append(self.fork(beams[p]))
        slots, pairs = [], []
        try:
            for b in new:
                slot, cow = self.append(b)
                slots.append(slot)
                if cow is not None:
                    pairs.append(cow)
        except AllocatorOOM:
            self.ref, self._free, self._next_id, self._seqs = snapshot
            raise
        for i, b in enumerate(beams):
            if not taken[i]:
                self.free(b)
        return new, slots, pairs

    def blocks_in_use(self) -> int:
        return self.num_blocks - len(self._free)

    # -- swapping between pools ---------------------------------------------
    def move_group(self, dst: "RefAllocator", seqs):
        """Move the sequences `seqs` (a group holding every reference to its
        blocks) into `dst`, all or nothing.  Returns (new ids in dst, pairs)
        where pairs lists (block here, block in dst) for every distinct block,
        in first-seen order; the device copies these pairs."""
        seqs = [int(s) for s in seqs]
        if dst.B != self.B:
            raise ValueError("pools of different block sizes")
        if len(set(seqs)) != len(seqs) or any(s not in self._seqs for s in seqs):
            raise ValueError("unknown or repeated sequence")
        uses: dict[int, int] = {}
        order: list[int] = []
        for s in seqs:
            for b in self._seqs[s]["blocks"]:
                if b not in uses:
                    uses[b] = 0
                    order.append(b)
                uses[b] += 1
        if any(self.ref[b] != n for b, n in uses.items()):
            raise ValueError("the group shares blocks with a sequence outside it")
        if len(order) > dst.num_free():
            raise AllocatorOOM(f"need {len(order)} blocks in the other pool, {dst.num_free()} free")
        remap = {}
        for b in order:
            c = dst._pop()
            dst.ref[c] = uses[b]
            remap[b] = c
        new_ids = []
        for s in seqs:
            st = self._seqs[s]
            sid = dst._next_id
            dst._next_id += 1
            dst._seqs[sid] = {"blocks": [remap[b] for b in st["blocks"]], "len": st["len"]}
            new_ids.append(sid)
        for s in seqs:
            self.free(s)
        return new_ids, [(b, remap[b]) for b in order]

    # -- batched step ------------------------------------------------------
    def append_batch(self, seqs):
        """One token for each sequence, in the given order.  All or nothing:
        on OOM every append of this call is undone and AllocatorOOM raised.
        Returns (slots, cow_pairs)."""
        snapshot = (list(self.ref), list(self._free),
                    {k: {"blocks": list(v["blocks"]), "len": v["len"]} for k, v in self._seqs.items()})
        slots, pairs = [], []
        try:
            for s in seqs:
                slot, cow = self.append(s)
                slots.append(slot)
                if cow is not None:
                    pairs.append(cow)
        except AllocatorOOM:
            self.ref, self._free, self._seqs = snapshot
            raise
        return slots, pairs
