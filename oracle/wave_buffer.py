"""Wave buffer block-cache policy, stated plainly -- TEST INFRASTRUCTURE ONLY.

Sources (the RetroInfer technical summaries; "de", "fr", "zh" name the
gist.science pages of arXiv 2505.02922):
  * a block cache of KV blocks on the GPU, for the temporal locality of the
    tokens attention retrieves from one decode step to the next (de 2.B
    "Block Cache", fr 2.B "Block Cache GPU", zh 2.B "KV Block Cache");
  * replacement is LRU, run by the CPU asynchronously while the GPU computes;
    cache access and cache update are decoupled (zh 2.B; de 2.B
    "Asynchronität"; fr 2.B "Gestion Asynchrone");
  * an execution buffer gathers the tokens attention needs -- from the steady
    zone, the cache and the CPU -- into contiguous GPU memory (de 2.B
    "Execution Buffer", zh 2.B).

READINGS (the pages give no block size, admission rule or eviction detail):
  * a block ("page") is `page_rows` consecutive rows of one unit's K/V in the
    index's cluster-contiguous order, so a retrieved cluster covers one or a
    few pages; every unit has its own cache of `slots` pages;
  * one replacement round per observed decode step, over the pages that step
    touched, in increasing page order: a cached page becomes the most recently
    used; a page not cached is admitted (at most `admit_max` per round and
    unit) into the lowest free slot, else into the slot of the least recently
    used page, unless that page was touched in this same round -- then every
    cached page was, and the round admits nothing more; an admitted page is
    the most recently used;
  * a page admitted in round t serves the steps after the round's copy lands;
    until then, and for every page not cached, the rows are read from host
    memory.  Where a row is read from does not change the attention output.
"""
from __future__ import annotations

from collections import OrderedDict


class LruPagePolicy:
    """The replacement rounds of one unit's page cache (readings above)."""

    def __init__(self, pages: int, slots: int, admit_max: int):
        if pages < 1 or slots < 0 or admit_max < 0:
            raise ValueError("pages >= 1, slots >= 0, admit_max >= 0")
        self.pages, self.slots, self.admit_max = pages, slots, admit_max
        self.slot_of = {}             # page -> slot
        self.lru = OrderedDict()      # page -> round last touched; first = least recently used
        self.free = list(range(slots))

    def round(self, touched, t):
        """One round for the pages touched at step t.  Returns (evicted, admitted): lists of
        (page, slot) pairs, in the order the round made them."""
        evicted, admitted = [], []
        n_admit = 0
        for p in sorted(set(int(x) for x in touched)):
            if not 0 <= p < self.pages:
                raise ValueError(f"page {p} outside [0, {self.pages})")
            if p in self.slot_of:         # hit: most recently used
                self.lru.move_to_end(p)
                self.lru[p] = t
                continue
            if n_admit >= self.admit_max:
                continue
            if self.free:
                s = min(self.free)
                self.free.remove(s)
            else:
                if not self.lru:
                    continue              # no slots at all
                victim, last = next(iter(self.lru.items()))
                if last == t:             # every cached page was touched in this round
                    continue
                del self.lru[victim]
                s = self.slot_of.pop(victim)
                evicted.append((victim, s))
            self.slot_of[p] = s
            self.lru[p] = t
            admitted.append((p, s))
            n_admit += 1
        return evicted, admitted


def pages_of_rows(row0: int, rows: int, page_rows: int):
    """The pages rows [row0, row0 + rows) fall in (a retrieved cluster's run), in order."""
    if rows <= 0:
        return []
    return list(range(row0 // page_rows, (row0 + rows - 1) // page_rows + 1))
