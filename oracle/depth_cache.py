"""Slot choice of the bounded depth KV cache, plain Python.

TEST INFRASTRUCTURE, like the rest of ``oracle``: only the tests may import it.

The summary's Sec. 6.2 ("bounded depth KV slot cache") keeps a fixed budget of
S slots, S much smaller than the number of depth entries written, and names
three ways to decide which entries stay:
  * dynamic selection: score the candidate entries by utility, keep the top S;
  * sliding window: keep the most recent entries, evict the older ones;
  * hybrid: part of the slots for the most recent entries, the rest for
    high-scoring ones.
The pages stop there (a future direction with no numbers). The readings taken
here, stated once:
  * an entry is one layer's depth K/V (one slot index for all KV heads and
    positions), and its age is the order in which it was written;
  * an entry's utility is the depth probability mass it received in the most
    recent read of the cache (``Oracle.depth_mass`` summed over KV heads); a
    new entry has not been read yet, so it is always admitted and one of the
    cached entries makes room;
  * ``recent`` = R slots are reserved for the R most recent entries, the new
    one included: R >= S is the sliding window, R <= 1 pure top-S by utility;
  * among the entries that may leave, the one with the least utility leaves;
    equal utilities: the older entry, then the lower slot index;
  * while a slot is empty, the lowest empty slot is filled.
"""
from __future__ import annotations


def victim(ages, utility, recent):
    """Slot that the next entry is written into.

    ages[s]    age of the entry in slot s (its write order), or -1 if empty
    utility[s] its utility (depth mass in the last read); ignored while a
               slot is empty
    recent     R, the number of most recent entries (the new one included)
               that stay regardless of utility
    """
    S = len(ages)
    empty = [s for s in range(S) if ages[s] < 0]
    if empty:
        return min(empty)
    # the R - 1 newest cached entries stay with the new one
    keep = max(0, min(recent, S) - 1)
    newest_first = sorted(range(S), key=lambda s: (-ages[s], s))
    protected = set(newest_first[:keep])
    may_leave = [s for s in range(S) if s not in protected]
    return min(may_leave, key=lambda s: (utility[s], ages[s], s))


def kept_after(ages, utility, recent, new_age):
    """The set of ages the cache holds after writing entry `new_age`, by the
    definition (the R most recent entries, then the highest-utility ones up to
    S), without going through `victim` -- used to check it."""
    S = len(ages)
    held = [(ages[s], utility[s], s) for s in range(S) if ages[s] >= 0]
    if len(held) < S:
        return sorted([a for a, _, _ in held] + [new_age])
    R = max(1, min(recent, S))
    by_age = sorted(held, key=lambda e: (-e[0], e[2]))
    recent_set = [new_age] + [a for a, _, _ in by_age[:R - 1]]
    rest = by_age[R - 1:]
    # of the others, S - R stay: the highest utility, then the younger, then
    # the higher slot index (the mirror of the eviction order)
    rest = sorted(rest, key=lambda e: (-e[1], -e[0], -e[2]))
    return sorted(recent_set + [a for a, _, _ in rest[:S - R]])
