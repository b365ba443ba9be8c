"""A model of the decode-attention kernel's split merge and length publication,
checked on CPU under random completion orders: the protocol itself,
independent of any device tool.

What is modelled, as `csrc/ekv_attn_body.cuh` does it per (sequence, KV head):
- every split's CTA writes its partial (max, sum, numerator) to its own slot,
  then arrives on a ticket; the arrival that finds `expected - 1` is the
  last, merges, and resets the ticket to zero for the next launch;
- up to GROUP splits merge in one level (the last CTA folds every partial
  into O); with more, the last CTA of each group of GROUP merges the group
  into the slot of its first split, and the last group merger merges the
  groups into O;
- with the fused append, the CTA that writes a KV head's O (or the head's
  only CTA when there is one split) arrives on the sequence's length ticket;
  the last of the Hkv arrivals publishes the new length and resets it.

Checked: O of each head is written once, from every split's partial, each
folded exactly once; the new length is published once, after every CTA of
the sequence has read the old one; every ticket is back at zero.
"""
import random

import pytest


def run(splits, hkv, group, rng):
    ticket = {}                        # (head, index) -> count; index 0 = groups
    len_ticket = [0]
    slots = {}                         # (head, slot) -> multiset of splits folded in
    out = {}                           # head -> multiset of splits
    published = []
    read_old = set()

    def arrive(key, expected):
        t = ticket.get(key, 0)
        ticket[key] = t + 1
        last = t == expected - 1
        if last:
            ticket[key] = 0
        return last

    def publish(h):
        t = len_ticket[0]
        len_ticket[0] = t + 1
        if t == hkv - 1:
            assert len(read_old) == hkv * splits, "length published before every CTA read it"
            published.append(h)
            len_ticket[0] = 0

    def cta(h, sp):
        read_old.add((h, sp))          # every CTA reads the old length first
        yield
        slots[(h, sp)] = [sp]          # its partial
        yield
        if splits == 1:
            out[h] = list(slots[(h, sp)])
            publish(h)
            return
        grp, ngrp = sp // group, -(-splits // group)
        gsize = min(group, splits - grp * group)
        if not arrive((h, 1 + grp), gsize):
            return
        yield
        members = range(grp * group, grp * group + gsize)
        if ngrp == 1:
            assert out.get(h) is None, "O written twice"
            out[h] = [s for m in members for s in slots[(h, m)]]
            publish(h)
            return
        folded = [s for m in members for s in slots[(h, m)]]
        slots[(h, grp * group)] = folded   # into the group's first slot
        yield
        if not arrive((h, 0), ngrp):
            return
        yield
        assert out.get(h) is None, "O written twice"
        out[h] = [s for g in range(ngrp) for s in slots[(h, g * group)]]
        publish(h)

    live = [cta(h, sp) for h in range(hkv) for sp in range(splits)]
    while live:
        c = rng.choice(live)
        try:
            next(c)
        except StopIteration:
            live.remove(c)
    for h in range(hkv):
        assert sorted(out[h]) == list(range(splits)), f"head {h} folded {sorted(out[h])}"
    assert len(published) == 1
    assert all(v == 0 for v in ticket.values()) and len_ticket[0] == 0


@pytest.mark.parametrize("splits", [1, 2, 3, 19, 31, 32, 33, 40, 64, 65, 76])
@pytest.mark.parametrize("hkv", [1, 2, 8])
def test_merge_protocol_random_orders(splits, hkv):
    for seed in range(25):
        run(splits, hkv, 32, random.Random(seed))


def test_merge_protocol_small_groups():
    for splits in range(1, 20):
        for seed in range(10):
            run(splits, 2, 4, random.Random(seed))
