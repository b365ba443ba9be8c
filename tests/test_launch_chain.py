"""A model of consecutive fused decode launches overlapped by programmatic
dependent launch, checked on CPU under random timings: the protocol itself,
independent of any device tool.

What is modelled, as `csrc/ekv_attn_body.cuh` and the runner do it:
- launches i = 0, 1, ... in one stream, launch i working on layer i mod L,
  each of C CTAs taking one SM of S (one CTA per SM);
- launch i + 1 may place CTAs once every CTA of launch i has triggered or
  exited; CTAs take free SMs in launch order;
- a CTA reads its layer's state (length, page table, pages) first; with
  dependent inputs it then waits for launch i - 1 to complete; it computes;
  before writing its partials it waits for launch i - 1 again; it appends to
  its layer and exits.  A launch completes when all its CTAs exited.
- the trigger: at the first instruction (an earlier placement), or after the
  CTA's own wait for launch i - 1 (the early wait with dependent inputs, else
  the one before the partials).

Checked: whenever a CTA reads its layer's state, the previous launch on that
layer has completed.  The trigger after the wait keeps that for any C <= S;
the trigger at the first instruction breaks it once C < S.
"""
import heapq
import random

import pytest


def simulate(n_launch, L, S, C, dependent, trigger, rng):
    """Returns the number of reads that found their layer's previous writer
    still running."""
    assert C <= S
    free = S
    eligible = 1                       # launches 0 .. eligible-1 may place CTAs
    placed = [0] * n_launch
    exited = [0] * n_launch
    triggered = [0] * n_launch
    done_at = [None] * n_launch
    events = []                        # (time, seq, kind, launch)
    seq = [0]
    waiting = {}                       # launch -> list of (kind, launch) resumed when launch-1 completes
    bad = [0]

    def push(t, kind, i):
        seq[0] += 1
        heapq.heappush(events, (t, seq[0], kind, i))

    def complete(i):
        return done_at[i] is not None

    def prev_same_layer_done(i):
        j = i - L
        return j < 0 or complete(j)

    def do_trigger(i):
        nonlocal eligible
        triggered[i] += 1
        if triggered[i] == C and eligible == i + 1 and i + 1 < n_launch:
            eligible = i + 2

    def wait_prev(i, t, then):
        if i == 0 or complete(i - 1):
            push(t, then, i)
        else:
            waiting.setdefault(i - 1, []).append((then, i))

    def place(t):
        nonlocal free
        for i in range(eligible):
            while placed[i] < C and free > 0:
                placed[i] += 1
                free -= 1
                push(t, "start", i)

    t = 0.0
    place(t)
    while events:
        t, _, kind, i = heapq.heappop(events)
        if kind == "start":
            if trigger == "first":
                do_trigger(i)
            if not prev_same_layer_done(i):      # the prologue reads the layer's state
                bad[0] += 1
            push(t + rng.uniform(0.5, 3.0), "prologue_done", i)
        elif kind == "prologue_done":
            if dependent:
                wait_prev(i, t, "early_wait_done")
            else:
                push(t, "early_wait_done", i)
        elif kind == "early_wait_done":
            if trigger == "after_wait" and dependent:
                do_trigger(i)
            push(t + rng.uniform(20.0, 40.0), "loop_done", i)
        elif kind == "loop_done":
            wait_prev(i, t, "epilogue_wait_done")
        elif kind == "epilogue_wait_done":
            if trigger == "after_wait" and not dependent:
                do_trigger(i)
            push(t + rng.uniform(0.5, 4.0), "exit", i)
        elif kind == "exit":
            exited[i] += 1
            free += 1
            if exited[i] == C:
                done_at[i] = t
                for then, j in waiting.pop(i, []):
                    push(t, then, j)
        place(t)
    assert triggered == [C] * n_launch   # every CTA triggers before it exits
    assert all(d is not None for d in done_at)
    return bad[0]


@pytest.mark.parametrize("C", [152, 144, 100, 40])
@pytest.mark.parametrize("dependent", [True, False])
@pytest.mark.parametrize("L", [2, 3])
def test_trigger_after_wait_keeps_layer_state_complete(C, dependent, L):
    for seed in range(30):
        assert simulate(24, L, 152, C, dependent, "after_wait", random.Random(seed)) == 0


def test_trigger_at_start_is_safe_only_with_every_sm_taken():
    for dependent in (True, False):
        for seed in range(30):
            assert simulate(24, 2, 152, 152, dependent, "first", random.Random(seed)) == 0
    races = sum(simulate(24, 2, 152, C, True, "first", random.Random(seed))
                for C in (144, 100, 40) for seed in range(30))
    assert races > 0
