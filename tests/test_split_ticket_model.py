"""Exhaustive check of the split-K tail's ticket protocol (the GEMM kernel's split_ticket and the
epilogue steps around it), as a model of its atomic steps explored over every interleaving of the
two K halves of a tile.

Each part publishes its raw sums of the other part's column half, then takes a ticket on a word
tagged with the call's epoch.  The second to take it finishes its own half; the first waits a
bounded window for the second (here: it may give up at any point) and, if it gives up first,
claims the word, publishes its other half too and leaves; the second then finishes the whole tile.
The model checks, in every reachable end state: both column halves are finished exactly once,
from sums that were published before they were read; nobody waits for a party that has not taken
its ticket; and the ticket and full words are back to zero (a CUDA-graph replay reuses the epoch).
No GPU is involved.
"""
import pytest

LEFT = 0x100


def _programs(epoch):
    """The steps of part p as generator functions over a shared state dict; a step that cannot
    run yet returns None (blocked), otherwise it returns the next step."""
    E = epoch

    def part(p):
        other = 1 - p
        st = {"role": None}

        def publish_writer(s):
            s["pub"][p].add(other)            # p's raw sums of the other part's column half
            return take_ticket

        def take_ticket(s):
            ep, cnt = s["T"]
            cnt = cnt + 1 if ep == E else 1   # a word of another epoch reads as count 0
            s["T"] = (E, cnt)
            if cnt == 2:
                st["role"] = "normal"
                return finish_own
            if cnt == LEFT + 1:
                s["T"] = (0, 0)
                st["role"] = "alone"
                return wait_full
            assert cnt == 1, cnt
            return first_wait

        def first_wait(s):
            # either the partner's ticket shows up, or the window runs out (both always possible)
            return ("choice", [see_partner, give_up])

        def see_partner(s):
            if s["T"] != (E, 2):
                return None                    # not yet: this branch blocks until it is
            s["T"] = (0, 0)
            st["role"] = "normal"
            return finish_own

        def give_up(s):
            if s["T"] == (E, 1):              # compare-and-swap (E, 1) -> (E, LEFT)
                s["T"] = (E, LEFT)
                st["role"] = "left"
                return publish_rest
            assert s["T"] == (E, 2), s["T"]
            s["T"] = (0, 0)
            st["role"] = "normal"
            return finish_own

        def publish_rest(s):
            s["pub"][p].add(p)                # its own half too
            s["F"] = E
            return done

        def wait_full(s):
            if s["F"] != E:
                return None
            return finish_both

        def finish_own(s):
            half = p                          # part p finishes column half p
            assert half in s["pub"][other], "read sums the other part had not published"
            s["finished"].append(half)
            return done

        def finish_both(s):
            for half in (0, 1):
                assert half in s["pub"][other]
                s["finished"].append(half)
            s["F"] = 0
            return done

        def done(s):
            return "done"

        return publish_writer, st

    return part(0), part(1)


def _explore(initial_T, epoch):
    """Depth-first search over the interleavings; returns the set of reachable end states."""
    (p0, st0), (p1, st1) = _programs(epoch)
    ends = []

    def state_copy(s):
        return {"T": s["T"], "F": s["F"], "pub": [set(s["pub"][0]), set(s["pub"][1])],
                "finished": list(s["finished"])}

    def dfs(s, pcs, depth):
        assert depth < 200, "a step loops without progress"
        if all(pc == "done" for pc in pcs):
            ends.append(s)
            return
        moved = False
        for who in (0, 1):
            pc = pcs[who]
            if pc == "done":
                continue
            s2 = state_copy(s)
            nxt = pc(s2)
            if isinstance(nxt, tuple) and nxt[0] == "choice":
                for alt in nxt[1]:
                    s3 = state_copy(s)
                    r = alt(s3)
                    if r is None:
                        continue
                    moved = True
                    new = list(pcs)
                    new[who] = r
                    dfs(s3, new, depth + 1)
                continue
            if nxt is None:
                continue
            moved = True
            new = list(pcs)
            new[who] = nxt
            dfs(s2, new, depth + 1)
        assert moved, ("deadlock", s, pcs)

    dfs({"T": initial_T, "F": 0, "pub": [set(), set()], "finished": []}, [p0, p1], 0)
    return ends


@pytest.mark.parametrize("initial_T", [(0, 0), (41, 1), (41, 2), (41, LEFT)])
def test_every_interleaving_finishes_each_half_once_and_cleans_up(initial_T):
    """From a zeroed word or one left by an earlier call (another epoch), every interleaving ends
    with both column halves finished exactly once and both words at zero."""
    ends = _explore(initial_T, epoch=7)
    assert ends
    for s in ends:
        assert sorted(s["finished"]) == [0, 1], s
        assert s["T"] == (0, 0) and s["F"] == 0, s


def test_a_replay_with_the_same_epoch_starts_clean():
    """A second call with the same epoch (a CUDA-graph replay) starts from the words the first
    call left, in every end state of the first, and behaves the same."""
    ends = _explore((0, 0), epoch=7)
    for s in ends:
        again = _explore(s["T"], epoch=7)
        assert all(sorted(e["finished"]) == [0, 1] and e["T"] == (0, 0) and e["F"] == 0 for e in again)


def test_count_of_interleavings_covers_the_leave_path():
    """The leave-and-finish-alone path occurs: in some end state one part published both halves
    (it left), and in others neither did (both finished their own half)."""
    ends = _explore((0, 0), epoch=3)
    alone = [s for s in ends if s["pub"][0] == {0, 1} or s["pub"][1] == {0, 1}]
    assert alone, "no interleaving took the leave path"
    assert len(ends) > len(alone)
