"""A model of the attention kernel's mbarrier protocol (csrc/ce_attention.cu),
run under random schedules on the CPU.

Each role of a CTA is a program that yields at every mbarrier wait: the TMA
producer (Q into two buffers, K into a three-stage ring, V into a two-stage
ring, K one tile ahead of V), the MMA thread (scores two tiles ahead of P V,
issued once the softmax holds the buffer's previous scores), and the softmax
warps (scores -> P into one of two P buffers, the output staged through the
item's own Q buffer when it is large enough).  The TMA engine completes loads
in any order; the tensor pipe runs MMAs in issue order and a commit arrives
when everything issued before it has run.  The model checks that no role ever
reads a stale buffer or overwrites one still in use, that no wait falls two
phases behind its barrier, and that every schedule ends (no deadlock).
A second test plants a mistake in the protocol and checks that the model
finds it.  The kernel's barrier counts (threads or warps) appear here as one
arrival per modelled softmax warp.
"""

import random

import pytest


class ProtocolError(AssertionError):
    pass


def check(cond, msg):
    if not cond:
        raise ProtocolError(msg)


class Barrier:
    """An mbarrier: a phase completes after `count` arrivals."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        check(self.pending >= 0, f"{self.name}: more arrivals than its count")
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, n):
        """Has phase n completed?  A parity wait cannot tell phase n from n + 2."""
        check(self.phase in (n, n + 1), f"{self.name}: waiting for phase {n} at {self.phase}")
        return self.phase == n + 1


def work_items(cta, grid, bh_count, T, causal):
    """The (head, query tile) items CTA `cta` of `grid` takes, in order: a work
    unit is one query tile, or under the causal mask the pair (last - u, u)."""
    q_tiles = (T + 127) // 128
    n_pairs = (q_tiles + 1) // 2
    n_units = bh_count * (n_pairs if causal else q_tiles)
    items = []
    for u in range(cta, n_units, grid):
        if not causal:
            items.append((u // q_tiles, u % q_tiles))
            continue
        bh, pr = divmod(u, n_pairs)
        items.append((bh, q_tiles - 1 - pr))
        if q_tiles - 1 - pr != pr:
            items.append((bh, pr))
    return items


def key_tiles(qt, T, causal):
    end = min(T, (qt + 1) * 128) if causal else T
    return (end + 127) // 128


def simulate(rng, bh_count, T, causal, grid, stage_in_q, warps=4, mutation=None):
    for cta in range(grid):
        run_cta(rng, work_items(cta, grid, bh_count, T, causal), T, causal, stage_in_q, warps,
                mutation)


def run_cta(rng, items, T, causal, stage_in_q, W, mutation):
    KS = 3  # K stages
    bar = {"o_free": Barrier("o_free", W)}
    for b in range(2):
        bar[f"q_full{b}"] = Barrier(f"q_full{b}", 1)
        bar[f"q_empty{b}"] = Barrier(f"q_empty{b}", 1 + (W if stage_in_q else 0))
        bar[f"v_full{b}"] = Barrier(f"v_full{b}", 1)
        bar[f"v_empty{b}"] = Barrier(f"v_empty{b}", 1)
        bar[f"s_full{b}"] = Barrier(f"s_full{b}", 1)
        bar[f"s_free{b}"] = Barrier(f"s_free{b}", W)
        bar[f"p_full{b}"] = Barrier(f"p_full{b}", W)
        bar[f"pv_done{b}"] = Barrier(f"pv_done{b}", 1)
    for b in range(KS):
        bar[f"k_full{b}"] = Barrier(f"k_full{b}", 1)
        bar[f"k_empty{b}"] = Barrier(f"k_empty{b}", 1)

    # what each buffer holds: (tile or item, still being written)
    q_buf = [[None, False], [None, False]]
    k_buf = [[None, False] for _ in range(KS)]
    v_buf = [[None, False], [None, False]]
    s_buf = [None, None]          # score buffers: the tile whose scores they hold
    s_readers = [0, 0]
    p_buf = [None, None]          # P buffers: the tile whose weights they hold
    staging = [0, 0]              # epilogue warps reading Q buffer b as staging
    state = {"o_item": None, "o_last": None, "pv_ran": set()}
    tma, pipe = [], []            # the TMA engine (any order) and the tensor pipe (in order)

    def wait(name, n):
        return lambda: bar[name].done(n)

    def producer():
        g = 0
        pending_v = None

        def load_v(t):
            s = t & 1
            if t >= 2 and mutation != "no_v_empty_wait":
                yield wait(f"v_empty{s}", (t >> 1) - 1)
            check(not v_buf[s][1], "V load into a stage still loading")
            v_buf[s][1] = True

            def land():
                v_buf[s][:] = [t, False]
                bar[f"v_full{s}"].arrive()
            tma.append(land)

        for it, (_, qt) in enumerate(items):
            qb = it & 1
            if it >= 2 and mutation != "no_q_release_wait":
                yield wait(f"q_empty{qb}", (it >> 1) - 1)
            check(staging[qb] == 0, "Q load over output staging still being read")
            check(not q_buf[qb][1], "Q load into a buffer still loading")
            q_buf[qb][1] = True

            def land_q(it=it, qb=qb):
                q_buf[qb][:] = [it, False]
                bar[f"q_full{qb}"].arrive()
            tma.append(land_q)
            for _ in range(key_tiles(qt, T, causal)):
                s = g % KS
                if g >= KS and mutation != "no_k_empty_wait":
                    yield wait(f"k_empty{s}", g // KS - 1)
                check(not k_buf[s][1], "K load into a stage still loading")
                k_buf[s][1] = True

                def land_k(s=s, g=g):
                    k_buf[s][:] = [g, False]
                    bar[f"k_full{s}"].arrive()
                tma.append(land_k)
                if pending_v is not None:
                    yield from load_v(pending_v)
                pending_v = g
                g += 1
                yield None
            # the item's last V before the next item's Q (whose buffer may still
            # hold an output being stored)
            yield from load_v(pending_v)
            pending_v = None
        # drain: nothing in flight into shared memory when the CTA ends
        for t in range(max(0, len(items) - 2), len(items)):
            yield wait(f"q_full{t & 1}", t >> 1)
        for t in range(max(0, g - KS), g):
            yield wait(f"k_full{t % KS}", t // KS)
        for t in range(max(0, g - 2), g):
            yield wait(f"v_full{t & 1}", t >> 1)

    def mma():
        g = gp = 0

        def issue_s(gs, it):
            ks, sb = gs % KS, gs & 1
            yield wait(f"k_full{ks}", gs // KS)
            if gs >= 2 and mutation != "no_s_free_wait":
                yield wait(f"s_free{sb}", (gs >> 1) - 1)

            def run():
                check(k_buf[ks] == [gs, False], "score MMA reads a stale K stage")
                check(q_buf[it & 1] == [it, False], "score MMA reads a stale Q buffer")
                check(s_readers[sb] == 0, "score MMA overwrites scores being read")
                s_buf[sb] = gs
            pipe.append(run)
            pipe.append(lambda: bar[f"s_full{sb}"].arrive())
            pipe.append(lambda: bar[f"k_empty{ks}"].arrive())

        def q_release(qb):
            pipe.append(lambda: bar[f"q_empty{qb}"].arrive())

        for it, (_, qt) in enumerate(items):
            n, qb, base = key_tiles(qt, T, causal), it & 1, g
            yield wait(f"q_full{qb}", it >> 1)
            yield from issue_s(base, it)
            if n > 1:
                yield from issue_s(base + 1, it)
            if n <= 2:
                q_release(qb)
            for j in range(n):
                if j + 2 < n:
                    yield from issue_s(base + j + 2, it)
                    if j + 3 == n:
                        q_release(qb)
                if j == 0 and it > 0 and mutation != "no_o_free_wait":
                    yield wait("o_free", it - 1)
                t, b = gp, gp & 1
                yield wait(f"p_full{b}", t >> 1)
                yield wait(f"v_full{b}", t >> 1)

                def run(t=t, b=b, j=j, it=it):
                    check(v_buf[b] == [t, False], "P V reads a stale V stage")
                    check(p_buf[b] == t, "P V reads another tile's P")
                    if j == 0:
                        check(state["o_item"] is None, "P V overwrites O before it was read out")
                    state["o_item"], state["o_last"] = it, t
                    state["pv_ran"].add(t)
                pipe.append(run)
                pipe.append(lambda b=b: bar[f"pv_done{b}"].arrive())
                pipe.append(lambda b=b: bar[f"v_empty{b}"].arrive())
                gp += 1
            g = base + n
        if gp:
            yield wait(f"pv_done{(gp - 1) & 1}", (gp - 1) >> 1)

    def softmax(w):
        g = 0
        for it, (_, qt) in enumerate(items):
            n = key_tiles(qt, T, causal)
            for j in range(n):
                sb = g & 1
                yield wait(f"s_full{sb}", g >> 1)
                check(s_buf[sb] == g, "softmax reads stale scores")
                s_readers[sb] += 1
                yield None
                s_readers[sb] -= 1
                bar[f"s_free{sb}"].arrive()
                if stage_in_q and j == 0 and it > 0:
                    # the previous item's output stores have read its Q buffer
                    bar[f"q_empty{(it - 1) & 1}"].arrive()
                yield None
                if j > 0 and rng.random() < 0.3:
                    # the lazy rescale of O after the previous P V
                    yield wait(f"pv_done{(g - 1) & 1}", (g - 1) >> 1)
                    check(state["o_last"] == g - 1, "O rescaled before the previous P V ran")
                if g >= 2 and mutation != "no_p_buffer_wait":
                    yield wait(f"pv_done{sb}", (g >> 1) - 1)
                check(g < 2 or g - 2 in state["pv_ran"], "P written over weights not yet read")
                p_buf[sb] = g
                yield None
                bar[f"p_full{sb}"].arrive()
                g += 1
            yield wait(f"pv_done{(g - 1) & 1}", (g - 1) >> 1)
            check(state["o_last"] == g - 1, "output read before the item's last P V")
            qb = it & 1
            if stage_in_q:
                check(q_buf[qb] == [it, False], "output staged in a Q buffer being reloaded")
                staging[qb] += 1
            yield None
            if stage_in_q:
                staging[qb] -= 1
            bar["o_free"].arrive()
            if bar["o_free"].pending == W:
                state["o_item"] = None

    roles = [producer(), mma()] + [softmax(w) for w in range(W)]
    blocked = [None] * len(roles)
    finished = [False] * len(roles)
    for _ in range(5_000_000):
        if all(finished):
            break
        ready = [i for i, r in enumerate(roles)
                 if not finished[i] and (blocked[i] is None or blocked[i]())]
        engines = (["tma"] if tma else []) + (["pipe"] if pipe else [])
        if not ready and not engines:
            raise ProtocolError("deadlock: every role waits and nothing is in flight")
        if engines and (not ready or rng.random() < 0.4):
            if rng.choice(engines) == "tma":
                tma.pop(rng.randrange(len(tma)))()
            else:
                pipe.pop(0)()
            continue
        i = rng.choice(ready)
        try:
            blocked[i] = next(roles[i])
        except StopIteration:
            finished[i], blocked[i] = True, None
    else:
        raise ProtocolError("schedule did not end")
    while tma:
        tma.pop(0)()
    while pipe:
        pipe.pop(0)()


def random_case(seed):
    rng = random.Random(seed)
    bh = rng.randint(1, 5)
    T = rng.choice([1, 64, 127, 128, 129, 200, 256, 300, 384, 512, 640, 1000])
    causal = rng.random() < 0.5
    q_tiles = (T + 127) // 128
    n_units = bh * (((q_tiles + 1) // 2) if causal else q_tiles)
    grid = min(rng.randint(1, n_units), 3)
    return rng, bh, T, causal, grid


@pytest.mark.parametrize("stage_in_q", [True, False], ids=["D128_staging_in_Q", "D64_own_staging"])
def test_protocol_under_random_schedules(stage_in_q):
    for seed in range(300):
        rng, bh, T, causal, grid = random_case(seed)
        simulate(rng, bh, T, causal, grid, stage_in_q)


@pytest.mark.parametrize("mutation", ["no_s_free_wait", "no_p_buffer_wait", "no_q_release_wait",
                                      "no_k_empty_wait", "no_v_empty_wait"])
def test_planted_protocol_mistakes_are_found(mutation):
    found = False
    for seed in range(300):
        rng, bh, T, causal, grid = random_case(seed)
        try:
            simulate(rng, bh, T, causal, grid, True, mutation=mutation)
        except ProtocolError:
            found = True
            break
    assert found, f"the model missed the planted mistake {mutation}"


def test_o_free_wait_is_implied_by_the_next_p_full():
    # the MMA thread waits for the previous item's output to be read out of TMEM
    # before the first P V of an item; that P V also waits for every softmax
    # warp's P of the item's first tile, which each warp writes only after its
    # own read-out, so the model finds no schedule where dropping the wait matters
    for seed in range(300):
        rng, bh, T, causal, grid = random_case(seed)
        simulate(rng, bh, T, causal, grid, True, mutation="no_o_free_wait")


# ---------------------------------------------------------------------------
# The swap of a row's two partial values between its two softmax threads
# (csrc/ce_attention.cu, `swap`): two slots per row and one named barrier per
# swap.  At swap k thread h writes slot h ^ (k % 2), meets its partner at the
# barrier, and reads slot h ^ (k % 2) ^ 1: each thread overwrites only the slot
# it read at the previous swap, so no write overtakes the partner's pending
# read.  The model runs the two threads under random schedules; a thread at a
# barrier waits until both have arrived there.
# ---------------------------------------------------------------------------
def run_swaps(rng, n, slot_of):
    slots = [None, None]
    arrived = [0, 0]          # barriers each thread has reached
    pc = [0, 0]               # 0: write, 1: at the barrier, 2: read (per swap)
    k = [0, 0]
    while k[0] < n or k[1] < n:
        ready = [t for t in (0, 1) if k[t] < n and (pc[t] != 1 or arrived[1 - t] > k[t])]
        check(ready, "deadlock")
        t = rng.choice(ready)
        w, r = slot_of(t, k[t])
        if pc[t] == 0:
            slots[w] = (t, k[t])
            arrived[t] += 1
            pc[t] = 1
        elif pc[t] == 1:
            pc[t] = 2
        else:
            check(slots[r] == (1 - t, k[t]),
                  f"thread {t} at swap {k[t]} read {slots[r]} from slot {r}")
            pc[t] = 0
            k[t] += 1


def test_row_swap_with_one_barrier():
    rng = random.Random(7)
    for _ in range(500):
        run_swaps(rng, 12, lambda h, k: (h ^ (k & 1), h ^ (k & 1) ^ 1))


def test_row_swap_planted_mistake_is_found():
    # each thread always writing its own slot needs a second barrier (before
    # the write): with one, a fast thread overwrites a value its partner has
    # not read yet
    rng = random.Random(7)
    with pytest.raises(ProtocolError):
        for _ in range(500):
            run_swaps(rng, 12, lambda h, k: (h, h ^ 1))
