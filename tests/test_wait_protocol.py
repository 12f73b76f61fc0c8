"""CPU models of the two hand-off protocols of the streaming kernel, run under
random interleavings, with the bounded waits and the failure paths.

1. The chunk ring between converter and compute warps.  Slot c % NSLOT holds
   chunk c.  Two mbarriers per slot: ``full`` (one arrival per converter
   thread) and ``empty`` (one arrival per compute warp that reads the slot).
   A converter thread waits on empty with parity ((c / NSLOT) + 1) & 1 before
   it writes chunk c (c >= NSLOT), then arrives on full; a reader waits on full
   with parity (c / NSLOT) & 1, reads, and arrives on empty when a converter
   will wait for it (c + NSLOT < nchunks).  An mbarrier is modelled by its
   pending count and phase: try_wait(parity) succeeds once the phase of that
   parity has completed, i.e. when (phase & 1) != parity.

2. The split-K exchange between the CTAs of a tile, across launches.  The
   tile's arrival word holds an epoch above ARRIVAL_BITS and an arrival count
   below; every CTA draws once; the CTA that draws last polls its peers'
   flagged words (flag = epoch | 2^31) and sums them in split order, clears
   them and moves the word to the next epoch; a CTA whose own waits ran out
   stores nothing and, if it drew last, still moves the word on.  Polls are
   bounded and an expiry sets the timeout status; the host then resets the
   words.

Each model is run clean (every run must finish, with the right data and no
expiry), with a stalled hand-off (every run must end, by expiry, with the
status set) and with planted mistakes in the model itself (a wrong parity, a
missing arrival, an epoch that does not move on), which the checks must catch."""
import random

import pytest

ARRIVAL_BITS = 10


class MBar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def try_wait(self, parity):
        return (self.phase & 1) != parity


class Violation(Exception):
    pass


def run_ring(nslot, nchunks, conv_threads, readers, seed, limit=400, stall_at=None, mistake=None):
    """One CTA's ring under a random schedule.  Returns (timed_out, steps).
    Raises Violation when a reader sees the wrong chunk or a converter
    overwrites a slot that is still being read."""
    rng = random.Random(seed)
    full = [MBar(conv_threads) for _ in range(nslot)]
    empty = [MBar(readers - (1 if mistake == "empty_count" else 0)) for _ in range(nslot)]
    parts = [[None] * conv_threads for _ in range(nslot)]  # chunk id each converter part holds
    reading = [0] * nslot  # readers inside a read of the slot
    done_reads = [0] * nchunks
    err = {"flag": False}

    def wait(bar, parity):
        polls = 0
        while not bar.try_wait(parity):
            if err["flag"] or polls >= limit:
                err["flag"] = True
                return False
            polls += 1
            yield
        return True

    def converter(t):
        for c in range(nchunks):
            if stall_at is not None and c >= stall_at:
                return
            s = c % nslot
            if c >= nslot:
                parity = ((c // nslot) + 1) & 1
                if mistake == "conv_parity":
                    parity ^= 1
                ok = yield from wait(empty[s], parity)
                if not ok:
                    return
                if reading[s] or done_reads[c - nslot] < readers:
                    raise Violation("chunk %d overwrites slot %d while chunk %d is read" % (c, s, c - nslot))
            parts[s][t] = c
            yield
            full[s].arrive()
            yield

    def reader(r):
        for c in range(nchunks):
            s = c % nslot
            parity = (c // nslot) & 1
            if mistake == "reader_parity":
                parity ^= 1
            ok = yield from wait(full[s], parity)
            if not ok:
                return
            reading[s] += 1
            for _ in range(rng.randint(0, 2)):
                yield
            if any(p != c for p in parts[s]):
                raise Violation("reader %d sees %r for chunk %d" % (r, parts[s], c))
            reading[s] -= 1
            done_reads[c] += 1
            arrive = c + nslot < nchunks
            if mistake == "missing_arrival":
                arrive = c + nslot < nchunks - 1
            if arrive:
                empty[s].arrive()
            yield

    agents = [converter(t) for t in range(conv_threads)] + [reader(r) for r in range(readers)]
    steps = 0
    while agents:
        a = rng.choice(agents)
        try:
            next(a)
        except StopIteration:
            agents.remove(a)
        steps += 1
        assert steps < 10_000_000
    return err["flag"], steps


RING_SHAPES = [
    # (NSLOT, chunks, converter threads, reading warps): the plain ring (4
    # slots), one row group per warp (2 slots), row-group CTAs (4 slots, half
    # the warps read each chunk), and a ring of one lap or less
    (4, 11, 3, 4),
    (2, 9, 2, 3),
    (4, 16, 2, 8),
    (4, 3, 2, 2),
    (2, 1, 1, 2),
]


@pytest.mark.parametrize("shape", RING_SHAPES)
def test_ring_clean_runs(shape):
    nslot, nchunks, conv, readers = shape
    for seed in range(60):
        timed_out, _ = run_ring(nslot, nchunks, conv, readers, seed)
        assert not timed_out, (shape, seed)


@pytest.mark.parametrize("shape", RING_SHAPES)
def test_ring_stalled_converters_time_out_and_end(shape):
    nslot, nchunks, conv, readers = shape
    for seed in range(20):
        for stall_at in (0, nchunks // 2):
            timed_out, _ = run_ring(nslot, nchunks, conv, readers, seed, stall_at=stall_at)
            assert timed_out, (shape, seed, stall_at)


@pytest.mark.parametrize("mistake", ["conv_parity", "reader_parity", "empty_count", "missing_arrival"])
def test_ring_planted_mistakes_are_caught(mistake):
    caught = 0
    for seed in range(60):
        try:
            timed_out, _ = run_ring(4, 11, 3, 4, seed, mistake=mistake)
        except Violation:
            caught += 1
            continue
        if timed_out:
            caught += 1
    assert caught > 0, mistake


# ---------------------------------------------------------------------------
# split-K exchange across launches


class Tile:
    """Device state of one tile: its arrival word and [splits] flagged words."""

    def __init__(self, splits):
        self.counter = 0
        self.words = [0] * splits
        self.status = 0
        self.y = None

    def host_reset(self):
        # what the status read does after an expiry, on an idle device
        self.counter = 0
        self.words = [0] * len(self.words)


def run_launch(tile, values, seed, fail=(), stall=False, poll_limit=50, mistake=None):
    """One launch of len(values) CTAs over the tile; `fail` lists the splits
    whose own waits ran out.  Writes tile.y (or leaves it) and tile.status."""
    rng = random.Random(seed)
    S = len(values)
    tile.y = None

    def cta(split):
        yield
        w = tile.counter
        tile.counter += 1  # atomicAdd
        last = (w & ((1 << ARRIVAL_BITS) - 1)) == S - 1
        nxt = ((w >> ARRIVAL_BITS) + 1) << ARRIVAL_BITS
        yield
        if split in fail:
            tile.status = 1
            if last and mistake != "failed_last_keeps_epoch":
                tile.counter = nxt
            return
        flag = (w >> ARRIVAL_BITS) | 0x80000000
        if not last:
            if stall:
                return
            tile.words[split] = (flag, values[split])
            return
        polls = 0
        while True:
            ready = all(tile.words[j] != 0 and tile.words[j][0] == flag for j in range(S) if j != split)
            if ready or polls >= poll_limit:
                break
            polls += 1
            yield
        total = 0
        for j in range(S):
            if j == split:
                total += values[j]
            else:
                word = tile.words[j]
                total += word[1] if word != 0 else 0
                tile.words[j] = 0
        if polls >= poll_limit:
            tile.status = 1
        tile.counter = nxt
        tile.y = total

    agents = [cta(s) for s in range(S)]
    while agents:
        a = rng.choice(agents)
        try:
            next(a)
        except StopIteration:
            agents.remove(a)


@pytest.mark.parametrize("splits", [2, 5, 19])
def test_split_exchange_clean_launches(splits):
    tile = Tile(splits)
    rng = random.Random(splits)
    for launch in range(200):
        values = [rng.randint(-1000, 1000) for _ in range(splits)]
        run_launch(tile, values, seed=launch)
        assert tile.status == 0 and tile.y == sum(values), launch
        assert tile.words == [0] * splits


@pytest.mark.parametrize("splits", [2, 5, 19])
def test_split_exchange_failures_then_recovery(splits):
    rng = random.Random(100 + splits)
    for launch in range(200):
        tile = Tile(splits)
        # a few clean launches move the epoch on first
        for k in range(rng.randint(0, 3)):
            run_launch(tile, [1] * splits, seed=launch * 7 + k)
        kind = launch % 3
        values = [rng.randint(-1000, 1000) for _ in range(splits)]
        if kind == 0:
            run_launch(tile, values, seed=launch, stall=True)
        elif kind == 1:
            run_launch(tile, values, seed=launch, fail={rng.randrange(splits)})
        else:
            run_launch(tile, values, seed=launch, fail=set(range(splits)))
        assert tile.status == 1, (launch, kind)
        # without the host's reset, and with it, the next launches are right
        for reset in (False, True):
            probe = Tile(splits)
            probe.counter, probe.words = tile.counter, list(tile.words)
            if reset:
                probe.host_reset()
            for k in range(3):
                vals = [rng.randint(-1000, 1000) for _ in range(splits)]
                run_launch(probe, vals, seed=launch * 13 + k)
                assert probe.status == 0 and probe.y == sum(vals), (launch, kind, reset, k)


def test_split_exchange_planted_epoch_mistake_is_caught():
    # a failed CTA that drew last but leaves the word at its epoch: the next
    # launch never sees its last arrival
    splits = 4
    broken = 0
    for launch in range(50):
        tile = Tile(splits)
        run_launch(tile, [1] * splits, seed=launch, fail={0, 1, 2, 3}, mistake="failed_last_keeps_epoch")
        run_launch(tile, [2] * splits, seed=launch + 1)
        if tile.y != 2 * splits:
            broken += 1
    assert broken == 50
