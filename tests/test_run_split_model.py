"""A Python restatement of the kernels' work split (RunWalker in
ssm_depthwise_causal_gb300/csrc/ccc_device.cuh: runs of equal rows, or of
equal cost with a per-sequence weight; the 32-way ballot searches; the rule
that moves a boundary out of a sequence's first W-1 rows; the segment walk),
fuzzed on random packed batches for what the kernels rely on: every valid
row handed out exactly once, padding rows never, every empty sequence once
when asked for, a walk that starts inside a sequence at least W-1 rows in,
and segments of a walk contiguous and batch-aligned.  The GPU parity tests
check the device code itself; this pins the index logic on the CPU, where
failures are cheap to read."""
import numpy as np
import pytest


def _clamp(v, rows):
    return 0 if v < 0 else (rows if v > rows else v)


def _search_first(pred, lo, hi, lane_value):
    """The device's 32-way ballot search: first i in [lo, hi] with pred(i),
    pred(hi) assumed true; lane_value(i) gives the value a lane tests."""
    while hi - lo >= 32:
        step = (hi - lo + 31) // 32
        m = [pred(lane_value(min(lo + j * step, hi)), min(lo + j * step, hi)) for j in range(32)]
        if not any(m):
            lo = min(lo + 31 * step, hi) + 1
        else:
            j = m.index(True)
            new_hi = min(lo + j * step, hi)
            if j > 0:
                lo = min(lo + (j - 1) * step, hi) + 1
            hi = new_hi
    cand = [lane <= hi - lo and pred(lane_value(lo + lane), lo + lane) for lane in range(32)]
    return lo + cand.index(True) if any(cand) else hi


class Walker:
    def __init__(self, cu, rows, run, runs, H, empties, B, alpha):
        self.cu, self.rows, self.H, self.empties, self.B = cu, rows, H, empties, B
        N = self.N = len(cu) - 1
        self.last = run == runs - 1
        self.fresh, self.s, self.e, self.r, self.n = True, 0, 0, 0, 0
        if N <= 0:
            self.R_lo = self.R_hi = 0
            return
        cuc = lambda i: _clamp(cu[i], rows) if i <= N else rows  # noqa: E731
        T = cuc(N)
        if alpha == 0:
            self.R_lo, self.R_hi = run * T // runs, (run + 1) * T // runs
        else:
            total = T + alpha * N

            def row_at(c):
                if c >= total:
                    return T
                f = _search_first(lambda v, i: v + alpha * i > c, 0, N, cuc)
                ns = max(f - 1, 0)
                s0, e0 = cuc(ns), cuc(ns + 1)
                ln = max(e0 - s0, 0)
                off = c - (s0 + alpha * (ns + 1))
                return s0 + min(max(off, 0), ln)
            self.R_lo, self.R_hi = row_at(run * total // runs), row_at((run + 1) * total // runs)
        R_lo = self.R_lo
        n = _search_first(lambda v, i: v >= R_lo, 0, N - 1, lambda i: cuc(i + 1))
        if n < N:
            sa, ea = cuc(n), cuc(n + 1)
            if ea == R_lo and sa < R_lo:
                n += 1
            elif sa < R_lo < ea and R_lo - sa < H:
                self.R_lo = sa
        self.n = n
        if n < N:
            self._load()

    def _load(self):
        s, e = _clamp(self.cu[self.n], self.rows), _clamp(self.cu[self.n + 1], self.rows)
        e = max(e, s)
        self.s, self.e = s, e
        self.r = min(max(s, self.R_lo), e)
        self.fresh = True

    def next(self):
        while self.n < self.N:
            s, e = self.s, self.e
            if self.fresh:
                if not (s < self.R_hi or (self.last and s == self.R_hi)):
                    return None
                if s < self.R_hi < e and self.R_hi - s < self.H:
                    return None
            stop = min(e, self.R_hi)
            if s == e:
                if self.fresh and self.empties:
                    item = (self.n, s, e, s, 0)
                    self.fresh = False
                    self.n += 1
                    if self.n < self.N:
                        self._load()
                    return item, False, False
            elif self.r < stop:
                nr = min(stop - self.r, self.B)
                item = (self.n, s, e, self.r, nr)
                cont = not self.fresh
                self.fresh = False
                self.r += nr
                return item, cont, self.r < stop
            if e > self.R_hi:
                return None
            self.n += 1
            if self.n < self.N:
                self._load()
        return None


def _check(cu, rows, runs, H, B, empties, alpha):
    N = len(cu) - 1
    covered = np.zeros(rows, int)
    empty_seen = np.zeros(N, int)
    for run in range(runs):
        w = Walker(cu, rows, run, runs, H, empties, B, alpha)
        prev = walk_start = None
        while True:
            x = w.next()
            if x is None:
                break
            (n, s, e, r0, nr), cont, more = x
            if nr == 0:
                assert s == e
                empty_seen[n] += 1
                prev = None
                continue
            covered[r0:r0 + nr] += 1
            if not cont:
                assert r0 - s == 0 or r0 - s >= H, "a walk starting inside a sequence needs H rows before it"
                walk_start = r0
            else:
                assert prev == (n, r0), "segments of a walk must be contiguous"
                assert (r0 - walk_start) % B == 0
            if more:
                assert nr == B
            prev = (n, r0 + nr)
    T = cu[N]
    assert np.all(covered[:T] == 1), np.nonzero(covered[:T] != 1)
    assert np.all(covered[T:] == 0)
    if empties:
        assert np.all(empty_seen[np.diff(cu) == 0] == 1)


@pytest.mark.parametrize("alpha", [0, 1, 10, 64])
def test_every_row_exactly_once(alpha):
    rng = np.random.default_rng(100 + alpha)
    for _ in range(150):
        N = int(rng.integers(1, 120))
        kind = rng.integers(0, 4)
        if kind == 0:
            lens = rng.integers(0, 5, N)
        elif kind == 1:
            lens = rng.integers(0, 200, N)
        elif kind == 2:
            lens = np.where(rng.random(N) < 0.3, 0, rng.integers(1, 70, N))
        else:
            lens = rng.integers(0, 3, N) * rng.integers(0, 100, N)
        cu = [int(v) for v in np.concatenate([[0], np.cumsum(lens)])]
        rows = cu[-1] + int(rng.integers(0, 5))
        runs = int(rng.choice([1, 2, 3, 7, 43, 86, int(rng.integers(1, 300))]))
        H = int(rng.integers(1, 4))
        B = int(rng.choice([4, 8, 64]))
        for empties in (False, True):
            _check(cu, rows, runs, H, B, empties, alpha)


def test_cost_split_balances_walks():
    """With the per-sequence weight the run holding many short sequences
    gets fewer rows than one inside a long sequence."""
    cu = [0] + list(np.cumsum([2000] + [10] * 200))
    runs, alpha = 8, 10
    rows_of = []
    for run in range(runs):
        w = Walker(cu, cu[-1], run, runs, 3, False, 64, alpha)
        n_rows = 0
        while (x := w.next()) is not None:
            n_rows += x[0][4]
        rows_of.append(n_rows)
    assert sum(rows_of) == cu[-1]
    assert rows_of[0] > rows_of[-1]          # the long sequence's run takes more rows
