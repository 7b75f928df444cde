"""Discrete-event model of the mbarrier protocols of the tcgen05 kernels
(csrc/attn_fwd2_sm103.cu, csrc/attn_bwd_sm103.cu, csrc/attn_proj_sm103.cu,
csrc/attn_split_sm103.cu), used by test_barrier_protocols.py.

Each role of a CTA (TMA producer, MMA issuer, elementwise warps) is a
generator that yields requests; a seeded scheduler interleaves them at
random, the tensor pipe executes queued MMAs in issue order, TMA copies land
in any order.  Hazard assertions check every read against the writes it
depends on, and every barrier wait is checked the way the hardware performs
it: a wait for a barrier's n-th completion is a parity test, which is only
exact when the barrier has completed n-1 or n times so far.

Requests:
  ('wait', bar, n)      block until bar has completed n+1 phases
  ('arrive', bar)       one arrival
  ('mma', label, fn)    queue work on the in-order tensor pipe (fn runs then)
  ('commit', bar)       queue one arrival behind the queued MMAs
  ('tma', bar, fn)      a copy: fn runs when it lands, then one arrival on bar
  ('tma', bar, fn, b)   a copy that completes b bytes of bar's transaction count
  ('arrive_tx', bar, b) one arrival that first expects b more bytes
  ('until', pred)       block until pred() holds (a wait that is not a
                        barrier's, e.g. for every bulk store to have read)
A commit may name a tuple of barriers (a multicast commit: one arrival on
each).
"""
import random


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"over-arrival on {self.name}"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count


class TxBar(Bar):
    """A barrier whose phase also waits for a transaction count (bytes
    expected by arrive_tx, completed by copies) to return to zero; copies may
    complete bytes before they are expected (the count goes negative)."""

    def __init__(self, name, count):
        super().__init__(name, count)
        self.tx = 0

    def _flip(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"over-arrival on {self.name}"
        self._flip()

    def expect(self, nbytes):
        self.tx += nbytes

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._flip()


class Deadlock(Exception):
    pass


class Sim:
    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.roles, self.pipe, self.tma = {}, [], []

    def add(self, name, gen):
        self.roles[name] = [gen, None]

    @staticmethod
    def _ready(req):
        if req[0] == 'until':
            return req[1]()
        _, bar, n = req
        assert bar.phase <= n + 1, f"{bar.name}: wait for completion {n} sees {bar.phase} (parity ambiguous)"
        assert bar.phase >= n, f"{bar.name}: wait for completion {n} sees {bar.phase} (parity wait passes early)"
        return bar.phase > n

    def _step(self, name):
        st = self.roles[name]
        gen, req = st
        if req is not None:
            if not self._ready(req):
                return False
            st[1] = None
        while True:
            try:
                r = next(gen)
            except StopIteration:
                del self.roles[name]
                return True
            if r[0] in ('wait', 'until'):
                if self._ready(r):
                    continue
                st[1] = r
                return True
            if r[0] == 'arrive':
                r[1].arrive()
            elif r[0] == 'arrive_tx':
                r[1].expect(r[2])
                r[1].arrive()
            elif r[0] in ('mma', 'commit'):
                self.pipe.append(r)
            elif r[0] == 'tma':
                self.tma.append(r)
            if self.rng.random() < 0.3:
                return True

    def run(self, max_iter=10 ** 6):
        for _ in range(max_iter):
            opts = list(self.roles) + (['@pipe'] if self.pipe else []) + (['@tma'] if self.tma else [])
            if not opts:
                return
            self.rng.shuffle(opts)
            progressed = False
            for o in opts:
                if o == '@pipe':
                    r = self.pipe.pop(0)
                    if r[0] == 'mma':
                        r[2]()
                    else:
                        for b in (r[1] if isinstance(r[1], tuple) else (r[1],)):
                            b.arrive()
                    progressed = True
                elif o == '@tma':
                    r = self.tma.pop(self.rng.randrange(len(self.tma)))
                    r[2]()
                    if len(r) == 4:
                        r[1].complete_tx(r[3])
                    else:
                        r[1].arrive()
                    progressed = True
                elif self._step(o):
                    progressed = True
                if progressed:
                    break
            if not progressed:
                raise Deadlock({n: (r[1][1].name, r[1][2]) for n, r in self.roles.items() if r[1]})
        raise RuntimeError("no termination")


def dkdv_cta(seed, n_steps, double_scores=True, n_stages=4, p_barrier_per_buffer=True, release_by_dp=False):
    """One CTA of bwd_dkdv_kernel: K/V once, then n_steps steps of a Q/dO ring
    of n_stages stages.  double_scores: head size 64, S^T issued a step ahead
    into two TMEM buffers (issue order S^T(n+1), dK(n-1), dP^T(n), dV(n));
    else head size 128 (S^T(n), dK(n-1), dP^T(n), dV(n)).  The two flags after
    it select variants that are not in the library (for the planted-mistake
    checks): one P^T barrier pair for both buffers, and ring stages reloaded
    on dp_full instead of their own release barrier."""
    dbl = double_scores
    sim = Sim(seed)
    kv_full = Bar("kv_full", 1)
    qdo_full = [Bar(f"qdo_full{i}", 1) for i in range(n_stages)]
    qdo_empty = [Bar(f"qdo_empty{i}", 1) for i in range(n_stages)]
    s_full = [Bar("s_full0", 1), Bar("s_full1", 1)]
    dp_full, ds_full, acc_done = Bar("dp_full", 1), Bar("ds_full", 8), Bar("acc_done", 1)
    nb = 2 if (dbl and p_barrier_per_buffer) else 1
    p_full = [[Bar(f"p_full{b}{h}", 8) for h in range(2)] for b in range(nb)]
    st = dict(q_land=[-1] * n_stages, s_exec=-1, dp_exec=-1, dv_exec=-1, dk_exec=-1,
              s_read={w: -1 for w in range(8)}, p_wr={(w, h): -1 for w in range(8) for h in range(2)},
              ds_wr={w: -1 for w in range(8)}, dp_read={w: -1 for w in range(8)})

    def pbar(n, h):
        b = (n & 1) if nb == 2 else 0
        return p_full[b][h], ((n >> 1) if nb == 2 else n)

    def producer():
        yield ('tma', kv_full, lambda: None)
        for n in range(n_steps):
            s = n % n_stages
            if n >= n_stages:
                yield ('wait', dp_full, n - 1) if release_by_dp else ('wait', qdo_empty[s], n // n_stages - 1)

            def land(n=n, s=s):
                assert st['dk_exec'] >= n - n_stages, "ring stage reloaded before dK read it"
                st['q_land'][s] = n
            yield ('tma', qdo_full[s], land)

    def issuer():
        yield ('wait', kv_full, 0)

        def issue_s(n):
            s = n % n_stages
            yield ('wait', qdo_full[s], n // n_stages)

            def ex(n=n, s=s):
                assert st['q_land'][s] == n
                if dbl and n >= 2:
                    assert st['dv_exec'] >= n - 2, "S^T overwrote P^T(n-2) before dV read it"
                    assert all(v >= n - 2 for v in st['s_read'].values())
                if not dbl and n >= 1:
                    assert st['dv_exec'] >= n - 1, "S^T overwrote P^T(n-1) before dV read it"
                st['s_exec'] = n
            yield ('mma', 'S', ex)
            yield ('commit', s_full[n & 1 if dbl else 0])

        def issue_dk(m):
            yield ('wait', ds_full, m)

            def ex(m=m):
                assert all(v >= m for v in st['ds_wr'].values()), "dK before dS^T written"
                assert st['q_land'][m % n_stages] == m, "dK read a reloaded stage"
                st['dk_exec'] = m
            yield ('mma', 'dK', ex)
            if not release_by_dp:
                yield ('commit', qdo_empty[m % n_stages])

        if dbl:
            yield from issue_s(0)
        for n in range(n_steps):
            if dbl:
                if n + 1 < n_steps:
                    yield from issue_s(n + 1)
            else:
                yield from issue_s(n)
            if n > 0:
                yield from issue_dk(n - 1)

            def exdp(n=n):
                assert st['dk_exec'] >= n - 1, "dP^T overwrote dS^T(n-1) before dK read it"
                assert all(v >= n - 1 for v in st['dp_read'].values())
                assert st['q_land'][n % n_stages] == n
                st['dp_exec'] = n
            yield ('mma', 'dP', exdp)
            yield ('commit', dp_full)
            for h in range(2):
                bar, k = pbar(n, h)
                yield ('wait', bar, k)

                def exdv(n=n, h=h):
                    assert all(st['p_wr'][(w, h)] >= n for w in range(8)), "dV before P^T written"
                    assert st['q_land'][n % n_stages] == n
                    if h == 1:
                        st['dv_exec'] = n
                yield ('mma', 'dV', exdv)
        yield from issue_dk(n_steps - 1)
        yield ('commit', acc_done)

    def elementwise(w):
        for n in range(n_steps):
            yield ('wait', s_full[n & 1 if dbl else 0], (n >> 1) if dbl else n)
            assert st['s_exec'] >= n
            st['s_read'][w] = n
            for h in range(2):
                st['p_wr'][(w, h)] = n
                yield ('arrive', pbar(n, h)[0])
            yield ('wait', dp_full, n)
            assert st['dp_exec'] >= n
            st['dp_read'][w] = n
            st['ds_wr'][w] = n
            yield ('arrive', ds_full)
        yield ('wait', acc_done, 0)
        assert st['dk_exec'] == n_steps - 1 and st['dv_exec'] == n_steps - 1
        # The epilogue stages dV and dK in the first Q and dO ring stages.
        assert not sim.tma, "gradient tiles staged over a ring stage a copy still fills"

    sim.add('producer', producer())
    sim.add('issuer', issuer())
    for w in range(8):
        sim.add(f'ew{w}', elementwise(w))
    sim.run()


def dq_rings(seed, steps, k_stages=3):
    """The K and V rings of bwd_dq_kernel at head size 128 for one item: K in
    k_stages stages released after the dQ MMA that reads it last; V in one
    stage, reloaded once dp_full shows dP (V's only reader) complete."""
    sim = Sim(seed)
    k_full = [Bar(f"k_full{i}", 1) for i in range(k_stages)]
    k_empty = [Bar(f"k_empty{i}", 1) for i in range(k_stages)]
    v_full = Bar("v_full", 1)
    s_full, s_free, dp_full, ds_full = Bar("s_full", 1), Bar("s_free", 8), Bar("dp_full", 1), Bar("ds_full", 8)
    st = dict(k_land=[-1] * k_stages, v_land=-1, s_exec=-1, dp_exec=-1, dq_exec=-1,
              s_read={w: -1 for w in range(8)}, ds_wr={w: -1 for w in range(8)})

    def producer():
        for g in range(steps):
            s = g % k_stages
            if g >= k_stages:
                yield ('wait', k_empty[s], g // k_stages - 1)

            def lk(g=g, s=s):
                assert st['dq_exec'] >= g - k_stages, "K stage reloaded before dQ read it"
                st['k_land'][s] = g
            yield ('tma', k_full[s], lk)
            if g >= 1:
                yield ('wait', dp_full, g - 1)

            def lv(g=g):
                assert st['dp_exec'] >= g - 1, "V reloaded before dP read it"
                st['v_land'] = g
            yield ('tma', v_full, lv)

    def issuer():
        def dq(m):
            yield ('wait', ds_full, m)

            def ex(m=m):
                assert all(v >= m for v in st['ds_wr'].values())
                assert st['k_land'][m % k_stages] == m
                st['dq_exec'] = m
            yield ('mma', 'dQ', ex)
            yield ('commit', k_empty[m % k_stages])

        for g in range(steps):
            s = g % k_stages
            yield ('wait', k_full[s], g // k_stages)
            if g > 0:
                yield ('wait', s_free, g - 1)

            def exs(g=g, s=s):
                assert st['k_land'][s] == g
                assert all(v >= g - 1 for v in st['s_read'].values())
                st['s_exec'] = g
            yield ('mma', 'S', exs)
            yield ('commit', s_full)
            if g > 0:
                yield from dq(g - 1)
            yield ('wait', v_full, g)

            def exdp(g=g):
                assert st['v_land'] == g
                assert st['dq_exec'] >= g - 1, "dP overwrote dS before dQ read it"
                st['dp_exec'] = g
            yield ('mma', 'dP', exdp)
            yield ('commit', dp_full)
        yield from dq(steps - 1)

    def elementwise(w):
        for g in range(steps):
            yield ('wait', s_full, g)
            assert st['s_exec'] >= g
            st['s_read'][w] = g
            yield ('arrive', s_free)
            yield ('wait', dp_full, g)
            assert st['dp_exec'] >= g
            st['ds_wr'][w] = g
            yield ('arrive', ds_full)

    sim.add('producer', producer())
    sim.add('issuer', issuer())
    for w in range(8):
        sim.add(f'ew{w}', elementwise(w))
    sim.run()


def fwd_pair_cta(seed, items, wait_o_free=True, wait_stage_free=True):
    """One CTA of the paired-head forward (fwd2_kernel, two query heads
    sharing each K/V tile): `items` lists the key tiles of each work item.
    Roles: producer (Q of an item after the previous item's last score MMA;
    K and V of a tile into a two-stage ring), issuer (S_A(0), S_B(0), then per
    tile PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)), four softmax warps per head
    (P written over the scores; O rescaled between PVs) and each head's
    epilogue through the one staging tile; after every role has finished
    (the issuer having waited for its drain commit) no MMA or copy may still
    be in flight.  The FP8 forward (fwd_fp8_kernel) runs the same protocol.
    The two flags drop waits of the library's protocol (planted-mistake
    checks).  The model shows the o_free
    wait to be implied by p_full: a head's softmax warps read O in the
    epilogue before they arrive on p_full for the next item's first tile,
    and that first PV waits for p_full."""
    sim = Sim(seed)
    q_full, q_empty = Bar("q_full", 1), Bar("q_empty", 1)
    kv_full = [Bar("kv_full0", 1), Bar("kv_full1", 1)]
    kv_empty = [Bar("kv_empty0", 1), Bar("kv_empty1", 1)]
    s_full = [Bar("s_full0", 1), Bar("s_full1", 1)]
    p_full = [Bar("p_full0", 4), Bar("p_full1", 4)]
    o_done = [Bar("o_done0", 1), Bar("o_done1", 1)]
    o_free = [Bar("o_free0", 4), Bar("o_free1", 4)]
    staged = [Bar("staged0", 4), Bar("staged1", 4)]
    stage_free = Bar("stage_free", 1)
    store_read = [Bar("store_read0", 1), Bar("store_read1", 1)]   # a storer's own wait on its copy
    drain = Bar("drain", 1)
    done = Bar("done", 1 + 1 + 8)
    tiles = [(it, j, n) for it, n in enumerate(items) for j in range(n)]
    first = {}
    for gk, (it, j, n) in enumerate(tiles):
        first.setdefault(it, gk)
    st = dict(q_land=-1, kv_land=[-1, -1], s_exec=[-1, -1], pv_exec=[-1, -1], s_read={}, p_wr={},
              o_read={}, stage_use=-1, store_read=-1)
    for x in range(2):
        for w in range(4):
            st['s_read'][(x, w)] = -1
            st['p_wr'][(x, w)] = -1
            st['o_read'][(x, w)] = -1

    def producer():
        gk = 0
        for it, n in enumerate(items):
            if it >= 1:
                yield ('wait', q_empty, it - 1)

            def lq(it=it):
                assert all(v >= first[it - 1] + items[it - 1] - 1 for v in st['s_exec']) if it >= 1 else True, \
                    "Q reloaded before the last score MMAs read it"
                st['q_land'] = it
            yield ('tma', q_full, lq)
            for j in range(n):
                s = gk % 2
                if gk >= 2:
                    yield ('wait', kv_empty[s], (gk >> 1) - 1)

                def lkv(gk=gk, s=s):
                    assert min(st['pv_exec']) >= gk - 2, "K/V stage reloaded before the PVs read it"
                    st['kv_land'][s] = gk
                yield ('tma', kv_full[s], lkv)
                gk += 1
        yield ('arrive', done)

    def issuer():
        def issue_s(x, gk, it):
            def ex(x=x, gk=gk, it=it):
                assert st['q_land'] == it and st['kv_land'][gk % 2] == gk
                assert st['pv_exec'][x] >= gk - 1, "S overwrote P before the PV read it"
                assert all(st['s_read'][(x, w)] >= gk - 1 for w in range(4))
                st['s_exec'][x] = gk
            yield ('mma', f'S{x}', ex)
            yield ('commit', s_full[x])

        g0 = 0
        for it, n in enumerate(items):
            yield ('wait', q_full, it)
            yield ('wait', kv_full[g0 % 2], g0 >> 1)
            yield from issue_s(0, g0, it)
            yield from issue_s(1, g0, it)
            if n == 1:
                yield ('commit', q_empty)
            for j in range(n):
                gk = g0 + j
                for x in range(2):
                    yield ('wait', p_full[x], gk)
                    if j == 0 and it >= 1 and wait_o_free:
                        yield ('wait', o_free[x], it - 1)

                    def expv(x=x, gk=gk, j=j, it=it):
                        assert all(st['p_wr'][(x, w)] >= gk for w in range(4)), "PV before P written"
                        assert st['kv_land'][gk % 2] == gk
                        if j == 0 and it >= 1:
                            assert all(st['o_read'][(x, w)] >= it - 1 for w in range(4)), \
                                "PV overwrote O before the epilogue read it"
                        st['pv_exec'][x] = gk
                    yield ('mma', f'PV{x}', expv)
                    if x == 1:
                        yield ('commit', kv_empty[gk % 2])
                    if j == n - 1:
                        yield ('commit', o_done[x])
                    if j + 1 < n:
                        if x == 0:
                            yield ('wait', kv_full[(gk + 1) % 2], (gk + 1) >> 1)
                        yield from issue_s(x, gk + 1, it)
                        if x == 1 and j + 1 == n - 1:
                            yield ('commit', q_empty)
            g0 += n
        yield ('commit', drain)
        yield ('wait', drain, 0)
        yield ('arrive', done)

    def softmax(x, w):
        gk = 0
        for it, n in enumerate(items):
            for j in range(n):
                yield ('wait', s_full[x], gk)
                assert st['s_exec'][x] >= gk
                # the O rescale of tile j: PV_x(j-1) has completed, PV_x(j) waits for this warp
                assert st['pv_exec'][x] == gk - 1 or (j == 0 and st['pv_exec'][x] < gk), "O rescaled under a PV"
                st['s_read'][(x, w)] = gk
                st['p_wr'][(x, w)] = gk
                yield ('arrive', p_full[x])
                gk += 1
            use = 2 * it + x
            yield ('wait', o_done[x], it)
            if use > 0 and wait_stage_free:
                yield ('wait', stage_free, use - 1)
            assert st['pv_exec'][x] >= gk - 1
            assert st['store_read'] >= use - 1, "staging tile rewritten before its store read it"
            st['o_read'][(x, w)] = it
            st['stage_use'] = use
            yield ('arrive', o_free[x])
            yield ('arrive', staged[x])
            if w == 0:
                # The group's first warp stores the tile and waits until the
                # copy engine has read it (bulk wait_group.read) before
                # releasing the staging tile.
                yield ('wait', staged[x], it)

                def read(use=use):
                    st['store_read'] = use
                yield ('tma', store_read[x], read)
                yield ('wait', store_read[x], it)
                yield ('arrive', stage_free)
        yield ('arrive', done)

    def teardown():
        yield ('wait', done, 0)
        assert not sim.pipe and not sim.tma, "CTA exits with MMAs or copies in flight"
        assert st['store_read'] == 2 * len(items) - 1

    sim.add('producer', producer())
    sim.add('issuer', issuer())
    for x in range(2):
        for w in range(4):
            sim.add(f'sm{x}{w}', softmax(x, w))
    sim.add('teardown', teardown())
    sim.run()


def proj_pair(seed, n_tiles, n_kb, n_stages=3, expect_both=True, acc_empty_wait=True, peer_empty_wait=True):
    """One CTA pair of the QKV projection (proj_kernel, tcgen05.mma.cta_group::2):
    n_tiles output tiles of n_kb k-blocks each, a ring of n_stages stages in
    each CTA.  Each CTA's producer copies its half of a stage (two copies of
    16 KB) and signals the first CTA's stage barrier, on which the first
    CTA's producer also expects the bytes of both halves; the first CTA's
    issuer runs the MMAs (reading both CTAs' stages, writing both CTAs'
    accumulators) and commits stage release, accumulator full and the final
    drain to both CTAs' barriers at once; both CTAs' four epilogue warps
    release an accumulator on the first CTA's barrier (count 8).  The issuer
    tests the next stage's barrier one k-block ahead (the same parity check,
    without blocking).  After every role has finished (the final cluster
    barrier) no MMA or copy may still be in flight.  The flags drop parts of
    the protocol (planted-mistake checks): the first CTA expecting one CTA's
    bytes, the issuer not waiting for the accumulator's release, the second
    CTA's producer not waiting for its stage's release."""
    sim = Sim(seed)
    half = 2 * 16384
    full = [TxBar(f"full{i}", 1) for i in range(n_stages)]             # first CTA's
    empty = [[Bar(f"empty{r}{i}", 1) for i in range(n_stages)] for r in range(2)]
    acc_full = [[Bar(f"acc_full{r}{b}", 1) for b in range(2)] for r in range(2)]
    acc_empty = [Bar(f"acc_empty{b}", 8) for b in range(2)]           # first CTA's
    drain = [Bar(f"drain{r}", 1) for r in range(2)]
    done = Bar("done", 2 + 1 + 1 + 8)
    st = dict(land=[[-1] * n_stages for _ in range(2)], mma_exec=-1,
              acc_tile=[-1, -1], acc_read={(r, w): -1 for r in range(2) for w in range(4)})

    def producer(r):
        for it in range(n_tiles * n_kb):
            s, u = it % n_stages, it // n_stages
            if u > 0 and (r == 0 or peer_empty_wait):
                yield ('wait', empty[r][s], u - 1)
            if r == 0:
                yield ('arrive_tx', full[s], 2 * half if expect_both else half)

            def land(it=it, s=s, r=r):
                assert st['mma_exec'] >= it - n_stages, "stage overwritten before the MMAs read it"
                st['land'][r][s] = it
            # The two copies (x rows, w rows) of this CTA's half; the first
            # one's landing is folded into the second's bytes.
            yield ('tma', full[s], lambda: None, half // 2)
            yield ('tma', full[s], land, half // 2)
        yield ('arrive', done)

    def issuer():
        def test(bar, n):
            return Sim._ready(('wait', bar, n))
        it = 0
        for lt in range(n_tiles):
            b = lt & 1
            if lt >= 2 and acc_empty_wait:
                yield ('wait', acc_empty[b], (lt >> 1) - 1)
            ready = test(full[it % n_stages], it // n_stages)
            for kb in range(n_kb):
                s, u = it % n_stages, it // n_stages
                if not ready:
                    yield ('wait', full[s], u)
                ready = test(full[(it + 1) % n_stages], (it + 1) // n_stages) if kb + 1 < n_kb else True

                def ex(it=it, s=s, lt=lt, kb=kb, b=b):
                    assert st['land'][0][s] == it and st['land'][1][s] == it, "MMA before both halves landed"
                    if kb == 0:
                        assert all(v >= lt - 2 for v in st['acc_read'].values()), \
                            "accumulator overwritten before both epilogues read it"
                    st['mma_exec'] = it
                    if kb == n_kb - 1:
                        st['acc_tile'][b] = lt
                yield ('mma', 'MMA', ex)
                yield ('commit', (empty[0][s], empty[1][s]))
                it += 1
            yield ('commit', (acc_full[0][b], acc_full[1][b]))
        yield ('commit', (drain[0], drain[1]))
        yield ('wait', drain[0], 0)
        yield ('arrive', done)

    def tmem_warp_peer():
        yield ('wait', drain[1], 0)
        yield ('arrive', done)

    def epilogue(r, w):
        for lt in range(n_tiles):
            b = lt & 1
            yield ('wait', acc_full[r][b], lt >> 1)
            assert st['acc_tile'][b] == lt, "epilogue read an accumulator the MMAs had not finished"
            st['acc_read'][(r, w)] = lt
            yield ('arrive', acc_empty[b])
        yield ('arrive', done)

    def teardown():
        yield ('wait', done, 0)
        assert not sim.pipe and not sim.tma, "pair released its memory with MMAs or copies in flight"
        assert st['mma_exec'] == n_tiles * n_kb - 1

    for r in range(2):
        sim.add(f'producer{r}', producer(r))
    sim.add('issuer', issuer())
    sim.add('tmem1', tmem_warp_peer())
    for r in range(2):
        for w in range(4):
            sim.add(f'epi{r}{w}', epilogue(r, w))
    sim.add('teardown', teardown())
    sim.run()


def dq_cta(seed, items, k_stages=3, v_stages=1, item_slots=4, wait_stage_free=True, wait_dq_free=True,
           k_release_on_s=False):
    """One persistent CTA of bwd_dq_kernel (head size 128: a 3-stage K ring and
    a one-stage V ring; head size 64: 4 and 4): `items` lists the key steps of
    each item the CTA claims.  Roles: the producer (claims items into a queue
    of item_slots slots; K, V and the item's dO), the Q producer (Q of item
    it into buffer it & 1 once the store of item it-2's dQ tile, staged in
    that buffer, has read it), the MMA issuer (order S(n), dQ(n-1), dP(n);
    two dQ accumulators, items alternating), and eight elementwise warps
    (P from S, dS over dP in TMEM; the epilogue of an item after the next
    item's first dS, staging dQ in the item's Q buffer; the first warp issues
    the tile store and releases the buffer once the store has read it, at
    its next dS arrival or the next item's start).  The flags change the
    protocol (planted-mistake checks): the Q reload without the wait for the
    store's read; the first dQ MMA of an item without the wait for the
    epilogue two items back (which the model shows to be implied: every
    elementwise warp runs that epilogue before its first dS arrival of the
    next item but one, and the dQ MMA waits for that dS); the K stage
    released after its score MMA instead of after its dQ MMA."""
    sim = Sim(seed)
    NKS, NVS, NIS = k_stages, v_stages, item_slots
    q_full = [Bar("q_full0", 1), Bar("q_full1", 1)]
    do_full, do_empty, drain = Bar("do_full", 1), Bar("do_empty", 1), Bar("drain", 1)
    k_full = [Bar(f"k_full{i}", 1) for i in range(NKS)]
    k_empty = [Bar(f"k_empty{i}", 1) for i in range(NKS)]
    v_full = [Bar(f"v_full{i}", 1) for i in range(NVS)]
    v_empty = [Bar(f"v_empty{i}", 1) for i in range(NVS)]
    s_full, s_free, dp_full, ds_full = Bar("s_full", 1), Bar("s_free", 8), Bar("dp_full", 1), Bar("ds_full", 8)
    acc_done = [Bar("acc_done0", 1), Bar("acc_done1", 1)]
    dq_free = [Bar("dq_free0", 8), Bar("dq_free1", 8)]
    staged = Bar("staged", 8)
    stage_free = [Bar("stage_free0", 1), Bar("stage_free1", 1)]
    store_read = Bar("store_read", 1)          # counts the stores' reads (waited on by 'until')
    item_full = [Bar(f"item_full{i}", 1) for i in range(NIS)]
    item_empty = [Bar(f"item_empty{i}", 10) for i in range(NIS)]
    done = Bar("done", 1 + 1 + 1 + 8)
    slot_val = [None] * NIS
    first_g = []
    g = 0
    for n in items:
        first_g.append(g)
        g += n
    last_g = [first_g[i] + items[i] - 1 for i in range(len(items))]
    W = range(8)
    st = dict(q_land=[-1, -1], do_land=-1, k_land=[-1] * NKS, v_land=[-1] * NVS, s_exec=-1, dp_exec=-1,
              dq_exec=-1, acc_item=[-1, -1], s_read={w: -1 for w in W}, dp_read={w: -1 for w in W},
              ds_wr={w: -1 for w in W}, acc_read={w: -1 for w in W}, staged_item=[-1, -1],
              store_read=[-1, -1], stores_pending=0)

    def next_item(it):
        slot = it % NIS
        yield ('wait', item_full[slot], it // NIS)
        yield ('arrive', item_empty[slot])

    def producer():
        for it in range(len(items) + 1):
            slot = it % NIS
            if it >= NIS:
                yield ('wait', item_empty[slot], it // NIS - 1)
            slot_val[slot] = it if it < len(items) else -1
            yield ('arrive', item_full[slot])
            if it == len(items):
                break
            for n in range(items[it]):
                gi = first_g[it] + n
                ks, u = gi % NKS, gi // NKS
                if u > 0:
                    yield ('wait', k_empty[ks], u - 1)

                def lk(gi=gi, ks=ks):
                    assert st['dq_exec'] >= gi - NKS and st['s_exec'] >= gi - NKS, "K stage reloaded under a reader"
                    st['k_land'][ks] = gi
                yield ('tma', k_full[ks], lk)
                if n == 0:
                    if it > 0:
                        yield ('wait', do_empty, it - 1)

                    def ld(it=it):
                        assert it == 0 or st['dp_exec'] >= last_g[it - 1], "dO reloaded before the last dP read it"
                        st['do_land'] = it
                    yield ('tma', do_full, ld)
                vs, vu = gi % NVS, gi // NVS
                if vu > 0:
                    yield ('wait', dp_full, gi - 1) if NVS == 1 else ('wait', v_empty[vs], vu - 1)

                def lv(gi=gi, vs=vs):
                    assert st['dp_exec'] >= gi - NVS, "V stage reloaded before dP read it"
                    st['v_land'][vs] = gi
                yield ('tma', v_full[vs], lv)
        yield ('arrive', done)

    def q_producer():
        for it in range(len(items) + 1):
            yield from next_item(it)
            if slot_val[it % NIS] < 0:
                break
            qb = it & 1
            if it >= 2 and wait_stage_free:
                yield ('wait', stage_free[qb], (it >> 1) - 1)

            def lq(it=it, qb=qb):
                if it >= 2:
                    assert st['s_exec'] >= last_g[it - 2], "Q reloaded before the last score MMA read it"
                    assert st['store_read'][qb] >= it - 2, "Q reloaded over a dQ tile its store had not read"
                st['q_land'][qb] = it
            yield ('tma', q_full[qb], lq)
        yield ('arrive', done)

    def issuer():
        pend = [None]

        def issue_dq():
            pg, pit, pfirst, plast = pend[0]
            yield ('wait', ds_full, pg)
            db = pit & 1
            if pfirst and pit >= 2 and wait_dq_free:
                yield ('wait', dq_free[db], (pit >> 1) - 1)

            def ex(pg=pg, pit=pit, pfirst=pfirst, db=db):
                assert all(v >= pg for v in st['ds_wr'].values()), "dQ before dS written"
                assert st['k_land'][pg % NKS] == pg
                if pfirst:
                    assert all(v >= pit - 2 for v in st['acc_read'].values()), \
                        "dQ accumulator overwritten before the epilogue read it"
                    st['acc_item'][db] = pit
                st['dq_exec'] = pg
            yield ('mma', 'dQ', ex)
            if not k_release_on_s:
                yield ('commit', k_empty[pg % NKS])
            if plast:
                yield ('commit', acc_done[db])

        for it in range(len(items) + 1):
            yield from next_item(it)
            if slot_val[it % NIS] < 0:
                break
            yield ('wait', q_full[it & 1], it >> 1)
            for n in range(items[it]):
                gi = first_g[it] + n
                ks, vs = gi % NKS, gi % NVS
                yield ('wait', k_full[ks], gi // NKS)
                if gi > 0:
                    yield ('wait', s_free, gi - 1)

                def exs(gi=gi, ks=ks, it=it):
                    assert st['q_land'][it & 1] == it and st['k_land'][ks] == gi
                    assert all(v >= gi - 1 for v in st['s_read'].values()), "S overwritten before it was read"
                    st['s_exec'] = gi
                yield ('mma', 'S', exs)
                yield ('commit', s_full)
                if k_release_on_s:
                    yield ('commit', k_empty[ks])
                if pend[0] is not None:
                    yield from issue_dq()
                if n == 0:
                    yield ('wait', do_full, it)
                yield ('wait', v_full[vs], gi // NVS)

                def exdp(gi=gi, vs=vs, it=it):
                    assert st['do_land'] == it and st['v_land'][vs] == gi
                    assert st['dq_exec'] >= gi - 1, "dP overwrote dS before dQ read it"
                    assert all(v >= gi - 1 for v in st['dp_read'].values())
                    st['dp_exec'] = gi
                yield ('mma', 'dP', exdp)
                yield ('commit', dp_full)
                if NVS > 1:
                    yield ('commit', v_empty[vs])
                if n == items[it] - 1:
                    yield ('commit', do_empty)
                pend[0] = (gi, it, n == 0, n == items[it] - 1)
        if pend[0] is not None:
            yield from issue_dq()
        yield ('commit', drain)
        yield ('wait', drain, 0)
        yield ('arrive', done)

    def elementwise(w):
        store_db = [-1]

        def release_store():
            if w == 0 and store_db[0] >= 0:
                yield ('until', lambda: st['reads_done'] == st['stores_issued'])
                yield ('arrive', stage_free[store_db[0]])
                store_db[0] = -1

        def epilogue(pit):
            db = pit & 1
            yield ('wait', acc_done[db], pit >> 1)
            assert st['dq_exec'] >= last_g[pit] and st['acc_item'][db] == pit, "epilogue read an unfinished dQ"
            assert st['s_exec'] >= last_g[pit], "dQ staged over a Q tile a score MMA still reads"
            assert st['store_read'][db] >= pit - 2, "dQ staged over a tile its store had not read"
            st['acc_read'][w] = pit
            yield ('arrive', dq_free[db])
            yield ('arrive', staged)
            if w == 0:
                yield ('wait', staged, pit)
                st['staged_item'][db] = pit
                st['stores_issued'] += 1

                def read(pit=pit, db=db):
                    assert st['staged_item'][db] == pit
                    st['store_read'][db] = pit
                    st['reads_done'] += 1
                yield ('tma', store_read, read)
                store_db[0] = db

        pend = -1
        for it in range(len(items) + 1):
            yield from next_item(it)
            if slot_val[it % NIS] < 0:
                break
            yield from release_store()
            for n in range(items[it]):
                gi = first_g[it] + n
                yield ('wait', s_full, gi)
                assert st['s_exec'] == gi
                st['s_read'][w] = gi
                yield ('arrive', s_free)
                yield ('wait', dp_full, gi)
                assert st['dp_exec'] == gi
                st['dp_read'][w] = gi
                st['ds_wr'][w] = gi
                yield ('arrive', ds_full)
                yield from release_store()
                if n == 0 and pend >= 0:
                    yield from epilogue(pend)
                    pend = -1
            pend = it
        if pend >= 0:
            yield from epilogue(pend)
        if w == 0:
            yield ('until', lambda: st['reads_done'] == st['stores_issued'])     # the final bulk wait
        yield ('arrive', done)

    def teardown():
        yield ('wait', done, 0)
        assert not sim.pipe and not sim.tma, "CTA exits with MMAs, copies or stores in flight"

    st['stores_issued'] = st['reads_done'] = 0
    sim.add('producer', producer())
    sim.add('qproducer', q_producer())
    sim.add('issuer', issuer())
    for w in W:
        sim.add(f'ew{w}', elementwise(w))
    sim.add('teardown', teardown())
    sim.run()


def split_fwd_cta(seed, n, pv_wait=True, v_release=True):
    """One CTA of split_fwd_kernel (float32 tensors as bf16 hi/lo parts, one
    128-query tile, key tiles 0..n-1): the producer loads Q once and each key
    tile's K and V parts into two-stage rings (K released once its score
    product has read it, V once its PV product has); the issuer runs the
    score products two tiles ahead into two score buffers (S(0), S(1), then
    per tile PV(j), S(j+2)); four softmax warps turn S(j) into P(j) (written
    over P(j-1) in TMEM) and rescale O, both after PV(j-1) has completed.
    The flags drop parts of the protocol (planted-mistake checks): the
    softmax warps not waiting for PV(j-1), and V stages reloaded without
    waiting for their PV."""
    sim = Sim(seed)
    q_full = Bar("q_full", 1)
    k_full = [Bar(f"k_full{s}", 1) for s in range(2)]
    k_empty = [Bar(f"k_empty{s}", 1) for s in range(2)]
    v_full = [Bar(f"v_full{s}", 1) for s in range(2)]
    v_empty = [Bar(f"v_empty{s}", 1) for s in range(2)]
    s_full = [Bar(f"s_full{s}", 1) for s in range(2)]
    p_full, pv_done, drain = Bar("p_full", 4), Bar("pv_done", 1), Bar("drain", 1)
    done = Bar("done", 1 + 1 + 4)
    W = range(4)
    st = dict(q_land=False, k_land=[-1, -1], v_land=[-1, -1], s_exec=-1, pv_exec=-1,
              s_read={w: -1 for w in W}, p_wr={w: -1 for w in W}, o_scaled={w: -1 for w in W})

    def producer():
        def lq():
            st['q_land'] = True
        yield ('tma', q_full, lq)
        for j in range(n):
            s = j & 1
            if j >= 2:
                yield ('wait', k_empty[s], (j >> 1) - 1)

            def lk(j=j, s=s):
                assert st['s_exec'] >= j - 2, "K stage reloaded before its score product read it"
                st['k_land'][s] = j
            yield ('tma', k_full[s], lk)
            if j >= 2 and v_release:
                yield ('wait', v_empty[s], (j >> 1) - 1)

            def lv(j=j, s=s):
                assert st['pv_exec'] >= j - 2, "V stage reloaded before its PV product read it"
                st['v_land'][s] = j
            yield ('tma', v_full[s], lv)
        yield ('arrive', done)

    def issuer():
        def issue_s(j):
            s = j & 1
            yield ('wait', k_full[s], j >> 1)

            def ex(j=j, s=s):
                assert st['q_land'] and st['k_land'][s] == j
                assert all(v >= j - 2 for v in st['s_read'].values()), "S overwritten before the softmax read it"
                st['s_exec'] = j
            yield ('mma', 'S', ex)
            yield ('commit', s_full[s])
            yield ('commit', k_empty[s])

        yield ('wait', q_full, 0)
        yield from issue_s(0)
        if n >= 2:
            yield from issue_s(1)
        for j in range(n):
            s = j & 1
            yield ('wait', p_full, j)
            yield ('wait', v_full[s], j >> 1)

            def expv(j=j, s=s):
                assert all(v >= j for v in st['p_wr'].values()), "PV before P written"
                assert all(v >= j for v in st['o_scaled'].values()), "PV before O rescaled"
                assert st['v_land'][s] == j
                st['pv_exec'] = j
            yield ('mma', 'PV', expv)
            yield ('commit', pv_done)
            yield ('commit', v_empty[s])
            if j + 2 < n:
                yield from issue_s(j + 2)
        yield ('commit', drain)
        yield ('wait', drain, 0)
        yield ('arrive', done)

    def softmax(w):
        for j in range(n):
            yield ('wait', s_full[j & 1], j >> 1)
            assert st['s_exec'] >= j
            st['s_read'][w] = j
            if j > 0 and pv_wait:
                yield ('wait', pv_done, j - 1)
            assert st['pv_exec'] >= j - 1, "P or O written under the previous PV product"
            st['o_scaled'][w] = j
            st['p_wr'][w] = j
            yield ('arrive', p_full)
        yield ('wait', pv_done, n - 1)
        assert st['pv_exec'] == n - 1
        yield ('arrive', done)

    def teardown():
        yield ('wait', done, 0)
        assert not sim.pipe and not sim.tma, "CTA exits with MMAs or copies in flight"

    sim.add('producer', producer())
    sim.add('issuer', issuer())
    for w in W:
        sim.add(f'sm{w}', softmax(w))
    sim.add('teardown', teardown())
    sim.run()


def split_dkdv_cta(seed, n_steps, s_before_p=False, release_after_dp=False):
    """One CTA of split_dkdv_kernel (float32 tensors as bf16 hi/lo parts; key
    tile stationary): K and V once, then per step a two-stage ring of Q, dO
    and row tables.  Issue order per step: dP^T(n) over dS^T(n-1) (read by
    dK(n-1), issued before), dV(n) once the elementwise warps wrote P^T(n)
    over S^T(n), S^T(n+1) over P^T(n) (read by dV(n), issued before), dK(n)
    once they wrote dS^T(n) over dP^T(n); the ring stage is released after
    dK(n).  The flags change the protocol (planted-mistake checks): S^T(n+1)
    issued before the wait for P^T(n), and the ring stage released after
    dP^T(n) instead of after dK(n)."""
    sim = Sim(seed)
    kv_full = Bar("kv_full", 1)
    qdo_full = [Bar(f"qdo_full{s}", 1) for s in range(2)]
    qdo_empty = [Bar(f"qdo_empty{s}", 1) for s in range(2)]
    s_full = [Bar(f"s_full{s}", 1) for s in range(2)]
    dp_full, p_full, ds_full = Bar("dp_full", 1), Bar("p_full", 8), Bar("ds_full", 8)
    acc_done, drain = Bar("acc_done", 1), Bar("drain", 1)
    done = Bar("done", 1 + 1 + 8)
    W = range(8)
    # TMEM S/P buffer and dP/dS buffer: what they hold ('S', n) / ('P', n) ...
    st = dict(land=[-1, -1], sbuf=None, dpbuf=None, dk_exec=-1, dv_exec=-1)

    def producer():
        yield ('tma', kv_full, lambda: None)
        for n in range(n_steps):
            s = n & 1
            if n >= 2:
                yield ('wait', qdo_empty[s], (n >> 1) - 1)

            def land(n=n, s=s):
                assert st['dk_exec'] >= n - 2 and st['dv_exec'] >= n - 2, "ring stage reloaded under a reader"
                st['land'][s] = n
            yield ('tma', qdo_full[s], land)
        yield ('arrive', done)

    def issuer():
        def issue_s(n):
            s = n & 1
            yield ('wait', qdo_full[s], n >> 1)

            def ex(n=n, s=s):
                assert st['land'][s] == n
                assert n == 0 or st['dv_exec'] >= n - 1, "S^T overwrote P^T before dV read it"
                st['sbuf'] = ('S', n)
            yield ('mma', 'S', ex)
            yield ('commit', s_full[s])

        yield ('wait', kv_full, 0)
        if n_steps > 0:
            yield from issue_s(0)
        for n in range(n_steps):
            s = n & 1

            def exdp(n=n, s=s):
                assert st['land'][s] == n
                assert n == 0 or st['dk_exec'] >= n - 1, "dP^T overwrote dS^T before dK read it"
                st['dpbuf'] = ('dP', n)
            yield ('mma', 'dP', exdp)
            yield ('commit', dp_full)
            if release_after_dp:
                yield ('commit', qdo_empty[s])
            if s_before_p and n + 1 < n_steps:
                yield from issue_s(n + 1)
            yield ('wait', p_full, n)

            def exdv(n=n, s=s):
                assert st['sbuf'] == ('P', n) and st['land'][s] == n, "dV read something other than P^T(n)"
                st['dv_exec'] = n
            yield ('mma', 'dV', exdv)
            if not s_before_p and n + 1 < n_steps:
                yield from issue_s(n + 1)
            yield ('wait', ds_full, n)

            def exdk(n=n, s=s):
                assert st['dpbuf'] == ('dS', n) and st['land'][s] == n, "dK read something other than dS^T(n)"
                st['dk_exec'] = n
            yield ('mma', 'dK', exdk)
            if not release_after_dp:
                yield ('commit', qdo_empty[s])
        yield ('commit', acc_done)
        yield ('commit', drain)
        yield ('wait', drain, 0)
        yield ('arrive', done)

    pw = {w: 0 for w in W}
    dw = {w: 0 for w in W}

    def elementwise(w):
        for n in range(n_steps):
            yield ('wait', s_full[n & 1], n >> 1)
            assert st['sbuf'] in (('S', n), ('P', n)), "elementwise read a score tile other than S^T(n)"
            pw[w] = n + 1
            if all(v == n + 1 for v in pw.values()):
                st['sbuf'] = ('P', n)
            yield ('arrive', p_full)
            yield ('wait', dp_full, n)
            assert st['dpbuf'] in (('dP', n), ('dS', n)), "elementwise read a dP^T tile other than dP^T(n)"
            dw[w] = n + 1
            if all(v == n + 1 for v in dw.values()):
                st['dpbuf'] = ('dS', n)
            yield ('arrive', ds_full)
        yield ('wait', acc_done, 0)
        assert st['dk_exec'] == n_steps - 1 and st['dv_exec'] == n_steps - 1
        yield ('arrive', done)

    def teardown():
        yield ('wait', done, 0)
        assert not sim.pipe and not sim.tma, "CTA exits with MMAs or copies in flight"

    sim.add('producer', producer())
    sim.add('issuer', issuer())
    for w in W:
        sim.add(f'ew{w}', elementwise(w))
    sim.add('teardown', teardown())
    sim.run()


def split_dq_cta(seed, n, k_release_after_s=False, one_s_buffer=False):
    """One CTA of split_dq_kernel (float32 tensors as bf16 hi/lo parts; query
    tile stationary, key tiles 0..n-1): Q and dO once, K in a three-stage ring
    (read by S(j) and dQ(j)), V in a two-stage ring (read by dP(j)).  Issue
    order per tile: dP(j) over dS(j-1) (read by dQ(j-1), issued before), S(j+1)
    into the other score buffer (its previous tile S(j-1) was read before the
    elementwise warps signalled dS(j-1), waited for before dQ(j-1)), dQ(j) once
    dS(j) is written.  The flags change the protocol (planted-mistake
    checks): K stages released after their score product, and one score
    buffer for all tiles."""
    sim = Sim(seed)
    qdo_full = Bar("qdo_full", 1)
    k_full = [Bar(f"k_full{s}", 1) for s in range(3)]
    k_empty = [Bar(f"k_empty{s}", 1) for s in range(3)]
    v_full = [Bar(f"v_full{s}", 1) for s in range(2)]
    v_empty = [Bar(f"v_empty{s}", 1) for s in range(2)]
    s_full = [Bar(f"s_full{s}", 1) for s in range(2)]
    dp_full, ds_full, acc_done, drain = Bar("dp_full", 1), Bar("ds_full", 8), Bar("acc_done", 1), Bar("drain", 1)
    done = Bar("done", 1 + 1 + 8)
    W = range(8)
    st = dict(k_land=[-1] * 3, v_land=[-1] * 2, sbuf=[-1, -1], s_exec=-1, dp_exec=-1, dq_exec=-1,
              s_read={w: -1 for w in W}, ds_wr={w: -1 for w in W})

    def sb(j):
        return 0 if one_s_buffer else (j & 1)

    def producer():
        yield ('tma', qdo_full, lambda: None)
        for j in range(n):
            ks, vs = j % 3, j & 1
            if j >= 3:
                yield ('wait', k_empty[ks], j // 3 - 1)

            def lk(j=j, ks=ks):
                assert st['dq_exec'] >= j - 3 and st['s_exec'] >= j - 3, "K stage reloaded under a reader"
                st['k_land'][ks] = j
            yield ('tma', k_full[ks], lk)
            if j >= 2:
                yield ('wait', v_empty[vs], (j >> 1) - 1)

            def lv(j=j, vs=vs):
                assert st['dp_exec'] >= j - 2, "V stage reloaded before dP read it"
                st['v_land'][vs] = j
            yield ('tma', v_full[vs], lv)
        yield ('arrive', done)

    def issuer():
        def issue_s(j):
            ks = j % 3
            yield ('wait', k_full[ks], j // 3)

            def ex(j=j, ks=ks):
                assert st['k_land'][ks] == j
                assert all(v >= j - (1 if one_s_buffer else 2) for v in st['s_read'].values()), \
                    "S overwritten before the elementwise warps read it"
                st['sbuf'][sb(j)] = j
                st['s_exec'] = j
            yield ('mma', 'S', ex)
            yield ('commit', s_full[j & 1])
            if k_release_after_s:
                yield ('commit', k_empty[ks])

        yield ('wait', qdo_full, 0)
        yield from issue_s(0)
        for j in range(n):
            vs = j & 1
            yield ('wait', v_full[vs], j >> 1)

            def exdp(j=j, vs=vs):
                assert st['v_land'][vs] == j
                assert st['dq_exec'] >= j - 1, "dP overwrote dS before dQ read it"
                st['dp_exec'] = j
            yield ('mma', 'dP', exdp)
            yield ('commit', dp_full)
            yield ('commit', v_empty[vs])
            if j + 1 < n:
                yield from issue_s(j + 1)
            yield ('wait', ds_full, j)

            def exdq(j=j):
                assert all(v >= j for v in st['ds_wr'].values()), "dQ before dS written"
                assert st['k_land'][j % 3] == j, "dQ read a reloaded K stage"
                st['dq_exec'] = j
            yield ('mma', 'dQ', exdq)
            if not k_release_after_s:
                yield ('commit', k_empty[j % 3])
        yield ('commit', acc_done)
        yield ('commit', drain)
        yield ('wait', drain, 0)
        yield ('arrive', done)

    def elementwise(w):
        for j in range(n):
            yield ('wait', s_full[j & 1], j >> 1)
            assert st['sbuf'][sb(j)] == j, "elementwise read a score tile other than S(j)"
            st['s_read'][w] = j
            yield ('wait', dp_full, j)
            assert st['dp_exec'] == j
            st['ds_wr'][w] = j
            yield ('arrive', ds_full)
        yield ('wait', acc_done, 0)
        assert st['dq_exec'] == n - 1
        yield ('arrive', done)

    def teardown():
        yield ('wait', done, 0)
        assert not sim.pipe and not sim.tma, "CTA exits with MMAs or copies in flight"

    sim.add('producer', producer())
    sim.add('issuer', issuer())
    for w in W:
        sim.add(f'ew{w}', elementwise(w))
    sim.add('teardown', teardown())
    sim.run()


def fwd_one_cta(seed, items, nk=3, nv=2, no=1, rope=False, store_release=True, rescale_wait=True,
                wait_rotated_k=True):
    """One CTA of the one-head forward (fwd_kernel): `items` lists the key
    tiles of each work item.  Roles: the producer (Q of item it into buffer
    it & 1 once item it-2's last score MMA and its output store have both
    released it; K in nk stages two tiles ahead of V in nv stages), the score
    issuer (S(g) into buffer g & 1 once the softmax read S(g-2)), the PV
    issuer (PV(g) from P buffer g & 1 into O buffer it % no, an item's first
    PV once the epilogue no items back read that O buffer), four softmax
    warps (P(g) over P(g-2) once PV(g-2) completed; O rescaled, when the row
    maximum grows, once PV(g-1) completed; the epilogue stages out in the
    item's Q buffer and the first warp stores it), and with RoPE four
    rotating warps (Q and every landed K tile rotated in place before the
    score MMA may read them).  The flags change the protocol
    (planted-mistake checks): the Q buffer released by the score MMAs alone,
    the O rescale without its wait, and the score issuer reading a K tile
    that has only landed."""
    sim = Sim(seed)
    rng = __import__("random").Random(seed * 7919 + 1)
    q_full = [Bar(f"q_full{i}", 1) for i in range(2)]
    q_ready = [Bar(f"q_ready{i}", 4) for i in range(2)]
    q_empty = [Bar(f"q_empty{i}", 2 if store_release else 1) for i in range(2)]
    o_free = [Bar(f"o_free{i}", 4) for i in range(no)]
    s_full = [Bar(f"s_full{i}", 1) for i in range(2)]
    s_free = [Bar(f"s_free{i}", 4) for i in range(2)]
    p_full = [Bar(f"p_full{i}", 4) for i in range(2)]
    pv_done = [Bar(f"pv_done{i}", 1) for i in range(2)]
    k_full = [Bar(f"k_full{i}", 1) for i in range(nk)]
    k_ready = [Bar(f"k_ready{i}", 4) for i in range(nk)]
    k_empty = [Bar(f"k_empty{i}", 1) for i in range(nk)]
    v_full = [Bar(f"v_full{i}", 1) for i in range(nv)]
    v_empty = [Bar(f"v_empty{i}", 1) for i in range(nv)]
    o_staged, drain, drain2 = Bar("o_staged", 4), Bar("drain", 1), Bar("drain2", 1)
    done = Bar("done", 1 + 1 + 1 + 4 + (4 if rope else 0))
    first, last = [], []
    g = 0
    for n in items:
        first.append(g)
        last.append(g + n - 1)
        g += n
    W = range(4)
    st = dict(q_item=[-1, -1], q_rot=[-1, -1], q_staged=[-1, -1], store_read=[-1, -1], k_land=[-1] * nk,
              k_rot=[-1] * nk, v_land=[-1] * nv, s_exec=-1, pv_exec=-1, o_item=[-1] * no,
              s_read={w: -1 for w in W}, p_wr={w: -1 for w in W}, o_read={w: -1 for w in W},
              o_scaled={w: -1 for w in W})

    def producer():
        kg = vg = 0
        for it, n in enumerate(items):
            qb = it & 1
            if it >= 2:
                yield ('wait', q_empty[qb], (it >> 1) - 1)

            def lq(it=it, qb=qb):
                if it >= 2:
                    assert st['s_exec'] >= last[it - 2], "Q reloaded before the last score MMA read it"
                    assert st['store_read'][qb] >= it - 2, "Q reloaded over an output tile its store had not read"
                st['q_item'][qb] = it
            yield ('tma', q_full[qb], lq)

            def load_k(gi):
                s, u = gi % nk, gi // nk
                if u > 0:
                    yield ('wait', k_empty[s], u - 1)

                def lk(gi=gi, s=s):
                    assert st['s_exec'] >= gi - nk, "K stage reloaded before its score MMA read it"
                    st['k_land'][s] = gi
                yield ('tma', k_full[s], lk)

            def load_v(gi):
                s, u = gi % nv, gi // nv
                if u > 0:
                    yield ('wait', v_empty[s], u - 1)

                def lv(gi=gi, s=s):
                    assert st['pv_exec'] >= gi - nv, "V stage reloaded before its PV read it"
                    st['v_land'][s] = gi
                yield ('tma', v_full[s], lv)
            base = first[it]
            for j in range(min(2, n)):
                yield from load_k(base + j)
            for j in range(n):
                yield from load_v(base + j)
                if j + 2 < n:
                    yield from load_k(base + j + 2)
        yield ('arrive', done)

    def score_issuer():
        for it, n in enumerate(items):
            qb = it & 1
            yield ('wait', (q_ready if rope else q_full)[qb], it >> 1)
            for j in range(n):
                gi = first[it] + j
                s, sb = gi % nk, gi & 1
                yield ('wait', (k_ready if rope and wait_rotated_k else k_full)[s], gi // nk)
                if gi >= 2:
                    yield ('wait', s_free[sb], (gi >> 1) - 1)

                def ex(gi=gi, s=s, it=it, qb=qb):
                    assert st['q_item'][qb] == it and st['k_land'][s] == gi
                    if rope:
                        assert st['q_rot'][qb] == it, "score MMA read an unrotated Q"
                        assert st['k_rot'][s] == gi, "score MMA read an unrotated K"
                    assert all(v >= gi - 2 for v in st['s_read'].values()), "S overwritten before it was read"
                    st['s_exec'] = gi
                yield ('mma', 'S', ex)
                yield ('commit', s_full[sb])
                yield ('commit', k_empty[s])
                if j == n - 1:
                    yield ('commit', q_empty[qb])
        yield ('commit', drain)
        yield ('wait', drain, 0)
        yield ('arrive', done)

    def pv_issuer():
        for it, n in enumerate(items):
            ob = it % no
            if it >= no:
                yield ('wait', o_free[ob], (it - no) // no)
            for j in range(n):
                gi = first[it] + j
                pb, sp = gi & 1, gi % nv
                yield ('wait', p_full[pb], gi >> 1)
                yield ('wait', v_full[sp], gi // nv)

                def ex(gi=gi, sp=sp, it=it, ob=ob, j=j):
                    assert all(v >= gi for v in st['p_wr'].values()), "PV before P written"
                    assert all(v >= gi for v in st['o_scaled'].values()), "PV before O rescaled"
                    assert st['v_land'][sp] == gi
                    if j == 0:
                        assert all(v >= it - no for v in st['o_read'].values()), \
                            "PV overwrote O before the epilogue read it"
                        st['o_item'][ob] = it
                    st['pv_exec'] = gi
                yield ('mma', 'PV', ex)
                yield ('commit', pv_done[pb])
                yield ('commit', v_empty[sp])
        yield ('commit', drain2)
        yield ('wait', drain2, 0)
        yield ('arrive', done)

    def softmax(w):
        for it, n in enumerate(items):
            ob, qb = it % no, it & 1
            for j in range(n):
                gi = first[it] + j
                sb = pb = gi & 1
                yield ('wait', s_full[sb], gi >> 1)
                assert st['s_exec'] >= gi
                st['s_read'][w] = gi
                yield ('arrive', s_free[sb])
                if gi >= 2:
                    yield ('wait', pv_done[pb], (gi - 2) >> 1)
                assert st['pv_exec'] >= gi - 2, "P written over a P the PV had not read"
                st['p_wr'][w] = gi
                if j >= 1 and rng.random() < 0.5:
                    if rescale_wait:
                        yield ('wait', pv_done[pb ^ 1], (gi - 1) >> 1)
                    assert st['pv_exec'] >= gi - 1, "O rescaled under a PV"
                st['o_scaled'][w] = gi
                yield ('arrive', p_full[pb])
            lg = last[it]
            yield ('wait', pv_done[lg & 1], lg >> 1)
            assert st['pv_exec'] >= lg and st['o_item'][ob] == it
            assert st['s_exec'] >= lg, "output staged over a Q tile a score MMA still reads"
            assert st['q_item'][qb] == it
            st['o_read'][w] = it
            st['q_staged'][qb] = it
            yield ('arrive', o_free[ob])
            yield ('arrive', o_staged)
            if w == 0:
                yield ('wait', o_staged, it)

                def read(it=it, qb=qb):
                    assert st['q_staged'][qb] == it and st['q_item'][qb] == it
                    st['store_read'][qb] = it
                yield ('tma', Bar("store", 1), read)
                yield ('until', lambda it=it, qb=qb: st['store_read'][qb] == it)
                if store_release:
                    yield ('arrive', q_empty[qb])
        yield ('arrive', done)

    def rotator(w):
        for it, n in enumerate(items):
            qb = it & 1
            yield ('wait', q_full[qb], it >> 1)
            assert st['q_item'][qb] == it
            if w == 0:
                st['q_rot'][qb] = it
            yield ('arrive', q_ready[qb])
            for j in range(n):
                gi = first[it] + j
                s = gi % nk
                yield ('wait', k_full[s], gi // nk)
                assert st['k_land'][s] == gi
                if w == 0:
                    st['k_rot'][s] = gi
                yield ('arrive', k_ready[s])
        yield ('arrive', done)

    def teardown():
        yield ('wait', done, 0)
        assert not sim.pipe and not sim.tma, "CTA exits with MMAs or copies in flight"

    sim.add('producer', producer())
    sim.add('score', score_issuer())
    sim.add('pv', pv_issuer())
    for w in W:
        sim.add(f'sm{w}', softmax(w))
    if rope:
        for w in W:
            sim.add(f'rot{w}', rotator(w))
    sim.add('teardown', teardown())
    sim.run()
