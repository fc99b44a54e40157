"""Discrete-event model of the mbarrier protocols of the split algorithm's dQ kernel and of
the forward kernel, for the CPU tests in test_protocol_cpu.py.

Each role of a kernel is a Python generator that yields the operations its CUDA code
performs, in program order: barrier waits and arrivals, tensor-memory / shared-memory
reads and writes, asynchronous copies (TMA) and asynchronous products (tcgen05.mma) with
their commits.  A scheduler interleaves the roles, the copies and the products of each
issuing thread (which execute in issue order) at random, and checks what the hardware
does not:

* a wait for phase k of a barrier passes when the barrier's phase parity differs from
  k's (mbarrier.try_wait.parity); it is an error if that happens before phase k has
  completed (the wait would pass early), or if phase k + 1 had already completed when the
  wait was first reached (the parity would alias a later phase);
* an arrival meant for phase k while the barrier is still collecting another phase is an
  error (it would complete the wrong phase);
* every buffer holds a tag naming the data in it; a read that finds another tag than the
  one the code relies on is a data race;
* no role may be left waiting (deadlock).

The models restate the kernels' barrier and buffer logic; they import nothing from the
package and run no GPU code.
"""

import itertools
import random


class ProtocolError(AssertionError):
    pass


class Sim:
    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.bars = {}
        self.bufs = {}
        self.agents = {}   # name -> [generator, pending request, first evaluation done]
        self.pipes = {}    # issuing thread -> list of products / commits in issue order
        self.copies = []   # asynchronous copies in flight: (barrier, phase, writes)

    def barrier(self, name, count=1):
        self.bars[name] = {"count": count, "arrived": 0, "done": 0}

    def add(self, name, gen):
        self.agents[name] = [gen, None, False]

    # ------------------------------------------------------------------ primitives
    def _arrive(self, bar, k, who):
        b = self.bars[bar]
        if b["done"] != k:
            raise ProtocolError(f"{who}: arrival for phase {k} of {bar} while it collects "
                                f"phase {b['done']}")
        b["arrived"] += 1
        if b["arrived"] == b["count"]:
            b["arrived"] = 0
            b["done"] += 1

    def _read(self, buf, tag, who):
        cur = self.bufs.get(buf)
        if cur != tag:
            raise ProtocolError(f"{who}: reads {buf} expecting {tag}, finds {cur}")

    def _wait_passes(self, bar, k):
        return (self.bars[bar]["done"] & 1) != (k & 1)

    # ------------------------------------------------------------------ roles
    def _runnable(self, name):
        gen, req, _ = self.agents[name]
        if req is None:
            return True
        return req[0] != "wait" or self._wait_passes(req[1], req[2])

    def _step_agent(self, name):
        st = self.agents[name]
        if st[1] is None:
            try:
                st[1] = next(st[0])
            except StopIteration:
                del self.agents[name]
                return
            st[2] = False
        req = st[1]
        kind = req[0]
        if kind == "wait":
            _, bar, k = req
            done = self.bars[bar]["done"]
            if not st[2]:
                st[2] = True
                if done >= k + 2:
                    raise ProtocolError(f"{name}: waits for phase {k} of {bar}, which has "
                                        f"completed {done} phases (parity aliases)")
            if not self._wait_passes(bar, k):
                return  # blocked
            if done < k + 1:
                raise ProtocolError(f"{name}: wait for phase {k} of {bar} passes with only "
                                    f"{done} phases completed")
        elif kind == "arrive":
            self._arrive(req[1], req[2], name)
        elif kind == "read":
            self._read(req[1], req[2], name)
        elif kind == "write":
            self.bufs[req[1]] = req[2]
        elif kind == "copy":  # (copy, barrier, phase, writes)
            self.copies.append((req[1], req[2], req[3]))
        elif kind in ("mma", "commit"):  # (mma, thread, reads, writes) / (commit, thread, bar, k)
            self.pipes.setdefault(req[1], []).append(req)
        else:
            raise ValueError(kind)
        st[1] = None

    # ------------------------------------------------------------------ asynchronous work
    def _step_pipe(self, thread):
        op = self.pipes[thread].pop(0)
        if op[0] == "mma":
            for buf, tag in op[2]:
                self._read(buf, tag, f"product of {thread}")
            for buf, tag in op[3]:
                self.bufs[buf] = tag
        else:
            self._arrive(op[2], op[3], f"commit of {thread}")

    def _step_copy(self, i):
        bar, k, writes = self.copies.pop(i)
        for buf, tag in writes:
            self.bufs[buf] = tag
        self._arrive(bar, k, "copy")

    def run(self, max_steps=2_000_000):
        for _ in range(max_steps):
            choices = [("a", n) for n in list(self.agents) if self._runnable(n)]
            choices += [("p", t) for t, q in self.pipes.items() if q]
            choices += [("c", i) for i in range(len(self.copies))]
            if not choices:
                if self.agents:
                    blocked = {n: st[1] for n, st in self.agents.items()}
                    raise ProtocolError(f"deadlock: {blocked}")
                return
            kind, x = self.rng.choice(choices)
            if kind == "a":
                self._step_agent(x)
            elif kind == "p":
                self._step_pipe(x)
            else:
                self._step_copy(x)
        raise ProtocolError("step limit")


# ============================================================================ dQ kernel

def dq_kernel(sim, totals, warps=2, kst=3, dsfull_per_parity=True):
    """The split algorithm's persistent dQ kernel on one CTA: `totals[t]` key tiles for the
    t-th query tile it claims.  `warps` compute warps stand for the eight (each arrives on
    the per-step barriers once).  dsfull_per_parity=False restores the single dS-full
    barrier the kernel had before (one barrier for every step)."""
    W = warps
    for b in ["QDO", "QDOE", "DPFULL", "ACC"]:
        sim.barrier(b)
    sim.barrier("DPFREE", W)
    for s in range(kst):
        sim.barrier(f"KF{s}")
        sim.barrier(f"KE{s}")
    for s in range(2):
        sim.barrier(f"VF{s}")
        sim.barrier(f"VE{s}")
        sim.barrier(f"SF{s}")
        sim.barrier(f"TF{s}")
        sim.barrier(f"TE{s}", 1 + W)
    if dsfull_per_parity:
        sim.barrier("DSFULL0", W)
        sim.barrier("DSFULL1", W)
    else:
        sim.barrier("DSFULL", W)
    slots = [None, None]
    ticket = itertools.count()

    def ds_bar(j):
        return (f"DSFULL{j & 1}", j >> 1) if dsfull_per_parity else ("DSFULL", j)

    def producer():
        q_loads = 0
        j = 0
        for T in itertools.count():
            slot = T & 1
            if T >= 2:
                yield ("wait", f"TE{slot}", (T - 2) >> 1)
            tile = next(ticket)
            if tile >= len(totals):
                tile = -1
            slots[slot] = tile
            yield ("arrive", f"TF{slot}", T >> 1)
            if tile < 0:
                return
            total = totals[tile]
            if total == 0:
                continue
            if q_loads > 0:
                yield ("wait", "QDOE", q_loads - 1)
            yield ("copy", "QDO", q_loads, [("Q", ("Q", tile))])
            q_loads += 1
            for _ in range(total):
                ks = j % kst
                if j >= kst:
                    yield ("wait", f"KE{ks}", (j - kst) // kst)
                yield ("copy", f"KF{ks}", j // kst, [(f"K{ks}", ("K", j))])
                vs = j & 1
                if j >= 2:
                    yield ("wait", f"VE{vs}", (j - 2) >> 1)
                yield ("copy", f"VF{vs}", j >> 1, [(f"V{vs}", ("V", j))])
                j += 1

    def mma():
        def issue_s(j, tile):
            ks = j % kst
            yield ("wait", f"KF{ks}", j // kst)
            yield ("mma", "mma", [("Q", ("Q", tile)), (f"K{ks}", ("K", j))],
                   [(f"S{j & 1}.{p}", ("S", j)) for p in range(W)])
            yield ("commit", "mma", f"SF{j & 1}", j >> 1)

        def issue_dp(j, tile):
            vs = j & 1
            yield ("wait", f"VF{vs}", j >> 1)
            yield ("mma", "mma", [("Q", ("Q", tile)), (f"V{vs}", ("V", j))],
                   [(f"DP.{p}", ("dP", j)) for p in range(W)])
            yield ("commit", "mma", "DPFULL", j)
            yield ("commit", "mma", f"VE{vs}", j >> 1)

        j0 = tq = 0
        for T in itertools.count():
            slot = T & 1
            yield ("wait", f"TF{slot}", T >> 1)
            tile = slots[slot]
            yield ("arrive", f"TE{slot}", T >> 1)
            if tile < 0:
                return
            total = totals[tile]
            if total == 0:
                continue
            yield ("wait", "QDO", tq)
            if j0 > 0:
                yield ("wait", "DPFREE", j0 - 1)
            yield from issue_s(j0, tile)
            yield from issue_dp(j0, tile)
            if total == 1:
                yield ("commit", "mma", "QDOE", tq)
            if total > 1:
                yield from issue_s(j0 + 1, tile)
            for it in range(total):
                j = j0 + it
                if it + 1 < total:
                    yield ("wait", "DPFREE", j)
                    yield from issue_dp(j + 1, tile)
                    if it + 2 == total:
                        yield ("commit", "mma", "QDOE", tq)
                yield ("wait",) + ds_bar(j)
                ks = j % kst
                reads = [(f"S{j & 1}.{p}", ("dS", j)) for p in range(W)] + [(f"K{ks}", ("K", j))]
                if it > 0:
                    reads += [(f"DQ.{p}", ("dQ", tile, it - 1)) for p in range(W)]
                yield ("mma", "mma", reads, [(f"DQ.{p}", ("dQ", tile, it)) for p in range(W)])
                yield ("commit", "mma", f"KE{ks}", j // kst)
                if it + 2 < total:
                    yield from issue_s(j + 2, tile)
            yield ("commit", "mma", "ACC", tq)
            j0 += total
            tq += 1

    def compute(p):
        j0 = tq = 0
        for T in itertools.count():
            slot = T & 1
            yield ("wait", f"TF{slot}", T >> 1)
            tile = slots[slot]
            yield ("arrive", f"TE{slot}", T >> 1)
            if tile < 0:
                return
            total = totals[tile]
            for it in range(total):
                j = j0 + it
                b = j & 1
                yield ("wait", f"SF{b}", j >> 1)
                yield ("wait", "DPFULL", j)
                yield ("read", f"DP.{p}", ("dP", j))
                yield ("arrive", "DPFREE", j)
                yield ("read", f"S{b}.{p}", ("S", j))
                yield ("write", f"S{b}.{p}", ("dS", j))
                yield ("arrive",) + ds_bar(j)
            if total > 0:
                yield ("wait", "ACC", tq)
                yield ("read", f"DQ.{p}", ("dQ", tile, total - 1))
                j0 += total
                tq += 1

    sim.add("producer", producer())
    sim.add("mma", mma())
    for p in range(W):
        sim.add(f"compute{p}", compute(p))


# ============================================================================ forward kernel

def forward_kernel(sim, nvis, warps=2, kst=2, vst=2, rescale=0.3, two_issuers=True,
                   s_waits_pd=True):
    """The forward kernel on one CTA: `nvis[i]` visible key tiles for its i-th item.
    `warps` softmax warps stand for the eight (each arrives on the P-full, O-empty and
    O-staged barriers once).  A softmax warp rescales its O rows before a key tile's P V
    product with probability `rescale` (seeded), after waiting for the previous product.
    two_issuers=False issues both kinds of product from one thread (the kernel's earlier
    form).  s_waits_pd=False drops the score products' wait for the P V product whose P
    they overwrite: safe for one issuing thread (issue order), a race for two."""
    W = warps
    rng = random.Random(sim.rng.random())
    for s in range(2):
        for b in ["QF", "QE", "SF", "PD", "ACC"]:
            sim.barrier(f"{b}{s}")
        for b in ["PF", "OE", "OS"]:
            sim.barrier(f"{b}{s}", W)
    for s in range(kst):
        sim.barrier(f"KF{s}")
        sim.barrier(f"KE{s}")
    for s in range(vst):
        sim.barrier(f"VF{s}")
        sim.barrier(f"VE{s}")
    sim.barrier("NB", W)  # the softmax warps' per-item named barrier, as a rendezvous
    resc = {(x, p): rng.random() < rescale for x in range(sum(nvis)) for p in range(W)}

    def k_producer():
        qn = c = 0
        for item, n in enumerate(nvis):
            if n == 0:
                continue
            qb = qn & 1
            if qn >= 2:
                yield ("wait", f"QE{qb}", (qn - 2) >> 1)
                yield ("wait", f"OS{qb}", (qn - 2) >> 1)
            yield ("copy", f"QF{qb}", qn >> 1, [(f"Q{qb}.{p}", ("Q", item)) for p in range(W)])
            for _ in range(n):
                ks = c % kst
                if c >= kst:
                    yield ("wait", f"KE{ks}", (c - kst) // kst)
                yield ("copy", f"KF{ks}", c // kst, [(f"K{ks}", ("K", c))])
                c += 1
            qn += 1

    def v_producer():
        c = 0
        for n in nvis:
            for _ in range(n):
                vs = c % vst
                if c >= vst:
                    yield ("wait", f"VE{vs}", (c - vst) // vst)
                yield ("copy", f"VF{vs}", c // vst, [(f"V{vs}", ("V", c))])
                c += 1

    def issue_s(thread, x, item, qb):
        ks = x % kst
        yield ("wait", f"KF{ks}", x // kst)
        yield ("mma", thread, [(f"Q{qb}.{p}", ("Q", item)) for p in range(W)] + [(f"K{ks}", ("K", x))],
               [(f"S{x & 1}.{p}", ("S", x)) for p in range(W)])
        yield ("commit", thread, f"SF{x & 1}", x >> 1)
        yield ("commit", thread, f"KE{ks}", x // kst)

    def issue_pv(thread, x, t, item, on, qb):
        yield ("wait", f"PF{x & 1}", x >> 1)
        if t == 0 and on >= 2:
            yield ("wait", f"OE{qb}", (on - 2) >> 1)
        vs = x % vst
        yield ("wait", f"VF{vs}", x // vst)
        reads = [(f"S{x & 1}.{p}", ("P", x)) for p in range(W)] + [(f"V{vs}", ("V", x))]
        if t > 0:
            reads += [(f"O{qb}.{p}", ("Or" if resc[(x, p)] else "O", item, t - 1)) for p in range(W)]
        yield ("mma", thread, reads, [(f"O{qb}.{p}", ("O", item, t)) for p in range(W)])
        yield ("commit", thread, f"VE{vs}", x // vst)
        yield ("commit", thread, f"PD{x & 1}", x >> 1)

    def s_issuer():
        g = on = 0
        for item, n in enumerate(nvis):
            if n == 0:
                continue
            qb = on & 1
            yield ("wait", f"QF{qb}", on >> 1)
            for t in range(n):
                x = g + t
                if x >= 2 and s_waits_pd:
                    yield ("wait", f"PD{x & 1}", (x - 2) >> 1)
                yield from issue_s("s", x, item, qb)
            yield ("commit", "s", f"QE{qb}", on >> 1)
            g += n
            on += 1

    def pv_issuer():
        g = on = 0
        for item, n in enumerate(nvis):
            if n == 0:
                continue
            qb = on & 1
            for t in range(n):
                yield from issue_pv("pv", g + t, t, item, on, qb)
            yield ("commit", "pv", f"ACC{qb}", on >> 1)
            g += n
            on += 1

    def one_issuer():
        g = on = 0
        for item, n in enumerate(nvis):
            if n == 0:
                continue
            qb = on & 1

            def s_after_pd(x):
                if x >= 2 and s_waits_pd:
                    yield ("wait", f"PD{x & 1}", (x - 2) >> 1)
                yield from issue_s("mma", x, item, qb)

            yield ("wait", f"QF{qb}", on >> 1)
            yield from s_after_pd(g)
            if n > 1:
                yield from s_after_pd(g + 1)
            for t in range(n):
                x = g + t
                yield from issue_pv("mma", x, t, item, on, qb)
                if t + 2 < n:
                    yield from s_after_pd(x + 2)
            yield ("commit", "mma", f"QE{qb}", on >> 1)
            yield ("commit", "mma", f"ACC{qb}", on >> 1)
            g += n
            on += 1

    def softmax(p):
        g = on = 0
        os_pend = None  # (buffer, phase, item) whose staged O this warp's store may still read

        def flush():
            nonlocal os_pend
            if os_pend is not None:
                qb_, ph, it_ = os_pend
                # bulk_wait_read_all: the store has read the staged rows
                yield ("read", f"Q{qb_}.{p}", ("Ostage", it_))
                yield ("arrive", f"OS{qb_}", ph)
                os_pend = None

        for item, n in enumerate(nvis):
            qb = on & 1
            for t in range(n):
                x = g + t
                b = x & 1
                yield ("wait", f"SF{b}", x >> 1)
                yield ("read", f"S{b}.{p}", ("S", x))
                if t > 0 and resc[(x, p)]:
                    yield ("wait", f"PD{(x - 1) & 1}", (x - 1) >> 1)
                    yield ("read", f"O{qb}.{p}", ("O", item, t - 1))
                    yield ("write", f"O{qb}.{p}", ("Or", item, t - 1))
                yield ("write", f"S{b}.{p}", ("P", x))
                yield ("arrive", f"PF{b}", x >> 1)
                if t == 0:
                    yield from flush()
            if n > 0:
                yield ("wait", f"ACC{qb}", on >> 1)
            yield ("arrive", "NB", item)
            yield ("wait", "NB", item)
            yield from flush()
            if n > 0:
                yield ("read", f"O{qb}.{p}", ("O", item, n - 1))
                yield ("write", f"Q{qb}.{p}", ("Ostage", item))
                yield ("arrive", f"OE{qb}", on >> 1)
                os_pend = (qb, on >> 1, item)
                g += n
                on += 1
        yield from flush()

    sim.add("k_producer", k_producer())
    sim.add("v_producer", v_producer())
    if two_issuers:
        sim.add("s_issuer", s_issuer())
        sim.add("pv_issuer", pv_issuer())
    else:
        sim.add("mma", one_issuer())
    for p in range(W):
        sim.add(f"softmax{p}", softmax(p))


# ============================================================================ main kernel

def main_kernel(sim, tiles, warps=2, drains=2, kst=1, issuers=1, do_waits_dp=True,
                ordered=False):
    """The fused backward's main kernel on one CTA (unordered mode): `tiles[t]` steps for
    the t-th key tile it claims.  `warps` compute warps stand for the eight and `drains`
    dQ-drain warps for the four.  kst: K stages (1 at Dp = 96 / 128, 2 at Dp <= 80).
    issuers=2 models a split of the MMA issue over two threads (S and dP from one, dV, dK
    and dQ from the other) with the completion waits that split needs; do_waits_dp=False
    drops the one it adds (dO is read by dP_i and dV_i, issued by different threads, so
    the producer reloads the dO buffer only once dP_i, not just dV_i, is complete).
    ordered=True adds the ordered mode's hand-over between the ordering warp and the
    drain (turn / turn-empty barriers and a two-slot turn word; the cross-CTA counter the
    ordering warp polls is outside a one-CTA model)."""
    W, D = warps, drains
    ones = ["V", "SFULL", "DPFULL", "DVDONE", "DQFULL", "DSEMPTY", "ACC", "NEXT", "VEMPTY"]
    for b in ones + [f"K{s}" for s in range(kst)] + [f"KEMPTY{s}" for s in range(kst)]:
        sim.barrier(b)
    for s in range(2):
        sim.barrier(f"QF{s}")
        sim.barrier(f"QE{s}")
        sim.barrier(f"TF{s}")
        sim.barrier(f"TE{s}", 1 + issuers + D + W + (1 if ordered else 0))
    sim.barrier("DOF")
    sim.barrier("DOE")
    for b in ["PFULL", "DSFULL", "DVEMPTY", "DKEMPTY"]:
        sim.barrier(b, W)
    sim.barrier("DQEMPTY", D)
    sim.barrier("TURN")
    sim.barrier("TURNE")
    ring = [None, None]
    ticket = itertools.count()

    def scheduler():
        for t in itertools.count():
            if t >= 1:
                yield ("wait", "NEXT", t - 1)
            if t >= 2:
                yield ("wait", f"TE{t & 1}", (t - 2) >> 1)
            tk = next(ticket)
            ring[t & 1] = (tk, tiles[tk]) if tk < len(tiles) else None
            yield ("arrive", f"TF{t & 1}", t >> 1)
            if ring[t & 1] is None:
                return

    def k_stage(kt):
        return (kt & 1, kt >> 1) if kst == 2 else (0, kt)

    def producer():
        git = nk = nv = 0
        for t in itertools.count():
            yield ("wait", f"TF{t & 1}", t >> 1)
            d = ring[t & 1]
            yield ("arrive", f"TE{t & 1}", t >> 1)
            if d is None:
                return
            tk, total = d
            if total == 0:
                yield ("arrive", "NEXT", t)
                continue

            def load_k():
                nonlocal nk
                ks, ph = k_stage(nk)
                nk += 1
                yield ("copy", f"K{ks}", ph, [(f"Ks{ks}", ("K", tk))])

            def load_v():
                nonlocal nv
                nv += 1
                yield ("copy", "V", nv - 1, [("Vs", ("V", tk))])

            kv_busy = nk > 0
            if kst == 2 and kv_busy:
                if nk >= 2:
                    yield ("wait", f"KEMPTY{nk & 1}", (nk >> 1) - 1)
                yield from load_k()
            if not kv_busy:
                yield from load_k()
                yield from load_v()
            for it in range(total):
                s = git & 1
                if it == total - 1:
                    yield ("arrive", "NEXT", t)
                if git >= 2:
                    yield ("wait", f"QE{s}", (git - 2) >> 1)
                yield ("copy", f"QF{s}", git >> 1, [(f"Q{s}", ("Q", git))])
                if it == 0 and kv_busy:
                    yield ("wait", "VEMPTY", nv - 1)
                    yield from load_v()
                if git >= 1:
                    yield ("wait", "DOE", git - 1)
                    if issuers == 2 and do_waits_dp:
                        yield ("wait", "DPFULL", git - 1)
                yield ("copy", "DOF", git, [("dO", ("dO", git))])
                if kst == 1 and it == 0 and kv_busy:
                    yield ("wait", "KEMPTY0", nk - 1)
                    yield from load_k()
                git += 1

    def mma_s(th, git, tk, ks):
        s = git & 1
        yield ("wait", f"QF{s}", git >> 1)
        yield ("mma", th, [(f"Ks{ks}", ("K", tk)), (f"Q{s}", ("Q", git))],
               [(f"S.{p}", ("S", git)) for p in range(W)])
        yield ("commit", th, "SFULL", git)

    def mma_dp(th, git, tk):
        yield ("wait", "DOF", git)
        yield ("mma", th, [("Vs", ("V", tk)), ("dO", ("dO", git))],
               [(f"DP.{p}", ("dP", git)) for p in range(W)] +
               [(f"DP.d{q}", ("dP", git)) for q in range(D)])
        yield ("commit", th, "DPFULL", git)

    def mma(role):
        # role: "all" (one issuer), "sdp" (S and dP), "rest" (dV, dK, dQ)
        git = kt = 0
        th = "mma" if role == "all" else role
        do_s = role in ("all", "sdp")
        do_rest = role in ("all", "rest")
        for t in itertools.count():
            yield ("wait", f"TF{t & 1}", t >> 1)
            d = ring[t & 1]
            yield ("arrive", f"TE{t & 1}", t >> 1)
            if d is None:
                return
            tk, total = d
            if total == 0:
                continue
            ks, kph = k_stage(kt)
            if do_s:
                if git > 0:
                    yield ("wait", "DVDONE", git - 1)
                yield ("wait", f"K{ks}", kph)
                yield from mma_s(th, git, tk, ks)
                if git > 0:
                    yield ("wait", "DQEMPTY", git - 1)
                yield ("wait", "V", kt)
                yield from mma_dp(th, git, tk)
                if total == 1:
                    yield ("commit", th, "VEMPTY", kt)
            for it in range(total):
                s = git & 1
                if do_rest:
                    yield ("wait", "PFULL", git)
                    if it == 0 and kt > 0:
                        yield ("wait", "DVEMPTY", kt - 1)
                    reads = [(f"S.{p}", ("P", git)) for p in range(W)] + [("dO", ("dO", git))]
                    if it > 0:
                        reads += [(f"DV.{p}", ("DV", kt, it - 1)) for p in range(W)]
                    yield ("mma", th, reads, [(f"DV.{p}", ("DV", kt, it)) for p in range(W)])
                    yield ("commit", th, "DOE", git)
                    yield ("commit", th, "DVDONE", git)
                if do_s and it + 1 < total:
                    yield ("wait", "DVDONE", git)
                    yield from mma_s(th, git + 1, tk, ks)
                if do_rest:
                    yield ("wait", "DSFULL", git)
                    if it == 0 and kt > 0:
                        yield ("wait", "DKEMPTY", kt - 1)
                    reads = [(f"DS.{p}", ("dS", git)) for p in range(W)] + [(f"Q{s}", ("Q", git))]
                    if it > 0:
                        reads += [(f"DK.{p}", ("DK", kt, it - 1)) for p in range(W)]
                    yield ("mma", th, reads, [(f"DK.{p}", ("DK", kt, it)) for p in range(W)])
                    yield ("commit", th, f"QE{s}", git >> 1)
                    # the dQ tile goes over the dP^T columns (all of them)
                    yield ("mma", th, [(f"DS.{p}", ("dS", git)) for p in range(W)] + [(f"Ks{ks}", ("K", tk))],
                           [(f"DP.d{q}", ("dQ", git)) for q in range(D)] +
                           [(f"DP.{p}", ("dQ", git)) for p in range(W)])
                    yield ("commit", th, "DQFULL", git)
                    yield ("commit", th, "DSEMPTY", git)
                if do_s and it + 1 < total:
                    yield ("wait", "DQEMPTY", git)
                    yield from mma_dp(th, git + 1, tk)
                    if it + 2 == total:
                        yield ("commit", th, "VEMPTY", kt)
                git += 1
            if do_rest:
                yield ("commit", th, "ACC", kt)
                yield ("commit", th, f"KEMPTY{ks}", kph)
            kt += 1

    def drain(q):
        git = 0
        for t in itertools.count():
            yield ("wait", f"TF{t & 1}", t >> 1)
            d = ring[t & 1]
            yield ("arrive", f"TE{t & 1}", t >> 1)
            if d is None:
                return
            for _ in range(d[1]):
                yield ("wait", "DQFULL", git)
                yield ("read", f"DP.d{q}", ("dQ", git))
                yield ("arrive", "DQEMPTY", git)
                if ordered and q == 0:
                    yield ("wait", "TURN", git)
                    yield ("read", f"turn{git & 1}", ("turn", git))
                    yield ("arrive", "TURNE", git)
                git += 1

    def compute(p):
        git = kt = 0
        for t in itertools.count():
            yield ("wait", f"TF{t & 1}", t >> 1)
            d = ring[t & 1]
            yield ("arrive", f"TE{t & 1}", t >> 1)
            if d is None:
                return
            total = d[1]
            for _ in range(total):
                yield ("wait", "SFULL", git)
                yield ("read", f"S.{p}", ("S", git))
                yield ("write", f"S.{p}", ("P", git))
                yield ("arrive", "PFULL", git)
                yield ("wait", "DPFULL", git)
                if git > 0:
                    yield ("wait", "DSEMPTY", git - 1)
                yield ("read", f"DP.{p}", ("dP", git))
                yield ("write", f"DS.{p}", ("dS", git))
                yield ("arrive", "DSFULL", git)
                git += 1
            if total > 0:
                yield ("wait", "DVDONE", git - 1)
                yield ("read", f"DV.{p}", ("DV", kt, total - 1))
                yield ("arrive", "DVEMPTY", kt)
                yield ("wait", "ACC", kt)
                yield ("read", f"DK.{p}", ("DK", kt, total - 1))
                yield ("arrive", "DKEMPTY", kt)
                kt += 1

    def ordering():
        git = 0
        for t in itertools.count():
            yield ("wait", f"TF{t & 1}", t >> 1)
            d = ring[t & 1]
            yield ("arrive", f"TE{t & 1}", t >> 1)
            if d is None:
                return
            for _ in range(d[1]):
                if git > 0:
                    yield ("wait", "TURNE", git - 1)
                yield ("write", f"turn{git & 1}", ("turn", git))
                yield ("arrive", "TURN", git)
                git += 1

    sim.add("scheduler", scheduler())
    if ordered:
        sim.add("ordering", ordering())
    sim.add("producer", producer())
    if issuers == 1:
        sim.add("mma", mma("all"))
    else:
        sim.add("mma_sdp", mma("sdp"))
        sim.add("mma_rest", mma("rest"))
    for q in range(D):
        sim.add(f"drain{q}", drain(q))
    for p in range(W):
        sim.add(f"compute{p}", compute(p))


# ============================================================================ dK / dV kernel

def dkdv_kernel(sim, total, warps=2, s_behind=True):
    """The split algorithm's dK/dV kernel on one CTA (one key tile, `total` steps).
    s_behind=True issues S_i+1 and dP_i+1 right behind dK_i (they overwrite P^T_i and
    dS^T_i, which dV_i and dK_i read, and the products of one thread run in issue order);
    False waits for dV_i's and dK_i's completion first (the kernel's earlier form)."""
    W = warps
    for b in ["KV", "SFULL", "DPFULL", "ACC", "DVDONE", "DKDONE"]:
        sim.barrier(b)
    for s in range(2):
        for b in ["QF", "QE", "DOF", "DOE"]:
            sim.barrier(f"{b}{s}")
    sim.barrier("PFULL", W)
    sim.barrier("DSFULL", W)

    def producer():
        if total == 0:
            return
        yield ("copy", "KV", 0, [("K", "K"), ("V", "V")])
        for it in range(total):
            s = it & 1
            if it >= 2:
                yield ("wait", f"QE{s}", (it - 2) >> 1)
            yield ("copy", f"QF{s}", it >> 1, [(f"Q{s}", ("Q", it)), (f"LSE{s}", ("lse", it))])
            if it >= 2:
                yield ("wait", f"DOE{s}", (it - 2) >> 1)
            yield ("copy", f"DOF{s}", it >> 1, [(f"dO{s}", ("dO", it))])

    def issue_s(it):
        s = it & 1
        yield ("wait", f"QF{s}", it >> 1)
        yield ("mma", "mma", [("K", "K"), (f"Q{s}", ("Q", it))], [(f"S.{p}", ("S", it)) for p in range(W)])
        yield ("commit", "mma", "SFULL", it)

    def issue_dp(it):
        s = it & 1
        yield ("wait", f"DOF{s}", it >> 1)
        yield ("mma", "mma", [("V", "V"), (f"dO{s}", ("dO", it))], [(f"DP.{p}", ("dP", it)) for p in range(W)])
        yield ("commit", "mma", "DPFULL", it)

    def mma():
        if total == 0:
            yield ("commit", "mma", "ACC", 0)
            return
        yield ("wait", "KV", 0)
        yield from issue_s(0)
        yield from issue_dp(0)
        for it in range(total):
            s = it & 1
            yield ("wait", "PFULL", it)
            reads = [(f"S.{p}", ("P", it)) for p in range(W)] + [(f"dO{s}", ("dO", it))]
            if it > 0:
                reads += [(f"DV.{p}", ("DV", it - 1)) for p in range(W)]
            yield ("mma", "mma", reads, [(f"DV.{p}", ("DV", it)) for p in range(W)])
            yield ("commit", "mma", f"DOE{s}", it >> 1)
            yield ("commit", "mma", "DVDONE", it)
            yield ("wait", "DSFULL", it)
            reads = [(f"DP.{p}", ("dS", it)) for p in range(W)] + [(f"Q{s}", ("Q", it))]
            if it > 0:
                reads += [(f"DK.{p}", ("DK", it - 1)) for p in range(W)]
            yield ("mma", "mma", reads, [(f"DK.{p}", ("DK", it)) for p in range(W)])
            yield ("commit", "mma", f"QE{s}", it >> 1)
            yield ("commit", "mma", "DKDONE", it)
            if it + 1 < total:
                if not s_behind:
                    yield ("wait", "DVDONE", it)
                yield from issue_s(it + 1)
                if not s_behind:
                    yield ("wait", "DKDONE", it)
                yield from issue_dp(it + 1)
        yield ("commit", "mma", "ACC", 0)

    def compute(p):
        for it in range(total):
            s = it & 1
            yield ("wait", "SFULL", it)
            yield ("read", f"LSE{s}", ("lse", it))
            yield ("read", f"S.{p}", ("S", it))
            yield ("write", f"S.{p}", ("P", it))
            yield ("arrive", "PFULL", it)
            yield ("wait", "DPFULL", it)
            yield ("read", f"LSE{s}", ("lse", it))  # D shares the stage with LSE2
            yield ("read", f"DP.{p}", ("dP", it))
            yield ("write", f"DP.{p}", ("dS", it))
            yield ("arrive", "DSFULL", it)
        yield ("wait", "ACC", 0)
        if total > 0:
            yield ("read", f"DK.{p}", ("DK", total - 1))
            yield ("read", f"DV.{p}", ("DV", total - 1))

    sim.add("producer", producer())
    sim.add("mma", mma())
    for p in range(W):
        sim.add(f"compute{p}", compute(p))


# ============================================================================ wide backward

def wide_bwd_kernel(sim, total, nst=2, warps=2, drains=2):
    """The wide backward kernel on one CTA (one key tile and output slice, `total` steps of
    64 queries), with one or two Q / dO stages.  dS^T is written into tensor memory over
    the dP^T columns (the A operand of dK) and into shared memory (the B operand of the
    transposed dQ product); the dQ^T columns are drained by the drain warps."""
    W, D = warps, drains
    for b in ["KV", "SF", "DPF", "DQF", "DSE", "ACC"]:
        sim.barrier(b)
    for s in range(nst):
        for b in ["QF", "QE", "DOF", "DOE"]:
            sim.barrier(f"{b}{s}")
    sim.barrier("PF", W)
    sim.barrier("DSF", W)
    sim.barrier("DQE", D)

    def producer():
        if total == 0:
            return
        yield ("copy", "KV", 0, [("K", "K"), ("V", "V")])
        for it in range(total):
            sq = it % nst
            if it >= nst:
                yield ("wait", f"QE{sq}", (it - nst) // nst)
            yield ("copy", f"QF{sq}", it // nst, [(f"Q{sq}", ("Q", it)), (f"LSE{sq}", ("lse", it))])
            if it >= nst:
                yield ("wait", f"DOE{sq}", (it - nst) // nst)
            yield ("copy", f"DOF{sq}", it // nst, [(f"dO{sq}", ("dO", it))])

    def do_s(i):
        sq = i % nst
        yield ("wait", f"QF{sq}", i // nst)
        yield ("mma", "mma", [("K", "K"), (f"Q{sq}", ("Q", i))], [(f"S.{p}", ("S", i)) for p in range(W)])
        yield ("commit", "mma", "SF", i)

    def do_dp(i):
        sq = i % nst
        yield ("wait", f"DOF{sq}", i // nst)
        yield ("mma", "mma", [("V", "V"), (f"dO{sq}", ("dO", i))], [(f"DP.{p}", ("dP", i)) for p in range(W)])
        yield ("commit", "mma", "DPF", i)

    def do_dv(i):
        sq = i % nst
        yield ("wait", "PF", i)
        reads = [(f"S.{p}", ("P", i)) for p in range(W)] + [(f"dO{sq}", ("dO", i))]
        if i > 0:
            reads += [(f"DV.{p}", ("DV", i - 1)) for p in range(W)]
        yield ("mma", "mma", reads, [(f"DV.{p}", ("DV", i)) for p in range(W)])
        yield ("commit", "mma", f"DOE{sq}", i // nst)

    def do_dk(i):
        sq = i % nst
        yield ("wait", "DSF", i)
        reads = [(f"DP.{p}", ("dS", i)) for p in range(W)] + [(f"Q{sq}", ("Q", i))]
        if i > 0:
            reads += [(f"DK.{p}", ("DK", i - 1)) for p in range(W)]
        yield ("mma", "mma", reads, [(f"DK.{p}", ("DK", i)) for p in range(W)])
        yield ("commit", "mma", f"QE{sq}", i // nst)

    def do_dq(i):
        if i >= 1:
            yield ("wait", "DQE", i - 1)
        yield ("mma", "mma", [("K", "K")] + [(f"DSs.{p}", ("dS", i)) for p in range(W)],
               [(f"DQ.{q}", ("dQ", i)) for q in range(D)])
        yield ("commit", "mma", "DQF", i)
        yield ("commit", "mma", "DSE", i)

    def mma():
        if total == 0:
            return
        yield ("wait", "KV", 0)
        if nst == 1:
            for it in range(total):
                yield from do_s(it)
                yield from do_dp(it)
                yield from do_dv(it)
                yield from do_dk(it)
                yield from do_dq(it)
        else:
            yield from do_s(0)
            yield from do_dp(0)
            for it in range(total):
                more = it + 1 < total
                yield from do_dv(it)
                if more:
                    yield from do_s(it + 1)
                yield from do_dk(it)
                if more:
                    yield from do_dp(it + 1)
                yield from do_dq(it)
        yield ("commit", "mma", "ACC", 0)

    def drain(q):
        for it in range(total):
            yield ("wait", "DQF", it)
            yield ("read", f"DQ.{q}", ("dQ", it))
            yield ("arrive", "DQE", it)

    def compute(p):
        for it in range(total):
            sq = it % nst
            yield ("wait", "SF", it)
            yield ("read", f"LSE{sq}", ("lse", it))
            yield ("read", f"S.{p}", ("S", it))
            yield ("write", f"S.{p}", ("P", it))
            yield ("arrive", "PF", it)
            yield ("wait", "DPF", it)
            if it >= 1:
                yield ("wait", "DSE", it - 1)
            yield ("read", f"LSE{sq}", ("lse", it))
            yield ("read", f"DP.{p}", ("dP", it))
            yield ("write", f"DP.{p}", ("dS", it))
            yield ("write", f"DSs.{p}", ("dS", it))
            yield ("arrive", "DSF", it)
        if total > 0:
            yield ("wait", "ACC", 0)
            yield ("read", f"DK.{p}", ("DK", total - 1))
            yield ("read", f"DV.{p}", ("DV", total - 1))

    sim.add("producer", producer())
    sim.add("mma", mma())
    for q in range(D):
        sim.add(f"drain{q}", drain(q))
    for p in range(W):
        sim.add(f"compute{p}", compute(p))
