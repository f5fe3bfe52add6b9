"""Host models of the attention kernel's work schedule and of one CTA's
mbarrier protocol (test infrastructure only; nothing here runs on a GPU).

Schedule: `dense_pieces`, `causal_pieces` and `varlen_pieces` list, for every
CTA, the pieces of work its roles walk (the kernel's `get_work`): whole tiles,
and for the balanced schedule the key-block ranges of the leftover tiles; causal
tiles longest first in snake order; packed sequences from a host-built tile
table.  The checks on it are the
kernel-independent facts: every (tile, key block) is covered exactly once, and
every TMA row and destination row lies inside its tensor.

Protocol: `run_cta` plays one CTA's roles (TMA producer, the S = QK^T issuer, the
O += PV issuer and the eight softmax warps) against mbarriers with phase
counters, the tensor pipe completing MMAs in issue order and TMA copies landing
in any order, with random timing.  Every wait states the phase it means; the
model asserts that the parity the kernel would wait on names that phase, that
neither a later phase has completed nor an earlier one is still open when the
wait starts (either way the parity would alias),
that no buffer is overwritten before its reader is done, and that the roles
finish (no deadlock).  The barrier layout follows the kernel: Q_FULL/Q_FREE per
Q buffer, S_FULL/P_FULL/P_FREE per score buffer (three; P is written over the
scores it came from), O_FINAL, O_FREE, KV_FULL/KV_FREE per ring stage, DRAIN.
"""
from __future__ import annotations

import random

BLOCK = 128
S_BUFS = 3
SOFTMAX_WARPS = 8


def ring_pos_k(j):
    """Ring position of K(j) within a piece (K0, K1, V0, K2, V1, K3, ...)."""
    return j if j < 2 else 2 * j - 1


def ring_pos_v(j, n):
    return 2 * j + 2 if j + 2 < n else n + j


def ring_item(i, n):
    """(block, is_v) of a piece's i-th ring item."""
    if n == 1:
        return 0, i == 1
    if i < 2:
        return i, False
    r = i - 2
    pairs = n - 2
    if r < 2 * pairs:
        return ((r >> 1), True) if (r & 1) == 0 else ((r >> 1) + 2, False)
    return n - 2 + (r - 2 * pairs), True


def cfg(D):
    """(Q buffers, K/V ring stages) of the kernel's configuration for head dimension D."""
    return (1, 4) if D == 128 else (2, 10)


# ------------------------------------------------------------------ schedule
def balanced_plan(tiles, n, G, min_piece=8, min_gain=16):
    """(dp_tiles, sk_iters, sk_ctas): whole waves, then the leftover tiles' key
    blocks cut into equal ranges when that saves a CTA at least
    max(min_gain, n // 8) blocks."""
    rem = tiles % G
    if rem == 0:
        return tiles, 0, 0
    sk = rem * n
    ctas = min(G, sk // min_piece)
    if ctas <= rem or n - (sk + ctas - 1) // ctas < max(min_gain, n // 8):
        return tiles, 0, 0
    return tiles - rem, sk, ctas


def dense_pieces(tiles, n, G, split=True):
    """Per CTA: [(tile, k0, nb)] in the order its roles walk them."""
    dp, sk, sk_ctas = balanced_plan(tiles, n, G) if split else (tiles, 0, 0)
    out = []
    for i in range(G):
        ps = [(t, 0, n) for t in range(i, dp, G)]
        if sk and i < sk_ctas:
            it0, it1 = sk * i // sk_ctas, sk * (i + 1) // sk_ctas
            t = it0 // n
            while it1 > it0 and t <= (it1 - 1) // n:
                lo, hi = max(it0 - t * n, 0), min(it1 - t * n, n)
                ps.append((dp + t, lo, hi - lo))
                t += 1
        out.append(ps)
    return out


def snake_unit(idx, i, G):
    return idx * G + (G - 1 - i if idx & 1 else i)


def causal_pieces(BH, n_qt, G, head_major):
    """Per CTA: [((bh, qt), 0, qt + 1)]: longest first, snake order."""
    units = BH * n_qt
    out = []
    for i in range(G):
        ps, idx = [], 0
        while True:
            u = snake_unit(idx, i, G)
            if u >= units:
                break
            if head_major:
                bh, qt = u // n_qt, n_qt - 1 - u % n_qt
            else:
                bh, qt = u % BH, n_qt - 1 - u // BH
            ps.append(((bh, qt), 0, qt + 1))
            idx += 1
        out.append(ps)
    return out


def varlen_table(seqlens, causal):
    """Tile list (sequence, query tile), longest first, ties in sequence order."""
    tiles = [(s, t) for s, L in enumerate(seqlens) for t in range((L + BLOCK - 1) // BLOCK)]
    nb = (lambda e: e[1] + 1) if causal else (lambda e: (seqlens[e[0]] + BLOCK - 1) // BLOCK)
    return sorted(tiles, key=lambda e: -nb(e))


def varlen_pieces(seqlens, H, G, causal):
    """Per CTA: [((seq, h, qt), row0, len, nb)]."""
    table = varlen_table(seqlens, causal)
    cu = [0]
    for L in seqlens:
        cu.append(cu[-1] + L)
    units = len(table) * H
    out = []
    for i in range(G):
        ps, idx = [], 0
        while True:
            u = snake_unit(idx, i, G)
            if u >= units:
                break
            t = u // H
            seq, tq = table[t]
            L = seqlens[seq]
            if causal:
                h, qt = u - t * H, tq
            else:
                nq = (L + BLOCK - 1) // BLOCK
                v = u - (t - tq) * H
                h, qt = v // nq, v % nq
            nb = qt + 1 if causal else (L + BLOCK - 1) // BLOCK
            ps.append(((seq, h, qt), cu[seq], L, nb))
            idx += 1
        out.append(ps)
    return out


# ------------------------------------------------------------------ protocol
class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.done = name, count, count, 0, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than its count"
        self._check()

    def expect_tx(self, n):
        self.tx += n
        self.arrive()

    def complete_tx(self, n):
        self.tx -= n
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count


class ProtocolError(AssertionError):
    pass


MUTATIONS = ("skip_buffer_wait", "two_buffer_parity", "skip_o_final_wait", "skip_q_free_wait",
             "skip_kv_free_wait", "early_p_signal")


def run_cta(piece_blocks, D=128, seed=0, rescale_rate=0.25, mutate=None, stall=0.85):
    """Play one CTA over pieces of the given key-block counts; raises on a
    parity alias, a buffer hazard or a deadlock.  Returns the number of steps.
    `mutate` plants one of MUTATIONS (a wait left out or a wrong parity), so
    that the tests can show the model catches it.  Each role skips a scheduling
    round with a probability of its own, drawn from [0, stall) per run (some
    warps fall well behind the others)."""
    assert mutate is None or mutate in MUTATIONS
    rnd = random.Random(seed)
    QB, NS = cfg(D)
    bars = {}

    def B(name, count=1):
        if name not in bars:
            bars[name] = Barrier(name, count)
        return bars[name]

    for i in range(QB):
        B(("QF", i)), B(("QFREE", i))
    for i in range(S_BUFS):
        B(("SF", i)), B(("PF", i), SOFTMAX_WARPS), B(("PFREE", i))
    B("OFIN"), B("OFREE", SOFTMAX_WARPS), B("DRAIN", 2)
    for s in range(NS):
        B(("KVF", s)), B(("KVFREE", s))

    events = []
    now = [0.0]
    pipe_end = [0.0]            # the tensor pipe completes MMAs in issue order
    last_mma = {"S": 0.0, "PV": 0.0}
    st = {"S": [None] * S_BUFS, "O": None, "O_issued": None, "stage": [None] * NS, "Q": [None] * QB}
    reads, writes = {}, {}

    def later(dt, fn):
        events.append((now[0] + dt, rnd.random(), fn))

    def mma(who, fn):
        t = max(now[0], pipe_end[0]) + rnd.uniform(0.2, 1.0)
        pipe_end[0] = last_mma[who] = t
        events.append((t, rnd.random(), fn))

    def commit(who, bar):
        events.append((max(now[0], last_mma[who]) + 1e-6, rnd.random(), bar.arrive))

    def wait(bar, parity, phase):
        if parity != (phase & 1):
            raise ProtocolError(f"{bar.name}: parity {parity} does not name phase {phase}")
        if bar.done < phase:
            raise ProtocolError(f"{bar.name}: wait for phase {phase} starts while phase {bar.done} is open")
        return ("wait", bar, phase)

    def producer():
        item = 0
        for u, n in enumerate(piece_blocks):
            qb = u % QB
            if u >= QB and mutate != "skip_q_free_wait":
                yield wait(B(("QFREE", qb)), (u // QB - 1) & 1, u // QB - 1)
            if st["Q"][qb] is not None and st["Q"][qb][1] != "free":
                raise ProtocolError(f"Q buffer {qb} reloaded while piece {st['Q'][qb][0]} still uses it")
            B(("QF", qb)).expect_tx(1)
            st["Q"][qb] = (u, "loading")

            def land_q(qb=qb, u=u):
                st["Q"][qb] = (u, "full")
                B(("QF", qb)).complete_tx(1)
            later(rnd.uniform(0.5, 3.0), land_q)
            for i in range(2 * n):
                blk, is_v = ring_item(i, n)
                s, rd = item % NS, item // NS
                if rd > 0 and mutate != "skip_kv_free_wait":
                    yield wait(B(("KVFREE", s)), (rd - 1) & 1, rd - 1)
                if st["stage"][s] is not None and st["stage"][s][2] != "free":
                    raise ProtocolError(f"ring stage {s} overwritten while {st['stage'][s][:2]} is in use")
                B(("KVF", s)).expect_tx(1)
                key = (u, ("V" if is_v else "K", blk))
                st["stage"][s] = key + ("loading",)

                def land(s=s, key=key):
                    st["stage"][s] = key + ("full",)
                    B(("KVF", s)).complete_tx(1)
                later(rnd.uniform(0.5, 3.0), land)
                item += 1
                yield ("step",)

    def s_issuer():
        g, item0, sb, sph = 0, 0, 0, 0
        for u, n in enumerate(piece_blocks):
            qb = u % QB
            yield wait(B(("QF", qb)), (u // QB) & 1, u // QB)
            if st["Q"][qb] != (u, "full"):
                raise ProtocolError(f"S MMA of piece {u} reads Q buffer holding {st['Q'][qb]}")
            if u > 0:
                yield wait(B("OFIN"), (u - 1) & 1, u - 1)
            for j in range(n):
                gs = g + j
                if gs >= S_BUFS and mutate != "skip_buffer_wait":
                    yield wait(B(("PFREE", sb)), sph ^ 1, gs // S_BUFS - 1)
                it = item0 + ring_pos_k(j)
                s = it % NS
                yield wait(B(("KVF", s)), (it // NS) & 1, it // NS)
                if st["stage"][s] != (u, ("K", j), "full"):
                    raise ProtocolError(f"S({u},{j}) reads stage {s} holding {st['stage'][s]}")
                if st["S"][sb] is not None and st["S"][sb][1] != "consumed":
                    raise ProtocolError(f"S({u},{j}) overwrites buffer {sb} holding {st['S'][sb]}")
                st["S"][sb] = ((u, j), "computing")

                def s_done(sb=sb, key=(u, j), s=s):
                    st["S"][sb] = (key, "full")
                    st["stage"][s] = st["stage"][s][:2] + ("free",)
                mma("S", s_done)
                commit("S", B(("SF", sb)))
                commit("S", B(("KVFREE", s)))
                if j == n - 1:
                    def q_free(qb=qb, u=u):
                        st["Q"][qb] = (u, "free")
                    mma("S", q_free)
                    commit("S", B(("QFREE", qb)))
                sb += 1
                if sb == S_BUFS:
                    sb, sph = 0, sph ^ 1
                yield ("step",)
            g += n
            item0 += 2 * n
        commit("S", B("DRAIN"))
        yield wait(B("DRAIN"), 0, 0)

    def pv_issuer():
        g, item0, pb, pph = 0, 0, 0, 0
        for u, n in enumerate(piece_blocks):
            for j in range(n):
                yield wait(B(("PF", pb)), pph, (g + j) // S_BUFS)
                if j == 0 and u > 0:
                    yield wait(B("OFREE"), (u - 1) & 1, u - 1)
                    if st["O"] != (u - 1, "read"):
                        raise ProtocolError(f"PV({u},0) overwrites O holding {st['O']}")
                it = item0 + ring_pos_v(j, n)
                s = it % NS
                yield wait(B(("KVF", s)), (it // NS) & 1, it // NS)
                if st["stage"][s] != (u, ("V", j), "full"):
                    raise ProtocolError(f"PV({u},{j}) reads stage {s} holding {st['stage'][s]}")
                if st["S"][pb] != ((u, j), "P"):
                    raise ProtocolError(f"PV({u},{j}) reads buffer {pb} holding {st['S'][pb]}")
                if j > 0 and st["O_issued"] != (u, j - 1):
                    raise ProtocolError(f"PV({u},{j}) issued after PV{st['O_issued']}")
                st["O_issued"] = (u, j)

                def pv_done(key=(u, j), pb=pb, s=s):
                    st["S"][pb] = (key, "consumed")
                    st["stage"][s] = st["stage"][s][:2] + ("free",)
                    st["O"] = (key[0], key[1], "done")
                mma("PV", pv_done)
                commit("PV", B(("PFREE", pb)))
                commit("PV", B(("KVFREE", s)))
                if j == n - 1:
                    commit("PV", B("OFIN"))
                pb += 1
                if pb == S_BUFS:
                    pb, pph = 0, pph ^ 1
                yield ("step",)
            g += n
            item0 += 2 * n
        commit("PV", B("DRAIN"))
        yield wait(B("DRAIN"), 0, 0)

    def softmax(w):
        g, sb, sph, pb, pph = 0, 0, 0, S_BUFS - 1, 1
        for u, n in enumerate(piece_blocks):
            for j in range(n):
                parity = ((g >> 1) & 1) if mutate == "two_buffer_parity" else sph
                yield wait(B(("SF", sb)), parity, g // S_BUFS)
                if st["S"][sb] not in (((u, j), "full"), ((u, j), "read")):
                    raise ProtocolError(f"softmax warp {w} reads buffer {sb} holding {st['S'][sb]} at ({u},{j})")
                reads[(sb, g)] = reads.get((sb, g), 0) + 1
                if reads[(sb, g)] == SOFTMAX_WARPS:
                    st["S"][sb] = ((u, j), "read")
                if mutate == "early_p_signal":
                    B(("PF", sb)).arrive()       # signalled before the scores are replaced by P
                yield ("step",)
                if j > 0 and rnd.random() < rescale_rate:
                    yield wait(B(("PFREE", pb)), pph, (g - 1) // S_BUFS)
                    if st["O"] != (u, j - 1, "done"):
                        raise ProtocolError(f"O rescale at ({u},{j}) sees O state {st['O']}")
                # this warp's rows of P(g) go over the scores it has read
                writes[(sb, g)] = writes.get((sb, g), 0) + 1
                if writes[(sb, g)] == SOFTMAX_WARPS:
                    if reads.get((sb, g), 0) != SOFTMAX_WARPS:
                        raise ProtocolError("P written before every warp read its scores")
                    st["S"][sb] = ((u, j), "P")
                if mutate != "early_p_signal":
                    B(("PF", sb)).arrive()
                g += 1
                pb, pph = sb, sph
                sb += 1
                if sb == S_BUFS:
                    sb, sph = 0, sph ^ 1
                yield ("step",)
            if mutate != "skip_o_final_wait":
                yield wait(B("OFIN"), u & 1, u)
            if st["O"] != (u, n - 1, "done"):
                raise ProtocolError(f"epilogue of piece {u} reads O state {st['O']}")
            reads[("O", u)] = reads.get(("O", u), 0) + 1
            if reads[("O", u)] == SOFTMAX_WARPS:
                st["O"] = (u, "read")
            B("OFREE").arrive()
            yield ("step",)

    roles = {"producer": producer(), "s_issuer": s_issuer(), "pv_issuer": pv_issuer()}
    for w in range(SOFTMAX_WARPS):
        roles[f"softmax{w}"] = softmax(w)
    blocked = {r: None for r in roles}
    p_stall = {r: rnd.uniform(0.0, stall) for r in roles}
    alive = set(roles)
    steps = 0
    while alive:
        steps += 1
        progressed = False
        order = sorted(alive)
        rnd.shuffle(order)
        for r in order:
            if rnd.random() < p_stall[r]:
                progressed = True
                continue
            bw = blocked[r]
            if bw is not None:
                _, bar, k = bw
                if bar.done <= k:
                    continue
                if bar.done != k + 1:
                    raise ProtocolError(f"{r} waits for phase {k} of {bar.name}, {bar.done} have completed")
                blocked[r] = None
            try:
                ev = next(roles[r])
                progressed = True
                while ev[0] == "wait":
                    _, bar, k = ev
                    if bar.done > k:
                        if bar.done != k + 1:
                            raise ProtocolError(f"{r} waits for phase {k} of {bar.name}, {bar.done} have completed")
                        ev = next(roles[r])
                    else:
                        blocked[r] = ev
                        break
            except StopIteration:
                alive.discard(r)
        if events:
            events.sort(key=lambda e: (e[0], e[1]))
            for _ in range(rnd.randint(1, min(4, len(events)))):
                t, _, fn = events.pop(0)
                now[0] = max(now[0], t)
                fn()
            progressed = True
        if not progressed and alive:
            raise ProtocolError("deadlock: " + ", ".join(
                f"{r} on {blocked[r][1].name} phase {blocked[r][2]}" for r in sorted(alive) if blocked[r]))
    return steps
