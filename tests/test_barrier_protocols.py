"""Schedule exploration of the kernels' shared-memory barrier protocols, on
the CPU.

Each role of a kernel is restated as a Python generator that performs the
role's waits (mbarrier phase-parity waits, as the kernels issue them) and
arrivals in the kernel's order; asynchronous engines are roles of their own:
TMA loads land in any order, tensor-core products and their commits complete
in issue order. A seeded random scheduler interleaves the roles. Every buffer
records which block it holds, and every read checks -- when it starts and
when it ends -- that the buffer holds the block the reader waited for, so an
early pass through a wait (a parity that aliases an older phase) or an
overwrite of a buffer in use shows as a violation; a state where no role can
move before all are done is a deadlock.

The barrier model follows the PTX mbarrier: a phase completes when its
pending count reaches zero (then the count resets), and a wait on parity P
passes while the current phase's parity differs from P, so a phase two
rounds old is indistinguishable from the one awaited.

Covered: the TMA ring of the mma.sync decode kernel (NS stages, KG key
groups, W warps per group); the e4m3 tensor-memory kernel's K and V rings,
double-buffered S^T, single P^T buffer, O^T accumulator and q operand; and
the int8 tensor-memory kernel, whose softmax groups also widen K into
double-buffered tensor memory one block ahead and V into a single fp16
buffer. The checker must also find the known failure of an odd-depth ring
shared by two key groups, and planted parity and ordering mistakes.
"""
import random

import pytest


class Violation(AssertionError):
    pass


class Bar:
    """One mbarrier: `count` arrivals complete a phase."""

    def __init__(self, count):
        self.count, self.left, self.phase = count, count, 0

    def arrive(self, n=1):
        for _ in range(n):
            self.left -= 1
            if self.left == 0:
                self.phase += 1
                self.left = self.count

    def passed(self, parity):
        return (self.phase & 1) != parity


def run(roles, rng, max_steps=200_000):
    """Interleave generator roles at random until all finish. A role yields a
    predicate and is resumed (running atomically to its next yield) only
    while the predicate holds."""
    live = {}
    for name, gen in roles.items():
        try:
            live[name] = (gen, next(gen))
        except StopIteration:
            pass
    steps = 0
    while live:
        ready = [n for n, (_, pred) in live.items() if pred()]
        if not ready:
            raise Violation(f"deadlock: {sorted(live)} all blocked")
        name = rng.choice(ready)
        gen, _ = live[name]
        try:
            live[name] = (gen, gen.send(None))
        except StopIteration:
            del live[name]
        steps += 1
        if steps > max_steps:
            raise Violation("no progress bound reached")
    return steps


def always():
    return True


# ---------------------------------------------------------------------------
# The mma.sync decode kernel's TMA ring: one producer warp fills NS stages in
# ring order; key group kg takes the tiles whose ring sequence number is kg
# modulo KG; each of the group's W warps waits the stage's full barrier,
# reads, and arrives on its empty barrier (count W). mutate="piece_local"
# restates an earlier assignment (tiles kg, kg + KG, ... of each piece).

def decode_ring_roles(NS, KG, W, pieces, rng, mutate=None):
    full = [Bar(1) for _ in range(NS)]
    empty = [Bar(W) for _ in range(NS)]
    slot = [None] * NS
    readers = [0] * NS
    inflight = []
    state = {"issuing": True}

    def producer():
        q = 0
        for n in pieces:
            for _ in range(n):
                st = q % NS
                if q >= NS:
                    par = ((q // NS) - 1) & 1
                    if mutate == "producer_parity":
                        par ^= 1
                    yield (lambda st=st, par=par: empty[st].passed(par))
                if readers[st]:
                    raise Violation(f"tile {q} issued into stage {st} while it is read")
                slot[st] = ("loading", q)
                inflight.append((st, q))
                q += 1
                yield always
        state["issuing"] = False

    def tma():
        while True:
            yield (lambda: bool(inflight) or not state["issuing"])
            if not inflight:
                return
            st, q = inflight.pop(rng.randrange(len(inflight)))
            slot[st] = q
            full[st].arrive()

    def consumer(kg):
        base = 0
        for n in pieces:
            k0 = kg if mutate == "piece_local" else (kg - base) % KG
            for k in range(k0, n, KG):
                q = base + k
                st = q % NS
                par = (q // NS) & 1
                if mutate == "consumer_parity":
                    par ^= 1
                yield (lambda st=st, par=par: full[st].passed(par))
                if slot[st] != q:
                    raise Violation(f"group {kg} read stage {st} for tile {q}, found {slot[st]}")
                readers[st] += 1
                yield always
                if slot[st] != q:
                    raise Violation(f"stage {st} changed under the read of tile {q}")
                readers[st] -= 1
                empty[st].arrive()
            base += n

    roles = {"producer": producer(), "tma": tma()}
    for kg in range(KG):
        for w in range(W):
            roles[f"consumer{kg}.{w}"] = consumer(kg)
    return roles


def random_pieces(rng, total, max_piece):
    pieces = []
    while total > 0:
        n = rng.randint(1, min(max_piece, total))
        pieces.append(n)
        total -= n
    return pieces


# stage counts and key groups of the shipped shapes (stages a multiple of KG)
RING_SHAPES = [(ns, kg, w) for ns in (2, 3, 4, 5, 6, 8, 12) for kg in (1, 2, 3, 4) for w in (1, 2)
               if ns % kg == 0]


@pytest.mark.parametrize("NS,KG,W", RING_SHAPES)
def test_decode_ring_is_safe(NS, KG, W):
    rng = random.Random(1000 * NS + 10 * KG + W)
    for _ in range(40):
        pieces = random_pieces(rng, rng.randint(1, 40), 12)
        run(decode_ring_roles(NS, KG, W, pieces, rng), rng)


def find_violation(make_roles, seeds):
    for seed in seeds:
        rng = random.Random(seed)
        try:
            run(make_roles(rng), rng)
        except Violation as e:
            return str(e)
    return None


def test_odd_ring_shared_by_two_key_groups_is_caught():
    """Five stages, two key groups: a stage alternates between the groups, and
    a group can pass a full wait on a phase two rounds old."""
    msg = find_violation(lambda rng: decode_ring_roles(5, 2, 1, [40], rng), range(200))
    assert msg is not None and "found" in msg


def test_piece_local_key_groups_are_caught():
    """Two key groups taking tiles by their index within each piece: after a
    piece of odd length a stage passes to the other group, which can skip a
    phase of it and then pass a wait on a phase two rounds old."""
    msg = find_violation(lambda rng: decode_ring_roles(4, 2, 1, random_pieces(rng, 40, 7), rng,
                                                       "piece_local"), range(400))
    assert msg is not None and "found" in msg


@pytest.mark.parametrize("mutate", ["producer_parity", "consumer_parity"])
def test_decode_ring_planted_parity_mistakes_are_caught(mutate):
    msg = find_violation(lambda rng: decode_ring_roles(4, 1, 2, [9, 5], rng, mutate), range(200))
    assert msg is not None


# ---------------------------------------------------------------------------
# The tensor-memory kernel: per 128-key block b, a K producer and a V producer
# fill rings of NBK and NBV stages; the MMA thread issues S^T = K Q^T into S
# buffer b % 2 and, one block behind, O^T += V^T P^T, committing S-full,
# K-empty, PV-done and V-empty; NG softmax warpgroups (four warps each, one
# per 8-row tile of the unit) read S^T, arrive on S-empty, may rescale O^T,
# write their rows of the single P^T buffer after the previous product
# completed, zero V rows of tail blocks (group 0), and arrive on P-full. Per
# piece the groups write the q operand and arrive on Q-full, and read O^T at
# the end.

def tc8_roles(NBK, NBV, pieces, tails, rescales, rng, mutate=None, NG=2):
    fullk, emptyk = [Bar(1) for _ in range(NBK)], [Bar(1) for _ in range(NBK)]
    fullv, emptyv = [Bar(1) for _ in range(NBV)], [Bar(1) for _ in range(NBV)]
    sfull, sempty = [Bar(1), Bar(1)], [Bar(4 * NG), Bar(4 * NG)]
    pfull, pvdone, qfull = Bar(4 * NG), Bar(1), Bar(1)
    st = {"K": [None] * NBK, "V": [None] * NBV, "S": [None, None], "P": [None] * NG, "Q": None,
          "s_read": [0, 0], "o_busy": 0, "loading": 0}
    inflight, pipe = [], []
    meet = {"n": 0}  # rendezvous counter of the groups (the named barrier of every softmax thread)
    nblocks = sum(pieces)

    def producer(ring, nb, full, empty):
        for b in range(nblocks):
            s = b % nb
            if b >= nb:
                yield (lambda s=s, par=((b // nb) - 1) & 1: empty[s].passed(par))
            st[ring][s] = ("loading", b)
            inflight.append((ring, s, b))
            yield always

    def tma():
        while True:
            yield (lambda: bool(inflight) or st["loading"] == 2)
            if not inflight:
                return
            ring, s, b = inflight.pop(rng.randrange(len(inflight)))
            st[ring][s] = b
            (fullk if ring == "K" else fullv)[s].arrive()

    def producers_done(gen):
        yield from gen
        st["loading"] += 1

    def check(cond, what):
        if not cond:
            raise Violation(what)

    def mma():
        bq = 0
        for p, nblk in enumerate(pieces):
            yield (lambda par=p & 1: qfull.passed(par))
            for i in range(nblk + 1):
                if i < nblk:
                    b = bq + i
                    sk, sb = b % NBK, b & 1
                    yield (lambda sk=sk, par=(b // NBK) & 1: fullk[sk].passed(par))
                    if b >= 2:
                        par = ((b >> 1) - 1) & 1
                        if mutate == "sempty_parity":
                            par ^= 1
                        yield (lambda sb=sb, par=par: sempty[sb].passed(par))
                    check(st["K"][sk] == b and st["Q"] == p and st["s_read"][sb] == 0,
                          f"S^T of block {b} issued on a wrong K / q operand or a busy S buffer")
                    st["S"][sb] = ("computing", b)
                    pipe.append(("QK", b, sk, sb, p))
                    pipe.append(("commit", sfull[sb]))
                    pipe.append(("commit", emptyk[sk]))
                if i >= 1:
                    b = bq + i - 1
                    sv = b % NBV
                    yield (lambda sv=sv, par=(b // NBV) & 1: fullv[sv].passed(par))
                    yield (lambda par=b & 1: pfull.passed(par))
                    check(st["V"][sv] == ("zeroed", b) or st["V"][sv] == b,
                          f"P.V of block {b} issued on V stage holding {st['V'][sv]}")
                    check(st["P"] == [b] * NG and st["o_busy"] == 0,
                          f"P.V of block {b} issued on P^T {st['P']} or a busy O^T")
                    if mutate == "early_v_release":
                        pipe.append(("commit", emptyv[sv]))
                    pipe.append(("PV", b, sv))
                    pipe.append(("commit", pvdone))
                    if mutate != "early_v_release":
                        pipe.append(("commit", emptyv[sv]))
                yield always
            bq += nblk

    def tensor_pipe():
        while True:
            yield (lambda: bool(pipe) or mma_done["v"])
            if not pipe:
                return
            op = pipe.pop(0)
            if op[0] == "commit":
                op[1].arrive()
            elif op[0] == "QK":
                _, b, sk, sb, p = op
                check(st["K"][sk] == b and st["Q"] == p, f"S^T of block {b} read a changed operand")
                check(st["s_read"][sb] == 0, f"S^T of block {b} written while S buffer {sb} is read")
                st["S"][sb] = b
            else:
                _, b, sv = op
                check(st["V"][sv] in (b, ("zeroed", b)) and st["P"] == [b] * NG and st["o_busy"] == 0,
                      f"P.V of block {b} read a changed operand or a busy O^T")

    mma_done = {"v": False}

    def mma_role():
        yield from mma()
        mma_done["v"] = True

    def rendezvous(target):
        meet["n"] += 1
        yield (lambda: meet["n"] >= target)

    def softmax(g):
        bq, meets = 0, 0
        for p, nblk in enumerate(pieces):
            # q set-up: the previous piece's S^T products are all complete
            check(not any(op[0] == "QK" for op in pipe), f"q of piece {p} written under an S^T product")
            if g == 0:
                st["Q"] = p
            meets += NG
            yield from rendezvous(meets)
            if g == 0:
                qfull.arrive()
            for i in range(nblk):
                b = bq + i
                sb, sv = b & 1, b % NBV
                yield (lambda sb=sb, par=(b >> 1) & 1: sfull[sb].passed(par))
                check(st["S"][sb] == b, f"group {g} read S buffer {sb} for block {b}: {st['S'][sb]}")
                st["s_read"][sb] += 1
                yield always
                check(st["S"][sb] == b, f"S buffer {sb} changed under block {b}")
                st["s_read"][sb] -= 1
                sempty[sb].arrive(4)
                if b >= 1 and mutate != "skip_pv_wait":
                    yield (lambda par=(b - 1) & 1: pvdone.passed(par))
                if rescales[b] and i > 0:
                    check(not any(op[0] == "PV" for op in pipe), f"O^T rescaled under a P.V product")
                    st["o_busy"] += 1
                    yield always
                    st["o_busy"] -= 1
                check(not any(op[0] == "PV" for op in pipe), f"P^T of block {b} written under a P.V product")
                st["P"][g] = b
                if g == 0 and tails[b]:
                    yield (lambda sv=sv, par=(b // NBV) & 1: fullv[sv].passed(par))
                    check(st["V"][sv] == b, f"tail rows of block {b} zeroed in V stage holding {st['V'][sv]}")
                    st["V"][sv] = ("zeroed", b)
                pfull.arrive(4)
                yield always
            bq += nblk
            # epilogue: O^T once the piece's last product is done
            yield (lambda par=(bq - 1) & 1: pvdone.passed(par))
            check(not any(op[0] == "PV" for op in pipe), "O^T read under a P.V product")
            st["o_busy"] += 1
            yield always
            st["o_busy"] -= 1
            meets += NG
            yield from rendezvous(meets)

    roles = {"K": producers_done(producer("K", NBK, fullk, emptyk)),
             "V": producers_done(producer("V", NBV, fullv, emptyv)), "tma": tma(), "mma": mma_role(),
             "pipe": tensor_pipe()}
    for g in range(NG):
        roles[f"softmax{g}"] = softmax(g)
    return roles


def tc8_case(rng, NBK, NBV, mutate=None, NG=2):
    pieces = [rng.randint(1, 6) for _ in range(rng.randint(1, 4))]
    n = sum(pieces)
    tails, rescales = [rng.random() < 0.3 for _ in range(n)], [rng.random() < 0.3 for _ in range(n)]
    return tc8_roles(NBK, NBV, pieces, tails, rescales, rng, mutate, NG)


@pytest.mark.parametrize("NG", [2, 3, 4])  # softmax groups = 8-row tiles of a unit
@pytest.mark.parametrize("NBK,NBV", [(2, 3), (4, 5)])  # D = 256, D = 128
def test_tensor_memory_kernel_protocol_is_safe(NBK, NBV, NG):
    for seed in range(200):
        rng = random.Random(7000 + 10 * NBK + 1000 * NG + seed)
        run(tc8_case(rng, NBK, NBV, NG=NG), rng)


@pytest.mark.parametrize("mutate", ["skip_pv_wait", "sempty_parity", "early_v_release"])
def test_tensor_memory_kernel_planted_mistakes_are_caught(mutate):
    msg = find_violation(lambda rng: tc8_case(rng, 2, 3, mutate), range(400))
    assert msg is not None


# ---------------------------------------------------------------------------
# The int8 tensor-memory kernel: the same K and V producers; each of the NG
# softmax groups widens its chunks of K block b + 1 into tensor-memory buffer
# (b + 1) % 2 before reading the scores of block b (block 0 of a piece right
# after the q set-up), then releases the K stage and arrives on K-ready (count
# 4 NG per buffer); the MMA issuer computes S^T of block b once K-ready (b % 2)
# completes -- no S-empty barrier: a group arrives on K-ready of block b + 2
# only after reading S^T of block b -- and, one block behind, O^T += V16^T P^T.
# After the previous product completed, each group writes its rows of P^T,
# widens its chunks of V block b into the single fp16 buffer (releasing the V
# stage), and arrives on P-full. mutate: "kready_parity" (the issuer waits on
# the wrong phase), "skip_pv_wait" (P^T and V16 written without waiting for the
# previous product), "k_two_ahead" (K widened two blocks ahead).

def tci8_roles(NBK, NBV, pieces, rescales, rng, mutate=None, NG=2):
    fullk, emptyk = [Bar(1) for _ in range(NBK)], [Bar(4 * NG) for _ in range(NBK)]
    fullv, emptyv = [Bar(1) for _ in range(NBV)], [Bar(4 * NG) for _ in range(NBV)]
    sfull, kready = [Bar(1), Bar(1)], [Bar(4 * NG), Bar(4 * NG)]
    pfull, pvdone, qfull = Bar(4 * NG), Bar(1), Bar(1)
    st = {"K": [None] * NBK, "V": [None] * NBV, "S": [None, None], "P": [None] * NG, "Q": None,
          "KT": [[None] * NG, [None] * NG], "V16": [None] * NG, "s_read": [0, 0], "o_busy": 0,
          "loading": 0}
    inflight, pipe = [], []
    meet = {"n": 0}
    nblocks = sum(pieces)
    mma_done = {"v": False}
    ahead = 2 if mutate == "k_two_ahead" else 1

    def check(cond, what):
        if not cond:
            raise Violation(what)

    def producer(ring, nb, full, empty):
        for b in range(nblocks):
            s = b % nb
            if b >= nb:
                yield (lambda s=s, par=((b // nb) - 1) & 1: empty[s].passed(par))
            st[ring][s] = ("loading", b)
            inflight.append((ring, s, b))
            yield always

    def producers_done(gen):
        yield from gen
        st["loading"] += 1

    def tma():
        while True:
            yield (lambda: bool(inflight) or st["loading"] == 2)
            if not inflight:
                return
            ring, s, b = inflight.pop(rng.randrange(len(inflight)))
            st[ring][s] = b
            (fullk if ring == "K" else fullv)[s].arrive()

    def mma():
        bq = 0
        for p, nblk in enumerate(pieces):
            yield (lambda par=p & 1: qfull.passed(par))
            for i in range(nblk + 1):
                if i < nblk:
                    b = bq + i
                    sb = b & 1
                    par = (b >> 1) & 1
                    if mutate == "kready_parity":
                        par ^= 1
                    yield (lambda sb=sb, par=par: kready[sb].passed(par))
                    check(st["KT"][sb] == [b] * NG and st["Q"] == p and st["s_read"][sb] == 0,
                          f"S^T of block {b} issued on K buffer {st['KT'][sb]}, a wrong q or a busy S buffer")
                    st["S"][sb] = ("computing", b)
                    pipe.append(("QK", b, sb, p))
                    pipe.append(("commit", sfull[sb]))
                if i >= 1:
                    b = bq + i - 1
                    yield (lambda par=b & 1: pfull.passed(par))
                    check(st["P"] == [b] * NG and st["V16"] == [b] * NG and st["o_busy"] == 0,
                          f"P.V of block {b} issued on P^T {st['P']}, V16 {st['V16']} or a busy O^T")
                    pipe.append(("PV", b))
                    pipe.append(("commit", pvdone))
                yield always
            bq += nblk

    def mma_role():
        yield from mma()
        mma_done["v"] = True

    def tensor_pipe():
        while True:
            yield (lambda: bool(pipe) or mma_done["v"])
            if not pipe:
                return
            op = pipe.pop(0)
            if op[0] == "commit":
                op[1].arrive()
            elif op[0] == "QK":
                _, b, sb, p = op
                check(st["KT"][sb] == [b] * NG and st["Q"] == p, f"S^T of block {b} read a changed operand")
                check(st["s_read"][sb] == 0, f"S^T of block {b} written while S buffer {sb} is read")
                st["S"][sb] = b
            else:
                _, b = op
                check(st["V16"] == [b] * NG and st["P"] == [b] * NG and st["o_busy"] == 0,
                      f"P.V of block {b} read a changed operand or a busy O^T")

    def rendezvous(target):
        meet["n"] += 1
        yield (lambda: meet["n"] >= target)

    def softmax(g):
        bq, meets = 0, 0

        def widen_k(b):
            sk = b % NBK
            yield (lambda sk=sk, par=(b // NBK) & 1: fullk[sk].passed(par))
            check(st["K"][sk] == b, f"group {g} widened K stage holding {st['K'][sk]} as block {b}")
            check(not any(op[0] == "QK" and op[2] == (b & 1) for op in pipe),
                  f"K buffer {b & 1} rewritten for block {b} under an S^T product")
            st["KT"][b & 1][g] = b
            yield always
            emptyk[sk].arrive(4)
            kready[b & 1].arrive(4)

        for p, nblk in enumerate(pieces):
            check(not any(op[0] == "QK" for op in pipe), f"q of piece {p} written under an S^T product")
            if g == 0:
                st["Q"] = p
            meets += NG
            yield from rendezvous(meets)
            if g == 0:
                qfull.arrive()
            for k in range(min(ahead, nblk)):
                yield from widen_k(bq + k)
            for i in range(nblk):
                b = bq + i
                sb, sv = b & 1, b % NBV
                if i + ahead < nblk:
                    yield from widen_k(b + ahead)
                yield (lambda sb=sb, par=(b >> 1) & 1: sfull[sb].passed(par))
                check(st["S"][sb] == b, f"group {g} read S buffer {sb} for block {b}: {st['S'][sb]}")
                st["s_read"][sb] += 1
                yield always
                check(st["S"][sb] == b, f"S buffer {sb} changed under block {b}")
                st["s_read"][sb] -= 1
                if b >= 1 and mutate != "skip_pv_wait":
                    yield (lambda par=(b - 1) & 1: pvdone.passed(par))
                if rescales[b] and i > 0:
                    check(not any(op[0] == "PV" for op in pipe), "O^T rescaled under a P.V product")
                    st["o_busy"] += 1
                    yield always
                    st["o_busy"] -= 1
                check(not any(op[0] == "PV" for op in pipe), f"P^T of block {b} written under a P.V product")
                st["P"][g] = b
                yield (lambda sv=sv, par=(b // NBV) & 1: fullv[sv].passed(par))
                check(st["V"][sv] == b, f"group {g} widened V stage holding {st['V'][sv]} as block {b}")
                check(not any(op[0] == "PV" for op in pipe), f"V16 of block {b} written under a P.V product")
                st["V16"][g] = b
                yield always
                emptyv[sv].arrive(4)
                pfull.arrive(4)
                yield always
            bq += nblk
            yield (lambda par=(bq - 1) & 1: pvdone.passed(par))
            check(not any(op[0] == "PV" for op in pipe), "O^T read under a P.V product")
            st["o_busy"] += 1
            yield always
            st["o_busy"] -= 1
            meets += NG
            yield from rendezvous(meets)

    roles = {"K": producers_done(producer("K", NBK, fullk, emptyk)),
             "V": producers_done(producer("V", NBV, fullv, emptyv)), "tma": tma(), "mma": mma_role(),
             "pipe": tensor_pipe()}
    for g in range(NG):
        roles[f"softmax{g}"] = softmax(g)
    return roles


def tci8_case(rng, NBK, NBV, mutate=None, NG=2):
    pieces = [rng.randint(1, 6) for _ in range(rng.randint(1, 4))]
    rescales = [rng.random() < 0.3 for _ in range(sum(pieces))]
    return tci8_roles(NBK, NBV, pieces, rescales, rng, mutate, NG)


@pytest.mark.parametrize("NG", [2, 3, 4])
@pytest.mark.parametrize("NBK,NBV", [(2, 2), (4, 4)])  # D = 256, D = 128
def test_int8_tensor_memory_kernel_protocol_is_safe(NBK, NBV, NG):
    for seed in range(200):
        rng = random.Random(9000 + 10 * NBK + 1000 * NG + seed)
        run(tci8_case(rng, NBK, NBV, NG=NG), rng)


@pytest.mark.parametrize("mutate", ["kready_parity", "skip_pv_wait", "k_two_ahead"])
def test_int8_tensor_memory_kernel_planted_mistakes_are_caught(mutate):
    msg = find_violation(lambda rng: tci8_case(rng, 2, 2, mutate), range(400))
    assert msg is not None


# ---------------------------------------------------------------------------
# The D-split score exchange of the mma.sync kernel: the DS warps of a pair
# split D; for each of the key group's tiles each warp writes its partial
# scores to its part of buffer (t / KG) % 2 (t = the tile's ring sequence
# number), meets its partners at a named barrier, and reads every part.
# mutate="parity_index" restates an earlier buffer index, t % 2, which does
# not alternate when KG is even.

def exchange_roles(DS, KG, kg, ntiles, mutate=None):
    tiles = [t for t in range(ntiles) if t % KG == kg]
    part = [[None] * DS, [None] * DS]
    reading = [0, 0]
    arrived = {"n": 0}

    def warp(dh):
        for i, t in enumerate(tiles):
            buf = t % 2 if mutate == "parity_index" else (t // KG) % 2
            if reading[buf]:
                raise Violation(f"part {dh} of tile {t} written while buffer {buf} is read")
            part[buf][dh] = t
            arrived["n"] += 1
            yield (lambda target=DS * (i + 1): arrived["n"] >= target)
            if part[buf] != [t] * DS:
                raise Violation(f"tile {t}: buffer {buf} holds {part[buf]}")
            reading[buf] += 1
            yield always
            if part[buf] != [t] * DS:
                raise Violation(f"buffer {buf} changed under tile {t}")
            reading[buf] -= 1

    return {f"warp{dh}": warp(dh) for dh in range(DS)}


@pytest.mark.parametrize("DS,KG", [(2, 1), (4, 1), (2, 2), (2, 3), (4, 2)])
def test_score_exchange_is_safe(DS, KG):
    for seed in range(200):
        rng = random.Random(seed)
        for kg in range(KG):
            run(exchange_roles(DS, KG, kg, 40), rng)


def test_score_exchange_indexed_by_tile_parity_fails_for_two_groups():
    msg = find_violation(lambda rng: exchange_roles(2, 2, 1, 40, "parity_index"), range(200))
    assert msg is not None
