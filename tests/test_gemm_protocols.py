"""Host-side models of the barrier protocols of the grouped GEMMs
(moe_expert_ffn_dg_gb300/csrc/dg_gemm_q4.cu for quantised weights,
dg_gemm.cu for bf16 weights), run on random tile sequences.

The kernel's roles hand shared-memory slots and TMEM accumulators to one
another through mbarriers, and an mbarrier wait compares only the parity of
the phase: a wait that is two phases early or late returns at the wrong time
instead of blocking.  This model runs every role of one CTA as a coroutine
with the kernel's loop structure, slot arithmetic and wait parities, the
pipeline constants read from the kernel source, and an adversarial random
interleaving of the roles and of the asynchronous completions (TMA copies
landing in any order, MMAs completing in issue order).  It checks that

* every wait returns on exactly the phase it means (no parity alias),
* no slot (code slab, scale slot, A stage quarter, token stage) and no
  accumulator is rewritten before its readers are done, and no MMA reads a
  stage before its operands are in place,
* every sequence runs to the end (no deadlock).

Planted mistakes (a stage ring shorter than the stages in flight, a skipped
wait before a slot or an accumulator is reused) must be caught, so the model
is known to see the failures it guards against.
"""

import os
import random
import re

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "moe_expert_ffn_dg_gb300",
                    "csrc")
SRC = os.path.join(CSRC, "dg_gemm_q4.cu")
SRC_BF16 = os.path.join(CSRC, "dg_gemm.cu")


# ----------------------------------------------------------------- constants

def _c_eval(expr: str, env: dict) -> int:
    """Evaluate a constant expression of the kernel source: integers, names
    already evaluated, comparisons, * / + - and right-nested ?: chains."""
    expr = expr.strip()
    if "?" in expr:
        cond, rest = expr.split("?", 1)
        depth, cut = 0, None
        for i, ch in enumerate(rest):  # the ':' that belongs to this '?'
            if ch == "?":
                depth += 1
            elif ch == ":":
                if depth == 0:
                    cut = i
                    break
                depth -= 1
        a, b = rest[:cut], rest[cut + 1:]
        return _c_eval(a, env) if _c_eval(cond, env) else _c_eval(b, env)
    py = re.sub(r"\b[A-Za-z_]\w*\b", lambda m: str(env[m.group(0)]), expr)
    if not re.fullmatch(r"[\d\s<>=!*/+\-()]+", py):
        raise ValueError(f"unexpected constant expression: {expr!r}")
    return int(eval(py.replace("/", "//")))  # digits and operators only; C division


def kernel_config(bn: int) -> dict:
    src = open(SRC).read()
    ring = int(re.search(r"constexpr int kStageRing = (\d+);", src).group(1))
    body = re.search(r"struct CfgQ \{(.*?)\n\};", src, re.S).group(1)
    env = {"BN": bn, "kStageRing": ring}
    for name, expr in re.findall(r"static constexpr int (k\w+) = ([^;]+);", body):
        try:
            env[name] = _c_eval(expr, env)
        except (KeyError, ValueError):
            pass  # byte sizes and the like that use names outside the block
    gpsl = re.search(r"constexpr int GPSL = QF == 8 \? (\d+) : (\d+);", src)
    return {"GPS": env["kGPS"], "NT": env["kNT"], "M": env["kM"], "SQ": env["kSQ"],
            "NB": env["kNB"], "R": ring, "GPSL8": int(gpsl.group(1)), "GPSL4": int(gpsl.group(2))}


# -------------------------------------------------------------------- model

class ProtocolError(AssertionError):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.completed = name, count, 0, 0

    def arrive(self, world):
        self.arrived += 1
        if self.arrived > self.count:
            raise ProtocolError(f"{self.name}: more arrivals than its count")
        if self.arrived == self.count:
            self.arrived = 0
            self.completed += 1
            world["version"] += 1


def wait(bar, target):
    """The kernel's parity wait, meant to return once bar has completed
    `target` phases: it returns when the completed count has target's
    parity, which must then be target itself."""
    while (bar.completed - target) % 2:
        yield
    if bar.completed != target:
        raise ProtocolError(f"{bar.name}: parity wait for completion {target} returned at "
                            f"completion {bar.completed}")


PLANTS = ("short_ring", "skip_a_free_wait", "skip_token_free_wait", "skip_acc_empty_wait")


def run_cta(cfg, tiles, seed, gpsl, plant=None):
    """One CTA's tile sequence (list of groups-of-64 per tile) through the
    protocol; plant names a deliberate mistake (PLANTS) for the self-test."""
    GPS, NT, M, SQ, NB, R = (cfg[k] for k in ("GPS", "NT", "M", "SQ", "NB", "R"))
    if plant == "short_ring":
        R = 2
    rnd = random.Random(seed)
    world = {"version": 0}
    NA = NT * M
    qfull = [Bar(f"qfull{i}", 1) for i in range(SQ)]
    qempty = [Bar(f"qempty{i}", 4 * NT) for i in range(SQ)]
    sfull = [Bar(f"sfull{i}", 1) for i in range(2)]
    sempty = [Bar(f"sempty{i}", 4 * NT) for i in range(2)]
    bfull = [Bar(f"bfull{i}", 1) for i in range(NB)]
    afull = [Bar(f"afull{i}", 4) for i in range(NA)]
    sdone = [Bar(f"sdone{i}", 1) for i in range(R)]
    acc_full = [Bar(f"acc_full{i}", 1) for i in range(2)]
    acc_empty = [Bar(f"acc_empty{i}", 4) for i in range(2)]

    nst = [(ng + GPS - 1) // GPS for ng in tiles]
    stage_tile = [t for t, n in enumerate(nst) for _ in range(n)]
    stage_last = [k == n - 1 for n in nst for k in range(n)]
    n_stages = len(stage_tile)

    def a_slot(st):
        team, n = st % NT, st // NT  # the team's n-th own stage
        return team + NT * (n % M)

    # data state
    slab_readers = [0] * SQ              # dequant warps still reading slab i
    slab_held = [None] * SQ              # use of the slot whose codes have landed
    scale_readers = [0] * 2
    scale_held = [None] * 2              # tile whose scales have landed
    a_state = {}                         # (slot, quarter) -> stage written, or None once read
    b_state = [None] * NB                # stage whose tokens sit in the slot (landed)
    b_free = [True] * NB                 # MMAs of the slot's previous stage completed
    acc_busy = [None] * 2                # tile whose MMAs accumulate / wait for the epilogue
    pending = []                         # TMA copies in flight: (barrier, on-land action)
    mma_queue = []                       # issued stages, completing in order
    hand = {"w": 0, "i": 0}

    def land(bar, action=None):
        pending.append((bar, action))

    # ---- warp 0: code slabs and per-tile scales
    def codes():
        qs, quse = 0, [0] * SQ
        for local, ng in enumerate(tiles):
            ss = local & 1
            yield from wait(sempty[ss], local >> 1)
            if scale_readers[ss]:
                raise ProtocolError("scale slot rewritten while read")

            def put_scales(ss=ss, local=local):
                scale_held[ss] = local
            land(sfull[ss], put_scales)
            for _ in range((ng + gpsl - 1) // gpsl):
                yield from wait(qempty[qs], quse[qs])
                if slab_readers[qs]:
                    raise ProtocolError("code slab rewritten while read")

                def put_codes(qs=qs, use=quse[qs]):
                    slab_held[qs] = use
                land(qfull[qs], put_codes)
                quse[qs] += 1
                qs = (qs + 1) % SQ

    # ---- warp 1: token stages
    def tokens():
        for st in range(n_stages):
            bs = st % NB
            if st >= NB and plant != "skip_token_free_wait":
                w = st - NB
                yield from wait(sdone[w % R], w // R + 1)
            if not b_free[bs]:
                raise ProtocolError(f"token stage {st} overwrites slot {bs} before its MMAs ended")
            b_free[bs] = False

            def put(bs=bs, st=st):
                b_state[bs] = st
            land(bfull[bs], put)
            yield

    # ---- warp 3: waiter, and warp 2: issuer (meeting at the named barrier)
    def waiter():
        st = 0
        for local, ng in enumerate(tiles):
            acc = local & 1
            for k in range(nst[local]):
                if k == 0 and plant != "skip_acc_empty_wait":
                    yield from wait(acc_empty[acc], local >> 1)
                n = st // NT  # the owning team's n-th stage
                a = a_slot(st)
                yield from wait(afull[a], n // M + 1)
                yield from wait(bfull[st % NB], st // NB + 1)
                hand["w"] += 1
                while hand["i"] < hand["w"]:
                    yield
                st += 1

    def issuer():
        st = 0
        for local, ng in enumerate(tiles):
            acc = local & 1
            for k in range(nst[local]):
                while hand["w"] <= hand["i"]:
                    yield
                hand["i"] += 1
                a, bs = a_slot(st), st % NB
                for q in range(4):
                    if a_state.get((a, q)) != st:
                        raise ProtocolError(f"MMA of stage {st} reads A slot {a} holding "
                                            f"{a_state.get((a, q))}")
                if b_state[bs] != st:
                    raise ProtocolError(f"MMA of stage {st} reads token slot {bs} holding "
                                        f"{b_state[bs]}")
                if k == 0:
                    if acc_busy[acc] is not None:
                        raise ProtocolError(f"tile {local} overwrites accumulator {acc} before "
                                            f"the epilogue read tile {acc_busy[acc]}")
                    acc_busy[acc] = local
                mma_queue.append(st)
                world["version"] += 1
                st += 1
                yield

    # ---- dequantising warps: team t, quarter q
    def dequant(t, q):
        qs, quse, s0, j = 0, [0] * SQ, 0, 0
        for local, ng in enumerate(tiles):
            ss = local & 1
            yield from wait(sfull[ss], (local >> 1) + 1)
            if scale_held[ss] != local:
                raise ProtocolError(f"tile {local} reads the scales of tile {scale_held[ss]}")
            scale_readers[ss] += 1
            for sl in range((ng + gpsl - 1) // gpsl):
                yield from wait(qfull[qs], quse[qs] + 1)
                if slab_held[qs] != quse[qs]:
                    raise ProtocolError(f"slab {qs}: use {quse[qs]} reads codes of use "
                                        f"{slab_held[qs]}")
                quse[qs] += 1
                slab_readers[qs] += 1
                k = (gpsl * sl) // GPS
                while k < (gpsl * sl + gpsl) // GPS and GPS * k < ng:
                    stg = s0 + k
                    k += 1
                    if stg % NT != t:
                        continue
                    a = a_slot(stg)
                    # the slot's previous stage, this team's M own stages back
                    if j >= M and plant != "skip_a_free_wait":
                        prev = stg - M * NT
                        yield from wait(sdone[prev % R], prev // R + 1)
                    j += 1
                    old = a_state.get((a, q), "free")
                    if old not in ("free", None):
                        raise ProtocolError(f"A slot {a} rewritten for stage {stg} while it "
                                            f"holds unread stage {old}")
                    a_state[(a, q)] = stg
                    afull[a].arrive(world)
                    yield
                slab_readers[qs] -= 1
                qempty[qs].arrive(world)
                qs = (qs + 1) % SQ
            s0 += nst[local]
            scale_readers[ss] -= 1
            sempty[ss].arrive(world)

    # ---- epilogue warps
    def epilogue(q):
        for local in range(len(tiles)):
            acc = local & 1
            yield from wait(acc_full[acc], (local >> 1) + 1)
            if acc_busy[acc] != local:
                raise ProtocolError(f"epilogue of tile {local} finds accumulator {acc} "
                                    f"holding {acc_busy[acc]}")
            yield
            epi_done[acc] += 1
            if epi_done[acc] == 4:
                epi_done[acc] = 0
                acc_busy[acc] = None
            acc_empty[acc].arrive(world)

    epi_done = [0, 0]
    roles = [codes(), tokens(), waiter(), issuer()]
    roles += [dequant(t, q) for t in range(NT) for q in range(4)]
    roles += [epilogue(q) for q in range(4)]
    live = list(roles)
    idle = 0
    while live or pending or mma_queue:
        choices = len(live) + (1 if pending else 0) + (1 if mma_queue else 0)
        pick = rnd.randrange(choices)
        before = world["version"] + len(pending) + len(mma_queue)
        if pick < len(live):
            co = live[pick]
            try:
                next(co)
            except StopIteration:
                live.remove(co)
                world["version"] += 1
        elif pending and pick == len(live):
            bar, action = pending.pop(rnd.randrange(len(pending)))
            if action:
                action()
            bar.arrive(world)
        else:
            st = mma_queue.pop(0)  # tcgen05 work completes in issue order
            a = a_slot(st)
            for q in range(4):
                a_state[(a, q)] = None  # read: the slot may be rewritten
            b_free[st % NB] = True
            sdone[st % R].arrive(world)
            if stage_last[st]:
                acc_full[stage_tile[st] & 1].arrive(world)
        after = world["version"] + len(pending) + len(mma_queue)
        idle = 0 if after != before else idle + 1
        if idle > 5000 * (len(live) + 1):
            raise ProtocolError("no role can make progress (deadlock)")
    return True


def random_tiles(rnd, n, lo=1, hi=48):
    return [rnd.randint(lo, hi) for _ in range(n)]


# -------------------------------------------------------------------- tests

def test_constants_are_read_from_the_kernel():
    for bn in (32, 64, 128, 256):
        cfg = kernel_config(bn)
        assert cfg["NB"] < cfg["R"] and cfg["M"] * cfg["NT"] < cfg["R"]
        assert cfg["GPS"] in (1, 2) and cfg["NT"] in (3, 4)
    assert kernel_config(32)["GPS"] == 2 and kernel_config(256)["GPS"] == 1


@pytest.mark.parametrize("bn", [32, 64, 128, 256])
@pytest.mark.parametrize("bits", [4, 8])
def test_protocol_has_no_alias_overwrite_or_deadlock(bn, bits):
    cfg = kernel_config(bn)
    gpsl = cfg["GPSL8"] if bits == 8 else cfg["GPSL4"]
    rnd = random.Random(1000 * bn + bits)
    for seed in range(6):
        # tile lengths as in the block: down (11 groups), gate_up (44), the
        # dense pair (33), and random ones including a single group
        tiles = random_tiles(rnd, 7) + [11, 44, 33, 1, 2, 11, 11]
        rnd.shuffle(tiles)
        assert run_cta(cfg, tiles, seed, gpsl)


def test_single_group_tiles_cycle_every_ring():
    # one stage per tile: the accumulators, scale slots and stage ring turn
    # over as fast as the protocol allows
    for bn in (32, 256):
        cfg = kernel_config(bn)
        for seed in range(4):
            assert run_cta(cfg, [1] * 40, seed, cfg["GPSL4"])


@pytest.mark.parametrize("plant", PLANTS)
def test_model_catches_planted_mistakes(plant):
    cfg = kernel_config(128)
    rnd = random.Random(7)
    caught = 0
    for seed in range(20):
        tiles = [1] * 12 if plant == "skip_acc_empty_wait" else random_tiles(rnd, 10, 1, 48)
        try:
            run_cta(cfg, tiles, seed, cfg["GPSL4"], plant=plant)
        except ProtocolError:
            caught += 1
    assert caught > 0, plant


# ------------------------------------------------------- bf16-weight kernel

def bf16_stages(bn: int) -> int:
    """Stages of the projection GEMMs' ring (the router GEMM keeps a ring of
    its own size, one CTA an SM)."""
    src = open(SRC_BF16).read()
    hdr = open(os.path.join(CSRC, "dg_kernels.h")).read()
    env = {"BN": bn}
    ctas = int(re.search(r"constexpr int kProjCtasPerSm = (\d+);", hdr).group(1))
    for name in ("kATileBytes", "kRingBytes"):
        env[name] = _c_eval(re.search(rf"constexpr int {name} = ([^;]+);", src).group(1), env)
    env["RING"] = env["kRingBytes"] // (1 if bn == 256 else ctas)
    body = re.search(r"struct Cfg \{(.*?)\n\};", src, re.S).group(1)
    for name, expr in re.findall(r"static constexpr int (k\w+) = ([^;]+);", body):
        env[name] = _c_eval(expr, env)
    return env["kStages"]


def run_bf16_cta(S, tiles, seed, plant=None):
    """The bf16 kernel: one producer fills a ring of S (weight, token) stages,
    one thread issues the MMAs and frees each stage with a commit, four
    epilogue warps drain the two accumulators."""
    rnd = random.Random(seed)
    world = {"version": 0}
    full = [Bar(f"full{i}", 1) for i in range(S)]
    empty = [Bar(f"empty{i}", 1) for i in range(S)]
    acc_full = [Bar(f"acc_full{i}", 1) for i in range(2)]
    acc_empty = [Bar(f"acc_empty{i}", 4) for i in range(2)]
    n_stages = sum(tiles)
    stage_tile = [t for t, n in enumerate(tiles) for _ in range(n)]
    stage_last = [k == n - 1 for n in tiles for k in range(n)]
    held = [None] * S          # stage whose operands sit in the slot (landed)
    free = [True] * S
    acc_busy = [None] * 2
    pending, mma_queue, epi_done = [], [], [0, 0]

    def producer():
        for st in range(n_stages):
            s = st % S
            if plant != "skip_empty_wait":
                yield from wait(empty[s], st // S)
            if not free[s]:
                raise ProtocolError(f"stage {st} overwrites slot {s} before its MMAs ended")
            free[s] = False

            def put(s=s, st=st):
                held[s] = st
            pending.append((full[s], put))
            yield

    def issuer():
        st = 0
        for local, n in enumerate(tiles):
            acc = local & 1
            yield from wait(acc_empty[acc], local >> 1)
            if acc_busy[acc] is not None:
                raise ProtocolError(f"tile {local} overwrites accumulator {acc}")
            acc_busy[acc] = local
            for _ in range(n):
                yield from wait(full[st % S], st // S + 1)
                if held[st % S] != st:
                    raise ProtocolError(f"MMA of stage {st} reads slot holding {held[st % S]}")
                mma_queue.append(st)
                world["version"] += 1
                st += 1
                yield

    def epilogue():
        for local in range(len(tiles)):
            acc = local & 1
            yield from wait(acc_full[acc], (local >> 1) + 1)
            if acc_busy[acc] != local:
                raise ProtocolError(f"epilogue of tile {local} finds tile {acc_busy[acc]}")
            yield
            epi_done[acc] += 1
            if epi_done[acc] == 4:
                epi_done[acc] = 0
                acc_busy[acc] = None
            acc_empty[acc].arrive(world)

    live = [producer(), issuer()] + [epilogue() for _ in range(4)]
    idle = 0
    while live or pending or mma_queue:
        choices = len(live) + (1 if pending else 0) + (1 if mma_queue else 0)
        pick = rnd.randrange(choices)
        before = world["version"] + len(pending) + len(mma_queue)
        if pick < len(live):
            co = live[pick]
            try:
                next(co)
            except StopIteration:
                live.remove(co)
                world["version"] += 1
        elif pending and pick == len(live):
            bar, action = pending.pop(rnd.randrange(len(pending)))
            action()
            bar.arrive(world)
        else:
            st = mma_queue.pop(0)
            held[st % S] = None
            free[st % S] = True
            empty[st % S].arrive(world)
            if stage_last[st]:
                acc_full[stage_tile[st] & 1].arrive(world)
        after = world["version"] + len(pending) + len(mma_queue)
        idle = 0 if after != before else idle + 1
        if idle > 5000 * (len(live) + 1):
            raise ProtocolError("no role can make progress (deadlock)")
    return True


@pytest.mark.parametrize("bn", [64, 128, 256])
def test_bf16_protocol_has_no_alias_overwrite_or_deadlock(bn):
    S = bf16_stages(bn)
    assert 3 <= S <= 8
    rnd = random.Random(bn)
    for seed in range(6):
        tiles = random_tiles(rnd, 8) + [44, 11, 33, 1, 1]
        rnd.shuffle(tiles)
        assert run_bf16_cta(S, tiles, seed)


def test_bf16_model_catches_a_skipped_slot_wait():
    caught = 0
    for seed in range(20):
        try:
            run_bf16_cta(bf16_stages(128), [11] * 8, seed, plant="skip_empty_wait")
        except ProtocolError:
            caught += 1
    assert caught > 0
