"""Executable model of the attention kernel's synchronisation protocol.

The fused kernel (transformer_attention_02_gb300/csrc/attn_kernel.cuh) runs
five roles in one CTA that hand work to each other through shared-memory
mbarriers: the K/V TMA producer, the Q TMA producer, the single-thread MMA
issuer, two softmax warpgroups and, in the rotary variant, four warps that
rotate the Q sub-tiles. This module re-states each role's control flow in Python, over the
same tile schedule, and runs the roles under an adversarial scheduler together
with the asynchronous agents they drive (TMA copies that land in any order,
the tensor core's in-order queue of MMAs and commits).

What it checks, on every interleaving it is given:
  * no deadlock: some role or agent can always make progress until every role
    has finished;
  * every mbarrier wait is sound: a thread waiting for phase k of a barrier
    (by its parity, as the hardware does) finds exactly k or k + 1 phases
    completed; k - 1 would let the parity test pass before the phase it wants,
    k + 2 would make it miss the phase (overrun);
  * no data race on shared memory or tensor memory: a TMA copy never lands in
    a ring slot or Q buffer that an unexecuted MMA still reads; every MMA reads
    the K/V block, Q sub-tile (rotated, in the rotary variant) and P it
    expects; S, P and O in tensor memory are written, read and rescaled in
    the order the algorithm needs (the softmax reads S only after the Q K^T
    that wrote it, rescales O only between two P V products, the epilogue
    reads O after the tile's last P V and before the next tile's first one);
  * the abort path terminates: when a bounded wait runs out (modelled by a
    wait that nothing will ever satisfy, as the kernel's stall hook does),
    every role leaves its loops and the shutdown waits (TMA copies landed,
    MMAs retired) complete by themselves.

The model is CPU-only test infrastructure; it shares no code with the kernel.
"""
from __future__ import annotations

import random
from collections import deque
from dataclasses import dataclass, field


class ProtocolError(AssertionError):
    pass


# ------------------------------------------------------------------ schedule

BLOCK_M = 128
BLOCK_N = 128
ROWS_PER_TILE = 2 * BLOCK_M


@dataclass
class Params:
    D: int = 128
    causal: bool = True
    B: int = 1
    Hq: int = 2
    Hkv: int = 2
    Sq: int = 512
    Sk: int = 512
    num_splits: int = 1          # key ranges (split-key mode when > 1)
    rope: bool = False           # rotary variant: Q rotated by four warps, "Q ready" has four arrivals
    additive: bool = False       # additive-mask variant: warpgroup 1's O leaves through its Q buffer
    pack_shift: int = 0          # GQA head packing: 2^pack_shift query heads share a tile's rows
    grid: int = 1                # persistent CTAs
    cta: int = 0                 # which CTA of the grid is modelled
    debug_stall: bool = False    # the MMA issuer first waits on a barrier nothing signals
    tile_slots: int = 8          # entries of the shared-memory tile ring
    head_group: int = 0          # slices per group of the tile order (0: all slices)
    steal_seed: int = -1         # >= 0: the CTA's tiles are its own and a random set taken over from CTAs
                                 # that had not started (cluster launch control), in launch order

    @property
    def tile_consumers(self) -> int:
        """Arrivals that free a tile-ring entry: the K/V producer, the MMA
        issuer, the eight softmax warps and, in the rotary variant, the four
        rotating warps."""
        return 1 + 1 + 8 + (4 if self.rope else 0)

    @property
    def slots(self) -> int:
        return 4 if self.D == 128 else 8

    @property
    def q_bufs(self) -> int:
        return 3

    @property
    def stage_o(self) -> bool:
        """The upper sub-tile's O goes out through its Q buffer (additive-mask
        variant at D = 128 with 16-bit output: no split keys, no head packing)."""
        return self.additive and self.D == 128 and self.num_splits == 1 and self.pack_shift == 0


@dataclass(frozen=True)
class Tile:
    b: int
    h: int
    hk: int
    m0: int
    split: int
    kb0: int
    nb: tuple
    n: int


def _ceil_div(a, b):
    return (a + b - 1) // b


def schedule(p: Params):
    """The CTA's work tiles in order. One CTA per tile is launched and each CTA
    starts with its own tile (blockIdx.x = cta) and then takes over tiles of
    CTAs that had not started, always in launch order: the model uses either
    the back-and-forth wave order of a persistent grid (steal_seed < 0) or a
    random increasing subset of the later tiles."""
    ps = p.pack_shift
    heads = p.Hkv if ps else p.Hq
    group = p.Hq // p.Hkv
    sub_rows = BLOCK_M >> ps
    n_mblk = _ceil_div(p.Sq, ROWS_PER_TILE >> ps)
    n_kb = _ceil_div(p.Sk, BLOCK_N)
    split_blocks = _ceil_div(n_kb, p.num_splits) if p.num_splits > 1 else n_kb
    n_splits = _ceil_div(n_kb, split_blocks) if p.num_splits > 1 else 1
    n_tiles = p.B * heads * n_mblk * n_splits
    out = []
    if p.steal_seed >= 0:
        rng = random.Random(p.steal_seed)
        order = [p.cta] + sorted(t for t in range(p.cta + 1, n_tiles) if rng.random() < 0.4)
    else:
        order = []
        w = 0
        while w * p.grid < n_tiles:
            order.append(w * p.grid + ((p.grid - 1 - p.cta) if (w & 1) else p.cta))
            w += 1
    slices = p.B * heads
    head_group = max(1, min(slices, p.head_group or slices))
    tail_levels = min(3, n_mblk) if p.causal else 0
    head_levels = n_mblk - tail_levels
    grouped = slices * head_levels * n_splits
    for tile in order:
        if tile >= n_tiles:
            continue
        if tile < grouped:                  # grouped slices, longest query block first
            per_slice = head_levels * n_splits
            g0 = tile // (head_group * per_slice) * head_group
            gs = min(head_group, slices - g0)
            local = tile - g0 * per_slice
            level, rem = divmod(local, gs * n_splits)
            split, r = divmod(rem, gs)
            bh = g0 + r
            mb = (n_mblk - 1 - level) if p.causal else level
        else:                               # the shortest levels of every slice, last
            level, rem = divmod(tile - grouped, slices * n_splits)
            split, bh = divmod(rem, slices)
            mb = (tail_levels - 1 - level) if p.causal else head_levels + level
        b, hh = divmod(bh, heads)
        h = hh * group if ps else hh
        hk = hh if ps else hh // group
        m0 = mb * 2 * sub_rows
        kb0 = split * split_blocks
        begin = kb0 * BLOCK_N
        end = min(p.Sk, begin + split_blocks * BLOCK_N)
        nb = []
        for s in range(2):
            first = m0 + s * sub_rows
            last = min(first + sub_rows - 1, p.Sq - 1)
            kv_end = begin
            if first < p.Sq:
                kv_end = min(end, max(0, last + (p.Sk - p.Sq) + 1)) if p.causal else end
            nb.append(_ceil_div(kv_end - begin, BLOCK_N) if kv_end > begin else 0)
        out.append(Tile(b, h, hk, m0, split, kb0, tuple(nb), max(nb)))
    return out


# --------------------------------------------------------------- simulation

class Barrier:
    def __init__(self, name: str, count: int):
        self.name = name
        self.count = count
        self.pending = count
        self.tx = 0
        self.completed = 0

    def arrive(self):
        self.pending -= 1
        self._maybe_complete()

    def expect_tx(self, n: int):
        self.tx += n

    def complete_tx(self, n: int):
        self.tx -= n
        self._maybe_complete()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = self.count


@dataclass
class Proc:
    name: str
    gen: object
    op: tuple = None
    done: bool = False
    blocked_since: int = 0


@dataclass
class Sim:
    p: Params
    rng: random.Random
    timeouts: bool = False
    bars: dict = field(default_factory=dict)
    res: dict = field(default_factory=dict)
    abort: bool = False
    timed_out: bool = False
    inflight: list = field(default_factory=list)
    mma_queue: deque = field(default_factory=deque)
    steps: int = 0

    def bar(self, name: str) -> Barrier:
        return self.bars[name]

    # -- checks applied when a thread evaluates a wait
    def poll(self, name: str, k: int) -> bool:
        bar = self.bars[name]
        c = bar.completed
        if not self.abort and not (k <= c <= k + 1):
            raise ProtocolError(f"{name}: waiting for phase {k} with {c} phases completed")
        return (c & 1) != (k & 1)

    def reads_pending(self, res_name: str) -> bool:
        return any(res_name in item[1] for item in self.mma_queue if item[0] == "mma")

    def tma_issue(self, bar: str, nbytes: int, res_name: str, tag, owner: str = ""):
        if self.reads_pending(res_name):
            raise ProtocolError(f"TMA into {res_name} while an unexecuted MMA still reads it")
        st = self.res.get(res_name)
        if isinstance(st, tuple) and st and st[0] == "loading":
            raise ProtocolError(f"TMA into {res_name} while another copy into it is in flight")
        if isinstance(st, tuple) and st and st[0] == "O":
            raise ProtocolError(f"TMA into {res_name} over the staged O of {st[1]} not yet stored")
        self.res[res_name] = ("loading", tag)
        self.inflight.append((bar, nbytes, res_name, tag, owner))

    def expect(self, res_name: str, want, what: str):
        got = self.res.get(res_name)
        if got != want:
            raise ProtocolError(f"{what}: {res_name} holds {got}, expected {want}")


def _tile_key(t: Tile):
    return (t.b, t.h, t.m0, t.split)


# ---------------------------------------------------------------- tile ring
# The Q warp computes each work tile once and publishes it in a ring of
# shared-memory entries (tile_full[slot], one arrival); every other role reads
# the entries in order and frees each one as soon as it holds a copy
# (tile_empty[slot], one arrival per consumer). After the last tile the
# producer publishes an end marker (None).

def ring_entries(tiles):
    return list(tiles) + [None]


def ring_fetch(sim: Sim, k: int, arrivals: int = 1):
    """Consumer side: wait for entry k, copy it, free it."""
    p = sim.p
    slot = k % p.tile_slots
    ok = yield ("wait", f"tile_full{slot}", k // p.tile_slots)
    if not ok:
        return False, None
    box = {}

    def read():
        got = sim.res.get(f"tile{slot}")
        if got is None or got[0] != k:
            raise ProtocolError(f"tile ring slot {slot}: entry {got and got[0]} read as entry {k}")
        box["t"] = got[1]
    yield ("act", read)
    for _ in range(arrivals):
        yield ("arrive", f"tile_empty{slot}")
    return True, box["t"]


def ring_produce(sim: Sim, k: int, entry, waited: bool = False):
    """Producer side: wait until entry k - slots has been freed, write entry k."""
    p = sim.p
    slot = k % p.tile_slots
    if k >= p.tile_slots and not waited:
        ok = yield ("wait", f"tile_empty{slot}", k // p.tile_slots - 1)
        if not ok:
            return False

    def write():
        sim.res[f"tile{slot}"] = (k, entry)
    yield ("act", write)
    yield ("arrive", f"tile_full{slot}")
    return True


# ------------------------------------------------------------------ roles
# Each role is a generator that yields the operations of the kernel role of
# the same name, in the same order:
#   ("wait", bar, phase)   bounded wait (returns False on abort or timeout)
#   ("drain", bar, phase)  shutdown wait (ignores the abort flag)
#   ("probe", bar, phase)  non-blocking test (returns the parity test)
#   ("arrive", bar) / ("expect_tx", bar, bytes) / ("tma", bar, bytes, res, tag)
#   ("mma", reads, fn) / ("commit", bar)   appended to the tensor core's queue
#   ("act", fn)           a synchronous action of the thread (loads, stores)

def role_tma(sim: Sim, tiles):
    """K/V producer (warp 9): the blocks in the order the MMA issuer takes
    them, K_0, then per block V_j and K_{j+1}; work tiles from the tile ring."""
    p = sim.p
    S = p.slots
    st = {"fill": 0, "alive": True}

    def load(kv, ti, blk):
        slot = st["fill"] % S
        if st["fill"] >= S:
            ok = yield ("wait", f"kv_empty{slot}", st["fill"] // S - 1)
            if not ok:
                st["alive"] = False
                return
        yield ("expect_tx", f"kv_full{slot}", 1)
        yield ("tma", f"kv_full{slot}", 1, f"kv{slot}", ("KV", kv, ti.b, ti.hk, ti.kb0 + blk))
        st["fill"] += 1

    k = 0
    while st["alive"]:
        ok, ti = yield from ring_fetch(sim, k)
        if not ok or ti is None:
            break
        k += 1
        if ti.n > 0:
            yield from load(0, ti, 0)
        for j in range(ti.n):
            if not st["alive"]:
                break
            yield from load(1, ti, j)
            if st["alive"] and j + 1 < ti.n:
                yield from load(0, ti, j + 1)
    kv_fill = st["fill"]
    for s in range(S):
        if kv_fill > s:
            last = s + S * ((kv_fill - 1 - s) // S)
            yield ("drain", f"kv_full{s}", last // S)


def q_slot(nq: int, t: int, nbufs: int = 3):
    """Buffer and use count of sub-tile t of the nq-th tile with key blocks.
    Sub-tiles take the Q buffers in turn (lower, upper, next lower, ...): with
    three buffers the next tile's upper sub-tile goes into the buffer the
    current lower sub-tile frees one block before the tile ends."""
    i = 2 * nq + t
    return i % nbufs, i // nbufs


def q_bufs_of(nq: int, nbufs: int = 3):
    return q_slot(nq, 0, nbufs)[0], q_slot(nq, 1, nbufs)[0]


def _q_tag(ti: Tile, t: int, p: Params):
    return ("Q", ti.b, ti.h, ti.m0 + t * (BLOCK_M >> p.pack_shift))


def _rotate(sim: Sim, buf: int, quarter: int):
    def fn():
        name = f"q{buf}"
        st = sim.res.get(name)
        if not (isinstance(st, tuple) and st and st[0] == "Q"):
            raise ProtocolError(f"rotation of {name} before its copy landed ({st})")
        if sim.reads_pending(name):
            raise ProtocolError(f"rotation of {name} while an MMA reads it")
        if ("rot", quarter) in st[4:]:
            raise ProtocolError(f"rows of quarter {quarter} of {name} rotated twice ({st})")
        sim.res[name] = st + (("rot", quarter),)
    return ("act", fn)


def role_qload(sim: Sim, tiles):
    """Q producer (warp 10) and producer of the tile ring: each entry is
    published when this warp is about to load that tile's Q (next_work of the
    kernel)."""
    p = sim.p
    uses = [0] * p.q_bufs
    nq = 0
    entries = ring_entries(tiles)
    st = {"produced": 0, "clc": 0, "drained": False, "staged": [0, 0]}
    staged = [None] * p.q_bufs          # (warpgroup, its staging index, tile key) of the O a buffer will hold

    def store_staged(buf):
        """Wait until the warpgroup has written the tile's O into buf, then copy
        it out (the tensor store reads the buffer before this warp goes on).
        Each warpgroup's stagings alternate between two barriers of its own: at
        most two of them are ever waiting to be stored, so no wait can fall a
        whole phase behind."""
        wg, idx, key = staged[buf]
        ok = yield ("wait", f"o_staged{wg}{idx % 2}", idx // 2)
        if not ok:
            return False

        def store(buf=buf, key=key, wg=wg):
            sim.expect(f"q{buf}", ("O", key, wg), f"store of the staged O of {key}, sub-tile {wg}")
            sim.res[f"q{buf}"] = "free"
        yield ("act", store)
        staged[buf] = None
        return True

    def produce():
        k = st["produced"]
        if k >= 1 and not st["drained"]:
            # the next tile index comes from a cluster-launch-control request
            # (or its failure: no CTA left), completing on the clc barrier
            slot = k % p.tile_slots
            if k >= p.tile_slots:
                ok = yield ("wait", f"tile_empty{slot}", k // p.tile_slots - 1)
                if not ok:
                    return -1, None
            yield ("expect_tx", "clc", 1)
            yield ("tma", "clc", 1, "clc_resp", ("CLC", st["clc"]))
            ok = yield ("wait", "clc", st["clc"])
            if not ok:
                yield ("drain", "clc", st["clc"])       # the response must land before the CTA exits
                return -1, None

            def read(n=st["clc"]):
                sim.expect("clc_resp", ("CLC", n), "launch-control response")
            yield ("act", read)
            st["clc"] += 1
            if entries[k] is None:
                st["drained"] = True
            ok = yield from ring_produce(sim, k, entries[k], waited=True)
        else:
            ok = yield from ring_produce(sim, k, entries[k])
        if not ok:
            return -1, None
        st["produced"] += 1
        return (1 if entries[k] is not None else 0), entries[k]

    def next_work():
        while True:
            r, t = yield from produce()
            if not (r > 0 and t.n == 0):
                return r, t

    def load(buf, ti, t):
        if uses[buf] > 0:
            ok = yield ("wait", f"q_empty{buf}", uses[buf] - 1)
            if not ok:
                return False
        if staged[buf] is not None and not (yield from store_staged(buf)):
            return False
        if p.stage_o and ti.nb[t] > 0:
            staged[buf] = (t, st["staged"][t], _tile_key(ti))
            st["staged"][t] += 1
        yield ("expect_tx", f"q_full{buf}", 1)
        yield ("tma", f"q_full{buf}", 1, f"q{buf}", _q_tag(ti, t, p))
        uses[buf] += 1
        return True

    while True:
        r, ti = yield from next_work()
        if r <= 0:
            break
        lb, ub = q_bufs_of(nq, p.q_bufs)
        if not (yield from load(lb, ti, 0)) or not (yield from load(ub, ti, 1)):
            break
        nq += 1
    # the O of the last tiles still waits in their buffers (in staging order)
    for buf in sorted((b for b in range(p.q_bufs) if staged[b] is not None), key=lambda b: staged[b][:2]):
        if not (yield from store_staged(buf)):
            break
    for b in range(p.q_bufs):
        if uses[b] > 0:
            yield ("drain", f"q_full{b}", uses[b] - 1)


def role_rope_q(sim: Sim, tiles, quarter: int):
    """Rotary variant, warp 12 + quarter: rotates its 32 rows of every Q sub-tile."""
    p = sim.p
    nq = 0
    k = 0
    while True:
        ok, ti = yield from ring_fetch(sim, k)
        if not ok or ti is None:
            return
        k += 1
        if ti.n == 0:
            continue
        for t in range(2):
            buf, use = q_slot(nq, t, p.q_bufs)
            ok = yield ("wait", f"q_full{buf}", use)
            if not ok:
                return
            yield _rotate(sim, buf, quarter)
            yield ("arrive", f"q_rdy{buf}")
        nq += 1


def _qk(sim: Sim, ti: Tile, t: int, q_buf: int, k_slot: int, blk: int):
    """S_t = Q_t K_blk^T (an MMA group) as the tensor core executes it."""
    p = sim.p
    key = _tile_key(ti)
    q_tag = _q_tag(ti, t, p)
    if p.rope:
        q_tag = q_tag + tuple(("rot", i) for i in range(4))
    k_tag = ("KV", 0, ti.b, ti.hk, ti.kb0 + blk)

    def fn():
        q_state = sim.res.get(f"q{q_buf}")
        if not (isinstance(q_state, tuple) and q_state[:4] == q_tag[:4] and set(q_state[4:]) == set(q_tag[4:])):
            raise ProtocolError(f"Q K^T of {key} sub-tile {t}: q{q_buf} holds {q_state}, expected {q_tag}")
        sim.expect(f"kv{k_slot}", k_tag, f"Q K^T of {key} sub-tile {t} block {blk}")
        s = sim.res.get(f"S{t}", "free")
        if s != "free":
            raise ProtocolError(f"Q K^T of {key} sub-tile {t} block {blk} overwrites S{t} holding {s}")
        sim.res[f"S{t}"] = ("S", key, t, blk)
    return ("mma", (f"q{q_buf}", f"kv{k_slot}"), fn)


def _pv(sim: Sim, ti: Tile, t: int, v_slot: int, blk: int):
    """O_t (+)= P_t V_blk as the tensor core executes it."""
    key = _tile_key(ti)
    v_tag = ("KV", 1, ti.b, ti.hk, ti.kb0 + blk)

    def fn():
        sim.expect(f"S{t}", ("P", key, t, blk), f"P V of {key} sub-tile {t} block {blk}")
        sim.expect(f"kv{v_slot}", v_tag, f"P V of {key} sub-tile {t} block {blk}")
        o = sim.res.get(f"O{t}", "free")
        if blk == 0:
            if not (o == "free" or (isinstance(o, tuple) and o[0] == "read")):
                raise ProtocolError(f"first P V of {key} sub-tile {t} overwrites O{t} holding {o}")
        elif o != ("O", key, t, blk - 1):
            raise ProtocolError(f"P V of {key} sub-tile {t} block {blk}: O{t} holds {o}")
        sim.res[f"S{t}"] = "free"
        sim.res[f"O{t}"] = ("O", key, t, blk)
    return ("mma", (f"S{t}", f"kv{v_slot}"), fn)


def role_mma(sim: Sim, tiles):
    """MMA issuer (warp 8, lane 0): the ping-pong issue order of role_mma."""
    p = sim.p
    S = p.slots
    st = {"kv_use": 0}
    p_cnt = [0, 0]
    nq = 0
    issued = False
    alive = True
    q_ready = "q_rdy" if p.rope else "q_full"

    def acquire(seen=False):
        slot = st["kv_use"] % S
        ok = True
        if not seen:
            ok = yield ("wait", f"kv_full{slot}", st["kv_use"] // S)
        st["kv_use"] += 1
        return slot, ok

    def probe_next():
        u = st["kv_use"]
        return (yield ("probe", f"kv_full{u % S}", u // S))

    def wait_p(t):
        ok = yield ("wait", f"p_full{t}", p_cnt[t])
        p_cnt[t] += 1
        return ok

    if p.debug_stall:
        alive = yield ("wait", "stall", 0)
    k = 0
    while alive:
        ok, ti = yield from ring_fetch(sim, k)
        if not ok or ti is None:
            break
        k += 1
        n, n0, n1 = ti.n, ti.nb[0], ti.nb[1]
        if n == 0:                  # no key block: nothing to issue
            continue
        q_buf = q_bufs_of(nq, p.q_bufs)
        ok = yield ("wait", f"{q_ready}{q_buf[0]}", q_slot(nq, 0, p.q_bufs)[1])
        if ok:
            ks, ok = yield from acquire()
        if not ok:
            alive = False
            break
        if n0 > 0:
            yield _qk(sim, ti, 0, q_buf[0], ks, 0)
            yield ("commit", "s_full0")
        issued = True
        ok = yield ("wait", f"{q_ready}{q_buf[1]}", q_slot(nq, 1, p.q_bufs)[1])
        if not ok:
            alive = False
            break
        nq += 1
        if n1 > 0:
            yield _qk(sim, ti, 1, q_buf[1], ks, 0)
            yield ("commit", "s_full1")
        yield ("commit", f"kv_empty{ks}")
        # each Q buffer is released after its sub-tile's last Q K^T
        if n0 <= 1:
            yield ("commit", f"q_empty{q_buf[0]}")
        if n1 <= 1:
            yield ("commit", f"q_empty{q_buf[1]}")
        v_seen = False
        for j in range(n):
            more = j + 1 < n
            vs, ok = yield from acquire(v_seen)
            if not ok:
                alive = False
                break
            k_seen = more and (yield from probe_next())
            if j < n0:
                if not (yield from wait_p(0)):
                    alive = False
                    break
                yield _pv(sim, ti, 0, vs, j)
                if j == n0 - 1:
                    yield ("commit", "o_full0")
            if more:
                ks, ok = yield from acquire(k_seen)
                if not ok:
                    alive = False
                    break
                if j + 1 < n0:
                    yield _qk(sim, ti, 0, q_buf[0], ks, j + 1)
                    yield ("commit", "s_full0")
                    if j + 1 == n0 - 1:
                        yield ("commit", f"q_empty{q_buf[0]}")
            if j < n1:
                if not (yield from wait_p(1)):
                    alive = False
                    break
                yield _pv(sim, ti, 1, vs, j)
                if j == n1 - 1:
                    yield ("commit", "o_full1")
            yield ("commit", f"kv_empty{vs}")
            if more:
                v_seen = yield from probe_next()
                if j + 1 < n1:
                    yield _qk(sim, ti, 1, q_buf[1], ks, j + 1)
                    yield ("commit", "s_full1")
                yield ("commit", f"kv_empty{ks}")
                if j + 1 == n1 - 1:
                    yield ("commit", f"q_empty{q_buf[1]}")
    if issued:
        yield ("commit", "drain")
        yield ("drain", "drain", 0)


def role_softmax(sim: Sim, tiles, t: int):
    """Softmax warpgroup t: per block, S_t -> P_t (rescaling O_t), then the
    epilogue; with stage_o it writes its O into its sub-tile's Q buffer and
    signals the Q warp, which stores it."""
    p = sim.p
    s_cnt = 0
    o_cnt = 0
    k = 0
    nq = 0
    n_staged = 0
    while True:
        ok, ti = yield from ring_fetch(sim, k, arrivals=4)     # each of the four warps frees the entry
        if not ok or ti is None:
            return
        k += 1
        nb = ti.nb[t]
        key = _tile_key(ti)
        qbuf = q_slot(nq, t, p.q_bufs)[0]
        if ti.n > 0:
            nq += 1
        if nb == 0:
            continue
        ok = True
        for j in range(nb):
            landed = yield ("wait", f"s_full{t}", s_cnt)
            s_cnt += 1
            if landed:
                def fn(j=j):
                    sim.expect(f"S{t}", ("S", key, t, j), f"softmax {t} block {j}")
                    if j > 0:      # the lazy rescale of O_t may run here
                        sim.expect(f"O{t}", ("O", key, t, j - 1), f"rescale of O{t} at block {j}")
                    sim.res[f"S{t}"] = ("P", key, t, j)
                yield ("act", fn)
            ok = landed
            if not ok:
                break
            yield ("arrive", f"p_full{t}")
        if not ok:
            return
        ok = yield ("wait", f"o_full{t}", o_cnt)
        if not ok:
            return
        o_cnt += 1

        def epi(nb=nb):
            sim.expect(f"O{t}", ("O", key, t, nb - 1), f"epilogue {t}")
            sim.res[f"O{t}"] = ("read", key, t)
        yield ("act", epi)
        if p.stage_o:
            sidx = n_staged
            n_staged += 1

            def stage(ti=ti, qbuf=qbuf):
                q = sim.res.get(f"q{qbuf}")
                if not (isinstance(q, tuple) and q[:4] == _q_tag(ti, t, p)[:4]):
                    raise ProtocolError(f"staging the O of {key} into q{qbuf}, which holds {q}")
                if sim.reads_pending(f"q{qbuf}"):
                    raise ProtocolError(f"staging the O of {key} into q{qbuf} while an MMA still reads it")
                sim.res[f"q{qbuf}"] = ("O", key, t)
            yield ("act", stage)
            for _ in range(4):                   # one arrival per warp, after its rows are written
                yield ("arrive", f"o_staged{t}{sidx % 2}")


# ---------------------------------------------------------------- scheduler

def make_sim(p: Params, seed: int, timeouts: bool = False):
    sim = Sim(p, random.Random(seed), timeouts=timeouts)
    names = [("q_full", p.q_bufs, 1), ("q_empty", p.q_bufs, 1), ("s_full", 2, 1), ("p_full", 2, 1),
             ("o_full", 2, 1), ("kv_full", p.slots, 1), ("kv_empty", p.slots, 1), ("q_rdy", p.q_bufs, 4)]
    for base, n, count in names:
        for i in range(n):
            sim.bars[f"{base}{i}"] = Barrier(f"{base}{i}", count)
    for i in range(p.tile_slots):
        sim.bars[f"tile_full{i}"] = Barrier(f"tile_full{i}", 1)
        sim.bars[f"tile_empty{i}"] = Barrier(f"tile_empty{i}", p.tile_consumers)
    sim.bars["clc"] = Barrier("clc", 1)
    for t in range(2):
        for i in range(2):
            sim.bars[f"o_staged{t}{i}"] = Barrier(f"o_staged{t}{i}", 4)
    sim.bars["drain"] = Barrier("drain", 1)
    sim.bars["stall"] = Barrier("stall", 1)
    tiles = schedule(p)
    procs = [Proc("tma", role_tma(sim, tiles)), Proc("qload", role_qload(sim, tiles)),
             Proc("mma", role_mma(sim, tiles)), Proc("softmax0", role_softmax(sim, tiles, 0)),
             Proc("softmax1", role_softmax(sim, tiles, 1))]
    if p.rope:
        procs += [Proc(f"rope_q{i}", role_rope_q(sim, tiles, i)) for i in range(4)]
    return sim, procs, tiles


def _advance(proc: Proc, value=None):
    try:
        proc.op = proc.gen.send(value) if proc.op is not None else next(proc.gen)
    except StopIteration:
        proc.done = True
        proc.op = None


def run(p: Params, seed: int = 0, timeouts: bool = False, bias: float = 0.5, max_steps: int = 2_000_000,
        abort_at: int = None):
    """One adversarially scheduled execution. Raises ProtocolError on a
    violation or a deadlock; returns the simulation state at the end.

    timeouts: a bounded wait that nothing can satisfy runs out (sets the
    abort flag) instead of being reported as a deadlock.
    abort_at: at that step some wait of the CTA is taken to have run out (the
    abort flag is raised wherever the roles are)."""
    sim, procs, tiles = make_sim(p, seed, timeouts)
    rng = sim.rng
    for pr in procs:
        _advance(pr)
    # per-run priorities: some agents run eagerly, others lag behind
    prio = {pr.name: rng.random() for pr in procs}
    prio["tma_agent"] = rng.random()
    prio["mma_agent"] = rng.random()

    def runnable(pr: Proc):
        op = pr.op
        kind = op[0]
        if kind == "wait":
            if sim.abort:
                return True
            return sim.poll(op[1], op[2])
        if kind == "drain":
            return sim.poll(op[1], op[2])
        return True

    while True:
        if all(pr.done for pr in procs):
            break                               # every thread has left: the kernel ends here
        sim.steps += 1
        if abort_at is not None and sim.steps == abort_at:
            sim.abort = True
            sim.timed_out = True
        if sim.steps > max_steps:
            raise ProtocolError("step limit reached (livelock?)")
        cands = [("proc", pr) for pr in procs if not pr.done and runnable(pr)]
        cands += [("tma", i) for i in range(len(sim.inflight))]
        if sim.mma_queue:
            cands.append(("mma", None))
        if not cands:
            blocked = [pr for pr in procs if not pr.done]
            waiting = [pr for pr in blocked if pr.op[0] == "wait"]
            if sim.timeouts and waiting:
                pr = rng.choice(waiting)          # the bounded wait runs out
                sim.abort = True
                sim.timed_out = True
                _advance(pr, False)
                continue
            raise ProtocolError("deadlock: " + ", ".join(f"{pr.name} at {pr.op}" for pr in blocked))
        # biased choice: prefer high-priority candidates, sometimes pick uniformly
        if rng.random() < bias:
            def weight(c):
                if c[0] == "proc":
                    return prio[c[1].name]
                return prio["tma_agent"] if c[0] == "tma" else prio["mma_agent"]
            kind, obj = max(cands, key=lambda c: weight(c) + 0.3 * rng.random())
        else:
            kind, obj = rng.choice(cands)
        if kind == "tma":
            bar, nbytes, res_name, tag, _owner = sim.inflight.pop(obj)
            sim.res[res_name] = tag
            sim.bars[bar].complete_tx(nbytes)
            continue
        if kind == "mma":
            item = sim.mma_queue.popleft()
            if item[0] == "mma":
                item[2]()
            else:
                sim.bars[item[1]].arrive()
            continue
        pr = obj
        op = pr.op
        k = op[0]
        val = None
        if k == "wait":
            # satisfied, or (after an abort) whatever the last poll of wait_phase saw
            val = sim.poll(op[1], op[2])
        elif k == "drain":
            val = True
        elif k == "probe":
            val = sim.poll(op[1], op[2])
        elif k == "arrive":
            sim.bars[op[1]].arrive()
        elif k == "expect_tx":
            sim.bars[op[1]].expect_tx(op[2])
            sim.bars[op[1]].arrive()
        elif k == "tma":
            sim.tma_issue(op[1], op[2], op[3], op[4], pr.name)
        elif k == "mma":
            sim.mma_queue.append(op)
        elif k == "commit":
            sim.mma_queue.append(("commit", op[1]))
        elif k == "act":
            op[1]()
        else:
            raise ProtocolError(f"unknown op {op}")
        _advance(pr, val)
        if pr.done and any(f[4] == pr.name for f in sim.inflight):
            # a warp may leave only once the copies it started have landed
            raise ProtocolError(f"{pr.name} left with an asynchronous copy in flight")

    if not sim.abort:
        if sim.inflight or sim.mma_queue:
            raise ProtocolError("kernel ended with copies or MMAs in flight")
        for t in range(2):
            o = sim.res.get(f"O{t}", "free")
            if not (o == "free" or o[0] == "read"):
                raise ProtocolError(f"O{t} not read out at the end: {o}")
        for b in range(p.q_bufs):
            q = sim.res.get(f"q{b}")
            if isinstance(q, tuple) and q and q[0] == "O":
                raise ProtocolError(f"the staged O of {q[1]} in q{b} was never stored")
    else:
        if sim.inflight or sim.mma_queue:
            raise ProtocolError("abort path ended with copies or MMAs in flight")
    return sim
