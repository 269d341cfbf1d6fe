"""The attention kernel's barrier protocol, checked on the CPU.

tests/protocol_model.py re-states every role of the kernel (K/V and Q
producers, the MMA issuer, the two softmax warpgroups, the four rotating
warps of the rotary variant) and runs them under many adversarial schedules
together with the asynchronous TMA copies and the tensor core's in-order MMA
queue. The cases cover both head dimensions (ring of 4 and 8 slots), causal and
non-causal tiles with ragged tails and Sq != Sk, sub-tiles with no key block,
GQA head packing, split-key mode, the rotary variant's four-arrival "Q ready"
barriers, the additive-mask variant's output staged in a Q buffer and stored
by the Q warp, and the abort path (a stalled wait that runs out; an abort raised at
an arbitrary moment). Planted protocol mistakes must each be caught.
"""
import os
import sys
import types

import pytest

import protocol_model as M

HERE = os.path.dirname(os.path.abspath(__file__))

CASES = [
    M.Params(),                                                        # causal, ring of 4
    M.Params(D=64),                                                    # ring of 8
    M.Params(causal=False, Sq=300, Sk=700),                            # ragged, upper sub-tile empty
    M.Params(Sq=1000, Sk=300),                                         # Sq > Sk: lower sub-tiles with no block
    M.Params(Sq=100, Sk=1000),
    M.Params(B=2, Hq=4, Hkv=2, Sq=1200, Sk=1200, grid=3, cta=2),        # snake waves, mixed lengths
    M.Params(B=2, Hq=4, Hkv=2, Sq=1200, Sk=1200, grid=3, cta=0, D=64),
    M.Params(num_splits=3, Sq=100, Sk=1500, grid=2, cta=1),            # split keys
    M.Params(num_splits=4, Sq=1, Sk=2000, Hq=8, Hkv=2, pack_shift=2, grid=2, cta=0),   # packed decode
    M.Params(Hq=8, Hkv=2, pack_shift=2, Sq=40, Sk=900),
    M.Params(rope=True),                                               # four-arrival "Q ready"
    M.Params(rope=True, D=64, causal=False, Sq=600, Sk=500),
    M.Params(rope=True, B=2, Hq=2, Hkv=1, Sq=700, Sk=700, grid=2, cta=1),
    M.Params(Sq=128, Sk=128, Hq=1, Hkv=1),                             # one block per tile
    M.Params(Sq=256, Sk=256, Hq=3, Hkv=3, causal=False),
    # tiles taken over from CTAs that had not started (cluster launch control)
    M.Params(B=2, Hq=4, Hkv=2, Sq=1200, Sk=1200, cta=3, steal_seed=1),
    M.Params(B=2, Hq=4, Hkv=2, Sq=1000, Sk=300, cta=0, steal_seed=2, D=64),
    M.Params(rope=True, B=2, Hq=2, Hkv=1, Sq=900, Sk=900, cta=1, steal_seed=3),
    M.Params(num_splits=3, Hq=4, Hkv=1, pack_shift=2, Sq=16, Sk=1500, cta=0, steal_seed=4),
    # additive-mask variant: warpgroup 1's O staged in its Q buffer, stored by the Q warp
    M.Params(additive=True),
    M.Params(additive=True, causal=False, Sq=300, Sk=700),
    M.Params(additive=True, B=2, Hq=4, Hkv=2, Sq=1200, Sk=1200, cta=3, steal_seed=1),
    M.Params(additive=True, Sq=1000, Sk=300, B=2, Hq=2, Hkv=2, grid=2, cta=1),
    M.Params(additive=True, num_splits=3, Sq=100, Sk=1500, grid=2, cta=1),     # split keys: no staging
]

SEEDS = range(12)


def _id(p):
    return f"D{p.D}_c{int(p.causal)}_B{p.B}H{p.Hq}-{p.Hkv}_S{p.Sq}-{p.Sk}_sp{p.num_splits}_r{int(p.rope)}" \
           f"_pk{p.pack_shift}_g{p.grid}.{p.cta}_st{p.steal_seed}_m{int(p.additive)}"


@pytest.mark.parametrize("p", CASES, ids=_id)
def test_protocol_has_no_deadlock_or_race(p):
    assert M.schedule(p), "the case must give the CTA some work"
    for seed in SEEDS:
        M.run(p, seed=seed, bias=(seed % 4) / 4)


@pytest.mark.parametrize("p", [CASES[0], CASES[1], CASES[7], CASES[10], CASES[15], CASES[21]], ids=_id)
def test_stalled_wait_aborts_every_role(p):
    """The stall hook: the MMA issuer waits on a barrier nothing signals; its
    wait runs out, and every role must then finish, shutdown waits included."""
    stalled = M.Params(**{**p.__dict__, "debug_stall": True})
    for seed in SEEDS:
        sim = M.run(stalled, seed=seed, timeouts=True)
        assert sim.timed_out


@pytest.mark.parametrize("p", [CASES[0], CASES[2], CASES[5], CASES[11], CASES[16], CASES[19], CASES[22]], ids=_id)
def test_abort_at_any_moment_terminates(p):
    """Some wait runs out at an arbitrary step: no role may hang afterwards."""
    total = M.run(p, seed=0).steps
    for seed in SEEDS:
        for frac in (0.05, 0.3, 0.6, 0.9):
            M.run(p, seed=seed, abort_at=max(2, int(total * frac)), timeouts=True)


# ------------------------------------------------------------ planted bugs

MUTATIONS = {
    # the MMA issuer never releases a ring slot after the V products
    "kv_empty_commit_dropped": ('            yield ("commit", f"kv_empty{vs}")\n', ""),
    # the producer waits for the slot's current phase instead of the previous one
    "ring_wait_wrong_phase": ('ok = yield ("wait", f"kv_empty{slot}", st["fill"] // S - 1)',
                              'ok = yield ("wait", f"kv_empty{slot}", st["fill"] // S)'),
    # the producer reuses a slot without waiting for its release
    "ring_wait_skipped": ('        if st["fill"] >= S:\n', "        if False:\n"),
    # V before K in the ring: the issuer takes the wrong tiles
    "ring_order_swapped": ('("KV", kv, ti.b, ti.hk, ti.kb0 + blk)', '("KV", 1 - kv, ti.b, ti.hk, ti.kb0 + blk)'),
    # Q buffers released one block early
    "q_release_early": ("                    if j + 1 == n0 - 1:\n", "                    if j + 2 == n0 - 1:\n"),
    # the next S_t written before P_t has been consumed
    "qk_before_pv": (
        "            if j < n0:\n"
        "                if not (yield from wait_p(0)):\n"
        "                    alive = False\n"
        "                    break\n"
        "                yield _pv(sim, ti, 0, vs, j)\n"
        "                if j == n0 - 1:\n"
        "                    yield (\"commit\", \"o_full0\")\n"
        "            if more:\n"
        "                ks, ok = yield from acquire(k_seen)\n"
        "                if not ok:\n"
        "                    alive = False\n"
        "                    break\n"
        "                if j + 1 < n0:\n"
        "                    yield _qk(sim, ti, 0, q_buf[0], ks, j + 1)\n"
        "                    yield (\"commit\", \"s_full0\")\n",
        "            if more:\n"
        "                ks, ok = yield from acquire(k_seen)\n"
        "                if not ok:\n"
        "                    alive = False\n"
        "                    break\n"
        "                if j + 1 < n0:\n"
        "                    yield _qk(sim, ti, 0, q_buf[0], ks, j + 1)\n"
        "                    yield (\"commit\", \"s_full0\")\n"
        "            if j < n0:\n"
        "                if not (yield from wait_p(0)):\n"
        "                    alive = False\n"
        "                    break\n"
        "                yield _pv(sim, ti, 0, vs, j)\n"
        "                if j == n0 - 1:\n"
        "                    yield (\"commit\", \"o_full0\")\n"),
    # "O ready" committed before the last P V product
    "o_full_early": ("                yield _pv(sim, ti, 0, vs, j)\n                if j == n0 - 1:\n"
                     "                    yield (\"commit\", \"o_full0\")",
                     "                if j == n0 - 1:\n                    yield (\"commit\", \"o_full0\")\n"
                     "                yield _pv(sim, ti, 0, vs, j)"),
    # the softmax does not wait for S
    "softmax_skips_s_wait": ('            landed = yield ("wait", f"s_full{t}", s_cnt)',
                             '            landed = True'),
    # "Q ready" of the rotary variant with three arrivals instead of four
    "rope_ready_one_arrival": ('("q_rdy", p.q_bufs, 4)', '("q_rdy", p.q_bufs, 3)'),
    # a rotating warp rotates the buffer before its copy has landed
    "rope_skips_q_wait": ('            ok = yield ("wait", f"q_full{buf}", use)\n            if not ok:\n                return\n            yield _rotate(sim, buf, quarter)',
                          '            ok = True\n            yield _rotate(sim, buf, quarter)'),
    # the softmax counts its S phases per tile instead of continuously
    "softmax_phase_reset": ("        ok = True\n        for j in range(nb):", "        ok = True\n        s_cnt = 0\n        for j in range(nb):"),
    # the issuer waits for Q of the upper sub-tile on the lower sub-tile's buffer
    "q_buffer_mixup": ('ok = yield ("wait", f"{q_ready}{q_buf[1]}", q_slot(nq, 1, p.q_bufs)[1])',
                       'ok = yield ("wait", f"{q_ready}{q_buf[0]}", q_slot(nq, 0, p.q_bufs)[1])'),
    # the tile-ring producer overwrites entries without waiting for them to be freed
    "ring_producer_skips_wait": ("    if k >= p.tile_slots:\n", "    if False:\n"),
    # one arrival too few frees a tile-ring entry (a consumer not counted)
    "ring_consumer_undercount": ("        return 1 + 1 + 8 + (4 if self.rope else 0)", "        return 1 + 8 + (4 if self.rope else 0)"),
    # the producer leaves without waiting for a launch-control response in flight
    "clc_drain_skipped": ('                yield ("drain", "clc", st["clc"])       # the response must land before the CTA exits\n', ""),
    # the producer reads the launch-control response without waiting for it
    "clc_wait_skipped": ('            ok = yield ("wait", "clc", st["clc"])', '            ok = True'),
    # the Q warp stores a staged O without waiting for warpgroup 1 to write it
    "stage_wait_skipped": ('ok = yield ("wait", f"o_staged{wg}{idx % 2}", idx // 2)', 'ok = True'),
    # the Q warp waits for the other warpgroup's staging
    "stage_wrong_warpgroup": ('ok = yield ("wait", f"o_staged{wg}{idx % 2}", idx // 2)',
                              'ok = yield ("wait", f"o_staged{1 - wg}{idx % 2}", idx // 2)'),
    # the Q warp reloads a buffer that still holds a staged O
    "stage_store_skipped": ("        if staged[buf] is not None and not (yield from store_staged(buf)):\n",
                            "        if False:\n"),
    # one warp of warpgroup 1 does not report its staged rows
    "stage_arrival_missing": ('            for _ in range(4):                   # one arrival per warp, after its rows are written',
                              '            for _ in range(3):'),
    # the Q warp leaves without storing the last tiles' staged O
    "stage_final_store_skipped": ("        if not (yield from store_staged(buf)):\n            break\n    for b in range(p.q_bufs):",
                                  "        break\n    for b in range(p.q_bufs):"),
    # the K/V producer stops draining its copies on shutdown
    "drain_skipped": ('            yield ("drain", f"kv_full{s}", last // S)', "            pass"),
}

MUTATION_CASES = [CASES[0], CASES[1], CASES[2], CASES[5], CASES[7], CASES[10], CASES[12], CASES[15], CASES[16],
                  CASES[19], CASES[21],
                  M.Params(B=2, Hq=4, Hkv=2, Sq=1200, Sk=1200, grid=1, tile_slots=1)]


def _mutant(name):
    src = open(os.path.join(HERE, "protocol_model.py")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation {name} no longer applies"
    mod = types.ModuleType(f"protocol_model_{name}")
    sys.modules[mod.__name__] = mod            # dataclasses look their module up
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def _caught(mod, **kw):
    try:
        mod.run(**kw)
    except mod.ProtocolError:
        return True
    return False


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_protocol_bug_is_caught(name):
    mod = _mutant(name)
    for p in MUTATION_CASES:
        q = mod.Params(**p.__dict__)
        for seed in SEEDS:
            if _caught(mod, p=q, seed=seed, bias=(seed % 4) / 4):
                return
    for p in MUTATION_CASES:                           # shutdown mistakes show on the abort path
        q = mod.Params(**p.__dict__)
        total = M.run(p, seed=0).steps
        for seed in SEEDS:
            for frac in (0.1, 0.3, 0.5, 0.7, 0.9):
                if _caught(mod, p=q, seed=seed, timeouts=True, abort_at=max(2, int(total * frac)),
                           bias=(seed % 4) / 4):
                    return
    pytest.fail(f"planted protocol bug {name!r} was not detected")
