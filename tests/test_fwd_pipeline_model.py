"""Happens-before model of the attention-forward kernel's pipeline (CPU only).

fa_fwd_kernel.cuh coordinates two TMA producer warps (Q and K; V), a
score-MMA issuer, a P.V-MMA issuer, eight softmax warps and four epilogue
warps through mbarriers (waited on by parity), hardware named barriers and
the asynchronous completion of TMA copies and tcgen05 MMAs.  This test
replays every role's sequence of barrier operations and buffer accesses in
the order the kernel executes them, under random interleavings and random
completion times of the copies and MMAs, and checks:

* no data race: every two conflicting accesses to a buffer (the Q, K and V
  stages in shared memory; the S, P and O regions of TMEM per lane quarter
  and half row; the row-max exchange slots and the two statistics slots the
  softmax warps hand to the epilogue warps) are ordered by happens-before.  Vector clocks travel through mbarrier phases, named
  barrier generations, MMA commits and TMA completions (the model and its
  rules are in _pipeline_model.py);
* parity safety: a wait for phase n of an mbarrier (parity n mod 2) starts
  with at least n phases complete and returns before phase n + 1 completes,
  so the parity cannot alias;
* every arrival lands in the phase it is meant for, on mbarriers and named
  barriers (no overrun), and no named-barrier generation is left incomplete;
* no deadlock.

Both designs are modelled: d = 128 (one softmax state per row split over two
warps, a P buffer, S released once read) and the d = 64 split design (two
independent half-row states, P over S, S released once P.V is done); in
both, the softmax warps leave each item's statistics in one of two slots
and the epilogue warps read them, then O once the item's last P.V is done.  Planted
protocol mistakes -- each a single wait or barrier left out -- are caught,
which shows that the check can fail.  Only the healthy path is modelled; the
abort path of the named barriers is checked in test_barrier_protocol.py.
"""
import random

import pytest

from _pipeline_model import Deadlock, Model, Violation

KSTAGES = {128: 3, 64: 4}
VSTAGES = {128: 2, 64: 4}
WARPS = 8  # softmax warps: warp w serves lane quarter w % 4, half row w // 4


EPI_WARPS = 4  # epilogue warps: warp 8 + q serves lane quarter q


def mbarrier_counts(split):
    """Expected arrivals per phase, as the kernel initialises them."""
    c = {"QFULL": 1, "QEMPTY": 1, "OFINAL": 1, "OFREE": EPI_WARPS, "DRAIN0": 1, "DRAIN1": 1}
    for slot in range(2):
        c[f"STFULL{slot}"] = WARPS
        c[f"STFREE{slot}"] = EPI_WARPS
    for s in range(max(KSTAGES.values())):
        c[f"KFULL{s}"] = c[f"KEMPTY{s}"] = 1
    for s in range(max(VSTAGES.values())):
        c[f"VFULL{s}"] = c[f"VEMPTY{s}"] = 1
    for b in range(2):
        c[f"SFULL{b}"] = 1
        if split:
            c[f"PFULL{b}"] = c[f"PFULL{2 + b}"] = WARPS // 2
            c[f"ODONE{b}"] = 1
        else:
            c[f"SREAD{b}"] = WARPS
    if not split:
        c["PFULL"] = WARPS
        c["ODONE"] = 1
    return c


# ----------------------------------------------------------------- the roles
# The roles yield the actions listed in _pipeline_model.


def producer_qk(items, D, mut):
    """Warp 12: K of every tile, and an item's Q after its first K tile,
    once the previous item's last score MMA is done."""
    KS = KSTAGES[D]
    gk = 0

    def load_q(k):
        yield ("wait", "QEMPTY", k - (2 if mut == "q_early" else 1))
        yield ("tma", "QFULL", k, ["Q"])

    for k, n in enumerate(items):
        for j in range(n):
            s = gk % KS
            yield ("wait", f"KEMPTY{s}", gk // KS - (2 if mut == "k_early" else 1))
            yield ("tma", f"KFULL{s}", gk // KS, [f"K{s}"])
            gk += 1
            if j == 0:
                yield from load_q(k)
    # drain: every copy lands before the CTA exits
    if items:
        yield ("wait", "QFULL", len(items) - 1)
    for g in range(max(0, gk - KS), gk):
        yield ("wait", f"KFULL{g % KS}", g // KS)


def producer_v(items, D, mut):
    """Warp 15: V of every tile as soon as its stage is free."""
    VS = VSTAGES[D]
    gv = 0
    for n in items:
        for _ in range(n):
            s = gv % VS
            yield ("wait", f"VEMPTY{s}", gv // VS - (2 if mut == "v_early" else 1))
            yield ("tma", f"VFULL{s}", gv // VS, [f"V{s}"])
            gv += 1
    for g in range(max(0, gv - VS), gv):
        yield ("wait", f"VFULL{g % VS}", g // VS)


def score_issuer(items, D, split, mut):
    KS = KSTAGES[D]
    s_all = [f"S{{}}.{q}.{h}" for q in range(4) for h in range(2)]
    g = 0

    def signal_s_ready(gg):
        yield ("wait", f"SFULL{gg & 1}", gg >> 1)
        if split:
            yield ("nb_arrive", 5 + gg % 3, 5)
            yield ("nb_arrive", 8 + gg % 3, 5)
        else:
            yield ("nb_arrive", 5 + gg % 3, 9)

    for k, n in enumerate(items):
        for j in range(n):
            b, s = g & 1, g % KS
            if g >= 1:
                yield from signal_s_ready(g - 1)
            if j == 0:
                yield ("wait", "QFULL", k)
            yield ("wait", f"KFULL{s}", g // KS)
            if g >= 2 and mut != "no_s_release":
                yield ("wait", f"ODONE{b}" if split else f"SREAD{b}", (g - 2) >> 1)
            yield ("mma", "S", ["Q", f"K{s}"], [x.format(b) for x in s_all], [])
            yield ("commit", "S", f"KEMPTY{s}", g // KS)
            yield ("commit", "S", f"SFULL{b}", g >> 1)
            if j == n - 1:
                yield ("commit", "S", "QEMPTY", k)
            g += 1
    if g >= 1:
        yield from signal_s_ready(g - 1)
    yield ("commit", "S", "DRAIN0", 0)
    yield ("wait", "DRAIN0", 0)


def pv_issuer(items, D, split, mut):
    VS = VSTAGES[D]
    g = 0
    for k, n in enumerate(items):
        if mut != "no_ofree":
            yield ("wait", "OFREE", k - 1)
        for j in range(n):
            s, b = g % VS, g & 1
            yield ("wait", f"VFULL{s}", g // VS)
            if split:
                for h in range(2):
                    yield ("wait", f"PFULL{2 * (0 if mut == 'pv_one_half' else h) + b}", g >> 1)
                    yield ("mma", "O", [f"S{b}.{q}.{h}" for q in range(4)] + [f"V{s}"], [],
                           [f"O{h}.{q}.{c}" for q in range(4) for c in range(2)] + [f"L{h}.{q}" for q in range(4)])
                yield ("commit", "O", f"VEMPTY{s}", g // VS)
                yield ("commit", "O", f"ODONE{b}", g >> 1)
            else:
                yield ("wait", "PFULL", g)
                yield ("mma", "O", [f"P.{q}.{h}" for q in range(4) for h in range(2)] + [f"V{s}"], [],
                       [f"O.{q}.{h}" for q in range(4) for h in range(2)])
                yield ("commit", "O", f"VEMPTY{s}", g // VS)
                yield ("commit", "O", "ODONE", g)
            if j == n - 1:
                yield ("commit", "O", "OFINAL", k)
            g += 1
    yield ("commit", "O", "DRAIN1", 0)
    yield ("wait", "DRAIN1", 0)


def softmax_warp(w, items, D, split, need, mut):
    """need[(key, g)]: the tile raises the row max enough to rescale; the key
    is the lane quarter at d = 128 (both halves of a row decide alike) and the
    warp in the split design (each half keeps its own reference max)."""
    q, h = w & 3, w >> 2
    g = 0
    for k, n in enumerate(items):
        for j in range(n):
            b = g & 1
            if split:
                yield ("nb_sync", 5 + 3 * h + g % 3, 5)
                yield ("rd", f"S{b}.{q}.{h}")
                if j > 0 and need[(w, g)]:
                    if mut != "no_rescale_wait":
                        yield ("wait", f"ODONE{(g - 1) & 1}", (g - 1) >> 1)
                    for r in (f"O{h}.{q}.0", f"O{h}.{q}.1", f"L{h}.{q}"):
                        yield ("wr", r)
                yield ("wr", f"S{b}.{q}.{h}")  # P over this half's scores
                yield ("arrive", f"PFULL{2 * h + b}", g >> 1)
            else:
                yield ("nb_sync", 5 + g % 3, 9)
                yield ("rd", f"S{b}.{q}.{h}")
                yield ("arrive", f"SREAD{b}", g >> 1)
                yield ("wr", f"MX.{q}.{b}.{h}")
                if mut != "no_pair":
                    yield ("nb_sync", 1 + q, 2)
                yield ("rd", f"MX.{q}.{b}.{h ^ 1}")
                waited = g == 0
                if j > 0 and need[(q, g)]:
                    if mut != "no_rescale_wait":
                        yield ("wait", "ODONE", g - 1)
                        waited = True
                    yield ("wr", f"O.{q}.{h}")
                if not waited and mut != "no_odone":
                    yield ("wait", "ODONE", g - 1)
                yield ("wr", f"P.{q}.{h}")
                yield ("arrive", "PFULL", g)
            g += 1
        # the item's statistics to the epilogue warps: slot k & 1, once the
        # epilogue warps have read what it held two items ago
        one = mut == "one_slot_no_free"
        slot = 0 if one else k & 1
        if split and mut != "no_stfree" and not one:
            yield ("wait", f"STFREE{slot}", (k >> 1) - 1)
        yield ("wr", f"ST{slot}.{q}.{h}")
        yield ("arrive", f"STFULL{slot}", k if one else k >> 1)


def epilogue_warp(q, items, split, mut):
    """Warp 8 + q: the statistics of lane quarter q, then (once the item's
    last P.V is done) O and l~ of its rows; O_FREE once they are read."""
    for k, n in enumerate(items):
        one = mut == "one_slot_no_free"
        slot = 0 if one else k & 1
        phase = k if one else k >> 1
        yield ("wait", f"STFULL{slot}", phase)
        yield ("rd", f"ST{slot}.{q}.0")
        yield ("rd", f"ST{slot}.{q}.1")
        if split:
            yield ("arrive", f"STFREE{slot}", phase)
        if mut != "no_ofinal":
            yield ("wait", "OFINAL", k)
        if split:
            for r in (f"O0.{q}.0", f"O0.{q}.1", f"L0.{q}", f"O1.{q}.0", f"O1.{q}.1", f"L1.{q}"):
                yield ("rd", r)
        else:
            yield ("rd", f"O.{q}.0")
            yield ("rd", f"O.{q}.1")
        yield ("arrive", "OFREE", k)


def simulate(D, seed, items=None, mut=None):
    rng = random.Random(seed * 7919 + D)
    if items is None:
        items = [rng.randint(1, 5) for _ in range(rng.randint(1, 4))]
    split = D == 64
    tiles = sum(items)
    p_need = rng.choice([0.0, 0.3, 1.0])
    keys = range(WARPS) if split else range(4)
    need = {(key, g): rng.random() < p_need for key in keys for g in range(tiles)}
    roles = {
        "producer_qk": producer_qk(items, D, mut),
        "producer_v": producer_v(items, D, mut),
        "score": score_issuer(items, D, split, mut),
        "pv": pv_issuer(items, D, split, mut),
    }
    for w in range(WARPS):
        roles[f"softmax{w}"] = softmax_warp(w, items, D, split, need, mut)
    for q in range(EPI_WARPS):
        roles[f"epilogue{q}"] = epilogue_warp(q, items, split, mut)
    Model(mbarrier_counts(split), seed).run(roles)


@pytest.mark.parametrize("D", [128, 64])
def test_forward_pipeline_is_race_free_and_parity_safe(D):
    for seed in range(120):
        simulate(D, seed)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("items", [[1], [1, 1, 1, 1, 1], [7], [2, 1, 3], [1, 6, 1]])
def test_forward_pipeline_item_shapes(D, items):
    """Single-tile items (the Q, O-free and O-final barriers turn over every
    tile), one long item (the K and V rings wrap several times) and mixes."""
    for seed in range(40):
        simulate(D, seed, items=items)


MUTANTS = [
    # (designs, mistake, what it breaks)
    ((128, 64), "no_s_release", "the score issuer reuses an S buffer without waiting for its readers"),
    ((128,), "no_odone", "P is written before the previous P.V has read the P buffer"),
    ((128, 64), "no_rescale_wait", "O is rescaled while the previous P.V may still add to it"),
    ((128,), "no_pair", "the partner's row max is read without the pair barrier"),
    ((64,), "pv_one_half", "a half's P.V waits for the other half's P only"),
    ((128, 64), "no_ofree", "the next item's first P.V overwrites O before the epilogue warps read it"),
    ((128, 64), "no_ofinal", "the epilogue warps read O before the item's last P.V is done"),
    ((128, 64), "k_early", "the producer refills a K stage one phase too early"),
    ((128, 64), "v_early", "the V producer refills a V stage one phase too early"),
    ((128, 64), "q_early", "the producer loads the next item's Q before the last score MMA read Q"),
    ((64,), "no_stfree", "the softmax warps overwrite a statistics slot before the epilogue read it"),
    ((128, 64), "one_slot_no_free", "one statistics slot, reused without waiting until it has been read"),
]


@pytest.mark.parametrize("designs, mut, what", MUTANTS, ids=[m[1] for m in MUTANTS])
def test_planted_protocol_mistakes_are_caught(designs, mut, what):
    for D in designs:
        caught = None
        for seed in range(400):
            try:
                simulate(D, seed, mut=mut)
            except (Violation, Deadlock) as e:
                caught = e
                break
        assert caught is not None, f"d = {D}: not caught: {what}"


def test_statistics_slot_reuse_at_d128_needs_no_wait():
    """At d = 128 the kernel writes a statistics slot without waiting for the
    epilogue warps to have read what it held two items ago: that read is
    implied.  The statistics of item k + 2 are written after P of item k + 2,
    whose write waited for a P.V of item k + 1 or later; those P.Vs follow
    the first P.V of item k + 1, which waited for "O read out" of item k, and
    the epilogue warps read item k's statistics before they arrive on that.
    The main tests run the kernel's protocol (no such wait at d = 128); this
    one runs long item sequences of single tiles, where the statistics turn
    over fastest.  In the split design (P over S, no P.V wait before a P) the
    wait is needed, as the planted mistake no_stfree shows."""
    for seed in range(200):
        simulate(128, seed, items=[1] * 8)
        simulate(128, seed, items=[1, 2, 1, 1, 3, 1])
