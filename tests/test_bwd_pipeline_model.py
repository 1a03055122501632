"""Happens-before model of the attention-backward kernel's pipeline (CPU only).

fa_bwd_kernel.cuh runs, per work item (128 keys of one head), steps of 64
query rows through a TMA producer, one MMA issuer, eight P/dS warps and four
dQ warps.  The producers signal the issuer through named barriers (P ready,
dP read, dS ready, dQ read, accumulators read); the issuer's MMAs signal
through commits (S full, dP full, dQ full, accumulators full, stage and K/V
empty).  Several buffers are released by implication rather than by a wait
of their own: S buffer b is rewritten once "dP(g-1) read" is met, because
every MMA issued before dP(g-1) -- among them dV(g-2), the last reader of
that buffer -- is then complete; dS buffer b is rewritten once dP(g) is
complete, because dK(g-2) and dQ(g-2), its readers, were issued before it.

This test replays every role's barrier operations and buffer accesses in the
kernel's order under random interleavings and random completion times (the
model and its rules are in _pipeline_model.py): no data race on K, V, the
Q/dO stages, the dS tiles, the dQ staging blocks or the S, dP, dQ, dV and dK
regions of TMEM; every parity wait safe; no overrun; no deadlock.  Planted
mistakes -- a signal met too late or not at all, a stage released early --
are caught.  The abort path of the named barriers is checked in
test_barrier_protocol.py.
"""
import random

import pytest

from _pipeline_model import Deadlock, Model, Violation

QSTAGES = 3
PDS = 8  # P/dS warps: warp w serves key lane quarter w % 4, query half w // 4


def mbarrier_counts():
    c = {"KVFULL": 1, "KVEMPTY": 1, "DPFULL": 1, "DQFULL": 1, "ACCFULL": 1, "DRAIN": 1, "SFULL0": 1, "SFULL1": 1}
    for s in range(QSTAGES):
        c[f"QFULL{s}"] = c[f"QEMPTY{s}"] = 1
    return c


ALL_S = [f"S{{}}.{q}.{h}" for q in range(4) for h in range(2)]
ALL_DP = [f"DP.{q}.{h}" for q in range(4) for h in range(2)]
ALL_DS = [f"DS{{}}.{q}.{h}" for q in range(4) for h in range(2)]
ALL_DQ = [f"DQ.{q}" for q in range(4)]
ALL_DV = [f"DV.{q}" for q in range(4)]
ALL_DK = [f"DK.{q}" for q in range(4)]
NB_PDS, NB_DQ = PDS + 1, 4 + 1  # warps meeting each named barrier (the issuer included)


def producer(items, mut):
    g = 0
    for k, n in enumerate(items):
        yield ("wait", "KVEMPTY", k - 1)
        yield ("tma", "KVFULL", k, ["K", "V"])
        for _ in range(n):
            s = g % QSTAGES
            yield ("wait", f"QEMPTY{s}", g // QSTAGES - 1)
            yield ("tma", f"QFULL{s}", g // QSTAGES, [f"Q{s}", f"DO{s}"])
            g += 1
    if items:
        yield ("wait", "KVFULL", len(items) - 1)
    for gg in range(max(0, g - QSTAGES), g):
        yield ("wait", f"QFULL{gg % QSTAGES}", gg // QSTAGES)


def issuer(items, mut):
    g = 0

    def issue_s_dp(gg):
        s, b = gg % QSTAGES, gg & 1
        yield ("wait", f"QFULL{s}", gg // QSTAGES)
        yield ("mma", "M", ["K", f"Q{s}"], [x.format(b) for x in ALL_S], [])
        yield ("commit", "M", f"SFULL{b}", gg >> 1)
        yield ("mma", "M", ["V", f"DO{s}"], ALL_DP, [])
        yield ("commit", "M", "DPFULL", gg)

    for k, n in enumerate(items):
        yield ("wait", "KVFULL", k)
        yield from issue_s_dp(g)
        for t in range(n):
            s, b = g % QSTAGES, g & 1
            more = t + 1 < n
            if t == 0 and k > 0:
                yield ("nb_sync", 7 + ((g - 1) & 1), NB_DQ)
                if mut != "no_acc_read":
                    yield ("nb_sync", 9 + ((k - 1) & 1), NB_DQ)
            yield ("nb_sync", 1 + b, NB_PDS)  # P(g) ready
            yield ("mma", "M", [x.format(b) for x in ALL_S] + [f"DO{s}"], [], ALL_DV)  # dV += P^T dO
            if mut == "qempty_after_dv":
                yield ("commit", "M", f"QEMPTY{s}", g // QSTAGES)
            if mut == "s_dp_before_dp_read" and more:
                yield from issue_s_dp(g + 1)
            yield ("nb_sync", 5 + b, NB_PDS)  # dP(g) read
            if mut != "s_dp_before_dp_read" and more:
                yield from issue_s_dp(g + 1)
            if mut != "no_ds_ready":
                yield ("nb_sync", 3 + b, NB_PDS)  # dS(g) ready
            yield ("mma", "M", [x.format(b) for x in ALL_DS] + [f"Q{s}"], [], ALL_DK)  # dK += dS^T Q
            if mut != "qempty_after_dv":  # dK(g) is the stage's last reader
                yield ("commit", "M", f"QEMPTY{s}", g // QSTAGES)
            if t > 0:
                yield ("nb_sync", 7 + ((g - 1) & 1), NB_DQ)  # dQ(g-1) read
            if mut == "no_ds_ready":
                yield ("nb_sync", 3 + b, NB_PDS)  # met late: the counts still match
            yield ("mma", "M", ["K"] + [x.format(b) for x in ALL_DS], ALL_DQ, [])  # dQ^T = K^T dS^T
            yield ("commit", "M", "DQFULL", g)
            if not more:
                yield ("commit", "M", "ACCFULL", k)
                yield ("commit", "M", "KVEMPTY", k)
            g += 1
    if items:
        yield ("nb_sync", 7 + ((g - 1) & 1), NB_DQ)
        if mut != "no_acc_read":
            yield ("nb_sync", 9 + ((len(items) - 1) & 1), NB_DQ)
    yield ("commit", "M", "DRAIN", 0)
    yield ("wait", "DRAIN", 0)


def dq_warp(q, items, D, mut):
    has_dims = q * 32 < D
    g = 0
    for k, n in enumerate(items):
        for _ in range(n):
            yield ("wait", "DQFULL", g)
            if has_dims:
                yield ("rd", f"DQ.{q}")
                yield ("nb_arrive", 7 + (g & 1), NB_DQ)
                if mut != "no_store_wait":
                    yield ("bulk_wait",)  # the previous reduce has read the staging block
                yield ("wr", f"STG.{q}")
                yield ("bulk", [f"STG.{q}"])  # TMA reduce-add into the fp32 dQ accumulator
            else:
                yield ("nb_arrive", 7 + (g & 1), NB_DQ)
            g += 1
        yield ("wait", "ACCFULL", k)
        yield ("rd", f"DV.{q}")
        yield ("rd", f"DK.{q}")
        yield ("nb_arrive", 9 + (k & 1), NB_DQ)
    yield ("bulk_wait",)


def pds_warp(w, items, mut):
    q, h = w & 3, w >> 2
    g = 0
    for n in items:
        for _ in range(n):
            b = g & 1
            yield ("wait", f"SFULL{b}", g >> 1)
            yield ("rd", f"S{b}.{q}.{h}")
            yield ("wr", f"S{b}.{q}.{h}")  # P over S
            yield ("nb_arrive", 1 + b, NB_PDS)
            if mut != "no_dp_wait":
                yield ("wait", "DPFULL", g)
            yield ("rd", f"DP.{q}.{h}")
            yield ("nb_arrive", 5 + b, NB_PDS)
            yield ("wr", f"DS{b}.{q}.{h}")
            yield ("nb_arrive", 3 + b, NB_PDS)
            g += 1


def simulate(D, seed, items=None, mut=None):
    rng = random.Random(seed * 104729 + D)
    if items is None:
        items = [rng.randint(1, 6) for _ in range(rng.randint(1, 4))]
    roles = {"producer": producer(items, mut)}
    roles["issuer"] = issuer(items, mut)
    for q in range(4):
        roles[f"dq{q}"] = dq_warp(q, items, D, mut)
    for w in range(PDS):
        roles[f"pds{w}"] = pds_warp(w, items, mut)
    Model(mbarrier_counts(), seed, queues=("M",)).run(roles)


@pytest.mark.parametrize("D", [128, 64])
def test_backward_pipeline_is_race_free_and_parity_safe(D):
    for seed in range(120):
        simulate(D, seed)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("items", [[1], [1, 1, 1, 1], [8], [2, 1, 5], [1, 7, 1]])
def test_backward_pipeline_item_shapes(D, items):
    """One-step items (K/V, the accumulators and the dQ signals turn over
    every step), one long item (the Q/dO ring wraps) and mixes."""
    for seed in range(40):
        simulate(D, seed, items=items)


MUTANTS = [
    ("s_dp_before_dp_read", "S and dP of the next step issued before dP(g) has been read out"),
    ("no_ds_ready", "dK(g) issued before the dS(g) tile is written"),
    ("no_acc_read", "the next item's first dV overwrites the accumulators before the epilogue read them"),
    ("qempty_after_dv", "the Q/dO stage released after dV instead of after dK, its last reader"),
    ("no_dp_wait", "the P/dS warps read dP before it is complete"),
    ("no_store_wait", "a dQ warp rewrites its staging block while the previous reduce may still read it"),
]


@pytest.mark.parametrize("mut, what", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_protocol_mistakes_are_caught(mut, what):
    caught = None
    for seed in range(400):
        try:
            simulate(128, seed, mut=mut)
        except (Violation, Deadlock) as e:
            caught = e
            break
    assert caught is not None, f"not caught: {what}"
