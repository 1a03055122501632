"""Work schedules of the persistent kernels (CPU only).

The integer walks of fa_fwd_kernel.cuh (item_of, item_of_rank, the
heavy/light pair walk and the cost-ordered snake) and of fa_bwd_kernel.cuh
(item_of, the pair walk), mirrored here with the grid sizes fa_api.cu
launches, are checked for every size and grid the GPU tests do not reach:

* every work item is taken by exactly one CTA, and every CTA gets work;
* a causal heavy/light pair costs the same number of key tiles in every head
  (an even number of query blocks);
* the cost-ordered walk balances the small causal problem it is chosen for
  (B4 H16 N2048: 98.6% against 84.2% for pairs, counting an item's epilogue
  as half a key tile).
"""
import pytest

BM = BN = 128  # forward: query rows per item, keys per tile
BKV, BQ = 128, 64  # backward: keys per item, query rows per step


# ------------------------------------------------------------ forward
def fwd_m_block(i, M):
    t = i % M
    return (t >> 1) if (t & 1) else (M - 1 - (t >> 1))


def fwd_n_kv(i, M, N, causal):
    n_all = (N + BN - 1) // BN
    q0 = fwd_m_block(i, M) * BM
    return min(n_all, (q0 + BM - 1) // BN + 1) if causal else n_all


def fwd_item_of_rank(r, BH, M):
    if r >= BH * M:
        return BH * M
    level = r // BH
    bh = r - level * BH
    m = M - 1 - level
    t = 2 * (M - 1 - m) if 2 * (M - 1 - m) < M else 2 * m + 1
    return bh * M + t


def fwd_walk(c, G, BH, M, snake):
    """Items CTA c takes, in order."""
    items = BH * M
    out, step = [], 0
    i = fwd_item_of_rank(c, BH, M) if snake else 2 * c
    while i < items:
        out.append(i)
        step += 1
        if snake:
            i = fwd_item_of_rank(step * G + ((G - 1 - c) if (step & 1) else c), BH, M)
        else:
            i = i + 1 if (step & 1) else i - 1 + 2 * G
    return out


def fwd_grid(BH, M, snake, sms):
    return min(BH * M if snake else (BH * M + 1) // 2, sms)


# ------------------------------------------------------------ backward
def bwd_walk(c, G, items):
    out, step, i = [], 0, 2 * c
    while i < items:
        out.append(i)
        step += 1
        i = i + 1 if (step & 1) else i - 1 + 2 * G
    return out


def bwd_item(i, num_kb, Np, causal):
    t = i % num_kb
    kb = (t >> 1) if (t & 1) else (num_kb - 1 - (t >> 1))
    m0 = (kb * BKV) // BQ if causal else 0
    return i // num_kb, kb, Np // BQ - m0


def _cover(walks, items):
    seen = [0] * items
    for w in walks:
        assert w, "a CTA without work"
        for i in w:
            seen[i] += 1
    assert all(s == 1 for s in seen), "an item taken twice or never"


@pytest.mark.parametrize("snake", [False, True])
def test_forward_walks_cover_every_item_once(snake):
    for BH in (1, 2, 3, 5, 16, 33):
        for N in (1, 127, 128, 129, 256, 1000, 2048, 4096, 5000):
            M = (N + BM - 1) // BM
            for sms in (1, 2, 3, 7, 152):
                G = fwd_grid(BH, M, snake, sms)
                _cover([fwd_walk(c, G, BH, M, snake) for c in range(G)], BH * M)


def test_item_of_rank_is_a_bijection_heaviest_first():
    for BH in (1, 3, 8):
        for M in range(1, 40):
            items = [fwd_item_of_rank(r, BH, M) for r in range(BH * M)]
            assert sorted(items) == list(range(BH * M))
            costs = [fwd_m_block(i, M) for i in items]
            assert costs == sorted(costs, reverse=True)


def test_causal_pairs_cost_the_same():
    for M in range(2, 64, 2):
        N = M * BM
        for BH in (1, 4):
            costs = {fwd_n_kv(2 * p, M, N, True) + fwd_n_kv(2 * p + 1, M, N, True) for p in range(BH * M // 2)}
            assert costs == {M + 1}


def test_snake_balances_the_small_causal_problem():
    BH, N, sms = 4 * 16, 2048, 152
    M = N // BM

    def balance(snake):
        G = fwd_grid(BH, M, snake, sms)
        loads = [sum(fwd_n_kv(i, M, N, True) + 0.5 for i in fwd_walk(c, G, BH, M, snake)) for c in range(G)]
        return sum(loads) / len(loads) / max(loads), len(loads)

    pairs, g_pairs = balance(False)
    snake, g_snake = balance(True)
    assert g_pairs == g_snake == sms
    assert pairs == pytest.approx(0.842, abs=1e-3)
    assert snake == pytest.approx(0.986, abs=1e-3)


def test_backward_walk_covers_every_item_once():
    for BH in (1, 2, 5, 16):
        for N in (1, 63, 64, 65, 130, 1000, 4096):
            num_kb = (N + BKV - 1) // BKV
            Np = (N + BQ - 1) // BQ * BQ
            items = BH * num_kb
            for sms in (1, 2, 3, 152):
                G = min((items + 1) // 2, sms)
                _cover([bwd_walk(c, G, items) for c in range(G)], items)
            for causal in (False, True):
                for i in range(items):
                    bh, kb, nq = bwd_item(i, num_kb, Np, causal)
                    assert 0 <= bh < BH and 0 <= kb < num_kb
                    assert nq >= 1  # the diagonal query block is always in range
