"""The selection argument of the top-k pass, checked on the CPU against brute
force ("LLM speculative decoding study notes 02", sec. 5.4: the kept set is
the k largest logits, ties at the k-th value to the lower token id).

The pass keeps one key per group of 16 f consecutive tokens (the group's
maximum) and claims that the top-k lies within k groups: with T the k-th
largest group maximum, every group above T and the first groups (token
order) equal to T.  This model follows the pass's steps on bf16 keys --
segments of 256-token multiples, 16 tokens per lane, groups folded over f
lanes, the first bound from the lanes' largest keys, the second round on
16-token pieces when f > 1 -- and compares the kept ids with a sort of
(key descending, id ascending).  It shares no code with the CUDA sources or
the oracle."""
import numpy as np
import pytest

EPL, STEP, SEG_ALIGN, WARPS = 16, 512, 256, 8


def key16(bits):
    x = bits.astype(np.int64)
    x = np.where(x == 0x8000, 0, x)
    nan = (x & 0x7FFF) > 0x7F80
    k = np.where(x & 0x8000, (~x) & 0xFFFF, x | 0x8000)
    return np.where(nan, 0, k)


def kth(vals, k, lo, hi):
    """Largest T in [lo, hi) with at least k values >= T (lo qualifies, hi
    does not); also how many values exceed T."""
    n_hi = 0
    while hi - lo > 1:
        mid = (lo + hi) // 2
        c = int((vals >= mid).sum())
        if c >= k:
            lo = mid
        else:
            hi, n_hi = mid, c
    return lo, n_hi


def first_k(vals, T, quota):
    out, ties = [], 0
    for i, v in enumerate(vals):
        if v > T:
            out.append(i)
        elif v == T:
            if ties < quota:
                out.append(i)
            ties += 1
    return out


def model(bits, k, map_cap):
    keys = key16(bits)
    V = len(keys)
    fold = 1
    while -(-V // (16 * fold)) > map_cap:
        fold *= 2
    assert fold <= 16
    n_groups = -(-V // (16 * fold))
    seg = -(-(-(-V // WARPS)) // SEG_ALIGN) * SEG_ALIGN
    gmax = np.zeros(n_groups, np.int64)
    lane_key = np.zeros(WARPS * 32, np.int64)
    padded = np.concatenate([keys, np.full(WARPS * seg + STEP - V, 0x7F)])  # -inf beyond V
    for w in range(WARPS):
        s0, n = w * seg, max(0, min(seg, V - w * seg))
        for eb in range(0, n, STEP):
            piece = padded[s0 + eb:s0 + eb + STEP].reshape(32, EPL).max(axis=1)
            for lane in range(0, 32, fold):
                t = eb + EPL * lane
                if t < n:
                    g = piece[lane:lane + fold].max()
                    gmax[(s0 + t) // (16 * fold)] = g
                    lane_key[w * 32 + lane] = max(lane_key[w * 32 + lane], g)
    if n_groups <= k:
        chosen, T = list(range(n_groups)), 1
    else:
        lo, _ = kth(lane_key, k, lane_key.min(), lane_key.max() + 1)
        T, n_above = kth(gmax, k, lo, lane_key.max() + 1)
        chosen = first_k(gmax, T, k - n_above)
        assert len(chosen) == k
    pieces = [g * fold + j for g in chosen for j in range(fold)]
    if fold > 1 and len(pieces) > k:
        pmax = np.array([keys[p * 16:p * 16 + 16].max() if p * 16 < V else 0 for p in pieces])
        T, n_above = kth(pmax, k, max(T, 1), pmax.max() + 1)
        pieces = [pieces[i] for i in first_k(pmax, T, k - n_above)]
    ids = np.concatenate([np.arange(p * 16, min(p * 16 + 16, V)) for p in pieces])
    kstar, n_above = kth(keys[ids], k, max(T, 1), keys[ids].max() + 1)
    return sorted(int(ids[i]) for i in first_k(keys[ids], kstar, k - n_above))


def brute(bits, k):
    keys = key16(bits)
    order = np.lexsort((np.arange(len(keys)), -keys))
    return sorted(int(i) for i in order[:k])


def to_bf16(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF).astype(np.uint32)


ROWS = {
    "normal": lambda rng, V: rng.normal(0, 4, V),
    "integer": lambda rng, V: np.round(rng.normal(0, 2, V)),
    "constant": lambda rng, V: np.full(V, 1.5),
    "sorted": lambda rng, V: -1.1 * np.log1p(np.arange(V)) + rng.normal(0, 3, V),
    "narrow": lambda rng, V: 100 + rng.normal(0, 0.05, V),
    "masked": lambda rng, V: np.where(np.arange(V) < 300, rng.normal(0, 3, V), -np.inf),
}


@pytest.mark.parametrize("kind", sorted(ROWS))
@pytest.mark.parametrize("V,map_cap", [(100, 14336), (20001, 14336), (40000, 1000), (70000, 300)])
def test_top_k_lies_within_k_groups(kind, V, map_cap):
    rng = np.random.default_rng(V + len(kind))
    bits = to_bf16(ROWS[kind](rng, V))
    for k in (1, 7, 50, 64):
        if k < V:
            assert model(bits, k, map_cap) == brute(bits, k), (kind, V, k, map_cap)
