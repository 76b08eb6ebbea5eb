"""Host-side measurement helpers (no GPU): the load statistics bench.py reports."""
import numpy as np

import oracle


def test_load_stats_counts_and_special_cases():
    """Load statistics of a routing: counts equal the oracle permutation's per-expert counts and
    per-group row counts; an even batch has max/mean 1 and cv 0; a batch sent to one expert has
    max/mean E."""
    from compressed_expert_two_b300 import workload
    rng = np.random.default_rng(7)
    T, G, K, kg, ke = 300, 4, 4, 2, 2
    E = G * K
    gm = np.arange(E) // K
    gidx = np.stack([rng.permutation(G)[:kg] for _ in range(T)]).astype(np.int32)
    eidx = np.concatenate([np.stack([g * K + rng.permutation(K)[:ke] for g in gidx[:, j]]) for j in range(kg)],
                          axis=1).astype(np.int32)
    st = workload.load_stats(gidx, eidx, G, E)
    ref = oracle.permute(eidx, gm, G, ke)
    counts = ref["expert_count"]
    assert st["expert"]["max"] == counts.max() and st["expert"]["min"] == counts.min()
    rows = np.diff(ref["row_begin"])
    assert st["group"]["max"] == rows.max() and st["group"]["min"] == rows.min()
    assert np.isclose(st["expert"]["max_over_mean"], counts.max() / counts.mean())
    even = workload.load_stats(np.tile(np.arange(G), T // G)[:, None], np.tile(np.arange(E), 2)[:, None], G, E)
    assert even["group"]["max_over_mean"] == 1.0 and even["expert"]["cv"] == 0.0
    one = workload.load_stats(np.zeros((T, 1), np.int32), np.zeros((T, 1), np.int32), G, E)
    assert one["expert"]["max_over_mean"] == E and one["group"]["max_over_mean"] == G


def test_load_stats_counts_only_active_assignments():
    """With the across-groups reading's picked-slot mask, unpicked (zero-gate) slots add no load."""
    from compressed_expert_two_b300 import workload
    eidx = np.array([[0, 1, 4, 5], [0, 2, 4, 6]], dtype=np.int32)
    active = np.array([[True, False, True, False], [True, True, False, False]])
    st = workload.load_stats(np.array([[0, 1], [0, 1]]), eidx, 2, 8, active=active)
    assert st["expert"]["max"] == 2 and st["expert"]["min"] == 0      # expert 0 twice, 1/5/6 never
    assert np.isclose(st["expert"]["max_over_mean"], 2 / (4 / 8))
