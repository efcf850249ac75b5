"""Pins for the commit oracle (CPU only): a hand-worked example crossing a
page boundary, and sentinel checks that nothing outside slots L .. L + a
changes."""

import numpy as np

import oracle


def test_hand_example_crosses_page_boundary():
    # 2 layers, 1 sequence, Hkv = 1, D = 2, P = 16, L = 14; pages: logical 0 ->
    # physical 2, logical 1 -> physical 0.  Path root(0) -> 2 -> 3, a = 2.
    layers, pages, Hkv, P, D = 2, 3, 1, 16, 2
    kc = np.full((layers, pages, Hkv, P, D), 0xDEAD, dtype=np.uint16)
    vc = np.full((layers, pages, Hkv, P, D), 0xBEEF, dtype=np.uint16)
    T = 4
    tk = np.arange(layers * T * Hkv * D, dtype=np.uint16).reshape(layers, T, Hkv, D) + 100
    tv = tk + 1000
    table = np.array([[2, 0, 1]], dtype=np.int32)
    k2, v2, nl = oracle.kv_commit(kc, vc, tk, tv, table, np.array([14]), np.array([0, 4]),
                                  [[0, 2, 3]], np.array([2]))
    assert list(nl) == [17]
    for layer in range(2):
        # slot 14 -> physical page 2 offset 14 <- node 0
        assert list(k2[layer, 2, 0, 14]) == list(tk[layer, 0, 0])
        # slot 15 -> physical page 2 offset 15 <- node 2
        assert list(k2[layer, 2, 0, 15]) == list(tk[layer, 2, 0])
        # slot 16 -> physical page 0 offset 0 <- node 3
        assert list(k2[layer, 0, 0, 0]) == list(tk[layer, 3, 0])
        assert list(v2[layer, 0, 0, 0]) == list(tv[layer, 3, 0])
    changed = (k2 != kc).any(axis=-1)
    assert changed.sum() == 2 * 3
    # inputs are untouched
    assert (kc == 0xDEAD).all()


def test_only_committed_slots_change():
    rng = np.random.default_rng(0)
    B, layers, Hkv, P, D = 3, 2, 2, 16, 8
    L = [5, 31, 16]
    a = [0, 3, 6]
    need = [-(-(L[b] + 8) // P) for b in range(B)]
    npg = sum(need)
    perm = rng.permutation(npg)
    table = np.full((B, max(need)), -1, np.int32)
    o = 0
    for b in range(B):
        table[b, : need[b]] = perm[o: o + need[b]]
        o += need[b]
    kc = rng.integers(0, 1 << 16, size=(layers, npg, Hkv, P, D)).astype(np.uint16)
    vc = rng.integers(0, 1 << 16, size=(layers, npg, Hkv, P, D)).astype(np.uint16)
    cu = np.array([0, 8, 16, 24])
    tk = rng.integers(0, 1 << 16, size=(layers, 24, Hkv, D)).astype(np.uint16)
    tv = rng.integers(0, 1 << 16, size=(layers, 24, Hkv, D)).astype(np.uint16)
    paths = [[0], [0, 1, 2, 3], [0, 1, 2, 3, 4, 5, 6]]
    k2, v2, nl = oracle.kv_commit(kc, vc, tk, tv, table, np.array(L), cu, paths, np.array(a))
    assert list(nl) == [L[b] + a[b] + 1 for b in range(B)]
    expect_k = kc.copy()
    for b in range(B):
        for j, node in enumerate(paths[b]):
            s = L[b] + j
            expect_k[:, table[b, s // P], :, s % P, :] = tk[:, cu[b] + node]
    np.testing.assert_array_equal(k2, expect_k)
    diff = (v2 != vc).any(axis=(0, 2, 4))
    assert diff.sum() <= sum(x + 1 for x in a)
