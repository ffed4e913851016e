"""Pins for the oracle's routing and token-to-expert sort (CPU only).

Routing is checked against brute-force sorting and scipy's softmax / expit
(library routines on a different path: a full softmax over all experts, then
renormalisation).  The sort is checked against a hand-derived case and the
invariants the pages state: sum of expert counts = routed slots,
a_map o c_map = identity, rows of an expert in ascending token order,
#virtual experts <= E + T*k/kBlockN.
"""
import math

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
import synth


def test_route_hand_case():
    lg = np.array([[1.0, 3.0, 3.0, -1.0, 2.0, 3.0]], np.float32)
    ids, w = oracle.route(lg, 3)
    assert ids.tolist() == [[1, 2, 5]]
    np.testing.assert_allclose(w, [[1 / 3] * 3], rtol=1e-15)
    ids, w = oracle.route(lg, 4)
    assert ids.tolist() == [[1, 2, 5, 4]]
    d = 3 + math.exp(-1)
    np.testing.assert_allclose(w, [[1 / d, 1 / d, 1 / d, math.exp(-1) / d]], rtol=1e-15)


@pytest.mark.parametrize("T,Eg,k", [(7, 8, 2), (5, 64, 16), (3, 896, 16)])
def test_route_matches_brute_force_and_softmax(T, Eg, k):
    rng = np.random.default_rng(T * Eg)
    lg = rng.normal(0, 1, (T, Eg)).astype(np.float32)
    lg[:, ::7] = np.round(lg[:, ::7])  # plenty of exact ties
    ids, w = oracle.route(lg, k)
    for t in range(T):
        order = sorted(range(Eg), key=lambda e: (-float(lg[t, e]), e))[:k]
        assert ids[t].tolist() == order
        p = softmax(lg[t].astype(np.float64))
        ref = p[order] / p[order].sum()
        np.testing.assert_allclose(w[t], ref, rtol=1e-13)
        assert abs(w[t].sum() - 1) < 1e-14
        assert all(w[t, j] >= w[t, j + 1] for j in range(k - 1))


def test_route_shared_expert_weight():
    cfg = synth.CONFIGS["skewed_shared_t256"].replace(T=16)
    lg = synth.logits_host(cfg)
    sl = synth.shared_logit_host(cfg)
    ids, w = oracle.route(lg, cfg.top_k, 1, sl, 0.5)
    assert (ids[:, -1] == cfg.E_global).all()
    ref = expit(synth.bf16_bits_to_f64(sl[:, 0])) * 0.5
    np.testing.assert_allclose(w[:, -1], ref, rtol=1e-14)
    # the routed part is unchanged by the shared append
    ids0, w0 = oracle.route(lg, cfg.top_k)
    np.testing.assert_array_equal(ids[:, :-1], ids0)
    np.testing.assert_array_equal(w[:, :-1], w0)


def _hand_sort_ids():
    return np.array([[3, 0, 4], [2, 3, 4], [1, 2, 4]], np.int32)


def test_sort_hand_case():
    s = oracle.sort(_hand_sort_ids(), E_global=4, E_local=2, expert_offset=2, num_shared=1, block_n=2)
    assert s["counts"].tolist() == [2, 2, 3]
    assert s["offsets"].tolist() == [0, 2, 4, 7]
    assert s["c_map"].tolist() == [2, -1, 4, 0, 3, 5, -1, 1, 6]
    assert s["a_map"].tolist() == [3, 7, 0, 4, 2, 5, 8]
    assert s["vinfo"].tolist() == [[0, 0, 2, 0], [1, 2, 2, 0], [2, 4, 2, 0], [2, 6, 1, 1]]


def check_sort_invariants(ids, s, E_global, E_local, expert_offset, S, B):
    T, kp = ids.shape
    flat = ids.reshape(-1)
    local = np.where((flat >= expert_offset) & (flat < expert_offset + E_local), flat - expert_offset, -1)
    local = np.where((flat >= E_global) & (flat < E_global + S), E_local + flat - E_global, local)
    R = int((local >= 0).sum())
    assert int(s["counts"].sum()) == R
    assert s["offsets"][-1] == R
    assert ((s["c_map"] >= 0) == (local >= 0)).all()
    # a_map o c_map = id on the routed slots, c_map o a_map = id on rows
    routed = np.nonzero(local >= 0)[0]
    np.testing.assert_array_equal(s["a_map"][s["c_map"][routed]], routed)
    np.testing.assert_array_equal(s["c_map"][s["a_map"]], np.arange(R))
    # rows of each expert hold that expert's slots in ascending slot order
    for e in range(E_local + S):
        rows = np.arange(s["offsets"][e], s["offsets"][e + 1])
        slots = s["a_map"][rows]
        assert (local[slots] == e).all()
        assert (np.diff(slots) > 0).all()
    # virtual experts tile each expert's rows in chunks of B, in order
    assert s["num_v"] <= (E_local + S) + R // B + (1 if R % B else 0)
    assert s["num_v"] <= (E_local + S) + (T * kp) // B
    cover = np.zeros(R, np.int32)
    for e_, first, tok, c in s["vinfo"]:
        assert 1 <= tok <= B and first == s["offsets"][e_] + c * B
        cover[first:first + tok] += 1
    assert (cover == 1).all()


@pytest.mark.parametrize("name,T,B", [("tiny", 4, 16), ("decode_t32", 32, 32), ("ep_slice_t64", 64, 16),
                                      ("skewed_shared_t256", 256, 32), ("decode_t32", 7, 16),
                                      ("decode_t32", 1, 32), ("prefill_t32768", 512, 128)])
def test_sort_invariants_on_routed_configs(name, T, B):
    cfg = synth.CONFIGS[name].replace(T=T, block_n=B)
    lg = synth.logits_host(cfg)
    sl = synth.shared_logit_host(cfg)
    ids, _ = oracle.route(lg, cfg.top_k, cfg.num_shared, sl, cfg.shared_scale)
    s = oracle.sort(ids, cfg.E_global, cfg.E_local, cfg.expert_offset, cfg.num_shared, B)
    check_sort_invariants(ids, s, cfg.E_global, cfg.E_local, cfg.expert_offset, cfg.num_shared, B)


def test_sort_masked_and_duplicate_ids():
    # -1 (masked) and out-of-slice ids get no row; a repeated id inside a token
    # still gets distinct rows in slot order.
    ids = np.array([[-1, 5, 5], [7, -1, 2], [5, 9, 3]], np.int32)
    s = oracle.sort(ids, E_global=10, E_local=6, expert_offset=2, num_shared=0, block_n=16)
    check_sort_invariants(ids, s, 10, 6, 2, 0, 16)
    assert s["c_map"].tolist() == [-1, 2, 3, 5, -1, 0, 4, -1, 1]


def test_sort_ep_slices_partition_the_rows():
    cfg = synth.CONFIGS["ep_slice_t64"]
    lg = synth.logits_host(cfg)
    ids, _ = oracle.route(lg, cfg.top_k)
    lo = oracle.sort(ids, 896, 448, 0, 0, 16)
    hi = oracle.sort(ids, 896, 448, 448, 0, 16)
    full = oracle.sort(ids, 896, 896, 0, 0, 16)
    assert lo["offsets"][-1] + hi["offsets"][-1] == full["offsets"][-1] == 64 * 16
    assert ((lo["c_map"] >= 0) ^ (hi["c_map"] >= 0)).all()
