"""Pins for the oracle's RoPE and tree-masked attention: closed forms and the path
equivalence the handbook page checks (each node's result equals an ordinary causal
pass over prefix + its own root-to-node chain)."""
import math

import numpy as np
import pytest

from oracle import attention, tree


def causal_attention_last_row(q_last, keys, values, scale):
    """Plain decode attention: the last query sees every key (no mask at all)."""
    s = [float(np.dot(q_last, k)) * scale for k in keys]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    z = sum(w)
    return sum((wi / z) * np.asarray(v, np.float64) for wi, v in zip(w, values))


def test_rope_closed_forms():
    x = np.array([[0.3, -1.7]])
    for p in (0, 1, 5, 1000):
        out = attention.apply_rope(x, [p], 10000.0)[0]
        c, s = math.cos(p), math.sin(p)
        assert np.allclose(out, [0.3 * c + 1.7 * s, -1.7 * c + 0.3 * s], atol=1e-14)
    # second frequency of D=4 is theta^(-2/4): 0.1 for theta = 100
    y = np.array([[0.0, 1.0, 0.0, 0.0]])
    out = attention.apply_rope(y, [10], 100.0)[0]
    assert np.allclose(out, [0.0, math.cos(1.0), 0.0, math.sin(1.0)], atol=1e-14)
    z = np.random.default_rng(0).normal(size=(3, 2, 64))
    assert np.allclose(attention.apply_rope(z, [0, 0, 0], 1e4), z)


def test_rope_is_a_rotation_by_relative_position():
    rng = np.random.default_rng(1)
    q, k = rng.normal(size=(1, 128)), rng.normal(size=(1, 128))
    d1 = attention.apply_rope(q, [70], 1e4) @ attention.apply_rope(k, [50], 1e4).T
    d2 = attention.apply_rope(q, [1020], 1e4) @ attention.apply_rope(k, [1000], 1e4).T
    assert math.isclose(float(d1[0, 0]), float(d2[0, 0]), rel_tol=1e-9)
    r = attention.apply_rope(q, [12345], 1e4)
    assert math.isclose(float(np.linalg.norm(r)), float(np.linalg.norm(q)), rel_tol=1e-12)


def test_equal_keys_give_the_mean_of_visible_values():
    rng = np.random.default_rng(2)
    keys = np.tile(rng.normal(size=(1, 8)), (6, 1))
    vals = rng.normal(size=(6, 8))
    mask = np.array([[1, 0, 1, 1, 0, 0]], dtype=bool)
    out = attention.masked_attention(rng.normal(size=(1, 8)), keys, vals, mask, 0.7)
    assert np.allclose(out[0], vals[[0, 2, 3]].mean(axis=0), atol=1e-14)


def tiny_case(parents, p_len=5, hq=4, hkv=2, d=8, seed=0):
    rng = np.random.default_rng(seed)
    t = len(parents)
    return dict(q=rng.normal(size=(t, hq, d)), k_new=rng.normal(size=(t, hkv, d)),
                v_new=rng.normal(size=(t, hkv, d)), k_prefix=rng.normal(size=(hkv, p_len, d)),
                v_prefix=rng.normal(size=(hkv, p_len, d)))


@pytest.mark.parametrize("parents", [
    [-1, 0, 0, 1, 1, 2],                       # the handbook's six-node example
    [-1, 0, 0, 1, 1, 2, 2, 3, 4, 5, 6],        # the [2,2,1] diagram
    [-1, 0, 1, 1, 0, 4, 2, 6, 6, 3],
])
def test_each_node_equals_causal_pass_over_its_chain(parents):
    c = tiny_case(parents)
    theta, scale = 1e4, 1 / math.sqrt(8)
    out, k_rot, _ = attention.tree_verify_attention(parents=parents, theta=theta, scale=scale, **c)
    p_len = c["k_prefix"].shape[1]
    hq, hkv = c["q"].shape[1], c["k_new"].shape[1]
    for i in range(len(parents)):
        chain, j = [], i
        while j != -1:
            chain.append(j)
            j = parents[j]
        chain.reverse()
        pos = list(range(p_len, p_len + len(chain)))      # consecutive positions
        for h in range(hq):
            kv = h // (hq // hkv)
            kc = attention.apply_rope(c["k_new"][chain, kv][:, None], pos, theta)[:, 0]
            keys = list(c["k_prefix"][kv]) + list(kc)
            vals = list(c["v_prefix"][kv]) + list(c["v_new"][chain, kv])
            qi = attention.apply_rope(c["q"][[i], h][:, None], [pos[-1]], theta)[0, 0]
            ref = causal_attention_last_row(qi, keys, vals, scale)
            assert np.allclose(out[i, h], ref, atol=1e-12, rtol=1e-12)


def test_root_only_tree_is_decode_attention():
    c = tiny_case([-1], p_len=9, seed=3)
    out, _, _ = attention.tree_verify_attention(parents=[-1], theta=1e4, scale=0.5, **c)
    for h in range(4):
        kv = h // 2
        q0 = attention.apply_rope(c["q"][:, h][:, None], [9], 1e4)[0, 0]
        k0 = attention.apply_rope(c["k_new"][:, kv][:, None], [9], 1e4)[0, 0]
        ref = causal_attention_last_row(q0, list(c["k_prefix"][kv]) + [k0],
                                        list(c["v_prefix"][kv]) + [c["v_new"][0, kv]], 0.5)
        assert np.allclose(out[0, h], ref, atol=1e-12)


def test_non_ancestors_do_not_matter():
    parents = [-1, 0, 0, 1, 1, 2, 2, 3, 4, 5, 6]
    c = tiny_case(parents, seed=4)
    out, _, _ = attention.tree_verify_attention(parents=parents, theta=1e4, scale=0.3, **c)
    mask = tree.tree_mask(parents)
    rng = np.random.default_rng(5)
    for victim in range(1, len(parents)):
        c2 = {k: v.copy() for k, v in c.items()}
        c2["k_new"][victim] = rng.normal(size=c2["k_new"][victim].shape)
        c2["v_new"][victim] = rng.normal(size=c2["v_new"][victim].shape)
        out2, _, _ = attention.tree_verify_attention(parents=parents, theta=1e4, scale=0.3, **c2)
        for i in range(len(parents)):
            same = np.allclose(out[i], out2[i], atol=1e-13)
            assert same == (not mask[i, victim]), (i, victim)   # root row: only itself


def test_gqa_head_mapping():
    parents = [-1, 0, 1]
    c = tiny_case(parents, hq=6, hkv=3, seed=6)
    out, _, _ = attention.tree_verify_attention(parents=parents, theta=1e4, scale=0.4, **c)
    for kv in range(3):
        single = {"q": c["q"][:, 2 * kv:2 * kv + 2], "k_new": c["k_new"][:, kv:kv + 1],
                  "v_new": c["v_new"][:, kv:kv + 1], "k_prefix": c["k_prefix"][kv:kv + 1],
                  "v_prefix": c["v_prefix"][kv:kv + 1]}
        o1, _, _ = attention.tree_verify_attention(parents=parents, theta=1e4, scale=0.4, **single)
        assert np.allclose(out[:, 2 * kv:2 * kv + 2], o1, atol=1e-14)
