"""tsv_accept_and_compact vs the oracle (walk and compaction), bit-exact."""
import numpy as np
import pytest
import torch

from oracle import accept, tree
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_verify_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def tokens_for(rng, parents, vocab=6):
    tok = [int(rng.integers(0, 1000))]
    for i in range(1, len(parents)):
        sib = {tok[j] for j in range(1, i) if parents[j] == parents[i]}
        free = [t for t in range(vocab + len(sib)) if t not in sib]
        tok.append(free[int(rng.integers(0, len(free)))])
    return np.array(tok, dtype=np.int32)


def planted_target(rng, tokens, parents, p=0.75, vocab=6):
    n = len(tokens)
    tgt = rng.integers(0, vocab, size=n).astype(np.int32)
    node = 0
    kids = tree.children_of(list(parents))
    while kids[node] and rng.random() < p:
        c = kids[node][int(rng.integers(0, len(kids[node])))]
        tgt[node] = tokens[c]
        node = c
    return tgt


def run(trees, tokens, targets, prefix, t_max, max_depth, cache=None, nn=None, valid=None):
    import tree_speculative_decoding_verify_gb300 as T
    b = len(trees)
    d = gc.dev()
    tok = np.full((b, t_max), -1, np.int32)
    tgt = np.zeros((b, t_max), np.int32)
    nxt = np.full((b, t_max), -1, np.int32)
    sib = np.full((b, t_max), -1, np.int32)
    for i, p in enumerate(trees):
        n = len(p)
        tok[i, :n], tgt[i, :n] = tokens[i], targets[i]
        a, s = tree.next_links(list(p))
        nxt[i, :n], sib[i, :n] = a, s
    nn = nn if nn is not None else [len(p) for p in trees]
    out = dict(accept_path=torch.full((b, max_depth + 1), 9, dtype=torch.int32, device=d),
               accept_len=torch.zeros(b, dtype=torch.int32, device=d),
               bonus_token=torch.zeros(b, dtype=torch.int32, device=d),
               slot_map=torch.zeros(b, max_depth + 1, 2, dtype=torch.int32, device=d),
               new_prefix_len=torch.zeros(b, dtype=torch.int32, device=d),
               err=torch.full((b,), 9, dtype=torch.int32, device=d))
    T.accept_and_compact(gc.i32(tok), gc.i32(nxt), gc.i32(sib), gc.i32(tgt), gc.i32(nn),
                         gc.i32(prefix), max_depth, cache, **out,
                         tree_valid=None if valid is None else gc.i32(valid))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def check_walk(got, trees, tokens, targets, prefix, max_depth, valid=None):
    for b, p in enumerate(trees):
        path, bonus = accept.greedy_walk(list(tokens[b]), list(p), list(targets[b]),
                                         True if valid is None else bool(valid[b]))
        assert got["err"][b] == 0
        assert got["accept_len"][b] == len(path)
        assert got["accept_path"][b].tolist() == path + [-1] * (max_depth + 1 - len(path))
        assert got["bonus_token"][b] == bonus
        assert got["new_prefix_len"][b] == prefix[b] + len(path)
        sm = accept.slot_map(int(prefix[b]), path)
        want = np.full((max_depth + 1, 2), -1, np.int32)
        want[:len(sm)] = sm
        np.testing.assert_array_equal(got["slot_map"][b], want)


def test_walk_random_trees():
    rng = np.random.default_rng(0)
    trees = [gc.random_tree(rng, int(rng.integers(1, 200)), 9) for _ in range(40)]
    tokens = [tokens_for(rng, p) for p in trees]
    targets = [planted_target(rng, t, p) for t, p in zip(tokens, trees)]
    prefix = rng.integers(0, 10000, size=40).astype(np.int32)
    got = run(trees, tokens, targets, prefix, 256, 9)
    check_walk(got, trees, tokens, targets, prefix, 9)


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_compaction_layers_and_pages(paged, dtype):
    import tree_speculative_decoding_verify_gb300 as T
    rng = np.random.default_rng(1)
    b, layers, hkv, d, t_max, depth = 6, 3, 4, 128, 61, 7
    trees = [gc.random_tree(rng, int(rng.integers(2, 62)), depth) for _ in range(b)]
    tokens = [tokens_for(rng, p) for p in trees]
    targets = [planted_target(rng, t, p, p=0.9) for t, p in zip(tokens, trees)]
    prefix = rng.integers(0, 300, size=b).astype(np.int32)
    cap = 448
    dev = gc.dev()
    if paged:
        per = cap // 64
        pool = b * per + 5
        table = rng.permutation(pool)[:b * per].reshape(b, per).astype(np.int32)
        k = torch.randn(layers, pool, hkv, 64, d, device=dev).to(dtype)
        v = torch.randn_like(k)
        cache = T.KVCache(k, v, gc.i32(table))
    else:
        table = None
        k = torch.randn(layers, b, hkv, cap, d, device=dev).to(dtype)
        v = torch.randn_like(k)
        cache = T.KVCache(k, v)

    def logical(t):  # [layers, b, hkv, cap, d] host view
        x = t.float().cpu().numpy()
        if not paged:
            return x
        out = np.zeros((layers, b, hkv, cap, d), np.float32)
        for bi in range(b):
            for j in range(cap // 64):
                out[:, bi, :, j * 64:(j + 1) * 64] = x[:, table[bi, j]]
        return out

    k0, v0 = logical(k), logical(v)
    got = run(trees, tokens, targets, prefix, t_max, depth, cache=cache)
    check_walk(got, trees, tokens, targets, prefix, depth)
    k1, v1 = logical(k), logical(v)
    for bi, p in enumerate(trees):
        path, _ = accept.greedy_walk(list(tokens[bi]), list(p), list(targets[bi]))
        np.testing.assert_array_equal(k1[:, bi], accept.compact(k0[:, bi], int(prefix[bi]), path))
        np.testing.assert_array_equal(v1[:, bi], accept.compact(v0[:, bi], int(prefix[bi]), path))


def test_bad_links_and_sizes():
    import tree_speculative_decoding_verify_gb300 as T
    d = gc.dev()
    tok = gc.i32([[5, 6, 7, 8], [5, 6, 7, 8], [5, 6, 7, 8]])
    nxt = gc.i32([[1, -1, -1, -1], [2, -1, -1, -1], [1, 3, -1, -1]])
    sib = gc.i32([[-1, 0, -1, -1], [-1, -1, 1, -1], [-1, 2, -1, -1]])
    tgt = gc.i32([[7, 0, 0, 0], [6, 0, 0, 0], [6, 8, 0, 0]])
    out = dict(accept_path=torch.zeros(3, 4, dtype=torch.int32, device=d),
               accept_len=torch.zeros(3, dtype=torch.int32, device=d),
               bonus_token=torch.zeros(3, dtype=torch.int32, device=d),
               slot_map=torch.zeros(3, 4, 2, dtype=torch.int32, device=d),
               new_prefix_len=torch.zeros(3, dtype=torch.int32, device=d),
               err=torch.zeros(3, dtype=torch.int32, device=d))
    # request 0: sibling link goes backwards; request 1: sibling link goes backwards
    # (2 -> 1); request 2: valid, accepts 0 -> 1 -> 3
    T.accept_and_compact(tok, nxt, sib, tgt, gc.i32([4, 4, 4]), gc.i32([0, 0, 0]), 3, None, **out)
    r = {k: v.cpu().numpy() for k, v in out.items()}
    assert r["err"].tolist() == [7, 7, 0]
    assert r["accept_len"].tolist() == [1, 1, 3]
    assert r["accept_path"][2].tolist() == [0, 1, 3, -1]
    T.accept_and_compact(tok, nxt, sib, tgt, gc.i32([0, 5, 4]), gc.i32([0, 0, -1]), 3, None, **out)
    assert out["err"].cpu().tolist() == [4, 4, 4]
    assert out["accept_len"].cpu().tolist() == [1, 1, 1]


def test_requests_without_a_tree_take_the_single_token_path():
    """tree_valid = 0 rows accept the root alone (bonus: the root's argmax) while the
    other requests of the batch walk their trees; the cache is untouched for them."""
    rng = np.random.default_rng(11)
    b, t_max, depth = 6, 40, 7
    trees = [gc.random_tree(rng, t_max, depth) for _ in range(b)]
    tokens, targets = [], []
    for p in trees:
        tok = rng.integers(0, 50, len(p)).astype(np.int32)
        tgt = rng.integers(0, 50, len(p)).astype(np.int32)
        for c in range(1, len(p)):  # plant matches so trees accept more than the root
            if rng.random() < 0.6:
                tgt[p[c]] = tok[c]
        tokens.append(tok)
        targets.append(tgt)
    valid = [1, 0, 1, 0, 0, 1]
    prefix = np.full(b, 100, np.int32)
    got = run(trees, tokens, targets, prefix, t_max, depth, valid=valid)
    check_walk(got, trees, tokens, targets, prefix, depth, valid=valid)
    assert all(got["accept_len"][i] == 1 for i in range(b) if not valid[i])
