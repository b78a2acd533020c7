"""One whole hot-path step (expansion -> selection -> metadata -> attention -> accept +
compaction) through the library vs the oracle's step on the same seeded inputs."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import step as ostep
from oracle import tree
from tests import gpu_cases as gc
from tests.test_gpu_sampling import valid_sample

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_verify_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("name", ["llama8b", "tiny"])
def test_whole_step_matches_oracle(name):
    import tree_speculative_decoding_verify_gb300 as T
    w = W.WORKLOADS[name]
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    d = gc.dev()
    b = 0
    tokens, parents, _ = gc.oracle_tree(w, b)
    target = W.plant_target(w, b, tokens, parents, mode="first" if name == "tiny" else "walk")
    p_len = w.max_prefix
    q, k_new, v_new = W.new_qkv(w)
    k_pre, v_pre = W.prefix_kv(w, b, p_len)
    rnd = gc.as_bf16_f64 if dt == torch.bfloat16 else (lambda x: np.asarray(x, np.float64))
    max_depth = (w.depth + 1) if w.fixed_parents is None else max(tree.depths(list(parents)))
    want = ostep.hot_path_step(
        gc.level_logits(w, b) if w.fixed_parents is None else None, w.top_k, w.total_tokens,
        int(tokens[0]), rnd(q[b]), rnd(k_new[b]), rnd(v_new[b]), rnd(k_pre), rnd(v_pre), target,
        w.theta, gc.scale_of(w), max_depth + 1) if w.fixed_parents is None else None

    cap = int(np.ceil((p_len + w.num_nodes + 16) / 64) * 64)
    kc = torch.zeros(1, w.num_kv_heads, cap, w.head_dim, dtype=dt, device=d)
    vc = torch.zeros_like(kc)
    kc[0, :, :p_len] = gc.to_dev(k_pre, dt)
    vc[0, :, :p_len] = gc.to_dev(v_pre, dt)
    cache = T.KVCache(kc, vc)
    shape = T.TreeShape(1, w.num_q_heads, w.num_kv_heads, w.head_dim, p_len, vocab=w.vocab,
                        top_k=w.top_k, depth=w.depth, total_tokens=w.total_tokens,
                        fixed_nodes=w.num_nodes if w.fixed_parents is not None else 0,
                        fixed_max_depth=max_depth)
    hp = T.HotPath(shape, cache)
    prefix = gc.i32([p_len])
    if w.fixed_parents is not None:
        hp.set_tree(gc.i32([tokens]), gc.i32([parents]), gc.i32([w.num_nodes]))
        levels = None
    else:
        levels = [torch.from_numpy(x[None]).to(d) for x in gc.level_logits(w, b)]
    hp.step(levels, gc.i32(W.root_tokens(w)[:1]) if levels else None, gc.to_dev(q, dt),
            gc.to_dev(k_new, dt), gc.to_dev(v_new, dt), prefix, gc.i32([target]), w.theta,
            gc.scale_of(w))
    torch.cuda.synchronize()

    assert hp.tokens.cpu().numpy()[0].tolist() == tokens.tolist()
    assert hp.parents.cpu().numpy()[0].tolist() == parents.tolist()
    assert hp.meta_err.item() == 0 and hp.attn_err.item() == 0 and hp.acc_err.item() == 0
    if want is None:   # fixed tree: compare the parts the oracle step covers piecewise
        from oracle import accept, attention
        want = {}
        out, k_rot, v_t = attention.tree_verify_attention(
            rnd(q[b]), rnd(k_new[b]), rnd(v_new[b]), rnd(k_pre), rnd(v_pre), list(parents),
            w.theta, gc.scale_of(w))
        want["out"] = out
        want["path"], want["bonus"] = accept.greedy_walk(list(tokens), list(parents), list(target))
        want["mask"] = tree.pack_mask(tree.tree_mask(list(parents)))
        want["pos"] = tree.position_ids(list(parents), p_len)
    np.testing.assert_array_equal(hp.mask.cpu().numpy()[0].view(np.uint32), want["mask"])
    np.testing.assert_array_equal(hp.position_ids.cpu().numpy()[0], want["pos"])
    got = hp.out.float().cpu().numpy()[0]
    diff = np.abs(got - want["out"])
    if dt == torch.bfloat16:
        assert diff.max() <= gc.BF16_ATOL_MAX and diff.mean() <= gc.BF16_ATOL_MEAN
    else:
        assert diff.max() <= gc.F32_ATOL_MAX
    path = want["path"]
    assert hp.accept_len.item() == len(path)
    assert hp.accept_path.cpu().numpy()[0][:len(path)].tolist() == path
    assert hp.bonus.item() == want["bonus"]
    assert hp.new_prefix_len.item() == p_len + len(path)
    assert len(path) >= 2
    if "k_cache" in want:
        n = len(path)
        kv_got = kc[0, :, :p_len + n].float().cpu().numpy()
        np.testing.assert_allclose(kv_got, want["k_cache"][:, :p_len + n], rtol=2.0 ** -7,
                                   atol=1e-6)
        np.testing.assert_array_equal(vc[0, :, :p_len + n].float().cpu().numpy(),
                                      want["v_cache"][:, :p_len + n])


def test_step_with_the_lm_head_stage():
    """The step with the target's lm_head in it: the greedy token of every node comes from
    tsv_lm_head_argmax over the nodes' hidden states, and the walk follows it. Hidden
    states are planted (a scaled copy of the wanted token's weight row plus noise) so the
    oracle's argmax walks a chosen path; the oracle's argmax feeds the oracle's walk."""
    import math

    import tree_speculative_decoding_verify_gb300 as T
    from oracle import accept, lm_head

    w = W.WORKLOADS["llama8b"].with_(vocab=2048, top_k=4, depth=2, total_tokens=8,
                                     prefix=("fixed", 200), num_q_heads=8, num_kv_heads=2)
    d = gc.dev()
    hdim, p_len = 256, 200
    tokens, parents, _ = gc.oracle_tree(w, 0)
    planted = W.plant_target(w, 0, tokens, parents)
    t_max = w.num_nodes
    weight = gc.as_bf16_f64(next(W.lm_head_weight_blocks(w, w.vocab, hdim))[1])
    noise = W.lm_head_hidden(w, t_max, hdim) * 0.05
    hidden = gc.as_bf16_f64(4.0 * weight[planted] + noise)
    target, _ = lm_head.lm_head_argmax(hidden, weight)
    assert target.tolist() == planted.tolist()  # the planted margins hold in fp64
    path, bonus = accept.greedy_walk(list(tokens), list(parents), list(target))

    q, k_new, v_new = W.new_qkv(w)
    cap = 256
    kc = torch.zeros(1, 2, cap, 128, dtype=torch.bfloat16, device=d)
    vc = torch.zeros_like(kc)
    shape = T.TreeShape(1, 8, 2, 128, p_len, vocab=w.vocab, top_k=w.top_k, depth=w.depth,
                        total_tokens=w.total_tokens, target_vocab=w.vocab)
    hp = T.HotPath(shape, T.KVCache(kc, vc))
    levels = [torch.from_numpy(x[None]).to(d) for x in gc.level_logits(w, 0)]
    bf = lambda x: gc.to_dev(x, torch.bfloat16)
    hp.step(levels, gc.i32(W.root_tokens(w)[:1]), bf(q), bf(k_new), bf(v_new), gc.i32([p_len]),
            None, w.theta, 1 / math.sqrt(128), hidden=bf(hidden[None]), lm_weight=bf(weight))
    torch.cuda.synchronize()
    assert hp.tokens.cpu().numpy()[0].tolist() == tokens.tolist()
    assert hp.target.cpu().numpy()[0, :t_max].tolist() == target.tolist()
    n = hp.accept_len.item()
    assert n == len(path) and n >= 1
    assert hp.accept_path.cpu().numpy()[0, :n].tolist() == list(path)
    assert hp.bonus.item() == bonus
    assert hp.kernels_per_step(lm_head=True) == hp.kernels_per_step() + 2


def test_step_with_non_greedy_acceptance():
    """The step with the non-greedy acceptance: at temperature 0 it is the greedy step
    (the same path, bonus and compacted cache) for any uniforms; at temperature 1 its path
    and token match the oracle's rejection walk on the step's tree."""
    import math

    import tree_speculative_decoding_verify_gb300 as T
    from oracle import sampling

    w = W.WORKLOADS["llama8b"].with_(vocab=2048, top_k=4, depth=2, total_tokens=8,
                                     prefix=("fixed", 200), num_q_heads=8, num_kv_heads=2)
    d = gc.dev()
    tokens, parents, _ = gc.oracle_tree(w, 0)
    t_max = w.num_nodes
    logits = W.target_logits(w, 0, tokens, parents, w.vocab, t_max)
    u = W.uniforms(w, 0, t_max)
    q, k_new, v_new = W.new_qkv(w)
    bf = lambda x: gc.to_dev(x, torch.bfloat16)
    levels = [torch.from_numpy(x[None]).to(d) for x in gc.level_logits(w, 0)]
    results = {}
    for mode in ("greedy", "t0", "t1"):
        kc = torch.zeros(1, 2, 256, 128, dtype=torch.bfloat16, device=d)
        kc[0, :, :200] = 1.0
        vc = kc.clone()
        shape = T.TreeShape(1, 8, 2, 128, 200, vocab=w.vocab, top_k=w.top_k, depth=w.depth,
                            total_tokens=w.total_tokens)
        hp = T.HotPath(shape, T.KVCache(kc, vc))
        args = (levels, gc.i32(W.root_tokens(w)[:1]), bf(q), bf(k_new), bf(v_new), gc.i32([200]))
        if mode == "greedy":
            target = np.argmax(logits, axis=1).astype(np.int32)
            hp.step(*args, gc.i32([target]), w.theta, 1 / math.sqrt(128))
        else:
            temp = 0.0 if mode == "t0" else 1.0
            smp = dict(target_logits=torch.from_numpy(logits[None]).to(d),
                       temperature=torch.tensor([temp], device=d),
                       top_k=torch.zeros(1, dtype=torch.int32, device=d),
                       top_p=torch.ones(1, device=d), min_p=torch.zeros(1, device=d),
                       u_node=torch.from_numpy(u[None, :t_max].copy()).to(d),
                       u_final=torch.from_numpy(u[t_max:].copy()).to(d))
            hp.step(*args, None, w.theta, 1 / math.sqrt(128), sampling=smp)
        torch.cuda.synchronize()
        n = hp.accept_len.item()
        results[mode] = (hp.accept_path.cpu().numpy()[0, :n].tolist(), hp.bonus.item(),
                         kc.cpu().clone())
    assert results["t0"][0] == results["greedy"][0] and results["t0"][1] == results["greedy"][1]
    assert torch.equal(results["t0"][2], results["greedy"][2])
    probs = [sampling.filter_probs(logits[i], 1.0) for i in range(len(tokens))]
    trace = []
    path, tok = sampling.rejection_walk(list(tokens), list(parents), probs, u[:t_max],
                                        float(u[t_max]), trace=trace)
    margin = min([abs(x - a) for kind, x, a in trace if kind == "test"], default=1.0)
    final = [(x, p) for kind, x, p in trace if kind == "final"][-1]
    if margin > 1e-5:
        assert results["t1"][0] == path
        # the sampled token: the oracle's, or (a near-tie of the inverse CDF) a token the
        # oracle's final distribution gives for a uniform within 1e-6 of this one
        assert results["t1"][1] == tok or valid_sample(results["t1"][1], final), (
            results["t1"][1], tok)
