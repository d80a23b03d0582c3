"""Pins of the CPU oracle to facts it does not compute itself.

Each test checks the oracle against something fixed by the pages (a printed
worked value, under tests/golden/), by mathematics (a closed form, an
invariant, brute force on a tiny vocabulary) or by an independent library
routine (torch's attention, RMSNorm and SiLU).  A plausible slip anywhere in
the oracle -- a dropped term, a wrong sign or index, a transposed operand --
fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

import synth
from oracle import (Oracle, apply_rope, attention, combine_spellings, field_scores, first_token_result,
                    kv_bytes_per_token, length_normalised_scores, logsumexp64, per_level_scores, rms_norm,
                    rope_cos_sin, scores_to_result, silu)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Worked values printed on the pages
# --------------------------------------------------------------------------
def test_worked_softmax_example():
    g = golden("softmax_worked_example.json")
    tol = 0.5 * 10 ** -g["printed_decimals"] + 1e-12
    r1 = scores_to_result(g["logits"], 1.0)
    r2 = scores_to_result(g["logits"], 2.0)
    np.testing.assert_allclose(r1.probs, g["probs_T1"], atol=tol)
    np.testing.assert_allclose(r2.probs, g["probs_T2"], atol=tol)
    assert r1.label == r2.label == g["argmax"]


def test_spelling_sets_worked_example():
    """The page's inputs are themselves rounded to three decimals, so the
    check is an interval one: with every printed input moved to either end of
    its rounding interval, the oracle's outputs must bracket the printed
    outputs (each again +- half a unit of the last printed digit)."""
    g = golden("spelling_sets_worked_example.json")
    h = 0.5 * 10 ** -g["printed_decimals"]
    labels = [p["label"] for p in g["paths"]]

    def run(shift_true, shift_false):
        # shift_x moves the inputs of label x's paths by +-h (all outputs are
        # monotone in each input, so the corners bound them)
        ps = []
        for p in g["paths"]:
            d = shift_true if p["label"] == 0 else shift_false
            ps.append(np.sum(np.log(np.asarray(p["token_probs"]) + d)))
        s = combine_spellings(ps, labels)
        return np.exp(s), scores_to_result(s), np.exp(ps[1])

    lo_t, _, qlo = run(-h, -h)
    hi_t, _, qhi = run(+h, +h)
    assert qlo - h <= g["quoted_true_path"] <= qhi + h
    for c in (0, 1):
        assert lo_t[c] - h <= g["label_probs_unnormalised"][c] <= hi_t[c] + h
    p_lo = run(-h, +h)[1].probs[0]
    p_hi = run(+h, -h)[1].probs[0]
    assert p_lo - h <= g["renormalised_true"] <= p_hi + h
    # at the printed inputs the answer flips to True, as the page says
    mid = run(0.0, 0.0)[1]
    assert mid.label == 0 and abs(mid.probs[0] - g["renormalised_true"]) < 2e-3


def test_kv_cache_bytes_closed_form():
    g = golden("kv_cache_size.json")
    per_tok = kv_bytes_per_token(g["n_layers"], g["n_kv_heads"], g["head_dim"], g["elem_bytes"])
    assert per_tok == 28 * 2 * 2 * 128 * 2 == 28672
    mib = g["tokens"] * per_tok / 2 ** 20
    assert abs(mib - g["printed_mib"]) < 0.5       # 31.55 MiB, printed as "32 MiB"
    c = synth.model_config("1.5b")
    assert kv_bytes_per_token(c.n_layers, c.n_kv_heads, c.head_dim) == per_tok


# --------------------------------------------------------------------------
# Closed forms and properties of the scorer
# --------------------------------------------------------------------------
def test_two_way_softmax_is_logistic():
    rng = np.random.default_rng(0)
    for _ in range(50):
        a, b = rng.normal(0, 3, 2)
        T = rng.uniform(0.2, 5)
        r = scores_to_result([a, b], T)
        assert abs(r.probs[0] - 1 / (1 + np.exp(-(a - b) / T))) < 1e-12


def test_temperature_keeps_argmax_and_mass():
    rng = np.random.default_rng(1)
    for _ in range(50):
        s = rng.normal(-5, 3, int(rng.integers(2, 20)))
        base = scores_to_result(s, 1.0)
        for T in (0.1, 0.5, 2.0, 7.0):
            r = scores_to_result(s, T)
            assert r.label == base.label
            assert r.mass == base.mass
        assert abs(base.probs.sum() - 1) < 1e-12


def test_tie_goes_to_first_declared():
    assert scores_to_result([1.0, 1.0, 0.0]).label == 0
    assert scores_to_result([0.0, 2.0, 2.0]).label == 1
    assert scores_to_result([-3.0, -3.0]).margin == 0.0


def test_log_sum_exp_against_direct_sum():
    rng = np.random.default_rng(2)
    z = rng.normal(0, 2, (5, 300))
    direct = np.log(np.exp(z).sum(axis=1))
    np.testing.assert_allclose(logsumexp64(z), direct, rtol=0, atol=1e-12)
    big = z + 1000.0                      # the max shift keeps it finite
    np.testing.assert_allclose(logsumexp64(big), direct + 1000.0, atol=1e-9)


# --------------------------------------------------------------------------
# Decoder blocks against independent library routines
# --------------------------------------------------------------------------
def test_rms_norm_matches_torch():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1.7, (7, 64))
    g = rng.normal(1, 0.1, 64)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (64,), torch.tensor(g), eps=1e-6).numpy()
    np.testing.assert_allclose(rms_norm(x, g, 1e-6), ref, rtol=1e-12, atol=1e-12)


def test_silu_matches_torch():
    x = np.linspace(-9, 9, 101)
    np.testing.assert_allclose(silu(x), torch.nn.functional.silu(torch.tensor(x)).numpy(), atol=1e-14)


@pytest.mark.parametrize("Hq,Hkv,n,m", [(4, 2, 9, 9), (12, 2, 5, 21), (6, 6, 3, 11)])
def test_attention_matches_torch_sdpa(Hq, Hkv, n, m):
    """Causal GQA attention == torch's scaled_dot_product_attention, both for
    a plain sequence and for a chunk on top of earlier keys."""
    rng = np.random.default_rng(4)
    dh = 16
    q = rng.normal(0, 1, (n, Hq, dh))
    k = rng.normal(0, 1, (m, Hkv, dh))
    v = rng.normal(0, 1, (m, Hkv, dh))
    k_pos = np.arange(m)
    q_pos = np.arange(m - n, m)                  # the chunk is the last n keys
    ours = attention(q, k, v, q_pos, k_pos)
    allowed = torch.tensor(k_pos[None, :] <= q_pos[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q).transpose(0, 1)[None], torch.tensor(k).transpose(0, 1)[None],
        torch.tensor(v).transpose(0, 1)[None], attn_mask=allowed, enable_gqa=True)
    np.testing.assert_allclose(ours, ref[0].transpose(0, 1).numpy(), atol=1e-12)


def test_rope_properties():
    rng = np.random.default_rng(5)
    dh, theta = 16, 1e4
    x = rng.normal(0, 1, (1, 1, dh))
    # position 0 is the identity
    np.testing.assert_allclose(apply_rope(x, np.array([0]), theta), x, atol=0)
    # a rotation keeps the norm
    pos = np.array([1234])
    assert abs(np.linalg.norm(apply_rope(x, pos, theta)) - np.linalg.norm(x)) < 1e-12
    # q.k after RoPE depends only on the distance of the positions
    q = rng.normal(0, 1, (1, 1, dh))
    k = rng.normal(0, 1, (1, 1, dh))
    dots = [np.sum(apply_rope(q, np.array([a + 7]), theta) * apply_rope(k, np.array([a]), theta))
            for a in (0, 5, 300, 9000)]
    np.testing.assert_allclose(dots, dots[0], atol=1e-10)
    # rotate-half pairing: e_i moves in the plane of (e_i, e_{i+dh/2}) by pos * theta^(-2i/dh)
    for i in (0, 3, 7):
        e = np.zeros((1, 1, dh))
        e[0, 0, i] = 1
        m = 11
        out = apply_rope(e, np.array([m]), theta)[0, 0]
        ang = m * theta ** (-2 * i / dh)
        want = np.zeros(dh)
        want[i], want[i + dh // 2] = np.cos(ang), np.sin(ang)
        np.testing.assert_allclose(out, want, atol=1e-12)
    # dh = 2 is the textbook 2-D rotation by angle = position
    v2 = np.array([[[0.3, -1.1]]])
    a = 2.5
    R = np.array([[np.cos(a), -np.sin(a)], [np.sin(a), np.cos(a)]])
    np.testing.assert_allclose(apply_rope(v2, np.array([a]), theta)[0, 0], R @ v2[0, 0], atol=1e-12)
    c, s = rope_cos_sin(np.array([3]), 4, 100.0, np.float64)
    np.testing.assert_allclose(c[0], np.cos([3, 3 / 10]), atol=1e-15)
    np.testing.assert_allclose(s[0], np.sin([3, 3 / 10]), atol=1e-15)


# --------------------------------------------------------------------------
# Whole-decoder invariants on the tiny model
# --------------------------------------------------------------------------
def test_causality(tiny_oracle64):
    rng = np.random.default_rng(6)
    ids = rng.integers(0, 512, 20)
    ids2 = ids.copy()
    ids2[12:] = rng.integers(0, 512, 8)
    h1, _ = tiny_oracle64.forward(ids, np.arange(20))
    h2, _ = tiny_oracle64.forward(ids2, np.arange(20))
    np.testing.assert_allclose(h1[:12], h2[:12], atol=1e-13)
    assert np.abs(h1[12:] - h2[12:]).max() > 1e-3


def test_rope_enters_relatively_on_q_and_k(tiny_oracle64):
    """Where RoPE enters the decoder.  Rotating q and k by their positions
    makes every attention score depend on the positions' difference only, so
    moving a whole sequence by one offset leaves the logits unchanged (1e-10,
    fp64) -- with or without a cached prefix.  A rotation of q alone, of k
    alone, or of v as well breaks that.  Positions still matter: opening a gap
    inside the sequence changes every row after it and none before it, which
    a decoder without RoPE would not do."""
    o = tiny_oracle64
    rng = np.random.default_rng(21)
    ids = rng.integers(0, 512, 24)
    pos = np.arange(24)
    base = o.logits(o.forward(ids, pos)[0])
    for off in (1, 37, 1000):
        moved = o.logits(o.forward(ids, pos + off)[0])
        np.testing.assert_allclose(moved, base, atol=1e-10, rtol=0)
    # a cached prefix at shifted positions, extended at the matching ones
    k = 10
    for off in (0, 300):
        hp, (kk, vv) = o.forward(ids[:k], pos[:k] + off)
        from oracle.pcd_oracle import KVCache
        cache = KVCache(kk, vv, pos[:k] + off)
        ht, _ = o.forward(ids[k:], pos[k:] + off, cache)
        np.testing.assert_allclose(o.logits(ht), base[k:], atol=1e-10, rtol=0)
    gap = np.concatenate([pos[:12], pos[12:] + 5])
    opened = o.logits(o.forward(ids, gap)[0])
    np.testing.assert_allclose(opened[:12], base[:12], atol=1e-10, rtol=0)
    assert np.abs(opened[12:] - base[12:]).max(axis=1).min() > 1e-4


def test_gqa_equals_mha_with_repeated_kv_heads(tiny_weights):
    """GQA with group G equals MHA whose KV head h is KV head h // G."""
    import copy
    cfg = tiny_weights.cfg
    G = cfg.n_q_heads // cfg.n_kv_heads
    mha = copy.deepcopy(tiny_weights)
    for lw in mha.layers:
        for k in ("wk", "wv"):
            w = lw[k].reshape(cfg.n_kv_heads, cfg.head_dim, cfg.d_model)
            lw[k] = np.repeat(w, G, axis=0).reshape(cfg.n_q_heads * cfg.head_dim, cfg.d_model)
    from dataclasses import replace
    mha.cfg = replace(cfg, n_kv_heads=cfg.n_q_heads)
    ids = np.random.default_rng(7).integers(0, 512, 15)
    a, _ = Oracle(tiny_weights, np.float64).forward(ids, np.arange(15))
    b, _ = Oracle(mha, np.float64).forward(ids, np.arange(15))
    np.testing.assert_allclose(a, b, atol=1e-12)


def test_residual_passthrough(tiny_weights):
    """With W_o = 0 and W_down = 0 every layer adds zero, so the final hidden
    state is RMSNorm(embedding row) and the logits are E . that."""
    import copy
    w = copy.deepcopy(tiny_weights)
    for lw in w.layers:
        lw["wo"][:] = 0
        lw["w_down"][:] = 0
    o = Oracle(w, np.float64)
    ids = np.array([3, 77, 500])
    h, _ = o.forward(ids, np.arange(3))
    E = w.embed.astype(np.float64)
    x = E[ids]
    want = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(h, want, atol=1e-12)
    np.testing.assert_allclose(o.logits(h), want @ E.T, atol=1e-12)


def test_warm_extend_equals_cold_prefill(tiny_oracle64):
    ids = np.random.default_rng(8).integers(0, 512, 40)
    cold = tiny_oracle64.prefill(ids)
    warm = tiny_oracle64.extend(tiny_oracle64.prefill(ids[:25]), ids[25:])
    for a, b in zip(cold.k + cold.v, warm.k + warm.v):
        np.testing.assert_allclose(a, b, atol=1e-13)


# --------------------------------------------------------------------------
# PCD on the tiny workload
# --------------------------------------------------------------------------
def test_shared_prefix_equals_independent_sequences(tiny_oracle, tiny_oracle64, request1):
    """Scoring every label on the one prefix cache gives what running
    prefix + scaffold + label as a fresh sequence gives ("Not an
    approximation. The same arithmetic.")."""
    for orc, tol in ((tiny_oracle64, 1e-11), (tiny_oracle, 1e-5)):
        cache = orc.prefill(request1.prefix)
        for f in request1.fields:
            a = orc.score_field(f, cache=cache)
            b = orc.score_field(f, prefix=request1.prefix, mode="independent")
            np.testing.assert_allclose(a.scores, b.scores, atol=tol)
            np.testing.assert_allclose(a.probs, b.probs, atol=tol)
            assert a.label == b.label


def test_teacher_forced_sum_by_brute_force(tiny_oracle64, request1):
    """A label's score is the log of the product of its tokens' full-vocab
    probabilities, each taken as exp(z_t) / sum_v exp(z_v) written out on
    the logits of the complete sequence (V = 512, no max shift needed)."""
    orc = tiny_oracle64
    cache = orc.prefill(request1.prefix)
    P = request1.prefix
    for f in request1.fields:
        res = orc.score_field(f, cache=cache)
        for c, lab in enumerate(f.labels):
            seq = np.concatenate([P, f.scaffold, lab])
            h, _ = orc.forward(seq, np.arange(len(seq)))
            z = orc.logits(h)
            prob = 1.0
            for j, t in enumerate(lab):
                row = z[len(P) + len(f.scaffold) - 1 + j]
                prob *= np.exp(row[t]) / np.exp(row).sum()
            assert abs(np.log(prob) - res.scores[c]) < 1e-10
            np.testing.assert_allclose(res.token_logprobs[c].sum(), res.scores[c], atol=1e-12)


def test_single_token_fields_gather_equals_mask(tiny_oracle64, request1):
    """For single-token labels the candidate-only softmax of the gathered
    logits equals the oracle's probabilities (the full-vocab normaliser
    cancels) and equals a full softmax with -inf on every non-candidate."""
    orc = tiny_oracle64
    cache = orc.prefill(request1.prefix)
    for f in request1.fields:
        if any(len(l) != 1 for l in f.labels):
            continue
        z = orc.readout_logits(cache, f.scaffold)
        ids = [int(l[0]) for l in f.labels]
        g = np.exp(z[ids] - z[ids].max())
        g /= g.sum()
        masked = np.full_like(z, -np.inf)
        masked[ids] = z[ids]
        mexp = np.exp(masked - masked.max())
        mexp /= mexp.sum()
        res = orc.score_field(f, cache=cache)
        np.testing.assert_allclose(res.probs, g, atol=1e-12)
        np.testing.assert_allclose(mexp[ids], g, atol=1e-12)
        full = np.exp(z - z.max())
        full /= full.sum()
        np.testing.assert_allclose(res.probs * res.mass, full[ids], atol=1e-12)


def test_probability_bounds(tiny_oracle, request1):
    cache = tiny_oracle.prefill(request1.prefix)
    for f in request1.fields:
        r = tiny_oracle.score_field(f, cache=cache)
        assert abs(r.probs.sum() - 1) < 1e-12
        assert 0 <= r.mass <= 1 and 0 <= r.first_mass <= 1
        assert r.mass <= r.first_mass + 1e-12      # every label starts with an allowed token
        np.testing.assert_allclose(r.probs * r.mass, np.exp(r.scores), rtol=1e-10)


def test_first_token_scoring_ties_where_trie_does_not(tiny_oracle64, request1):
    """Labels sharing their first token get one logit under first-token
    scoring, so the argmax falls to the lowest index whatever the model
    prefers; summing along the trie tells them apart."""
    orc = tiny_oracle64
    cache = orc.prefill(request1.prefix)
    f = request1.fields[3]
    assert len({int(l[0]) for l in f.labels}) == 1
    z = orc.readout_logits(cache, f.scaffold)
    ft, first_mass = first_token_result(z, f.labels)
    assert np.all(ft.probs == ft.probs[0]) and ft.label == 0
    trie = orc.score_field(f, cache=cache)
    assert len(np.unique(np.round(trie.scores, 9))) == len(f.labels)
    assert abs(first_mass - trie.first_mass) < 1e-12
    # enum A has distinct first tokens: first-token probs are not all equal
    ft2, _ = first_token_result(orc.readout_logits(cache, request1.fields[2].scaffold),
                                request1.fields[2].labels)
    assert len(np.unique(ft2.probs)) == len(request1.fields[2].labels)


def test_field_order_and_subset_invariance(tiny_oracle, request1):
    cache = tiny_oracle.prefill(request1.prefix)
    full = tiny_oracle.score(cache, request1.fields)
    perm = [2, 0, 3]
    part = tiny_oracle.score(cache, [request1.fields[i] for i in perm])
    for j, i in enumerate(perm):
        np.testing.assert_array_equal(part[j].scores, full[i].scores)


# --------------------------------------------------------------------------
# Alternative scorers: per-level product and length-normalised mean
# --------------------------------------------------------------------------
def test_per_level_hand_example():
    """Labels (5,1), (5,3), (7).  Root: P(5) = 0.3, P(7) = 0.1, so the first
    level gives 0.75 / 0.25; after token 5: P(1) = 0.2, P(3) = 0.6, so the
    second level gives 0.25 / 0.75.  Products: 0.1875, 0.5625, 0.25.
    Counting token 5 once per label at the root (0.3 + 0.3 + 0.1) or leaving
    the second level unrenormalised gives other numbers."""
    labels = [[5, 1], [5, 3], [7]]
    lps = [np.log([0.3, 0.2]), np.log([0.3, 0.6]), np.log([0.1])]
    np.testing.assert_allclose(np.exp(per_level_scores(labels, lps)), [0.1875, 0.5625, 0.25], atol=1e-15)
    # the summed-log-prob score of the same labels: 0.06, 0.18, 0.1
    np.testing.assert_allclose(np.exp(field_scores("sum", labels, lps)), [0.06, 0.18, 0.1], atol=1e-15)


def test_per_level_single_token_is_subset_softmax():
    """With one-token labels there is a single level, and its renormalised
    distribution is torch's softmax over the candidate logits."""
    rng = np.random.default_rng(7)
    z = rng.normal(0, 3, 64)
    cands = [3, 17, 40, 41, 63]
    lp = z - logsumexp64(z[None, :])[0]
    got = np.exp(per_level_scores([[c] for c in cands], [lp[[c]] for c in cands]))
    want = torch.softmax(torch.tensor(z[cands], dtype=torch.float64), 0).numpy()
    np.testing.assert_allclose(got, want, atol=1e-14)


def _random_trie_model(seed, vocab=6, depth=3, n_labels=9):
    """A toy model: every prefix u has its own next-token distribution over
    a 6-token vocabulary; the labels are distinct random paths of length
    1..depth with no label a prefix of another."""
    rng = np.random.default_rng(seed)
    dist = {}

    def p(u):
        if u not in dist:
            w = rng.gamma(0.7, 1.0, vocab)
            dist[u] = w / w.sum()
        return dist[u]

    labels = []
    while len(labels) < n_labels:
        lab = tuple(int(t) for t in rng.integers(0, vocab, rng.integers(1, depth + 1)))
        if any(lab == o[:len(lab)] or o == lab[:len(o)] for o in labels):
            continue
        labels.append(lab)
    lps = [np.array([np.log(p(lab[:j])[lab[j]]) for j in range(len(lab))]) for lab in labels]
    return labels, lps, p


@pytest.mark.parametrize("seed", range(6))
def test_per_level_by_brute_force(seed):
    """Product over the label's levels of P_u(t) / sum of P_u over the
    tokens that some label continues with after u, taken straight from the
    toy model's node distributions.  The result is a distribution over the
    labels, and a multi-level label never beats its first-level share."""
    labels, lps, p = _random_trie_model(seed)
    got = np.exp(per_level_scores(labels, lps))
    for c, lab in enumerate(labels):
        prob = 1.0
        for j in range(len(lab)):
            u = lab[:j]
            allowed = {o[j] for o in labels if len(o) > j and o[:j] == u}
            prob *= p(u)[lab[j]] / sum(p(u)[t] for t in allowed)
        assert abs(got[c] - prob) < 1e-13
        firsts = {o[0] for o in labels}
        assert got[c] <= p(())[lab[0]] / sum(p(())[t] for t in firsts) + 1e-15
    assert abs(got.sum() - 1.0) < 1e-13


def test_length_normalised_mean():
    """HIGH is one token at log-prob -0.5, MEDIUM two tokens at -0.3 each:
    summing favours HIGH (-0.5 > -0.6), the per-token mean favours MEDIUM
    (-0.3 > -0.5), the length bias the mean is there to remove."""
    lps = [np.array([-0.5]), np.array([-0.3, -0.3])]
    np.testing.assert_allclose(length_normalised_scores(lps), [-0.5, -0.3], atol=1e-15)
    assert scores_to_result(field_scores("sum", [[1], [2, 3]], lps)).label == 0
    assert scores_to_result(field_scores("mean", [[1], [2, 3]], lps)).label == 1
    # one-token labels: the mean is the sum
    one = [np.array([-1.25]), np.array([-0.75])]
    np.testing.assert_array_equal(field_scores("mean", [[1], [2]], one), field_scores("sum", [[1], [2]], one))


def test_scoring_rules_keep_the_mass(tiny_oracle64, request1):
    """The scoring rule changes label, probabilities and margin, never the
    full-vocabulary candidate mass or the first-token mass; the per-level
    rule at T = 1 is already normalised, so its probabilities are exp(s)."""
    orc = tiny_oracle64
    cache = orc.prefill(request1.prefix)
    for f in request1.fields:
        base = orc.score_field(f, cache=cache)
        for rule in ("mean", "level"):
            g = synth.Field(f.scaffold, f.labels, f.temperature, f.kind, rule)
            r = orc.score_field(g, cache=cache)
            assert r.mass == base.mass and r.log_mass == base.log_mass and r.first_mass == base.first_mass
            if rule == "level":
                np.testing.assert_allclose(r.probs, np.exp(r.scores), atol=1e-12)
            else:
                lens = np.array([len(l) for l in f.labels])
                np.testing.assert_allclose(r.scores * lens, base.scores, atol=1e-12)


def test_spelled_labels_by_brute_force(tiny_oracle64):
    """Labels with several spellings: at T = 1 a label's probability is the
    sum over its spellings of the product of the spelling's token
    probabilities, each token's probability written out from the logits of
    the complete sequence, divided by that sum over every spelling; the mass
    is the latter sum.  Under the per-level rule the label probabilities
    (the sums of their paths' per-level products) add up to 1."""
    from synth.requests import make_custom
    orc = tiny_oracle64
    req = make_custom(3, 512, 20, [("spelled", 2, 2), ("spelled", 3, 3)])
    cache = orc.prefill(req.prefix)
    P = req.prefix
    for f in req.fields:
        res = orc.score_field(f, cache=cache)
        path_p = []
        for lab in f.labels:
            seq = np.concatenate([P, f.scaffold, lab])
            h, _ = orc.forward(seq, np.arange(len(seq)))
            z = orc.logits(h)
            prob = 1.0
            for j, t in enumerate(lab):
                row = z[len(P) + len(f.scaffold) - 1 + j]
                prob *= np.exp(row[t]) / np.exp(row).sum()
            path_p.append(prob)
        path_p = np.array(path_p)
        n_lab = int(f.label_of.max()) + 1
        lab_p = np.array([path_p[f.label_of == i].sum() for i in range(n_lab)])
        np.testing.assert_allclose(res.probs, lab_p / path_p.sum(), atol=1e-10)
        np.testing.assert_allclose(np.exp(res.scores), lab_p, rtol=1e-9)
        assert abs(res.mass - path_p.sum()) < 1e-10 * max(1.0, path_p.sum()) + 1e-15
        assert res.label == int(np.argmax(lab_p))
        lvl = orc.score_field(synth.Field(f.scaffold, f.labels, 1.0, f.kind, "level", f.label_of), cache=cache)
        assert abs(np.exp(lvl.scores).sum() - 1.0) < 1e-12
        assert lvl.mass == res.mass


def test_first_field_first_by_brute_force(tiny_oracle64, request1):
    """First field first: field 0 is scored right after the prefix; every
    other label's probability is the product of its tokens' probabilities
    written out from the logits of the complete sequence prefix || field 0's
    scaffold || field 0's winning label || separator || scaffold || label."""
    orc = tiny_oracle64
    P = request1.prefix
    sep = np.array([7, 11])
    cache = orc.prefill(P)
    res = orc.score_first_field_first(cache, request1.fields, sep)
    plain = orc.score_field(request1.fields[0], cache=cache)
    np.testing.assert_array_equal(res[0].scores, plain.scores)
    f0 = request1.fields[0]
    line = np.concatenate([f0.scaffold, f0.labels[plain.label], sep])
    for f, r in zip(request1.fields[1:], res[1:]):
        for c, lab in enumerate(f.labels):
            seq = np.concatenate([P, line, f.scaffold, lab])
            h, _ = orc.forward(seq, np.arange(len(seq)))
            z = orc.logits(h)
            prob = 1.0
            for j, t in enumerate(lab):
                row = z[len(P) + len(line) + len(f.scaffold) - 1 + j]
                prob *= np.exp(row[t]) / np.exp(row).sum()
            assert abs(np.log(prob) - r.scores[c]) < 1e-10
    # the written spelling of a label with several is its first listed path
    from synth.requests import make_custom
    sp = make_custom(9, 512, 12, [("spelled", 3, 3)]).fields[0]
    fake = scores_to_result([0.0, -1.0, -2.0])   # label 0 wins
    for want in range(3):
        fake.label = want
        first_path = sp.labels[int(np.flatnonzero(sp.label_of == want)[0])]
        np.testing.assert_array_equal(orc.answer_line(sp, fake, sep),
                                      np.concatenate([sp.scaffold, first_path, sep]))


def test_workload_shapes():
    """The generators give the branch sizes the workloads are described with."""
    r2 = synth.make_request(2)
    assert len(r2.prefix) == 512 and len(r2.fields) == 28
    assert sum(f.kind == "bool" for f in r2.fields) == 10
    for f in r2.fields:
        assert len(f.scaffold) == 8
        toks = np.concatenate(f.labels)
        assert len(np.unique(toks)) == len(toks)            # no sharing within a field
    r3 = synth.make_request(3)
    f = r3.fields[0]
    assert len(f.labels) == 255 and {len(l) for l in f.labels} == {3}
    assert len({int(l[0]) for l in f.labels}) == 1
    assert len({(int(l[1]), int(l[2])) for l in f.labels}) == 255
    r4 = synth.make_request(4)
    assert len(r4.prefix) == 8192 and len(r4.fields) == 29 and len(r4.fields[-1].labels) == 218
    reqs = synth.make_requests(5, n_requests=8)
    assert all(512 <= len(r.prefix) <= 4096 for r in reqs)
    assert all(np.array_equal(r.prefix[:512], reqs[0].prefix[:512]) for r in reqs)
