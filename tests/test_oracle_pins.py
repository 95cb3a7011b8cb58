"""Pins of the fp64 oracle against things other than itself (no GPU needed).

* the hand-worked commit example (tests/golden), re-evaluated from its closed forms;
* scipy's softmax and numpy's argmax on random bf16 logits;
* a dense block-causal attention over a whole multi-block sequence (a different
  formulation: one masked matrix product per head, no pages);
* special cases: equal keys give the mean of V, one dominant key gives its V row, MHA,
  permuted pages, softmax rows summing to one;
* the LM head against a BLAS matrix product.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import brute
from workloads import (f32_to_bf16_bits, bf16_bits_to_f32, make_attention, make_logits,
                       make_mask_fixed_fraction)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "commit_worked_example.txt")


def _closed(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"E": math.exp, "LN": math.log}))


def _parse_golden():
    rows, cases = {}, []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = [p.strip() for p in line.split("|")]
        if parts[0].startswith("row"):
            r = int(parts[0].split()[1])
            rows[r] = dict(logits=[float(x) for x in parts[1].split(",")], tok=int(parts[2]),
                           conf1=float(parts[3]), conf05=float(parts[4]),
                           closed1=parts[5], closed05=parts[6])
        elif parts[0].startswith("case"):
            cases.append(dict(name=parts[0].split()[1], mask=[int(c) for c in parts[1]],
                              replace=parts[2], tau=float(parts[3]), T=float(parts[4]),
                              commit=[int(c) for c in parts[5]]))
        elif parts[0].startswith("rcase"):
            cases.append(dict(name=parts[0].split()[1], mask=[int(c) for c in parts[1]],
                              replace=parts[2], rule=parts[3], k=int(parts[4]), tau=0.5, T=1.0,
                              commit=[int(c) for c in parts[5]]))
        elif parts[0].startswith("erow"):
            r = int(parts[0].split()[1])
            rows[r].update(h1=float(parts[1]), h05=float(parts[2]), hclosed1=parts[3],
                           hclosed05=parts[4])
        elif parts[0].startswith("ecase"):
            cases.append(dict(name=parts[0].split()[1], mask=[int(c) for c in parts[1]],
                              replace=parts[2], rule="entropy_bounded", budget=float(parts[3]),
                              T=float(parts[4]), commit=[int(c) for c in parts[5]]))
    return rows, cases


def test_golden_closed_forms_match_printed_decimals():
    rows, _ = _parse_golden()
    assert len(rows) == 4
    for r in rows.values():
        assert abs(_closed(r["closed1"]) - r["conf1"]) < 5e-7
        assert abs(_closed(r["closed05"]) - r["conf05"]) < 5e-7


@pytest.mark.parametrize("case", ["A", "B", "C", "D", "E"])
def test_commit_worked_example(case):
    rows, cases = _parse_golden()
    c = [x for x in cases if x["name"] == case][0]
    logits = np.array([rows[r]["logits"] for r in range(4)], dtype=np.float32)
    closed = {r: (rows[r]["closed1"] if c["T"] == 1 else rows[r]["closed05"]) for r in range(4)}
    toks = {r: rows[r]["tok"] for r in range(4)}
    if c["replace"] != "-":
        rr, vals = c["replace"].split("=")
        logits[int(rr)] = [float(x) for x in vals.split(",")]
        closed[int(rr)] = "1/4"
        toks[int(rr)] = 0
    bits = f32_to_bf16_bits(logits)
    assert np.array_equal(bf16_bits_to_f32(bits), logits)  # exact in bf16
    mask = np.array([c["mask"]], dtype=np.uint8)
    res = oracle.confidence_commit(bits, mask, c["tau"], c["T"])
    for i in range(4):
        if mask[0, i]:
            assert res.tok[0, i] == toks[i]
            assert abs(res.conf[0, i] - _closed(closed[i])) <= 1e-12
        else:
            assert res.tok[0, i] == -1 and res.conf[0, i] == -np.inf
    assert list(res.commit[0]) == c["commit"]
    if case == "D":
        assert res.near[0, 0] & 1  # conf exactly at the threshold is flagged
    if case == "E":
        assert res.near[0, 0] & 2 and res.near[0, 2] & 2  # confidence tie flagged


RULES = {"topk": oracle.RULE_TOPK, "sequential": oracle.RULE_SEQUENTIAL,
         "anti_sequential": oracle.RULE_ANTI_SEQUENTIAL}


@pytest.mark.parametrize("case", ["F", "G", "H", "I", "J", "K", "L", "M"])
def test_commit_rules_worked_example(case):
    rows, cases = _parse_golden()
    c = [x for x in cases if x["name"] == case][0]
    logits = np.array([rows[r]["logits"] for r in range(4)], dtype=np.float32)
    if c["replace"] != "-":
        rr, vals = c["replace"].split("=")
        logits[int(rr)] = [float(x) for x in vals.split(",")]
    bits = f32_to_bf16_bits(logits)
    mask = np.array([c["mask"]], dtype=np.uint8)
    res = oracle.confidence_commit(bits, mask, c["tau"], c["T"], rule=RULES[c["rule"]], k=c["k"])
    assert list(res.commit[0]) == c["commit"]
    if case == "I":
        assert res.near[0, 1] & 2 and res.near[0, 2] & 2  # the tie at the cut is flagged


def test_golden_entropy_closed_forms():
    """The printed entropies match their closed forms, and the oracle's entropies match both
    (all four rows masked, T = 1 and T = 0.5)."""
    rows, _ = _parse_golden()
    logits = np.array([rows[r]["logits"] for r in range(4)], dtype=np.float32)
    bits = f32_to_bf16_bits(logits)
    mask = np.ones((1, 4), np.uint8)
    for T, key, ckey in ((1.0, "h1", "hclosed1"), (0.5, "h05", "hclosed05")):
        res = oracle.confidence_commit(bits, mask, 0.5, T)
        for r in range(4):
            closed = _closed(rows[r][ckey])
            assert abs(closed - rows[r][key]) < 5e-7
            assert abs(res.ent[0, r] - closed) <= 1e-12


@pytest.mark.parametrize("case", ["N", "O", "P", "Q", "R", "S", "T", "U", "W"])
def test_entropy_bounded_worked_example(case):
    rows, cases = _parse_golden()
    c = [x for x in cases if x["name"] == case][0]
    logits = np.array([rows[r]["logits"] for r in range(4)], dtype=np.float32)
    if c["replace"] != "-":
        rr, vals = c["replace"].split("=")
        logits[int(rr)] = [float(x) for x in vals.split(",")]
    bits = f32_to_bf16_bits(logits)
    mask = np.array([c["mask"]], dtype=np.uint8)
    res = oracle.confidence_commit(bits, mask, c["budget"], c["T"],
                                   rule=oracle.RULE_ENTROPY_BOUNDED)
    assert list(res.commit[0]) == c["commit"]
    assert np.all(np.isinf(res.ent[0][mask[0] == 0]))
    if case == "T":
        assert res.near[0, 0] & 2 and res.near[0, 2] & 2   # the entropy tie is flagged


@pytest.mark.parametrize("T", [1.0, 0.5, 1.7])
def test_entropy_against_scipy(T):
    """The oracle's entropy of random bf16 rows equals scipy's entropy of scipy's softmax."""
    from scipy.special import softmax
    from scipy.stats import entropy
    rng = np.random.default_rng(47)
    B, L, V = 3, 4, 3001
    bits = make_logits(rng, B * L, V, peak_height=(0.0, 16.0))
    mask = np.ones((B, L), np.uint8)
    res = oracle.confidence_commit(bits, mask, 0.5, T)
    x = bf16_bits_to_f32(bits).astype(np.float64).reshape(B, L, V)
    want = entropy(softmax(x / T, axis=-1), axis=-1)
    assert np.allclose(res.ent, want, rtol=1e-10, atol=1e-12)
    assert np.array_equal(res.ent32, res.ent.astype(np.float32))


def test_entropy_special_cases():
    """Uniform rows give ln V; one dominant logit gives (almost) 0; two equal dominant logits
    give ln 2; the entropy never exceeds ln V."""
    V = 1000
    x = np.zeros((3, V), np.float32)
    x[1, 7] = 120.0
    x[2, 3] = x[2, 900] = 120.0
    bits = f32_to_bf16_bits(x)
    res = oracle.confidence_commit(bits, np.ones((1, 3), np.uint8), 0.5, 1.0)
    assert abs(res.ent[0, 0] - math.log(V)) <= 1e-12
    assert res.ent[0, 1] < 1e-40
    assert abs(res.ent[0, 2] - math.log(2)) <= 1e-12


def test_entropy_bounded_against_numpy():
    """The entropy rule against a stable argsort of float32 entropies and a float32 running sum
    taken in that order; at least one commit in every block with a masked position."""
    rng = np.random.default_rng(53)
    B, L, V = 24, 16, 400
    bits = make_logits(rng, B * L, V, peak_height=(0.0, 14.0))
    mask = make_mask_fixed_fraction(rng, B, L, 0.7)
    mask[5] = 0
    for budget in (0.0, 0.5, 3.0, 20.0):
        res = oracle.confidence_commit(bits, mask, budget, 1.0, rule=oracle.RULE_ENTROPY_BOUNDED)
        for b in range(B):
            pos = np.nonzero(mask[b])[0]
            if len(pos) == 0:
                assert res.commit[b].sum() == 0
                continue
            order = pos[np.argsort(res.ent32[b, pos], kind="stable")]
            want, run = [order[0]], np.float32(res.ent32[b, order[0]])
            for i in order[1:]:
                nxt = np.float32(run + res.ent32[b, i])
                if not nxt <= np.float32(budget):
                    break
                want.append(i)
                run = nxt
            assert set(np.nonzero(res.commit[b])[0].tolist()) == set(int(i) for i in want)


@pytest.mark.parametrize("k", [1, 2, 3, 9])
def test_commit_rules_against_numpy(k):
    """Top-k against a stable argsort of float32 confidences; sequential rules against the
    masked positions in order; every rule commits min(k, masked) masked positions."""
    rng = np.random.default_rng(31 + k)
    B, L, V = 12, 8, 500
    bits = make_logits(rng, B * L, V, peak_height=(0.0, 12.0))
    mask = make_mask_fixed_fraction(rng, B, L, 0.6)
    mask[3] = 0
    for rule in (oracle.RULE_TOPK, oracle.RULE_SEQUENTIAL, oracle.RULE_ANTI_SEQUENTIAL):
        res = oracle.confidence_commit(bits, mask, 0.5, 1.0, rule=rule, k=k)
        for b in range(B):
            pos = np.nonzero(mask[b])[0]
            n = min(k, len(pos))
            if rule == oracle.RULE_TOPK:
                order = pos[np.argsort(-res.conf32[b, pos], kind="stable")]
                want = set(order[:n].tolist())
            elif rule == oracle.RULE_SEQUENTIAL:
                want = set(pos[:n].tolist())
            else:
                want = set(pos[len(pos) - n:].tolist())
            got = set(np.nonzero(res.commit[b])[0].tolist())
            assert got == want, (rule, b)
        assert np.all(res.commit <= mask)


def test_commit_rule_arguments_checked():
    bits = f32_to_bf16_bits(np.zeros((4, 8), np.float32))
    mask = np.ones((1, 4), np.uint8)
    with pytest.raises(ValueError):
        oracle.confidence_commit(bits, mask, 0.5, 1.0, rule=oracle.RULE_TOPK, k=0)
    with pytest.raises(ValueError):
        oracle.confidence_commit(bits, mask, 0.5, 1.0, rule=7)


@pytest.mark.parametrize("T", [1.0, 0.5, 1.7])
def test_commit_against_scipy_softmax(T):
    rng = np.random.default_rng(7)
    B, L, V = 6, 8, 997
    bits = make_logits(rng, B * L, V, peak_height=(0.0, 12.0))
    mask = make_mask_fixed_fraction(rng, B, L, 0.6)
    res = oracle.confidence_commit(bits, mask, 0.3, T)
    x = bf16_bits_to_f32(bits).astype(np.float64)
    tok_ref, conf_ref = brute.confidence_scipy(x, T)
    m = mask.reshape(-1) == 1
    assert np.array_equal(res.tok.reshape(-1)[m], tok_ref[m])
    np.testing.assert_allclose(res.conf.reshape(-1)[m], conf_ref[m], rtol=1e-12)
    assert np.all(res.tok.reshape(-1)[~m] == -1)


def test_commit_invariants_and_special_values():
    rng = np.random.default_rng(11)
    B, L, V = 40, 8, 513
    bits = make_logits(rng, B * L, V, peak_height=(0.0, 30.0))
    frac = rng.uniform(0.0, 1.0, size=B)
    frac[:3] = 0.0  # SAVING blocks
    mask = make_mask_fixed_fraction(rng, B, L, frac)
    res = oracle.confidence_commit(bits, mask, 0.6, 1.0)
    for b in range(B):
        masked = mask[b] == 1
        assert np.all(res.commit[b][~masked] == 0)          # commit within the mask
        if masked.any():
            assert res.commit[b].sum() >= 1                  # at least one per block
            assert np.all((res.conf[b][masked] >= 1.0 / V - 1e-15) & (res.conf[b][masked] <= 1.0))
        else:
            assert res.commit[b].sum() == 0                  # SAVING block: nothing
    # all-equal logits: conf is exactly 1/V, token 0
    flat = np.full((1, 1 * 4, 300), f32_to_bf16_bits(np.float32(1.5)), dtype=np.uint16)
    r = oracle.confidence_commit(flat.reshape(4, 300), np.ones((1, 4), np.uint8), 0.9, 1.0)
    assert np.all(r.tok == 0) and np.allclose(r.conf, 1.0 / 300, rtol=0, atol=1e-15)
    # one dominant logit: confidence tends to one
    big = np.zeros((1, 50), dtype=np.float32)
    big[0, 17] = 120.0
    r = oracle.confidence_commit(f32_to_bf16_bits(big), np.ones((1, 1), np.uint8), 0.9, 1.0)
    assert r.tok[0, 0] == 17 and r.conf[0, 0] == 1.0 and r.commit[0, 0] == 1
    # ties in the logits go to the lowest vocabulary index
    tie = np.zeros((1, 64), dtype=np.float32)
    tie[0, [5, 9, 40]] = 3.0
    r = oracle.confidence_commit(f32_to_bf16_bits(tie), np.ones((1, 1), np.uint8), 0.9, 1.0)
    assert r.tok[0, 0] == 5


def test_apply_commit():
    mask = np.array([[1, 1, 0, 1]], np.uint8)
    com = np.array([[0, 1, 0, 1]], np.uint8)
    assert list(oracle.apply_commit(mask, com)[0]) == [1, 0, 0, 0]


def _scatter_sequence(rng, n_tok, Hkv, D, P, pool_pages, k_seq, v_seq):
    """Place one sequence's tokens into a shuffled pool; unused slots hold NaN."""
    n_pages = (n_tok + P - 1) // P
    ids = rng.permutation(pool_pages)[:n_pages].astype(np.int32)
    kp = np.full((pool_pages, P, Hkv, D), 0x7FC0, np.uint16)
    vp = np.full((pool_pages, P, Hkv, D), 0x7FC0, np.uint16)
    for t in range(n_tok):
        kp[ids[t // P], t % P] = k_seq[t]
        vp[ids[t // P], t % P] = v_seq[t]
    return kp, vp, ids


@pytest.mark.parametrize("Hq,Hkv,L,P", [(4, 2, 3, 4), (6, 6, 4, 16), (8, 2, 5, 3)])
def test_attention_matches_dense_block_causal(Hq, Hkv, L, P):
    rng = np.random.default_rng(Hq * 100 + L)
    D, n_blocks = 16, 5
    n = L * n_blocks
    q_seq = f32_to_bf16_bits(rng.standard_normal((n, Hq, D), dtype=np.float32))
    k_seq = f32_to_bf16_bits(rng.standard_normal((n, Hkv, D), dtype=np.float32))
    v_seq = f32_to_bf16_bits(rng.standard_normal((n, Hkv, D), dtype=np.float32))
    dense = brute.dense_block_causal_attention(bf16_bits_to_f32(q_seq), bf16_bits_to_f32(k_seq),
                                               bf16_bits_to_f32(v_seq), L, Hq, Hkv)
    kp, vp, ids = _scatter_sequence(rng, n, Hkv, D, P, 3 * ((n + P - 1) // P), k_seq, v_seq)
    for blk in range(n_blocks):
        prefix = blk * L
        kv = prefix + L
        table = np.full((1, (n + P - 1) // P), -1, np.int32)
        table[0, :(kv + P - 1) // P] = ids[:(kv + P - 1) // P]
        # the cache holds only tokens < kv; later slots of the last page are poisoned
        kpb, vpb = kp.copy(), vp.copy()
        for t in range(kv, ((kv + P - 1) // P) * P):
            kpb[ids[t // P], t % P] = 0x7FC0
            vpb[ids[t // P], t % P] = 0x7FC0
        q = q_seq[prefix:prefix + L][None]
        out = oracle.block_attention(q, kpb, vpb, table, np.array([prefix], np.int32), L, Hq, Hkv,
                                     D, P)
        np.testing.assert_allclose(out[0], dense[prefix:prefix + L], rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    rng = np.random.default_rng(3)
    Hq, Hkv, D, P, L = 8, 4, 32, 16, 4
    # equal keys: output is the mean of V over the kv tokens
    inp = make_attention(rng, 2, L, Hq, Hkv, D, prefix_range=(20, 37), P=P, poison=True)
    k_eq = inp.k_ref.copy()
    k_eq[:] = f32_to_bf16_bits(np.float32(0.25))
    kvl = inp.kv_lens
    out = oracle.block_attention(inp.q, k_eq, inp.v_ref, inp.page_table_ref, inp.prefix_lens, L,
                                 Hq, Hkv, D, P)
    for b in range(2):
        vs = np.stack([bf16_bits_to_f32(inp.v_ref[inp.page_table_ref[b, t // P], t % P])
                       for t in range(kvl[b])]).astype(np.float64)
        mean = vs.mean(axis=0)  # [Hkv, D]
        for h in range(Hq):
            np.testing.assert_allclose(out[b, :, h, :], np.broadcast_to(mean[h // 2], (L, D)),
                                       rtol=1e-12, atol=1e-14)
    # one dominant key: output equals that token's V row
    inp = make_attention(rng, 1, L, Hq, Hkv, D, prefix_range=(40, 40), P=P)
    q = np.zeros((1, L, Hq, D), np.float32)
    q[..., 0] = 64.0
    k = np.zeros(inp.k_ref.shape, np.float32)
    j = 23
    k[inp.page_table_ref[0, j // P], j % P, :, 0] = 64.0
    out = oracle.block_attention(f32_to_bf16_bits(q), f32_to_bf16_bits(k), inp.v_ref,
                                 inp.page_table_ref, inp.prefix_lens, L, Hq, Hkv, D, P)
    vj = bf16_bits_to_f32(inp.v_ref[inp.page_table_ref[0, j // P], j % P]).astype(np.float64)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, :, h, :], np.broadcast_to(vj[h // 2], (L, D)), atol=1e-12)
    # permuting the pool (pages and table together) changes nothing
    inp = make_attention(rng, 3, L, Hq, Hkv, D, prefix_range=(5, 50), P=P)
    base = oracle.block_attention(inp.q, inp.k_ref, inp.v_ref, inp.page_table_ref, inp.prefix_lens,
                                  L, Hq, Hkv, D, P)
    perm = rng.permutation(inp.k_ref.shape[0])
    inv = np.argsort(perm)
    table = np.where(inp.page_table_ref >= 0, inv[np.maximum(inp.page_table_ref, 0)], -1)
    out = oracle.block_attention(inp.q, inp.k_ref[perm], inp.v_ref[perm], table.astype(np.int32),
                                 inp.prefix_lens, L, Hq, Hkv, D, P)
    assert np.array_equal(out, base)
    # softmax rows sum to one
    for (b, i, h) in [(0, 0, 0), (1, 3, 7), (2, 2, 5)]:
        p = oracle.attention_probs(inp.q, inp.k_ref, inp.page_table_ref, inp.prefix_lens, L, Hq,
                                   Hkv, D, P, b, i, h)
        assert abs(p.sum() - 1.0) < 1e-12 and np.all(p >= 0)


def test_attention_gqa_grouping_is_contiguous():
    """Query head h reads KV head h // (Hq/Hkv): with distinct constant V per KV head and
    equal keys, the output of head h is exactly that constant."""
    rng = np.random.default_rng(5)
    Hq, Hkv, D, P, L = 8, 2, 16, 16, 4
    inp = make_attention(rng, 1, L, Hq, Hkv, D, prefix_range=(9, 9), P=P, poison=False)
    v = np.zeros(inp.v_ref.shape, np.float32)
    v[:, :, 0, :] = 1.0
    v[:, :, 1, :] = -2.0
    out = oracle.block_attention(inp.q, inp.k_ref, f32_to_bf16_bits(v), inp.page_table_ref,
                                 inp.prefix_lens, L, Hq, Hkv, D, P)
    assert np.allclose(out[0, :, :4, :], 1.0) and np.allclose(out[0, :, 4:, :], -2.0)


def test_lm_head_against_blas():
    rng = np.random.default_rng(9)
    n_rows, H, V = 12, 96, 211
    hidden = f32_to_bf16_bits(rng.standard_normal((n_rows, H), dtype=np.float32))
    w = f32_to_bf16_bits(rng.standard_normal((V, H), dtype=np.float32) * np.float32(0.02))
    rows = np.array([0, 3, 4, 11], np.int32)
    out = oracle.lm_head(hidden, w, rows)
    ref = brute.lm_head_matmul(hidden, w, rows)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    cols = np.array([0, 7, 210, 100], np.int32)
    sub = oracle.lm_head(hidden, w, rows, cols)
    np.testing.assert_allclose(sub, ref[:, cols], rtol=1e-12, atol=1e-13)


def test_round_logits_to_bf16():
    rng = np.random.default_rng(13)
    x = rng.standard_normal(100000).astype(np.float32)
    # values exact in float32 round exactly as the generator's float32 rounding does
    assert np.array_equal(oracle.round_logits_to_bf16(x.astype(np.float64)), f32_to_bf16_bits(x))
    # an fp64 value just above a bf16 midpoint rounds up even when float32 would tie
    one = 1.0
    mid = one + 2.0 ** -8          # halfway between 1 and the next bf16 (1 + 2^-7)
    assert oracle.round_logits_to_bf16(np.array([mid]))[0] == 0x3F80          # tie -> even
    assert oracle.round_logits_to_bf16(np.array([mid + 2.0 ** -40]))[0] == 0x3F81
    assert oracle.round_logits_to_bf16(np.array([-(mid + 2.0 ** -40)]))[0] == 0xBF81


def test_attention_oracle_rejects_pages_outside_the_pool():
    """A page id of a needed token outside the pool is an argument error, not a read."""
    rng = np.random.default_rng(11)
    a = make_attention(rng, 2, 4, 8, 8, 128, prefix_range=(20, 40), poison=False)
    bad = a.page_table_ref.copy()
    bad[1, 0] = a.k_ref.shape[0]
    with pytest.raises(ValueError):
        oracle.block_attention(a.q, a.k_ref, a.v_ref, bad, a.prefix_lens, a.L, a.Hq, a.Hkv,
                               a.D, a.P)
    bad[1, 0] = -1
    with pytest.raises(ValueError):
        oracle.attention_probs(a.q, a.k_ref, bad, a.prefix_lens, a.L, a.Hq, a.Hkv, a.D, a.P,
                               1, 0, 0)


def test_active_rows_by_hand():
    mask = np.array([[1, 0, 1, 0], [0, 0, 0, 0], [1, 1, 0, 1]], np.uint8)
    assert oracle.active_rows(mask).tolist() == [0, 2, 8, 9, 11]
    assert oracle.active_rows(mask, np.array([1, 1, 0], np.uint8)).tolist() == [0, 2]


def test_written_block_kv_is_what_attention_reads():
    """After the write, the block's keys are the new ones: with every new key equal to the
    query (scaled large) and new values constant, the block's output is that constant."""
    rng = np.random.default_rng(13)
    a = make_attention(rng, 2, 4, 8, 8, 128, prefix_range=(30, 50), poison=False)
    k_new = np.zeros((2, 4, 8, 128), np.uint16)
    v_new = np.zeros((2, 4, 8, 128), np.uint16)
    big = f32_to_bf16_bits(np.full((2, 4, 8, 128), 4.0, np.float32))
    k_new[:] = big
    v_new[:] = f32_to_bf16_bits(np.full((2, 4, 8, 128), 0.75, np.float32))
    q = f32_to_bf16_bits(np.full(a.q.shape, 4.0, np.float32))
    k, v = oracle.write_block_kv(a.k_ref, a.v_ref, a.page_table_ref, a.prefix_lens, k_new, v_new)
    out = oracle.block_attention(q, k, v, a.page_table_ref, a.prefix_lens, a.L, a.Hq, a.Hkv, a.D,
                                 a.P)
    # block keys score 4*4*128/sqrt(128) ~ 181 above the prefix keys (N(0, 0.5^2) entries)
    assert np.allclose(out, 0.75, atol=1e-6)
    untouched = np.ones(a.k_ref.shape[0], bool)
    for b in range(2):
        for i in range(4):
            j = int(a.prefix_lens[b]) + i
            untouched[a.page_table_ref[b][j // 16]] = False
    assert np.array_equal(k[untouched], a.k_ref[untouched])


def test_block_kv_write_by_hand_across_a_page_boundary():
    """Prefix 14, L = 4, pages of 16, page-table row [5, 2, 7]: block tokens 0 and 1 land in
    page 5, slots 14 and 15; tokens 2 and 3 in page 2, slots 0 and 1 (coordinates worked out by
    hand).  Every other slot of the pool keeps its value."""
    Hkv, D = 2, 3
    k0 = np.arange(8 * 16 * Hkv * D, dtype=np.uint16).reshape(8, 16, Hkv, D)
    v0 = k0 + 7000
    kn = (50000 + np.arange(4 * Hkv * D, dtype=np.uint16)).reshape(1, 4, Hkv, D)
    vn = kn + 5000
    pt = np.array([[5, 2, 7]], np.int32)
    k, v = oracle.write_block_kv(k0, v0, pt, np.array([14], np.int32), kn, vn, P=16)
    want_k, want_v = k0.copy(), v0.copy()
    for tok, (page, slot) in enumerate([(5, 14), (5, 15), (2, 0), (2, 1)]):
        want_k[page, slot] = kn[0, tok]
        want_v[page, slot] = vn[0, tok]
    assert np.array_equal(k, want_k) and np.array_equal(v, want_v)


def test_block_kv_write_against_gathered_sequences():
    """The written cache read back a second way: each sequence's pages gathered whole and laid
    end to end give its tokens in order; the block's L tokens follow the untouched prefix, and
    pages no sequence uses keep their contents."""
    rng = np.random.default_rng(29)
    B, L, Hkv, D = 5, 7, 2, 128
    a = make_attention(rng, B, L, 4, Hkv, D, prefix_range=(0, 60), poison=False)
    kn = f32_to_bf16_bits(rng.normal(0, 0.5, (B, L, Hkv, D)).astype(np.float32))
    vn = f32_to_bf16_bits(rng.normal(0, 0.5, (B, L, Hkv, D)).astype(np.float32))
    k, v = oracle.write_block_kv(a.k_ref, a.v_ref, a.page_table_ref, a.prefix_lens, kn, vn)
    used = np.zeros(a.k_ref.shape[0], bool)
    for b in range(B):
        pages = a.page_table_ref[b][a.page_table_ref[b] >= 0]
        used[pages] = True
        n = int(a.prefix_lens[b])
        for pool0, pool1, new in ((a.k_ref, k, kn), (a.v_ref, v, vn)):
            before = pool0[pages].reshape(-1, Hkv, D)
            after = pool1[pages].reshape(-1, Hkv, D)
            assert np.array_equal(after[:n], before[:n])
            assert np.array_equal(after[n:n + L], new[b])
            assert np.array_equal(after[n + L:], before[n + L:])
    assert np.array_equal(k[~used], a.k_ref[~used]) and np.array_equal(v[~used], a.v_ref[~used])


def test_prefill_oracle_against_dense_block_causal_attention():
    """A fresh prompt of three blocks: the block-by-block paged prefill equals dense attention
    with the block-causal mask over the whole prompt."""
    rng = np.random.default_rng(17)
    B, L, Hq, Hkv, D, n = 2, 4, 8, 4, 128, 12
    a = make_attention(rng, B, n - L, Hq, Hkv, D, prefix_lens=np.zeros(B, np.int64),
                       poison=False)   # pages for n tokens per sequence (n - L + L)
    q = f32_to_bf16_bits(rng.normal(0, 0.5, (B, n, Hq, D)).astype(np.float32))
    kn = f32_to_bf16_bits(rng.normal(0, 0.5, (B, n, Hkv, D)).astype(np.float32))
    vn = f32_to_bf16_bits(rng.normal(0, 0.5, (B, n, Hkv, D)).astype(np.float32))
    out, _, _ = oracle.prefill_attention(q, kn, vn, a.k_ref, a.v_ref, a.page_table_ref,
                                         np.zeros(B, np.int32), L, Hq, Hkv, D)
    for b in range(B):
        ref = brute.dense_block_causal_attention(bf16_bits_to_f32(q[b]), bf16_bits_to_f32(kn[b]),
                                                 bf16_bits_to_f32(vn[b]), L, Hq, Hkv)
        assert np.allclose(out[b], ref, rtol=1e-12, atol=1e-12)
