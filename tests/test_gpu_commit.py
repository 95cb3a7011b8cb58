"""Parity of the CUDA confidence/commit kernel with the fp64 oracle, through the C-ABI."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import bf16_tensor, compare_commit, compare_entropy, dev, host

pytestmark = pytest.mark.gpu


def run_gpu(lib, logits_bits, mask, threshold, temperature, rule=None, k=1, entropy=False):
    """tok, conf, commit (and the entropies when `entropy`) of one call; rule None uses the
    threshold entry point without entropies."""
    import torch
    B, L = mask.shape
    V = logits_bits.size // (B * L)
    lg = bf16_tensor(logits_bits.reshape(B * L, V))
    mk = dev(mask)
    tok = torch.empty((B, L), dtype=torch.int32, device="cuda")
    conf = torch.empty((B, L), dtype=torch.float32, device="cuda")
    com = torch.full((B, L), 7, dtype=torch.uint8, device="cuda")
    ent = torch.full((B, L), -5.0, dtype=torch.float32, device="cuda") if entropy else None
    if rule is None and not entropy:
        lib.bdlm_confidence_commit(lg, mk, B, L, V, threshold, temperature, tok, conf, com)
    else:
        lib.bdlm_confidence_commit_rule(lg, mk, B, L, V, 0 if rule is None else rule, k,
                                        threshold, temperature, tok, conf, com, entropy_out=ent)
    torch.cuda.synchronize()
    if entropy:
        return host(tok), host(conf), host(com), host(ent)
    return host(tok), host(conf), host(com)


def check(lib, ci, threshold=None, temperature=None):
    thr = ci.threshold if threshold is None else threshold
    T = ci.temperature if temperature is None else temperature
    ref = oracle.confidence_commit(ci.logits, ci.mask, thr, T)
    tok, conf, com = run_gpu(lib, ci.logits, ci.mask, thr, T)
    near = compare_commit(ref, tok, conf, com, ci.mask)
    assert lib.bdlm_device_error() == 0
    return ref, near


def test_worked_example(lib):
    x = np.array([[0, 0, 0, 0], [4, 0, 0, 0], [0, 2, 0, 0], [0, 3, 3, 0]], np.float32)
    bits = W.f32_to_bf16_bits(x)
    for mask, tau, T, want in [([1, 1, 1, 1], 0.9, 1.0, [0, 1, 0, 0]),
                               ([1, 0, 1, 1], 0.9, 1.0, [0, 0, 1, 0]),
                               ([1, 1, 1, 1], 0.9, 0.5, [0, 1, 1, 0]),
                               ([1, 1, 1, 1], 0.25, 1.0, [1, 1, 1, 1])]:
        m = np.array([mask], np.uint8)
        tok, conf, com = run_gpu(lib, W.poison_unmasked_rows(bits, m), m, tau, T)
        assert list(com[0]) == want
        assert list(tok[0][m[0] == 1]) == [t for t, k in zip([0, 0, 1, 1], mask) if k]


@pytest.mark.parametrize("config", [1, 2, 4])
@pytest.mark.parametrize("supplementary", [False, True])
def test_configs_full_size(lib, config, supplementary):
    c = W.CONFIGS[config]
    rng = np.random.default_rng(W.seed_for(config, 1 if supplementary else 0))
    ci = W.commit_inputs(config, rng, c["B"], c["L"], c["V"], supplementary=supplementary)
    ref, (near_diff, near_blocks) = check(lib, ci)
    # every block with a masked position commits at least one
    assert np.all(ref.commit.sum(1)[ci.mask.sum(1) > 0] >= 1)
    print(f"config {config} supp={supplementary}: near-threshold blocks {near_blocks}, "
          f"differing {near_diff}, multi-commit blocks {(ref.commit.sum(1) > 1).sum()}")


@pytest.mark.parametrize("B,L,V", [(3, 4, 4), (2, 1, 151939), (5, 7, 1001), (2, 64, 3000),
                                   (1, 3, 1), (9, 5, 8), (4, 16, 151936 + 5)])
@pytest.mark.parametrize("T", [1.0, 0.5, 1.7])
def test_odd_shapes(lib, B, L, V, T):
    rng = np.random.default_rng(B * 1000 + L * 10 + V)
    frac = rng.uniform(0.0, 1.0, size=B)
    frac[0] = 1.0
    if B > 2:
        frac[1] = 0.0  # a SAVING block: nothing masked
    mask = W.make_mask_fixed_fraction(rng, B, L, frac)
    logits = W.make_logits(rng, B * L, V, peak_height=(0.0, 14.0))
    ci = W.CommitInputs(B, L, V, W.poison_unmasked_rows(logits, mask), mask, 0.4, T)
    check(lib, ci)


def test_ties_go_to_lowest_index_and_position(lib):
    B, L, V = 2, 6, 5000
    x = np.zeros((B * L, V), np.float32)
    x[:, [17, 4000, 4999]] = 5.0           # equal maxima in different CTAs' ranges
    bits = W.f32_to_bf16_bits(x)
    mask = np.ones((B, L), np.uint8)
    tok, conf, com = run_gpu(lib, bits, mask, 0.9, 1.0)
    assert np.all(tok == 17)
    assert np.all(com.sum(1) == 1) and np.all(com[:, 0] == 1)  # equal confidences -> lowest i


def test_repeated_calls_stay_correct(lib):
    """Nothing carries over between calls: many calls in a row stay correct."""
    rng = np.random.default_rng(5)
    mask = W.make_mask_fixed_fraction(rng, 16, 4, 0.5)
    logits = W.poison_unmasked_rows(W.make_logits(rng, 64, 20000, peak_height=(0, 12)), mask)
    ref = oracle.confidence_commit(logits, mask, 0.3, 1.0)
    for _ in range(5):
        tok, conf, com = run_gpu(lib, logits, mask, 0.3, 1.0)
        compare_commit(ref, tok, conf, com, mask)


def test_apply_commit(lib):
    import torch
    rng = np.random.default_rng(8)
    mask = (rng.uniform(size=(64, 8)) < 0.6).astype(np.uint8)
    com = (rng.uniform(size=(64, 8)) < 0.3).astype(np.uint8) & mask
    m = dev(mask)
    lib.bdlm_apply_commit(m, dev(com), mask.size)
    torch.cuda.synchronize()
    assert np.array_equal(host(m), oracle.apply_commit(mask, com))


RULES = [("topk", oracle.RULE_TOPK), ("sequential", oracle.RULE_SEQUENTIAL),
         ("anti_sequential", oracle.RULE_ANTI_SEQUENTIAL)]


@pytest.mark.parametrize("name,rule", RULES)
@pytest.mark.parametrize("k", [1, 2, 5])
def test_commit_rules(lib, name, rule, k):
    """Top-k / sequential / anti-sequential commits against the oracle: config-4-like blocks
    (L = 64, masked fraction U[0.1, 0.9]) and blocks without any masked position."""
    rng = np.random.default_rng(100 + 10 * rule + k)
    B, L, V = 6, 64, 20000
    mask = np.zeros((B, L), np.uint8)
    for b in range(B):
        mask[b] = W.make_mask_fixed_fraction(rng, 1, L, rng.uniform(0.1, 0.9))[0]
    mask[2] = 0
    logits = W.poison_unmasked_rows(W.make_logits(rng, B * L, V, peak_height=(0, 16)), mask)
    ref = oracle.confidence_commit(logits, mask, 0.5, 1.0, rule=rule, k=k)
    tok, conf, com = run_gpu(lib, logits, mask, 0.5, 1.0, rule=lib.BDLM_COMMIT_TOPK
                             if name == "topk" else lib.BDLM_COMMIT_SEQUENTIAL
                             if name == "sequential" else lib.BDLM_COMMIT_ANTI_SEQUENTIAL, k=k)
    compare_commit(ref, tok, conf, com, mask)
    assert np.all(com.sum(1) == np.minimum(k, mask.sum(1)))
    assert lib.bdlm_device_error() == 0


def test_topk_full_size_config2(lib):
    """Config 2 with the top-2 rule (k = L / 2 per step)."""
    c = W.CONFIGS[2]
    rng = np.random.default_rng(W.seed_for(2, 3))
    ci = W.commit_inputs(2, rng, c["B"], c["L"], c["V"], supplementary=True)
    ref = oracle.confidence_commit(ci.logits, ci.mask, ci.threshold, 1.0, rule=oracle.RULE_TOPK,
                                   k=2)
    tok, conf, com = run_gpu(lib, ci.logits, ci.mask, ci.threshold, 1.0,
                             rule=lib.BDLM_COMMIT_TOPK, k=2)
    compare_commit(ref, tok, conf, com, ci.mask)


def test_threshold_rule_equals_default_entry_point(lib):
    rng = np.random.default_rng(8)
    mask = W.make_mask_fixed_fraction(rng, 8, 4, 0.75)
    logits = W.poison_unmasked_rows(W.make_logits(rng, 32, 9000, peak_height=(0, 14)), mask)
    a = run_gpu(lib, logits, mask, 0.4, 1.0)
    b = run_gpu(lib, logits, mask, 0.4, 1.0, rule=lib.BDLM_COMMIT_THRESHOLD, k=3)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_rule_arguments_rejected(lib):
    import torch
    lg = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    mk = torch.ones((1, 4), dtype=torch.uint8, device="cuda")
    tok = torch.empty((1, 4), dtype=torch.int32, device="cuda")
    conf = torch.empty((1, 4), dtype=torch.float32, device="cuda")
    com = torch.empty((1, 4), dtype=torch.uint8, device="cuda")
    for rule, k, thr in ((9, 1, 0.5), (lib.BDLM_COMMIT_TOPK, 0, 0.5), (-1, 1, 0.5),
                         (lib.BDLM_COMMIT_ENTROPY_BOUNDED, 1, -0.1)):
        with pytest.raises(lib.BdlmError):
            lib.bdlm_confidence_commit_rule(lg, mk, 1, 4, 16, rule, k, thr, 1.0, tok, conf, com)


@pytest.mark.parametrize("config", [1, 2, 4])
def test_entropy_configs_full_size(lib, config):
    """Entropies of every masked position at full size (the supplementary peaks, so rows range
    from flat to nearly one-hot) within 1e-4 + 1e-5 H of the oracle; the threshold rule's
    tokens, confidences and commits unchanged by asking for them."""
    c = W.CONFIGS[config]
    rng = np.random.default_rng(W.seed_for(config, 5))
    ci = W.commit_inputs(config, rng, c["B"], c["L"], c["V"], supplementary=True)
    ref = oracle.confidence_commit(ci.logits, ci.mask, ci.threshold, ci.temperature)
    tok, conf, com, ent = run_gpu(lib, ci.logits, ci.mask, ci.threshold, ci.temperature,
                                  entropy=True)
    compare_commit(ref, tok, conf, com, ci.mask)
    err = compare_entropy(ref, ent, ci.mask)
    plain = run_gpu(lib, ci.logits, ci.mask, ci.threshold, ci.temperature)
    for x, y in zip(plain, (tok, conf, com)):
        assert np.array_equal(x, y)
    print(f"config {config}: entropy max abs err {err:.2e}, "
          f"range {ref.ent[ci.mask == 1].min():.3f} .. {ref.ent[ci.mask == 1].max():.3f}")


@pytest.mark.parametrize("B,L,V", [(3, 4, 4), (2, 1, 151939), (5, 7, 1001), (2, 64, 3000),
                                   (1, 3, 1), (4, 16, 151936 + 5)])
@pytest.mark.parametrize("T", [1.0, 0.5])
def test_entropy_odd_shapes(lib, B, L, V, T):
    rng = np.random.default_rng(B * 7000 + L * 10 + V)
    frac = rng.uniform(0.0, 1.0, size=B)
    frac[0] = 1.0
    mask = W.make_mask_fixed_fraction(rng, B, L, frac)
    logits = W.poison_unmasked_rows(W.make_logits(rng, B * L, V, peak_height=(0.0, 14.0)), mask)
    ref = oracle.confidence_commit(logits, mask, 0.4, T)
    tok, conf, com, ent = run_gpu(lib, logits, mask, 0.4, T, entropy=True)
    compare_commit(ref, tok, conf, com, mask)
    compare_entropy(ref, ent, mask)


@pytest.mark.parametrize("budget", [0.0, 1.0, 5.0, 60.0])
def test_entropy_bounded_rule(lib, budget):
    """entropy_bounded against the oracle on config-4-like blocks (L = 64, masked fraction
    U[0.1, 0.9], peaks U[0, 16] so the entropies spread), with a block that has no masked
    position; blocks whose decision the oracle flags as near the budget or a near-tie are
    counted, not failed."""
    rng = np.random.default_rng(300 + int(budget * 10))
    B, L, V = 8, 64, 20000
    mask = np.zeros((B, L), np.uint8)
    for b in range(B):
        mask[b] = W.make_mask_fixed_fraction(rng, 1, L, rng.uniform(0.1, 0.9))[0]
    mask[3] = 0
    logits = W.poison_unmasked_rows(W.make_logits(rng, B * L, V, peak_height=(0, 16)), mask)
    ref = oracle.confidence_commit(logits, mask, budget, 1.0, rule=oracle.RULE_ENTROPY_BOUNDED)
    tok, conf, com, ent = run_gpu(lib, logits, mask, budget, 1.0,
                                  rule=lib.BDLM_COMMIT_ENTROPY_BOUNDED, entropy=True)
    near_diff, near_blocks = compare_commit(ref, tok, conf, com, mask)
    compare_entropy(ref, ent, mask)
    has = mask.sum(1) > 0
    assert np.all(com.sum(1)[has] >= 1) and np.all(com.sum(1)[~has] == 0)
    assert lib.bdlm_device_error() == 0
    print(f"budget {budget}: commits per block {com.sum(1).tolist()}, near blocks "
          f"{near_blocks}, differing {near_diff}")


def test_entropy_bounded_full_size_config4(lib):
    c = W.CONFIGS[4]
    rng = np.random.default_rng(W.seed_for(4, 6))
    ci = W.commit_inputs(4, rng, c["B"], c["L"], c["V"], supplementary=True)
    ref = oracle.confidence_commit(ci.logits, ci.mask, 4.0, 1.0,
                                   rule=oracle.RULE_ENTROPY_BOUNDED)
    tok, conf, com, ent = run_gpu(lib, ci.logits, ci.mask, 4.0, 1.0,
                                  rule=lib.BDLM_COMMIT_ENTROPY_BOUNDED, entropy=True)
    compare_commit(ref, tok, conf, com, ci.mask)
    compare_entropy(ref, ent, ci.mask)
