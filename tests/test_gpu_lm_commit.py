"""The fused LM head + confidence/commit (bdlm_lm_head_commit) through the C-ABI.

Checked against the oracle the way the unfused step is: the logits the fused kernel stores
(when asked) match the fp64 LM head within |err| <= 1e-2 + 1e-2 |ref|, and tok/conf/commit
equal the oracle's commit over those same bf16 logits (tokens and commits exact, except
blocks with a position within 1e-5 of the threshold; confidences within 1e-5 relative).  The
scored rows are the masked rows of DENOISING sequences; every other position must read
tok = -1, conf = -inf, commit = 0, and logits rows that are not scored stay untouched.  The
fused results also match the unfused calls (bdlm_lm_head, then
bdlm_confidence_commit_rule over the scored rows) exactly for tokens and commits.  The entropy
of every scored position is within 1e-4 + 1e-5 H of the oracle's over the same logits (+inf
elsewhere), and the entropy-bounded rule decides like the oracle."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import bf16_tensor, compare_commit, compare_entropy, dev, host

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2


def make_case(seed, B, L, H, V, mask_frac, den_frac, wstd):
    rng = np.random.default_rng(seed)
    hidden = W._normal_bf16(rng, (B * L, H), 1.0)
    w = W._normal_bf16(rng, (V, H), wstd)
    mask = W.make_mask_fixed_fraction(rng, B, L, mask_frac)
    den = None if den_frac is None else W.denoising_sequences(rng, B, den_frac)
    return rng, hidden, w, mask, den


def run_fused(lib, hidden, w, mask, den, B, L, H, V, rule, k, thr, T, want_logits=True):
    import torch
    tok = torch.full((B, L), -9, dtype=torch.int32, device="cuda")
    conf = torch.full((B, L), 9.0, dtype=torch.float32, device="cuda")
    com = torch.full((B, L), 9, dtype=torch.uint8, device="cuda")
    ent = torch.full((B, L), -5.0, dtype=torch.float32, device="cuda")
    logits = None
    if want_logits:
        logits = torch.full((B * L, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.bdlm_lm_head_commit(bf16_tensor(hidden), bf16_tensor(w), dev(mask),
                            None if den is None else dev(den), B, L, H, V, rule, k, thr, T, tok,
                            conf, com, logits, entropy_out=ent)
    torch.cuda.synchronize()
    assert lib.bdlm_device_error() == 0
    lg = None if logits is None else logits.view(torch.int16).cpu().numpy().view(np.uint16)
    return host(tok), host(conf), host(com), lg, host(ent)


def scored_mask(mask, den):
    m = mask.astype(bool)
    if den is not None:
        m &= den.astype(bool)[:, None]
    return m.astype(np.uint8)


def check_against_oracle(lib, case, B, L, H, V, rule, k, thr, T, col_sample=None):
    rng, hidden, w, mask, den = case
    tok, conf, com, lg, ent = run_fused(lib, hidden, w, mask, den, B, L, H, V, rule, k, thr, T)
    sm = scored_mask(mask, den)
    rows = np.nonzero(sm.reshape(-1))[0].astype(np.int32)
    others = np.setdiff1d(np.arange(B * L), rows)
    assert np.all(lg[others] == 0x7FC0), "a row that is not scored was written"
    if len(rows):
        cols = None
        if col_sample is not None:
            cols = np.sort(rng.choice(V, col_sample, replace=False)).astype(np.int32)
        ref = oracle.lm_head(hidden, w, rows, cols)
        got = (lg[rows].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        if cols is not None:
            got = got[:, cols]
        excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
        assert excess.max() <= 0, f"logits: max excess {excess.max()}"
    ref_c = oracle.confidence_commit(lg, sm, thr, T, rule=rule, k=k)
    near, _ = compare_commit(ref_c, tok, conf, com, sm)
    compare_entropy(ref_c, ent, sm)
    return tok, conf, com, near


# (seed, B, L, H, V, masked fraction, DENOISING fraction or None, W std, rule, k, tau, T)
CASES = [
    (1, 64, 4, 256, 4104, 0.5, 0.75, 0.2, 0, 1, 0.5, 1.0),     # V tail of 8 columns
    (2, 128, 4, 512, 1000, 1.0, None, 0.15, 0, 1, 0.3, 0.7),   # 512 rows: two row tiles
    (3, 48, 16, 256, 2048, 0.9, None, 0.2, 1, 3, 0.0, 1.0),    # ~690 rows: three row tiles
    (4, 3, 64, 128, 136, 0.5, None, 0.3, 2, 5, 0.0, 1.0),      # one partial vocabulary tile
    (5, 8, 1, 64, 256, 1.0, 0.5, 0.3, 3, 1, 0.0, 2.0),         # L = 1
    (6, 40, 32, 320, 1288, 0.3, 0.75, 0.2, 0, 1, 0.9, 1.0),
    (7, 65, 2, 2560, 640, 1.0, None, 0.05, 0, 1, 0.2, 1.0),    # 130 rows: a ragged sub-tile
    (8, 1, 4, 128, 64, 0.5, None, 0.5, 0, 1, 0.9, 1.0),        # V smaller than one share
    (9, 64, 16, 256, 2048, 0.8, 0.75, 0.3, 4, 1, 2.0, 1.0),    # entropy budget 2 nats
    (10, 150, 4, 512, 4104, 0.7, None, 0.25, 4, 1, 0.5, 0.8),  # entropy rule on CTA pairs
]


@pytest.mark.parametrize("seed,B,L,H,V,mf,df,wstd,rule,k,thr,T", CASES)
def test_fused_matches_oracle(lib, seed, B, L, H, V, mf, df, wstd, rule, k, thr, T):
    case = make_case(seed, B, L, H, V, mf, df, wstd)
    check_against_oracle(lib, case, B, L, H, V, rule, k, thr, T)


def test_fused_equals_unfused_and_logits_are_optional(lib):
    """Same tokens and commits as bdlm_lm_head + bdlm_confidence_commit_rule over the scored
    rows; confidences equal to float32 summation order; storing the logits changes nothing."""
    import torch
    B, L, H, V = 96, 4, 512, 4104
    case = make_case(11, B, L, H, V, 0.6, 0.75, 0.2)
    _, hidden, w, mask, den = case
    tok, conf, com, lg, _ = run_fused(lib, hidden, w, mask, den, B, L, H, V, 0, 1, 0.4, 1.0)
    tok2, conf2, com2, _, _ = run_fused(lib, hidden, w, mask, den, B, L, H, V, 0, 1, 0.4, 1.0,
                                        want_logits=False)
    assert np.array_equal(tok, tok2) and np.array_equal(com, com2)
    assert np.array_equal(conf, conf2)
    sm = scored_mask(mask, den)
    rows = np.nonzero(sm.reshape(-1))[0].astype(np.int32)
    logits = torch.full((B * L, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.bdlm_lm_head(bf16_tensor(hidden), bf16_tensor(w), dev(rows), len(rows), B * L, H, V,
                     logits)
    t3 = torch.empty((B, L), dtype=torch.int32, device="cuda")
    c3 = torch.empty((B, L), dtype=torch.float32, device="cuda")
    m3 = torch.empty((B, L), dtype=torch.uint8, device="cuda")
    lib.bdlm_confidence_commit_rule(logits, dev(sm), B, L, V, 0, 1, 0.4, 1.0, t3, c3, m3)
    torch.cuda.synchronize()
    assert np.array_equal(logits.view(torch.int16).cpu().numpy().view(np.uint16)[rows], lg[rows])
    assert np.array_equal(host(t3), tok) and np.array_equal(host(m3), com)
    s = sm.astype(bool)
    rel = np.abs(host(c3)[s].astype(np.float64) - conf[s]) / conf[s]
    assert rel.max() <= 1e-5
    assert np.array_equal(host(c3)[~s], conf[~s])


def test_nothing_scored(lib):
    B, L, H, V = 6, 4, 64, 256
    case = make_case(12, B, L, H, V, 0.5, None, 0.2)
    _, hidden, w, mask, _ = case
    den = np.zeros(B, np.uint8)              # every sequence SAVING
    tok, conf, com, lg, ent = run_fused(lib, hidden, w, mask, den, B, L, H, V, 0, 1, 0.5, 1.0)
    assert np.all(tok == -1) and np.all(np.isneginf(conf)) and np.all(com == 0)
    assert np.all(np.isposinf(ent))
    assert np.all(lg == 0x7FC0)
    tok, conf, com, _, _ = run_fused(lib, hidden, w, np.zeros_like(mask), None, B, L, H, V, 0, 1,
                                     0.5, 1.0)
    assert np.all(tok == -1) and np.all(com == 0)


def test_config2_shape(lib):
    """Batch 128, block 4, SDAR-4B hidden 2560, V = 151936, half of each block masked: 256
    scored rows, one row tile.  Logits checked on sampled columns, the commit on all."""
    c = W.CONFIGS[2]
    B, L, V, H = c["B"], c["L"], c["V"], 2560
    case = make_case(W.seed_for(2) + 7, B, L, H, V, 0.5, None, 0.02)
    tok, conf, com, near = check_against_oracle(lib, case, B, L, H, V, 0, 1, 0.75, 1.0,
                                                col_sample=256)
    print(f"config-2 fused: {int(com.sum())} commits, {near} near-threshold blocks differ")


def test_config5_first_step_shape(lib):
    """Batch 128, block 4, SDAR-8B hidden 4096: all 512 rows scored (two row tiles)."""
    c = W.CONFIGS[5]
    B, L, V, H = c["B"], c["L"], c["V"], c["H"]
    case = make_case(W.seed_for(5) + 3, B, L, H, V, 1.0, None, 0.02)
    check_against_oracle(lib, case, B, L, H, V, 0, 1, 0.75, 1.0, col_sample=128)
