"""The device-side round loop (one CUDA graph with a conditional WHILE node) against an fp64
oracle chain, step by step.

For every step s the oracle chain runs, on the host and in the order the round defines it:
the block's K/V of step s written into the cache (oracle.write_block_kv), block attention
over that cache (oracle.block_attention), the LM head on the scored rows -- masked, in a
DENOISING sequence -- rounded once to bf16 (oracle.lm_head, oracle.round_logits_to_bf16), the
confidence and the block decision by the loop's rule (oracle.confidence_commit) and the mask
update (oracle.apply_commit).  The loop must give the same per-step attention output (within
1e-2 + 1e-2 |ref|), the same tokens and commits (bit for bit), confidences within 1e-5, the
same final mask and bit-identical K/V pools, and stop after the same number of steps.

The LM-head inputs are exact: hidden = k/8 and W = k/32 for small integers k, with a few
hidden rows per step set to the signs of one vocabulary row of W on 256 dims (a large logit),
so every dot product is exact in fp32 and the GPU's bf16 logits equal the oracle's.  A block
whose commit differs only on a decision the oracle flags as within 1e-5 of the threshold or
of a tie is counted, not failed, and the chain then follows the GPU's commit for it.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import bf16_tensor, dev, host

pytestmark = pytest.mark.gpu


class Case:
    def __init__(self, seed, B=12, L=4, Hq=8, Hkv=4, H=512, V=4104, S=4, frac=0.75,
                 prefix=(40, 400), saving_masked=False, peaks_per_step=None):
        import torch
        rng = np.random.default_rng(seed)
        self.B, self.L, self.Hq, self.Hkv, self.H, self.V, self.S = B, L, Hq, Hkv, H, V, S
        self.a = W.make_attention(rng, B, L, Hq, Hkv, 128, prefix_range=prefix, poison=False)
        R = B * L
        self.q_h = W._normal_bf16(rng, (S, B, L, Hq, 128), 0.5)
        self.kn_h = W._normal_bf16(rng, (S, B, L, Hkv, 128), 0.5)
        self.vn_h = W._normal_bf16(rng, (S, B, L, Hkv, 128), 0.5)
        w = rng.integers(-8, 9, size=(V, H)).astype(np.float32) / 32
        hid = rng.integers(-8, 9, size=(S, R, H)).astype(np.float32) / 8
        n_pk = peaks_per_step if peaks_per_step is not None else max(2, R // 3)
        for s in range(S):
            for r in rng.choice(R, n_pk, replace=False):
                t = int(rng.integers(0, V))
                hid[s, r, :256] = np.where(w[t, :256] >= 0, 1.0, -1.0)
        self.w_h = W.f32_to_bf16_bits(w)
        self.hid_h = W.f32_to_bf16_bits(hid)
        self.mask0 = W.make_mask_fixed_fraction(rng, B, L, frac)
        self.mask0[1] = 0                               # a block with nothing to do
        self.den = W.denoising_sequences(rng, B, 0.75)
        if not saving_masked:
            self.mask0[self.den == 0] = 0               # SAVING sequences have no masked slot
        self.q, self.kn, self.vn = bf16_tensor(self.q_h), bf16_tensor(self.kn_h), bf16_tensor(self.vn_h)
        self.hid, self.w = bf16_tensor(self.hid_h), bf16_tensor(self.w_h)
        self.k0, self.v0 = bf16_tensor(self.a.k_ref), bf16_tensor(self.a.v_ref)
        self.pt, self.pl = dev(self.a.page_table_ref), dev(self.a.prefix_lens)
        self.torch = torch

    def desc(self, lib):
        a = self.a
        return lib.attn_desc(self.B, self.L, self.Hq, self.Hkv, 128, a.page_table_ref.shape[1],
                             a.k_ref.shape[0])


def run_loop(lib, c, rule, k, thr, launches=1, regrow=False):
    torch = c.torch
    kp, vp = c.k0.clone(), c.v0.clone()
    mask = dev(c.mask0)
    tok = torch.full((c.S, c.B, c.L), -9, dtype=torch.int32, device="cuda")
    conf = torch.full((c.S, c.B, c.L), 9.0, dtype=torch.float32, device="cuda")
    com = torch.full((c.S, c.B, c.L), 9, dtype=torch.uint8, device="cuda")
    out = torch.full((c.S, c.B, c.L, c.Hq, 128), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    done = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    den = dev(c.den)
    d = lib.round_loop_desc(c.desc(lib), c.S, c.H, c.V, rule, k, thr, 1.0, q_steps=c.q,
                            k_new_steps=c.kn, v_new_steps=c.vn, hidden_steps=c.hid, k_pages=kp,
                            v_pages=vp, page_table=c.pt, prefix_lens=c.pl, w=c.w, mask=mask,
                            denoising=den, tok_steps=tok, conf_steps=conf, commit_steps=com,
                            steps_done=done, attn_out_steps=out)
    loop = lib.bdlm_round_loop_create(d)
    try:
        for i in range(launches):
            if i > 0:
                mask.copy_(dev(c.mask0))
                kp.copy_(c.k0)
                vp.copy_(c.v0)
                if regrow:
                    # a bigger LM-head call grows the library workspace: the loop re-captures
                    big = torch.zeros((4096, 1024), dtype=torch.bfloat16, device="cuda")
                    lib.bdlm_lm_head(big, big, torch.arange(4096, dtype=torch.int32,
                                                            device="cuda"), 4096, 4096, 1024,
                                     1024, torch.empty((4096, 1024), dtype=torch.bfloat16,
                                                       device="cuda"))
            lib.bdlm_round_loop_launch(loop)
        torch.cuda.synchronize()
    finally:
        lib.bdlm_round_loop_destroy(loop)
    assert lib.bdlm_device_error() == 0
    kp_h = kp.view(torch.int16).cpu().numpy().view(np.uint16)
    vp_h = vp.view(torch.int16).cpu().numpy().view(np.uint16)
    return dict(tok=host(tok), conf=host(conf), com=host(com), done=int(done.item()),
                mask=host(mask), kp=kp_h, vp=vp_h, out=out.float().cpu().numpy())


def check_against_oracle_chain(c, got, rule, k, thr):
    """Replays the loop's steps in the oracle and compares every step; returns the number of
    blocks whose commit differed on a flagged near-tie."""
    a, L, R = c.a, c.L, c.B * c.L
    kp, vp = a.k_ref.copy(), a.v_ref.copy()
    mask = c.mask0.copy()
    scoring = (c.den != 0)[:, None]
    near_blocks, steps = 0, 0
    for s in range(c.S):
        steps = s + 1
        kp, vp = oracle.write_block_kv(kp, vp, a.page_table_ref, a.prefix_lens, c.kn_h[s],
                                       c.vn_h[s])
        ref_out = oracle.block_attention(c.q_h[s], kp, vp, a.page_table_ref, a.prefix_lens, L,
                                         c.Hq, c.Hkv, 128, 16)
        err = np.abs(got["out"][s] - ref_out) - (1e-2 + 1e-2 * np.abs(ref_out))
        assert err.max() <= 0, f"step {s}: attention differs from the oracle by {err.max()}"
        rows = oracle.active_rows(mask, c.den)
        lg = np.full((R, c.V), 0x7FC0, np.uint16)
        if len(rows):
            lg[rows] = oracle.round_logits_to_bf16(oracle.lm_head(c.hid_h[s], c.w_h, rows))
        scored = (mask != 0) & scoring
        ref = oracle.confidence_commit(lg, scored.astype(np.uint8), thr, 1.0, rule=rule, k=k)
        tok, conf, com = got["tok"][s], got["conf"][s], got["com"][s]
        assert np.array_equal(tok[scored], ref.tok[scored]), f"step {s}: tokens differ"
        assert np.all(tok[~scored] == -1) and np.all(np.isneginf(conf[~scored]))
        rel = np.abs(conf[scored].astype(np.float64) - ref.conf[scored]) / ref.conf[scored]
        assert rel.max(initial=0.0) <= 1e-5, f"step {s}: confidence rel err {rel.max()}"
        commit = ref.commit.copy()
        for b in range(c.B):
            if not np.array_equal(com[b], ref.commit[b]):
                assert np.any(ref.near[b]), f"step {s} block {b}: commit differs"
                near_blocks += 1
                commit[b] = com[b]             # both are correct: follow the GPU's choice
        assert np.all(com[~scored] == 0)
        mask = oracle.apply_commit(mask, commit)
        if not mask.any():
            break
    assert got["done"] == steps, f"loop ran {got['done']} steps, the oracle chain {steps}"
    assert np.all(got["tok"][steps:] == -9) and np.all(got["com"][steps:] == 9)  # past the end
    assert np.isnan(got["out"][steps:]).all()
    assert np.array_equal(got["mask"], mask)
    assert np.array_equal(got["kp"], kp) and np.array_equal(got["vp"], vp)
    return near_blocks


@pytest.mark.parametrize("rule,k,thr", [(0, 1, 0.6), (1, 1, 0.5), (1, 2, 0.5), (2, 2, 0.5),
                                        (3, 1, 0.5), (4, 1, 1.5)])
def test_loop_matches_oracle_chain(lib, rule, k, thr):
    c = Case(seed=40 + rule + 10 * k)
    got = run_loop(lib, c, rule, k, thr)
    near = check_against_oracle_chain(c, got, rule, k, thr)
    assert np.all(got["mask"] == 0)                  # every block committed
    print(f"rule {rule} k {k}: {got['done']} steps, {near} near-tie blocks")


def test_loop_on_cta_pairs_matches_oracle_chain(lib):
    """160 rows (> 128): the fused LM head runs on CTA pairs inside the loop."""
    c = Case(seed=71, B=40, S=4, prefix=(16, 300))
    got = run_loop(lib, c, 0, 1, 0.6)
    check_against_oracle_chain(c, got, 0, 1, 0.6)


def test_masked_positions_of_saving_sequences_are_not_scored(lib):
    """Masked positions of SAVING sequences are never scored or committed: the loop runs every
    step slot and leaves them masked, in step with the oracle chain."""
    c = Case(seed=19, S=3, saving_masked=True)
    assert (c.mask0[c.den == 0] != 0).any()
    got = run_loop(lib, c, 0, 1, 0.6)
    check_against_oracle_chain(c, got, 0, 1, 0.6)
    assert got["done"] == c.S
    assert np.array_equal(got["mask"][c.den == 0], c.mask0[c.den == 0])


def test_loop_stops_early_and_relaunches(lib):
    """With more step slots than the block needs the loop stops when the mask is empty; a
    second launch of the same graph (inputs reset) gives the same answers, also after the
    library workspace has been reallocated in between."""
    c = Case(seed=7, S=9, L=4)
    first = run_loop(lib, c, 0, 1, 0.6)
    assert first["done"] <= 4
    check_against_oracle_chain(c, first, 0, 1, 0.6)
    again = run_loop(lib, c, 0, 1, 0.6, launches=2, regrow=True)
    for key in ("tok", "conf", "com", "mask", "kp", "vp"):
        assert np.array_equal(first[key], again[key]), key
    assert first["done"] == again["done"]
