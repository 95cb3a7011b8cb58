"""The chained denoising round (attention -> selective LM head -> commit -> mask update),
repeated for a whole block, against the fp64 oracle.

Exact chain: hidden and W are small integers times powers of two, so every LM-head dot
product is exact in fp32 and the GPU's logits round to the same bf16 as the oracle's; every
token, confidence and commit decision of every step is then comparable (decisions the oracle
flags as within 1e-5 of the threshold or of a tie are counted, not failed, and the block is
no longer compared once it diverges).
Full size (B=128, L=4, SDAR-8B LM head, 4 steps): the GPU runs the whole batch; the oracle
checks sampled sequences' attention and logits, every step's tokens, confidences and commits
over the GPU's stored bf16 logits of every active row, and the chain's invariants.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import bf16_tensor, compare_commit, dev

pytestmark = pytest.mark.gpu


def _exact_lm_inputs(rng, n_rows, H, V, peaks):
    """hidden = k/8, W = k/32 with small integers k: products are multiples of 2^-8 and every
    partial sum of H of them is exact in fp32.  `peaks` (row, token) pairs get a W row that
    agrees in sign with the row's hidden vector on its first 256 dims (a large logit)."""
    hidden = rng.integers(-8, 9, size=(n_rows, H)).astype(np.float32) / 8
    w = rng.integers(-8, 9, size=(V, H)).astype(np.float32) / 32
    for r, t in peaks:
        w[t, :256] = np.sign(hidden[r, :256]) * 0.25
    return W.f32_to_bf16_bits(hidden), W.f32_to_bf16_bits(w)


def _gpu_step(lib, mask_d, hidden_d, w_d, act, B, L, H, V, tau, T, logits_d):
    import torch
    if len(act):
        lib.bdlm_lm_head(hidden_d, w_d, dev(act), len(act), B * L, H, V, logits_d)
    tok = torch.empty((B, L), dtype=torch.int32, device="cuda")
    conf = torch.empty((B, L), dtype=torch.float32, device="cuda")
    com = torch.empty((B, L), dtype=torch.uint8, device="cuda")
    lib.bdlm_confidence_commit(logits_d, mask_d, B, L, V, tau, T, tok, conf, com)
    lib.bdlm_apply_commit(mask_d, com, B * L)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), conf.cpu().numpy(), com.cpu().numpy()


def test_exact_chain_small(lib):
    import torch
    rng = np.random.default_rng(W.seed_for(5, 99))
    B, L, H, V, steps, tau, T = 12, 4, 512, 4096 + 8, 4, 0.75, 1.0
    mask = np.ones((B, L), np.uint8)
    mask_d = dev(mask.copy())
    logits_d = torch.full((B * L, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    live = np.ones(B, bool)       # blocks still compared
    near_blocks = 0
    for s in range(steps):
        peaks = [(int(r), int(rng.integers(0, V))) for r in rng.choice(B * L, 6, replace=False)]
        hidden, w = _exact_lm_inputs(rng, B * L, H, V, peaks)
        act = np.nonzero(mask.reshape(-1))[0].astype(np.int32)
        tok, conf, com = _gpu_step(lib, mask_d, bf16_tensor(hidden), bf16_tensor(w), act, B, L,
                                   H, V, tau, T, logits_d)
        # oracle: fp64 logits of the active rows, stored as bf16 like the GPU stores them
        lg = np.full((B * L, V), 0x7FC0, np.uint16)
        if len(act):
            ref64 = oracle.lm_head(hidden, w, act)
            lg[act] = oracle.round_logits_to_bf16(ref64)
        got_lg = logits_d.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got_lg[act], lg[act]), "exact logits differ"
        ref = oracle.confidence_commit(lg, mask, tau, T)
        m = mask == 1
        assert np.array_equal(tok[m], ref.tok[m])
        assert np.all(np.abs(conf[m] - ref.conf[m]) <= 1e-5 * np.abs(ref.conf[m]))
        for b in range(B):
            if not live[b]:
                continue
            if not np.array_equal(com[b], ref.commit[b]):
                assert np.any(ref.near[b]), f"step {s} block {b}: commit differs"
                near_blocks += 1
                live[b] = False
            assert com[b].sum() >= 1 or mask[b].sum() == 0
        mask = oracle.apply_commit(mask, ref.commit)
        assert np.array_equal(mask_d.cpu().numpy()[live], mask[live])
    assert np.all(mask[live] == 0), "every block is fully committed after L steps"
    print(f"exact chain: {near_blocks} blocks diverged on flagged near-ties")


def test_config5_full_size_chain(lib):
    """B=128, L=4, 4 steps, SDAR-8B LM head (H=4096, V=151936, W ~ N(0, 0.02^2))."""
    import torch
    c = W.CONFIGS[5]
    B, L, H, V, tau, T = c["B"], c["L"], c["H"], c["V"], c["threshold"], c["temperature"]
    rng = np.random.default_rng(W.seed_for(5))
    prefix = rng.integers(c["prefix"][0], c["prefix"][1] + 1, size=B).astype(np.int32)
    w = W._normal_bf16(rng, (V, H), 0.02)
    w_d = bf16_tensor(w)
    mask = np.ones((B, L), np.uint8)
    mask_d = dev(mask.copy())
    logits_d = torch.full((B * L, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    sample = np.array([0, int(np.argmax(prefix))], np.int32)
    for s in range(c["steps"]):
        # attention of this step (fresh Q/K/V; the same prefix lengths every step)
        a = W.make_attention(rng, B, L, c["Hq"], c["Hkv"], c["D"], prefix_lens=prefix)
        shape = (a.pool_pages, a.P, a.Hkv, a.D)
        kp = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        vp = kp.clone()
        ids = torch.from_numpy(a.ref_page_ids.astype(np.int64)).cuda()
        kp[ids] = bf16_tensor(a.k_ref)
        vp[ids] = bf16_tensor(a.v_ref)
        out = torch.empty((B, L, a.Hq, a.D), dtype=torch.bfloat16, device="cuda")
        desc = lib.attn_desc(B, L, a.Hq, a.Hkv, a.D, a.page_table.shape[1], a.pool_pages)
        lib.bdlm_block_attention(desc, bf16_tensor(a.q), kp, vp, dev(a.page_table), dev(prefix),
                                 L, out)
        del kp, vp
        # LM head on the still-masked rows, then commit and mask update
        hidden = W._normal_bf16(rng, (B * L, H), 1.0)
        act = np.nonzero(mask.reshape(-1))[0].astype(np.int32)
        assert len(act) == B * (L - s), "fallback commits exactly one position per step here"
        tok, conf, com = _gpu_step(lib, mask_d, bf16_tensor(hidden), w_d, act, B, L, H, V, tau,
                                   T, logits_d)
        got_out = out.float().cpu().numpy().astype(np.float64)
        ref_out = oracle.block_attention(a.q, a.k_ref, a.v_ref, a.page_table_ref, a.prefix_lens,
                                         L, a.Hq, a.Hkv, a.D, a.P, seqs=sample)
        assert np.all(np.abs(got_out[sample] - ref_out[sample])
                      <= 1e-2 + 1e-2 * np.abs(ref_out[sample]))
        rows = np.array([r for r in act if r // L in sample][:4], np.int32)
        if len(rows):
            ref_lg = oracle.lm_head(hidden, w, rows)
            got_lg = logits_d.float().cpu().numpy()[rows].astype(np.float64)
            assert np.all(np.abs(got_lg - ref_lg) <= 1e-2 + 1e-2 * np.abs(ref_lg))
        # the step's commit against the oracle over the GPU's bf16 logits of every active row
        lg_bits = logits_d.view(torch.int16).cpu().numpy().view(np.uint16)
        ref = oracle.confidence_commit(lg_bits, mask, tau, T)
        near_differ, near_total = compare_commit(ref, tok, conf, com, mask)
        print(f"step {s}: {near_differ} of {near_total} near-threshold blocks differ")
        # invariants of the step on every block
        m = mask == 1
        assert np.all(com[~m] == 0) and np.all(com.sum(1) >= 1)
        mask = mask & (1 - com)
        assert np.array_equal(mask_d.cpu().numpy(), mask)
    assert mask.sum() == 0, "every block committed after 4 steps"
    assert lib.bdlm_device_error() == 0
