"""The device-side round loop (one CUDA graph with a conditional WHILE node) against the same
calls made one by one from the host: identical per-step tokens, confidences and commits, the
same final mask and KV cache; the loop stops as soon as every position is committed."""
import numpy as np
import pytest

import workloads as W
from gpu_util import bf16_tensor, dev, host

pytestmark = pytest.mark.gpu


class Case:
    def __init__(self, seed, B=12, L=4, Hq=8, Hkv=4, H=512, V=4104, S=4, frac=0.75,
                 prefix=(40, 400), saving_masked=False):
        import torch
        rng = np.random.default_rng(seed)
        self.B, self.L, self.Hq, self.Hkv, self.H, self.V, self.S = B, L, Hq, Hkv, H, V, S
        self.a = W.make_attention(rng, B, L, Hq, Hkv, 128, prefix_range=prefix, poison=False)
        R = B * L
        self.q = bf16_tensor(W._normal_bf16(rng, (S, B, L, Hq, 128), 0.5))
        self.kn = bf16_tensor(W._normal_bf16(rng, (S, B, L, Hkv, 128), 0.5))
        self.vn = bf16_tensor(W._normal_bf16(rng, (S, B, L, Hkv, 128), 0.5))
        self.hid = bf16_tensor(W._normal_bf16(rng, (S, R, H), 1.0))
        self.w = bf16_tensor(W._normal_bf16(rng, (V, H), 0.05))
        self.mask0 = W.make_mask_fixed_fraction(rng, B, L, frac)
        self.mask0[1] = 0                               # a block with nothing to do
        self.den = W.denoising_sequences(rng, B, 0.75)
        if not saving_masked:
            self.mask0[self.den == 0] = 0               # SAVING sequences have no masked slot
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
    done = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    den = dev(c.den)
    d = lib.round_loop_desc(c.desc(lib), c.S, c.H, c.V, rule, k, thr, 1.0, q_steps=c.q,
                            k_new_steps=c.kn, v_new_steps=c.vn, hidden_steps=c.hid, k_pages=kp,
                            v_pages=vp, page_table=c.pt, prefix_lens=c.pl, w=c.w, mask=mask,
                            denoising=den, tok_steps=tok, conf_steps=conf, commit_steps=com,
                            steps_done=done)
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
    return host(tok), host(conf), host(com), int(done.item()), host(mask), kp, vp


def run_eager(lib, c, rule, k, thr):
    """The same round, call by call from the host, until no position is masked."""
    torch = c.torch
    kp, vp = c.k0.clone(), c.v0.clone()
    mask = dev(c.mask0)
    den = dev(c.den)
    out = torch.empty((c.B, c.L, c.Hq, 128), dtype=torch.bfloat16, device="cuda")
    tok = torch.empty((c.B, c.L), dtype=torch.int32, device="cuda")
    conf = torch.empty((c.B, c.L), dtype=torch.float32, device="cuda")
    com = torch.empty((c.B, c.L), dtype=torch.uint8, device="cuda")
    steps = []
    for s in range(c.S):
        lib.bdlm_write_block_kv(c.desc(lib), c.kn[s], c.vn[s], kp, vp, c.pt, c.pl)
        lib.bdlm_block_attention(c.desc(lib), c.q[s], kp, vp, c.pt, c.pl, c.L, out)
        lib.bdlm_lm_head_commit(c.hid[s], c.w, mask, den, c.B, c.L, c.H, c.V, rule, k, thr,
                                1.0, tok, conf, com)
        lib.bdlm_apply_commit(mask, com, c.B * c.L)
        torch.cuda.synchronize()
        steps.append((host(tok), host(conf), host(com)))
        if host(mask).sum() == 0:
            break
    return steps, host(mask), kp, vp


@pytest.mark.parametrize("rule,k,thr", [(0, 1, 0.6), (1, 1, 0.5), (2, 2, 0.5)])
def test_loop_matches_host_driven_round(lib, rule, k, thr):
    c = Case(seed=40 + rule)
    tok, conf, com, done, mask, kp, vp = run_loop(lib, c, rule, k, thr)
    steps, mask_e, kp_e, vp_e = run_eager(lib, c, rule, k, thr)
    assert done == len(steps)
    for s, (t, f, m) in enumerate(steps):
        assert np.array_equal(tok[s], t) and np.array_equal(com[s], m)
        assert np.array_equal(conf[s], f)
    assert np.all(tok[done:] == -9) and np.all(com[done:] == 9)   # slices past the end
    assert np.array_equal(mask, mask_e)
    assert c.torch.equal(kp, kp_e) and c.torch.equal(vp, vp_e)
    assert np.all(mask == 0)                                      # every block committed


def test_loop_stops_early_and_relaunches(lib):
    """With more step slots than the block needs the loop stops when the mask is empty; a
    second launch of the same graph (inputs reset) gives the same answers, also after the
    library workspace has been reallocated in between."""
    c = Case(seed=7, S=9, L=4)
    first = run_loop(lib, c, 0, 1, 0.6)
    assert first[3] <= 4
    again = run_loop(lib, c, 0, 1, 0.6, launches=2, regrow=True)
    for x, y in zip(first[:3], again[:3]):
        assert np.array_equal(x, y)
    assert first[3] == again[3]
    assert np.array_equal(first[4], again[4])


def test_masked_positions_of_saving_sequences_are_not_scored(lib):
    """Masked positions of SAVING sequences are never scored or committed: the loop runs every
    step slot, in step with the host-driven round, and leaves them masked."""
    c = Case(seed=19, S=3, saving_masked=True)
    assert (c.mask0[c.den == 0] != 0).any()
    tok, conf, com, done, mask, kp, vp = run_loop(lib, c, 0, 1, 0.6)
    steps, mask_e, kp_e, vp_e = run_eager(lib, c, 0, 1, 0.6)
    assert done == c.S == len(steps)
    for s, (t, f, m) in enumerate(steps):
        assert np.array_equal(tok[s], t) and np.array_equal(com[s], m)
        assert np.array_equal(conf[s], f)
        saving = c.den == 0
        assert np.all(t[saving] == -1) and np.all(m[saving] == 0)
    assert np.array_equal(mask, mask_e)
    assert np.array_equal(mask[c.den == 0], c.mask0[c.den == 0])
    assert c.torch.equal(kp, kp_e) and c.torch.equal(vp, vp_e)
