"""The device-side round pieces through the C-ABI: active rows from the mask, the LM head with
a device-side row count, and the block K/V write, against the oracle's definitions."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import bf16_tensor, dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,L,frac,flags", [(128, 4, 0.5, False), (64, 32, 0.3, True),
                                            (3, 1, 1.0, False), (40, 64, 0.05, True)])
def test_active_rows(lib, B, L, frac, flags):
    import torch
    rng = np.random.default_rng(B + L)
    mask = W.make_mask_fixed_fraction(rng, B, L, frac)
    mask[0] = 0
    den = W.denoising_sequences(rng, B) if flags else None
    idx = torch.full((B * L,), -7, dtype=torch.int32, device="cuda")
    n = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    lib.bdlm_active_rows(dev(mask), None if den is None else dev(den), B, L, idx, n)
    torch.cuda.synchronize()
    want = oracle.active_rows(mask, den)
    assert int(n.item()) == len(want)
    assert np.array_equal(host(idx)[:len(want)], want)


def test_active_rows_of_an_all_unmasked_batch(lib):
    import torch
    mask = np.zeros((5, 4), np.uint8)
    idx = torch.zeros((20,), dtype=torch.int32, device="cuda")
    n = torch.full((1,), 9, dtype=torch.int32, device="cuda")
    lib.bdlm_active_rows(dev(mask), None, 5, 4, idx, n)
    torch.cuda.synchronize()
    assert int(n.item()) == 0


def test_lm_head_device_count(lib):
    """Planned for 512 rows, run for the 300 active rows the device reports: those logits
    match the oracle (sampled columns), every other row is left untouched."""
    import torch
    rng = np.random.default_rng(21)
    n_rows, H, V = 512, 1024, 8192 + 8
    act = np.sort(rng.choice(n_rows, 300, replace=False)).astype(np.int32)
    inp = W.lm_head_inputs(rng, n_rows, H, V, act)
    idx = torch.full((n_rows,), 0, dtype=torch.int32, device="cuda")
    idx[:300] = dev(act)
    n = torch.tensor([300], dtype=torch.int32, device="cuda")
    logits = torch.full((n_rows, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.bdlm_lm_head_device_count(bf16_tensor(inp.hidden), bf16_tensor(inp.w), idx, n, n_rows,
                                  n_rows, H, V, logits)
    torch.cuda.synchronize()
    got = logits.float().cpu().numpy().astype(np.float64)
    cols = np.sort(rng.choice(V, 64, replace=False)).astype(np.int32)
    ref = oracle.lm_head(inp.hidden, inp.w, act, cols)
    g = got[act][:, cols]
    assert np.all(np.abs(g - ref) <= 1e-2 + 1e-2 * np.abs(ref))
    rest = np.setdiff1d(np.arange(n_rows), act)
    assert np.all(np.isnan(got[rest]))
    assert lib.bdlm_device_error() == 0


def test_lm_head_device_count_zero(lib):
    import torch
    rng = np.random.default_rng(2)
    inp = W.lm_head_inputs(rng, 64, 256, 1024, np.arange(64, dtype=np.int32))
    n = torch.zeros((1,), dtype=torch.int32, device="cuda")
    logits = torch.full((64, 1024), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.bdlm_lm_head_device_count(bf16_tensor(inp.hidden), bf16_tensor(inp.w),
                                  dev(inp.active_idx), n, 64, 64, 256, 1024, logits)
    torch.cuda.synchronize()
    assert torch.all(torch.isnan(logits))


@pytest.mark.parametrize("B,L,Hkv", [(5, 4, 8), (3, 16, 2), (2, 64, 1), (4, 7, 3), (3, 64, 16)])
def test_write_block_kv(lib, B, L, Hkv):
    import torch
    rng = np.random.default_rng(B * 100 + L)
    a = W.make_attention(rng, B, L, 2 * Hkv, Hkv, 128, prefix_range=(0, 300), poison=False)
    k_new = W._normal_bf16(rng, (B, L, Hkv, 128), 0.5)
    v_new = W._normal_bf16(rng, (B, L, Hkv, 128), 0.5)
    kp, vp = bf16_tensor(a.k_ref), bf16_tensor(a.v_ref)
    desc = lib.attn_desc(B, L, 2 * Hkv, Hkv, 128, a.page_table_ref.shape[1], a.k_ref.shape[0])
    lib.bdlm_write_block_kv(desc, bf16_tensor(k_new), bf16_tensor(v_new), kp, vp,
                            dev(a.page_table_ref), dev(a.prefix_lens))
    torch.cuda.synchronize()
    k_ref, v_ref = oracle.write_block_kv(a.k_ref, a.v_ref, a.page_table_ref, a.prefix_lens,
                                         k_new, v_new)
    assert np.array_equal(host(kp.view(torch.int16)).view(np.uint16), k_ref)
    assert np.array_equal(host(vp.view(torch.int16)).view(np.uint16), v_ref)
    assert lib.bdlm_device_error() == 0


def test_write_block_kv_bad_page_is_flagged(lib):
    import torch
    rng = np.random.default_rng(3)
    a = W.make_attention(rng, 2, 4, 8, 8, 128, prefix_range=(20, 40), poison=False)
    pt = a.page_table_ref.copy()
    j = int(a.prefix_lens[1])
    pt[1, j // 16] = a.k_ref.shape[0] + 5      # outside the pool
    kp, vp = bf16_tensor(a.k_ref), bf16_tensor(a.v_ref)
    desc = lib.attn_desc(2, 4, 8, 8, 128, pt.shape[1], a.k_ref.shape[0])
    k_new = W._normal_bf16(rng, (2, 4, 8, 128), 0.5)
    lib.bdlm_write_block_kv(desc, bf16_tensor(k_new), bf16_tensor(k_new), kp, vp, dev(pt),
                            dev(a.prefix_lens))
    torch.cuda.synchronize()
    assert lib.bdlm_device_error() & lib.BDLM_DEVERR_PAGE
