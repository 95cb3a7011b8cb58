"""Parity of the CUDA selective LM head with the fp64 oracle, through the C-ABI.

Tolerance: |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| per logit (fp32 accumulation, one
rounding to bf16).  Rows that are not active must keep their previous contents."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import bf16_tensor, dev

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2


def run_gpu(lib, inp: W.LmHeadInputs):
    import torch
    logits = torch.full((inp.n_rows, inp.V), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.bdlm_lm_head(bf16_tensor(inp.hidden), bf16_tensor(inp.w), dev(inp.active_idx),
                     len(inp.active_idx), inp.n_rows, inp.H, inp.V, logits)
    torch.cuda.synchronize()
    return logits.float().cpu().numpy().astype(np.float64)


def check(lib, inp, rows_sample=None, cols=None):
    got = run_gpu(lib, inp)
    act = inp.active_idx
    inactive = np.setdiff1d(np.arange(inp.n_rows), act)
    assert np.all(np.isnan(got[inactive])), "an inactive row was written"
    rows = act if rows_sample is None else rows_sample
    ref = oracle.lm_head(inp.hidden, inp.w, rows, cols)
    g = got[rows] if cols is None else got[rows][:, cols]
    excess = np.abs(g - ref) - (ATOL + RTOL * np.abs(ref))
    assert excess.max() <= 0, f"max excess {excess.max()}"
    assert lib.bdlm_device_error() == 0
    return np.abs(g - ref).max()


@pytest.mark.parametrize("n_rows,n_act,H,V", [(40, 23, 256, 1000), (8, 1, 64, 136),
                                              (300, 300, 512, 2048), (700, 600, 128, 4104),
                                              (130, 129, 2560, 640), (64, 64, 72, 128 + 8),
                                              (100, 100, 320, 1000), (512, 256, 2560, 1288)])
def test_small_shapes(lib, n_rows, n_act, H, V):
    rng = np.random.default_rng(n_rows + H + V)
    act = np.sort(rng.choice(n_rows, size=n_act, replace=False)).astype(np.int32)
    check(lib, W.lm_head_inputs(rng, n_rows, H, V, act))


@pytest.mark.parametrize("L,H,n_sample", [(16, 2560, 6), (32, 2560, 4)])
def test_config3_full_size_sampled(lib, L, H, n_sample):
    """Config-3 shape: B=64, 75% DENOISING sequences, all their rows active."""
    c = W.CONFIGS[3]
    rng = np.random.default_rng(W.seed_for(3, L))
    den = W.denoising_sequences(rng, c["B"])
    act = W.rows_of_sequences(den, L)
    inp = W.lm_head_inputs(rng, c["B"] * L, H, c["V"], act)
    pick = np.unique(np.concatenate([act[:1], act[-1:], rng.choice(act, n_sample - 2)]))
    err = check(lib, inp, rows_sample=pick)
    cols = np.sort(rng.choice(c["V"], 96, replace=False)).astype(np.int32)
    check(lib, inp, cols=cols)
    print(f"config 3 L={L}: {len(act)} active rows, max abs err {err:.3e}")


def test_config5_step_shape_sampled(lib):
    c = W.CONFIGS[5]
    rng = np.random.default_rng(W.seed_for(5))
    act = np.arange(0, c["B"] * c["L"], dtype=np.int32)
    inp = W.lm_head_inputs(rng, c["B"] * c["L"], c["H"], c["V"], act)
    check(lib, inp, rows_sample=np.array([0, 257, 511], np.int32))


def test_bad_row_index_is_flagged(lib):
    rng = np.random.default_rng(4)
    inp = W.lm_head_inputs(rng, 16, 64, 256, np.array([0, 3], np.int32))
    import torch
    logits = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")
    act = dev(np.array([0, 3], np.int32))
    lib.bdlm_lm_head(bf16_tensor(inp.hidden), bf16_tensor(inp.w), act, 2, 16, 64, 256, logits)
    torch.cuda.synchronize()
    assert lib.bdlm_device_error() == 0
    bad = dev(np.array([0, 1], np.int32))
    bad[1] = 1000  # outside [0, n_rows): gathered as zeros, flagged, never written
    logits.fill_(0)
    lib.bdlm_lm_head(bf16_tensor(inp.hidden), bf16_tensor(inp.w), bad, 2, 16, 64, 256, logits)
    torch.cuda.synchronize()
    assert lib.bdlm_device_error() & lib.BDLM_DEVERR_ROW
    assert torch.all(logits[1:] == 0)
