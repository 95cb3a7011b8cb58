"""The failure path every kernel shares, provoked without a fault: a bounded wait on an
mbarrier that nothing arrives on gives up, the kernel records BDLM_DEVERR_TIMEOUT in the
device error word, bdlm_device_error() reports and clears it, and the context stays usable
(a block attention afterwards still matches the oracle)."""
import time

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import bf16_tensor, dev

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_is_reported_and_the_context_survives(lib):
    import torch
    assert lib.bdlm_device_error() == 0
    t0 = time.perf_counter()
    lib.bdlm_selftest_wait_timeout(20000)          # 20 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert 0.015 < elapsed < 5.0, elapsed          # it waited its limit, then gave up
    assert lib.bdlm_device_error() == lib.BDLM_DEVERR_TIMEOUT
    assert lib.bdlm_device_error() == 0            # read and cleared

    rng = np.random.default_rng(77)
    a = W.make_attention(rng, 2, 4, 32, 8, 128, prefix_range=(20, 300), poison=False)
    out = torch.empty((a.B, a.L, a.Hq, a.D), dtype=torch.bfloat16, device="cuda")
    desc = lib.attn_desc(a.B, a.L, a.Hq, a.Hkv, a.D, a.page_table_ref.shape[1], a.k_ref.shape[0])
    lib.bdlm_block_attention(desc, bf16_tensor(a.q), bf16_tensor(a.k_ref), bf16_tensor(a.v_ref),
                             dev(a.page_table_ref), dev(a.prefix_lens), a.L, out)
    torch.cuda.synchronize()
    ref = oracle.block_attention(a.q, a.k_ref, a.v_ref, a.page_table_ref, a.prefix_lens, a.L,
                                 a.Hq, a.Hkv, a.D, a.P)
    got = out.float().cpu().numpy().astype(np.float64)
    assert (np.abs(got - ref) - (1e-2 + 1e-2 * np.abs(ref))).max() <= 0
    assert lib.bdlm_device_error() == 0
