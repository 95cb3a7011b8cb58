"""Block prefill through the C-ABI against the oracle: the prompt's pages bit-exact and the
block-causal attention output within 1e-2 + 1e-2 |ref|."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import bf16_tensor, dev, host

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2


def run(lib, B, L, Hq, Hkv, n, prefix_range, seed):
    import torch
    rng = np.random.default_rng(seed)
    lens = rng.integers(prefix_range[0], prefix_range[1] + 1, size=B)
    # pages for the cached prefix and the prompt (the generator's block length is the prompt)
    a = W.make_attention(rng, B, n, Hq, Hkv, 128, prefix_lens=lens, poison=False)
    q = W._normal_bf16(rng, (B, n, Hq, 128), 0.5)
    kn = W._normal_bf16(rng, (B, n, Hkv, 128), 0.5)
    vn = W._normal_bf16(rng, (B, n, Hkv, 128), 0.5)
    kp, vp = bf16_tensor(a.k_ref), bf16_tensor(a.v_ref)
    out = torch.full((B, n, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    desc = lib.attn_desc(B, L, Hq, Hkv, 128, a.page_table_ref.shape[1], a.k_ref.shape[0])
    lib.bdlm_prefill_attention(desc, n, bf16_tensor(q), bf16_tensor(kn), bf16_tensor(vn), kp, vp,
                               dev(a.page_table_ref), dev(a.prefix_lens), out)
    torch.cuda.synchronize()
    ref, k_ref, v_ref = oracle.prefill_attention(q, kn, vn, a.k_ref, a.v_ref, a.page_table_ref,
                                                 a.prefix_lens, L, Hq, Hkv, 128)
    assert np.array_equal(host(kp.view(torch.int16)).view(np.uint16), k_ref)
    assert np.array_equal(host(vp.view(torch.int16)).view(np.uint16), v_ref)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    assert excess.max() <= 0, f"max excess {excess.max()}"
    assert lib.bdlm_device_error() == 0


@pytest.mark.parametrize("B,L,Hq,Hkv,n,prefix", [(3, 4, 32, 8, 64, (0, 0)),
                                                (2, 16, 32, 8, 256, (0, 0)),
                                                (4, 4, 16, 8, 48, (0, 300)),
                                                (2, 64, 32, 8, 128, (17, 100))])
def test_prefill(lib, B, L, Hq, Hkv, n, prefix):
    run(lib, B, L, Hq, Hkv, n, prefix, seed=B * 1000 + n)


def test_prefill_rejects_a_ragged_prompt(lib):
    import torch
    desc = lib.attn_desc(1, 4, 8, 8, 128, 4, 4)
    z = torch.zeros((1, 6, 8, 128), dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    pl = torch.zeros((1,), dtype=torch.int32, device="cuda")
    pool = torch.zeros((4, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.BdlmError):
        lib.bdlm_prefill_attention(desc, 6, z, z, z, pool, pool, pt, pl, z)
