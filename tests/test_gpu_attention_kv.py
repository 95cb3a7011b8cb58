"""Block attention with the block's K/V-cache write fused in (bdlm_block_attention_kv), through
the C-ABI, against the fp64 oracle.

The block's own slots in the cache hold NaN before the call, so any read of a slot before its
new K/V is written there shows up as NaN in the output.  After the call the K/V pools must equal
oracle.write_block_kv of the initial pools bit for bit (untouched slots included), and the
output must match oracle.block_attention over the written cache within 1e-2 + 1e-2 |ref|.  The
fused call must also give exactly the output of the unfused pair (bdlm_write_block_kv, then
bdlm_block_attention) on the same inputs."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import bf16_tensor, dev

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2


def make_case(rng, B, L, Hq, Hkv, prefix_lens=None, prefix_range=(0, 0), pool_pages=None):
    a = W.make_attention(rng, B, L, Hq, Hkv, 128, prefix_range=prefix_range,
                         prefix_lens=prefix_lens, pool_pages=pool_pages, poison=True)
    kn = W._normal_bf16(rng, (B, L, Hkv, 128), 0.5)
    vn = W._normal_bf16(rng, (B, L, Hkv, 128), 0.5)
    k0, v0 = a.k_ref.copy(), a.v_ref.copy()
    for b in range(B):   # the block's slots are stale (NaN) until the call writes them
        for i in range(L):
            t = int(a.prefix_lens[b]) + i
            k0[a.page_table_ref[b, t // 16], t % 16] = W.BF16_NAN
            v0[a.page_table_ref[b, t // 16], t % 16] = W.BF16_NAN
    return a, kn, vn, k0, v0


def pools_on_device(a, k0, v0):
    import torch
    shape = (a.pool_pages, a.P, a.Hkv, a.D)
    kp = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    ids = torch.from_numpy(a.ref_page_ids.astype(np.int64)).cuda()
    kp[ids] = bf16_tensor(k0)
    vp[ids] = bf16_tensor(v0)
    return kp, vp, ids


def run(lib, a, kn, vn, k0, v0, fused=True, page_table=None, prefix_lens=None):
    import torch
    kp, vp, ids = pools_on_device(a, k0, v0)
    out = torch.full((a.B, a.L, a.Hq, a.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    pt = a.page_table if page_table is None else page_table
    pl = a.prefix_lens if prefix_lens is None else prefix_lens
    desc = lib.attn_desc(a.B, a.L, a.Hq, a.Hkv, a.D, pt.shape[1], a.pool_pages)
    if fused:
        lib.bdlm_block_attention_kv(desc, bf16_tensor(a.q), bf16_tensor(kn), bf16_tensor(vn), kp,
                                    vp, dev(pt), dev(pl), a.L, out)
    else:
        lib.bdlm_write_block_kv(desc, bf16_tensor(kn), bf16_tensor(vn), kp, vp, dev(pt), dev(pl))
        lib.bdlm_block_attention(desc, bf16_tensor(a.q), kp, vp, dev(pt), dev(pl), a.L, out)
    torch.cuda.synchronize()
    kr = kp[ids].view(torch.int16).cpu().numpy().view(np.uint16)
    vr = vp[ids].view(torch.int16).cpu().numpy().view(np.uint16)
    return out, kr, vr


def check(lib, a, kn, vn, k0, v0, seqs=None):
    out, kr, vr = run(lib, a, kn, vn, k0, v0)
    kw, vw = oracle.write_block_kv(k0, v0, a.page_table_ref, a.prefix_lens, kn, vn)
    assert np.array_equal(kr, kw) and np.array_equal(vr, vw), "K/V pools differ"
    ref = oracle.block_attention(a.q, kw, vw, a.page_table_ref, a.prefix_lens, a.L, a.Hq, a.Hkv,
                                 a.D, a.P, seqs=seqs)
    sel = np.arange(a.B) if seqs is None else np.asarray(seqs)
    got = out.float().cpu().numpy().astype(np.float64)[sel]
    assert np.all(np.isfinite(got)), "a stale (NaN) block slot was read"
    excess = np.abs(got - ref[sel]) - (ATOL + RTOL * np.abs(ref[sel]))
    assert excess.max() <= 0, f"max excess {excess.max()}"
    assert lib.bdlm_device_error() == 0
    return out


@pytest.mark.parametrize("L", [1, 4, 7, 16, 32, 64])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 2)])
def test_small_shapes(lib, L, Hq, Hkv):
    """Blocks starting mid-page and at page starts, an empty prefix, and (16 query heads per KV
    head at L = 64) several query-row groups writing the same tokens."""
    rng = np.random.default_rng(9000 + L * 10 + Hq)
    lens = np.array([0, 14, 31, 64 + 5], np.int64)
    a, kn, vn, k0, v0 = make_case(rng, 4, L, Hq, Hkv, prefix_lens=lens)
    check(lib, a, kn, vn, k0, v0)


@pytest.mark.parametrize("L,lens", [(4, (893, 894, 895, 896, 2000)),       # 896-token splits
                                    (16, (2040, 2047, 2032, 4090, 100)),   # 2048-token splits
                                    (64, (2040, 2000, 1990, 3000, 5000)),
                                    (32, (4000, 4090, 1000, 2030, 17))])
def test_blocks_straddling_kv_splits(lib, L, lens):
    """Sequences long enough to be cut into KV splits, with blocks that cross a split boundary:
    each split's item writes the block tokens it reads."""
    rng = np.random.default_rng(L * 31 + lens[0])
    a, kn, vn, k0, v0 = make_case(rng, len(lens), L, 32, 8, prefix_lens=np.array(lens))
    check(lib, a, kn, vn, k0, v0)


def test_whole_sequence_mode(lib):
    """Enough sequences for whole-sequence items (no splits)."""
    rng = np.random.default_rng(4242)
    a, kn, vn, k0, v0 = make_case(rng, 160, 4, 32, 8, prefix_range=(0, 1200))
    check(lib, a, kn, vn, k0, v0)


def test_fused_equals_unfused_bit_for_bit(lib):
    import torch
    rng = np.random.default_rng(99)
    a, kn, vn, k0, v0 = make_case(rng, 24, 16, 32, 8, prefix_range=(0, 3000))
    o1, k1, v1 = run(lib, a, kn, vn, k0, v0, fused=True)
    o2, k2, v2 = run(lib, a, kn, vn, k0, v0, fused=False)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)


@pytest.mark.parametrize("config,L,sample", [(2, 4, 16), (4, 64, 2)])
def test_configs_full_size_sampled(lib, config, L, sample):
    c = W.CONFIGS[config]
    rng = np.random.default_rng(W.seed_for(config, 77))
    a, kn, vn, k0, v0 = make_case(rng, c["B"], L, c["Hq"], c["Hkv"], prefix_range=c["prefix"],
                                  pool_pages=c.get("pool_pages"))
    order = np.argsort(a.prefix_lens)
    pick = np.unique(np.concatenate([order[:1], order[-1:],
                                     rng.choice(a.B, size=sample - 2, replace=False)]))
    check(lib, a, kn, vn, k0, v0, seqs=pick)


def test_bad_page_ids_and_lengths_are_flagged_not_faulted(lib):
    rng = np.random.default_rng(5)
    a, kn, vn, k0, v0 = make_case(rng, 4, 4, 32, 8, prefix_range=(50, 300))
    pt = a.page_table.copy()
    last = (a.prefix_lens + 3) // 16
    pt[1, last[1]] = a.pool_pages + 5     # the block's page outside the pool
    run(lib, a, kn, vn, k0, v0, page_table=pt)
    assert lib.bdlm_device_error() & lib.BDLM_DEVERR_PAGE
    pl = a.prefix_lens.copy()
    pl[2] = pt.shape[1] * 16 + 100        # longer than the page table
    run(lib, a, kn, vn, k0, v0, prefix_lens=pl)
    assert lib.bdlm_device_error() & lib.BDLM_DEVERR_LENGTH
    check(lib, a, kn, vn, k0, v0)         # the library still works afterwards
