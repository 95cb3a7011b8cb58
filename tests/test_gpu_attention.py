"""Parity of the CUDA block attention with the fp64 oracle, through the C-ABI.

Tolerance: |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| per element (bf16 output, fp32
accumulation, P rounded to bf16 before the PV product)."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import bf16_tensor, dev

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2


def device_pools(a: W.AttnInputs, fill_nan=True):
    import torch
    shape = (a.pool_pages, a.P, a.Hkv, a.D)
    fill = float("nan") if fill_nan else 0.0
    kp = torch.full(shape, fill, dtype=torch.bfloat16, device="cuda")
    vp = torch.full(shape, fill, dtype=torch.bfloat16, device="cuda")
    ids = torch.from_numpy(a.ref_page_ids.astype(np.int64)).cuda()
    kp[ids] = bf16_tensor(a.k_ref)
    vp[ids] = bf16_tensor(a.v_ref)
    return kp, vp


def run_gpu(lib, a: W.AttnInputs, page_table=None, prefix_lens=None, sm_scale=0.0):
    import torch
    kp, vp = device_pools(a)
    out = torch.full((a.B, a.L, a.Hq, a.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    pt = a.page_table if page_table is None else page_table
    pl = a.prefix_lens if prefix_lens is None else prefix_lens
    desc = lib.attn_desc(a.B, a.L, a.Hq, a.Hkv, a.D, pt.shape[1], a.pool_pages, sm_scale=sm_scale)
    lib.bdlm_block_attention(desc, bf16_tensor(a.q), kp, vp, dev(pt), dev(pl), a.L, out)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def check(lib, a, seqs=None, sm_scale=None):
    got = run_gpu(lib, a, sm_scale=0.0 if sm_scale is None else sm_scale)
    ref = oracle.block_attention(a.q, a.k_ref, a.v_ref, a.page_table_ref, a.prefix_lens, a.L,
                                 a.Hq, a.Hkv, a.D, a.P, sm_scale=sm_scale, seqs=seqs)
    sel = np.arange(a.B) if seqs is None else np.asarray(seqs)
    g, r = got[sel], ref[sel]
    assert np.all(np.isfinite(g)), "non-finite output"
    excess = np.abs(g - r) - (ATOL + RTOL * np.abs(r))
    assert excess.max() <= 0, f"max excess {excess.max()} at {np.unravel_index(excess.argmax(), excess.shape)}"
    assert lib.bdlm_device_error() == 0
    return np.abs(g - r).max()


@pytest.mark.parametrize("L", [1, 4, 7, 16, 32, 64])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 8), (8, 8), (16, 2)])
def test_small_shapes(lib, L, Hq, Hkv):
    rng = np.random.default_rng(L * 1000 + Hq * 10 + Hkv)
    a = W.make_attention(rng, 3, L, Hq, Hkv, 128, prefix_range=(0, 700))
    a.prefix_lens[0] = 0                      # the block alone
    check(lib, a)


@pytest.mark.parametrize("L,prefix", [(4, (1000, 3000)), (16, (2000, 5000)), (64, (2040, 4200))])
def test_multiple_splits_and_chunks(lib, L, prefix):
    rng = np.random.default_rng(L + prefix[0])
    a = W.make_attention(rng, 4, L, 32, 8, 128, prefix_range=prefix)
    check(lib, a)


@pytest.mark.parametrize("L,kv", [
    (64, [64, 4096, 4097, 8192, 8193, 12417, 200]),    # two sub-groups: splits of <= 4096 tokens
    (32, [3072, 3073, 6144, 6145, 9217, 32, 1000]),     # one sub-group: splits of <= 3072 tokens
])
def test_even_splits_longest_first(lib, L, kv):
    """Query rows on M with KV lengths at and just past multiples of the longest split: every
    sequence is cut into equal splits of whole tiles, the last one taking what is left, and the
    items go out sequence by sequence, longest splits first."""
    rng = np.random.default_rng(L * 3 + len(kv))
    lens = np.asarray(kv, dtype=np.int64) - L
    a = W.make_attention(rng, len(kv), L, 32, 8, 128, prefix_lens=lens)
    check(lib, a)


@pytest.mark.parametrize("L,Hq,B,prefix", [(4, 32, 96, (100, 1900)), (8, 32, 160, (0, 1200)),
                                          (4, 16, 200, (3000, 4100)), (4, 32, 96, (2044, 2044))])
def test_whole_sequences_longest_first(lib, L, Hq, B, prefix):
    """Enough (sequence, KV head) items for whole sequences, longest first, with no KV
    splits: items of several tensor-memory chunks, sequences of equal length (ties in the
    order), the longest page table the mode takes, and every output checked."""
    rng = np.random.default_rng(B * 10 + L)
    lens = rng.integers(prefix[0], prefix[1] + 1, size=B)
    lens[1] = lens[0]
    lens[-1] = 0
    a = W.make_attention(rng, B, L, Hq, 8, 128, prefix_lens=lens)
    check(lib, a)


def test_config1(lib):
    c = W.CONFIGS[1]
    a = W.make_attention(np.random.default_rng(W.seed_for(1)), 1, 4, 16, 8, 128,
                         prefix_range=(60, 60), identity_pages=True)
    assert a.page_table.tolist() == [[0, 1, 2, 3]]
    check(lib, a)


@pytest.mark.parametrize("config,L,sample", [(2, 4, 24), (3, 16, 6), (3, 32, 6), (4, 64, 2)])
def test_configs_full_size_sampled(lib, config, L, sample):
    """The full workload on the GPU; the oracle recomputes a sample of sequences (always
    the shortest and the longest) exactly."""
    c = W.CONFIGS[config]
    rng = np.random.default_rng(W.seed_for(config, L))
    a = W.make_attention(rng, c["B"], L, c["Hq"], c["Hkv"], c["D"], prefix_range=c["prefix"],
                         pool_pages=c.get("pool_pages"))
    order = np.argsort(a.prefix_lens)
    pick = np.unique(np.concatenate([order[:1], order[-1:],
                                     rng.choice(a.B, size=sample - 2, replace=False)]))
    err = check(lib, a, seqs=pick)
    print(f"config {config} L={L}: sampled {len(pick)} sequences, max abs err {err:.3e}")


def test_custom_scale_and_permuted_pool(lib):
    rng = np.random.default_rng(77)
    a = W.make_attention(rng, 5, 8, 32, 8, 128, prefix_range=(100, 1500), pool_factor=3.0)
    check(lib, a, sm_scale=0.05)


def test_bad_page_ids_and_lengths_are_flagged_not_faulted(lib):
    import torch
    rng = np.random.default_rng(3)
    a = W.make_attention(rng, 4, 4, 32, 8, 128, prefix_range=(50, 300))
    pt = a.page_table.copy()
    pt[1, 0] = a.pool_pages + 5          # outside the pool
    pt[2, 1] = -7
    run_gpu(lib, a, page_table=pt)
    assert lib.bdlm_device_error() & lib.BDLM_DEVERR_PAGE
    pl = a.prefix_lens.copy()
    pl[3] = pt.shape[1] * 16 + 100       # longer than the page table
    pl[0] = -5
    run_gpu(lib, a, prefix_lens=pl)
    assert lib.bdlm_device_error() & lib.BDLM_DEVERR_LENGTH
    # the library still works afterwards
    check(lib, a)


@pytest.mark.parametrize("L", [32, 16, 64])
def test_rows_on_m_rescale_after_a_sharp_key(lib, L):
    """More than 32 query rows per KV head (query rows on the UMMA M side).  One key in the
    third 128-token tile is planted as 3x a query of its KV head, so that row's max rises
    far above the first tiles' and the kernel must rescale the row's output before the next
    PV product; every other row keeps the lazily kept max.  At L = 64 (256 rows per KV head:
    two 128-row sub-groups) a second key in the fourth tile does the same for a row of the
    second sub-group."""
    rng = np.random.default_rng(515)
    B, Hq, Hkv = 2, 32, 8
    G = Hq // Hkv
    a = W.make_attention(rng, B, L, Hq, Hkv, 128, prefix_range=(600, 900))
    plants = [(3, 300)] + ([(50, 420)] if L == 64 else [])   # (query position, first token)
    for b in range(B):
        for i, t0 in plants:
            for g in (1, 6):
                t = t0 + 7 * g                               # a prefix token in tile t0 // 128
                r = a.page_table_ref[b, t // 16]
                qf = W.bf16_bits_to_f32(a.q[b, i, g * G + 1])
                a.k_ref[r, t % 16, g] = W.f32_to_bf16_bits(3.0 * qf)
    check(lib, a)


@pytest.mark.parametrize("Hq,lens", [
    # 256 query rows per KV head (two sub-groups): KV 126977 is cut into 32 even splits of 4096
    # tokens, the last of which holds only the chunk's last token
    (32, [126913]),
    # 128 rows (one sub-group): KV 70657 / 70684, 24 splits of 3072, the last holding 1 / 28
    # tokens of the chunk
    (16, [70593, 70620]),
])
def test_prefill_chunk_across_a_split_boundary(lib, Hq, lens):
    """Block prefill whose chunk straddles a KV split boundary: the queries of the chunk's first
    blocks see no key of the last split (their partial is empty: max -inf, sum 0) and the
    merge must ignore it."""
    import torch
    from gpu_util import host
    rng = np.random.default_rng(2048 + Hq)
    B, L, Hkv, n = len(lens), 4, 8, 64
    lens = np.array(lens)
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
    ref, k_ref, _ = oracle.prefill_attention(q, kn, vn, a.k_ref, a.v_ref, a.page_table_ref,
                                             a.prefix_lens, L, Hq, Hkv, 128)
    assert np.array_equal(host(kp.view(torch.int16)).view(np.uint16), k_ref)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    assert excess.max() <= 0, f"max excess {excess.max()}"
    assert lib.bdlm_device_error() == 0


@pytest.mark.parametrize("B,L,Hq,Hkv,prefix", [
    (3, 40, 32, 8, (0, 700)),      # 160 rows: sub-group 1 holds 32 of them
    (2, 16, 32, 2, (100, 900)),    # 16 query heads per KV head
    (3, 12, 16, 1, (0, 600)),      # 192 rows, one KV head
    (3, 33, 16, 2, (0, 500)),      # 264 rows: row groups of 256 and 8
    (2, 64, 32, 8, (2040, 4200)),  # KV splits, ragged last tiles
    (40, 64, 32, 8, (0, 1500)),    # enough items for whole sequences, longest first
    (40, 64, 32, 8, (1984, 1984)),  # whole sequences, every one of the longest length taken
    (3, 50, 24, 8, (0, 700)),      # 3 query heads per KV head: 150 rows
])
def test_256_row_groups(lib, B, L, Hq, Hkv, prefix):
    """129-256 query rows per KV head (two 128-row sub-groups sharing each K/V stage): ragged
    row counts, row groups of 256 and fewer, splits with ragged last tiles, whole sequences,
    and an odd number of query heads per KV head."""
    rng = np.random.default_rng(B * 7 + L * 131 + Hq)
    a = W.make_attention(rng, B, L, Hq, Hkv, 128, prefix_range=prefix)
    check(lib, a)

