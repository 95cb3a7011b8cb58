"""The seeded input generators: determinism, shapes, page tables, masks, poison."""
import numpy as np

import workloads as W


def test_bf16_rounding_is_rne():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, np.nan, 3.0e38], np.float32)
    b = W.f32_to_bf16_bits(x)
    assert b[0] == 0x3F80 and b[1] == 0x3F80 and b[2] == 0x3F82 and b[4] == 0x7FC0
    assert W.bf16_bits_to_f32(b[3]) == -2.5


def test_attention_inputs_deterministic_and_consistent():
    a = W.make_attention(np.random.default_rng(1), 5, 4, 8, 4, 32, prefix_range=(3, 70), P=16)
    b = W.make_attention(np.random.default_rng(1), 5, 4, 8, 4, 32, prefix_range=(3, 70), P=16)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.k_ref, b.k_ref)
    assert np.array_equal(a.page_table, b.page_table)
    kv = a.kv_lens
    for s in range(5):
        n = (kv[s] + 15) // 16
        assert np.all(a.page_table[s, :n] >= 0) and np.all(a.page_table[s, n:] == -1)
        assert np.array_equal(a.ref_page_ids[a.page_table_ref[s, :n]], a.page_table[s, :n])
        used = kv[s] - (n - 1) * 16
        last = a.k_ref[a.page_table_ref[s, n - 1]]
        assert np.all(last[used:] == 0x7FC0)
        assert not np.any(last[:used] == 0x7FC0)
    # pool ids are distinct
    ids = a.page_table[a.page_table >= 0]
    assert len(np.unique(ids)) == len(ids) and ids.max() < a.pool_pages


def test_masks_and_logits():
    rng = np.random.default_rng(2)
    m = W.make_mask_fixed_fraction(rng, 50, 64, rng.uniform(0.1, 0.9, 50))
    assert np.all(m.sum(1) >= 1)
    ci = W.commit_inputs(1, np.random.default_rng(W.seed_for(1)), 1, 4, 1000)
    assert list(ci.mask[0]) == [0, 1, 0, 1]
    assert np.all(ci.logits[0] == 0x7FC0) and not np.any(ci.logits[1] == 0x7FC0)
    ci4 = W.commit_inputs(4, np.random.default_rng(W.seed_for(4)), 3, 64, 2000)
    assert ci4.logits.shape == (192, 2000)
