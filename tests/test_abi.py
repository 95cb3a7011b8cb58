"""The C-ABI library loads, exports every function include/bdlm.h declares, and rejects
bad arguments on the host before touching a GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bdlm.h")


@pytest.fixture(scope="module")
def so():
    from block_diffusion_gb300 import build, load_library
    build.build()  # incremental: recompiles only sources newer than their objects
    return load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bdlm_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_round():
    names = declared_functions()
    for n in ("bdlm_block_attention", "bdlm_lm_head", "bdlm_confidence_commit",
              "bdlm_apply_commit", "bdlm_status_string", "bdlm_device_error", "bdlm_release"):
        assert n in names


def test_library_exports_every_declared_symbol(so):
    for name in declared_functions():
        assert hasattr(so, name), name
    import block_diffusion_gb300 as bd
    assert set(bd.EXPORTS) <= set(declared_functions())


def test_status_strings(so):
    import block_diffusion_gb300 as bd
    assert bd.status_string(0) == "ok"
    assert "invalid" in bd.status_string(-1)


def test_host_side_validation_rejects_bad_arguments(so):
    import block_diffusion_gb300 as bd
    P = 0x1000  # never dereferenced: every call below fails validation first
    bad = [
        lambda: so.bdlm_confidence_commit(P, P, 1, 0, 10, 0.5, 1.0, P, P, P, None),   # L = 0
        lambda: so.bdlm_confidence_commit(P, P, 1, 65, 10, 0.5, 1.0, P, P, P, None),  # L > 64
        lambda: so.bdlm_confidence_commit(P, P, 1, 4, 10, 0.5, 0.0, P, P, P, None),   # T = 0
        lambda: so.bdlm_confidence_commit(P, P, 1, 4, 10, 1.5, 1.0, P, P, P, None),   # tau > 1
        lambda: so.bdlm_confidence_commit(None, P, 1, 4, 10, 0.5, 1.0, P, P, P, None),  # null
        lambda: so.bdlm_lm_head(P, P, P, 4, 8, 12, 64, P, None),      # H % 8 != 0
        lambda: so.bdlm_lm_head(P, P, P, 9, 8, 16, 64, P, None),      # n_active > n_rows
        lambda: so.bdlm_lm_head(P + 2, P, P, 4, 8, 16, 64, P, None),  # misaligned hidden
        lambda: so.bdlm_apply_commit(P, P, -1, None),
        # fused LM head + commit: hidden, w, mask, den, B, L, H, V, rule, k, tau, T, tok, conf,
        # entropy, commit, logits, stream
        lambda: so.bdlm_lm_head_commit(P, P, P, None, 2, 65, 16, 64, 0, 1, 0.5, 1.0, P, P, None,
                                       P, None, None),                         # L > 64
        lambda: so.bdlm_lm_head_commit(P, P, P, None, 2, 4, 12, 64, 0, 1, 0.5, 1.0, P, P, None,
                                       P, None, None),                         # H % 8 != 0
        lambda: so.bdlm_lm_head_commit(P, P, P, None, 2, 4, 16, 60, 0, 1, 0.5, 1.0, P, P, None,
                                       P, None, None),                         # V % 8 != 0
        lambda: so.bdlm_lm_head_commit(P, P, P, None, 2, 4, 16, 64, 5, 1, 0.5, 1.0, P, P, None,
                                       P, None, None),                         # unknown rule
        lambda: so.bdlm_lm_head_commit(P, P, P, None, 2, 4, 16, 64, 1, 0, 0.5, 1.0, P, P, None,
                                       P, None, None),                         # k = 0
        lambda: so.bdlm_lm_head_commit(P, P, P, None, 2, 4, 16, 64, 0, 1, 0.5, -1.0, P, P, None,
                                       P, None, None),                         # T < 0
        lambda: so.bdlm_lm_head_commit(P, P, P, None, 2, 4, 16, 64, 4, 1, -0.5, 1.0, P, P, None,
                                       P, None, None),                         # budget < 0
        lambda: so.bdlm_lm_head_commit(P, P, None, None, 2, 4, 16, 64, 0, 1, 0.5, 1.0, P, P,
                                       None, P, None, None),                   # null mask
        lambda: so.bdlm_lm_head_commit(P, P, P, None, 2, 4, 16, 64, 0, 1, 0.5, 1.0, P, P, None,
                                       P, P + 8, None),                        # misaligned logits
        # commit with a rule: logits, mask, B, L, V, rule, k, tau, T, tok, conf, entropy, commit
        lambda: so.bdlm_confidence_commit_rule(P, P, 1, 4, 10, 5, 1, 0.5, 1.0, P, P, None, P,
                                               None),                          # unknown rule
        lambda: so.bdlm_confidence_commit_rule(P, P, 1, 4, 10, 4, 1, -1.0, 1.0, P, P, None, P,
                                               None),                          # budget < 0
        lambda: so.bdlm_confidence_commit_rule(P, P, 1, 4, 10, 4, 1, float("inf"), 1.0, P, P,
                                               None, P, None),                 # budget inf
        lambda: so.bdlm_confidence_commit_rule(P, P, 1, 4, 10, 0, 1, 1.5, 1.0, P, P, None, P,
                                               None),                          # tau > 1
        lambda: so.bdlm_confidence_commit_rule(P, P, 1, 4, 10, 1, 0, 0.5, 1.0, P, P, None, P,
                                               None),                          # k = 0
    ]
    for f in bad:
        assert f() == bd.BDLM_ERR_INVALID
    d = bd.attn_desc(2, 4, 32, 8, 64, 10, 100)          # D != 128
    assert so.bdlm_block_attention(ctypes.byref(d), P, P, P, P, P, 4, P, None) == -1
    d = bd.attn_desc(2, 4, 30, 8, 128, 10, 100)         # Hq % Hkv != 0
    assert so.bdlm_block_attention(ctypes.byref(d), P, P, P, P, P, 4, P, None) == -1
    d = bd.attn_desc(2, 4, 32, 8, 128, 10, 100)
    assert so.bdlm_block_attention(ctypes.byref(d), P, P, P, P, P, 5, P, None) == -1  # L mismatch
    d = bd.attn_desc(2, 4, 32, 8, 128, 10, 100, page_size=32)
    assert so.bdlm_block_attention(ctypes.byref(d), P, P, P, P, P, 4, P, None) == -1
    # empty problems are no-ops that succeed without a device
    assert so.bdlm_confidence_commit(P, P, 0, 4, 10, 0.5, 1.0, P, P, P, None) == 0
    assert so.bdlm_lm_head(P, P, P, 0, 8, 16, 64, P, None) == 0
    assert so.bdlm_apply_commit(P, P, 0, None) == 0
    assert so.bdlm_lm_head_commit(P, P, P, None, 0, 4, 16, 64, 0, 1, 0.5, 1.0, P, P, None, P,
                                  None, None) == 0
    assert so.bdlm_confidence_commit_rule(P, P, 0, 4, 10, 4, 1, 2.0, 1.0, P, P, None, P,
                                          None) == 0


def test_selftest_wait_limit_is_validated(so):
    assert so.bdlm_selftest_wait_timeout(0, None) == -1
    assert so.bdlm_selftest_wait_timeout(2000001, None) == -1
