"""bdlm_confidence_commit_noalloc against bdlm_confidence_commit, through the C-ABI.

The no-allocation entry point serves callers that cannot let the library call cudaMalloc
(an engine that owns all of the GPU's memory, a loop that cannot absorb an allocation's
implicit synchronisation).  It must give the same tokens, confidences (within the 1e-5
relative tolerance used elsewhere) and commit masks as the allocating entry point, on two
calls in a row that reuse its fixed scratch array, and agree with the fp64 oracle; its device
error word (read through bdlm_device_error) stays clear.  This file is collected last so that
a run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import compare_commit

pytestmark = pytest.mark.gpu


def _noalloc(lib_so):
    f = lib_so.bdlm_confidence_commit_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, I, I, I, F, F, P, P, P, P]
    f.restype = I
    return f


def _inputs(seed, B, L, V):
    rng = np.random.default_rng(seed)
    mask = W.make_mask_fixed_fraction(rng, B, L, rng.uniform(0.2, 1.0, size=B))
    logits = W.make_logits(rng, B * L, V, peak_height=(4.0, 20.0))
    return W.poison_unmasked_rows(logits, mask), mask


def test_noalloc_matches_allocating_entry_point_twice(lib):
    import torch
    so = lib.load_library()
    noalloc = _noalloc(so)
    s = torch.cuda.current_stream().cuda_stream
    for seed, (B, L, V) in [(1, (128, 4, 151936)), (2, (16, 64, 151936 + 8))]:
        logits, mask = _inputs(seed, B, L, V)
        lg = torch.from_numpy(logits.view(np.int16)).cuda().view(torch.bfloat16)
        mk = torch.from_numpy(mask).cuda()
        outs = []
        for use_noalloc in (False, True):
            tok = torch.full((B, L), 7, dtype=torch.int32, device="cuda")
            conf = torch.zeros((B, L), dtype=torch.float32, device="cuda")
            com = torch.full((B, L), 9, dtype=torch.uint8, device="cuda")
            if use_noalloc:
                rc = noalloc(lg.data_ptr(), mk.data_ptr(), B, L, V, 0.5, 1.0, tok.data_ptr(),
                             conf.data_ptr(), com.data_ptr(), s)
                assert rc == 0, lib.status_string(rc)
            else:
                lib.bdlm_confidence_commit(lg, mk, B, L, V, 0.5, 1.0, tok, conf, com)
            torch.cuda.synchronize()
            outs.append((tok.cpu().numpy(), conf.cpu().numpy(), com.cpu().numpy()))
        (t0, c0, m0), (t1, c1, m1) = outs
        m = mask == 1
        assert np.array_equal(t0, t1)
        rel = np.abs(c1[m].astype(np.float64) - c0[m]) / np.abs(c0[m])
        assert rel.max() <= 1e-5
        assert np.all(np.isneginf(c1[~m]))
        assert np.array_equal(m0, m1)
        # and the oracle, on the same bf16 logits
        ref = oracle.confidence_commit(logits, mask, 0.5, 1.0)
        compare_commit(ref, t1, c1, m1, mask)
    # no bounded wait gave up in either entry point (bdlm_device_error reads both words)
    assert lib.bdlm_device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    so = lib.load_library()
    noalloc = _noalloc(so)
    P = 0x1000  # never dereferenced: the size check comes first
    assert noalloc(P, P, 2049, 1, 100, 0.5, 1.0, P, P, P, None) == lib.BDLM_ERR_UNSUPPORTED
    assert noalloc(P, P, 4, 4, 262145, 0.5, 1.0, P, P, P, None) == lib.BDLM_ERR_UNSUPPORTED
