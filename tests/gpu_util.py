"""Helpers shared by the GPU parity tests: host arrays to device tensors and comparisons."""
import numpy as np


def dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def host(t):
    return t.cpu().numpy()


def bf16_tensor(bits):
    import torch
    return dev(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def bf16_to_np_f64(t):
    import torch
    return t.float().cpu().numpy().astype(np.float64)


def compare_commit(ref, tok, conf, commit, mask, rtol_conf=1e-5):
    """Tokens exact and confidences within rtol on masked rows; commit masks exact except
    in blocks holding a position the oracle flags as near the threshold or a near-tie of
    the fallback (counted, not failed).  Returns (n_near_blocks_differing, n_near_total)."""
    m = mask.astype(bool)
    assert np.array_equal(tok[m], ref.tok[m]), "argmax tokens differ"
    assert np.all(tok[~m] == -1)
    assert np.all(np.isneginf(conf[~m]))
    rel = np.abs(conf[m].astype(np.float64) - ref.conf[m]) / np.abs(ref.conf[m])
    assert rel.max(initial=0.0) <= rtol_conf, f"confidence rel err {rel.max()}"
    differ = np.any(commit != ref.commit, axis=1)
    near_blk = np.any(ref.near != 0, axis=1)
    bad = differ & ~near_blk
    assert not bad.any(), f"commit differs in blocks {np.nonzero(bad)[0][:10]}"
    return int((differ & near_blk).sum()), int(near_blk.sum())


def compare_entropy(ref, ent, mask):
    """Entropies of masked positions within 1e-4 + 1e-5 H of the oracle's (float32
    accumulation over the vocabulary); +inf at unmasked positions.  Returns the largest
    absolute error."""
    m = mask.astype(bool)
    err = np.abs(ent[m].astype(np.float64) - ref.ent[m])
    tol = 1e-4 + 1e-5 * np.abs(ref.ent[m])
    assert np.all(err <= tol), f"entropy error {err.max()} (tol {tol[np.argmax(err)]})"
    assert np.all(np.isposinf(ent[~m]))
    return float(err.max(initial=0.0))
