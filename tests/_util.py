"""Helpers shared by the tests: seeded inputs and the parity bars."""
import numpy as np

import oracle
import synth


def q4k_weights(seed, tid, N, K, sigma=0.02):
    """(f32 weights, oracle-packed Q4_K bytes)."""
    w = synth.normal(seed, tid, (N, K), sigma)
    return w, oracle.q4k_pack(w)


def check_f32(got, ref, a, what, rel=1e-5, abs_=1e-6, cos_min=0.999999):
    """GEMV / decode bar: |err| <= rel * sum|w x| + abs per output, and cosine >= cos_min."""
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    a = np.asarray(a, np.float64).ravel()
    err = np.abs(got - ref)
    bound = rel * a + abs_
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, "%s: %d/%d outputs out of bound; worst idx %d err %.3g bound %.3g" % (
        what, bad.size, got.size, bad[np.argmax(err[bad] / bound[bad])], err[bad].max(), bound[bad].min())
    if np.linalg.norm(ref) > 0 and got.size > 1:
        cos = float(got @ ref / (np.linalg.norm(got) * np.linalg.norm(ref)))
        assert cos >= cos_min, "%s: cosine %.9f < %g" % (what, cos, cos_min)
    return float((err / bound).max()) if got.size else 0.0
