"""Speculation bookkeeping of the C library (host code) against the oracle.

These entry points do no device work, so they run here without a GPU; the
comparison is exact (integers), on seeded random rounds.
"""

from __future__ import annotations

import numpy as np
import pytest

from oracle import mtp_oracle as O


@pytest.fixture(scope="module")
def M():
    import mtp_speculative_draft_gb300 as M
    return M


def _as_dict(s, kmax):
    return {"rounds": s.rounds, "drafted": s.drafted, "accepted": s.accepted,
            "accept_hist": list(s.accept_hist)[:kmax + 1],
            "depth_drafted": list(s.depth_drafted)[:kmax],
            "depth_accepted": list(s.depth_accepted)[:kmax],
            "draft_ns": s.draft_ns, "verify_ns": s.verify_ns}


def test_stats_match_oracle(M):
    rng = np.random.default_rng(11)
    s, ref = M.SpecStats(), O.spec_stats_new()
    kmax = 0
    for _ in range(500):
        k = int(rng.integers(0, 17))
        a = int(rng.integers(0, k + 1))
        dns, vns = int(rng.integers(0, 10 ** 6)), int(rng.integers(0, 10 ** 7))
        M.mtp_spec_note_round(s, k, a, dns, vns)
        O.spec_note_round(ref, k, a, dns, vns)
        kmax = max(kmax, k)
    got = _as_dict(s, kmax)
    assert got == ref
    assert M.mtp_spec_tokens_per_round(s) == O.spec_tokens_per_round(ref)
    # bins past the deepest round stay zero
    assert not any(list(s.accept_hist)[kmax + 1:]) and not any(list(s.depth_drafted)[kmax:])


def test_accept_matches_oracle(M):
    rng = np.random.default_rng(12)
    for _ in range(300):
        k = int(rng.integers(0, 17))
        drafts = rng.integers(0, 50, size=k)
        verify = rng.integers(0, 50, size=k + 1)
        cut = int(rng.integers(0, k + 1))   # plant a matching prefix of random length
        verify[:cut] = drafts[:cut]
        assert M.mtp_spec_accept(drafts, verify) == O.spec_accept(drafts, verify)


def test_rewind_matches_oracle(M):
    rng = np.random.default_rng(13)
    for _ in range(100):
        lens = rng.integers(0, 5000, size=int(rng.integers(0, 8))).tolist()
        keep = int(rng.integers(0, 5000))
        assert M.mtp_spec_rewind(lens, keep) == O.spec_rewind(lens, keep)


def test_bad_rounds_are_rejected_unchanged(M):
    from mtp_speculative_draft_gb300._lib import MtpError, load
    s = M.SpecStats()
    M.mtp_spec_note_round(s, 2, 1)
    before = _as_dict(s, 16)
    for k, a in [(3, 4), (17, 0), (-1, 0), (2, -1)]:
        with pytest.raises(MtpError):
            M.mtp_spec_note_round(s, k, a)
    assert _as_dict(s, 16) == before
    assert load().mtp_spec_accept(None, None, 0) == 0
    assert load().mtp_spec_accept(None, None, 3) == -1
    assert load().mtp_spec_accept(None, None, 17) == -1
    with pytest.raises(MtpError):
        M.mtp_spec_rewind([1, 2], -1)


def test_mimo_plan_commit_match_oracle(M):
    """Per-layer round state over random rounds, gaps and stale states."""
    rng = np.random.default_rng(14)
    for trial in range(40):
        layers = int(rng.integers(1, 5))
        c = [M.MimoLayerState() for _ in range(layers)]
        r = [O.mimo_layer_state_new() for _ in range(layers)]
        t, lo = int(rng.integers(0, 30)), 0
        for _ in range(30):
            if rng.random() < 0.1:                     # the history restarts part-way
                lo = int(rng.integers(max(0, t - 5), t + 1))
            hist_end = t + 1 if rng.random() < 0.9 else t  # sometimes lacks t
            ids_len = t + 2 if rng.random() < 0.95 else t + 1
            for l in range(layers):
                n, start = M.mtp_mimo_plan_layer(c[l], l, t, lo, hist_end, ids_len)
                ref = O.mimo_plan_layer(r[l], l, t, lo, hist_end, ids_len)
                assert (n > 0) == (ref is not None)
                if ref is not None:
                    assert start == ref and n == t + 1 - ref
                    M.mtp_mimo_commit_layer(c[l], l, t, ids_len)
                    O.mimo_commit_layer(r[l], l, t, ids_len)
                assert (c[l].committed, c[l].base, c[l].kv_len) == (r[l]["committed"], r[l]["base"],
                                                                    r[l]["kv_len"])
            t += int(rng.integers(1, 5))
