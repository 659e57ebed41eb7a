"""The measured SPS(B) table's host logic (no GPU): the verify_len spread of a
budget, the table built from sampled step times, and the stored table."""

import json
import os

import numpy as np
import pytest

from speculative_decoding_verification_padding_gb300 import sps


@pytest.mark.parametrize("B", [0, 256, 300, 511, 512, 900, 1280, 5000])
def test_verify_lens_spread_a_budget(B):
    gamma = np.full(256, 4, dtype=np.int32)
    L = sps.verify_lens(B, gamma)
    assert (L >= 0).all() and (L <= gamma).all()
    assert L.sum() == int(np.clip(B - 256, 0, gamma.sum()))
    assert L.max() - L.min() <= 1                         # as even as possible
    assert (np.diff(L) <= 0).all()                        # lower requests first


def test_verify_lens_respect_per_request_limits():
    gamma = np.array([0, 3, 1, 5], dtype=np.int32)
    L = sps.verify_lens(4 + 7, gamma)
    assert list(L) == [0, 3, 1, 3]


def test_table_is_non_increasing_and_matches_the_samples():
    pts = [256, 512, 768, 1024, 1280]
    secs = [1.0e-3, 1.3e-3, 1.25e-3, 1.9e-3, 2.4e-3]      # one noisy dip
    t = sps.table_from_samples(pts, secs, 1280)
    assert t.shape == (1281,) and t.dtype == np.float32
    assert (np.diff(t.astype(np.float64)) <= 0).all()
    assert t[256] == np.float32(1 / 1.0e-3)
    assert t[1280] == np.float32(1 / 2.4e-3)
    assert t[0] == t[256]                                 # constant before the first sample


@pytest.mark.skipif(not os.path.exists(sps.MEASURED), reason="no measured table stored")
def test_stored_table_is_well_formed():
    d = json.load(open(sps.MEASURED))
    t = np.asarray(d["sps"], dtype=np.float64)
    assert len(t) == 1281 and (t > 0).all() and (np.diff(t) <= 0).all()
    assert len(d["points"]) == len(d["seconds"]) >= 3
