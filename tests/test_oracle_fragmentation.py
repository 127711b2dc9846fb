"""Pins for the fragmentation arithmetic against the numbers the pages print
(fixture: tests/golden/fragmentation_pages.json, each entry cited)."""

import json
import os

import numpy as np

from oracle.fragmentation import contiguous_waste, paged_slots, paged_waste
from workloads import lognormal_lengths

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "fragmentation_pages.json")))


def test_contiguous_example_from_the_page():
    g = GOLDEN["contiguous_example"]
    _, unused = contiguous_waste([g["tokens_used"]], g["max_seq_len"])
    assert unused.tolist() == [g["unused_slots"]]


def test_worst_case_paged_slack_is_block_size_minus_one():
    g = GOLDEN["paged_worst_case"]
    bs = g["block_size"]
    lens = np.arange(1, 10 * bs + 1)
    _, slack = paged_waste(lens, bs)
    assert slack.max() == g["max_slack_tokens"]
    assert (slack[lens % bs == 1] == g["max_slack_tokens"]).all()
    assert (slack[lens % bs == 0] == 0).all()
    assert (paged_slots(lens, bs) >= lens).all()


def test_realistic_lengths_paged_below_bound_and_contiguous_in_range():
    """13B-shaped lengths (log-normal, median 350, clipped to [16, 2048]) under
    paging at the default block size waste less than the page's bound, while a
    2048-slot contiguous reservation wastes within the page's 60-80% band."""
    rng = np.random.default_rng(2)
    lens = lognormal_lengths(rng, 4096, 350.0, 0.75, 16, 2048)
    bs = GOLDEN["default_block_size"]["block_size"]
    frac_paged, _ = paged_waste(lens, bs)
    frac_contig, _ = contiguous_waste(lens, 2048)
    assert frac_paged < GOLDEN["paged_waste_bound"]["max_fraction"]
    lo, hi = GOLDEN["contiguous_waste_range"]["low"], GOLDEN["contiguous_waste_range"]["high"]
    assert lo <= frac_contig <= hi


def test_paged_waste_is_exact_on_a_hand_case():
    frac, slack = paged_waste([1, 16, 17], 16)
    assert slack.tolist() == [15, 0, 15]
    assert abs(frac - 30 / 64) < 1e-15
