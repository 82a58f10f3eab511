"""The host padding plan against the token counts the pages print (CPU only)."""
import json
import os

import pytest

from video_dit_attention_gb300.padding import plan_token_padding

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "padding_plan.json")


def test_pages_padding_numbers():
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert plan_token_padding(c["seq_len"], c["multiple"], c["shards"]) == c["padded"], c["cite"]


def test_rejects_bad_plans():
    for args in [(-1, 128, 1), (10, 0, 1), (10, 128, 0)]:
        with pytest.raises(ValueError):
            plan_token_padding(*args)


def test_exact_multiples_are_unchanged():
    assert plan_token_padding(4736) == 4736 and plan_token_padding(0) == 0 and plan_token_padding(1) == 128
