"""The oracle still reproduces the stored align cases (guards later edits)."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "align_cases.json")


def test_align_golden_cases():
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    assert len(cases) >= 6
    for c in cases:
        ids = np.array(c["ids"], dtype=np.int32).reshape(-1)
        s, e, npp, cnt = oracle.moe_align_block_size(ids, c["E"], c["block"])
        assert s.tolist() == c["sorted_ids"], c["name"]
        assert e.tolist() == c["expert_ids"], c["name"]
        assert npp == c["num_tokens_post_padded"], c["name"]
        assert cnt.tolist() == c["expert_counts"], c["name"]
