"""Writes the stored expected values under tests/golden/ by calling only the
oracle package. Re-run after a deliberate change to the oracle's arithmetic:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

# Hand-written routing cases for moe_align_block_size (vLLM PR #12185, note 1):
# decode with many experts, one hot expert, duplicates inside a token, an
# out-of-range id (dropped), and an empty batch.
ALIGN_CASES = [
    dict(name="decode_e256", ids=[[17, 3, 255, 128, 0, 64, 200, 99]], E=256, block=16),
    dict(name="hot_expert", ids=[[2, 2], [2, 5], [2, 0], [1, 2]], E=8, block=16),
    dict(name="dup_in_token", ids=[[4, 4], [4, 1]], E=8, block=32),
    dict(name="bad_id_dropped", ids=[[0, 9], [3, -1], [0, 3]], E=8, block=16),
    dict(name="empty", ids=[], E=8, block=16),
    dict(name="spill_two_blocks", ids=[[1]] * 17 + [[0]], E=2, block=16),
]


def main():
    out = []
    for c in ALIGN_CASES:
        sorted_ids, expert_ids, npp, counts = oracle.moe_align_block_size(
            __import__("numpy").array(c["ids"], dtype="int32").reshape(-1), c["E"], c["block"])
        out.append(dict(c, sorted_ids=sorted_ids.tolist(), expert_ids=expert_ids.tolist(),
                        num_tokens_post_padded=npp, expert_counts=counts.tolist()))
    with open(os.path.join(HERE, "align_cases.json"), "w") as f:
        json.dump(dict(source="written by tests/golden/make_golden.py from the oracle",
                       cases=out), f, indent=1)


if __name__ == "__main__":
    main()
