"""The oracle still reproduces its stored output on the tiny golden case."""
import json
import os
import sys

import torch

import oracle

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
sys.path.insert(0, GOLD)
from tiny_case import tiny_inputs  # noqa: E402


def test_oracle_matches_stored_tiny_case():
    with open(os.path.join(GOLD, "oracle_tiny.json")) as f:
        doc = json.load(f)
    args, kw = tiny_inputs()
    out, a = oracle.pre_attention(*args, **kw)
    assert list(out.shape) == doc["out_shape"]
    assert out.view(torch.int16).flatten().tolist() == doc["out_bits"]
    assert a.view(torch.int16).flatten().tolist() == doc["workspace_bits"]
    # the guarded token (index -1) is zero in the workspace and in every output
    assert all(v == 0 for v in a[2].view(torch.int16).tolist())
