"""Write tests/golden/oracle_tiny.json from the oracle alone.

The pages print no worked example, so the only stored values are the
oracle's own output on one tiny, fully specified input; they guard the
oracle against unintended changes (the independent pins live in
test_oracle_pins.py).  Run from the repository root:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402

from tiny_case import tiny_inputs  # noqa: E402


def main():
    args, kw = tiny_inputs()
    out, a = oracle.pre_attention(*args, **kw)
    doc = {
        "about": "oracle output of the tiny case in tiny_case.py (bf16 bit patterns as int16)",
        "source": "written by tests/golden/make_golden.py, which calls only oracle/",
        "workspace_bits": a.view(torch.int16).flatten().tolist(),
        "out_shape": list(out.shape),
        "out_bits": out.view(torch.int16).flatten().tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json")
    with open(path, "w") as f:
        json.dump(doc, f)
    print("wrote", path)


if __name__ == "__main__":
    main()
