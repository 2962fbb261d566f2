"""Writes tiny_decode.json: a small decode case and the oracle's fp64 outputs.

Run from the repository root: ``python tests/golden/make_golden.py``.  It calls
only ``oracle/`` and ``workloads/`` (the seeded input generator); the stored
inputs are bit patterns, so the fixture does not depend on the generator
reproducing the same numbers on another machine.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from workloads import make_dense_case  # noqa: E402


def main():
    case, _, _ = make_dense_case(lengths=[7, 13], num_q_heads=4, num_kv_heads=2, head_dim=8,
                                 block_size=4, dtype=torch.float16, seed=20261200)
    scale = float(np.float32(1 / np.sqrt(8)))
    out = oracle.attention(case.query, case.key_cache, case.value_cache, case.block_tables,
                           case.seq_lens, scale)
    tmp, es, ml = oracle.partials(case.query, case.key_cache, case.value_cache,
                                  case.block_tables, case.seq_lens, scale, 8)

    def bits(t):
        return t.view(torch.int16).numpy().view(np.uint16).tolist()

    doc = {
        "about": "fp16 paged decode, 2 seqs (L=7,13), Hq=4, Hkv=2, d=8, bs=4; "
                 "outputs written by oracle/ via tests/golden/make_golden.py",
        "dtype": "f16", "scale": scale, "partition_size": 8,
        "query_bits": bits(case.query), "key_cache_bits": bits(case.key_cache),
        "value_cache_bits": bits(case.value_cache),
        "block_tables": case.block_tables.tolist(), "seq_lens": case.seq_lens.tolist(),
        "out": out.tolist(), "exp_sums": es.tolist(), "max_logits": ml.tolist(),
        "tmp_out": tmp.tolist(),
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_decode.json"),
              "w") as f:
        json.dump(doc, f)


if __name__ == "__main__":
    main()
