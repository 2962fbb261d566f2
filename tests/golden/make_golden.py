"""Writes tiny_decode.json, tiny_prefill.json and tiny_moe.json: small cases and
the oracle's fp64 outputs (decode; prefix prefill; MoE router, sort, gather and
scatter-back).

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
from workloads import make_dense_case, make_dense_prefill_case, make_moe_case  # noqa: E402


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
    here = os.path.dirname(os.path.abspath(__file__))
    with open(os.path.join(here, "tiny_decode.json"), "w") as f:
        json.dump(doc, f)

    pc, _, _ = make_dense_prefill_case(ctx_lens=[5, 0], q_lens=[6, 3], num_q_heads=4,
                                       num_kv_heads=2, head_dim=8, block_size=4,
                                       dtype=torch.bfloat16, seed=20261201)
    pout = oracle.prefill(pc.query, pc.case.key_cache, pc.case.value_cache,
                          pc.case.block_tables, pc.case.seq_lens, pc.q_start, scale)
    pdoc = {
        "about": "bf16 prefix prefill, 2 seqs (context 5 + chunk 6, context 0 + chunk 3), "
                 "Hq=4, Hkv=2, d=8, bs=4; outputs written by oracle/ via make_golden.py",
        "dtype": "bf16", "scale": scale,
        "query_bits": bits(pc.query), "key_cache_bits": bits(pc.case.key_cache),
        "value_cache_bits": bits(pc.case.value_cache),
        "block_tables": pc.case.block_tables.tolist(), "seq_lens": pc.case.seq_lens.tolist(),
        "q_start": pc.q_start.tolist(), "out": pout.tolist(),
    }
    with open(os.path.join(here, "tiny_prefill.json"), "w") as f:
        json.dump(pdoc, f)

    mc = make_moe_case(num_tokens=6, num_experts=32, topk=4, hidden_size=8, seed=20261202)
    w, ids = oracle.topk_softmax(mc.logits, 4, True)
    sp, off, pos = oracle.moe_sort(ids, 32)
    y = oracle.moe_gather(mc.hidden, sp, 4)
    mout = oracle.moe_scatter(torch.from_numpy(y.view(np.int16)).view(torch.bfloat16), pos, w, 4)
    mdoc = {
        "about": "MoE routing, 6 tokens, top-4 of 32 experts (renormalised), hidden 8, bf16; "
                 "outputs written by oracle/ via make_golden.py",
        "logits_bits": bits(mc.logits), "hidden_bits": bits(mc.hidden),
        "weights": w.tolist(), "ids": ids.tolist(), "sorted_pairs": sp.tolist(),
        "offsets": off.tolist(), "pair_pos": pos.tolist(), "out": mout.tolist(),
    }
    with open(os.path.join(here, "tiny_moe.json"), "w") as f:
        json.dump(mdoc, f)


if __name__ == "__main__":
    main()
