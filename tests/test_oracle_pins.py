"""The oracle against its pins (CPU only)."""
import pytest

from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(orc, pin):
    pin(orc)


def test_oracle_rejects_table_outside_cache(orc):
    from workloads import make_dense_case
    case, _, _ = make_dense_case(lengths=[9], num_q_heads=2, num_kv_heads=1, head_dim=8,
                                 block_size=4, seed=1)
    case.block_tables[0, 1] = case.key_cache.shape[0]
    with pytest.raises(ValueError):
        orc.attention(case.query, case.key_cache, case.value_cache, case.block_tables,
                      case.seq_lens, 0.5)


def test_oracle_rejects_length_beyond_table(orc):
    from workloads import make_dense_case
    case, _, _ = make_dense_case(lengths=[9], num_q_heads=2, num_kv_heads=1, head_dim=8,
                                 block_size=4, seed=1)
    case.seq_lens[0] = 4 * case.block_tables.shape[1] + 1
    with pytest.raises(ValueError):
        orc.attention(case.query, case.key_cache, case.value_cache, case.block_tables,
                      case.seq_lens, 0.5)


def test_partition_count_golden(orc):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "partition_counts.txt")
    rows = [line.split() for line in open(path) if line.strip() and not line.startswith("#")]
    for L, P, used, page in rows:
        assert orc.num_partitions(int(L), int(P)) == int(used)
        # the page's figure is the floor; the last partition is partial
        assert int(L) // int(P) == int(page) and int(L) % int(P) > 0


def test_tiny_golden_fixture(orc):
    """Regression fixture written by tests/golden/make_golden.py (oracle only)."""
    import json
    import os
    import numpy as np
    doc = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_decode.json")))
    q = np.array(doc["query_bits"], dtype=np.uint16)
    k = np.array(doc["key_cache_bits"], dtype=np.uint16)
    v = np.array(doc["value_cache_bits"], dtype=np.uint16)
    bt = np.array(doc["block_tables"], dtype=np.int32)
    sl = np.array(doc["seq_lens"], dtype=np.int32)
    out = orc.attention(q, k, v, bt, sl, doc["scale"], dtype="f16")
    assert np.abs(out - np.array(doc["out"])).max() <= 1e-13
    tmp, es, ml = orc.partials(q, k, v, bt, sl, doc["scale"], doc["partition_size"], dtype="f16")
    assert np.allclose(es, np.array(doc["exp_sums"]), rtol=1e-13, atol=0, equal_nan=True)
    assert np.allclose(ml, np.array(doc["max_logits"]), rtol=1e-13, atol=1e-15, equal_nan=True)


def test_tiny_prefill_golden_fixture(orc):
    """Regression fixture written by tests/golden/make_golden.py (oracle only)."""
    import json
    import os
    import numpy as np
    doc = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_prefill.json")))
    u16 = lambda k: np.array(doc[k], dtype=np.uint16)
    out = orc.prefill(u16("query_bits"), u16("key_cache_bits"), u16("value_cache_bits"),
                      np.array(doc["block_tables"], dtype=np.int32),
                      np.array(doc["seq_lens"], dtype=np.int32),
                      np.array(doc["q_start"], dtype=np.int32), doc["scale"], dtype="bf16")
    assert np.abs(out - np.array(doc["out"])).max() <= 1e-13


def test_tiny_moe_golden_fixture(orc):
    """Regression fixture written by tests/golden/make_golden.py (oracle only)."""
    import json
    import os
    import numpy as np
    import torch
    doc = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_moe.json")))
    logits = torch.from_numpy(np.array(doc["logits_bits"], dtype=np.uint16).view(np.int16)) \
        .view(torch.bfloat16)
    hidden = np.array(doc["hidden_bits"], dtype=np.uint16)
    w, ids = orc.topk_softmax(logits, 4, True)
    assert (ids == np.array(doc["ids"])).all()
    assert np.abs(w - np.array(doc["weights"])).max() <= 1e-15
    sp, off, pos = orc.moe_sort(ids, 32)
    assert (sp == np.array(doc["sorted_pairs"])).all() and (off == np.array(doc["offsets"])).all()
    assert (pos == np.array(doc["pair_pos"])).all()
    y = orc.moe_gather(hidden, sp, 4)
    out = orc.moe_scatter(y, pos, w, 4, dtype="bf16")
    assert np.abs(out - np.array(doc["out"])).max() <= 1e-13
