"""The work counts bench.py divides by, checked against brute force on small
cases (CPU only): decode's algorithmic bytes and prefill's attention FLOPs."""
import numpy as np

import bench
from paged_kv_split_gb300 import inputs


def test_decode_algorithmic_bytes_brute_force():
    case = inputs.make_case("ab", [17, 40, 0, 100], 8, 2, 64, 16, seed=5, sliding_window=30)
    ab = bench.algorithmic_bytes(case, 0)
    keys = pages = 0
    for L in case.seq_lens:
        seen = [j for j in range(int(L)) if int(L) - 1 - j < 30]
        keys += len(seen)
        pages += len({j // 16 for j in seen})
    kv = keys * case.num_kv_heads * 2 * case.head_dim * 2
    qo = 2 * case.num_seqs * case.num_q_heads * case.head_dim * 2
    assert ab["keys"] == keys
    assert ab["total"] == kv + qo + 4 * pages


def test_prefill_flops_brute_force():
    for w in (0, 7):
        case = inputs.make_prefill_case("pf", [17, 40, 9], [5, 40, 1], 8, 2, 64, 16, seed=6,
                                        sliding_window=w)
        total = 0
        for b, (L, ql) in enumerate(zip(case.seq_lens, case.extra["q_lens"])):
            for i in range(int(ql)):
                p = int(L) - int(ql) + i
                total += sum(1 for j in range(p + 1) if w == 0 or p - j < w)
        assert bench.prefill_flops(case) == 4.0 * case.head_dim * case.num_q_heads * total
        # a sample of rows counts only those rows
        assert bench.prefill_flops(case, [(1, 38, 40)]) == \
            4.0 * case.head_dim * case.num_q_heads * sum(
                min(38 + k + 1, w) if w else 38 + k + 1 for k in range(2))
