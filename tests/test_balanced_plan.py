"""The balanced plan (pd_balanced_plan, host only): it must cover every
(sequence, kv head) key range exactly once, in order, give every CTA the same
cost (its pages plus 40 keys' worth for each extra piece) to within the
page rounding at its two ends and a piece's cost at each, and describe itself
consistently. CPU only."""
import numpy as np
import pytest

from paged_kv_split_gb300 import inputs


def _plan(lens, Hq=32, Hkv=8, D=128, bs=16, mbs=None, W=0, dt=0, sms=152):
    from paged_kv_split_gb300 import binding as B
    lens = np.asarray(lens, np.int32)
    mbs = mbs or max(1, int(-(-lens.max() // bs)) if len(lens) else 1)
    return B.pd_balanced_plan(lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                              max_blocks_per_seq=mbs, sliding_window=W, kv_dtype=dt,
                              num_sms=sms), mbs


def _decode(plan, B, Hkv):
    w = plan.words
    nc, npc = int(w[1]), int(w[2])
    assert w[0] == 0x50444231 and (nc, npc) == (plan.num_ctas, plan.num_pieces)
    cta = w[8:8 + nc + 1]
    poff = (8 + nc + 1 + 3) // 4 * 4
    pieces = w[poff:poff + 4 * npc].reshape(npc, 4)
    seg = w[poff + 4 * npc:poff + 4 * npc + 2 * B * Hkv].reshape(B * Hkv, 2)
    return cta, pieces, seg


def _key_range(L, W):
    lo = L - W if (W > 0 and L > W) else 0
    return lo, L


def _pages(t0, t1, bs):
    return (t1 - 1) // bs - t0 // bs + 1


CASES = [
    ("llama8b", inputs.llama8b().seq_lens, dict()),
    ("ragged_small", [1, 15, 16, 17, 0, 100, 33], dict(Hq=8, Hkv=2, D=64)),
    ("window", [16384] * 3 + [100, 4097], dict(Hq=8, Hkv=4, D=256, W=4096)),
    ("one_long", [32768], dict(bs=32)),
    ("many_short", inputs.uniform_int(77, 1100, 1, 60), dict(Hq=4, Hkv=2, D=64)),
    ("all_empty", [0, 0, 0], dict()),
    ("fewer_pages_than_ctas", [20, 5], dict(Hq=4, Hkv=1, D=64)),
]


@pytest.mark.parametrize("name,lens,kw", CASES, ids=[c[0] for c in CASES])
def test_plan_covers_every_range_once_and_balances(name, lens, kw):
    lens = np.asarray(lens, np.int32)
    Hkv, bs, W = kw.get("Hkv", 8), kw.get("bs", 16), kw.get("W", 0)
    G = kw.get("Hq", 32) // Hkv
    D = kw.get("D", 128)
    plan, mbs = _plan(lens, **kw)
    B = len(lens)
    cta, pieces, seg = _decode(plan, B, Hkv)
    nc, npc = plan.num_ctas, plan.num_pieces
    total_pages = sum(_pages(*_key_range(int(L), W), bs) * Hkv for L in lens if L > 0)
    if total_pages == 0:
        assert nc == 0 and npc == 0
        assert (seg[:, 1] == 0).all()
        return
    assert 1 <= nc <= min(total_pages, 152 * 4)
    assert cta[0] == 0 and cta[-1] == npc and (np.diff(cta) >= 1).all()
    # every (sequence, kv head): its pieces are consecutive and tile its key range in order
    for b in range(B):
        lo, hi = _key_range(int(lens[b]), W)
        for g in range(Hkv):
            first, count = seg[b * Hkv + g]
            if hi <= lo:
                assert count == 0
                continue
            ps = pieces[first:first + count]
            assert (ps[:, 0] == b * Hkv + g).all()
            assert ps[0, 1] == lo and ps[-1, 2] == hi
            assert (ps[1:, 1] == ps[:-1, 2]).all() and (ps[:, 2] > ps[:, 1]).all()
            assert (ps[:, 1][1:] % bs == 0).all()  # cuts fall on page boundaries
            assert ((ps[:, 3] & 1) == (1 if count == 1 else 0)).all()
    assert seg[:, 1].sum() == npc
    # balance: the cost of a CTA's share (pages, plus 40 / bs pages for every
    # piece after its first) is the same for every CTA up to the rounding at
    # the share's two ends (a page, and a piece's cost at each end)
    per_cta = np.array([sum(_pages(int(p[1]), int(p[2]), bs)
                            for p in pieces[cta[c]:cta[c + 1]]) for c in range(nc)])
    assert per_cta.sum() == total_pages
    kappa = 40 / bs
    cost = per_cta + kappa * (np.diff(cta) - 1)
    assert cost.max() - cost.min() <= 2 + 2 * kappa
    assert plan.workspace_bytes >= npc * G * (D + 2) * 4


def test_plan_rejects_bad_arguments():
    from paged_kv_split_gb300 import binding as B
    with pytest.raises(B.PdError):
        B.pd_balanced_plan(np.array([10], np.int32), num_q_heads=6, num_kv_heads=4, head_dim=128,
                           block_size=16, max_blocks_per_seq=4, num_sms=152)
    with pytest.raises(B.PdError):
        B.pd_balanced_plan(np.array([10], np.int32), num_q_heads=8, num_kv_heads=8, head_dim=96,
                           block_size=16, max_blocks_per_seq=4, num_sms=152)


def test_schedule_preference_follows_length_spread():
    from paged_kv_split_gb300 import binding as B

    def prefer(lens, **kw):
        args = dict(num_q_heads=32, num_kv_heads=8, max_blocks_per_seq=1024, block_size=32,
                    head_dim=128, num_sms=152)
        args.update(kw)
        return B.pd_prefer_balanced(np.asarray(lens, np.int32), **args)
    # equal lengths: the split schedule already gives every CTA the same work
    assert not prefer([32768] * 4)
    # very unequal lengths: the balanced plan
    assert prefer(inputs.lognormal_lengths(5, 64, np.log(2048.0), 1.0, 512, 16384),
                  num_q_heads=64, max_blocks_per_seq=1024, block_size=16)
    assert not prefer([])
    with pytest.raises(B.PdError):
        prefer([10], num_q_heads=6, num_kv_heads=4)
