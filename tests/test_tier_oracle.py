"""Pins of the tiered store's policy oracle (oracle/tier.py) against the
formulas of "Colibrì 深度解析" §三 and hand-derived tick sequences."""
from oracle import tier as T


def test_frequency_first_recency_breaks_ties():
    # the page's own example: 256 routes, unused for 300 ticks, outranks 50
    # routes used 5 ticks ago
    assert T.score(256, 0, 300) > T.score(50, 295, 300)
    # a recent access is worth at most 255 points, one count 256
    assert T.recent(1000, 1000) == 255 and T.recent(1000, 700) == 0
    assert T.score(11, 0, 10_000) > T.score(10, 10_000, 10_000)
    # equal heat: the more recent wins
    assert T.score(7, 90, 100) > T.score(7, 80, 100)


def test_promotion_hysteresis_and_saturation():
    assert T.should_promote(5, 0) and not T.should_promote(4, 0)
    assert T.should_promote(130, 100) and not T.should_promote(129, 100)  # 100 + 25 + 4
    m = 2 ** 32 - 1
    assert not T.should_promote(m, m)       # a saturated counter never wraps the threshold
    assert T.should_promote(m, (m - 4) * 4 // 5 - 1)


def test_hand_sequence_one_slot():
    # 4 routed experts, one slot, initially free
    st = T.TierState(4, 0, [-1])
    ups = []
    for _ in range(5):          # expert 0 routed once per tick: heat 1, 2, 3, 4, 5
        ups.append(st.tick([1, 0, 0, 0], max_uploads=4))
    assert st.heat[0] == 5
    assert ups == [[], [], [], [], [(0, 0)]]          # admitted when heat 5 > 0 + 0 + 4
    assert st.owner == [0] and st.slot_of == [0, -1, -1, -1]
    # expert 1 routed three times per tick, expert 0 not at all: heat 0 stays 5
    # (5 - 5 // 8 = 5); heat 1 goes 3, 6, 9 (6 // 8 = 0), then 9 - 1 + 3 = 11,
    # the first value above 5 + 5 // 4 + 4 = 10
    got = [st.tick([0, 3, 0, 0], max_uploads=4) for _ in range(4)]
    assert [st.heat[0], st.heat[1]] == [5, 11]
    assert got == [[], [], [], [(1, 0)]]
    assert st.slot_of == [-1, 0, -1, -1] and st.clock == 9 and st.last == [5, 9, 0, 0]


def test_free_slots_fill_lowest_first_and_shared_stay():
    # 3 routed + 1 shared expert; slots: shared in 0, two free
    st = T.TierState(3, 1, [3, -1, -1])
    for _ in range(4):
        st.tick([2, 2, 0], max_uploads=8)
    # heats 2, 4, 6 -> both pass 4 on the third tick, higher score first
    assert st.owner == [3, 0, 1] or st.owner == [3, 1, 0]
    assert st.slot_of[3] == 0                         # the shared expert never moves
    st2 = T.TierState(3, 1, [3, -1, -1])
    seq = [st2.tick([2, 3, 0], max_uploads=8) for _ in range(3)]
    # heats after ticks: e0 2, 4, 6; e1 3, 6, 9 -> tick 2 admits e1 (6 > 4) to
    # slot 1; tick 3 admits e0 (6 > 4) to slot 2
    assert seq == [[], [(1, 1)], [(0, 2)]]


def test_max_uploads_counts_moves_only():
    st = T.TierState(4, 0, [-1, -1, -1])
    for _ in range(6):
        ups = st.tick([3, 3, 3, 0], max_uploads=2)
    assert sum(o >= 0 for o in st.owner) == 3
    # heats 3 after one tick (none above 4), 6 after two: equal scores, so
    # lower ids first, two moves; the third expert on the next tick
    st = T.TierState(4, 0, [-1, -1, -1])
    assert st.tick([3, 3, 3, 0], max_uploads=2) == []
    assert st.tick([3, 3, 3, 0], max_uploads=2) == [(0, 0), (1, 1)]
    assert st.tick([3, 3, 3, 0], max_uploads=2) == [(2, 2)]
