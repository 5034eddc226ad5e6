"""Host logic of the expert cache (the GPU as an expert cache whose misses are
fetched: vLLM-Moet page, "2-bit experts on vLLM v0.24.0", "Experts beyond
VRAM"; the cache holds the most-used experts: Tandem-vLLM page, "How it
works").  moe_expert_cache_plan is the cache's planning step, a host-only
function of the library: which slot each missing expert takes, and which
expert it replaces (eviction by routing counts).  No GPU is needed."""
import numpy as np
import pytest

import bit_vq_routed_gb300 as bv

plan = bv.moe_expert_cache_plan


def state(E, S):
    return np.full(S, -1, np.int32), np.zeros(E, np.uint64), np.zeros(E, np.uint64)


def test_slot_bytes_of_the_decode_shapes():
    # VQ2: codes I*H/4 (x2) + H*I/4, scales 2 bytes per 128 inputs; FP4: H*I/2 per
    # matrix + one byte per 32 inputs (each buffer padded to 256 bytes: all are
    # multiples already at these shapes)
    H, I = 4096, 2048
    assert bv.moe_expert_cache_slot_bytes(H, I, bv.MOE_FMT_VQ2) == 3 * (H * I // 4) + 3 * (H * I // 128 * 2)
    assert bv.moe_expert_cache_slot_bytes(H, I, bv.MOE_FMT_VQ2) == 6_684_672
    assert bv.moe_expert_cache_slot_bytes(H, I, bv.MOE_FMT_FP4) == 13_369_344
    assert bv.moe_expert_cache_slot_bytes(H, I, 7) == 0
    assert bv.moe_expert_cache_slot_bytes(0, I, bv.MOE_FMT_VQ2) == 0
    # a buffer that is not a multiple of 256 bytes is padded: H=256, I=128:
    # scales of gate/up = 128*2*2 = 512, of down = 256*1*2 = 512; codes 8192 each
    assert bv.moe_expert_cache_slot_bytes(256, 128, bv.MOE_FMT_VQ2) == 3 * 8192 + 3 * 512
    # FP4 at H=256, I=128: down scales = 256 * 4 = 1024, gate/up scales 128 * 8 = 1024
    assert bv.moe_expert_cache_slot_bytes(256, 128, bv.MOE_FMT_FP4) == 3 * 16384 + 3 * 1024


def test_slot_layout_of_the_binding_matches_the_library():
    from bit_vq_routed_gb300.layer import slot_layout
    for H, I in ((4096, 2048), (256, 128), (512, 384)):
        for fmt in (bv.MOE_FMT_VQ2, bv.MOE_FMT_FP4):
            lay, total = slot_layout(H, I, fmt)
            assert total == bv.moe_expert_cache_slot_bytes(H, I, fmt)
            assert all(o % 256 == 0 for o, _ in lay)
            assert all(lay[b][0] + lay[b][1] <= lay[b + 1][0] for b in range(5))


def test_free_slots_fill_in_order_and_hits_repeats_do_not():
    se, cnt, last = state(10, 4)
    fill, ev, left = plan(10, se, cnt, last, 1, [7, 3, 7, 9])
    assert list(fill) == [0, 1, -1, 2] and list(ev) == [-1, -1, -1, -1] and left == 0
    assert list(se) == [7, 3, 9, -1]
    assert cnt[7] == 1 and cnt[3] == 1 and cnt[9] == 1 and cnt.sum() == 3  # once per step, repeats too
    assert last[7] == 1 and last[0] == 0
    fill, ev, left = plan(10, se, cnt, last, 2, [3, 9, 1])
    assert list(fill) == [-1, -1, 3] and left == 0
    assert list(se) == [7, 3, 9, 1] and cnt[3] == 2


def test_victim_is_least_routed_then_oldest_then_lowest_id():
    E, S = 16, 3
    se = np.array([4, 5, 6], np.int32)
    cnt = np.zeros(E, np.uint64)
    last = np.zeros(E, np.uint64)
    cnt[[4, 5, 6]] = [5, 2, 2]
    last[[4, 5, 6]] = [3, 2, 1]
    # counts 5, 2, 2: 5 and 6 tie on count; 6 was named longer ago
    fill, ev, _ = plan(E, se, cnt, last, 10, [11])
    assert fill[0] == 2 and ev[0] == 6 and list(se) == [4, 5, 11]
    # now 5 (count 2, step 2) against 11 (count 1, step 10): 11 is the least routed
    fill, ev, _ = plan(E, se, cnt, last, 11, [12])
    assert ev[0] == 11 and fill[0] == 2
    # equal counts and steps: the lower id goes
    se = np.array([9, 8], np.int32)
    cnt = np.zeros(E, np.uint64)
    last = np.zeros(E, np.uint64)
    cnt[[8, 9]] = 1
    last[[8, 9]] = 4
    fill, ev, _ = plan(E, se, cnt, last, 5, [0])
    assert ev[0] == 8 and fill[0] == 1


def test_named_experts_are_never_evicted_and_overflow_is_unplaced():
    E, S = 12, 3
    se = np.array([0, 1, 2], np.int32)
    cnt = np.zeros(E, np.uint64)
    last = np.zeros(E, np.uint64)
    cnt[[0, 1, 2]] = [1, 9, 9]
    last[[0, 1, 2]] = 1
    # the step names 0 (least routed, but named: kept), 5 and 6: 5 replaces one
    # of 1 / 2 (equal counts and steps: the lower id, 1), 6 replaces 2
    fill, ev, left = plan(E, se, cnt, last, 2, [5, 0, 6])
    assert list(ev) == [1, -1, 2] and left == 0
    assert sorted(se.tolist()) == [0, 5, 6]
    # four distinct experts, three slots, all named: the last one finds no slot
    fill, ev, left = plan(E, se, cnt, last, 3, [7, 0, 5, 6])
    assert left == 1 and fill[0] == -1
    assert sorted(se.tolist()) == [0, 5, 6]
    assert cnt[7] == 1  # it was still counted
    # no slots at all: everything unplaced, counts still kept
    se0 = np.zeros(0, np.int32)
    c0, l0 = np.zeros(E, np.uint64), np.zeros(E, np.uint64)
    fill, ev, left = plan(E, se0, c0, l0, 1, [1, 2, 2])
    assert left == 2 and list(fill) == [-1, -1, -1] and c0[2] == 1


def test_bad_arguments_are_rejected_and_nothing_changes():
    E = 8
    se = np.array([1, 2, -1], np.int32)
    cnt = np.zeros(E, np.uint64)
    last = np.zeros(E, np.uint64)
    last[1] = 4
    snap = (se.copy(), cnt.copy(), last.copy())

    def unchanged():
        return np.array_equal(se, snap[0]) and np.array_equal(cnt, snap[1]) and np.array_equal(last, snap[2])

    for bad_req, step in (([8], 5), ([-1], 5), ([3], 4), ([3], 3)):
        with pytest.raises(bv.MoeError) as ei:
            plan(E, se, cnt, last, step, bad_req)
        assert ei.value.status == bv.MOE_ERR_INVALID_ARG and unchanged()
    se2 = np.array([1, 1, -1], np.int32)  # one expert in two slots
    with pytest.raises(bv.MoeError):
        plan(E, se2, cnt, last, 5, [3])
    se3 = np.array([1, 9, -1], np.int32)  # an expert id out of range
    with pytest.raises(bv.MoeError):
        plan(E, se3, cnt, last, 5, [3])
    assert cnt.sum() == 0


def _model_step(E, slots, cnt, last, step, req):
    """The eviction rule as stated, written with Python's sorted(): a second
    formulation to compare the library's loop with."""
    named = []
    for e in req:
        if e not in named:
            named.append(e)
            cnt[e] += 1
            last[e] = step
    fills, left = [], 0
    for e in named:
        if e in slots:
            continue
        free = [s for s, v in enumerate(slots) if v < 0]
        if free:
            s = free[0]
        else:
            cands = [(cnt[v], last[v], v, s) for s, v in enumerate(slots) if last[v] != step]
            if not cands:
                left += 1
                continue
            s = sorted(cands)[0][3]
        fills.append((e, s, slots[s]))
        slots[s] = e
    return fills, left


@pytest.mark.parametrize("S,k", [(4, 2), (10, 8), (24, 8), (7, 3)])
def test_random_steps_follow_the_rule_and_keep_the_invariants(S, k):
    E = 32
    rng = np.random.default_rng(S * 100 + k)
    # Zipf-like popularity so that some experts are hot
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    se, cnt, last = state(E, S)
    m_slots, m_cnt, m_last = [-1] * S, [0] * E, [0] * E
    hits = fills_total = unplaced = 0
    for step in range(1, 200):
        T = int(rng.integers(1, 3))
        req = np.concatenate([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
        resident_before = set(int(v) for v in se if v >= 0)
        fill, ev, left = plan(E, se, cnt, last, step, req)
        mf, ml = _model_step(E, m_slots, m_cnt, m_last, step, req.tolist())
        got = [(int(req[i]), int(fill[i]), int(ev[i])) for i in range(req.size) if fill[i] >= 0]
        assert got == mf and left == ml
        assert se.tolist() == m_slots and cnt.tolist() == m_cnt and last.tolist() == m_last
        # invariants: no expert twice, every placed named expert resident, no
        # named expert evicted, distinct named = hits + fills + unplaced
        held = [int(v) for v in se if v >= 0]
        assert len(held) == len(set(held)) <= S
        named = set(int(e) for e in req)
        assert all(int(e) in held for e in named) or left > 0
        assert not (set(int(v) for v in ev if v >= 0) & named)
        h = len(named & resident_before)
        assert h + len(got) + left == len(named)
        hits += h
        fills_total += len(got)
        unplaced += left
    if S >= 2 * k:
        assert unplaced == 0
    # the hottest expert (id 0) stays resident once the cache is warm
    assert 0 in se.tolist()
    assert hits > 0 and fills_total > 0
