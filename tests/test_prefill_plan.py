"""kv_prefill's host plan (kv_prefill_plan, the same function kv_prefill calls), on the CPU.

For every small state and chunk: the head, the direct-sealed groups and the rest tile the chunk
[N0, N1) exactly; the groups sealed from the journal were appended first (by earlier calls or
the head); the head never overflows the ring; the newest T positions lie in the rest (so the
exact tail is written); and the sealed end after the call is the one the plain route reaches:
appends of journal-sized pieces, each followed by seal(keep) (SJ-KVaRN §2.1: staged positions,
full groups older than the newest keep committed in a batch). Refusals: past max_ctx, or more
unsealed positions than the ring holds.
"""

import pytest

from quantized_kv_cache_gb300 import _lib, configs

G = 128


def plain_route(N0, S0, n, keep, R):
    """Sealed end after appending n positions in pieces that fit the ring, sealing after each."""
    N, S = N0, S0
    left = n
    while left:
        room = R - (max(N, 128) - S)
        assert room > 0
        c = min(left, room)
        N += c
        left -= c
        S += G * configs.groups_to_seal(N, S, keep)
    return S


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_plan_tiles_the_chunk_and_matches_the_plain_route(lib):
    checked = 0
    for R in (256, 384, 640):
        T = 64
        for keep in (T, 128, 200, R - 128):
            for S0 in range(128, 128 + 4 * G, G):
                starts = [0, 37, 127, 128] if S0 == 128 else []
                starts += list(range(max(S0, 128), S0 + R + 1, 29))
                for N0 in starts:
                    if max(N0, 128) - S0 > R:                  # not a reachable state
                        continue
                    for n in (1, 5, 40, 127, 128, 129, 300, R, 3 * R + 71):
                        max_ctx = N0 + n + (0 if n == 300 else 5)
                        N1 = N0 + n
                        lim = N1 - keep - S0
                        if max(N1, 128) - (S0 + (lim // G * G if lim >= G else 0)) > R:
                            with pytest.raises(_lib.KVQError) as e:          # refused, nothing planned
                                _lib.kv_prefill_plan(N0, S0, n, keep, R, max_ctx)
                            assert e.value.code == _lib.ENOSPC
                            continue
                        r = _lib.kv_prefill_plan(N0, S0, n, keep, R, max_ctx)
                        head, jseal, direct, rest = (r[0], r[1]), (r[2], r[3]), (r[4], r[5]), (r[6], r[7])
                        S1 = direct[1]
                        cover = list(range(*head)) + list(range(*direct)) + list(range(*rest))
                        assert sorted(cover) == list(range(N0, N1)), (R, keep, S0, N0, n, r)
                        assert len(cover) == n                                  # disjoint
                        assert jseal[0] == S0                                   # appended before sealed:
                        assert jseal[1] == jseal[0] or jseal[1] <= max(N0, head[1])
                        assert direct[0] == jseal[1] and (direct[1] - direct[0]) % G == 0
                        assert max(head[1], 128) - S0 <= R                      # the head fits the ring
                        assert max(N1, 128) - S1 <= R                           # so does what stays unsealed
                        assert all(p >= rest[0] for p in range(max(N1 - T, 128, N0), N1))
                        if keep + G - 1 <= R:   # the plain route can run: its ring never fills
                            assert S1 == plain_route(N0, S0, n, keep, R), (R, keep, S0, N0, n, r)
                        checked += 1
    assert checked > 2000


def test_plan_refusals(lib):
    # past max_ctx
    with pytest.raises(_lib.KVQError) as e:
        _lib.kv_prefill_plan(1000, 128, 100, 128, 512, 1099)
    assert e.value.code == _lib.ENOSPC
    # keep so large that the unsealed rest overflows the ring
    with pytest.raises(_lib.KVQError) as e:
        _lib.kv_prefill_plan(0, 128, 4 * 512, 2 * 512, 512, 1 << 20)
    assert e.value.code == _lib.ENOSPC
    with pytest.raises(_lib.KVQError) as e:
        _lib.kv_prefill_plan(0, 128, 0, 128, 512, 1 << 20)
    assert e.value.code == 1
    # a sealed end off the group grid (the library only ever holds 128 + 128 k)
    for bad in (129, 200, 255, 127):
        with pytest.raises(_lib.KVQError) as e:
            _lib.kv_prefill_plan(1000, bad, 100, 128, 1024, 1 << 20)
        assert e.value.code == 1
    # the whole context in one call: everything older than keep sealed straight from the input
    r = _lib.kv_prefill_plan(0, 128, 131072, 1024, 5248, 1 << 20)
    assert r[:2] == [0, 128] and r[2:4] == [128, 128] and r[4:6] == [128, 130048] and r[6:] == [130048, 131072]
