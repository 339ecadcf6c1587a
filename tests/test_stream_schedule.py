"""The token-balanced decode schedule's arithmetic, restated on the CPU (no GPU needed).

The decode kernel's walk (`StreamWalk` in `tq_decode_common.cuh`: which units and token
ranges each CTA takes) and the combine kernel's record ranges (`stream_unit_ctas`) are
warp-collective device code.  This is a scalar restatement of the same arithmetic, fuzzed
over length sets, CTA counts and per-unit start allowances, checking what the kernels rely
on: every token of every unit is taken by exactly one CTA, segments start on 8-token
boundaries and hold at least one token, the combine finds exactly the CTAs that wrote a
unit's records, and the record slots (CTA + unit) are distinct and inside the workspace's
SMs + units records."""
import numpy as np
import pytest

MIN_W = 256


def unit_ext(ovh, n):
    return ovh + ((n + 7) // 8) * 8 if n > 0 else 0


def extent(lens, hkv, n_cta, ovh):
    tot = sum(unit_ext(ovh, n) for n in lens) * hkv
    w = -(-tot // n_cta)
    return tot, max(((w + 7) // 8) * 8, MIN_W)


def walk(lens, hkv, n_cta, ovh, c):
    """Segments (b, h, a0, a1) of CTA c, in the order the kernel takes them."""
    tot, W = extent(lens, hkv, n_cta, ovh)
    P = c * W
    if P >= tot:
        return []
    end = min(P + W, tot)
    base = 0
    for b, n in enumerate(lens):
        sp = unit_ext(ovh, n) * hkv
        if base + sp > P:
            break
        base += sp
    else:
        raise AssertionError("position past the total")
    ln, ext = lens[b], unit_ext(ovh, lens[b])
    h = (P - base) // ext
    us = base + h * ext
    a0 = max(P - (us + ovh), 0)
    valid = end > us + ovh
    segs = []
    while valid:
        segs.append((b, h, a0, min(ln, end - (us + ovh))))
        ue = us + ext
        if end <= ue:
            break
        us, a0 = ue, 0
        h += 1
        if h == hkv:
            h = 0
            b += 1
            while b < len(lens) and lens[b] == 0:
                b += 1
            if b >= len(lens):
                break
            ln, ext = lens[b], unit_ext(ovh, lens[b])
        valid = end > us + ovh
    return segs


def unit_ctas(lens, hkv, n_cta, ovh, b, h):
    """(first CTA, count) whose positions cover unit (b, h): the combine's record range."""
    _, W = extent(lens, hkv, n_cta, ovh)
    before = sum(unit_ext(ovh, n) for n in lens[:b])
    ext = unit_ext(ovh, lens[b])
    us = before * hkv + h * ext
    first = (us + ovh) // W
    return first, ((us + ext - 1) // W - first + 1) if ext > 0 else 0


def check(lens, hkv, n_cta, ovh):
    B = len(lens)
    covered = {(b, h): [] for b in range(B) for h in range(hkv)}
    ctas = {(b, h): [] for b in range(B) for h in range(hkv)}
    slots = set()
    for c in range(n_cta):
        for (b, h, a0, a1) in walk(lens, hkv, n_cta, ovh, c):
            assert a0 % 8 == 0 and a1 > a0 and a1 <= lens[b], (c, b, h, a0, a1)
            covered[(b, h)].append((a0, a1))
            ctas[(b, h)].append(c)
            slot = c + b * hkv + h
            assert slot not in slots
            assert slot < n_cta + B * hkv  # inside the SMs + units records of the workspace
            slots.add(slot)
    for (b, h), rs in covered.items():
        rs.sort()
        pos = 0
        for a0, a1 in rs:
            assert a0 == pos, (b, h, rs)
            pos = a1
        assert pos == lens[b], (b, h, rs, lens[b])
        first, count = unit_ctas(lens, hkv, n_cta, ovh, b, h)
        assert ctas[(b, h)] == list(range(first, first + count)), (b, h, ctas[(b, h)], first, count)


@pytest.mark.parametrize("ovh", [64, 320, 384, 768, 1536])
def test_walk_covers_every_token_once(ovh):
    rng = np.random.default_rng(ovh)
    for trial in range(150):
        B = int(rng.integers(1, 70))
        hkv = int(rng.choice([1, 2, 4, 8]))
        kind = trial % 3
        if kind == 0:    # ragged, with empty and tiny sequences
            lens = rng.integers(0, 3000, size=B)
            lens[rng.random(B) < 0.2] = 0
            lens[rng.random(B) < 0.2] = rng.integers(1, 10)
        elif kind == 1:  # equal lengths (whole waves or not)
            lens = np.full(B, int(rng.integers(1, 20000)))
        else:            # a few long sequences among short ones
            lens = rng.integers(1, 64, size=B)
            lens[rng.integers(0, B)] = int(rng.integers(8000, 40000))
        lens = [int(x) for x in lens]
        if sum(lens) == 0:
            lens[0] = 1
        n_cta = int(rng.choice([1, 7, 148, 152]))
        check(lens, hkv, n_cta, ovh)


def test_walk_edge_shapes():
    # the decode tests' shapes (several segments per CTA, 1-9 tokens, >32 sequences)
    check([0, 1, 7, 8, 9, 128] + [100] * 58, 8, 152, 768)
    check([0, 1, 7, 8, 9, 256] + [64] * 27, 2, 152, 384)
    check([16384] * 32, 8, 152, 320)                       # 256 equal units on 152 CTAs
    check([1] * 200, 1, 152, 768)                          # more sequences than CTAs
    check([5], 1, 152, 64)                                 # one token-light unit
