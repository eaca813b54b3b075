"""The split forward grid's schedule (no GPU): the arithmetic attn_fwd_kernel uses when a
non-causal dense grid has fewer query blocks than SMs, restated here.

The units (block k, key tile j), block-major, are cut into G ranges [floor(c U / G),
floor((c + 1) U / G)), one per CTA c (U = blocks x key tiles). CTA c walks the blocks its
range meets, from floor(u_lo / nk) while block * nk < u_hi, each over the key tiles inside its
range; the CTA holding unit u is floor(((u + 1) G - 1) / U); a block's parts are the CTAs from
the one holding its first unit to the one holding its last, and part (k, c) writes slot k + c.
Checked: every unit is computed exactly once, each block's parts are the CTAs that visit it,
the slots of all parts are distinct and below blocks + 256 (the workspace's slot count), and
the part counts agree with what the merging CTA expects."""
import pytest


def schedule(n_items, nk, G):
    U = n_items * nk
    seen = {}
    for c in range(G):
        u_lo, u_hi = c * U // G, (c + 1) * U // G
        item = u_lo // nk
        while item >= 0:
            base = item * nk
            j_lo, j_hi = max(u_lo, base) - base, min(u_hi, base + nk) - base
            assert 0 <= j_lo < j_hi <= nk
            seen.setdefault(item, []).append((c, j_lo, j_hi))
            item = item + 1 if (item + 1) * nk < u_hi else -1
    return U, seen


def cta_of(u, U, G):
    return ((u + 1) * G - 1) // U


@pytest.mark.parametrize("n_items,nk,G", [(128, 32, 152), (1, 512, 152), (3, 7, 21),
                                          (151, 2, 152), (100, 3, 152), (5, 64, 152),
                                          (2, 2, 4), (64, 33, 152)])
def test_split_schedule(n_items, nk, G):
    U, seen = schedule(n_items, nk, G)
    assert sorted(seen) == list(range(n_items))
    slots = set()
    for k, parts in seen.items():
        cover = sorted((j_lo, j_hi) for _, j_lo, j_hi in parts)
        assert cover[0][0] == 0 and cover[-1][1] == nk
        assert all(a[1] == b[0] for a, b in zip(cover, cover[1:]))  # no gap, no overlap
        c_first, c_last = cta_of(k * nk, U, G), cta_of((k + 1) * nk - 1, U, G)
        assert [c for c, _, _ in parts] == list(range(c_first, c_last + 1))
        for c, _, _ in parts:
            assert (k + c) not in slots
            slots.add(k + c)
    assert max(slots) < n_items + 256
    # the CTA that holds unit u is the one whose range contains it
    for u in range(U):
        c = cta_of(u, U, G)
        assert c * U // G <= u < (c + 1) * U // G


def split_ctas(n_items, nk, sms):
    """The host's split grid size (attn_fwd): a whole number of ranges per block, at most one
    per SM; with more than half as many blocks as SMs (only when forced) one range per SM."""
    per_block = min(nk, sms // n_items)
    return n_items * per_block if per_block >= 2 else min(n_items * nk, sms)


@pytest.mark.parametrize("n_items,nk", [(32, 32), (50, 9), (1, 512), (76, 2), (7, 3), (64, 33),
                                        (3, 2)])
def test_split_grid_size_gives_each_cta_one_block(n_items, nk):
    G = split_ctas(n_items, nk, 152)
    assert n_items < G <= 152 and G % n_items == 0
    U, seen = schedule(n_items, nk, G)
    visits = {}
    for k, parts in seen.items():
        assert len(parts) == G // n_items  # every block has the same number of parts
        for c, j_lo, j_hi in parts:
            visits[c] = visits.get(c, 0) + 1
    assert sorted(visits) == list(range(G)) and set(visits.values()) == {1}
