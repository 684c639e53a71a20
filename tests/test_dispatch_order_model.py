"""CPU check of the forward kernel's CTA dispatch order (no GPU).

A Python statement of the integer arithmetic of the launcher's group choice
(attn_api.cu, launch) and the kernel's cta_coords (attn_fwd_kernel.cuh): the
1-D launch index is mapped to the logical (x, y, z) of a CTA, with x the query
block counted from the last, y the query head and z the batch or sequence.
Checked here: the map is a bijection onto the logical grid; inside a group
every CTA of a larger x (a shorter causal block) starts after every CTA of a
smaller x; groups are contiguous ranges of (y, z) pairs of near-equal size.
A list-scheduling model of the GPU (one CTA per SM, each SM taking the next
CTA in launch order) shows the grouped order removing the causal tail of the
plain 3-D order on the batched and packed workloads.  The backward launch
(attn_bwd_kernel.cuh, bwd_cta_coords) uses the same map with x the key block
(block 0, read by every query block, is the longest); the model shows the same
for its CTAs, whose lengths are the query steps they walk."""

import heapq

import pytest

from exact_tiled_attention_19_gb300 import workloads as W

SMS = 152


def group_sizes(gx, gy, gz, num_sms=SMS):
    """(q, rem): groups of near-equal size, q + 1 pairs in the first rem
    groups and q in the rest, with about G pairs each, G the smallest power
    of two with G * gx >= num_sms (or all pairs)."""
    pairs = gy * gz
    G = 1
    while G * gx < num_sms and G < pairs:
        G *= 2
    groups = (pairs + G - 1) // G
    return pairs // groups, pairs % groups


def cta_coords(lin, gx, gy, gz, q, rem):
    big = rem * (q + 1)
    pi = lin // gx
    if pi < big:
        size = q + 1
        first = pi // size * size
    else:
        size = q
        first = big + (pi - big) // q * q
    r = lin - first * gx
    x = r // size
    pair = first + (r - x * size)
    z = pair // gy
    return x, pair - z * gy, z, first


@pytest.mark.parametrize("gx,gy,gz", [(1, 1, 1), (16, 16, 4), (32, 32, 2), (59, 16, 16), (3, 7, 5), (2, 1000, 1),
                                      (1, 152, 1), (5, 3, 1), (9, 11, 13), (4, 64, 1)])
def test_cta_coords_is_a_bijection_longest_first_within_groups(gx, gy, gz):
    q, rem = group_sizes(gx, gy, gz)
    assert q >= 1 and 0 <= rem
    seen = set()
    last_x_of_group = {}
    group_pairs = {}
    for lin in range(gx * gy * gz):
        x, y, z, g = cta_coords(lin, gx, gy, gz, q, rem)
        assert lin < 2 ** 31 and g * gx <= lin
        assert 0 <= x < gx and 0 <= y < gy and 0 <= z < gz
        assert (x, y, z) not in seen
        seen.add((x, y, z))
        # launch order inside a group: x never decreases
        assert x >= last_x_of_group.get(g, 0)
        last_x_of_group[g] = x
        group_pairs.setdefault(g, set()).add(y + gy * z)
    assert len(seen) == gx * gy * gz
    sizes = [len(v) for v in group_pairs.values()]
    assert max(sizes) - min(sizes) <= 1
    # groups are contiguous pair ranges, in launch order
    starts = [min(group_pairs[g]) for g in sorted(group_pairs)]
    assert starts == sorted(starts)
    for g in group_pairs:
        ps = sorted(group_pairs[g])
        assert ps == list(range(ps[0], ps[-1] + 1))


def _causal_ctas(w, order):
    """(launch order) list of per-CTA tile counts for a square causal workload
    with two 128-row sub-tiles per CTA: block t streams tiles 0 .. 2t+1."""
    lens = [lq for lq, _ in w.lengths()]
    gx = max((L + 255) // 256 for L in lens)
    gy, gz = w.Hq, len(lens)

    def work(x, y, z):
        L = lens[z]
        t = gx - 1 - x
        nb, kt = (L + 255) // 256, (L + 127) // 128
        return min(2 * t + 2, kt) if t < nb else 0

    if order == "grid":
        return [work(x, y, z) for z in range(gz) for y in range(gy) for x in range(gx)]
    q, rem = group_sizes(gx, gy, gz)
    return [work(*cta_coords(lin, gx, gy, gz, q, rem)[:3]) for lin in range(gx * gy * gz)]


def _makespan(tiles, fixed=2.0):
    heap = [0.0] * SMS
    for n in tiles:
        t = heapq.heappop(heap)
        heapq.heappush(heap, t + (fixed + n if n > 0 else 0.2))
    return max(heap)


@pytest.mark.parametrize("name,gain", [("b4_h16_n4096_d128_bf16", 0.10), ("gqa_b2_h32x8_n8192_d128_bf16", 0.05),
                                       ("varlen16_h16_d128_bf16", 0.01)])
def test_grouped_order_removes_the_causal_tail(name, gain):
    w = W.WORKLOADS[name]
    grid, grouped = _makespan(_causal_ctas(w, "grid")), _makespan(_causal_ctas(w, "grouped"))
    ideal = sum(2.0 + n for n in _causal_ctas(w, "grid") if n > 0) / SMS
    assert grouped <= grid * (1 - gain)
    assert grouped <= ideal * 1.03


def div_magic_of(d):
    """The launcher's (m, k): l = ceil(log2 d), k = 31 + l, m = ceil(2^k / d)."""
    l = 0
    while (1 << l) < d:
        l += 1
    k = 31 + l
    return -(-(1 << k) // d), k


@pytest.mark.parametrize("d", [1, 2, 3, 5, 7, 16, 59, 127, 152, 1000, 4097, 65535, 65536, 2 ** 20 + 1,
                               2 ** 30 - 1, 2 ** 30 + 1, 2 ** 31 - 1])
def test_multiply_shift_division_is_exact_below_2_31(d):
    import random
    m, k = div_magic_of(d)
    assert 0 < m < 2 ** 32 and k <= 62
    rng = random.Random(d)
    ns = {0, 1, d - 1, d, d + 1, 2 ** 31 - 1, 2 ** 31 - 2} | {rng.randrange(2 ** 31) for _ in range(20000)}
    ns |= {j * d + r for j in (1, 2, 1000, (2 ** 31 - 1) // d) for r in (0, d - 1) if j * d + r < 2 ** 31}
    for n in ns:
        if 0 <= n < 2 ** 31:
            assert (n * m) >> k == n // d, (n, d)


def _backward_ctas(B, Hq, Hkv, N, order):
    """(launch order) per-CTA step counts of the causal backward launch: key
    block kb walks the query blocks kb .. N/128 - 1 of each of the group's
    Hq / Hkv query heads."""
    gx, gy, gz = (N + 127) // 128, Hkv, B

    def work(x, y, z):
        return (gx - x) * (Hq // Hkv)

    if order == "grid":
        return [work(x, y, z) for z in range(gz) for y in range(gy) for x in range(gx)]
    q, rem = group_sizes(gx, gy, gz)
    return [work(*cta_coords(lin, gx, gy, gz, q, rem)[:3]) for lin in range(gx * gy * gz)]


@pytest.mark.parametrize("shape,gain", [((4, 16, 16, 4096), 0.02), ((2, 32, 8, 8192), 0.05)])
def test_grouped_order_shortens_the_backward_tail(shape, gain):
    grid, grouped = _makespan(_backward_ctas(*shape, "grid")), _makespan(_backward_ctas(*shape, "grouped"))
    ideal = sum(2.0 + n for n in _backward_ctas(*shape, "grid")) / SMS
    assert grouped <= grid * (1 - gain)
    assert grouped <= ideal * 1.05
