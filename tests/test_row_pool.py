"""The backward's row pool, host side: the layout the planner gives the pool
kernel (per-CTA heads, then a queue of segments of consecutive rows) must cover
every row exactly once, whatever M and the grid size. Host-only arithmetic of the
library (no GPU): rmsnorm_row_pool_layout / rmsnorm_row_pool_segment."""
import pytest

from rmsnorm_fwd_bwd_gb300 import binding as B

CASES = [(65536, 456), (65536, 608), (32768, 456), (16384, 152), (16384, 304), (8192, 456), (8192, 608),
         (4096, 608), (4096, 456), (2432, 608), (2431, 608), (1000, 456), (7, 3), (12, 3), (13, 3),
         (100003, 456), (1 << 20, 608), (999999, 152)]


def segments(M, G):
    head, nseg = B.rmsnorm_row_pool_layout(M, G)
    return head, [B.rmsnorm_row_pool_segment(M, G, k) for k in range(nseg)]


@pytest.mark.parametrize("M,G", CASES)
def test_heads_and_segments_cover_every_row_once(M, G):
    head, segs = segments(M, G)
    if head == 0:
        assert segs == []
        return
    # heads: CTA b takes rows b + j*G, j < head, i.e. exactly rows [0, G*head)
    assert 1 <= head and G * head < M
    at = G * head
    for first, last in segs:
        assert first == at and last > first
        at = last
    assert at == M


@pytest.mark.parametrize("M,G", CASES)
def test_pool_only_with_four_rows_per_cta(M, G):
    head, segs = segments(M, G)
    assert (head > 0) == (M >= 4 * G and G * head < M)
    if head:
        # most rows stay with their static owner: 90% (92% below 64 rows per CTA), less
        # at most G rows of rounding
        share = 0.90 if M // G >= 64 else 0.92
        assert G * head <= share * M and G * head > share * M - G


@pytest.mark.parametrize("M,G", [c for c in CASES if c[0] >= 4 * c[1]])
def test_segments_shrink_towards_the_end(M, G):
    """Three tiers of 4-16, half and a quarter of that (>= 4) rows; within a tier
    every segment but the tier's last has the tier's length."""
    _, segs = segments(M, G)
    lens = [b - a for a, b in segs]
    assert max(lens) <= 16 and min(lens) >= 1
    R = M // G
    l1 = min(max(R // 8, 4), 16)
    assert max(lens) <= l1
    # non-increasing apart from the short last segment of a tier, which the next
    # tier's first segment may exceed (three tiers: at most two such steps up)
    assert sum(1 for a, b in zip(lens, lens[1:]) if b > a) <= 2
    assert sum(1 for n in lens if n not in (l1, max(l1 // 2, 4), max(l1 // 4, 4))) <= 3


def test_bad_arguments():
    assert B._load().rmsnorm_row_pool_layout(10, 0, None, None) != 0
    with pytest.raises(B.RMSNormError):
        B.rmsnorm_row_pool_layout(-1, 4)
    with pytest.raises(B.RMSNormError):
        B.rmsnorm_row_pool_segment(65536, 456, 10 ** 6)
    with pytest.raises(B.RMSNormError):
        B.rmsnorm_row_pool_segment(65536, 456, -1)


def test_tuning_switches_validate_their_arguments():
    """rmsnorm_set_row_pool takes 0, 1 or 2; rmsnorm_set_row_pool_shape takes head
    shares below 100% and non-negative lengths (0: the default). Host-only: they
    set the next plans and launch nothing."""
    assert B.rmsnorm_set_row_pool(3) == 9       # RMSNORM_ERR_ARG
    assert B.rmsnorm_set_row_pool(-1) == 9
    assert B.rmsnorm_set_row_pool_shape(100, 0, 0, 0) == 9
    assert B.rmsnorm_set_row_pool_shape(0, 0, -1, 0) == 9
    assert B.rmsnorm_set_row_pool(1) == 0
    assert B.rmsnorm_set_row_pool_shape(0, 0, 0, 0) == 0
