"""Host-side arithmetic the GQA kernel's scheduling relies on, checked by brute
force (no GPU).

A launch in which no request can reach two splits skips the scanning prologue
and numbers its items (request, kv head) directly.  That holds when the split
cap is 1, or when every request's attended pages fit in one minimum split:
with a sliding window of W tokens over L keys, the attended keys are
[max(L - W, 0), L) (the Flint decode page's window: the last W positions,
the current token included), and the pages they touch number at most
(W + 2P - 2) // P for page size P.  The minimum split is 256 tokens, i.e.
256 // P pages."""
import pytest


def cdiv(a, b):
    return -(-a // b)


def attended_pages(L, W, P):
    start = L - W if (W > 0 and L > W) else 0
    return cdiv(L, P) - start // P


@pytest.mark.parametrize("P", [16, 32])
def test_window_page_bound_holds_and_is_tight(P):
    for W in range(1, 600):
        bound = (W + 2 * P - 2) // P
        worst = max(attended_pages(L, W, P) for L in range(0, 4 * W + 4 * P))
        assert worst == bound, (P, W, worst, bound)


@pytest.mark.parametrize("P, widest", [(16, 241), (32, 225)])
def test_widest_window_that_never_splits(P, widest):
    """The kernel takes the no-scan path exactly for windows up to `widest`."""
    min_pages = 256 // P
    fits = [W for W in range(1, 1000) if (W + 2 * P - 2) // P <= min_pages]
    assert max(fits) == widest and fits == list(range(1, widest + 1))
    # a window of 128 tokens (the Flint sliding-window layer) is on that path
    assert 128 in fits
