"""The fused step's launch-window split, restated from include/zero.h for the
tests: ceil(length / ZERO_FUSED_WINDOW_ELEMS) windows of about equal length
(none longer than ZERO_FUSED_WINDOW_ELEMS + 15) over a shard, every inner cut on a 16-element (32-byte) boundary of row 0
(whose element 0 sits `phase` elements past a 32-byte boundary: its offset in
the row, for the 32-byte aligned torch buffers of the tests), and a remainder
of under 64 elements joined to the last window.  Used to put sampled oracle
checks on every cut, and to pin the binding's launch count."""

WINDOW_ELEMS = 10485760   # ZERO_FUSED_WINDOW_ELEMS


def window_cuts(length: int, phase: int = 0, window: int = WINDOW_ELEMS):
    """[(w0, w1), ...] windows tiling [0, length) in order."""
    if length <= 0:
        return []
    nwin = -(-length // window)
    target = -(-(-(-length // nwin)) // 16) * 16
    cuts, w0, cut = [], 0, target - (phase & 15)
    while w0 < length:
        w1 = min(cut, length)
        if length - w1 < 64:
            w1 = length
        cuts.append((w0, w1))
        w0, cut = w1, cut + target
    return cuts


def inner_cuts(length: int, phase: int = 0):
    """The element indices where one launch window ends and the next begins."""
    return [w0 for w0, _ in window_cuts(length, phase)[1:]]
