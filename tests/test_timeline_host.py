"""Host logic of the per-CTA timeline tool, without a GPU: decoding the device buffer,
grouping CTA records into launches, idle-gap accounting and the per-layer critical-path
report, on synthetic records whose answers are known by construction."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from diffusion_lookahead_decoding_gb300 import timeline as T  # noqa: E402


def _buffer(recs):
    """The device buffer layout: a 16-byte header {count, capacity, 0, 0}, then records of
    {tag, cta, sm, pad} (u32) and {t0, t_ready, t1} (u64)."""
    n = len(recs)
    buf = np.zeros(4 + n * 10, dtype=np.int32)
    buf[0], buf[1] = n, n
    body = buf[4:].view(np.uint32).reshape(n, 10)
    for i, (tag, cta, sm, t0, tw, t1) in enumerate(recs):
        body[i, 0:4] = (tag, cta, sm, 0)
        body[i, 4:10] = np.array([t0, tw, t1], dtype=np.uint64).view(np.uint32)
    return buf


class _Host:
    """Stands in for the device tensor: the decoder only indexes and copies to host."""

    def __init__(self, a):
        self.a = a

    def __getitem__(self, k):
        r = self.a[k]
        return _Host(r) if isinstance(r, np.ndarray) else _Scalar(r)

    def cpu(self):
        return self

    def numpy(self):
        return self.a


class _Scalar:
    def __init__(self, v):
        self.v = v

    def item(self):
        return int(self.v)


def test_records_decode_and_drop_ready_stamps_outside_the_cta():
    recs = [(13, 0, 5, 1000, 1500, 2000),      # ready inside [start, end]
            (13, 1, 6, 1000, 0, 2100),         # no ready stamp
            (30, 2, 7, 3000, 2500, 4000),      # a stamp before the start is not a ready time
            (30, 3, 8, 3000, 5000, 4000)]      # nor one after the end
    out = T._records(_Host(_buffer(recs)))
    assert out.shape == (4, 6)
    np.testing.assert_array_equal(out[:, 0], [13, 13, 30, 30])          # tags
    np.testing.assert_array_equal(out[:, 1], [1000, 1000, 3000, 3000])  # starts
    np.testing.assert_array_equal(out[:, 2], [1500, 0, 0, 0])           # ready
    np.testing.assert_array_equal(out[:, 3], [2000, 2100, 4000, 4000])  # ends
    np.testing.assert_array_equal(out[:, 4], [0, 1, 2, 3])              # CTA index
    np.testing.assert_array_equal(out[:, 5], [5, 6, 7, 8])              # SM


def _rec(tag, t0, t1, tw=0, cta=0, sm=0):
    return [tag, t0, tw, t1, cta, sm]


def test_launches_split_one_kernel_at_gaps_and_sort_by_start():
    r = np.array([
        _rec(11, 0, 500), _rec(11, 100, 900), _rec(11, 950, 1200),    # launch A (overlapping CTAs)
        _rec(11, 5000, 5400), _rec(11, 5100, 5600),                   # launch B, 3.8 us later
        _rec(20, 1300, 4000),                                         # another kernel in between
    ], dtype=np.int64)
    ls = T.launches(r)
    assert [(tg, len(c)) for _, tg, c in ls] == [(11, 3), (20, 1), (11, 2)]
    assert [s for s, _, _ in ls] == [0, 1300, 5000]


def test_gaps_count_only_intervals_with_no_resident_cta():
    r = np.array([
        _rec(1, 0, 10_000), _rec(2, 2_000, 12_000),    # overlap: no gap
        _rec(3, 15_000, 20_000),                       # 3 us gap
        _rec(4, 21_000, 22_000),                       # 1 us gap: below the 2 us threshold
        _rec(5, 30_000, 31_000),                       # 8 us gap
    ], dtype=np.int64)
    span, idle, n = T.gaps(r)
    assert span == 31_000
    assert (idle, n) == (11_000, 2)
    assert T.gaps(r, min_ns=500)[1:] == (12_000, 3)


def test_report_increments_follow_the_last_cta_of_each_kernel():
    """One forward: embed, then per layer q/k/v, attention, output projection, norm,
    gate/up, down, norm, then the LM head and the merge.  Each kernel's last CTA ends a
    known time after the previous kernel's last CTA; the report's per-slot means must be
    those increments."""
    slots = [13, 20, 10, 30, 11, 10, 30]   # tags of the seven kernels of a layer
    incr = [21, 15, 13, 8, 48, 32, 8]      # us after the previous kernel's last CTA end
    n_layers = 3
    rows, t = [], 0
    rows.append(_rec(31, 0, 1_000))        # embed
    t = 1_000
    for _ in range(n_layers):
        for tg, d in zip(slots, incr):
            t += 2_000                     # the kernel's last CTA ends d + 2 us after its
            start = t - 2_500              # predecessor's, and it starts 0.5 us before that end
            rows.append(_rec(tg, start, t + d * 1000 - 300, cta=0))
            rows.append(_rec(tg, start + 10, t + d * 1000, cta=1))   # the last CTA
            t += d * 1000
    rows.append(_rec(12, t - 500, t + 216_000))   # LM head
    t += 216_000
    rows.append(_rec(32, t - 500, t + 12_000))    # merge
    text = T.report(np.array(rows, dtype=np.int64), n_layers, layer=1)
    body = text.split("critical-path increment")[1].split("relative to the previous")[0]
    lines = {ln.split()[0]: ln.split() for ln in body.splitlines() if ln.startswith("  ")}
    for name, d in zip(T.SLOTS, incr):
        assert abs(float(lines[name][1]) - (d + 2.0)) < 1e-6, (name, lines[name])
    assert abs(float(lines["layer"][1]) - (sum(incr) + 14.0)) < 1e-6
    assert "lmstats: +216.00" in text and "merge: +12.00" in text
