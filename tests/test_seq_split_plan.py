"""The sequence split's launch plan, on the CPU: the job of every CTA of its two passes
(segment, map kind, chunk range, where its state comes from and goes), the scan between
them and the slots of the segment states and maps, emulated on small random affine chunk
maps H <- A_c H + B_c.  The plan must give every chunk's output from its true incoming
state exactly once, the true final state, slots inside the workspace extent
(units x 3 nseg x dk x 128 floats), and a first pass of one wave on the GPU it is
planned for.  The kernels' own results are compared with the oracle by the GPU tests."""
import numpy as np
import pytest


def segments(units, nchunks, dv, sms):
    """The segment count (1: no split): dv = 128, at least five SMs per (b, h), a first pass
    of 1 + 2 (nseg - 2) CTAs per (b, h) in one wave, at most 16 segments of >= 16 chunks."""
    if dv != 128 or units < 1 or sms // units < 5:
        return 1
    n = min((sms // units - 1) // 2 + 2, 16, nchunks // 16)
    return n if n >= 3 else 1


def jobs(pass_, nseg):
    return 1 if pass_ == 0 else (1 + 2 * (nseg - 2) if pass_ == 1 else nseg - 1)


def slot(unit, nseg, kind, s, dk=4, cols=4):
    return ((unit * 3 * nseg + kind * nseg + s) * dk) * cols


def run_plan(nch, nseg, units, rng, d=4):
    cps = -(-nch // nseg)
    A = rng.standard_normal((units, nch, d, d)) * 0.3
    Bm = rng.standard_normal((units, nch, d, d))
    S0 = rng.standard_normal((units, d, d))
    seg = np.full(units * 3 * nseg * d * d, np.nan)
    got = np.full((units, nch, d, d), np.nan)
    fin = {}
    for pass_ in (1, 2):
        if pass_ == 2:   # the scan: state(s) = M_{s-1} state(s-1) + N_{s-1}
            for u in range(units):
                for s in range(2, nseg):
                    g = lambda kind, t: seg[slot(u, nseg, kind, t, d, d):slot(u, nseg, kind, t, d, d) + d * d].reshape(d, d)
                    seg[slot(u, nseg, 0, s, d, d):slot(u, nseg, 0, s, d, d) + d * d] = \
                        (g(2, s - 1) @ g(0, s - 1) + g(1, s - 1)).ravel()
        J = jobs(pass_, nseg)
        for blk in range(units * J):
            u, j = divmod(blk, J)
            sg, kind = 0, 0
            if pass_ == 1 and j >= 1:
                sg, kind = 1 + (j - 1) // 2, 1 + (j - 1) % 2
            elif pass_ == 2:
                sg = 1 + j
            cs, ce = sg * cps, min(nch, (sg + 1) * cps)
            assert ce > cs
            if pass_ == 1 and sg == 0:
                H = S0[u].copy()
            elif pass_ == 2:
                o = slot(u, nseg, 0, sg, d, d)
                H = seg[o:o + d * d].reshape(d, d).copy()
                assert np.all(np.isfinite(H)), "a segment's incoming state is read before it is written"
            else:
                H = np.eye(d) if kind == 2 else np.zeros((d, d))
            for c in range(cs, ce):
                if kind == 0:
                    assert np.all(np.isnan(got[u, c])), "a chunk's output is written twice"
                    got[u, c] = H
                H = A[u, c] @ H + (0 if kind == 2 else Bm[u, c])
            if pass_ == 1:
                o = slot(u, nseg, 0 if sg == 0 else kind, 1 if sg == 0 else sg, d, d)
                assert 0 <= o and o + d * d <= seg.size
                seg[o:o + d * d] = H.ravel()
            elif sg == nseg - 1:
                fin[u] = H
    # the serial recurrence
    for u in range(units):
        H = S0[u].copy()
        for c in range(nch):
            assert np.allclose(got[u, c], H), (nch, nseg, u, c)
            H = A[u, c] @ H + Bm[u, c]
        assert np.allclose(fin[u], H)


@pytest.mark.parametrize("nseg", range(3, 17))
def test_plan_reproduces_the_serial_recurrence(nseg):
    rng = np.random.default_rng(nseg)
    for nch in (16 * nseg, 16 * nseg + 1, 16 * nseg + nseg - 1, 16 * nseg + 37):
        run_plan(nch, nseg, units=2, rng=rng)


def test_segment_count_fits_one_wave():
    for sms in (132, 148, 152, 160):
        for units in range(1, 64):
            for nch in (16, 47, 48, 100, 128, 512, 1024):
                n = segments(units, nch, 128, sms)
                assert n == 1 or 3 <= n <= 16
                if n >= 3:
                    assert units * jobs(1, n) <= sms, (sms, units, nch, n)
                    assert nch // n >= 16
    # the long-sequence workloads on a 152-SM GB300: six segments
    assert segments(16, 1024, 128, 152) == 6 and segments(16, 128, 128, 152) == 6
    # many (b, h) or dv = 64: no split
    assert segments(64, 32, 128, 152) == 1 and segments(1, 1024, 64, 152) == 1
