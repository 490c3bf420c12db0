"""Host logic of conv_fwd_from_host, checked without a GPU: the slices it
cuts a problem into (conv_fwd_from_host_slices plans host-only for a given
SM count) tile the output rows in order, and before each slice runs the
device holds every input row that slice's output rows read.  The reads are
enumerated here tap by tap from the convolution's definition (output row
(n, od, oh, ow) reads input depth od*sd - pd + t*dd and row oh*sh - ph +
r*dh for every tap (t, r) that lands inside x), independently of the
library's reach rule."""
import random

import pytest

import conv_workloads as cw


@pytest.fixture(scope="module")
def pkg():
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


def _out_dim(i, f, s, p, d):
    return (i + 2 * p - d * (f - 1) - 1) // s + 1


def _held(reach, plane, H):
    whole, part, rows = reach
    return H if plane < whole else (rows if plane < part else 0)


def _check_plan(pkg, xs, ws, st, pa, di, num_sms, chunks):
    N, D, H, W, C = xs
    K, T, R, S, _ = ws
    Do, Ho, Wo = (_out_dim(D, T, st[0], pa[0], di[0]), _out_dim(H, R, st[1], pa[1], di[1]),
                  _out_dim(W, S, st[2], pa[2], di[2]))
    M = N * Do * Ho * Wo
    plan = pkg.conv_fwd_from_host_slices(xs, ws, st, pa, di, num_sms=num_sms, chunks=chunks)
    rows, reach = plan["rows"], plan["reach"]
    assert 1 <= len(rows) <= 32 and len(reach) == len(rows)
    # the slices tile [0, M) in order
    assert rows[0][0] == 0 and rows[-1][1] == M
    assert all(lo < hi for lo, hi in rows)
    assert all(a[1] == b[0] for a, b in zip(rows, rows[1:]))
    # the last slice has all of x
    assert reach[-1][0] == N * D
    # every input row read below each slice's end is held by then
    need = {}
    i = 0
    for row in range(M):
        ow = row % Wo
        oh = (row // Wo) % Ho
        q = row // (Wo * Ho)
        n, od = divmod(q, Do)
        for t in range(T):
            d = od * st[0] - pa[0] + t * di[0]
            if not 0 <= d < D:
                continue
            for r in range(R):
                h = oh * st[1] - pa[1] + r * di[1]
                if 0 <= h < H:
                    p = n * D + d
                    need[p] = max(need.get(p, -1), h)
        while i < len(rows) and row + 1 == rows[i][1]:
            for p, hmax in need.items():
                assert _held(reach[i], p, H) > hmax, (xs, ws, st, pa, di, i, p, hmax, reach[i])
            i += 1
    return plan


def test_headline_slice_plan(pkg):
    """The video conv on 152 SMs: 512 x 256 units, blocks of 19 m-tiles
    (9728 rows, two waves of 76 CTA pairs); one block first (split over two
    weight groups), one, then doubling up to a sixth of the rest, one last."""
    wl = cw.BY_NAME["video_conv3d_bf16"]
    plan = pkg.conv_fwd_from_host_slices(wl.x_shape, wl.w_shape, wl.stride, wl.pad, wl.dil,
                                         num_sms=152)
    blocks = [(hi - lo) / 9728 for lo, hi in plan["rows"]]
    assert blocks[:-1] == [1, 1, 2, 4, 4, 4, 4, 1]
    assert plan["rows"][-1] == (204288, 216000)
    assert plan["weight_groups"] == 2
    # the first slice reads rows 0..82 of input planes 0 and 1 only
    assert plan["reach"][0] == (0, 2, 83)


@pytest.mark.parametrize("chunks", [0, 2, 3, 7])
def test_slices_hold_every_input_row_read(pkg, chunks):
    """Seeded random geometries (strides, dilations and padding in D and H,
    several images), few SMs so that the problems span many waves; only
    plans of two or more slices count."""
    rng = random.Random(900 + chunks)
    checked = 0
    while checked < 12:
        N, D, H, W = rng.randint(1, 3), rng.randint(1, 9), rng.randint(3, 40), rng.randint(2, 24)
        C = rng.choice([8, 16, 32])
        T, R, S = rng.randint(1, 3), rng.randint(1, 3), rng.randint(1, 3)
        st = (rng.randint(1, 2), rng.randint(1, 3), rng.randint(1, 2))
        di = (rng.randint(1, 2), rng.randint(1, 2), 1)
        pa = (rng.randint(0, 2), rng.randint(0, 3), rng.randint(0, 1))
        dims = [_out_dim(D, T, st[0], pa[0], di[0]), _out_dim(H, R, st[1], pa[1], di[1]),
                _out_dim(W, S, st[2], pa[2], di[2])]
        if min(dims) < 1 or N * dims[0] * dims[1] * dims[2] > 6000:
            continue
        if T == 1 and R == 1 and S == 1:
            continue   # pointwise: a GEMM, unsliced
        xs, ws = (N, D, H, W, C), (rng.choice([32, 64, 96]), T, R, S, C)
        try:
            plan = _check_plan(pkg, xs, ws, st, pa, di, rng.choice([2, 4, 8]), chunks)
        except pkg.ConvError as e:
            assert e.status == pkg.CONV_ERR_UNSUPPORTED
            continue
        checked += len(plan["rows"]) >= 2


def test_unsliced_plans(pkg):
    # one slice asked for, and a point-output GEMM (never sliced): all of x first
    for xs, ws, st, chunks in (((2, 6, 12, 10, 64), (96, 3, 3, 3, 64), 1, 1),
                               ((300, 1, 14, 14, 3), (200, 1, 14, 14, 3), (1, 14, 14), 0)):
        plan = _check_plan(pkg, xs, ws, pkg._triple(st), (0, 0, 0) if chunks == 0 else (1, 1, 1),
                           (1, 1, 1), 152, chunks)
        assert len(plan["rows"]) == 1 and plan["weight_groups"] == 1


def test_slice_query_argument_errors(pkg):
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_fwd_from_host_slices((1, 4, 8, 8, 16), (32, 3, 3, 3, 16), 1, 1, 1,
                                      num_sms=152, chunks=-1)
    assert e.value.status == pkg.CONV_ERR_INVALID
