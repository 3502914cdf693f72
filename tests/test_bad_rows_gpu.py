"""Row indices outside [0, T*k) never become addresses.

The dispatch pass writes dest_row = -1 for a pair it cannot place (an
expert index outside [0, E)), and a caller may pass anything.  moe_permute,
moe_combine and moe_combine_backward must then skip that pair and touch no
memory outside their buffers.  Each buffer
here is a view into a larger allocation with one guard row on each side, so
a missing check would land in the guard rows (inside the allocation) rather
than fault; the guards are filled with a sentinel, or NaN where a read would
show, and must come back unchanged.  The calls go through the C ABI.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

T, K, D = 64, 4, 128
P = T * K
BAD = {5: -1, 17: P, 130: -1}  # pair -> row index outside [0, P); each lands in a guard row if unchecked
SENTINEL = 0x3F7F                   # a bf16 bit pattern no kernel here writes for these inputs


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_expert_gb300._lib import lib as l
    return l


def _guarded(rows, cols, fill_bits):
    """A [rows, cols] bf16 view with one guard row on each side, all filled with fill_bits."""
    buf = torch.full((rows + 2, cols), fill_bits, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    return buf, buf[1:rows + 1]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _rows():
    """(valid rows, the same with BAD applied), both on the device."""
    g = torch.Generator().manual_seed(3)
    good = torch.randperm(P, generator=g).to(torch.int32)
    bad = good.clone()
    for p, r in BAD.items():
        bad[p] = r
    return good.cuda(), bad.cuda()


def test_permute_skips_rows_outside_the_buffer(lib):
    g = torch.Generator().manual_seed(1)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16).cuda()
    good, bad = _rows()
    buf, xp = _guarded(P, D, SENTINEL)
    before = buf.clone()
    assert lib.moe_permute(_ptr(x), T, D, _ptr(bad), K, _ptr(xp), _stream()) == 0
    torch.cuda.synchronize()
    assert torch.equal(buf[0], before[0]) and torch.equal(buf[-1], before[-1]), "a guard row changed"
    for p in range(P):
        r = int(good[p])
        if p in BAD:
            assert torch.equal(xp[r], before[1 + r]), f"row of skipped pair {p} was written"
        else:
            assert torch.equal(xp[r], x[p // K]), p


def test_combine_leaves_bad_slots_out_of_the_sum(lib):
    g = torch.Generator().manual_seed(2)
    ybuf, y = _guarded(P, D, 0x7FC0)  # NaN guards: a read of them would poison the sum
    y.copy_(torch.randn(P, D, generator=g).to(torch.bfloat16).cuda())
    w = torch.rand(T, K, generator=g).cuda()
    good, bad = _rows()
    obuf, out = _guarded(T, D, SENTINEL)
    before = obuf.clone()
    assert lib.moe_combine(_ptr(y), _ptr(bad), _ptr(w), T, K, D, _ptr(out), _stream()) == 0
    # the same sum with those slots present at weight 0 (adding +-0 changes no fp32 sum)
    w0 = w.clone().view(-1)
    good0 = good.clone()
    for p in BAD:
        w0[p] = 0.0
    ref = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
    assert lib.moe_combine(_ptr(y), _ptr(good0), _ptr(w0), T, K, D, _ptr(ref), _stream()) == 0
    torch.cuda.synchronize()
    assert torch.equal(obuf[0], before[0]) and torch.equal(obuf[-1], before[-1]), "a guard row changed"
    assert torch.isfinite(out.float()).all(), "a guard row of y was read"
    assert torch.equal(out, ref)


def test_combine_backward_skips_bad_slots(lib):
    g = torch.Generator().manual_seed(4)
    dout = torch.randn(T, D, generator=g).to(torch.bfloat16).cuda()
    ybuf, y = _guarded(P, D, 0x7FC0)
    y.copy_(torch.randn(P, D, generator=g).to(torch.bfloat16).cuda())
    w = torch.rand(T, K, generator=g).cuda()
    good, bad = _rows()
    dbuf, dy = _guarded(P, D, SENTINEL)
    before = dbuf.clone()
    dw = torch.full((T, K), 7.0, device="cuda")
    assert lib.moe_combine_backward(_ptr(dout), _ptr(y), _ptr(bad), _ptr(w), T, K, D, _ptr(dy), _ptr(dw),
                                    _stream()) == 0
    dy_ref = torch.empty(P, D, dtype=torch.bfloat16, device="cuda")
    dw_ref = torch.empty(T, K, device="cuda")
    assert lib.moe_combine_backward(_ptr(dout), _ptr(y), _ptr(good), _ptr(w), T, K, D, _ptr(dy_ref),
                                    _ptr(dw_ref), _stream()) == 0
    torch.cuda.synchronize()
    assert torch.equal(dbuf[0], before[0]) and torch.equal(dbuf[-1], before[-1]), "a guard row changed"
    flat = dw.view(-1)
    for p in range(P):
        r = int(good[p])
        if p in BAD:
            assert float(flat[p]) == 0.0, p
            assert torch.equal(dy[r], before[1 + r]), f"row of skipped pair {p} was written"
        else:
            assert float(flat[p]) == float(dw_ref.view(-1)[p]), p
            assert torch.equal(dy[r], dy_ref[r]), p


def test_get_device_status_returns_the_recorded_error(lib):
    import sparse_expert_gb300 as moe
    idx = torch.tensor([[0, 1], [2, 9], [1, 3]], dtype=torch.int32, device="cuda")
    res = moe.moe_dispatch_scan(idx, 4)
    assert lib.moe_get_device_status(_ptr(res["workspace"]), _stream()) == 5  # MOE_ERR_BAD_INDEX
    res = moe.moe_dispatch_scan(idx.clamp(max=3), 4)
    assert lib.moe_get_device_status(_ptr(res["workspace"]), _stream()) == 0
