"""msda_query_order_static: the query order for callers that may not allocate.

Some callers cannot call cudaMalloc on their path (an allocation-free real-time loop, a
plugin whose host owns all device memory), so the library offers the query order with
its scratch in a fixed device array instead of a caller workspace.  These tests call it
through the C ABI and compare it with msda_query_order on two calls in a row, with
different sizes, so that scratch left over by the first call would show up in the second.

The order of queries that share a Morton cell is not fixed (atomic slots), so the two
orders are compared on what is unique: both are permutations, and the cell (key) of the
query at every position is the same.  The keys come from msda_query_order's workspace,
whose second region holds one int32 key per query.

This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest

import workloads

ORDER_BUCKETS = 4096


def _msda():
    import scale_deformable_attention_msda3d_b300 as m
    m.load()
    return m


def test_rejects_problems_beyond_the_fixed_scratch():
    msda = _msda()
    fake = 0x10000  # never dereferenced: the size check comes first
    for B, Nq in ((65, 10), (2, 600000), (1, (1 << 20) + 1)):
        d = msda.make_dims(B, 1, Nq, 8, 32, 4, 4, msda.MSDA_F32)
        st = msda.query_order_static_raw(2, d, fake, fake, 0)
        assert st == msda.MSDA_ERR_UNSUPPORTED
        assert "at most" in msda.msda_last_error()
    d = msda.make_dims(64, 1, (1 << 20) // 64, 8, 32, 4, 4, msda.MSDA_F32)
    assert msda.query_order_static_raw(2, d, fake, 0, 0) == msda.MSDA_ERR_INVALID_ARG
    # nothing to order: OK without touching the device
    d = msda.make_dims(3, 1, 0, 8, 32, 4, 4, msda.MSDA_F32)
    assert msda.query_order_static_raw(3, d, 0, 0, 0) == msda.MSDA_OK


@pytest.mark.gpu
def test_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    msda = _msda()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    for name in ("volume3d", "decoder2d"):          # two calls, different B, Nq and ndim
        w = workloads.WORKLOADS[name]
        loc = torch.from_numpy(workloads.make_inputs(w)["sampling_locations"]).to(dev)
        B, Nq, nd = w.B, w.Nq, w.ndim
        # the existing entry point, with a workspace
        nbytes = msda.query_order_workspace_bytes(B, Nq, w.M, w.L, w.P, nd)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        ref = msda.msda_query_order(loc, workspace=ws)
        # the fixed-scratch entry point, through the C ABI
        got = torch.full((B, Nq), -1, dtype=torch.int32, device=dev)
        dims = msda.make_dims(B, 1, Nq, w.M, 4, w.L, w.P, msda.MSDA_F32)
        st = msda.query_order_static_raw(nd, dims, loc.data_ptr(), got.data_ptr(),
                                         stream.cuda_stream)
        assert st == msda.MSDA_OK, msda.msda_last_error()
        torch.cuda.synchronize()
        ref_h, got_h = ref.cpu().numpy(), got.cpu().numpy()
        off = ((B * ORDER_BUCKETS * 4 + 255) // 256) * 256
        keys = ws[off:off + B * Nq * 4].view(torch.int32).reshape(B, Nq).cpu().numpy()
        for b in range(B):
            assert np.array_equal(np.sort(got_h[b]), np.arange(Nq)), (name, b)
            assert np.array_equal(np.sort(ref_h[b]), np.arange(Nq)), (name, b)
            k_ref, k_got = keys[b][ref_h[b]], keys[b][got_h[b]]
            assert np.all(np.diff(k_ref) >= 0), (name, b)
            assert np.array_equal(k_ref, k_got), (name, b)
