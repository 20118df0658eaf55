"""Host-side checks of the C ABI (no GPU): the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the device.

Every call here either fails validation or is an empty no-op, so no CUDA API call is
made; pointer arguments are plain integers that are never dereferenced.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import scale_deformable_attention_msda3d_b300 as msda
from scale_deformable_attention_msda3d_b300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msda.h")

FAKE = 0x10000          # 16-byte aligned, never dereferenced
FAKE_MIS = 0x10004      # misaligned


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msda\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return msda.load()


def test_header_and_binding_agree():
    assert declared_functions() == sorted(_binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and through a fresh handle with plain dlopen semantics
    raw = ctypes.CDLL(msda.library_path())
    for name in declared_functions():
        getattr(raw, name)


def test_abi_version(lib):
    assert msda.msda_abi_version() == 10300


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        _binding.load(str(tmp_path / "no_such_libmsda.so"))


SH2 = np.array([[4, 6], [2, 3]], dtype=np.int64)
LS2 = np.array([0, 24], dtype=np.int64)
SH3 = np.array([[2, 4, 6], [1, 2, 3]], dtype=np.int64)
LS3 = np.array([0, 48], dtype=np.int64)


def dims(**kw):
    d = dict(B=2, Nin=30, Nq=5, M=2, D=8, L=2, P=4, value_dtype=msda.MSDA_F32)
    d.update(kw)
    return msda.make_dims(**d)


def fwd(nd=2, d=None, sh=None, ls=None, ptrs=None):
    d = d or (dims() if nd == 2 else dims(Nin=54))
    sh = SH2 if (sh is None and nd == 2) else (SH3 if sh is None else sh)
    ls = LS2 if (ls is None and nd == 2) else (LS3 if ls is None else ls)
    p = dict(value=FAKE, loc=FAKE, attn=FAKE, out=FAKE)
    p.update(ptrs or {})
    return msda.forward_raw(nd, d, p["value"], sh, ls, p["loc"], p["attn"], p["out"], 0)


def bwd(nd=2, d=None, ptrs=None):
    d = d or dims()
    p = dict(value=FAKE, loc=FAKE, attn=FAKE, go=FAKE, gv=FAKE, gl=FAKE, ga=FAKE)
    p.update(ptrs or {})
    return msda.backward_raw(nd, d, p["value"], SH2, LS2, p["loc"], p["attn"], p["go"],
                             p["gv"], p["gl"], p["ga"], 0)


@pytest.mark.parametrize("case,status,msg", [
    (dict(d=dims(value_dtype=7)), msda.MSDA_ERR_INVALID_ARG, "value_dtype"),
    (dict(d=dims(Nq=-1)), msda.MSDA_ERR_INVALID_ARG, ">= 0"),
    (dict(d=dims(M=0)), msda.MSDA_ERR_INVALID_ARG, ">= 1"),
    (dict(d=dims(D=0)), msda.MSDA_ERR_INVALID_ARG, ">= 1"),
    (dict(d=dims(L=17)), msda.MSDA_ERR_UNSUPPORTED, "MSDA_MAX_LEVELS"),
    (dict(d=dims(P=33)), msda.MSDA_ERR_UNSUPPORTED, "MSDA_MAX_POINTS"),
    (dict(d=dims(D=6)), msda.MSDA_ERR_UNSUPPORTED, "D * sizeof"),
    (dict(d=dims(D=12)), msda.MSDA_ERR_UNSUPPORTED, "D * sizeof"),
    (dict(d=dims(D=256)), msda.MSDA_ERR_UNSUPPORTED, "D * sizeof"),
    (dict(d=dims(D=4, value_dtype=msda.MSDA_BF16)), msda.MSDA_ERR_UNSUPPORTED, "D * sizeof"),
    (dict(d=dims(Nin=31)), msda.MSDA_ERR_INVALID_ARG, "add up to"),
    (dict(ls=np.array([0, 23])), msda.MSDA_ERR_INVALID_ARG, "prefix sum"),
    (dict(ls=np.array([1, 24])), msda.MSDA_ERR_INVALID_ARG, "prefix sum"),
    (dict(sh=np.array([[4, 6], [0, 3]])), msda.MSDA_ERR_INVALID_ARG, "spatial_shapes"),
    (dict(sh=np.array([[4, -6], [2, 3]])), msda.MSDA_ERR_INVALID_ARG, "spatial_shapes"),
    (dict(d=dims(Nin=2 ** 30 + 5)), msda.MSDA_ERR_UNSUPPORTED, "2^30"),
    (dict(ptrs=dict(value=0)), msda.MSDA_ERR_INVALID_ARG, "value is NULL"),
    (dict(ptrs=dict(loc=0)), msda.MSDA_ERR_INVALID_ARG, "sampling_locations is NULL"),
    (dict(ptrs=dict(attn=0)), msda.MSDA_ERR_INVALID_ARG, "attention_weights is NULL"),
    (dict(ptrs=dict(out=0)), msda.MSDA_ERR_INVALID_ARG, "out is NULL"),
    (dict(ptrs=dict(value=FAKE_MIS)), msda.MSDA_ERR_INVALID_ARG, "aligned"),
    (dict(ptrs=dict(out=FAKE_MIS)), msda.MSDA_ERR_INVALID_ARG, "aligned"),
])
def test_forward_rejects_bad_arguments(lib, case, status, msg):
    st = fwd(**case)
    assert st == status, (st, msda.msda_last_error())
    assert msg in msda.msda_last_error()


def test_forward_3d_rejects_bad_arguments(lib):
    assert fwd(nd=3, d=dims(Nin=54), sh=np.array([[2, 4, 6], [1, 2, 4]])) == \
        msda.MSDA_ERR_INVALID_ARG
    # an extent of 2^23 or more is outside what the kernels support
    assert fwd(nd=3, d=dims(Nin=54), sh=np.array([[2, 4, 2 ** 24], [1, 2, 3]])) == \
        msda.MSDA_ERR_UNSUPPORTED


def test_null_metadata_and_dims(lib):
    d = dims()
    fn = lib.msda2d_forward
    st = fn(None, _binding._VP(FAKE), None, None, _binding._VP(FAKE), _binding._VP(FAKE),
            _binding._VP(FAKE), _binding._VP(0))
    assert st == msda.MSDA_ERR_INVALID_ARG and "dims" in msda.msda_last_error()
    st = fn(ctypes.byref(d), _binding._VP(FAKE), None, None, _binding._VP(FAKE),
            _binding._VP(FAKE), _binding._VP(FAKE), _binding._VP(0))
    assert st == msda.MSDA_ERR_INVALID_ARG and "spatial_shapes" in msda.msda_last_error()


@pytest.mark.parametrize("ptrs,msg", [
    (dict(gv=0), "grad_value is NULL"), (dict(go=0), "grad_out is NULL"),
    (dict(gl=FAKE_MIS), "grad_sampling_locations is not 16-byte aligned"),
    (dict(ga=0), "grad_attention_weights is NULL"),
])
def test_backward_rejects_bad_arguments(lib, ptrs, msg):
    st = bwd(ptrs=ptrs)
    assert st == msda.MSDA_ERR_INVALID_ARG
    assert msg in msda.msda_last_error()


def test_empty_calls_are_ok_without_touching_the_device(lib):
    # no queries: nothing to compute, null tensor pointers are fine
    assert fwd(d=dims(Nq=0), ptrs=dict(value=0, loc=0, attn=0, out=0)) == msda.MSDA_OK
    assert fwd(d=dims(B=0), ptrs=dict(value=0, loc=0, attn=0, out=0)) == msda.MSDA_OK
    assert fwd(nd=3, d=dims(Nq=0, Nin=54)) == msda.MSDA_OK
    # empty batch backward: no grad_value rows to zero
    assert bwd(d=dims(B=0), ptrs=dict(gv=0, go=0)) == msda.MSDA_OK


def test_error_message_is_per_thread(lib):
    import threading
    fwd(d=dims(M=0))
    seen = {}

    def other():
        seen["msg"] = msda.msda_last_error()

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert seen["msg"] == ""
    assert ">= 1" in msda.msda_last_error()


def test_torch_layer_rejects_host_tensors():
    torch = pytest.importorskip("torch")
    v = torch.zeros(1, 24, 2, 8)
    loc = torch.zeros(1, 3, 2, 1, 4, 2)
    a = torch.zeros(1, 3, 2, 1, 4)
    with pytest.raises(msda.MsdaError):
        msda.msda2d_forward(v, np.array([[4, 6]]), np.array([0]), loc, a)


def test_query_order_workspace_size(lib):
    st, n = msda.query_order_workspace_raw(2, dims(B=3, Nq=1000))
    assert st == msda.MSDA_OK
    # per-batch histogram of 4096 ints, then one int per query, each 256-byte aligned
    assert n == 3 * 4096 * 4 + ((3 * 1000 * 4 + 255) // 256) * 256
    assert msda.query_order_workspace_raw(4, dims())[0] == msda.MSDA_ERR_INVALID_ARG
    assert msda.query_order_workspace_raw(2, dims(P=0))[0] == msda.MSDA_ERR_INVALID_ARG
    assert msda.query_order_workspace_raw(3, dims(Nq=2 ** 31))[0] == msda.MSDA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,msg", [
    (dict(order=0), "query_order is NULL"),
    (dict(order=FAKE + 2), "4-byte aligned"),
    (dict(ws=0), "workspace is NULL"),
    (dict(ws_bytes=1024), "needed"),
    (dict(loc=FAKE_MIS), "aligned"),
])
def test_query_order_rejects_bad_arguments(lib, kw, msg):
    d = dims()
    args = dict(loc=FAKE, order=FAKE, ws=FAKE, ws_bytes=1 << 24)
    args.update(kw)
    st = msda.query_order_raw(2, d, args["loc"], args["order"], args["ws"], args["ws_bytes"], 0)
    assert st == msda.MSDA_ERR_INVALID_ARG
    assert msg in msda.msda_last_error()


def test_ordered_forward_rejects_bad_order(lib):
    for order, msg in ((0, "query_order is NULL"), (FAKE + 1, "4-byte aligned")):
        st = msda.forward_ordered_raw(2, dims(), FAKE, SH2, LS2, FAKE, FAKE, order, FAKE, 0)
        assert st == msda.MSDA_ERR_INVALID_ARG and msg in msda.msda_last_error()
    # the core's own checks still run first
    st = msda.forward_ordered_raw(2, dims(M=0), FAKE, SH2, LS2, FAKE, FAKE, FAKE, FAKE, 0)
    assert st == msda.MSDA_ERR_INVALID_ARG
    # nothing to do: OK without touching the device
    assert msda.forward_ordered_raw(2, dims(Nq=0), 0, SH2, LS2, 0, 0, 0, 0, 0) == msda.MSDA_OK


def test_ordered_backward_rejects_bad_order(lib):
    for order, msg in ((0, "query_order is NULL"), (FAKE + 1, "4-byte aligned")):
        st = msda.backward_ordered_raw(2, dims(), FAKE, SH2, LS2, FAKE, FAKE, order, FAKE, FAKE,
                                       FAKE, FAKE, 0)
        assert st == msda.MSDA_ERR_INVALID_ARG and msg in msda.msda_last_error()
    # the core's own checks still run first
    st = msda.backward_ordered_raw(2, dims(M=0), FAKE, SH2, LS2, FAKE, FAKE, FAKE, FAKE, FAKE,
                                   FAKE, FAKE, 0)
    assert st == msda.MSDA_ERR_INVALID_ARG
    # an empty batch: OK without touching the device
    assert msda.backward_ordered_raw(2, dims(B=0), 0, SH2, LS2, 0, 0, 0, 0, 0, 0, 0,
                                     0) == msda.MSDA_OK


@pytest.mark.parametrize("tau", [-0.1, float("nan"), float("inf")])
def test_pruned_forward_rejects_bad_threshold(lib, tau):
    st = msda.forward_pruned_raw(2, dims(), FAKE, SH2, LS2, FAKE, FAKE, tau, FAKE, 0)
    assert st == msda.MSDA_ERR_INVALID_ARG and "threshold" in msda.msda_last_error()


def test_fused_forward_rejects_bad_reference_points(lib):
    for ref, msg in ((0, "reference_points is NULL"), (FAKE_MIS, "reference_points is not")):
        st = msda.forward_fused_raw(2, dims(), FAKE, SH2, LS2, ref, FAKE, FAKE, FAKE, 0)
        assert st == msda.MSDA_ERR_INVALID_ARG and msg in msda.msda_last_error()
    # the core's checks apply to the offsets / logits slots as to locations / weights
    st = msda.forward_fused_raw(2, dims(), FAKE, SH2, LS2, FAKE, 0, FAKE, FAKE, 0)
    assert st == msda.MSDA_ERR_INVALID_ARG and "sampling_offsets is NULL" in msda.msda_last_error()
    st = msda.forward_fused_raw(2, dims(), FAKE, SH2, LS2, FAKE, FAKE, 0, FAKE, 0)
    assert st == msda.MSDA_ERR_INVALID_ARG and "attention_logits is NULL" in msda.msda_last_error()
    st = msda.forward_fused_raw(3, dims(Nin=54), FAKE, SH3, LS3, FAKE, FAKE, FAKE, FAKE_MIS, 0)
    assert st == msda.MSDA_ERR_INVALID_ARG and "out is not 16-byte aligned" in msda.msda_last_error()
    assert msda.forward_fused_raw(2, dims(Nq=0), 0, SH2, LS2, 0, 0, 0, 0, 0) == msda.MSDA_OK


def test_fused_backward_validates_before_any_launch(lib):
    """Every pointer of msda{2,3}d_backward_fused is checked (NULL / 16-byte alignment)
    before anything is enqueued; grad_reference_points may be NULL."""
    args = dict(value=FAKE, ref=FAKE, off=FAKE, z=FAKE, go=FAKE, gv=FAKE, goff=FAKE, gz=FAKE,
                gref=FAKE)
    names = dict(value="value", ref="reference_points", off="sampling_offsets",
                 z="attention_logits", go="grad_out", gv="grad_value",
                 goff="grad_sampling_offsets", gz="grad_attention_logits",
                 gref="grad_reference_points")

    def call(nd, d, a):
        sh, ls = (SH2, LS2) if nd == 2 else (SH3, LS3)
        return msda.backward_fused_raw(nd, d, a["value"], sh, ls, a["ref"], a["off"], a["z"],
                                       a["go"], a["gv"], a["goff"], a["gz"], a["gref"], 0)

    for nd, d in ((2, dims()), (3, dims(Nin=54))):
        for key, name in names.items():
            bad = dict(args, **{key: FAKE_MIS})
            st = call(nd, d, bad)
            assert st == msda.MSDA_ERR_INVALID_ARG, (nd, key)
            assert f"{name} is not 16-byte aligned" in msda.msda_last_error(), (nd, key)
            if key == "gref":
                continue
            st = call(nd, d, dict(args, **{key: 0}))
            assert st == msda.MSDA_ERR_INVALID_ARG and f"{name} is NULL" in msda.msda_last_error()
    # nothing to do: B = 0 is OK without touching any pointer
    assert call(2, dims(B=0), dict.fromkeys(args, 0)) == msda.MSDA_OK


def test_extents_of_2_23_or_more_are_unsupported(lib):
    """Extents up to 2^23 - 1 pass validation (the call then stops at the NULL value
    pointer, before any launch); 2^23 returns MSDA_ERR_UNSUPPORTED."""
    big = (1 << 23) - 1
    for nd, sh in ((2, np.array([[1, big]])), (3, np.array([[big, 1, 1]]))):
        d = msda.make_dims(1, big, 4, 1, 4, 1, 4, msda.MSDA_F32)
        st = msda.forward_raw(nd, d, 0, sh, np.array([0]), FAKE, FAKE, FAKE, 0)
        assert st == msda.MSDA_ERR_INVALID_ARG and "value is NULL" in msda.msda_last_error()
        sh2 = sh.copy()
        sh2[sh2 == big] = big + 1
        d2 = msda.make_dims(1, big + 1, 4, 1, 4, 1, 4, msda.MSDA_F32)
        st = msda.forward_raw(nd, d2, FAKE, sh2, np.array([0]), FAKE, FAKE, FAKE, 0)
        assert st == msda.MSDA_ERR_UNSUPPORTED and "2^23" in msda.msda_last_error()


# ------------------------------------------------------------------ MSDA_ERR_CUDA

# Runs in a child process that sees no CUDA device (CUDA_VISIBLE_DEVICES=""): every call
# below passes validation, so its first CUDA runtime call (a kernel launch, a memset or
# cudaGetDevice) fails and the library must return MSDA_ERR_CUDA with the runtime's
# message.  The pointers are aligned integers that nothing dereferences: without a device
# nothing is enqueued.
_NO_DEVICE_SCRIPT = r"""
import json, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import scale_deformable_attention_msda3d_b300 as msda
msda.load()
F = 0x10000
SH = {2: np.array([[4, 6], [2, 3]]), 3: np.array([[2, 4, 6], [1, 2, 3]])}
LS = {2: np.array([0, 24]), 3: np.array([0, 48])}
NIN = {2: 30, 3: 54}
res = {}
for nd in (2, 3):
    for dt in (msda.MSDA_F32, msda.MSDA_BF16):
        d = msda.make_dims(2, NIN[nd], 5, 2, 8, 2, 4, dt)
        sh, ls = SH[nd], LS[nd]
        calls = {
            "forward": lambda: msda.forward_raw(nd, d, F, sh, ls, F, F, F, 0),
            "forward_fused": lambda: msda.forward_fused_raw(nd, d, F, sh, ls, F, F, F, F, 0),
            "forward_pruned": lambda: msda.forward_pruned_raw(nd, d, F, sh, ls, F, F, 0.01, F, 0),
            "forward_ordered": lambda: msda.forward_ordered_raw(nd, d, F, sh, ls, F, F, F, F, 0),
            "backward": lambda: msda.backward_raw(nd, d, F, sh, ls, F, F, F, F, F, F, 0),
            "backward_ordered": lambda: msda.backward_ordered_raw(nd, d, F, sh, ls, F, F, F, F, F,
                                                                  F, F, 0),
            "backward_fused": lambda: msda.backward_fused_raw(nd, d, F, sh, ls, F, F, F, F, F, F,
                                                              F, F, 0),
            "query_order": lambda: msda.query_order_raw(nd, d, F, F, F, 1 << 24, 0),
            "query_order_static": lambda: msda.query_order_static_raw(nd, d, F, F, 0),
        }
        for name, fn in calls.items():
            st = int(fn())
            res[f"{name}/{nd}d/{dt}"] = [st, msda.msda_last_error()]
print(json.dumps(res))
"""


def test_cuda_errors_map_to_msda_err_cuda_without_a_device():
    """Every public compute call returns MSDA_ERR_CUDA, with the runtime's error in
    msda_last_error(), when its first CUDA runtime call fails (here: no visible device)."""
    import json
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _NO_DEVICE_SCRIPT, ROOT], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert len(res) == 2 * 2 * 9
    for key, (st, msg) in res.items():
        assert st == msda.MSDA_ERR_CUDA, (key, st, msg)
        # "<what>: <cudaError name> (<description>)"
        assert re.search(r": cudaError\w+ \(", msg), (key, msg)


def test_query_order_grid_too_large_is_a_cuda_error_with_nothing_enqueued(lib):
    """B * Nq beyond what one grid of one warp per query can hold: the launch layer
    returns cudaErrorInvalidConfiguration before its first enqueue (the histogram clear
    included), so the call fails with MSDA_ERR_CUDA without touching the device."""
    d = dims(B=9, Nq=2 ** 31 - 1)                     # 1.9e10 queries > 2^34
    st, need = msda.query_order_workspace_raw(2, d)
    assert st == msda.MSDA_OK
    st = msda.query_order_raw(2, d, FAKE, FAKE, FAKE, need, 0)
    assert st == msda.MSDA_ERR_CUDA, msda.msda_last_error()
    assert "cudaErrorInvalidConfiguration" in msda.msda_last_error()


def test_normal_build_has_no_bounds_checks(lib):
    """libmsda.so reports no checks, its status call is a no-op and its self-test is
    unsupported (all without a CUDA call)."""
    assert msda.msda_build_flags() == 0
    assert msda.msda_debug_bounds_status() == msda.MSDA_OK
    assert msda.msda_debug_bounds_selftest(0) == msda.MSDA_ERR_UNSUPPORTED
    assert "debug build" in msda.msda_last_error()


def test_debug_build_loads_and_exports_every_symbol():
    """libmsda_debug.so (MSDA_DEBUG_BOUNDS) exports the same entry points and says so in
    its build flags; without a device its status call fails as a CUDA error."""
    import json
    import subprocess
    import sys
    from scale_deformable_attention_msda3d_b300 import build
    path = build.build(debug=True)
    raw = ctypes.CDLL(path)
    for name in declared_functions():
        getattr(raw, name)
    script = ("import json, sys; sys.path.insert(0, sys.argv[1]); "
              "import scale_deformable_attention_msda3d_b300 as m; m.load(); "
              "print(json.dumps([m.msda_build_flags(), m.msda_debug_bounds_status(), "
              "m.msda_last_error()]))")
    env = dict(os.environ, MSDA_LIBRARY=path, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", script, ROOT], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    flags, st, msg = json.loads(r.stdout.strip().splitlines()[-1])
    assert flags == msda.MSDA_BUILD_DEBUG_BOUNDS
    assert st == msda.MSDA_ERR_CUDA and "bounds-check record" in msg
