"""The C-ABI library builds, loads without a GPU, exports every entry point
declared in include/moe.h, and rejects bad arguments on the host before any
CUDA call (these checks run on the CPU)."""
import ctypes
import re
from pathlib import Path

import pytest

import moe_routing_swiglu_gb300 as moe
from moe_routing_swiglu_gb300 import _build

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.load_library()


def declared_functions():
    text = (ROOT / "include" / "moe.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_chain():
    names = declared_functions()
    for required in ("moe_route", "moe_dispatch", "moe_experts_create", "moe_experts_forward_dispatched",
                     "moe_combine", "moe_forward"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(moe.SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    for code, name in moe.STATUS_NAMES.items():
        assert lib.moe_status_string(code).decode() == name
    assert lib.moe_status_string(99).decode() == "MOE_ERR_UNKNOWN"
    assert lib.moe_version() == 10100


P = ctypes.c_void_p
FAKE = P(0x100000)  # never dereferenced: every case below fails a host check first


def _route(lib, logits=FAKE, dtype=2, T=4, E=8, k=2, idx=FAKE, w=FAKE):
    return lib.moe_route(logits, dtype, T, E, k, 1, idx, w, None, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(logits=None), 1), (dict(idx=None), 1), (dict(w=None), 1),
    (dict(dtype=7), 3), (dict(dtype=-1), 3),
    (dict(k=0), 4), (dict(k=9), 4), (dict(k=-3), 4),
    (dict(E=0, k=1), 2), (dict(E=1025, k=1), 2), (dict(T=-1), 2),
    (dict(T=1 << 31, k=2), 2),
])
def test_route_rejects_bad_arguments(lib, kwargs, status):
    assert _route(lib, **kwargs) == status
    assert lib.moe_last_error().decode() != ""


def test_route_with_no_tokens_is_a_no_op(lib):
    assert _route(lib, logits=None, idx=None, w=None, T=0) == 0


def _dispatch(lib, idx=FAKE, T=4, E=8, k=2, x=None, H=0, counts=FAKE, offsets=FAKE, row_src=FAKE,
              inv=FAKE, xd=None, ws=P(0x200000), ws_bytes=1 << 20, dtype=2):
    return lib.moe_dispatch(idx, T, E, k, x, dtype, H, counts, offsets, row_src, inv, xd, ws,
                            ws_bytes, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(idx=None), 1), (dict(counts=None), 1), (dict(inv=None), 1), (dict(row_src=None), 1),
    (dict(xd=FAKE), 1),                                   # x_dispatched without x
    (dict(xd=FAKE, x=FAKE, H=16, dtype=5), 3),
    (dict(xd=FAKE, x=FAKE, H=0), 2),
    (dict(k=0), 4), (dict(k=9), 4), (dict(E=0, k=1), 2),
    (dict(ws=None), 6), (dict(ws_bytes=0), 6),
    (dict(ws=P(0x200010)), 5),                           # workspace not 256-byte aligned
])
def test_dispatch_rejects_bad_arguments(lib, kwargs, status):
    assert _dispatch(lib, **kwargs) == status


def test_dispatch_workspace_size(lib):
    assert lib.moe_dispatch_workspace_size(4096, 128, 8) >= 16 * 128 * 4
    assert lib.moe_dispatch_workspace_size(-1, 8, 2) == 0
    assert lib.moe_dispatch_workspace_size(0, 8, 2) % 256 == 0


def _route_dispatch(lib, logits=FAKE, ldt=2, T=4, E=8, k=2, idx=FAKE, w=FAKE, x=None, xdt=2, H=0, counts=FAKE,
                    offsets=FAKE, row_src=FAKE, inv=FAKE, xd=None, ws=P(0x200000), ws_bytes=1 << 20):
    return lib.moe_route_dispatch(logits, ldt, T, E, k, 1, idx, w, None, x, xdt, H, counts, offsets, row_src, inv,
                                  xd, ws, ws_bytes, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(logits=None), 1), (dict(idx=None), 1), (dict(w=None), 1), (dict(counts=None), 1),
    (dict(offsets=None), 1), (dict(row_src=None), 1), (dict(inv=None), 1),
    (dict(xd=FAKE), 1),                                   # x_dispatched without x
    (dict(xd=FAKE, x=FAKE, H=16, xdt=7), 3), (dict(xd=FAKE, x=FAKE, H=0), 2),
    (dict(ldt=5), 3), (dict(E=0, k=1), 2), (dict(E=1025), 2), (dict(T=-1), 2),
    (dict(k=0), 4), (dict(k=9), 4),
    (dict(ws=None), 6), (dict(ws_bytes=256), 6),          # the histograms need more than the barrier word
    (dict(ws=P(0x200010)), 5),
])
def test_route_dispatch_rejects_bad_arguments(lib, kwargs, status):
    """Every check runs on the host before anything is enqueued."""
    assert _route_dispatch(lib, **kwargs) == status
    assert lib.moe_last_error().decode() != ""


def test_route_dispatch_workspace_size(lib):
    """256 bytes for the barrier word, then one E-word histogram per block
    (at most one block per token, at most 2048 blocks)."""
    assert lib.moe_route_dispatch_workspace_size(-1, 8) == 0
    assert lib.moe_route_dispatch_workspace_size(4, 0) == 0
    assert lib.moe_route_dispatch_workspace_size(4, 1025) == 0
    for T, E in [(0, 8), (1, 1), (16, 128), (4096, 128), (70000, 8), (300, 1024)]:
        n = lib.moe_route_dispatch_workspace_size(T, E)
        assert n % 256 == 0 and n >= 256 + min(max(T, 1), 2048) * E * 4
    assert lib.moe_route_dispatch_workspace_size(10 ** 6, 128) == lib.moe_route_dispatch_workspace_size(2048, 128)


def test_grouped_route_dispatch_rejects_bad_arguments(lib):
    o = moe.GroupRoutingOptions(2, 4, 2, True, True, 1.0)
    bad = moe.GroupRoutingOptions(0, 4, 2, True, True, 1.0)

    def call(opts=o, E=8, counts=FAKE, ws=P(0x200000), ws_bytes=1 << 20, bias=None):
        return lib.moe_route_sigmoid_grouped_dispatch(FAKE, 2, 4, E, bias, None if opts is None else ctypes.byref(opts),
                                                      FAKE, FAKE, None, None, 2, 0, counts, FAKE, FAKE, FAKE, None,
                                                      ws, ws_bytes, None)

    assert call(opts=None) == 1
    assert call(opts=bad) == 4
    assert call(E=0) == 2
    assert call(counts=None) == 1
    assert call(ws=None) == 6
    assert call(ws=P(0x200010)) == 5
    assert call(bias=P(0x100002)) == 5


@pytest.mark.parametrize("args,status", [
    ((None, 4, FAKE, 4, FAKE, 4, 16, 0), 1), ((FAKE, 4, None, 4, FAKE, 4, 16, 0), 1),
    ((FAKE, 4, FAKE, 4, None, 4, 16, 0), 1), ((FAKE, -1, FAKE, 4, FAKE, 4, 16, 0), 2),
    ((FAKE, 4, FAKE, 4, FAKE, 4, 0, 0), 2), ((FAKE, 4, FAKE, 3, FAKE, 4, 16, 0), 2),  # gather writes 4 rows into 3
    ((FAKE, 3, FAKE, 4, FAKE, 4, 16, 1), 2),                                          # scatter reads 4 rows of 3
])
def test_permute_rows_rejects_bad_arguments(lib, args, status):
    assert lib.moe_permute_rows(*args, None) == status


def test_permute_rows_zero_rows_is_a_no_op(lib):
    assert lib.moe_permute_rows(None, 0, None, 0, None, 0, 16, 0, None) == 0


def _create(lib, gate=FAKE, up=FAKE, down=FAKE, dtype=2, E=8, H=64, I=128, out=True):
    h = ctypes.c_void_p()
    return lib.moe_experts_create(gate, up, down, dtype, E, H, I, ctypes.byref(h) if out else None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(gate=None), 1), (dict(up=None), 1), (dict(down=None), 1), (dict(out=False), 1),
    (dict(dtype=3), 3), (dict(E=0), 2), (dict(E=2000), 2), (dict(H=0), 2), (dict(I=-4), 2),
    (dict(H=20), 5), (dict(I=100), 5),             # 16-bit rows must be 16-byte multiples
    (dict(gate=P(0x100008)), 5),                       # misaligned weights
])
def test_experts_create_rejects_bad_arguments(lib, kwargs, status):
    assert _create(lib, **kwargs) == status


def test_null_handles_are_rejected(lib):
    assert lib.moe_forward(None, FAKE, FAKE, 2, 4, 2, 1, FAKE, None, None, FAKE, 1 << 20, None) == 1
    assert lib.moe_experts_forward_dispatched(None, FAKE, FAKE, 4, FAKE, FAKE, 1 << 20, None) == 1
    assert lib.moe_forward_workspace_size(None, 4, 2) == 0
    assert lib.moe_forward_host(None, FAKE, FAKE, 2, 4, 2, 1, FAKE, None, None, FAKE, 1 << 20, None) == 1
    assert lib.moe_forward_host_workspace_size(None, 4, 2, 2) == 0
    assert lib.moe_experts_forward_dispatched_workspace_size(None, 4) == 0
    lib.moe_experts_destroy(None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(y=None), 1), (dict(dtype=9), 3), (dict(wdt=9), 3), (dict(k=0), 4), (dict(H=0), 2),
])
def test_combine_rejects_bad_arguments(lib, kwargs, status):
    a = dict(y=FAKE, dtype=2, inv=FAKE, w=FAKE, wdt=2, T=4, k=2, H=64, out=FAKE)
    a.update(kwargs)
    assert lib.moe_combine(a["y"], a["dtype"], a["inv"], a["w"], a["wdt"], a["T"], a["k"], a["H"],
                           a["out"], None) == status


def _grouped(lib, logits=FAKE, dtype=2, T=4, E=8, bias=None, opts=None, idx=FAKE, w=FAKE, **opt_kw):
    o = dict(top_k=2, groups=4, selected_groups=2, group_top_two=True, renormalize=True, scale=1.0)
    o.update(opt_kw)
    options = moe.GroupRoutingOptions(**o) if opts is None else opts
    ref = ctypes.byref(options) if options is not False else None
    return lib.moe_route_sigmoid_grouped(logits, dtype, T, E, bias, ref, idx, w, None, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(logits=None), 1), (dict(idx=None), 1), (dict(w=None), 1), (dict(opts=False), 1),
    (dict(dtype=3), 3), (dict(E=0), 2), (dict(E=1025), 2), (dict(T=-1), 2),
    (dict(top_k=0), 4), (dict(top_k=65, E=128, groups=1, selected_groups=1), 4),
    (dict(top_k=5, selected_groups=2), 4),                  # 2 groups of 2 experts hold only 4
    (dict(groups=3), 2), (dict(groups=0), 2), (dict(groups=129, E=258), 2),
    (dict(selected_groups=0), 2), (dict(selected_groups=5), 2),
    (dict(groups=8, selected_groups=2, top_k=1), 2),        # top-two needs two experts per group
    (dict(scale=0.0), 2), (dict(scale=-1.0), 2), (dict(scale=float("inf")), 2), (dict(scale=float("nan")), 2),
    (dict(bias=P(0x100002)), 5),
])
def test_grouped_route_rejects_bad_arguments(lib, kwargs, status):
    assert _grouped(lib, **kwargs) == status
    assert lib.moe_last_error().decode() != ""


def test_grouped_route_accepts_the_edges_on_the_host(lib):
    """T = 0 enqueues nothing, so valid options return MOE_OK without a GPU."""
    assert _grouped(lib, T=0, logits=None, idx=None, w=None) == 0
    assert _grouped(lib, T=0, E=1024, groups=128, selected_groups=128, top_k=64, group_top_two=True) == 0
    assert _grouped(lib, T=0, E=7, groups=1, selected_groups=1, top_k=7, group_top_two=False) == 0


def test_grouped_forward_rejects_bad_arguments(lib):
    o = moe.GroupRoutingOptions(2, 4, 2, True, True, 1.0)
    args = [FAKE, FAKE, 2, 4, None, ctypes.byref(o), FAKE, None, None, FAKE, 1 << 20, None]
    assert lib.moe_forward_sigmoid_grouped(None, *args) == 1
    assert lib.moe_forward_sigmoid_grouped(FAKE, FAKE, FAKE, 2, 4, None, None, FAKE, None, None, FAKE, 1 << 20,
                                           None) == 1


@pytest.mark.parametrize("kwargs,status", [
    (dict(ex=None), 1), (dict(offsets=None), 1), (dict(x=None), 1), (dict(ws=None), 6), (dict(ws=P(0x200010)), 5),
])
def test_gate_up_gather_rejects_bad_arguments(lib, kwargs, status):
    """Checks that run before the handle is read (the rest need a real handle
    and run in the GPU tests)."""
    a = dict(ex=FAKE, x=FAKE, T=4, row_src=FAKE, k=2, offsets=FAKE, rows=8, h=FAKE, ws=P(0x200000))
    a.update(kwargs)
    assert lib.moe_experts_gate_up_gather(a["ex"], a["x"], a["T"], a["row_src"], a["k"], a["offsets"], a["rows"],
                                          a["h"], a["ws"], 1 << 10, None) == status


def _rw(lib, logits=FAKE, dtype=2, T=4, E=8, idx=FAKE, itype=1, k=2, scoring=0, scale=1.0, out=FAKE,
        opts=True):
    o = moe.RouterWeightOptions(scoring, True, scale)
    return lib.moe_router_weights(logits, dtype, T, E, idx, itype, k, ctypes.byref(o) if opts else None, out, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(logits=None), 1), (dict(idx=None), 1), (dict(out=None), 1), (dict(opts=False), 1),
    (dict(dtype=5), 3), (dict(itype=3), 3), (dict(itype=-1), 3),
    (dict(E=0), 2), (dict(E=1025), 2), (dict(T=-1), 2),
    (dict(k=0), 4), (dict(k=9), 4), (dict(k=65, E=100), 4),
    (dict(scoring=2), 2), (dict(scale=0.0), 2), (dict(scale=float("inf")), 2),
])
def test_router_weights_rejects_bad_arguments(lib, kwargs, status):
    assert _rw(lib, **kwargs) == status


def test_training_entry_points_reject_null_buffers(lib):
    o = moe.RouterWeightOptions("sigmoid", False, 1.0)
    assert lib.moe_router_backward(FAKE, 2, 4, 8, FAKE, 1, 2, ctypes.byref(o), None, FAKE, None) == 1
    assert lib.moe_router_backward(FAKE, 2, 0, 8, None, 1, 2, ctypes.byref(o), None, None, None) == 0
    assert lib.moe_combine_backward(FAKE, 2, FAKE, FAKE, FAKE, 2, None, 4, 2, 64, FAKE, FAKE, None) == 1
    assert lib.moe_combine_backward(FAKE, 2, FAKE, None, FAKE, 2, FAKE, 4, 2, 64, FAKE, FAKE, None) == 1
    assert lib.moe_combine_backward(FAKE, 9, FAKE, FAKE, FAKE, 2, FAKE, 4, 2, 64, FAKE, FAKE, None) == 3
    assert lib.moe_combine_backward(FAKE, 2, FAKE, FAKE, FAKE, 2, FAKE, 4, 0, 64, FAKE, FAKE, None) == 4
    assert lib.moe_dispatch_backward(None, 2, FAKE, 4, 2, 64, FAKE, None) == 1
    assert lib.moe_dispatch_backward(FAKE, 2, FAKE, 4, 2, 0, FAKE, None) == 2
    assert lib.moe_experts_forward_training(None, FAKE, FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 10, None) == 1
    assert lib.moe_experts_backward(None, FAKE, FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                    1 << 10, None) == 1
    assert lib.moe_experts_backward_workspace_size(None, 4) == 0


def test_selftest_rejects_bad_limit(lib):
    assert lib.moe_selftest_bounded_wait(0, None) == 2
    assert lib.moe_selftest_bounded_wait(10_000_001, None) == 2


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="no fallback"):
        moe.load_library(tmp_path / "missing.so")
