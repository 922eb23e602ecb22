"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory when they dispatch (for example a plugin driven
through the C ABI by a host framework that owns every device allocation, or a
serving loop whose memory budget is fixed at start-up). It keeps its scratch
in a fixed array inside the library instead of a caller workspace.

Checked through the C ABI against moe_dispatch, bit for bit, on two calls in
a row with different shapes (the second call must not depend on what the
first left in the shared scratch), and the over-size rejection."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"
P = ctypes.c_void_p


def _buffers(T, k, E, H, dtype):
    n = T * k
    return dict(counts=torch.empty(E, dtype=torch.int32, device=DEV),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV),
                row_src=torch.full((n,), -7, dtype=torch.int32, device=DEV),
                inv=torch.empty(n, dtype=torch.int32, device=DEV),
                xd=torch.empty(n, H, dtype=dtype, device=DEV))


def _call(lib, fn, idx, x, E, b, stream, ws=None):
    T, k = idx.shape
    H = x.shape[1]
    dt = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[x.dtype]
    args = [P(idx.data_ptr()), T, E, k, P(x.data_ptr()), dt, H, P(b["counts"].data_ptr()),
            P(b["offsets"].data_ptr()), P(b["row_src"].data_ptr()), P(b["inv"].data_ptr()), P(b["xd"].data_ptr())]
    if ws is not None:
        args += [P(ws.data_ptr()), ws.numel()]
    return fn(*args, stream)


def _case(T, k, E, H, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    p = torch.rand(E, generator=g) ** 4 + 1e-3
    idx = torch.stack([torch.multinomial(p, k, replacement=False, generator=g) for _ in range(T)]).to(torch.int32)
    x = torch.randn(T, H, generator=g).to(dtype)
    return idx.to(DEV), x.to(DEV)


def test_noalloc_dispatch_matches_moe_dispatch_twice(cuda_lib):
    lib = cuda_lib.load_library()
    stream = P(torch.cuda.current_stream().cuda_stream)
    # the first case exceeds the one-block dispatch limit, so the fixed scratch is used
    cases = [(70000, 2, 64, 64, 11, torch.float16), (700, 8, 128, 512, 12, torch.bfloat16)]
    for T, k, E, H, seed, dtype in cases:
        idx, x = _case(T, k, E, H, seed, dtype)
        ref = _buffers(T, k, E, H, dtype)
        ws = torch.empty(lib.moe_dispatch_workspace_size(T, E, k), dtype=torch.uint8, device=DEV)
        assert _call(lib, lib.moe_dispatch, idx, x, E, ref, stream, ws) == 0
        got = _buffers(T, k, E, H, dtype)
        assert _call(lib, lib.moe_dispatch_noalloc, idx, x, E, got, stream) == 0, lib.moe_last_error()
        torch.cuda.synchronize()
        for key in ("counts", "offsets", "row_src", "inv"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["xd"].view(torch.int16), ref["xd"].view(torch.int16))
        assert int(got["counts"].sum()) == T * k
        assert np.array_equal(np.sort(got["inv"].cpu().numpy()), np.arange(T * k))


def test_noalloc_dispatch_rejects_requests_beyond_its_scratch(cuda_lib):
    lib = cuda_lib.load_library()
    stream = P(torch.cuda.current_stream().cuda_stream)
    T, k, E = 600_000, 2, 1024            # ceil(1.2e6 / 2048) * 1024 * 4 B > 1 MiB
    assert lib.moe_dispatch_workspace_size(T, E, k) > (1 << 20)
    idx = torch.zeros(1, 1, dtype=torch.int32, device=DEV)   # never read: the size check comes first
    null = P(idx.data_ptr())
    st = lib.moe_dispatch_noalloc(null, T, E, k, None, 2, 0, null, null, null, null, None, stream)
    assert st == 2 and b"1 MiB" in lib.moe_last_error()
