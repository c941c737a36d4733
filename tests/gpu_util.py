"""Shared helpers of the GPU parity tests: tolerances and comparison with the oracle."""
import numpy as np
import torch

# Output tolerance |gpu - oracle| <= atol + rtol * |oracle| per storage dtype, and the
# absolute tolerance on the natural-log LSE.
TOL = {torch.bfloat16: (2e-2, 2e-2), torch.float16: (5e-3, 5e-3), torch.float32: (1e-5, 1e-5)}
LSE_TOL = 1e-3


def assert_matches_oracle(o, lse, ref_o, ref_lse, dtype, what=""):
    atol, rtol = TOL[dtype]
    o = o.float().cpu().numpy().astype(np.float64)
    ref_o = np.asarray(ref_o, dtype=np.float64)
    assert o.shape == ref_o.shape, (o.shape, ref_o.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    excess = np.abs(o - ref_o) - (atol + rtol * np.abs(ref_o))
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"{what}: output off by {np.abs(o - ref_o)[worst]:.3e} at {worst} "
                               f"(gpu {o[worst]:.5f}, oracle {ref_o[worst]:.5f})")
    if lse is not None:
        lse = lse.float().cpu().numpy().astype(np.float64)
        ref_lse = np.asarray(ref_lse, dtype=np.float64)
        both_inf = np.isneginf(lse) & np.isneginf(ref_lse)
        with np.errstate(invalid="ignore"):
            d = np.where(both_inf, 0.0, np.abs(lse - ref_lse))
        assert np.isfinite(d).all() and d.max() <= LSE_TOL, f"{what}: lse off by {np.nanmax(d):.3e}"


def kernel_nodes(fn, stream):
    """Capture fn's launches on `stream` into a CUDA graph through the driver API (the
    kernels come from this library's own runtime, so no profiler is involved) and
    return (function name, grid, block) of every kernel node."""
    import ctypes
    cu = ctypes.CDLL("libcuda.so.1")
    vp = ctypes.c_void_p
    h, graph = vp(stream.cuda_stream), vp()
    assert cu.cuStreamBeginCapture_v2(h, 2) == 0  # CU_STREAM_CAPTURE_MODE_RELAXED
    try:
        fn()
    finally:
        assert cu.cuStreamEndCapture(h, ctypes.byref(graph)) == 0
    try:
        n = ctypes.c_size_t(0)
        assert cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) == 0
        nodes = (vp * max(n.value, 1))()
        assert cu.cuGraphGetNodes(graph, nodes, ctypes.byref(n)) == 0
        out = []
        for i in range(n.value):
            t = ctypes.c_int(-1)
            assert cu.cuGraphNodeGetType(vp(nodes[i]), ctypes.byref(t)) == 0
            if t.value != 0:  # CU_GRAPH_NODE_TYPE_KERNEL
                continue
            # CUDA_KERNEL_NODE_PARAMS_v2: func, grid[3], block[3], shared bytes, params, extra, kern, ctx
            par = (ctypes.c_uint64 * 16)()
            assert cu.cuGraphKernelNodeGetParams_v2(vp(nodes[i]), par) == 0
            dims = (ctypes.c_uint32 * 32).from_buffer(par)
            name = ctypes.c_char_p()
            if par[0]:
                assert cu.cuFuncGetName(ctypes.byref(name), vp(par[0])) == 0
            else:
                assert cu.cuKernelGetName(ctypes.byref(name), vp(par[7])) == 0
            out.append((name.value.decode(), tuple(dims[2:5]), tuple(dims[5:8])))
        return out
    finally:
        cu.cuGraphDestroy(graph)
