"""Topology of a captured iq_prepare_q call: kernel nodes only -- no
separate RoPE, Hadamard or FP4 kernel, no memcpy and no memset node.  The
quantizer and the GEMM kernel of the call's route are two kernel nodes; with
the quantizer fused into the CTA-pair kernel (iq_set_quant_fusion) that route
is one.  This is the check the TensorRT-LLM PR "Fuse DeepSeek-V4 Indexer
Q projection with CuTe DSL" makes on its fused path (Description: no
standalone RoPE or FP4-concat kernel in the captured graph).

The graph is captured on a torch stream with the driver API (libcuda through
ctypes) so that its nodes can be listed.
"""

import ctypes

import numpy as np
import pytest
import torch

from fp4_fp8_quant_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CU_STREAM_CAPTURE_MODE_THREAD_LOCAL = 1
CU_GRAPH_NODE_TYPE_KERNEL = 0


def _driver():
    cu = ctypes.CDLL("libcuda.so.1")
    begin = getattr(cu, "cuStreamBeginCapture_v2", None) or cu.cuStreamBeginCapture
    begin.argtypes = [ctypes.c_void_p, ctypes.c_int]
    cu.cuStreamEndCapture.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
    cu.cuGraphGetNodes.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_size_t)]
    cu.cuGraphNodeGetType.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    cu.cuGraphDestroy.argtypes = [ctypes.c_void_p]
    return cu, begin


def _node_types(call, stream):
    cu, begin = _driver()
    h = ctypes.c_void_p(stream.cuda_stream)
    assert begin(h, CU_STREAM_CAPTURE_MODE_THREAD_LOCAL) == 0
    try:
        call()
    finally:
        graph = ctypes.c_void_p()
        rc = cu.cuStreamEndCapture(h, ctypes.byref(graph))
    assert rc == 0
    try:
        n = ctypes.c_size_t(0)
        assert cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) == 0
        nodes = (ctypes.c_void_p * n.value)()
        assert cu.cuGraphGetNodes(graph, nodes, ctypes.byref(n)) == 0
        types = []
        for i in range(n.value):
            t = ctypes.c_int(-1)
            assert cu.cuGraphNodeGetType(nodes[i], ctypes.byref(t)) == 0
            types.append(t.value)
        return types
    finally:
        cu.cuGraphDestroy(graph)


@pytest.mark.parametrize("M,fused,kernels", [(24, True, 2), (100, True, 2), (300, True, 1), (4632, True, 1),
                                              (100, False, 2), (300, False, 2), (4632, False, 2)])
def test_captured_prepare_q_kernel_nodes(cuda_device, M, fused, kernels):
    from fp4_fp8_quant_gb300 import iq
    prev = iq.set_quant_fusion(fused)
    try:
        _check_topology(iq, M, kernels)
    finally:
        iq.set_quant_fusion(prev)


def _check_topology(iq, M, kernels):
    x, wq, wsf, pos = W.chain_workload(M, seed=600 + M, outlier_p=0.001, outlier_scale=50.0)
    lat = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    w, ws, p = torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda(), torch.from_numpy(pos).cuda()
    q = torch.empty((M, 4096), dtype=torch.uint8, device="cuda")
    s = torch.empty((M, 256), dtype=torch.uint8, device="cuda")
    work = torch.empty(iq.prepare_q_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work)     # set-up outside the capture
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    types = _node_types(lambda: iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work, stream=stream), stream)
    assert types == [CU_GRAPH_NODE_TYPE_KERNEL] * kernels, types
