"""nvfp4_fc2_host_noalloc: the host-to-host FC2 step for callers that cannot
allocate device memory (a plug-in whose host program owns the GPU's memory,
code that must not allocate once it runs).  Its three device buffers come
from a fixed array inside the library instead of from the caller.

Called through the C ABI, twice in a row on different inputs, its host
output must match what nvfp4_fc2_host (the same step on caller-provided
device buffers) returns for the same inputs, under the GEMM tolerance the
other tests use (the same kernels on the same bytes: bit for bit in
practice).  A request larger than the array is refused with a message.

This file is collected last, so that a run which stops at the first failure
has run every other test first; it also passes on its own in a fresh
process."""
import ctypes

import numpy as np
import pytest
import torch

import diffusion_transformer_mlp_gb300 as fc2
import oracle
import synth
from diffusion_transformer_mlp_gb300 import _lib

pytestmark = pytest.mark.gpu

M, N, K = 256, 512, 1024


def _pinned(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()


def _noalloc(L, x_host, w, out_host, stream):
    vp = ctypes.c_void_p
    return L.nvfp4_fc2_host_noalloc(vp(x_host.data_ptr()), M, K, x_host.stride(0), vp(w.qdata.data_ptr()),
                                    vp(w.scales.data_ptr()), vp(w.rec.data_ptr()), N, vp(out_host.data_ptr()),
                                    vp(0), vp(stream.cuda_stream))


def test_noalloc_step_matches_host_step_twice():
    L = _lib.load()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    w = fc2.nvfp4_quantize_weight(
        torch.from_numpy(synth.weight(N, K, seed=40).view(np.int16)).view(torch.bfloat16).cuda())
    inputs = [_pinned(synth.activation(M, K, seed=41)), _pinned(synth.activation(M, K, seed=42))]
    # the reference: nvfp4_fc2_host on device buffers the caller allocates
    refs = [fc2.fc2_host(x, w) for x in inputs]
    outs = [torch.empty(M, N, dtype=torch.bfloat16).pin_memory() for _ in inputs]
    for x, out in zip(inputs, outs):  # two calls in a row on one stream
        st = _noalloc(L, x, w, out, stream)
        assert st == _lib.NVFP4_OK, _lib.last_error()
    stream.synchronize()
    for ref, out in zip(refs, outs):
        ok, worst = oracle.check_gemm_tolerance(out.float().numpy().astype(np.float64),
                                                ref.float().numpy().astype(np.float64))
        assert ok, f"worst error / bound = {worst}"
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert not torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_noalloc_step_refuses_more_than_its_array():
    L = _lib.load()
    vp = ctypes.c_void_p
    m, k, n = 4096, 14336, 5376  # about 390 MB of scratch, far above the array
    buf = torch.zeros(16, dtype=torch.uint8)
    st = L.nvfp4_fc2_host_noalloc(vp(buf.data_ptr()), m, k, 2 * k, vp(16), vp(16), vp(16), n,
                                  vp(buf.data_ptr()), vp(0), vp(0))
    assert st == _lib.NVFP4_EUNSUPPORTED
    assert "bytes of scratch" in _lib.last_error()
