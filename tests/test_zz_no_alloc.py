"""The scratch-free entry point, decode_paged_static_scratch.

Callers that cannot allocate device memory (code inside an allocator's
callbacks, plugin hosts that hand out no device buffers, processes whose
device footprint is fixed after start-up) use this entry point: it runs the
same decode as decode_paged but keeps its split-K partials in a scratch
array built into the library instead of a caller-provided workspace.

The test calls it through the C ABI (ctypes) twice in a row and compares each
result with decode_paged's on the same inputs and with the fp64 oracle, within
the 2e-3 tolerance the parity tests use, and checks that the second call
takes no device memory (the first call on a device may: that is when CUDA's
lazy module loading brings the array in). This file is collected last so that
a stop-at-first-failure run has already run every other test; it also passes
on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_split_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 2e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = binding.load()
    P = ctypes.c_void_p
    fn = lib.decode_paged_static_scratch
    fn.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                   ctypes.POINTER(binding.PdDims), P, P]
    fn.restype = ctypes.c_int
    return lib


def _device(w):
    k, v = w.k_cache.to(DEV), w.v_cache.to(DEV)
    if w.kv_int8:
        k, v = k.view(torch.int8), v.view(torch.int8)
    return (w.q.to(DEV), k, v, w.block_table.to(DEV), w.seq_lens.to(DEV))


def _call_static(lib, w, t, num_splits, out, flag):
    q, k, v, bt, sl = t
    dims = binding.dims_of(q, k, bt, w.qlen, None, w.k_scale, w.v_scale)
    stream = torch.cuda.current_stream().cuda_stream
    return lib.decode_paged_static_scratch(q.data_ptr(), k.data_ptr(), v.data_ptr(), bt.data_ptr(),
                                           sl.data_ptr(), w.scale, w.window, w.qlen, num_splits,
                                           out.data_ptr(), ctypes.byref(dims), flag.data_ptr(),
                                           stream)


def _oracle(w):
    return oracle.decode_paged(w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(),
                               w.block_table.numpy(), w.seq_lens.numpy(), w.scale, w.window,
                               w.qlen, w.k_scale, w.v_scale, w.kv_fp8, kv_int8=w.kv_int8)


def test_static_scratch_matches_decode_paged_and_the_oracle(lib):
    # balanced split over every SM: the split-K partials live in the scratch
    # (fp16 KV; and e4m3 KV with three query tokens, the tensor-memory kernel)
    cases = [inputs.gqa_d256(2),
             inputs.make_workload(B=5, Hq=32, Hkv=8, D=128, qlen=1,
                                  seq_lens=[3000, 0, 17, 900, 4096], seed=31),
             inputs.make_workload(B=3, Hq=24, Hkv=4, D=256, qlen=3, seq_lens=[5000, 2, 777],
                                  kv="fp8", seed=33)]
    for w in cases:
        t = _device(w)
        q, k, v, bt, sl = t
        want = binding.decode_paged(q, k, v, bt, sl, w.scale, w.window, w.qlen, 0,
                                    k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        ref = _oracle(w).reshape(-1, w.D)
        outs = [torch.full_like(q, float("nan")) for _ in range(2)]
        flags = [torch.zeros(1, dtype=torch.int32, device=DEV) for _ in range(2)]
        torch.cuda.synchronize()
        for n in range(2):  # two calls in a row share the scratch
            free0 = torch.cuda.mem_get_info()[0]
            assert _call_static(lib, w, t, 0, outs[n], flags[n]) == 0
            torch.cuda.synchronize()
            if n == 1:
                assert torch.cuda.mem_get_info()[0] == free0, "the second call took device memory"
            assert int(flags[n].item()) == 0
            got = outs[n].float()
            err = (got - want.float()).abs().max().item()
            assert err <= TOL, f"{w.name}: max abs difference from decode_paged {err}"
            g = got.cpu().numpy().reshape(-1, w.D)
            assert np.all(np.isfinite(g)), f"{w.name}: non-finite output"
            err_ref = float(np.max(np.abs(g - ref)))
            assert err_ref <= TOL, f"{w.name}: max abs error against the oracle {err_ref}"


def test_static_scratch_rejects_plans_beyond_its_size(lib):
    # a fixed split of 8 over 64 sequences x 8 KV heads needs 4096 partial slots
    # of 8 rows x 256 floats (32 MiB) plus their (m, l) pairs: more than the
    # scratch
    w = inputs.make_workload(B=64, Hq=8, Hkv=8, D=256, qlen=1, seq_lens=[64] * 64, seed=32)
    t = _device(w)
    need = binding.workspace_bytes(binding.dims_of(t[0], t[1], t[3], w.qlen), w.qlen, 8)
    assert need > (32 << 20)
    out = torch.empty_like(t[0])
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _call_static(lib, w, t, 8, out, flag) == 6  # PD_ERR_WORKSPACE
