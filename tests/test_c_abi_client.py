"""The C ABI on its own: tests/c_abi_client.c, a plain C program, includes
include/pdecode.h, links libpdecode.so and the CUDA runtime, and calls
decode_paged with device memory it allocates itself -- no Python or torch on
the call path. On the CPU the client must compile and link; on a GPU its
output must match the fp64 oracle on the same inputs (max abs error 2e-3,
exact zeros for rows with no visible key, no device error bits)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from paged_split_decode_gb300 import binding, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_client.c")
TOL = 2e-3


def build_client(out_dir):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    lib_dir = os.path.dirname(binding.lib_path())
    exe = os.path.join(out_dir, "c_abi_client")
    subprocess.run([nvcc, "-O2", "-I", os.path.join(ROOT, "include"), SRC, "-L", lib_dir, "-lpdecode",
                    "-Xlinker", "-rpath", "-Xlinker", lib_dir, "-o", exe], check=True, capture_output=True,
                   text=True)
    return exe


def test_client_compiles_and_links(tmp_path):
    if not os.path.exists(binding.lib_path()):
        pytest.skip("libpdecode.so not built")
    assert os.path.exists(build_client(str(tmp_path)))


def _write_case(d, w, kind, splits):
    num_blocks, bs, Hkv, D = w.k_cache.shape
    params = [w.B, w.Hq, Hkv, D, bs, num_blocks, w.block_table.shape[1], w.qlen, kind, w.window, splits,
              w.scale, w.k_scale, w.v_scale]
    with open(os.path.join(d, "params.txt"), "w") as f:
        f.write(" ".join(repr(float(x)) if isinstance(x, float) else str(int(x)) for x in params) + "\n")
    raw = {"q.bin": w.q.contiguous().view(torch.uint8), "k.bin": w.k_cache.contiguous().view(torch.uint8),
           "v.bin": w.v_cache.contiguous().view(torch.uint8),
           "block_table.bin": w.block_table.contiguous(), "seq_lens.bin": w.seq_lens.contiguous()}
    for name, t in raw.items():
        t.numpy().tofile(os.path.join(d, name))


@pytest.mark.gpu
@pytest.mark.parametrize("kv,splits", [("f16", 0), ("f16", 3), ("fp8", 0)])
def test_client_matches_oracle(tmp_path, kv, splits):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()
    exe = build_client(str(tmp_path))
    w = inputs.make_workload(B=3, Hq=24, Hkv=4, D=256, qlen=1, seq_lens=[1000, 0, 2500], kv=kv, seed=17,
                             name=f"c_client_{kv}")
    kind = binding.PD_KV_FP8_E4M3 if kv == "fp8" else binding.PD_KV_F16
    _write_case(str(tmp_path), w, kind, splits)
    run = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True)
    assert run.returncode == 0, run.stderr
    assert open(os.path.join(tmp_path, "flag.txt")).read().strip() == "0"
    got = np.fromfile(os.path.join(tmp_path, "out.bin"), dtype=np.float16).astype(np.float64)
    ref = oracle.decode_paged(w.q.numpy(), w.k_cache.numpy(), w.v_cache.numpy(), w.block_table.numpy(),
                              w.seq_lens.numpy(), w.scale, w.window, w.qlen, w.k_scale, w.v_scale, w.kv_fp8)
    got = got.reshape(ref.shape)
    assert np.all(np.isfinite(got))
    assert float(np.max(np.abs(got - ref))) <= TOL
    empty = np.all(ref == 0.0, axis=-1)
    assert np.all(got[empty] == 0.0)
