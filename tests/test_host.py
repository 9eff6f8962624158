"""Host-side checks that need no GPU: the library builds for sm_103a, loads,
exports exactly what include/pdecode.h declares, and its pure host functions
(planning, workspace sizing, argument validation) behave as documented."""
import ctypes
import os
import re
import subprocess

import pytest

from paged_split_decode_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pdecode.h")).read()
    src = re.sub(r"#define PD_API.*", "", src)
    return sorted(set(re.findall(r"^PD_API\s+[\w\s\*]*?\b(\w+)\s*\(", src, re.M)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", binding.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted(line.split()[-1] for line in out.splitlines() if line.strip())
    assert exported == declared_functions()


def test_build_targets_sm_103a_only():
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    for code in range(8):
        assert binding.status_str(code)
    assert binding.status_str(0) == "ok"


def _dims(**kw):
    base = dict(B=32, Hq=24, Hkv=4, D=256, block_size=16, num_blocks=10000, max_blocks_per_seq=256)
    base.update(kw)
    return binding.make_dims(**base)


def test_workspace_and_grid_plans(lib):
    d = _dims()
    up = lambda x: (x + 255) // 256 * 256
    # one row tile per head and Hkv % 4 == 0: head-group tiles (fp16 D=256:
    # two KV heads per tile), one persistent CTA per SM; balanced: two
    # partial slots per CTA, 2 heads x 8 padded rows of (m, l) and of D floats
    # per slot (a unit's pieces follow from the sequence lengths: nothing else
    # is stored)
    assert binding.grid_ctas(d, 1, 0, sm_count=152) == 152
    ws = binding.workspace_bytes(d, 1, 0, sm_count=152)
    assert ws == up(304 * 16 * 2 * 4) + 304 * 16 * 256 * 4
    # no split: no workspace at all; one CTA per unit (B * Hkv / 2 units)
    assert binding.workspace_bytes(d, 1, 1, sm_count=152) == 0
    assert binding.grid_ctas(d, 1, 1, sm_count=152) == 64
    # fixed split: units * S slots
    assert binding.workspace_bytes(d, 1, 3, sm_count=152) == \
        up(192 * 16 * 2 * 4) + 192 * 16 * 256 * 4
    assert binding.grid_ctas(d, 1, 3, sm_count=152) == 152
    # fp8 D=256: four KV heads per tile, 32 rows per slot, B * Hkv / 4 units
    d8 = _dims(kv_fp8=True)
    assert binding.workspace_bytes(d8, 1, 0, sm_count=152) == \
        up(304 * 32 * 2 * 4) + 304 * 32 * 256 * 4
    assert binding.grid_ctas(d8, 1, 1, sm_count=152) == 32
    # per-head tiles (Hkv = 2): two CTAs per SM, 8 padded rows per slot
    d2 = _dims(Hq=12, Hkv=2)
    assert binding.grid_ctas(d2, 1, 0, sm_count=152) == 304
    assert binding.workspace_bytes(d2, 1, 0, sm_count=152) == \
        up(608 * 8 * 2 * 4) + 608 * 8 * 256 * 4
    assert binding.grid_ctas(d2, 1, 1, sm_count=152) == 64
    # qlen 3 x G 6 = 18 rows -> three row tiles of 8, per-head tiles
    ws3 = binding.workspace_bytes(_dims(B=8), 3, 0, sm_count=152)
    assert ws3 == up(608 * 24 * 2 * 4) + 608 * 24 * 256 * 4


def test_automatic_split_for_few_units(lib):
    up = lambda x: (x + 255) // 256 * 256
    # B=1..3 at L <= 4096 (2..6 units of at most 257 tiles, <= 24 tiles per
    # CTA slot): each unit is cut into floor(128 / units) pieces, one per CTA
    for B, units in ((1, 2), (2, 4), (3, 6)):
        assert binding.grid_ctas(_dims(B=B), 1, 0, sm_count=152) == units * (128 // units)
        # the workspace stays the balanced split's (two slots per CTA slot)
        assert binding.workspace_bytes(_dims(B=B), 1, 0, sm_count=152) == \
            up(304 * 16 * 2 * 4) + 304 * 16 * 256 * 4
    # long tables (bandwidth-bound): balanced over every CTA slot
    assert binding.grid_ctas(_dims(B=1, max_blocks_per_seq=2048), 1, 0, sm_count=152) == 152
    assert binding.grid_ctas(_dims(B=8), 1, 0, sm_count=152) == 152
    # e4m3 verify (tensor-memory kernel, 32 per-head units): fixed, 4 pieces each
    assert binding.grid_ctas(_dims(B=8, kv_fp8=True, max_blocks_per_seq=512), 3, 0, sm_count=152) == 128


@pytest.mark.parametrize("kw,qlen", [
    (dict(D=64), 1), (dict(D=96), 1), (dict(block_size=8), 1), (dict(Hq=24, Hkv=5), 1),
    (dict(Hq=40, Hkv=1), 1), (dict(), 9), (dict(Hq=24, Hkv=4), 6),
])
def test_unsupported_or_bad_shapes_are_rejected(lib, kw, qlen):
    assert binding.workspace_bytes(_dims(**kw), qlen, 0, sm_count=152) == 0
    assert binding.grid_ctas(_dims(**kw), qlen, 0, sm_count=152) == 0


def _call(lib, dims, q=16, k=16, v=16, bt=16, sl=16, out=16, qlen=1, splits=0, ws=None, wsb=0, flag=None):
    return lib.decode_paged(q, k, v, bt, sl, 0.1, 0, qlen, splits, out, ctypes.byref(dims), ws, wsb,
                            flag, None)


def test_decode_paged_validates_before_touching_the_device(lib):
    d = _dims()
    assert _call(lib, _dims(D=64)) == 4          # unsupported head size
    assert _call(lib, _dims(Hkv=5)) == 2         # Hq % Hkv
    bad = _dims()
    bad.kv_dtype = 7
    assert _call(lib, bad) == 3                  # dtype
    i8 = _dims()
    i8.kv_dtype = 2                              # int8 is a known kind
    assert binding.workspace_bytes(i8, 1, 0, sm_count=152) > 0
    assert _call(lib, d, q=None) == 1            # null pointer
    assert _call(lib, d, out=None) == 1
    assert _call(lib, d, q=0x1008) == 5          # misaligned (not 16 B)
    assert _call(lib, d, bt=0x1002) == 5
    assert _call(lib, d, splits=-1) == 2
    assert _call(lib, _dims(B=0)) == 0           # nothing to do


def test_combine_validates(lib):
    assert lib.decode_paged_combine(16, 16, 16, 4, 0, 256, 16, None) == 2   # S = 0
    assert lib.decode_paged_combine(16, 16, 16, 4, 2, 100, 16, None) == 2   # D % 8
    assert lib.decode_paged_combine(None, 16, 16, 4, 2, 256, 16, None) == 1
    assert lib.decode_paged_combine(16, 16, 0x1004, 4, 2, 256, 16, None) == 5
    assert lib.decode_paged_combine(16, 16, 16, 0, 2, 256, 16, None) == 0   # no rows


@pytest.mark.parametrize("byte", ["fp8", "int8"])
@pytest.mark.parametrize("qlen,kw", [(1, {}), (1, dict(Hq=12, Hkv=2)), (3, dict(B=8)), (2, dict(D=128))])
def test_bf16_q_byte_kinds_plan_like_their_fp16_q_kinds(lib, byte, qlen, kw):
    """A bfloat16 q over fp8 / int8 caches runs the same shapes as an fp16 q:
    the same grids and workspaces, for every split mode."""
    flag = {"kv_fp8": True} if byte == "fp8" else {"kv_int8": True}
    f16q = _dims(**flag, **kw)
    bq = _dims(**flag, q_bf16=True, **kw)
    assert bq.kv_dtype == f16q.kv_dtype + 3
    for S in (0, 1, 3):
        assert binding.grid_ctas(bq, qlen, S, sm_count=152) == binding.grid_ctas(f16q, qlen, S, sm_count=152) > 0
        assert binding.workspace_bytes(bq, qlen, S, sm_count=152) == \
            binding.workspace_bytes(f16q, qlen, S, sm_count=152)


def test_bf16_q_needs_a_bf16_or_byte_cache():
    with pytest.raises(TypeError):
        _dims(q_bf16=True)
    bad = _dims(kv_fp8=True, q_bf16=True)
    bad.kv_dtype = 6
    assert binding.workspace_bytes(bad, 1, 0, sm_count=152) == 0
