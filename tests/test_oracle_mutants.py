"""The oracle's pins have teeth: plant one mistake at a time in a copy of the
oracle's C source, build the copy on the CPU, and check that at least one pin
in test_oracle.py fails on it. The oracle itself is never modified."""
import importlib.util
import os
import shutil
import sys

import pytest

import test_oracle as pins
import test_oracle_writer as writer_pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in pd_oracle.c, planted replacement)
MUTANTS = [
    ("gqa_index", "int kh = h / G;", "int kh = h % d->Hkv;"),
    ("window_off_by_one", "if (window > 0 && p - window + 1 > 0) first = p - window + 1;",
     "if (window > 0 && p - window > 0) first = p - window;"),
    ("causal_position", "long p = (long)L - qlen + i;", "long p = (long)L - 1 - i;"),
    ("scale_dropped", "s[j - lo] = scale * dot;", "s[j - lo] = dot;"),
    ("softmax_sign", "double w = exp(s[j - lo] - M);", "double w = exp(M - s[j - lo]);"),
    ("f16_subnormal_exponent", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("e4m3_bias", "v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 9);"),
    ("combine_weight_sign", "double w = (ms == -INFINITY) ? 0.0 : exp(ms - M);",
     "double w = (ms == -INFINITY) ? 0.0 : exp(M - ms);"),
    ("online_rescale_missing", "l *= a;", "l *= 1.0;"),
    ("v_scale_unused", "o[x] += w * cache_at(d, v_cache, d->v_scale, blk, slot, kh, x);",
     "o[x] += w * cache_at(d, v_cache, d->k_scale, blk, slot, kh, x);"),
    ("int8_unsigned", "double pdo_i8_to_f64(uint8_t c) { return (double)(int8_t)c; }",
     "double pdo_i8_to_f64(uint8_t c) { return (double)c; }"),
    ("split_chunk_bound", "if (cb1 > first_block + n_blocks) cb1 = first_block + n_blocks;",
     "if (cb1 > first_block + n_blocks - 1) cb1 = first_block + n_blocks - 1;"),
    ("writer_scale_multiplies", "float kq = (float)(b16 ? pdo_bf16_to_f64(kx) : pdo_f16_to_f64(kx)) / ks;",
     "float kq = (float)(b16 ? pdo_bf16_to_f64(kx) : pdo_f16_to_f64(kx)) * ks;"),
    ("e4m3_ties_away", "if (d < best_d || (d == best_d && (c & 1) == 0)) {",
     "if (d <= best_d) {"),
    ("i8_ties_up", "r = (fmod(f, 2.0) == 0.0) ? f : f + 1.0;", "r = f + 1.0;"),
    ("i8_clamp_asymmetric", "if (v <= -127.0) return -127;", "if (v <= -128.0) return -128;"),
    ("writer_offset_transposed", "long dst = (blk * d->block_size + off) * row;",
     "long dst = (off * d->num_blocks + blk) * row;"),
    ("writer_padding_written", "if (slot < 0) continue;", "if (slot < 0) slot = -slot;"),
    ("bf16_exponent_bias", "v = ldexp((double)(128 + f), e - 134);", "v = ldexp((double)(128 + f), e - 133);"),
    ("bf16_q_read_as_f16", "return d->kv_kind >= 3 ? pdo_bf16_to_f64(bits) : pdo_f16_to_f64(bits);",
     "return pdo_f16_to_f64(bits);"),
    ("bf16q_e4m3_cache_read_as_f16", "if (d->kv_kind == 1 || d->kv_kind == 4)\n",
     "if (d->kv_kind == 1)\n"),
    ("writer_bf16_tokens_read_as_f16", "const int b16 = d->kv_kind >= 4;", "const int b16 = 0;"),
    ("writer_bf16_cache_quantised", "if (d->kv_kind == 0 || d->kv_kind == 3) {", "if (d->kv_kind == 0) {"),
    ("writer_bf16_cache_byte_stores", "((uint16_t*)k_cache)[dst + e] = kx;",
     "if (d->kv_kind == 3) ((uint8_t*)k_cache)[dst + e] = (uint8_t)kx; else ((uint16_t*)k_cache)[dst + e] = kx;"),
]


def _load_mutant(tmp_path, name, old, new):
    src = open(os.path.join(ROOT, "oracle", "pd_oracle.c")).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    pkg = tmp_path / f"oracle_{name}"
    pkg.mkdir()
    (pkg / "pd_oracle.c").write_text(src.replace(old, new))
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), pkg / "__init__.py")
    spec = importlib.util.spec_from_file_location(f"oracle_{name}", pkg / "__init__.py",
                                                  submodule_search_locations=[str(pkg)])
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod
    spec.loader.exec_module(mod)
    mod.build(force=True)
    return mod


def _pin_calls():
    import json
    cases = json.load(open(os.path.join(pins.GOLDEN, "closed_forms.json")))["cases"]
    calls = [(pins.test_f16_decoder_every_pattern, {}), (pins.test_e4m3fn_decoder_every_code, {}),
             (pins.test_e4m3fn_spec_points, {}), (pins.test_int8_decoder_every_code, {}),
             (pins.test_bf16_decoder_every_pattern, {})]
    calls += [(pins.test_golden_closed_forms, {"case": c}) for c in cases]
    calls += [(pins.test_oracle_matches_dense_bruteforce, {"ci": ci, "kv": kv})
              for ci in range(len(pins.TINY)) for kv in pins.KV_KINDS]
    calls += [(pins.test_split_mode_matches_one_shot, {"ci": ci, "kv": "f16"}) for ci in (2, 5)]
    calls += [(pins.test_combine_edge_cases, {}), (pins.test_split_partials_recombine, {})]
    calls += [(writer_pins.test_e4m3fn_encoder_golden_points, {}),
              (writer_pins.test_i8_encoder_golden_points, {}),
              (writer_pins.test_e4m3fn_encoder_matches_torch_cast, {}),
              (writer_pins.test_i8_encoder_matches_numpy, {})]
    calls += [(writer_pins.test_writer_layout_and_codes, {"kind": k}) for k in writer_pins.KINDS]
    return calls


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    mod = _load_mutant(tmp_path, name, old, new)
    caught = []
    for fn, kw in _pin_calls():
        try:
            fn(mod, **kw)
        except (AssertionError, ValueError) as e:  # a pin fired
            caught.append(fn.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
