"""The oracle against its pins, and the pins' power against planted mistakes.

CPU only.  Every mutant below is ``oracle/oracle.c`` with one plausible mistake
planted by text substitution and compiled into a temporary library; each must
fail at least one pin while the real oracle passes all of them.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

_SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement) -- the first occurrence is replaced.
MUTANTS = [
    ("mask without the history offset (N x N triangle)",
     "const long long n_keys = P + i + 1;", "const long long n_keys = i + 1;"),
    ("mask drops the row's own new key",
     "const long long n_keys = P + i + 1;", "const long long n_keys = P + i;"),
    ("every new row sees every new key",
     "const long long n_keys = P + i + 1;", "const long long n_keys = P + N;"),
    ("GQA head taken modulo instead of by group",
     "const int h = hq / g;", "const int h = hq % H_kv;"),
    ("scale dropped",
     "scores[j] = scale * dot;", "scores[j] = dot;"),
    ("softmax weights not normalised",
     "for (int d = 0; d < D; ++d) o[d] /= wsum;", "for (int d = 0; d < D; ++d) o[d] /= 1.0;"),
    ("value rows read from the K cache",
     "o[d] += w * (v_scale * load_elem(v_cache, v_row + d, kv_dtype));",
     "o[d] += w * (v_scale * load_elem(k_cache, v_row + d, kv_dtype));"),
    ("every new row uses the first query row",
     "* (size_t)N + (size_t)i) * (size_t)D;\n                const size_t kv_head",
     "* (size_t)N + (size_t)0) * (size_t)D;\n                const size_t kv_head"),
    ("append writes the new tokens at the start of the row",
     "(size_t)(P + i)) * row;", "(size_t)(i)) * row;"),
    ("bf16 widened with the wrong shift",
     "[idx] << 16;", "[idx] << 15;"),
    ("fp16 exponent bias off by one",
     "ldexp((double)(1024 + frac), expo - 25)", "ldexp((double)(1024 + frac), expo - 24)"),
    ("e4m3 exponent bias off by one",
     "v = ldexp((double)(8 + frac), expo - 10);", "v = ldexp((double)(8 + frac), expo - 9);"),
    ("e4m3 ties rounded away from even",
     "(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    ("e4m3 append without the scale",
     "e4m3_from_float(kx / k_scale)", "e4m3_from_float(kx)"),
    ("e4m3 attention ignores the V scale",
     "o[d] += w * (v_scale * load_elem(v_cache, v_row + d, kv_dtype));",
     "o[d] += w * (load_elem(v_cache, v_row + d, kv_dtype));"),
    ("fp16 subnormals scaled as normals",
     "v = ldexp((double)frac, -24);", "v = ldexp((double)(1024 + frac), -25);"),
    ("size formula without the factor 2 for K and V",
     "(2LL * L * H_kv", "(1LL * L * H_kv"),
    ("paged: page slot and page index swapped",
     "const long long j = t / page_size;", "const long long j = t % page_size;"),
    ("paged: block table read with the wrong row stride",
     "block_table[(size_t)b * (size_t)max_pages + (size_t)j]", "block_table[(size_t)b + (size_t)j]"),
    ("paged: pages gathered as token-major [page, slot, head]",
     "const size_t src = (((size_t)page * H_kv + h) * (size_t)page_size + (size_t)(t % page_size)) * row;",
     "const size_t src = (((size_t)page * page_size + (size_t)(t % page_size)) * H_kv + h) * row;"),
    ("paged: append writes the token at the page start",
     "(size_t)page_size + (size_t)(t % page_size)) * row;\n                const size_t src",
     "(size_t)page_size + (size_t)(0)) * row;\n                const size_t src"),
]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(oracle_lib, pin):
    pin(oracle_lib)


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(mutant_dir, name, old, new):
    with open(_SRC) as f:
        src = f.read()
    assert old in src, f"mutation anchor not found: {old!r}"
    tag = str(abs(hash(name)))
    path_c = os.path.join(mutant_dir, f"mutant_{tag}.c")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new, 1))
    lib = oracle.Oracle(oracle.compile_library(path_c, os.path.join(mutant_dir, f"mutant_{tag}.so")))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake: {name}"
