"""The C-ABI library loads and exports every declared entry point; host-side
argument checks return their documented status before touching a GPU.  CPU only."""
import ctypes
import os
import re

import pytest

from helpers import *  # noqa: F401,F403

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvd.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "kv_cache_bytes.txt")


@pytest.fixture(scope="module")
def lib():
    from kv_cache_decode_append_gb300 import build as kbuild
    from kv_cache_decode_append_gb300 import kvd
    kbuild.build()
    return kvd.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvd_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("kvd_append", "kvd_decode_attention", "kvd_decode_workspace_bytes", "kvd_decode_plan",
              "kvd_workspace_init", "kvd_cache_bytes", "kvd_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib.path)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_cache_bytes_matches_the_pages_table(lib):
    import kv_cache_decode_append_gb300 as kvd
    units = {"B": 1, "KiB": 1024, "MiB": 1024 ** 2}
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        L, B, H, D, T, s, expected, unit, match = line.split()
        got = kvd.kvd_cache_bytes(int(L), int(B), int(H), int(D), int(T), "f32" if s == "4" else "bf16")
        got /= units[unit]
        if match == "exact":
            assert got == float(expected)
        else:
            assert round(got, len(expected.split(".")[1])) == float(expected)
    assert kvd.kvd_cache_bytes(-1, 1, 1, 1, 1, "f32") == 0


def test_status_strings(lib):
    import kv_cache_decode_append_gb300 as kvd
    assert kvd.kvd_status_string(0) == "KVD_OK"
    assert kvd.kvd_status_string(4) == "KVD_ERR_WORKSPACE"
    assert kvd.kvd_status_string(99) == "KVD_UNKNOWN_STATUS"


# Fake, 256-byte aligned addresses: every call below must be rejected on the
# host before any pointer is dereferenced or any CUDA call is made.
A = 1 << 20


def _attn(lib, q=A, k=A, v=A, out=A, past=A, B=1, H_q=4, H_kv=2, T_max=64, D=64, N=1,
          max_past=10, dtype=1):
    return lib.kvd_decode_attention(q, k, v, out, past, B, H_q, H_kv, T_max, D, N, max_past,
                                    0.0, dtype, None, 0, None, None)


def _append(lib, k=A, v=A, kn=A, vn=A, past=A, B=1, H_kv=2, T_max=64, D=64, N=1, max_past=10, dtype=1):
    return lib.kvd_append(k, v, kn, vn, past, B, H_kv, T_max, D, N, max_past, dtype, None, None)


def test_attention_argument_errors(lib):
    assert _attn(lib, q=0) == 1
    assert _attn(lib, past=0) == 1
    assert _attn(lib, H_q=3, H_kv=2) == 1
    assert _attn(lib, N=0) == 1
    assert _attn(lib, B=-1) == 1
    assert _attn(lib, max_past=-1) == 1
    assert _attn(lib, D=96) == 3
    assert _attn(lib, dtype=7) == 3
    assert _attn(lib, H_q=16, H_kv=1, N=65) == 3     # 1040 query rows per KV head
    assert _attn(lib, q=A + 8) == 1                   # misaligned
    assert _attn(lib, out=A + 4) == 1
    assert _attn(lib, max_past=64, N=1, T_max=64) == 2  # P + N > T_max
    assert _attn(lib, B=0) == 0                       # empty batch: nothing to do


def test_append_argument_errors(lib):
    assert _append(lib, k=0) == 1
    assert _append(lib, vn=0) == 1
    assert _append(lib, N=0) == 1
    assert _append(lib, T_max=0) == 1
    assert _append(lib, dtype=9) == 3
    assert _append(lib, D=3, dtype=1) == 3            # 6-byte rows are not whole 16-byte chunks
    assert _append(lib, kn=A + 2) == 1
    assert _append(lib, max_past=60, N=5, T_max=64) == 2
    assert _append(lib, B=0) == 0


def test_workspace_query_rejects_bad_shapes(lib):
    assert lib.kvd_decode_workspace_bytes(1, 3, 2, 64, 1, 10, 1) == 0
    assert lib.kvd_decode_workspace_bytes(1, 4, 2, 80, 1, 10, 1) == 0
    assert lib.kvd_decode_workspace_bytes(1, 4, 2, 64, 0, 10, 1) == 0


def _paged_attn(lib, q=A, k=A, v=A, out=A, table=A, past=A, B=1, H_q=4, H_kv=2, D=64, N=1,
                page_size=64, max_pages=4, num_pages=8, max_past=10, dtype=1):
    return lib.kvd_paged_decode_attention(q, k, v, out, table, past, B, H_q, H_kv, D, N, page_size,
                                          max_pages, num_pages, max_past, 0.0, dtype, None, 0, None, None)


def _paged_append(lib, k=A, v=A, kn=A, vn=A, table=A, past=A, B=1, H_kv=2, D=64, N=1, page_size=64,
                  max_pages=4, num_pages=8, max_past=10, dtype=1):
    return lib.kvd_paged_append(k, v, kn, vn, table, past, B, H_kv, D, N, page_size, max_pages, num_pages,
                                max_past, dtype, None, None)


def test_paged_argument_errors(lib):
    for call in (_paged_attn, _paged_append):
        assert call(lib, table=0) == 1                    # no block table
        assert call(lib, page_size=48) == 1               # not a power of two
        assert call(lib, page_size=32) == 1               # smaller than a tile
        assert call(lib, max_pages=0) == 1
        assert call(lib, num_pages=0) == 1
        assert call(lib, max_past=256, N=1) == 2          # 4 pages x 64 tokens hold 256
        assert call(lib, k=A + 8) == 1                    # misaligned pages
        assert call(lib, B=0) == 0
    assert _paged_attn(lib, D=96) == 3
    assert _paged_attn(lib, H_q=3) == 1
    assert lib.kvd_paged_decode_step(A, A, A, 0, A, A, A, A, 1, 4, 2, 64, 1, 64, 4, 8, 10, 0.0, 1,
                                     None, 0, None, None) == 1   # k_new missing


def _append8(lib, k=A, v=A, kn=A, vn=A, past=A, B=1, H_kv=2, T_max=64, D=64, N=1, max_past=10, new_dtype=1,
             k_scale=0.5, v_scale=0.5):
    return lib.kvd_append_e4m3(k, v, kn, vn, past, B, H_kv, T_max, D, N, max_past, new_dtype, k_scale, v_scale,
                               None, None)


def _attn8(lib, q=A, k=A, v=A, out=A, past=A, B=1, H_q=4, H_kv=2, T_max=64, D=128, N=1, max_past=10,
           k_scale=0.5, v_scale=0.5):
    return lib.kvd_decode_attention_e4m3(q, k, v, out, past, B, H_q, H_kv, T_max, D, N, max_past, 0.0, k_scale,
                                         v_scale, None, 0, None, None)


def test_e4m3_argument_errors(lib):
    assert _append8(lib, new_dtype=3) == 3              # new rows are fp32 / bf16 / fp16, not codes
    assert _append8(lib, k=0) == 1
    assert _append8(lib, k_scale=0.0) == 1              # scales: finite and positive
    assert _append8(lib, v_scale=float("inf")) == 1
    assert _append8(lib, k_scale=float("nan")) == 1
    assert _append8(lib, D=8) == 3                      # 8 codes are not a whole 16-byte chunk
    assert _append8(lib, kn=A + 4) == 1                 # misaligned
    assert _append8(lib, max_past=60, N=5, T_max=64) == 2
    assert _append8(lib, B=0) == 0
    assert _attn8(lib, k_scale=-1.0) == 1
    assert _attn8(lib, v_scale=float("nan")) == 1
    assert _attn8(lib, q=A + 8) == 1
    assert _attn8(lib, D=96) == 3
    assert _attn8(lib, H_q=16, H_kv=1, N=65) == 3       # 1040 query rows per KV head
    assert _attn8(lib, max_past=64, T_max=64) == 2
    assert _attn8(lib, B=0) == 0
    assert _attn(lib, dtype=3) == 3                     # an E4M3 cache only through the _e4m3 calls (scales)
    assert lib.kvd_decode_step_e4m3(A, A, A, 0, A, A, A, 1, 4, 2, 64, 128, 1, 10, 0.0, 0.5, 0.5,
                                    None, 0, None, None) == 1   # k_new missing
    assert lib.kvd_decode_step_e4m3(A, A, A, A, A + 8, A, A, 1, 4, 2, 64, 128, 1, 10, 0.0, 0.5, 0.5,
                                    None, 0, None, None) == 1   # v_new misaligned


def test_decode_step_argument_errors(lib):
    def step(kn=A, vn=A, **kw):
        args = dict(q=A, k=A, v=A, out=A, past=A, B=1, H_q=4, H_kv=2, T_max=64, D=64, N=1, max_past=10, dtype=1)
        args.update(kw)
        return lib.kvd_decode_step(args["q"], args["k"], args["v"], kn, vn, args["out"], args["past"], args["B"],
                                   args["H_q"], args["H_kv"], args["T_max"], args["D"], args["N"],
                                   args["max_past"], 0.0, args["dtype"], None, 0, None, None)
    assert step(kn=0) == 1
    assert step(vn=A + 2) == 1
    assert step(q=0) == 1
    assert step(H_q=6, H_kv=4) == 1
    assert step(D=80) == 3
    assert step(max_past=60, N=5, T_max=64) == 2
    assert step(B=0) == 0


def test_decode_step_host_argument_errors(lib):
    def step(staging=A, staging_bytes=1 << 20, **kw):
        args = dict(q=A, k=A, v=A, kn=A, vn=A, out=A, past=A, B=1, H_q=4, H_kv=2, T_max=64, D=64, N=1,
                    max_past=10, dtype=1)
        args.update(kw)
        return lib.kvd_decode_step_host(args["q"], args["k"], args["v"], args["kn"], args["vn"], args["out"],
                                        args["past"], args["B"], args["H_q"], args["H_kv"], args["T_max"], args["D"],
                                        args["N"], args["max_past"], 0.0, args["dtype"], staging, staging_bytes, None,
                                        0, None, None)
    assert step(q=0) == 1
    assert step(past=0) == 1
    assert step(H_q=6, H_kv=4) == 1
    assert step(D=80) == 3
    assert step(dtype=3) == 3                      # E4M3 caches: not through this entry point
    assert step(max_past=60, N=5, T_max=64) == 2
    assert step(staging=None) == 4
    assert step(staging=A + 16) == 4               # staging must be 256-byte aligned
    assert step(staging_bytes=1791) == 4           # one byte short (next test)
    assert step(B=0, staging=None) == 0


def test_decode_step_host_packed_argument_errors(lib):
    def step(block=A, staging=A, staging_bytes=1 << 20, **kw):
        args = dict(k=A, v=A, out=A, B=1, H_q=4, H_kv=2, T_max=64, D=64, N=1, max_past=10, dtype=1)
        args.update(kw)
        return lib.kvd_decode_step_host_packed(block, args["k"], args["v"], args["out"], args["B"], args["H_q"],
                                               args["H_kv"], args["T_max"], args["D"], args["N"], args["max_past"],
                                               0.0, args["dtype"], staging, staging_bytes, None, 0, None, None)
    assert step(block=0) == 1
    assert step(out=0) == 1
    assert step(D=80) == 3
    assert step(dtype=3) == 3
    assert step(staging=None) == 4
    assert step(staging_bytes=1791) == 4
    assert step(B=0, staging=None) == 0


def test_host_staging_bytes(lib):
    # q and out: 1*4*1*64 bf16 = 512 B each; k_new, v_new: 256 B each; past_len: 4 B -> 256
    assert lib.kvd_host_staging_bytes(1, 4, 2, 64, 1, 1) == 512 + 512 + 256 + 256 + 256
    assert lib.kvd_host_staging_bytes(3, 8, 2, 128, 5, 0) == 2 * (3 * 8 * 5 * 128 * 4) + 2 * (3 * 2 * 5 * 128 * 4) + 256
    assert lib.kvd_host_staging_bytes(1, 4, 2, 64, 1, 3) == 0   # E4M3
    assert lib.kvd_host_staging_bytes(1, 6, 4, 64, 1, 1) == 0   # H_q % H_kv != 0
    # the inputs alone: q, k_new, v_new from 256-byte boundaries, then past_len unpadded
    assert lib.kvd_host_staging_inputs_bytes(1, 4, 2, 64, 1, 1) == 512 + 256 + 256 + 4
    assert lib.kvd_host_staging_inputs_bytes(1, 4, 2, 64, 1, 3) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built CUDA library every entry point raises: there is no fallback path."""
    from kv_cache_decode_append_gb300 import kvd
    monkeypatch.setattr(kvd, "_loaded", None)
    monkeypatch.setattr(kvd._build, "LIB_PATH", str(tmp_path / "libkvd.so"))
    with pytest.raises(RuntimeError, match="missing"):
        kvd.load()
    with pytest.raises(RuntimeError, match="missing"):
        kvd.raw.kvd_cache_bytes(1, 1, 1, 64, 1, 0)
