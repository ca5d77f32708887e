"""CPU-side checks of the C ABI: the library builds for sm_103a, loads without a
GPU, exports every symbol include/mla.h declares, and rejects host-visible bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libmla():
    from head_latent_attention_29_b300 import _build
    _build.build()
    import head_latent_attention_29_b300 as mla
    return mla.lib()


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "mla.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text)))


def test_header_declares_the_hot_path():
    syms = _declared_symbols()
    for name in ["mla_cache_append", "mla_absorb_q", "mla_decode_attn", "mla_decode_workspace_size",
                 "mla_out_up", "mla_gate", "mla_get_device_error", "mla_status_string", "mla_abi_version"]:
        assert name in syms


def test_library_exports_every_declared_symbol(libmla):
    for name in _declared_symbols():
        assert hasattr(libmla, name), name


def test_abi_version_and_status_strings(libmla):
    assert libmla.mla_abi_version() == 1
    for st in range(7):
        s = libmla.mla_status_string(st).decode()
        assert s.startswith("MLA_")
    assert libmla.mla_status_string(99).decode() == "MLA_ERR_UNKNOWN"


def test_workspace_size_rules(libmla):
    ws = libmla.mla_decode_workspace_size
    assert ws(32, 128, 512, 0) > 32 * 128 * 512 * 4          # partials for at least one run per sequence
    assert ws(64, 128, 512, 0) > ws(32, 128, 512, 0)
    assert ws(32, 128, 256, 0) == 0                         # bf16 tensor-core path needs d_c = 512
    assert ws(32, 256, 512, 0) == 0                         # and at most 128 heads
    assert ws(1, 4, 32, 1) > 0                              # fp32 path takes any small shape
    assert ws(0, 4, 32, 1) == 0


def test_host_validation_rejects_bad_arguments(libmla):
    import head_latent_attention_29_b300 as mla
    INVALID = 1
    null = ctypes.c_void_p(0)
    # null cache / null data pointer
    assert libmla.mla_cache_append(None, null, null, null, null, 1, 10000.0, null) == INVALID
    c = mla._Cache(0, 0, 1, 8, 512, 64, 0, 576)
    assert libmla.mla_cache_append(ctypes.byref(c), null, null, null, null, 1, 10000.0, null) == INVALID
    # misaligned cache pointer, bad row stride, odd RoPE width
    c = mla._Cache(0x1008, 0, 1, 8, 512, 64, 0, 576)
    assert libmla.mla_decode_attn(null, ctypes.byref(c), null, 128, 0.1, null, 0, null, null, null) == INVALID
    c = mla._Cache(0x1000, 0, 1, 8, 512, 64, 0, 570)
    assert libmla.mla_decode_attn(null, ctypes.byref(c), null, 128, 0.1, null, 0, null, null, null) == INVALID
    c = mla._Cache(0x1000, 0, 1, 8, 512, 63, 0, 576)
    assert libmla.mla_decode_attn(null, ctypes.byref(c), null, 128, 0.1, null, 0, null, null, null) == INVALID
    # non-positive sizes and null tensors
    assert libmla.mla_absorb_q(null, null, null, null, null, 0, 128, 128, 512, 64, 0, 10000.0, null) == INVALID
    assert libmla.mla_out_up(null, null, null, 1, 1, 1, 1, 0, null) == INVALID
    assert libmla.mla_gate(null, null, null, 1, 1, 1, 0, null) == INVALID
    # unknown dtype
    assert libmla.mla_out_up(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), 1, 1, 1, 1, 7, null) == INVALID


def test_unsupported_bf16_shapes_are_refused(libmla):
    import head_latent_attention_29_b300 as mla
    UNSUPPORTED = 2
    c = mla._Cache(0x1000, 0, 1, 8, 256, 64, 0, 320)   # d_c = 256 has no tensor-core kernel
    p = ctypes.c_void_p(0x2000)
    assert libmla.mla_decode_attn(p, ctypes.byref(c), p, 128, 0.1, p, 1 << 20, p, None, None) == UNSUPPORTED
    c = mla._Cache(0x1000, 0, 1, 8, 512, 64, 0, 576)   # more than 128 heads
    assert libmla.mla_decode_attn(p, ctypes.byref(c), p, 256, 0.1, p, 1 << 20, p, None, None) == UNSUPPORTED


def test_bf16_head_gemms_refuse_what_the_tensor_cores_do_not_take(libmla):
    # bf16 absorb / out-up / gate / kv_down run on the tensor-core kernels only: a
    # shape those kernels do not take is MLA_ERR_UNSUPPORTED and a misaligned
    # pointer MLA_ERR_INVALID_ARG, decided on the host before anything launches
    # (no silent switch to a CUDA-core kernel)
    import head_latent_attention_29_b300 as mla
    INVALID, UNSUPPORTED = 1, 2
    a, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008)
    out_up = libmla.mla_out_up
    assert out_up(a, a, a, 32, 128, 512, 96, 0, None) == UNSUPPORTED     # d_v % 128
    assert out_up(a, a, a, 32, 128, 500, 128, 0, None) == UNSUPPORTED    # d_c % 64
    assert out_up(odd, a, a, 32, 128, 512, 128, 0, None) == INVALID      # o_lat not 16-byte aligned
    assert out_up(a, odd, a, 32, 128, 512, 128, 0, None) == INVALID
    assert out_up(a, a, odd, 32, 128, 512, 128, 0, None) == INVALID
    absorb = libmla.mla_absorb_q
    assert absorb(a, a, a, a, a, 32, 128, 100, 512, 64, 0, 1e4, None) == UNSUPPORTED   # d_k % 64
    assert absorb(a, a, a, a, a, 32, 128, 128, 500, 64, 0, 1e4, None) == UNSUPPORTED   # d_c % 128
    assert absorb(odd, a, a, a, a, 32, 128, 128, 512, 64, 0, 1e4, None) == INVALID
    assert absorb(a, a, a, a, odd, 32, 128, 128, 512, 64, 0, 1e4, None) == INVALID
    assert absorb(a, ctypes.c_void_p(0x10002), a, a, a, 32, 128, 128, 512, 64, 0, 1e4, None) == INVALID
    gate = libmla.mla_gate
    assert gate(a, a, a, 3, 100, 256, 0, None) == UNSUPPORTED            # d_model % 64
    assert gate(a, a, a, 3, 128, 200, 0, None) == UNSUPPORTED            # width % 128
    assert gate(odd, a, a, 3, 128, 256, 0, None) == INVALID
    c = mla._Cache(0x1000, 0, 4, 300, 512, 64, 0, 576)
    kvd = libmla.mla_kv_down_append
    assert kvd(ctypes.byref(c), a, a, a, 1e-6, a, a, 4, 200, 1e4, a, 1 << 20, None) == UNSUPPORTED  # d_model % 64
    assert kvd(ctypes.byref(c), odd, a, a, 1e-6, a, a, 4, 256, 1e4, a, 1 << 20, None) == INVALID
    # the append-and-absorb call: mla_absorb_q's limits, plus a 16-byte aligned c_kv
    fused = libmla.mla_absorb_q_append
    assert fused(None, a, a, a, a, 4, a, a, a, a, a, 32, 128, 128, 1e4, None) == INVALID            # no cache
    assert fused(ctypes.byref(c), a, a, a, a, -1, a, a, a, a, a, 32, 128, 128, 1e4, None) == INVALID  # T < 0
    assert fused(ctypes.byref(c), a, a, a, a, 4, a, a, a, a, a, 32, 128, 100, 1e4, None) == UNSUPPORTED  # d_k % 64
    assert fused(ctypes.byref(c), odd, a, a, a, 4, a, a, a, a, a, 32, 128, 128, 1e4, None) == INVALID  # c_kv
    assert fused(ctypes.byref(c), a, ctypes.c_void_p(0x10002), a, a, 4, a, a, a, a, a, 32, 128, 128, 1e4,
                 None) == INVALID                                                                      # k_r
    assert fused(ctypes.byref(c), a, a, a, a, 4, odd, a, a, a, a, 32, 128, 128, 1e4, None) == INVALID  # q_nope
    assert fused(ctypes.byref(c), a, a, a, a, 4, a, a, a, a, a, 32, 128, 128, 0.0, None) == INVALID    # base
    c192 = mla._Cache(0x1000, 0, 4, 300, 192, 64, 0, 256)   # d_c % 128 != 0: no tensor-core absorb
    assert fused(ctypes.byref(c192), a, a, a, a, 4, a, a, a, a, a, 32, 128, 128, 1e4, None) == UNSUPPORTED


def test_product_path_fails_loudly_without_the_library(tmp_path, monkeypatch):
    import head_latent_attention_29_b300 as mla
    monkeypatch.setattr(mla, "_lib_handle", None)
    monkeypatch.setattr(mla, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        mla.lib()


def test_library_built_from_other_sources_is_refused(libmla, monkeypatch):
    # the build compiles a hash of its sources into the library; the binding
    # compares it with the sources beside it, whatever the files' times
    import head_latent_attention_29_b300 as mla
    from head_latent_attention_29_b300 import _build
    assert libmla.mla_build_source_hash().decode() == _build.source_hash() == _build.built_hash()
    assert not _build.needs_build()
    monkeypatch.setattr(mla, "_lib_handle", None)
    monkeypatch.setattr(_build, "source_hash", lambda: "0123456789abcdef")
    with pytest.raises(ImportError, match="built from other sources"):
        mla.lib()


def test_paged_cache_validation(libmla):
    import head_latent_attention_29_b300 as mla
    INVALID, UNSUPPORTED = 1, 2
    assert ctypes.sizeof(mla._PagedCache) == 48
    assert mla.PAGE_ROWS == 64
    p = ctypes.c_void_p(0x2000)
    ok = dict(data=0x1000, dtype=0, num_pages=16, d_c=512, d_r=64, row_stride=576, block_table=0x3000, B=2,
              max_blocks=8)

    def paged(**kw):
        f = dict(ok, **kw)
        return mla._PagedCache(f["data"], f["dtype"], f["num_pages"], f["d_c"], f["d_r"], f["row_stride"],
                               f["block_table"], f["B"], f["max_blocks"])

    def decode(c, H=128):
        return libmla.mla_decode_attn_paged(p, ctypes.byref(c), p, H, 0.1, p, 1 << 20, p, None, None)

    assert libmla.mla_decode_attn_paged(p, None, p, 128, 0.1, p, 1 << 20, p, None, None) == INVALID
    assert decode(paged(block_table=0)) == INVALID          # a paged cache needs its block table
    assert decode(paged(block_table=0x3002)) == INVALID     # int32 entries: 4-byte aligned
    assert decode(paged(data=0x1008)) == INVALID            # pool base 16-byte aligned
    assert decode(paged(num_pages=0)) == INVALID
    assert decode(paged(max_blocks=0)) == INVALID
    assert decode(paged(max_blocks=1 << 26)) == INVALID     # 64 x max_blocks must fit int32 positions
    assert decode(paged(row_stride=570)) == INVALID
    assert decode(paged(d_r=63)) == INVALID
    assert decode(paged(d_c=256, row_stride=320)) == UNSUPPORTED
    assert decode(paged(), H=256) == UNSUPPORTED
    assert decode(paged(dtype=1, row_stride=576)) == UNSUPPORTED  # fp32 pools have no paged kernel
    assert libmla.mla_cache_append_paged(ctypes.byref(paged(block_table=0)), p, p, p, p, 1, 10000.0, None) == INVALID
    assert libmla.mla_cache_append_paged(ctypes.byref(paged()), p, p, p, p, -1, 10000.0, None) == INVALID
    assert libmla.mla_cache_append_paged(ctypes.byref(paged()), p, p, p, p, 0, 10000.0, None) == 0


def test_kv_down_validation_and_workspace(libmla):
    import head_latent_attention_29_b300 as mla
    INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 5
    ws = libmla.mla_kv_down_workspace_size
    # decode batch: 5 column tiles x 30 K ranges of fp32 partials
    assert ws(32, 7168, 512, 64, 0) == 30 * 32 * 576 * 4
    assert ws(32768, 7168, 512, 64, 0) == 32768 * 576 * 4   # 640 tiles: no K split
    assert ws(40, 64, 32, 8, 1) == 40 * 40 * 4               # fp32: CUDA-core path, one range
    assert ws(0, 7168, 512, 64, 0) == 0
    p = ctypes.c_void_p(0x2000)
    c = mla._Cache(0x1000, 0, 4, 300, 512, 64, 0, 576)

    def call(cache=c, T=4, eps=1e-6, d_model=1024, wsb=1 << 20, ws_ptr=p, base=1e4):
        return libmla.mla_kv_down_append(ctypes.byref(cache) if cache is not None else None, p, p, p, eps, p, p, T,
                                         d_model, base, ws_ptr, wsb, None)

    assert call(cache=None) == INVALID
    assert call(T=-1) == INVALID
    assert call(T=0) == 0
    assert call(eps=float("nan")) == INVALID
    assert call(eps=-1.0) == INVALID
    assert call(d_model=0) == INVALID
    assert call(base=0.0) == INVALID
    assert call(wsb=16) == WORKSPACE                        # far below the partials' size
    assert call(ws_ptr=ctypes.c_void_p(0x2008)) == WORKSPACE  # 16-byte aligned scratch
    assert call(cache=mla._Cache(0x1000, 0, 4, 300, 511, 65, 0, 576)) == INVALID  # odd d_r
    assert call(cache=mla._Cache(0x1000, 0, 4, 300, 511, 64, 0, 576)) == UNSUPPORTED  # odd d_c
    assert call(cache=mla._Cache(0x1000, 1, 4, 300, 1024, 64, 0, 1088)) == UNSUPPORTED  # row over 1024
    pc = mla._PagedCache(0x1000, 0, 16, 512, 64, 576, 0, 2, 8)  # paged without a block table
    assert libmla.mla_kv_down_append_paged(ctypes.byref(pc), p, p, p, 1e-6, p, p, 4, 1024, 1e4, p, 1 << 20,
                                           None) == INVALID


def test_nvtx_ranges_switch_on_without_a_tool(tmp_path):
    # MLA_NVTX=1 wraps every compute entry point in an NVTX range; with no profiler
    # attached the calls are no-ops and the entry points behave as before
    import subprocess
    import sys
    code = (
        "import ctypes, head_latent_attention_29_b300 as mla\n"
        "lib = mla.lib()\n"
        "c = mla._Cache(0x1008, 0, 1, 8, 512, 64, 0, 576)\n"
        "assert lib.mla_decode_attn(None, ctypes.byref(c), None, 128, 0.1, None, 0, None, None, None) == 1\n"
        "assert lib.mla_cache_append(None, None, None, None, None, 1, 1e4, None) == 1\n"
        "print('ok')\n"
    )
    env = dict(os.environ, MLA_NVTX="1", PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stderr


def test_header_compiles_as_c_and_layouts_match_the_binding(tmp_path, libmla):
    # a plain C consumer of include/mla.h: the header must be valid C99, every
    # declared entry point must link against the built library, and the structs
    # the caller fills must have the layout the Python binding assumes
    import shutil
    import subprocess
    import head_latent_attention_29_b300 as mla
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    syms = _declared_symbols()
    src = tmp_path / "consumer.c"
    src.write_text(
        "#include <stddef.h>\n#include <stdint.h>\n#include <stdio.h>\n#include \"mla.h\"\n"
        "int main(void) {\n"
        "  volatile uintptr_t a;\n"
        + "".join(f"  a = (uintptr_t)&{s};\n  printf(\"%d\\n\", (int)(a != 0));\n" for s in syms)
        + "  printf(\"%zu %zu %zu %zu %zu\\n\", sizeof(mla_cache), offsetof(mla_cache, dtype), "
          "offsetof(mla_cache, d_r), offsetof(mla_cache, row_stride), offsetof(mla_cache, N_max));\n"
          "  printf(\"%zu %zu %zu %zu %zu\\n\", sizeof(mla_paged_cache), offsetof(mla_paged_cache, num_pages), "
          "offsetof(mla_paged_cache, row_stride), offsetof(mla_paged_cache, block_table), "
          "offsetof(mla_paged_cache, max_blocks));\n"
          "  return 0;\n}\n")
    exe = tmp_path / "consumer"
    lib_dir = os.path.dirname(mla.LIB_PATH)
    cc = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                         "-L", lib_dir, "-l:libmla.so", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.split()
    assert lines[:len(syms)] == ["1"] * len(syms)
    c = [int(x) for x in lines[len(syms):len(syms) + 5]]
    p = [int(x) for x in lines[len(syms) + 5:len(syms) + 10]]
    C, P = mla._Cache, mla._PagedCache
    assert c == [ctypes.sizeof(C), C.dtype.offset, C.d_r.offset, C.row_stride.offset, C.N_max.offset]
    assert p == [ctypes.sizeof(P), P.num_pages.offset, P.row_stride.offset, P.block_table.offset,
                 P.max_blocks.offset]


def test_prefill_explicit_validation(libmla):
    import head_latent_attention_29_b300 as mla
    INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 5
    assert libmla.mla_prefill_explicit_workspace_size(4, 0, 8192, 128) == 2 * 4 * 8192 * 128 * 128 * 2
    assert libmla.mla_prefill_explicit_workspace_size(1, 37, 200, 2) == 2 * 237 * 2 * 128 * 2
    assert libmla.mla_prefill_explicit_workspace_size(0, 0, 1, 2) == 0
    p = ctypes.c_void_p(0x2000)
    c = mla._Cache(0x1000, 0, 2, 300, 512, 64, 0, 576)

    def call(cache=c, start=0, S=200, H=4, causal=1, scale=0.07, base=1e4, ptr=p, wsb=1 << 30):
        return libmla.mla_prefill_explicit(ptr, p, ctypes.byref(cache), p, p, start, S, causal, H, scale, base, p,
                                           wsb, p, None, None)

    assert call(ptr=ctypes.c_void_p(0)) == INVALID
    assert call(ptr=ctypes.c_void_p(0x2008)) == INVALID         # 16-byte aligned queries
    assert call(S=0) == INVALID
    assert call(start=-1) == INVALID
    assert call(start=101, S=200) == INVALID                    # start + S beyond N_max = 300
    assert call(scale=float("nan")) == INVALID
    assert call(base=0.0) == INVALID
    assert call(H=3) == UNSUPPORTED                             # the K/V rebuild pairs heads
    assert call(cache=mla._Cache(0x1000, 0, 2, 300, 512, 0, 0, 512)) == UNSUPPORTED  # needs the 64-wide key
    assert call(cache=mla._Cache(0x1000, 1, 2, 300, 512, 64, 0, 576)) == UNSUPPORTED  # bf16 only
    assert call(wsb=1024) == WORKSPACE
