"""The C ABI library loads, exports every symbol the header declares, and
rejects bad arguments on the host before touching a GPU (runs without one)."""

import ctypes
import os
import re

import pytest

from mla_latent_kv_71_b300 import mla

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "mla.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["mla_absorb_q", "mla_decode_attn", "mla_combine_splits", "mla_out_proj"]:
        assert n in names
    assert set(names) == set(mla.SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = mla.library()
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_version():
    lib = mla.library()
    assert lib.mla_version() >= 100
    for code in range(6):
        assert lib.mla_status_string(code)
    assert b"invalid" in lib.mla_status_string(1)


@pytest.mark.parametrize("dtype", [mla.MLA_BF16, mla.MLA_FP32])
def test_null_pointers_are_rejected_on_the_host(dtype):
    lib = mla.library()
    assert lib.mla_absorb_q(None, None, None, 1, 1, 128, 512, dtype, None) == 1
    assert lib.mla_decode_attn(None, None, None, None, None, None, 1, 1, 128, 512, 64, 64, 1, 1,
                               0.07, 0, None, None, None, 0, dtype, None) == 1
    assert lib.mla_combine_splits(None, None, 1, 1, 512, None, None, dtype, None) == 1
    assert lib.mla_out_proj(None, None, None, None, None, 1, 1, 128, 512, 128, None, 0, dtype,
                            None) == 1


def test_bad_sizes_are_rejected_on_the_host():
    lib = mla.library()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    assert lib.mla_decode_attn(fake, fake, fake, fake, fake, None, 0, 1, 128, 512, 64, 64, 1, 1,
                               0.07, 0, fake, fake, fake, 0, mla.MLA_BF16, None) == 1
    assert lib.mla_combine_splits(fake, fake, 0, 1, 512, fake, fake, mla.MLA_BF16, None) == 1
    assert lib.mla_combine_splits(fake, fake, 2, 1, 6, fake, fake, mla.MLA_BF16, None) == 1
    misaligned = ctypes.c_void_p((1 << 20) + 2)
    assert lib.mla_absorb_q(misaligned, fake, fake, 1, 1, 128, 512, mla.MLA_BF16, None) == 1


def test_shapes_the_bf16_kernels_do_not_cover_are_refused_on_the_host():
    # MLA_ERR_UNSUPPORTED (2), returned before any launch: widths or page size
    # other than the kernel's, a pool beyond 32-bit row indices, and a plan
    # whose 32-bit arithmetic would overflow (units x (pages per unit + 3)).
    lib = mla.library()
    fake = ctypes.c_void_p(1 << 20)

    def call(B=1, T=1, H=128, d_c=512, d_r=64, page=64, max_pages=1, num_pages=1):
        return lib.mla_decode_attn(fake, fake, fake, fake, fake, None, B, T, H, d_c, d_r, page,
                                   max_pages, num_pages, 0.07, 0, fake, fake, fake, 1 << 30,
                                   mla.MLA_BF16, None)

    assert call(d_c=256) == 2
    assert call(d_r=32) == 2
    assert call(page=32) == 2
    assert call(num_pages=(1 << 31) // 64 + 1) == 2
    assert call(B=1 << 19, max_pages=4096) == 2  # 2^19 units x 4099 > 2^31


def test_prologue_calls_reject_bad_arguments_on_the_host():
    lib = mla.library()
    fake = ctypes.c_void_p(1 << 20)

    def append(d=7168, d_c=512, d_r=64, N=4, dtype=mla.MLA_BF16, h=fake, pool=fake):
        return lib.mla_cache_append(h, fake, fake, fake, fake, fake, pool, N, d, d_c, d_r, 2, 64,
                                    4, 8, 10000.0, fake, 1 << 30, dtype, None)

    def project(d=1536, H=128, d_h=128, d_r=64, N=4, dtype=mla.MLA_BF16, q_pe=fake):
        return lib.mla_project_q(fake, fake, fake, fake, q_pe, N, H, d_h, d_r, d, 10000.0, fake,
                                 1 << 30, dtype, None)

    for dtype in (mla.MLA_BF16, mla.MLA_FP32):
        assert append(h=None, dtype=dtype) == 1
        assert append(N=0, dtype=dtype) == 1
        assert append(d_r=63, dtype=dtype) == 1              # RoPE needs pairs
        assert append(pool=ctypes.c_void_p((1 << 20) + 4), dtype=dtype) == 1
        assert project(q_pe=None, dtype=dtype) == 1
        assert project(d_r=63, dtype=dtype) == 1
        assert project(d_h=127, dtype=dtype) == 2           # RoPE pairs must not straddle tiles
        assert append(d_c=511, dtype=dtype) == 2
    assert append(d_c=384 + 64) == 2                          # bf16: d_c % 128
    assert append(d=7168 + 32) == 2                           # bf16: d % 64
    assert append(d_r=36) == 2                                # bf16: d_r % 8
    assert append(d=102, d_c=60, d_r=10, dtype=mla.MLA_FP32) == 2  # fp32: d % 4
    assert project(H=3, d_h=6, d_r=4) == 2                    # bf16: H*(d_h+d_r) % 128
    assert project(d=1536 + 32) == 2                          # bf16: d % 64
    assert project(d=102, dtype=mla.MLA_FP32) == 2            # fp32: d % 4
    assert lib.mla_cache_append_workspace_size(4, 7168, 512, mla.MLA_FP32) == 0
    assert lib.mla_project_q_workspace_size(4, 128, 128, 64, 1536, mla.MLA_FP32) == 0


def test_merged_output_calls_reject_bad_arguments_on_the_host():
    lib = mla.library()
    fake = ctypes.c_void_p(1 << 20)
    assert lib.mla_fold_out_weights(None, fake, fake, 128, 128, 512, 7168, mla.MLA_BF16, None) == 1
    assert lib.mla_fold_out_weights(fake, fake, fake, 128, 128, 500, 7168, mla.MLA_BF16, None) == 2
    assert lib.mla_out_proj_merged(fake, None, fake, 64, 128, 512, 7168, fake, 1 << 30,
                                   mla.MLA_BF16, None) == 1
    assert lib.mla_out_proj_merged(fake, fake, fake, 64, 128, 512, 7100, fake, 1 << 30,
                                   mla.MLA_BF16, None) == 2   # bf16: d % 128
    assert lib.mla_out_proj_merged_workspace_size(64, 128, 512, 7168, mla.MLA_FP32) == 0
