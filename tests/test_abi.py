"""C ABI checks that need no GPU: the library loads, exports every entry point
include/tq.h declares, builds host-only handles whose R, S and codebooks agree
with the oracle's independent construction, and rejects bad arguments before
launching anything."""
import ctypes
import os
import re

import numpy as np
import pytest

from online_kv_cache_tq_gb300 import binding as B
from online_kv_cache_tq_gb300 import build as libbuild
from oracle import engine

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tq.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_]\w*\s*\*?\s+(tq_\w+)\s*\(", text, flags=re.M)))


def test_header_declarations_are_exported(lib):
    names = declared_functions()
    assert "tq_quantize_append" in names and "tq_decode_attention" in names
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(B.EXPORTED) == names


def test_status_strings(lib):
    for code in range(7):
        assert B.tq_status_string(code)
    assert B.tq_status_string(99) == "unknown status"


@pytest.mark.parametrize("k_bits,v_bits,qjl", [(3, 3, 128), (4, 2, 128), (2, 4, 128), (5, 1, 128), (2, 2, 0)])
def test_host_builder_agrees_with_oracle(lib, k_bits, v_bits, qjl):
    book = B.Codebook(k_bits=k_bits, v_bits=v_bits, qjl_m=qjl, seed=7, device=-1)
    ref = engine.build(k_bits=k_bits, v_bits=v_bits, qjl_m=qjl, seed=7)
    rot, proj = B.tq_codebook_matrices(book)
    assert np.max(np.abs(rot - ref["rot"])) < 1e-12
    if qjl:
        assert np.max(np.abs(proj - ref["proj"])) < 1e-12
    for which, name in ((0, "k"), (1, "v")):
        levels, bounds, bits = B.tq_codebook_levels(book, which)
        assert bits == ref[name + "_bits"]
        assert np.max(np.abs(levels - ref[name + "_levels"])) < 1e-12
        # both builders restore the exact symmetry: the tie at 0 is decided alike
        assert np.array_equal(levels, -levels[::-1]) and bounds[len(bounds) // 2] == 0.0
        assert np.max(np.abs(bounds - ref[name + "_bounds"])) < 1e-12
    sizes = B.tq_cache_field_bytes(book)
    expect = engine.field_bytes(ref)
    for field, nbytes in sizes.items():
        assert nbytes == expect.get(field, 0)
    book.close()


def test_config_validation(lib):
    for kw, status in ((dict(k_bits=1, qjl_m=128), 2), (dict(v_bits=5), 2), (dict(qjl_m=12), 1),
                       (dict(block_size=0), 1), (dict(d=100), 1), (dict(d=64), 2)):
        args = dict(d=128, k_bits=3, v_bits=3, qjl_m=128, seed=0, block_size=64)
        args.update(kw)
        cfg = B.tq_config(args["d"], args["k_bits"], args["v_bits"], args["qjl_m"], args["seed"], args["block_size"])
        handle = ctypes.c_void_p()
        device = 0 if kw.get("d") == 64 else -1
        got = lib.tq_codebook_build(ctypes.byref(cfg), device, ctypes.byref(handle))
        assert got == status, kw
    assert lib.tq_codebook_build(None, -1, None) == 1


def test_host_only_handle_rejected_by_kernels(lib):
    book = B.Codebook(device=-1)
    view = B.tq_cache_view(16, 16, 16, 16, 16, 16, 1, 1, 64)
    assert lib.tq_quantize_append(book.handle, 16, 16, 0, 1, 1, 16, ctypes.byref(view), None) == 1
    assert lib.tq_decode_attention(book.handle, 16, 0, 1, 1, 1, ctypes.byref(view), None, 1, 16, 64, 0.0,
                                   16, 256, 1 << 20, None) == 1
    # the host-buffer step validates the whole step before it queues a copy
    ws_bytes = lib.tq_decode_step_host_workspace_bytes(book.handle, 1, 1, 1, 64, 0, 0)
    assert ws_bytes > 0
    assert lib.tq_decode_step_host(book.handle, 16, 16, 0, 16, 0, 1, 1, 1, ctypes.byref(view), 16, 1, 16, 64,
                                   0.0, 16, 256, ws_bytes, None) == 1
    assert lib.tq_decode_step_host(None, 16, 16, 0, 16, 0, 1, 1, 1, ctypes.byref(view), 16, 1, 16, 64, 0.0,
                                   16, 256, ws_bytes, None) == 1
    assert lib.tq_decode_step_host_workspace_bytes(book.handle, 1, 1, 1, 64, 7, 0) == 0
    code = ctypes.c_int()
    assert lib.tq_get_last_device_error(book.handle, None, ctypes.byref(code)) == 1
    assert lib.tq_codebook_destroy(None) == 1
    book.close()


def test_workspace_size_grows_with_context(lib):
    # room for one partial entry per (query head, 512-token chunk) -- what the
    # CUDA-core kernel writes -- and never less than the tensor-core kernel's
    # per-segment entries, which do not grow with the context
    book = B.Codebook(device=-1)
    small = B.tq_decode_workspace_bytes(book, 64, 64, 4096)
    large = B.tq_decode_workspace_bytes(book, 64, 64, 4097)
    assert small % 256 == 0 and large > small
    short = B.tq_decode_workspace_bytes(book, 2, 8, 512)
    assert short == B.tq_decode_workspace_bytes(book, 2, 8, 513) > 0
    assert B.tq_decode_workspace_bytes(book, 0, 8, 512) == 0
    book.close()


def test_sixteen_bit_norms_field_sizes_and_checks(lib):
    # norm_bits 16: every stored norm is 2 bytes, 102 bytes per (token, head) at 3/3 bits
    book = B.Codebook(k_bits=3, v_bits=3, qjl_m=128, device=-1, norm_bits=16)
    sizes = B.tq_cache_field_bytes(book)
    assert [sizes[n] for n in B.FIELDS] == [32, 16, 2, 2, 48, 2]
    assert sum(sizes.values()) == 102
    book.close()
    with pytest.raises(B.TQError) as err:
        B.Codebook(device=-1, norm_bits=8)
    assert err.value.status == 1


def test_polar_codec_handle_fields_and_checks(lib):
    # PolarQuant: 64-byte records for keys and values (token-major), float32
    # radii, no QJL fields: 136 bytes per (token, head); no codebook to read
    book = B.Codebook(k_bits=0, v_bits=0, qjl_m=0, device=-1, codec=B.TQ_CODEC_POLAR)
    sizes = B.tq_cache_field_bytes(book)
    assert [sizes[n] for n in B.FIELDS] == [64, 0, 4, 0, 64, 4]
    assert sizes == engine.field_bytes(engine.build(codec="polar")) | {"k_qjl": 0, "k_rnorm": 0}
    with pytest.raises(B.TQError) as err:
        B.tq_codebook_levels(book, 0)
    assert err.value.status == 2
    # the rotation is the same seeded draw as a TurboQuant handle's
    other = B.Codebook(k_bits=3, v_bits=3, qjl_m=0, device=-1)
    assert np.array_equal(B.tq_codebook_matrices(book)[0], B.tq_codebook_matrices(other)[0])
    other.close()
    book.close()
    for kw, status in ((dict(qjl_m=128), 2), (dict(norm_bits=16), 2), (dict(codec=2), 1)):
        args = dict(k_bits=0, v_bits=0, qjl_m=0, norm_bits=32, codec=B.TQ_CODEC_POLAR)
        args.update(kw)
        with pytest.raises(B.TQError) as err:
            B.Codebook(device=-1, **args)
        assert err.value.status == status, kw
