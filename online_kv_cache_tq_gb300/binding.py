"""Thin ctypes binding of the C ABI (argument marshalling only).

Every function here has the name of the C entry point it wraps and does no
arithmetic of the method: it converts Python/torch arguments to pointers and
sizes, calls the library and raises ``TQError`` on a non-OK status.  Torch
tensors are accepted for device buffers (their ``data_ptr()`` is passed);
streams default to torch's current CUDA stream.  The library must be built
(``online_kv_cache_tq_gb300.build.build()``); loading fails loudly otherwise.
"""
import ctypes
import os

from . import build as _build

TQ_OK = 0
TQ_BF16 = 0
TQ_FP32 = 1
TQ_CODEC_TURBOQUANT = 0
TQ_CODEC_POLAR = 1
STATUS_NAMES = {0: "TQ_OK", 1: "TQ_ERR_INVALID_ARG", 2: "TQ_ERR_UNSUPPORTED", 3: "TQ_ERR_CUDA",
                4: "TQ_ERR_OOM", 5: "TQ_ERR_WORKSPACE", 6: "TQ_ERR_DEVICE"}
FIELDS = ("k_codes", "k_qjl", "k_norm", "k_rnorm", "v_codes", "v_norm")

# Entry points declared in include/tq.h, checked by the ABI test.
EXPORTED = ("tq_codebook_build", "tq_codebook_destroy", "tq_codebook_levels", "tq_codebook_matrices",
            "tq_cache_field_bytes", "tq_quantize_append", "tq_reconstruction_error", "tq_decode_workspace_bytes",
            "tq_decode_attention", "tq_decode_step", "tq_decode_step_host", "tq_decode_step_host_workspace_bytes",
            "tq_decode_step_prepare", "tq_decode_prepare", "tq_decode_partials", "tq_decode_finish",
            "tq_decode_attention_static", "tq_decode_kernel_kind", "tq_decode_plan", "tq_debug_withhold_commit",
            "tq_decode_parts_workspace_bytes", "tq_decode_attention_parts",
            "tq_get_last_device_error",
            "tq_status_string")


class TQError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s failed: %s" % (where, STATUS_NAMES.get(status, status)))


class tq_config(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("k_bits", ctypes.c_int), ("v_bits", ctypes.c_int),
                ("qjl_m", ctypes.c_int), ("seed", ctypes.c_uint64), ("block_size", ctypes.c_int),
                ("norm_bits", ctypes.c_int), ("codec", ctypes.c_int)]


class tq_cache_view(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("k_qjl", ctypes.c_void_p), ("k_norm", ctypes.c_void_p),
                ("k_rnorm", ctypes.c_void_p), ("v_codes", ctypes.c_void_p), ("v_norm", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("block_size", ctypes.c_int)]


class tq_decode_plan_info(ctypes.Structure):
    _fields_ = [("tensor_cores", ctypes.c_int), ("merge_in_partials", ctypes.c_int),
                ("partials_ctas", ctypes.c_int), ("chunk_tokens", ctypes.c_int), ("merge_ctas", ctypes.c_int)]


class tq_context_part(ctypes.Structure):
    _fields_ = [("book", ctypes.c_void_p), ("cache", ctypes.POINTER(tq_cache_view)), ("block_table", ctypes.c_void_p),
                ("max_blocks", ctypes.c_int), ("context_lens", ctypes.c_void_p), ("max_context", ctypes.c_int)]


_LIB = None


def library_path():
    return _build.LIB_PATH


def load():
    """Load libtq.so (never builds; raises if the library is missing)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError("libtq.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.tq_codebook_build.argtypes = [ctypes.POINTER(tq_config), i32, ctypes.POINTER(vp)]
    lib.tq_codebook_destroy.argtypes = [vp]
    lib.tq_codebook_levels.argtypes = [vp, i32, vp, vp, ctypes.POINTER(i32)]
    lib.tq_codebook_matrices.argtypes = [vp, vp, vp]
    lib.tq_cache_field_bytes.argtypes = [vp, ctypes.POINTER(sz * 6)]
    lib.tq_quantize_append.argtypes = [vp, vp, vp, i32, i32, i32, vp, ctypes.POINTER(tq_cache_view), vp]
    lib.tq_reconstruction_error.argtypes = [vp, vp, i32, i32, i32, i32, vp, ctypes.POINTER(tq_cache_view), vp, vp]
    lib.tq_decode_workspace_bytes.argtypes = [vp, i32, i32, i32]
    lib.tq_decode_workspace_bytes.restype = sz
    lib.tq_decode_attention.argtypes = [vp, vp, i32, i32, i32, i32, ctypes.POINTER(tq_cache_view), vp, i32,
                                        vp, i32, ctypes.c_float, vp, vp, sz, vp]
    lib.tq_decode_step.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, i32, ctypes.POINTER(tq_cache_view), vp,
                                   i32, vp, i32, ctypes.c_float, vp, vp, sz, vp]
    lib.tq_decode_step_host.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, i32, ctypes.POINTER(tq_cache_view),
                                        vp, i32, vp, i32, ctypes.c_float, vp, vp, sz, vp]
    lib.tq_decode_step_host_workspace_bytes.argtypes = [vp, i32, i32, i32, i32, i32, i32]
    lib.tq_decode_step_host_workspace_bytes.restype = sz
    lib.tq_decode_step_prepare.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                           ctypes.POINTER(tq_cache_view), vp, i32, vp, i32, vp, sz, vp]
    lib.tq_decode_prepare.argtypes = [vp, vp, i32, i32, i32, i32, vp, sz, vp]
    lib.tq_decode_partials.argtypes = [vp, i32, i32, i32, ctypes.POINTER(tq_cache_view), vp, i32, vp, i32,
                                       ctypes.c_float, vp, vp, sz, vp]
    lib.tq_decode_finish.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp, sz, vp]
    lib.tq_decode_attention_static.argtypes = [vp, vp, i32, i32, i32, i32, ctypes.POINTER(tq_cache_view), vp,
                                               i32, vp, i32, ctypes.c_float, vp, vp]
    lib.tq_decode_kernel_kind.argtypes = [vp, i32, i32, ctypes.POINTER(i32)]
    lib.tq_decode_plan.argtypes = [vp, i32, i32, i32, i32, ctypes.POINTER(tq_decode_plan_info)]
    lib.tq_debug_withhold_commit.argtypes = [vp, i32]
    lib.tq_decode_parts_workspace_bytes.argtypes = [ctypes.POINTER(tq_context_part), ctypes.POINTER(tq_context_part),
                                                    i32, i32]
    lib.tq_decode_parts_workspace_bytes.restype = sz
    lib.tq_decode_attention_parts.argtypes = [ctypes.POINTER(tq_context_part), ctypes.POINTER(tq_context_part), vp,
                                              i32, i32, i32, i32, ctypes.c_float, vp, vp, sz, vp]
    lib.tq_get_last_device_error.argtypes = [vp, vp, ctypes.POINTER(i32)]
    lib.tq_status_string.argtypes = [i32]
    lib.tq_status_string.restype = ctypes.c_char_p
    for name in EXPORTED:
        if name not in ("tq_decode_workspace_bytes", "tq_decode_step_host_workspace_bytes", "tq_status_string"):
            getattr(lib, name).restype = i32
    _LIB = lib
    return lib


def _check(status, where):
    if status != TQ_OK:
        raise TQError(status, where)


def _ptr(x):
    """Device/host address of a tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Codebook:
    """Owner of a tq_codebook handle."""

    def __init__(self, d=128, k_bits=3, v_bits=3, qjl_m=128, seed=0, block_size=64, device=0, norm_bits=32,
                 codec=0):
        self.config = tq_config(d, k_bits, v_bits, qjl_m, seed, block_size, norm_bits, codec)
        self.device = device
        self.handle = tq_codebook_build(self.config, device)

    def close(self):
        if self.handle:
            tq_codebook_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def qjl_m(self):
        return self.config.qjl_m

    @property
    def block_size(self):
        return self.config.block_size

    @property
    def norm_bits(self):
        return 16 if self.config.norm_bits == 16 else 32

    @property
    def codec(self):
        return self.config.codec


def tq_codebook_build(config, device=0):
    handle = ctypes.c_void_p()
    _check(load().tq_codebook_build(ctypes.byref(config), device, ctypes.byref(handle)), "tq_codebook_build")
    return handle


def tq_codebook_destroy(handle):
    _check(load().tq_codebook_destroy(handle), "tq_codebook_destroy")


def tq_codebook_levels(book, which):
    """(levels, bounds, bits) as lists of floats (fp64 host copies)."""
    import numpy as np
    lib = load()
    bits = ctypes.c_int()
    _check(lib.tq_codebook_levels(book.handle, which, None, None, ctypes.byref(bits)), "tq_codebook_levels")
    levels = np.zeros(1 << bits.value)
    bounds = np.zeros((1 << bits.value) - 1)
    _check(lib.tq_codebook_levels(book.handle, which, levels.ctypes.data, bounds.ctypes.data, None),
           "tq_codebook_levels")
    return levels, bounds, bits.value


def tq_codebook_matrices(book):
    """(R [d][d], S [m][d]) fp64 host copies."""
    import numpy as np
    d, m = book.config.d, book.config.qjl_m
    rot = np.zeros((d, d))
    proj = np.zeros((m, d))
    _check(load().tq_codebook_matrices(book.handle, rot.ctypes.data, proj.ctypes.data if m else None),
           "tq_codebook_matrices")
    return rot, proj


def tq_cache_field_bytes(book):
    arr = (ctypes.c_size_t * 6)()
    _check(load().tq_cache_field_bytes(book.handle, ctypes.byref(arr)), "tq_cache_field_bytes")
    return dict(zip(FIELDS, list(arr)))


def make_cache_view(cache, num_blocks, n_kv_heads, block_size):
    """tq_cache_view from a dict of device tensors keyed by field name."""
    return tq_cache_view(*[_ptr(cache.get(f)) for f in FIELDS], num_blocks, n_kv_heads, block_size)


def tq_quantize_append(book, k, v, dtype, n_tokens, n_kv_heads, slot_mapping, view, stream=None):
    _check(load().tq_quantize_append(book.handle, _ptr(k), _ptr(v), dtype, n_tokens, n_kv_heads,
                                     _ptr(slot_mapping), ctypes.byref(view), _stream(stream)),
           "tq_quantize_append")


def tq_decode_workspace_bytes(book, batch, n_q_heads, max_context):
    return load().tq_decode_workspace_bytes(book.handle, batch, n_q_heads, max_context)


def tq_decode_attention(book, q, dtype, batch, n_q_heads, n_kv_heads, view, block_table, max_blocks,
                        context_lens, max_context, scale, out, workspace, workspace_bytes, stream=None):
    _check(load().tq_decode_attention(book.handle, _ptr(q), dtype, batch, n_q_heads, n_kv_heads,
                                      ctypes.byref(view), _ptr(block_table), max_blocks, _ptr(context_lens),
                                      max_context, scale, _ptr(out), _ptr(workspace), workspace_bytes,
                                      _stream(stream)),
           "tq_decode_attention")


def tq_decode_step(book, k_new, v_new, kv_dtype, q, q_dtype, batch, n_q_heads, n_kv_heads, view, block_table,
                   max_blocks, context_lens, max_context, scale, out, workspace, workspace_bytes, stream=None):
    _check(load().tq_decode_step(book.handle, _ptr(k_new), _ptr(v_new), kv_dtype, _ptr(q), q_dtype, batch,
                                 n_q_heads, n_kv_heads, ctypes.byref(view), _ptr(block_table), max_blocks,
                                 _ptr(context_lens), max_context, scale, _ptr(out), _ptr(workspace),
                                 workspace_bytes, _stream(stream)),
           "tq_decode_step")


def tq_decode_step_host_workspace_bytes(book, batch, n_q_heads, n_kv_heads, max_context, kv_dtype, q_dtype):
    return load().tq_decode_step_host_workspace_bytes(book.handle, batch, n_q_heads, n_kv_heads, max_context,
                                                      kv_dtype, q_dtype)


def tq_decode_step_host(book, k_new, v_new, kv_dtype, q, q_dtype, batch, n_q_heads, n_kv_heads, view, block_table,
                        max_blocks, context_lens, max_context, scale, out, workspace, workspace_bytes, stream=None):
    """tq_decode_step with k_new, v_new, q, context_lens and out in host memory
    (tensors on the CPU, preferably pinned, or int addresses)."""
    _check(load().tq_decode_step_host(book.handle, _ptr(k_new), _ptr(v_new), kv_dtype, _ptr(q), q_dtype, batch,
                                      n_q_heads, n_kv_heads, ctypes.byref(view), _ptr(block_table), max_blocks,
                                      _ptr(context_lens), max_context, scale, _ptr(out), _ptr(workspace),
                                      workspace_bytes, _stream(stream)),
           "tq_decode_step_host")


def tq_decode_step_prepare(book, k_new, v_new, kv_dtype, q, q_dtype, batch, n_q_heads, n_kv_heads, view,
                           block_table, max_blocks, context_lens, max_context, workspace, workspace_bytes,
                           stream=None):
    _check(load().tq_decode_step_prepare(book.handle, _ptr(k_new), _ptr(v_new), kv_dtype, _ptr(q), q_dtype, batch,
                                         n_q_heads, n_kv_heads, ctypes.byref(view), _ptr(block_table),
                                         max_blocks, _ptr(context_lens), max_context, _ptr(workspace),
                                         workspace_bytes, _stream(stream)),
           "tq_decode_step_prepare")


def tq_reconstruction_error(book, x, dtype, which, n_tokens, n_kv_heads, slot_mapping, view, stats, stream=None):
    """Add reconstruction-error sums of appended vectors into ``stats`` (a
    device float64 tensor of 4): sum ||x - x_hat||, sum ||x - x_hat||^2,
    sum ||x||^2, count.  which: 0 keys, 1 values."""
    _check(load().tq_reconstruction_error(book.handle, _ptr(x), dtype, which, n_tokens, n_kv_heads,
                                          _ptr(slot_mapping), ctypes.byref(view), _ptr(stats), _stream(stream)),
           "tq_reconstruction_error")


def tq_decode_prepare(book, q, dtype, batch, n_q_heads, max_context, workspace, workspace_bytes, stream=None):
    _check(load().tq_decode_prepare(book.handle, _ptr(q), dtype, batch, n_q_heads, max_context, _ptr(workspace),
                                    workspace_bytes, _stream(stream)), "tq_decode_prepare")


def tq_decode_partials(book, batch, n_q_heads, n_kv_heads, view, block_table, max_blocks, context_lens,
                       max_context, scale, workspace, workspace_bytes, stream=None, out=None):
    """``out`` None: leave split-K partials for tq_decode_finish; a float32
    [batch][n_q_heads][128] device tensor: leave the final output there."""
    _check(load().tq_decode_partials(book.handle, batch, n_q_heads, n_kv_heads, ctypes.byref(view),
                                     _ptr(block_table), max_blocks, _ptr(context_lens), max_context, scale,
                                     _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)),
           "tq_decode_partials")


def tq_decode_finish(book, batch, n_q_heads, context_lens, max_context, max_blocks, out, workspace,
                     workspace_bytes, stream=None):
    _check(load().tq_decode_finish(book.handle, batch, n_q_heads, _ptr(context_lens), max_context, max_blocks,
                                   _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)),
           "tq_decode_finish")


def tq_decode_attention_static(book, q, dtype, batch, n_q_heads, n_kv_heads, view, block_table, max_blocks,
                               context_lens, max_context, scale, out, stream=None):
    """Decode attention with the library's built-in scratch (no workspace argument)."""
    _check(load().tq_decode_attention_static(book.handle, _ptr(q), dtype, batch, n_q_heads, n_kv_heads,
                                             ctypes.byref(view), _ptr(block_table), max_blocks, _ptr(context_lens),
                                             max_context, scale, _ptr(out), _stream(stream)),
           "tq_decode_attention_static")


def tq_decode_kernel_kind(book, n_q_heads, n_kv_heads):
    """1 when decode partials run on the tensor cores for this shape, else 0."""
    flag = ctypes.c_int()
    _check(load().tq_decode_kernel_kind(book.handle, n_q_heads, n_kv_heads, ctypes.byref(flag)),
           "tq_decode_kernel_kind")
    return flag.value


def tq_get_last_device_error(book, stream=None):
    """Synchronise the stream and return (and clear) the device error code."""
    code = ctypes.c_int()
    status = load().tq_get_last_device_error(book.handle, _stream(stream), ctypes.byref(code))
    if status not in (TQ_OK, 6):
        raise TQError(status, "tq_get_last_device_error")
    return code.value


def tq_status_string(status):
    return load().tq_status_string(status).decode()


def tq_decode_plan(book, batch, n_q_heads, n_kv_heads, max_context):
    """dict(tensor_cores, merge_in_partials, partials_ctas, chunk_tokens, merge_ctas) for a decode shape."""
    info = tq_decode_plan_info()
    _check(load().tq_decode_plan(book.handle, batch, n_q_heads, n_kv_heads, max_context, ctypes.byref(info)),
           "tq_decode_plan")
    return {name: getattr(info, name) for name, _ in info._fields_}


def tq_debug_withhold_commit(book, enable):
    """Test aid for the bounded waits (see include/tq.h)."""
    _check(load().tq_debug_withhold_commit(book.handle, 1 if enable else 0), "tq_debug_withhold_commit")


def context_part(book, view, block_table, max_blocks, context_lens, max_context):
    """A tq_context_part (keeps the cache view alive with it)."""
    part = tq_context_part(book.handle, ctypes.pointer(view), _ptr(block_table), max_blocks, _ptr(context_lens),
                           max_context)
    part._keep = (view, block_table, context_lens)
    return part


def tq_decode_parts_workspace_bytes(first, second, batch, n_q_heads):
    return load().tq_decode_parts_workspace_bytes(ctypes.byref(first), ctypes.byref(second), batch, n_q_heads)


def tq_decode_attention_parts(first, second, q, dtype, batch, n_q_heads, n_kv_heads, scale, out, workspace,
                              workspace_bytes, stream=None):
    _check(load().tq_decode_attention_parts(ctypes.byref(first), ctypes.byref(second), _ptr(q), dtype, batch,
                                            n_q_heads, n_kv_heads, scale, _ptr(out), _ptr(workspace),
                                            workspace_bytes, _stream(stream)), "tq_decode_attention_parts")
