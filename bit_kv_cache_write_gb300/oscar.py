"""Thin ctypes binding of liboscar (include/oscar.h). Same names as the C ABI.

Only argument marshalling happens here: tensors become device pointers and
sizes, host arrays become host pointers. Every step of the write and decode
path runs in the library's CUDA kernels. There is no fallback: if liboscar.so is
missing or fails to load, every call raises.
"""

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboscar.so")

OSCAR_OK = 0
STATUS_NAMES = {
    0: "OSCAR_OK", -1: "OSCAR_ERR_INVALID_ARG", -2: "OSCAR_ERR_UNSUPPORTED", -3: "OSCAR_ERR_NOT_CALIBRATED",
    -4: "OSCAR_ERR_CUDA", -5: "OSCAR_ERR_BOUNDS", -6: "OSCAR_ERR_NO_MEMORY", -7: "OSCAR_ERR_WORKSPACE",
}


class OscarError(RuntimeError):
    def __init__(self, status, where, message):
        self.status = status
        super().__init__("%s: %s (%s) %s" % (where, STATUS_NAMES.get(status, status), oscar_status_string(status), message))


class oscar_config_t(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("group", ctypes.c_int), ("page_size", ctypes.c_int),
                ("sink", ctypes.c_int), ("recent", ctypes.c_int), ("sm_scale", ctypes.c_float),
                ("debug_bounds", ctypes.c_int), ("codebook", ctypes.c_int)]

OSCAR_CODEBOOK_UNIFORM, OSCAR_CODEBOOK_LLOYD_MAX = 0, 1


_lib = None
_vp, _i, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "oscar_create": (_i, [ctypes.POINTER(oscar_config_t), ctypes.POINTER(_vp)]),
    "oscar_destroy": (None, [_vp]),
    "oscar_calibrate_upload": (_i, [_vp, _i, _vp, _vp, _vp, _vp, _vp]),
    "oscar_write_tokens": (_i, [_vp, _i, _vp, _vp, _vp, _i, _vp, _i64, _vp]),
    "oscar_demote_recent": (_i, [_vp, _i, _vp, _i64, _vp, _vp, _i64, _vp, _i, _vp]),
    "oscar_decode_workspace_size": (_sz, [_vp, _i, _i]),
    "oscar_decode": (_i, [_vp, _i, _vp, _vp, _i64, _vp, _i, _vp, _i, _vp, _i64, _vp, _i, _vp,
                          _vp, _vp, _sz, _i, _vp]),
    "oscar_decode_shared_prefix_workspace_size": (_sz, [_vp, _i, _i, _i]),
    "oscar_decode_shared_prefix": (_i, [_vp, _i, _vp, _vp, _i64, _vp, _i, _vp, _i, _vp, _i, _vp, _i64, _vp, _i, _vp,
                                        _vp, _vp, _sz, _i, _vp]),
    "oscar_int2_page_bytes": (_sz, [_vp]),
    "oscar_bf16_page_bytes": (_sz, [_vp]),
    "oscar_status_string": (ctypes.c_char_p, [_i]),
    "oscar_last_error": (ctypes.c_char_p, []),
    "oscar_debug_error": (_i, [_vp, ctypes.POINTER(_i), ctypes.POINTER(ctypes.c_longlong)]),
    "oscar_decode_static_workspace": (_i, [_vp, _i, _vp, _vp, _i64, _vp, _i, _vp, _i, _vp, _i64, _vp, _i, _vp,
                                           _vp, _i, _vp]),
    "oscar_calibration_workspace_size": (_sz, [_i, _i, _i, _i]),
    "oscar_calibration_targets": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_double, _vp, _vp, _vp, _sz,
                                       _vp]),
    "oscar_profile_enable": (_i, [_vp, _i]),
    "oscar_profile_read": (_i, [_vp, _i, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong)]),
}

OSCAR_KERNEL_WRITE, OSCAR_KERNEL_QROT, OSCAR_KERNEL_SPLIT, OSCAR_KERNEL_MERGE = 0, 1, 2, 3


def lib():
    """Load liboscar.so once. Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("liboscar.so not found at %s: build it with "
                               "`python -m bit_kv_cache_write_gb300.build`" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(handle, name)
            f.restype = res
            f.argtypes = args
        _lib = handle
    return _lib


def oscar_status_string(status):
    return lib().oscar_status_string(int(status)).decode()


def oscar_last_error():
    return lib().oscar_last_error().decode()


def _check(status, where):
    if status != OSCAR_OK:
        raise OscarError(status, where, oscar_last_error())


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dptr(t, dtype, name):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def oscar_create(n_layers, n_q_heads, n_kv_heads, head_dim, group, page_size=16, sink=64, recent=256,
                 sm_scale=0.0, debug_bounds=0, codebook=OSCAR_CODEBOOK_UNIFORM):
    """Create a context on the current CUDA device; returns an opaque handle (int)."""
    cfg = oscar_config_t(n_layers, n_q_heads, n_kv_heads, head_dim, group, page_size, sink, recent,
                         float(sm_scale), int(debug_bounds), int(codebook))
    ctx = _vp()
    _check(lib().oscar_create(ctypes.byref(cfg), ctypes.byref(ctx)), "oscar_create")
    return ctx.value


def oscar_destroy(ctx):
    lib().oscar_destroy(ctx)


def oscar_calibrate_upload(ctx, layer, R_k, R_v, T_k, T_v, stream=None):
    """R_k, R_v: host fp32 [H_kv][d][d]; T_k, T_v: host fp32 [H_kv][d]."""
    arrs = [np.ascontiguousarray(a, dtype=np.float32) for a in (R_k, R_v, T_k, T_v)]
    ptrs = [a.ctypes.data_as(_vp) for a in arrs]
    _check(lib().oscar_calibrate_upload(ctx, layer, *ptrs, _stream(stream)), "oscar_calibrate_upload")


def oscar_int2_page_bytes(ctx):
    return lib().oscar_int2_page_bytes(ctx)


def oscar_bf16_page_bytes(ctx):
    return lib().oscar_bf16_page_bytes(ctx)


def oscar_write_tokens(ctx, layer, k, v, slots, int2_pool, stream=None):
    """k, v: bf16 [n][H_kv][d]; slots: int64 [n]; int2_pool: uint8 tensor of whole pages."""
    import torch
    n = slots.numel()
    pages = int2_pool.numel() // oscar_int2_page_bytes(ctx)
    _check(lib().oscar_write_tokens(ctx, layer, _dptr(k, torch.bfloat16, "k"), _dptr(v, torch.bfloat16, "v"),
                                    _dptr(slots, torch.int64, "slots"), n, _dptr(int2_pool, torch.uint8, "int2_pool"),
                                    pages, _stream(stream)), "oscar_write_tokens")


def oscar_demote_recent(ctx, layer, bf16_pool, src_slots, int2_pool, dst_slots, stream=None):
    import torch
    if src_slots.numel() != dst_slots.numel():
        raise ValueError("src_slots and dst_slots differ in length")
    bf_pages = bf16_pool.numel() * 2 // oscar_bf16_page_bytes(ctx)
    i2_pages = int2_pool.numel() // oscar_int2_page_bytes(ctx)
    _check(lib().oscar_demote_recent(ctx, layer, _dptr(bf16_pool, torch.bfloat16, "bf16_pool"), bf_pages,
                                     _dptr(src_slots, torch.int64, "src_slots"),
                                     _dptr(int2_pool, torch.uint8, "int2_pool"), i2_pages,
                                     _dptr(dst_slots, torch.int64, "dst_slots"), src_slots.numel(),
                                     _stream(stream)), "oscar_demote_recent")


def oscar_decode_workspace_size(ctx, batch, max_hist):
    return lib().oscar_decode_workspace_size(ctx, batch, max_hist)


def oscar_decode(ctx, layer, q, int2_pool, int2_tables, hist_len, max_hist, bf16_pool, bf16_tables, bf16_len,
                 out, workspace, stream=None):
    """q: bf16 [B][H_q][d]; tables int32 [B][stride]; lengths int32 [B]; out fp32 [B][H_q][d]; workspace uint8."""
    import torch
    batch = q.shape[0]
    i2_pages = int2_pool.numel() // oscar_int2_page_bytes(ctx) if int2_pool is not None else 0
    bf_pages = bf16_pool.numel() * 2 // oscar_bf16_page_bytes(ctx)
    _check(lib().oscar_decode(
        ctx, layer, _dptr(q, torch.bfloat16, "q"),
        _dptr(int2_pool, torch.uint8, "int2_pool"), i2_pages,
        _dptr(int2_tables, torch.int32, "int2_tables"), int2_tables.shape[1] if int2_tables is not None else 0,
        _dptr(hist_len, torch.int32, "hist_len"), int(max_hist),
        _dptr(bf16_pool, torch.bfloat16, "bf16_pool"), bf_pages,
        _dptr(bf16_tables, torch.int32, "bf16_tables"), bf16_tables.shape[1],
        _dptr(bf16_len, torch.int32, "bf16_len"),
        _dptr(out, torch.float32, "out"), _dptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), batch, _stream(stream)), "oscar_decode")


def oscar_decode_shared_prefix_workspace_size(ctx, batch, prefix_pages, max_hist):
    return lib().oscar_decode_shared_prefix_workspace_size(ctx, batch, prefix_pages, max_hist)


def oscar_decode_shared_prefix(ctx, layer, q, int2_pool, prefix_table, int2_tables, hist_len, max_hist, bf16_pool,
                               bf16_tables, bf16_len, out, workspace, stream=None):
    """oscar_decode with a prefix shared by the whole batch: prefix_table int32 [P] (full pages), then each
    sequence's own pages in int2_tables [B][stride] with hist_len counting the tokens after the prefix."""
    import torch
    batch = q.shape[0]
    i2_pages = int2_pool.numel() // oscar_int2_page_bytes(ctx)
    bf_pages = bf16_pool.numel() * 2 // oscar_bf16_page_bytes(ctx)
    _check(lib().oscar_decode_shared_prefix(
        ctx, layer, _dptr(q, torch.bfloat16, "q"),
        _dptr(int2_pool, torch.uint8, "int2_pool"), i2_pages,
        _dptr(prefix_table, torch.int32, "prefix_table"), prefix_table.numel() if prefix_table is not None else 0,
        _dptr(int2_tables, torch.int32, "int2_tables"), int2_tables.shape[1] if int2_tables is not None else 0,
        _dptr(hist_len, torch.int32, "hist_len"), int(max_hist),
        _dptr(bf16_pool, torch.bfloat16, "bf16_pool"), bf_pages,
        _dptr(bf16_tables, torch.int32, "bf16_tables"), bf16_tables.shape[1],
        _dptr(bf16_len, torch.int32, "bf16_len"),
        _dptr(out, torch.float32, "out"), _dptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), batch, _stream(stream)), "oscar_decode_shared_prefix")


def oscar_calibration_workspace_size(n, n_q_heads, n_kv_heads, head_dim):
    return lib().oscar_calibration_workspace_size(n, n_q_heads, n_kv_heads, head_dim)


def oscar_calibration_targets(q_cal, k_cal, v_cal, sm_scale, target_k, target_v, workspace, stream=None):
    """q_cal fp32 [n][H_q][d], k_cal/v_cal fp32 [m][H_kv][d] -> target_k/target_v fp64 [H_kv][d][d] (device)."""
    import torch
    n, h_q, d = q_cal.shape
    m, h_kv = k_cal.shape[0], k_cal.shape[1]
    _check(lib().oscar_calibration_targets(
        _dptr(q_cal, torch.float32, "q_cal"), _dptr(k_cal, torch.float32, "k_cal"),
        _dptr(v_cal, torch.float32, "v_cal"), n, m, h_q, h_kv, d, float(sm_scale),
        _dptr(target_k, torch.float64, "target_k"), _dptr(target_v, torch.float64, "target_v"),
        _dptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream)),
        "oscar_calibration_targets")


def oscar_decode_static_workspace(ctx, layer, q, int2_pool, int2_tables, hist_len, max_hist, bf16_pool,
                                  bf16_tables, bf16_len, out, stream=None):
    """oscar_decode for callers that cannot allocate: the scratch is the library's static device array.

    Same arguments as oscar_decode without the workspace. The library rejects
    sizes whose workspace exceeds its fixed maximum. Calls that overlap on the
    GPU share that array and race.
    """
    import torch
    batch = q.shape[0]
    i2_pages = int2_pool.numel() // oscar_int2_page_bytes(ctx) if int2_pool is not None else 0
    bf_pages = bf16_pool.numel() * 2 // oscar_bf16_page_bytes(ctx)
    _check(lib().oscar_decode_static_workspace(
        ctx, layer, _dptr(q, torch.bfloat16, "q"),
        _dptr(int2_pool, torch.uint8, "int2_pool"), i2_pages,
        _dptr(int2_tables, torch.int32, "int2_tables"), int2_tables.shape[1] if int2_tables is not None else 0,
        _dptr(hist_len, torch.int32, "hist_len"), int(max_hist),
        _dptr(bf16_pool, torch.bfloat16, "bf16_pool"), bf_pages,
        _dptr(bf16_tables, torch.int32, "bf16_tables"), bf16_tables.shape[1],
        _dptr(bf16_len, torch.int32, "bf16_len"),
        _dptr(out, torch.float32, "out"), batch, _stream(stream)), "oscar_decode_static_workspace")


def oscar_debug_error(ctx):
    """Returns (status, kind, index) and clears the device error word."""
    kind = _i(0)
    index = ctypes.c_longlong(0)
    st = lib().oscar_debug_error(ctx, ctypes.byref(kind), ctypes.byref(index))
    return st, kind.value, index.value


def oscar_profile_enable(ctx, enable):
    _check(lib().oscar_profile_enable(ctx, int(bool(enable))), "oscar_profile_enable")


def oscar_profile_read(ctx, kernel):
    """(total_ms, launches) of one kernel class since the last read; synchronizes."""
    ms = ctypes.c_double(0.0)
    n = ctypes.c_longlong(0)
    _check(lib().oscar_profile_read(ctx, int(kernel), ctypes.byref(ms), ctypes.byref(n)), "oscar_profile_read")
    return ms.value, n.value


class Oscar:
    """Owning wrapper around one context: the same calls as methods, with ctx bound."""

    def __init__(self, **cfg):
        self.cfg = dict(cfg)
        self.ctx = oscar_create(**cfg)

    def close(self):
        if self.ctx:
            oscar_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def calibrate_upload(self, layer, R_k, R_v, T_k, T_v, stream=None):
        oscar_calibrate_upload(self.ctx, layer, R_k, R_v, T_k, T_v, stream)

    def write_tokens(self, layer, k, v, slots, int2_pool, stream=None):
        oscar_write_tokens(self.ctx, layer, k, v, slots, int2_pool, stream)

    def demote_recent(self, layer, bf16_pool, src_slots, int2_pool, dst_slots, stream=None):
        oscar_demote_recent(self.ctx, layer, bf16_pool, src_slots, int2_pool, dst_slots, stream)

    def decode_workspace_size(self, batch, max_hist):
        return oscar_decode_workspace_size(self.ctx, batch, max_hist)

    def decode(self, layer, q, int2_pool, int2_tables, hist_len, max_hist, bf16_pool, bf16_tables, bf16_len,
               out, workspace, stream=None):
        oscar_decode(self.ctx, layer, q, int2_pool, int2_tables, hist_len, max_hist, bf16_pool, bf16_tables,
                     bf16_len, out, workspace, stream)

    def decode_static_workspace(self, layer, q, int2_pool, int2_tables, hist_len, max_hist, bf16_pool, bf16_tables,
                                bf16_len, out, stream=None):
        oscar_decode_static_workspace(self.ctx, layer, q, int2_pool, int2_tables, hist_len, max_hist, bf16_pool,
                                      bf16_tables, bf16_len, out, stream)

    def decode_shared_prefix_workspace_size(self, batch, prefix_pages, max_hist):
        return oscar_decode_shared_prefix_workspace_size(self.ctx, batch, prefix_pages, max_hist)

    def decode_shared_prefix(self, layer, q, int2_pool, prefix_table, int2_tables, hist_len, max_hist, bf16_pool,
                             bf16_tables, bf16_len, out, workspace, stream=None):
        oscar_decode_shared_prefix(self.ctx, layer, q, int2_pool, prefix_table, int2_tables, hist_len, max_hist,
                                   bf16_pool, bf16_tables, bf16_len, out, workspace, stream)

    def int2_page_bytes(self):
        return oscar_int2_page_bytes(self.ctx)

    def bf16_page_bytes(self):
        return oscar_bf16_page_bytes(self.ctx)

    def debug_error(self):
        return oscar_debug_error(self.ctx)

    def profile_enable(self, enable):
        oscar_profile_enable(self.ctx, enable)

    def profile_read(self, kernel):
        return oscar_profile_read(self.ctx, kernel)
