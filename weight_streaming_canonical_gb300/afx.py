"""ctypes binding of libafx (include/afx.h): same names, argument marshalling only.

Host arrays are numpy; device buffers and streams are torch CUDA tensors
and torch streams (torch is used only for device memory and streams).
Every step of the unpack runs in libafx.  Importing this module loads the
library and raises ImportError if it has not been built: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# AFX_DEBUG_BOUNDS=1 in the environment loads the bounds-checked build
# (`python -m weight_streaming_canonical_gb300.build --debug-bounds`)
DEBUG_BOUNDS = os.environ.get("AFX_DEBUG_BOUNDS", "0") == "1"
LIB_PATH = (os.path.join(_HERE, "_build_debug", "libafx_debug.so") if DEBUG_BOUNDS
            else os.path.join(_HERE, "_build", "libafx.so"))

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH} missing); run "
        "`python -m weight_streaming_canonical_gb300.build` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

AFX_OK, AFX_E_ARG, AFX_E_FORMAT, AFX_E_CORRUPT, AFX_E_CUDA, AFX_E_NOSPACE, AFX_E_TIMEOUT = 0, -1, -2, -3, -4, -5, -6
AFX_DEV_BAD_BLOCK, AFX_DEV_BAD_CHUNK, AFX_DEV_BAD_CODE, AFX_DEV_BAD_SHAPE = 0x1, 0x2, 0x4, 0x8
AFX_DEV_TIMEOUT = 0x10
AFX_DEV_UNDRAINED = 0x20
AFX_MAX_CODE_LEN = 24
AFX_BLOCK_CAPACITY = 32768
AFX_HEADER_BYTES = 512
AFX_STATIC_WORKSPACE_BYTES = 4 << 20
AFX_OP_DECODE, AFX_OP_GEMV = 0, 1
AFX_FMT_BF16, AFX_FMT_FP16, AFX_FMT_E4M3 = 0, 1, 2


class afx_code(ctypes.Structure):
    _fields_ = [
        ("count", ctypes.c_uint64 * 256),
        ("code", ctypes.c_uint32 * 256),
        ("len", ctypes.c_uint8 * 256),
        ("nsym", ctypes.c_uint32),
        ("max_len", ctypes.c_uint32),
        ("fill", ctypes.c_uint32),
        ("format", ctypes.c_uint32),
    ]


class afx_desc(ctypes.Structure):
    _fields_ = [
        ("n", ctypes.c_uint64),
        ("total_bits", ctypes.c_uint64),
        ("chunk_bytes", ctypes.c_uint32),
        ("block_chunks", ctypes.c_uint32),
        ("n_chunks", ctypes.c_uint64),
        ("n_blocks", ctypes.c_uint64),
        ("off_exp", ctypes.c_uint64),
        ("exp_bytes", ctypes.c_uint64),
        ("off_sm", ctypes.c_uint64),
        ("off_hi", ctypes.c_uint64),
        ("off_chunk", ctypes.c_uint64),
        ("off_block", ctypes.c_uint64),
        ("container_bytes", ctypes.c_uint64),
        ("max_len", ctypes.c_uint32),
        ("nsym", ctypes.c_uint32),
        ("fill", ctypes.c_uint32),
        ("format", ctypes.c_uint32),
        ("len", ctypes.c_uint8 * 256),
    ]


class afx_op(ctypes.Structure):
    _fields_ = [
        ("desc", afx_desc),
        ("offset", ctypes.c_uint64),
        ("kind", ctypes.c_uint32),
        ("rows", ctypes.c_uint32),
        ("cols", ctypes.c_uint32),
        ("batch", ctypes.c_uint32),
        ("x_dev", ctypes.c_void_p),
        ("out_dev", ctypes.c_void_p),
        ("workspace_dev", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_uint64),
        ("out_host", ctypes.c_void_p),
    ]


class afx_layer(ctypes.Structure):
    _fields_ = [
        ("host_blob", ctypes.c_void_p),
        ("blob_bytes", ctypes.c_uint64),
        ("ops", ctypes.POINTER(afx_op)),
        ("n_ops", ctypes.c_uint32),
        ("reserved", ctypes.c_uint32),
    ]


_vp, _u32, _u64, _i32p = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p
_lib.afx_build_code.argtypes = [_vp, _u64, _u32, ctypes.POINTER(afx_code)]
_lib.afx_build_code_fmt.argtypes = [_vp, _u64, _u32, _u32, ctypes.POINTER(afx_code)]
_lib.afx_encode_bound.argtypes = [_u64, ctypes.POINTER(afx_code), _u32, _u32, ctypes.POINTER(afx_desc)]
_lib.afx_encode.argtypes = [_vp, _u64, ctypes.POINTER(afx_code), ctypes.POINTER(afx_desc), _vp, _u64]
_lib.afx_parse_header.argtypes = [_vp, _u64, ctypes.POINTER(afx_desc)]
_lib.afx_decode.argtypes = [ctypes.POINTER(afx_desc), _vp, _vp, _vp, _i32p]
_lib.afx_decode_gemv_workspace.argtypes = [ctypes.POINTER(afx_desc), _u32, ctypes.POINTER(ctypes.c_uint64)]
_lib.afx_decode_table_kind.argtypes = [ctypes.POINTER(afx_desc), ctypes.POINTER(ctypes.c_uint32),
                                       ctypes.POINTER(ctypes.c_uint32)]
_lib.afx_decode_gemv.argtypes = [ctypes.POINTER(afx_desc), _vp, _u32, _u32, _vp, _u32, _vp, _vp, _u64, _vp, _i32p]
_PP = ctypes.POINTER(ctypes.c_void_p)
_lib.afx_decode_batch.argtypes = [ctypes.POINTER(afx_desc), _PP, _PP, _u32, _vp, _i32p]
_lib.afx_decode_chunks_a_lane.argtypes = [ctypes.POINTER(afx_desc), _PP, _u32, ctypes.POINTER(ctypes.c_uint32)]
_lib.afx_decode_gemv_batch.argtypes = [ctypes.POINTER(afx_desc), _PP, ctypes.POINTER(ctypes.c_uint32),
                                       ctypes.POINTER(ctypes.c_uint32), _PP, _u32, _PP, _PP,
                                       ctypes.POINTER(ctypes.c_uint64), _u32, _vp, _i32p]
_lib.afx_decode_gemv_static.argtypes = [ctypes.POINTER(afx_desc), _vp, _u32, _u32, _vp, _u32, _vp, _vp, _i32p]
_lib.afx_stream_run.argtypes = [ctypes.POINTER(afx_layer), _u32, ctypes.POINTER(ctypes.c_void_p), _u32, _u64, _vp,
                                _vp, _vp, _i32p]
_lib.afx_test_restore_stalled.argtypes = [ctypes.POINTER(afx_desc), _vp, _vp, _u32, _vp, _i32p]
_lib.afx_sync.argtypes = [_vp, _u32, _vp, ctypes.POINTER(ctypes.c_int32)]
_lib.afx_sync.restype = ctypes.c_int
class afx_plan_tensor(ctypes.Structure):
    _fields_ = [("decoded_bytes", ctypes.c_uint64), ("compressed_bytes", ctypes.c_uint64)]


class afx_plan_rates(ctypes.Structure):
    _fields_ = [("link_gbs", ctypes.c_double), ("restore_gbs", ctypes.c_double), ("overlapped", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


AFX_RESIDENT_DECODED, AFX_RESIDENT_COMPRESSED, AFX_STREAM_COMPRESSED, AFX_STREAM_RAW = 0, 1, 2, 3
_lib.afx_plan_residency.argtypes = [ctypes.POINTER(afx_plan_tensor), _u32, _u64, ctypes.POINTER(afx_plan_rates),
                                    ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_uint64)]
_lib.afx_debug_bounds_report.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32)]
_lib.afx_prefill.argtypes = [ctypes.POINTER(afx_desc), _vp, _u32, _u32, _vp, _u32, _vp, _vp, _vp, _vp, _i32p]
_lib.afx_prefill_batch.argtypes = [ctypes.POINTER(afx_desc), ctypes.POINTER(ctypes.c_void_p),
                                   ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32),
                                   ctypes.POINTER(ctypes.c_void_p), _u32, ctypes.POINTER(ctypes.c_void_p), _u32,
                                   ctypes.POINTER(ctypes.c_void_p), _vp, _vp, _vp, _i32p]
AFX_PREFILL_GEMM_WORKSPACE_BYTES = 32 << 20
_lib.afx_tile_order.argtypes = [_vp, _u32, _u32, _vp]
_lib.afx_prefill_fused_workspace.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
_lib.afx_prefill_fused.argtypes = [ctypes.POINTER(afx_desc), _vp, _u32, _u32, _vp, _u32, _vp, _vp, _u64, _vp, _i32p]
_lib.afx_prefill_fused_batch.argtypes = [ctypes.POINTER(afx_desc), ctypes.POINTER(ctypes.c_void_p),
                                         ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32),
                                         ctypes.POINTER(ctypes.c_void_p), _u32, ctypes.POINTER(ctypes.c_void_p), _u32,
                                         _vp, _u64, _vp, _i32p]
_lib.afx_last_error.argtypes = []
_lib.afx_last_error.restype = ctypes.c_char_p
_lib.afx_status_string.argtypes = [ctypes.c_int]
_lib.afx_status_string.restype = ctypes.c_char_p
for _f in (_lib.afx_build_code, _lib.afx_build_code_fmt, _lib.afx_encode_bound, _lib.afx_encode, _lib.afx_parse_header, _lib.afx_decode,
           _lib.afx_decode_batch, _lib.afx_decode_gemv_workspace, _lib.afx_decode_gemv, _lib.afx_decode_gemv_batch,
           _lib.afx_decode_gemv_static, _lib.afx_stream_run, _lib.afx_test_restore_stalled,
           _lib.afx_plan_residency, _lib.afx_debug_bounds_report, _lib.afx_prefill, _lib.afx_prefill_batch,
           _lib.afx_tile_order, _lib.afx_prefill_fused, _lib.afx_prefill_fused_batch,
           _lib.afx_prefill_fused_workspace):
    _f.restype = ctypes.c_int


class AfxError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        super().__init__(f"{fn}: {afx_status_string(status)} ({status})" + (f": {detail}" if detail else ""))
        self.status = status


def afx_last_error() -> str:
    return _lib.afx_last_error().decode()


def afx_status_string(status: int) -> str:
    return _lib.afx_status_string(int(status)).decode()


def _check(fn: str, st: int) -> None:
    if st != AFX_OK:
        raise AfxError(fn, st, afx_last_error() if st in (AFX_E_CUDA, AFX_E_NOSPACE) else "")


def _host_u16(w) -> np.ndarray:
    a = np.ascontiguousarray(w).reshape(-1)
    if a.dtype != np.uint16:
        raise TypeError(f"expected BF16 bit patterns as uint16, got {a.dtype}")
    return a


def element_bytes(fmt: int) -> int:
    """Bytes per element of a format: 2 for BF16 and FP16, 1 for E4M3."""
    return 1 if fmt == AFX_FMT_E4M3 else 2


def _host_elems(w, fmt: int) -> np.ndarray:
    a = np.ascontiguousarray(w).reshape(-1)
    want = np.uint8 if fmt == AFX_FMT_E4M3 else np.uint16
    if a.dtype != want:
        raise TypeError(f"expected {np.dtype(want).name} bit patterns for format {fmt}, got {a.dtype}")
    return a


def _check_out(desc: afx_desc, out) -> None:
    if out.numel() * out.element_size() < desc.n * element_bytes(desc.format) or \
            out.element_size() != element_bytes(desc.format):
        raise ValueError(f"the output must hold n elements of {element_bytes(desc.format)} bytes")


def _dev_ptr(t) -> int:
    if t is None:
        return 0
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t.data_ptr()


def _buf_ptr(t) -> int:
    """A CUDA tensor, or a pinned host tensor (read or written by the kernel over the host link)."""
    if t.is_cuda:
        return _dev_ptr(t)
    if not t.is_pinned() or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor or a contiguous pinned host tensor")
    return t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


# ---- C entry points ---------------------------------------------------------

def afx_build_code(w, max_len: int = AFX_MAX_CODE_LEN) -> afx_code:
    a = _host_u16(w)
    code = afx_code()
    _check("afx_build_code", _lib.afx_build_code(a.ctypes.data, a.size, max_len, ctypes.byref(code)))
    return code


def afx_build_code_fmt(w, fmt: int, max_len: int = AFX_MAX_CODE_LEN) -> afx_code:
    a = _host_elems(w, fmt)
    code = afx_code()
    _check("afx_build_code_fmt", _lib.afx_build_code_fmt(a.ctypes.data, a.size, fmt, max_len, ctypes.byref(code)))
    return code


def afx_encode_bound(n: int, code: afx_code, chunk_bytes: int = 0, block_chunks: int = 0) -> afx_desc:
    d = afx_desc()
    _check("afx_encode_bound", _lib.afx_encode_bound(n, ctypes.byref(code), chunk_bytes, block_chunks, ctypes.byref(d)))
    return d


def afx_encode(w, code: afx_code, desc: afx_desc, out: np.ndarray | None = None) -> np.ndarray:
    a = _host_elems(w, desc.format)
    if out is None:
        out = np.empty(desc.container_bytes, np.uint8)
    if out.dtype != np.uint8 or not out.flags["C_CONTIGUOUS"]:
        raise ValueError("out must be a contiguous uint8 array")
    _check("afx_encode", _lib.afx_encode(a.ctypes.data, a.size, ctypes.byref(code), ctypes.byref(desc),
                                          out.ctypes.data, out.size))
    return out


def afx_parse_header(container) -> afx_desc:
    c = np.ascontiguousarray(container, dtype=np.uint8).reshape(-1)
    d = afx_desc()
    _check("afx_parse_header", _lib.afx_parse_header(c.ctypes.data, c.size, ctypes.byref(d)))
    return d


def afx_decode(desc: afx_desc, container_dev, out_dev, stream=None, status_dev=None) -> None:
    """out_dev: CUDA (or pinned host) tensor of n elements of the container's format:
    16-bit (uint16/int16/bfloat16/float16) for BF16 and FP16, 8-bit (uint8) for E4M3."""
    _check_out(desc, out_dev)
    _check("afx_decode", _lib.afx_decode(ctypes.byref(desc), _buf_ptr(container_dev), _buf_ptr(out_dev),
                                          _stream_handle(stream), _dev_ptr(status_dev)))


def afx_test_restore_stalled(desc: afx_desc, container_dev, out_dev, wait_polls: int, status_dev,
                             stream=None) -> None:
    """Failure injection: a restore whose staging copies never come (see afx.h)."""
    _check("afx_test_restore_stalled",
           _lib.afx_test_restore_stalled(ctypes.byref(desc), _dev_ptr(container_dev), _dev_ptr(out_dev), wait_polls,
                                         _stream_handle(stream), _dev_ptr(status_dev)))


def _ptrs(tensors) -> ctypes.Array:
    return (ctypes.c_void_p * len(tensors))(*[_dev_ptr(t) for t in tensors])


def afx_decode_batch(descs, containers_dev, outs_dev, stream=None, status_dev=None) -> None:
    """Restore several containers in one launch (lists of equal length)."""
    if not (len(descs) == len(containers_dev) == len(outs_dev)):
        raise ValueError("descs, containers_dev and outs_dev must have the same length")
    for d, o in zip(descs, outs_dev):
        _check_out(d, o)
    arr = (afx_desc * len(descs))(*descs)
    bufs_in = (ctypes.c_void_p * len(containers_dev))(*[_buf_ptr(t) for t in containers_dev])
    bufs_out = (ctypes.c_void_p * len(outs_dev))(*[_buf_ptr(t) for t in outs_dev])
    _check("afx_decode_batch", _lib.afx_decode_batch(arr, bufs_in, bufs_out, len(descs),
                                                      _stream_handle(stream), _dev_ptr(status_dev)))


def afx_decode_gemv_batch(descs, containers_dev, shapes, xs_dev, ys_dev, workspaces_dev, stream=None,
                          status_dev=None) -> None:
    """Several fused restore+GEMV products in one launch; shapes = [(rows, cols)], one batch size for all."""
    count = len(descs)
    batch = xs_dev[0].shape[0] if xs_dev and xs_dev[0].dim() == 2 else 1
    for x, y, (r, c) in zip(xs_dev, ys_dev, shapes):
        if (x.shape[0] if x.dim() == 2 else 1) != batch or y.numel() < batch * r:
            raise ValueError("every x must have the same batch and every y must hold batch * rows floats")
    arr = (afx_desc * count)(*descs)
    rows = (ctypes.c_uint32 * count)(*[r for r, _ in shapes])
    cols = (ctypes.c_uint32 * count)(*[c for _, c in shapes])
    wsb = (ctypes.c_uint64 * count)(*[w.numel() * w.element_size() for w in workspaces_dev])
    _check("afx_decode_gemv_batch", _lib.afx_decode_gemv_batch(
        arr, _ptrs(containers_dev), rows, cols, _ptrs(xs_dev), batch, _ptrs(ys_dev), _ptrs(workspaces_dev), wsb,
        count, _stream_handle(stream), _dev_ptr(status_dev)))


AFX_TABLE_FILL, AFX_TABLE_LUT12, AFX_TABLE_STATES, AFX_TABLE_PARTIAL = 0, 1, 2, 3


def afx_decode_table_kind(desc: afx_desc) -> tuple:
    """(kind, rows): the decoder the restore kernels use for this container
    launched alone on the current device (AFX_TABLE_*) and its state-table
    node rows."""
    kind, rows = ctypes.c_uint32(0), ctypes.c_uint32(0)
    _check("afx_decode_table_kind", _lib.afx_decode_table_kind(ctypes.byref(desc), ctypes.byref(kind),
                                                               ctypes.byref(rows)))
    return int(kind.value), int(rows.value)


def afx_decode_chunks_a_lane(descs, containers) -> list:
    """For each container, the chunks a lane (1 or 2; 0 for a fill or an
    empty tensor) that afx_decode_batch of these containers would take on
    the current device."""
    if len(descs) != len(containers):
        raise ValueError("descs and containers must have the same length")
    arr = (afx_desc * len(descs))(*descs)
    bufs = (ctypes.c_void_p * len(containers))(*[_buf_ptr(t) for t in containers])
    out = (ctypes.c_uint32 * max(1, len(descs)))()
    _check("afx_decode_chunks_a_lane", _lib.afx_decode_chunks_a_lane(arr, bufs, len(descs), out))
    return [int(out[i]) for i in range(len(descs))]


def afx_decode_gemv_workspace(desc: afx_desc, batch: int) -> int:
    v = ctypes.c_uint64(0)
    _check("afx_decode_gemv_workspace", _lib.afx_decode_gemv_workspace(ctypes.byref(desc), batch, ctypes.byref(v)))
    return int(v.value)


def afx_decode_gemv(desc: afx_desc, container_dev, rows: int, cols: int, x_dev, y_dev, workspace_dev,
                    stream=None, status_dev=None) -> None:
    """x_dev: CUDA [batch][cols] 16-bit BF16; y_dev: CUDA float32 [batch][rows]."""
    batch = x_dev.shape[0] if x_dev.dim() == 2 else 1
    if y_dev.numel() < batch * rows:
        raise ValueError("y_dev too small")
    ws_bytes = workspace_dev.numel() * workspace_dev.element_size() if workspace_dev is not None else 0
    _check("afx_decode_gemv", _lib.afx_decode_gemv(
        ctypes.byref(desc), _dev_ptr(container_dev), rows, cols, _dev_ptr(x_dev), batch, _dev_ptr(y_dev),
        _dev_ptr(workspace_dev), ws_bytes, _stream_handle(stream), _dev_ptr(status_dev)))


def afx_decode_gemv_static(desc: afx_desc, container_dev, rows: int, cols: int, x_dev, y_dev, stream=None,
                           status_dev=None) -> None:
    """afx_decode_gemv with the library's own fixed device workspace (no allocation by the call)."""
    batch = x_dev.shape[0] if x_dev.dim() == 2 else 1
    if y_dev.numel() < batch * rows:
        raise ValueError("y_dev too small")
    _check("afx_decode_gemv_static", _lib.afx_decode_gemv_static(
        ctypes.byref(desc), _dev_ptr(container_dev), rows, cols, _dev_ptr(x_dev), batch, _dev_ptr(y_dev),
        _stream_handle(stream), _dev_ptr(status_dev)))


def afx_stream_run(layers, dev_bufs, buf_bytes: int, compute_stream=None, copy_stream=None, status_dev=None,
                   d2h_stream=None) -> None:
    """layers: list of (pinned host uint8 tensor, [afx_op, ...]); dev_bufs: list of CUDA uint8 tensors."""
    arr = (afx_layer * len(layers))()
    keep = []
    for i, (blob, ops) in enumerate(layers):
        op_arr = (afx_op * len(ops))(*ops)
        keep.append(op_arr)
        arr[i].host_blob = blob.data_ptr()
        arr[i].blob_bytes = blob.numel() * blob.element_size()
        arr[i].ops = op_arr
        arr[i].n_ops = len(ops)
    bufs = (ctypes.c_void_p * len(dev_bufs))(*[_dev_ptr(b) for b in dev_bufs])
    _check("afx_stream_run", _lib.afx_stream_run(arr, len(layers), bufs, len(dev_bufs), buf_bytes,
                                                  _stream_handle(compute_stream), _stream_handle(copy_stream),
                                                  _stream_handle(d2h_stream) if d2h_stream is not None else None,
                                                  _dev_ptr(status_dev)))


def afx_prefill(desc: afx_desc, container_dev, rows: int, cols: int, x_dev, y_dev, w_scratch_dev, gemm_workspace_dev,
                stream=None, status_dev=None) -> None:
    """y_dev[t] = W x_dev[t] for every token t: x_dev [n_tokens][cols] in the container's format (BF16 or
    FP16), y_dev float32 [n_tokens][rows]."""
    n_tokens = x_dev.shape[0]
    if x_dev.numel() != n_tokens * cols or y_dev.numel() != n_tokens * rows:
        raise ValueError("x_dev must be [n_tokens][cols] and y_dev [n_tokens][rows]")
    if w_scratch_dev.numel() * w_scratch_dev.element_size() < 2 * rows * cols:
        raise ValueError("w_scratch_dev must hold rows * cols 16-bit elements")
    _check("afx_prefill", _lib.afx_prefill(ctypes.byref(desc), _dev_ptr(container_dev), rows, cols, _dev_ptr(x_dev),
                                            n_tokens, _dev_ptr(y_dev), _dev_ptr(w_scratch_dev),
                                            _dev_ptr(gemm_workspace_dev), _stream_handle(stream), _dev_ptr(status_dev)))


def afx_prefill_batch(descs, containers_dev, shapes, xs_dev, ys_dev, w_scratch_dev, gemm_workspace_dev,
                      restore_stream=None, gemm_stream=None, status_dev=None) -> None:
    """afx_prefill over several matrices (shapes = [(rows, cols)]).  w_scratch_dev: two buffers of the
    largest rows * cols BF16 (restores pipelined with products), or [one buffer of all matrices, None]
    (one restore launch, then the products)."""
    n = len(descs)
    n_tokens = xs_dev[0].shape[0]
    arr = (afx_desc * n)(*descs)
    rows = (ctypes.c_uint32 * n)(*[r for r, _ in shapes])
    cols = (ctypes.c_uint32 * n)(*[c for _, c in shapes])
    scratch = (ctypes.c_void_p * 2)(*[(_dev_ptr(t) if t is not None else None) for t in w_scratch_dev])
    _check("afx_prefill_batch", _lib.afx_prefill_batch(arr, _ptrs(containers_dev), rows, cols, _ptrs(xs_dev), n_tokens,
                                                        _ptrs(ys_dev), n, scratch, _dev_ptr(gemm_workspace_dev),
                                                        _stream_handle(restore_stream), _stream_handle(gemm_stream),
                                                        _dev_ptr(status_dev)))


def afx_tile_order(w, rows: int, cols: int) -> np.ndarray:
    """The [rows][cols] BF16 patterns w in the tile order the fused prefill product reads (uint16, flat)."""
    w = np.ascontiguousarray(w, dtype=np.uint16).reshape(-1)
    if w.size != rows * cols:
        raise ValueError("w must hold rows * cols elements")
    out = np.empty(rows * cols, dtype=np.uint16)
    _check("afx_tile_order", _lib.afx_tile_order(w.ctypes.data, rows, cols, out.ctypes.data))
    return out


def afx_prefill_fused_workspace() -> int:
    """Bytes of device workspace afx_prefill_fused needs on the current device (one ring per SM)."""
    v = ctypes.c_uint64()
    _check("afx_prefill_fused_workspace", _lib.afx_prefill_fused_workspace(ctypes.byref(v)))
    return v.value


def afx_prefill_fused(desc: afx_desc, container_dev, rows: int, cols: int, x_dev, y_dev, workspace_dev, stream=None,
                      status_dev=None) -> None:
    """y_dev[t] = W x_dev[t] for every token t, W restored from a slice-ordered container inside the product:
    x_dev BF16 [n_tokens][cols], y_dev float32 [n_tokens][rows], workspace_dev a CUDA tensor of
    afx_prefill_fused_workspace() bytes."""
    n_tokens = x_dev.shape[0]
    if x_dev.numel() != n_tokens * cols or y_dev.numel() != n_tokens * rows:
        raise ValueError("x_dev must be [n_tokens][cols] and y_dev [n_tokens][rows]")
    _check("afx_prefill_fused", _lib.afx_prefill_fused(ctypes.byref(desc), _dev_ptr(container_dev), rows, cols,
                                                        _dev_ptr(x_dev), n_tokens, _dev_ptr(y_dev),
                                                        _dev_ptr(workspace_dev),
                                                        workspace_dev.numel() * workspace_dev.element_size(),
                                                        _stream_handle(stream), _dev_ptr(status_dev)))


def afx_prefill_fused_batch(descs, containers_dev, shapes, xs_dev, ys_dev, workspace_dev, stream=None,
                            status_dev=None) -> None:
    """afx_prefill_fused over several matrices (shapes = [(rows, cols)]), one launch per 16."""
    n = len(descs)
    n_tokens = xs_dev[0].shape[0]
    arr = (afx_desc * n)(*descs)
    rows = (ctypes.c_uint32 * n)(*[r for r, _ in shapes])
    cols = (ctypes.c_uint32 * n)(*[c for _, c in shapes])
    _check("afx_prefill_fused_batch", _lib.afx_prefill_fused_batch(arr, _ptrs(containers_dev), rows, cols,
                                                                    _ptrs(xs_dev), n_tokens, _ptrs(ys_dev), n,
                                                                    _dev_ptr(workspace_dev),
                                                                    workspace_dev.numel() * workspace_dev.element_size(),
                                                                    _stream_handle(stream), _dev_ptr(status_dev)))


def afx_plan_residency(tensors, device_budget_bytes: int, link_gbs: float, restore_gbs: float,
                       overlapped: bool = True) -> tuple[list[int], float, int]:
    """tensors: [(decoded_bytes, compressed_bytes)].  Returns (placements, step_ms, resident_bytes)."""
    n = len(tensors)
    arr = (afx_plan_tensor * max(n, 1))(*[afx_plan_tensor(int(S), int(C)) for S, C in tensors])
    rates = afx_plan_rates(float(link_gbs), float(restore_gbs), 1 if overlapped else 0, 0)
    out = (ctypes.c_uint32 * max(n, 1))()
    ms, res = ctypes.c_double(), ctypes.c_uint64()
    _check("afx_plan_residency", _lib.afx_plan_residency(arr, n, int(device_budget_bytes), ctypes.byref(rates), out,
                                                          ctypes.byref(ms), ctypes.byref(res)))
    return [int(v) for v in out[:n]], ms.value, res.value


def afx_sync(stream=None, timeout_ms: int = 0, status_dev=None) -> tuple[int, int]:
    """Bounded host wait for the work queued on `stream`, then the status word.
    Returns (AFX_OK, 0), (AFX_E_CORRUPT, bits) or (AFX_E_TIMEOUT, 0); raises on a CUDA error."""
    word = ctypes.c_int32(0)
    st = _lib.afx_sync(_stream_handle(stream), int(timeout_ms), _buf_ptr(status_dev) if status_dev is not None else None,
                       ctypes.byref(word))
    if st not in (AFX_OK, AFX_E_CORRUPT, AFX_E_TIMEOUT):
        _check("afx_sync", st)
    return int(st), int(word.value)


def afx_debug_bounds_report() -> tuple[int, bool]:
    """(bits of the failed bounds checks since the last call, whether the loaded library checks)."""
    bits, checked = ctypes.c_uint32(), ctypes.c_uint32()
    _check("afx_debug_bounds_report", _lib.afx_debug_bounds_report(ctypes.byref(bits), ctypes.byref(checked)))
    return bits.value, bool(checked.value)


# ---- conveniences over the entry points ---------------------------------------

def encode(w, chunk_bytes: int = 0, max_len: int = AFX_MAX_CODE_LEN, fmt: int = AFX_FMT_BF16) -> tuple[np.ndarray, afx_desc]:
    """Container (uint8 numpy) and its description for the element patterns w
    (uint16 for BF16 and FP16, uint8 for E4M3)."""
    a = _host_elems(w, fmt)
    code = afx_build_code_fmt(a, fmt, max_len)
    desc = afx_encode_bound(a.size, code, chunk_bytes, 0)
    return afx_encode(a, code, desc), desc


def desc_dict(d: afx_desc) -> dict:
    return {f: (list(getattr(d, f)) if f == "len" else int(getattr(d, f))) for f, _ in afx_desc._fields_}
