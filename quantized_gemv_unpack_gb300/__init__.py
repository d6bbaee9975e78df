"""Python binding of libqmv (fused dequantize-and-matvec for compressed-LLM decode on GB300).

Argument marshalling only: every function forwards to the C ABI of
``include/qmv.h`` under the same name. Device buffers are torch CUDA tensors
(or raw integer addresses); streams default to torch's current stream. A
failing call raises ``QmvError`` with the library's message. There is no
fallback: if ``libqmv.so`` has not been built, importing a call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqmv.so")

QMV_ABI_VERSION = 1
QMV_GROUP = 128
QMV_MAX_SECTIONS = 8
QMV_MAX_M = 16
QMV_MAX_BATCH = 448

QMV_OK, QMV_ERR_ARG, QMV_ERR_ALIGN, QMV_ERR_UNSUPPORTED = 0, -1, -2, -3
QMV_ERR_CORRUPT, QMV_ERR_CUDA, QMV_ERR_TIMEOUT = -4, -5, -6
QMV_TERNARY2, QMV_INT4, QMV_CASS, QMV_CASS_MX, QMV_TERNARY2_SPARSE, QMV_TERNARY2_LUT, QMV_INT4_LUT = 1, 2, 3, 4, 5, 6, 7
QMV_FLAG_PATH_FMA, QMV_FLAG_PATH_MMA = 1, 2   # qmv_desc.flags: force the fp16-FMA or the tensor-core matvec kernel
QMV_FLAG_TEST_WAIT_TIMEOUT = 0x100           # qmv_desc.flags, testing only: the matvec's first wait gives up

# the exported C symbols (one per declaration in include/qmv.h)
EXPORTS = ("qmv_pack_desc", "qmv_pack_ternary", "qmv_pack_int4", "qmv_unpack", "qmv_run_ternary",
           "qmv_run_int4", "qmv_run_batch", "qmv_sparse_pack_host", "cass_pack_host", "cass_mx_pack_host", "cass_kv_encode", "cass_decode_draft", "cass_reconstruct",
           "cass_speculate_step", "moe_workspace_size", "moe_qmv_run", "moe_qmv_run_static",
           "qmv_file_write", "qmv_file_open", "qmv_file_count", "qmv_file_tensor", "qmv_file_find", "qmv_file_load",
           "qmv_file_read_host", "qmv_file_close", "qmv_crc32", "qmv_check_status", "qmv_last_error")


class QmvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"qmv status {status}: {message}")
        self.status = status


class qmv_desc(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_uint32), ("format", ctypes.c_uint32),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("group", ctypes.c_int32), ("n_symbols", ctypes.c_int32),
                ("off", ctypes.c_int64 * QMV_MAX_SECTIONS), ("bytes", ctypes.c_int64 * QMV_MAX_SECTIONS),
                ("total_bytes", ctypes.c_int64), ("flags", ctypes.c_uint64)]

    def sections(self):
        return [(int(self.off[i]), int(self.bytes[i])) for i in range(QMV_MAX_SECTIONS)]


class qmv_task(ctypes.Structure):
    _fields_ = [("desc", ctypes.POINTER(qmv_desc)), ("w", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("ldx", ctypes.c_int64), ("ldy", ctypes.c_int64)]


_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_DESC = ctypes.POINTER(qmv_desc)
_SIGS = {
    "qmv_pack_desc": (_I32, [_I32, _I64, _I64, ctypes.c_int32, _DESC]),
    "qmv_pack_ternary": (_I32, [_DESC, _P, _P, _P]),
    "qmv_pack_int4": (_I32, [_DESC, _P, _P, _P]),
    "qmv_unpack": (_I32, [_DESC, _P, _P, _P, _P]),
    "qmv_run_ternary": (_I32, [_DESC, _P, _P, _I32, _I64, _P, _I64, _P]),
    "qmv_run_int4": (_I32, [_DESC, _P, _P, _I32, _I64, _P, _I64, _P]),
    "qmv_run_batch": (_I32, [_I32, ctypes.POINTER(qmv_task), _I32, _I32, _P]),
    "cass_pack_host": (_I32, [_P, _I64, _I64, _P, _I64, _DESC, _P, _I64]),
    "cass_mx_pack_host": (_I32, [_P, _I64, _I64, _P, _I64, _DESC, _P, _I64]),
    "qmv_sparse_pack_host": (_I32, [_DESC, _P, _DESC, _P, _I64]),
    "cass_kv_encode": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _DESC, _P, _I64, _P]),
    "cass_decode_draft": (_I32, [_DESC, _P, _P, _I32, _I64, _P, _I64, _P, _P]),
    "cass_reconstruct": (_I32, [_DESC, _P, _P, _I32, _I64, _P, _I64, _P, _P]),
    "cass_speculate_step": (_I32, [_DESC, _P, _P, _I32, _I64, _P, _P, _I64, _P]),
    "moe_workspace_size": (ctypes.c_size_t, [_I32, _I32, _I32, _I64, _I64]),
    "moe_qmv_run": (_I32, [_DESC, _DESC, _P, _I64, _I64, _I32, _P, _I32, _P, _I32, _I64, _P, _I64, _P,
                           ctypes.c_size_t, _P]),
    "moe_qmv_run_static": (_I32, [_DESC, _DESC, _P, _I64, _I64, _I32, _P, _I32, _P, _I32, _I64, _P, _I64, _P]),
    "qmv_file_write": (_I32, [ctypes.c_char_p, _I32, ctypes.POINTER(ctypes.c_char_p), _DESC, ctypes.POINTER(_P)]),
    "qmv_file_open": (_I32, [ctypes.c_char_p, ctypes.POINTER(_P)]),
    "qmv_file_count": (_I32, [_P]),
    "qmv_file_tensor": (_I32, [_P, _I32, ctypes.c_char_p, _DESC]),
    "qmv_file_find": (_I32, [_P, ctypes.c_char_p]),
    "qmv_file_load": (_I32, [_P, _I32, _P, _I64, _P]),
    "qmv_file_read_host": (_I32, [_P, _I32, _P, _I64]),
    "qmv_file_close": (None, [_P]),
    "qmv_crc32": (ctypes.c_uint32, [_P, ctypes.c_size_t, ctypes.c_uint32]),
    "qmv_check_status": (_I32, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "qmv_last_error": (ctypes.c_char_p, []),
}


def lib():
    """The loaded libqmv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with quantized_gemv_unpack_gb300.build.build() "
                              "(there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def qmv_last_error() -> str:
    return lib().qmv_last_error().decode()


def _check(rc: int):
    if rc != QMV_OK:
        raise QmvError(rc, qmv_last_error())


def _ptr(t):
    """Device/host address of a torch tensor, a NumPy array, an int or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _rows(t):
    """(M, leading dimension) of a 2-D (or 1-D) activation/output tensor."""
    if t.dim() == 1:
        return 1, t.shape[0]
    return t.shape[0], t.stride(0)


# ----------------------------------------------------------------------------- layout and packing

def qmv_pack_desc(format: int, N: int, K: int, group: int = QMV_GROUP) -> qmv_desc:
    d = qmv_desc()
    _check(lib().qmv_pack_desc(format, N, K, group, ctypes.byref(d)))
    return d


def qmv_pack_ternary(desc: qmv_desc, w, packed, stream=None):
    _check(lib().qmv_pack_ternary(ctypes.byref(desc), _ptr(w), _ptr(packed), _stream(stream)))


def qmv_pack_int4(desc: qmv_desc, w, packed, stream=None):
    _check(lib().qmv_pack_int4(ctypes.byref(desc), _ptr(w), _ptr(packed), _stream(stream)))


def qmv_unpack(desc: qmv_desc, packed, q, scales=None, stream=None):
    _check(lib().qmv_unpack(ctypes.byref(desc), _ptr(packed), _ptr(q), _ptr(scales), _stream(stream)))


# ----------------------------------------------------------------------------- matvec

def qmv_run_ternary(desc: qmv_desc, w, x, y, stream=None):
    M, ldx = _rows(x)
    _, ldy = _rows(y)
    _check(lib().qmv_run_ternary(ctypes.byref(desc), _ptr(w), _ptr(x), M, ldx, _ptr(y), ldy, _stream(stream)))


def qmv_run_int4(desc: qmv_desc, w, x, y, stream=None):
    M, ldx = _rows(x)
    _, ldy = _rows(y)
    _check(lib().qmv_run_int4(ctypes.byref(desc), _ptr(w), _ptr(x), M, ldx, _ptr(y), ldy, _stream(stream)))


class Batch:
    """A prepared qmv_run_batch argument list. It keeps the descriptors, the ctypes
    arrays and the tensors (packed weights, x, y) alive for as long as it exists: the
    launch reads them through raw pointers, and memory that the caller's allocator took
    back and handed out again would otherwise be read as weights."""

    def __init__(self, format: int, tasks, M: int):
        self.format = format
        self.M = M
        self.descs = [t[0] for t in tasks]
        self.tensors = [tuple(t[1:]) for t in tasks]
        self.arr = (qmv_task * len(tasks))()
        for i, (d, w, x, y) in enumerate(tasks):
            _, ldx = _rows(x)
            _, ldy = _rows(y)
            self.arr[i] = qmv_task(ctypes.pointer(d), _ptr(w), _ptr(x), _ptr(y), ldx, ldy)

    def run(self, stream=None):
        _check(lib().qmv_run_batch(self.format, self.arr, len(self.arr), self.M, _stream(stream)))


def qmv_run_batch(format: int, tasks, M: int, stream=None):
    """tasks: list of (desc, w, x, y). Prefer ``Batch`` when the same list runs many times."""
    Batch(format, tasks, M).run(stream)


# ----------------------------------------------------------------------------- Cassandra

def _host_pack(fn, w_bf16_bits, calib_bf16_bits):
    import numpy as np
    w = np.ascontiguousarray(w_bf16_bits, dtype=np.uint16)
    c = np.ascontiguousarray(calib_bf16_bits, dtype=np.uint16)
    N, K = w.shape
    R = c.shape[0]
    d = qmv_desc()
    _check(fn(w.ctypes.data, N, K, c.ctypes.data, R, ctypes.byref(d), None, 0))
    out = np.zeros(d.total_bytes, dtype=np.uint8)
    _check(fn(w.ctypes.data, N, K, c.ctypes.data, R, ctypes.byref(d), out.ctypes.data, out.nbytes))
    return d, out


def cass_pack_host(w_bf16_bits, calib_bf16_bits):
    """Host packer: NumPy uint16 [N][K] weights and [R][K] calibration rows -> (desc, uint8 buffer)."""
    return _host_pack(lib().cass_pack_host, w_bf16_bits, calib_bf16_bits)


def qmv_sparse_pack_host(dense_desc: qmv_desc, dense_packed_host):
    """Flagged sparse ternary packer: a host copy (NumPy uint8) of a dense ternary buffer ->
    (desc, uint8 buffer) with all-zero 16 x 128 tiles left out."""
    import numpy as np
    src = np.ascontiguousarray(dense_packed_host, dtype=np.uint8)
    d = qmv_desc()
    _check(lib().qmv_sparse_pack_host(ctypes.byref(dense_desc), src.ctypes.data, ctypes.byref(d), None, 0))
    out = np.zeros(d.total_bytes, dtype=np.uint8)
    _check(lib().qmv_sparse_pack_host(ctypes.byref(dense_desc), src.ctypes.data, ctypes.byref(d), out.ctypes.data,
                                      out.nbytes))
    return d, out


def cass_kv_encode(kv, codebook, slot_words: int, packed=None, stream=None) -> qmv_desc:
    """Online KV encoder: kv device bf16 [T][ld] (one token per row), codebook NumPy uint8 [256]
    (the exponents in rank order). Returns the QMV_CASS descriptor; with packed (device uint8 of
    at least desc.total_bytes) also encodes into it. packed=None is a size query."""
    import numpy as np
    cb = np.ascontiguousarray(codebook, dtype=np.uint8)
    T, ld = _rows(kv)
    D = kv.shape[1]
    d = qmv_desc()
    _check(lib().cass_kv_encode(_ptr(kv), T, D, ld, cb.ctypes.data, slot_words, ctypes.byref(d),
                                _ptr(packed) if packed is not None else None,
                                packed.numel() if packed is not None else 0, _stream(stream)))
    return d


def cass_mx_pack_host(w_bf16_bits, calib_bf16_bits):
    """Cassandra-2 (MX) host packer, same arguments and result as cass_pack_host."""
    return _host_pack(lib().cass_mx_pack_host, w_bf16_bits, calib_bf16_bits)


def cass_decode_draft(desc: qmv_desc, packed, x, y=None, w_draft=None, stream=None):
    M, ldx = _rows(x)
    ldy = _rows(y)[1] if y is not None else 0
    _check(lib().cass_decode_draft(ctypes.byref(desc), _ptr(packed), _ptr(x), M, ldx, _ptr(y), ldy,
                                   _ptr(w_draft), _stream(stream)))


def cass_reconstruct(desc: qmv_desc, packed, x, y=None, w_out=None, stream=None):
    M, ldx = _rows(x)
    ldy = _rows(y)[1] if y is not None else 0
    _check(lib().cass_reconstruct(ctypes.byref(desc), _ptr(packed), _ptr(x), M, ldx, _ptr(y), ldy,
                                  _ptr(w_out), _stream(stream)))


def cass_speculate_step(desc: qmv_desc, packed, x, y_draft, y_target, stream=None):
    """x: bf16 [n_draft + 1][ldx] (row 0 the current token); y_draft [n_draft][ldy]; y_target
    [n_draft + 1][ldy] with the same ldy."""
    M, ldx = _rows(x)
    nd, ldy = _rows(y_draft)
    mt, ldy2 = _rows(y_target)
    if nd != M - 1 or mt != M or ldy2 != ldy:
        raise ValueError("x must have n_draft + 1 rows, y_draft n_draft and y_target n_draft + 1, one ldy")
    _check(lib().cass_speculate_step(ctypes.byref(desc), _ptr(packed), _ptr(x), nd, ldx, _ptr(y_draft),
                                     _ptr(y_target), ldy, _stream(stream)))


# ----------------------------------------------------------------------------- MoE

def moe_workspace_size(E: int, topk: int, M: int, H: int, I: int) -> int:
    return int(lib().moe_workspace_size(E, topk, M, H, I))


def moe_qmv_run(gateup_desc: qmv_desc, down_desc: qmv_desc, experts, expert_stride: int, down_off: int, E: int,
                logits, topk: int, x, y, workspace, stream=None):
    M, ldx = _rows(x)
    _, ldy = _rows(y)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().moe_qmv_run(ctypes.byref(gateup_desc), ctypes.byref(down_desc), _ptr(experts), expert_stride,
                             down_off, E, _ptr(logits), topk, _ptr(x), M, ldx, _ptr(y), ldy, _ptr(workspace),
                             ws_bytes, _stream(stream)))


QMV_MOE_STATIC_SCRATCH_BYTES = 2 * 1024 * 1024


def moe_qmv_run_static(gateup_desc: qmv_desc, down_desc: qmv_desc, experts, expert_stride: int, down_off: int,
                       E: int, logits, topk: int, x, y, stream=None):
    """moe_qmv_run without a caller workspace: for callers that cannot allocate device memory, the
    library's fixed device scratch array is used instead (see include/qmv.h)."""
    M, ldx = _rows(x)
    _, ldy = _rows(y)
    _check(lib().moe_qmv_run_static(ctypes.byref(gateup_desc), ctypes.byref(down_desc), _ptr(experts),
                                    expert_stride, down_off, E, _ptr(logits), topk, _ptr(x), M, ldx, _ptr(y), ldy,
                                    _stream(stream)))


# ----------------------------------------------------------------------------- status

# ----------------------------------------------------------------------------- packed-weight files

QMV_FILE_NAME_BYTES = 64


def qmv_crc32(data, crc: int = 0) -> int:
    """CRC-32 (zip polynomial) of a bytes-like object or a host NumPy array."""
    import numpy as np
    a = np.ascontiguousarray(np.frombuffer(data, dtype=np.uint8) if isinstance(data, (bytes, bytearray)) else data)
    return int(lib().qmv_crc32(_ptr(a), a.nbytes, crc))


def qmv_file_write(path: str, items):
    """items: [(name, qmv_desc, host buffer of desc.total_bytes bytes: NumPy array or CPU tensor)]."""
    n = len(items)
    names = (ctypes.c_char_p * n)(*[nm.encode() for nm, _, _ in items])
    descs = (qmv_desc * n)(*[d for _, d, _ in items])
    for _, d, b in items:
        nb = b.nbytes if hasattr(b, "nbytes") else b.numel() * b.element_size()
        if nb < d.total_bytes:
            raise ValueError("buffer smaller than desc.total_bytes")
        if hasattr(b, "is_cuda") and b.is_cuda:
            raise ValueError("qmv_file_write takes host buffers")
    bufs = (_P * n)(*[_ptr(b) for _, _, b in items])
    _check(lib().qmv_file_write(path.encode(), n, names, descs, bufs))


class QmvFile:
    """An open packed-weight file (qmv_file_open ... qmv_file_close)."""

    def __init__(self, path: str):
        h = _P()
        _check(lib().qmv_file_open(path.encode(), ctypes.byref(h)))
        self._h = h

    def __len__(self):
        return int(lib().qmv_file_count(self._h))

    def tensor(self, index: int):
        """(name, qmv_desc) of tensor `index`."""
        name = ctypes.create_string_buffer(QMV_FILE_NAME_BYTES)
        d = qmv_desc()
        _check(lib().qmv_file_tensor(self._h, index, name, ctypes.byref(d)))
        return name.value.decode(), d

    def find(self, name: str) -> int:
        i = lib().qmv_file_find(self._h, name.encode())
        if i < 0:
            _check(i)
        return int(i)

    def load(self, index: int, dst, stream=None):
        """Copy tensor `index` (CRC-checked) into the device buffer dst."""
        nb = dst.numel() * dst.element_size()
        _check(lib().qmv_file_load(self._h, index, _ptr(dst), nb, _stream(stream)))

    def read_host(self, index: int, dst):
        nb = dst.nbytes if hasattr(dst, "nbytes") else dst.numel() * dst.element_size()
        _check(lib().qmv_file_read_host(self._h, index, _ptr(dst), nb))

    def close(self):
        if self._h:
            lib().qmv_file_close(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def qmv_check_status(stream=None) -> int:
    """Synchronize the stream and return (and clear) the device error word; raises on CUDA failure."""
    code = ctypes.c_int32(0)
    rc = lib().qmv_check_status(_stream(stream), ctypes.byref(code))
    if rc == QMV_ERR_CUDA:
        _check(rc)
    return int(code.value)
