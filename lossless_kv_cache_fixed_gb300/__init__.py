"""Speculative KV coding on GB300 -- Python binding of libskv.so.

The functions named ``skv_*`` mirror the C ABI in ``include/skv.h`` one to one
and only marshal arguments (ctypes structs, raw device pointers, the current
CUDA stream).  ``Codec`` is a convenience wrapper that owns the workspace and
output buffers as torch tensors; every step of the coder runs in the CUDA
kernels of ``csrc/``.  There is no fallback: if the library is missing, every
call raises.
"""
from __future__ import annotations

import ctypes as C
import os

from .build import LIB, build  # noqa: F401

SKV_BF16, SKV_E4M3 = 0, 1
SKV_OP_ENCODE, SKV_OP_DECODE, SKV_OP_IDEAL_BITS, SKV_OP_MODEL_BITS = 0, 1, 2, 3
SKV_FLAG_DECODE_BISECT = 1
SKV_FLAG_BLOCK_SCALE = 2
SKV_FLAG_ORDER0 = 4
SKV_FLAG_ADAPTIVE = 8
SKV_RANGE_FIRST = 1
SKV_RANGE_PARTIAL = 2
SKV_RANGE_BITS = 4
SKV_OK, SKV_ERR_ARG, SKV_ERR_CAPACITY, SKV_ERR_SYMBOL = 0, -1, -2, -3
SKV_ERR_PARAM, SKV_ERR_CORRUPT, SKV_ERR_CUDA = -4, -5, -6
NSYM = {SKV_BF16: 65282, SKV_E4M3: 254}

EXPORTS = ("skv_max_encoded_bytes", "skv_workspace_bytes", "skv_encode", "skv_encode_with_bits",
           "skv_encode_with_bits_fused", "skv_encode_range", "skv_encode_finish",
           "skv_encode_range_bits", "skv_encode_commit",
           "skv_model_fingerprint", "skv_merge_parts", "skv_decode",
           "skv_decode_range", "skv_decode_status", "skv_ideal_bits", "skv_model_bits",
           "skv_ideal_bits_noalloc", "skv_ideal_bits_noalloc_max_channels",
           "skv_build_ecdf", "skv_phi_table", "skv_strerror", "skv_version")


class SkvParams(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("token_block", C.c_int32), ("lanes", C.c_int32),
                ("flags", C.c_int32), ("sigma", C.c_void_p), ("ecdf", C.c_void_p),
                ("phat", C.c_void_p)]


class SkvShape(C.Structure):
    _fields_ = [("layers", C.c_int32), ("kv", C.c_int32), ("heads", C.c_int32),
                ("tokens", C.c_int32), ("head_dim", C.c_int32)]


class SkvError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s: %s (%d)" % (what or "skv", skv_strerror(status), status))


_lib = None


def lib():
    """The loaded libskv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError("libskv.so is not built (%s); run __graft_entry__.build()" % LIB)
        L = C.CDLL(LIB)
        P, S = C.POINTER(SkvParams), C.POINTER(SkvShape)
        vp, sz = C.c_void_p, C.c_size_t
        sig = {
            "skv_max_encoded_bytes": (sz, [P, S]),
            "skv_workspace_bytes": (sz, [P, S, C.c_int]),
            "skv_encode": (C.c_int, [P, S, vp, vp, vp, sz, C.POINTER(sz), vp, sz, vp]),
            "skv_encode_with_bits": (C.c_int, [P, S, vp, vp, vp, sz, C.POINTER(sz), vp,
                                               C.POINTER(C.c_double), vp, sz, vp]),
            "skv_encode_with_bits_fused": (C.c_int, [P, S, C.POINTER(C.c_int)]),
            "skv_encode_range": (C.c_int, [P, S, vp, vp, C.c_uint64, C.c_uint64, C.c_int, vp, sz,
                                           vp]),
            "skv_encode_finish": (C.c_int, [P, S, vp, sz, C.POINTER(sz), vp, sz, vp]),
            "skv_encode_range_bits": (C.c_int, [P, S, C.POINTER(C.c_double), vp, sz, vp]),
            "skv_encode_commit": (C.c_int, [P, S, C.c_uint64, C.c_uint64, vp, sz, vp, vp, sz,
                                            vp]),
            "skv_model_fingerprint": (C.c_int, [P, S, C.POINTER(C.c_uint64), vp, sz, vp]),
            "skv_merge_parts": (C.c_int, [P, S, C.c_uint64, C.POINTER(vp), C.POINTER(sz), C.c_int,
                                          vp, sz, C.POINTER(sz)]),
            "skv_decode": (C.c_int, [P, S, vp, sz, vp, vp, vp, sz, vp]),
            "skv_decode_range": (C.c_int, [P, S, vp, sz, C.c_uint64, C.c_uint64, vp, vp, vp,
                                           C.c_uint64, C.c_int, vp, sz, vp]),
            "skv_decode_status": (C.c_int, [vp, vp]),
            "skv_ideal_bits": (C.c_int, [P, S, vp, vp, vp, C.POINTER(C.c_double), vp, sz, vp]),
            "skv_model_bits": (C.c_int, [P, S, vp, vp, vp, C.POINTER(C.c_double), vp, sz, vp]),
            "skv_ideal_bits_noalloc": (C.c_int, [P, S, vp, vp, vp, C.POINTER(C.c_double), vp]),
            "skv_ideal_bits_noalloc_max_channels": (sz, []),
            "skv_build_ecdf": (C.c_int, [vp, vp, vp]),
            "skv_phi_table": (C.c_int, [vp]),
            "skv_strerror": (C.c_char_p, [C.c_int]),
            "skv_version": (C.c_int, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


# ---- one-to-one wrappers of the C ABI ----

def skv_max_encoded_bytes(params: SkvParams, shape: SkvShape) -> int:
    return int(lib().skv_max_encoded_bytes(C.byref(params), C.byref(shape)))


def skv_workspace_bytes(params: SkvParams, shape: SkvShape, op: int) -> int:
    return int(lib().skv_workspace_bytes(C.byref(params), C.byref(shape), op))


def skv_encode(params, shape, kv_ptr, mu_ptr, out_ptr, out_capacity, ws_ptr, ws_bytes, stream):
    """Returns (status, container bytes)."""
    nb = C.c_size_t(0)
    rc = lib().skv_encode(C.byref(params), C.byref(shape), kv_ptr, mu_ptr, out_ptr, out_capacity,
                          C.byref(nb), ws_ptr, ws_bytes, stream)
    return rc, nb.value


def skv_encode_with_bits(params, shape, kv_ptr, mu_ptr, out_ptr, out_capacity, per_scalar_ptr,
                         ws_ptr, ws_bytes, stream):
    """Returns (status, container bytes, ideal bits)."""
    nb = C.c_size_t(0)
    tot = C.c_double(0)
    rc = lib().skv_encode_with_bits(C.byref(params), C.byref(shape), kv_ptr, mu_ptr, out_ptr,
                                    out_capacity, C.byref(nb), per_scalar_ptr, C.byref(tot), ws_ptr,
                                    ws_bytes, stream)
    return rc, nb.value, tot.value


def skv_encode_with_bits_fused(params, shape):
    """Returns (status, 1 if skv_encode_with_bits computes the bits inside the encoder)."""
    f = C.c_int(0)
    rc = lib().skv_encode_with_bits_fused(C.byref(params), C.byref(shape), C.byref(f))
    return rc, f.value


def skv_encode_range(params, shape, kv_ptr, mu_ptr, chunk_begin, chunk_end, range_flags, ws_ptr,
                     ws_bytes, stream):
    """Enqueues the encode of chunks [chunk_begin, chunk_end); returns the argument status."""
    return lib().skv_encode_range(C.byref(params), C.byref(shape), kv_ptr, mu_ptr, chunk_begin,
                                  chunk_end, range_flags, ws_ptr, ws_bytes, stream)


def skv_encode_range_bits(params, shape, ws_ptr, ws_bytes, stream):
    """Returns (status, ideal bits of the ranges encoded with SKV_RANGE_BITS)."""
    tot = C.c_double(0.0)
    rc = lib().skv_encode_range_bits(C.byref(params), C.byref(shape), C.byref(tot), ws_ptr,
                                     ws_bytes, stream)
    return rc, tot.value


def skv_encode_finish(params, shape, out_ptr, out_capacity, ws_ptr, ws_bytes, stream):
    """Returns (status, container bytes)."""
    nb = C.c_size_t(0)
    rc = lib().skv_encode_finish(C.byref(params), C.byref(shape), out_ptr, out_capacity,
                                 C.byref(nb), ws_ptr, ws_bytes, stream)
    return rc, nb.value


def skv_encode_commit(params, shape, chunk_begin, chunk_end, out_ptr, out_capacity,
                      end_bytes_ptr, ws_ptr, ws_bytes, stream):
    """Enqueues the placement of chunks [chunk_begin, chunk_end); returns the argument status."""
    return lib().skv_encode_commit(C.byref(params), C.byref(shape), chunk_begin, chunk_end,
                                   out_ptr, out_capacity, end_bytes_ptr, ws_ptr, ws_bytes, stream)


def skv_model_fingerprint(params, shape, ws_ptr, ws_bytes, stream):
    """Returns (status, the model fingerprint of a container's header)."""
    fp = C.c_uint64(0)
    rc = lib().skv_model_fingerprint(C.byref(params), C.byref(shape), C.byref(fp), ws_ptr,
                                     ws_bytes, stream)
    return rc, fp.value


def skv_merge_parts(params, shape, fingerprint, parts, out):
    """parts: host uint8 numpy arrays (containers of consecutive layer ranges);
    out: a host uint8 numpy array.  Returns (status, container bytes)."""
    n = len(parts)
    ptrs = (C.c_void_p * n)(*[pt.ctypes.data for pt in parts])
    sizes = (C.c_size_t * n)(*[pt.nbytes for pt in parts])
    nb = C.c_size_t(0)
    rc = lib().skv_merge_parts(C.byref(params), C.byref(shape), fingerprint, ptrs, sizes, n,
                               out.ctypes.data, out.nbytes, C.byref(nb))
    return rc, nb.value


def skv_decode(params, shape, in_ptr, in_bytes, mu_ptr, kv_out_ptr, ws_ptr, ws_bytes, stream):
    return lib().skv_decode(C.byref(params), C.byref(shape), in_ptr, in_bytes, mu_ptr, kv_out_ptr,
                            ws_ptr, ws_bytes, stream)


def skv_decode_range(params, shape, in_ptr, in_bytes, chunk_begin, chunk_end, mu_ptr,
                     kv_out_ptr, pages_ptr, num_pages, range_flags, ws_ptr, ws_bytes, stream):
    """Enqueues the decode of chunks [chunk_begin, chunk_end); returns the argument status."""
    return lib().skv_decode_range(C.byref(params), C.byref(shape), in_ptr, in_bytes, chunk_begin,
                                  chunk_end, mu_ptr, kv_out_ptr, pages_ptr, num_pages,
                                  range_flags, ws_ptr, ws_bytes, stream)


def skv_decode_status(ws_ptr, stream):
    return lib().skv_decode_status(ws_ptr, stream)


def skv_ideal_bits(params, shape, kv_ptr, mu_ptr, per_scalar_ptr, ws_ptr, ws_bytes, stream):
    """Returns (status, total bits)."""
    tot = C.c_double(0)
    rc = lib().skv_ideal_bits(C.byref(params), C.byref(shape), kv_ptr, mu_ptr, per_scalar_ptr,
                              C.byref(tot), ws_ptr, ws_bytes, stream)
    return rc, tot.value


def skv_model_bits(params, shape, kv_ptr, mu_ptr, per_scalar_ptr, ws_ptr, ws_bytes, stream):
    """Returns (status, total bits under the coder's own frequencies)."""
    tot = C.c_double(0)
    rc = lib().skv_model_bits(C.byref(params), C.byref(shape), kv_ptr, mu_ptr, per_scalar_ptr,
                              C.byref(tot), ws_ptr, ws_bytes, stream)
    return rc, tot.value


def skv_ideal_bits_noalloc(params, shape, kv_ptr, mu_ptr, per_scalar_ptr, stream):
    """Returns (status, total bits); scratch is the library's fixed device array."""
    tot = C.c_double(0)
    rc = lib().skv_ideal_bits_noalloc(C.byref(params), C.byref(shape), kv_ptr, mu_ptr,
                                      per_scalar_ptr, C.byref(tot), stream)
    return rc, tot.value


def skv_ideal_bits_noalloc_max_channels() -> int:
    return int(lib().skv_ideal_bits_noalloc_max_channels())


def skv_build_ecdf(counts):
    """counts: numpy uint64[65536] by bf16 pattern -> (E_q uint32[65283], p-hat float32[65282])."""
    import numpy as np
    counts = np.ascontiguousarray(counts, dtype=np.uint64)
    if counts.size != 65536:
        raise ValueError("counts must have 65536 entries")
    E = np.zeros(65283, dtype=np.uint32)
    ph = np.zeros(65282, dtype=np.float32)
    rc = lib().skv_build_ecdf(counts.ctypes.data, E.ctypes.data, ph.ctypes.data)
    if rc:
        raise SkvError(rc, "skv_build_ecdf")
    return E, ph


def skv_phi_table():
    import numpy as np
    T = np.zeros(8193, dtype=np.uint32)
    rc = lib().skv_phi_table(T.ctypes.data)
    if rc:
        raise SkvError(rc, "skv_phi_table")
    return T


def skv_strerror(status: int) -> str:
    return lib().skv_strerror(int(status)).decode()


def skv_version() -> int:
    return int(lib().skv_version())


# ---- torch convenience wrapper (buffers only) ----

def _stream_handle(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


class Codec:
    """Owns device buffers for one (model, shape) and calls the C ABI.

    sigma: float32 [L, 2, H, D] on the device; ecdf: int32/uint32 [65283]
    (bf16); phat: float32 [65282] (bf16, ideal bits only).  With
    SKV_FLAG_ORDER0 sigma and mu may be None (the baseline reads neither).
    """

    def __init__(self, dtype, L, H, T, D, token_block, lanes, sigma, ecdf=None, phat=None,
                 flags=0):
        import torch
        self.dtype = dtype
        self.sigma = None if sigma is None else sigma.contiguous()
        self.ecdf, self.phat = ecdf, phat
        self.params = SkvParams(dtype, token_block, lanes, flags, _ptr(self.sigma),
                                ecdf.data_ptr() if ecdf is not None else None,
                                phat.data_ptr() if phat is not None else None)
        self.shape = SkvShape(L, 2, H, T, D)
        self.n = L * 2 * H * T * D
        self.device = (sigma if sigma is not None else ecdf).device
        self._ws = {}
        self.max_bytes = skv_max_encoded_bytes(self.params, self.shape)
        if self.max_bytes == 0:
            raise SkvError(SKV_ERR_ARG, "Codec")
        self.torch = torch

    def workspace(self, op):
        if op not in self._ws:
            nb = skv_workspace_bytes(self.params, self.shape, op)
            self._ws[op] = self.torch.empty(max(nb, 256), dtype=self.torch.uint8,
                                            device=self.device)
        return self._ws[op]

    def kv_dtype(self):
        return self.torch.int16 if self.dtype == SKV_BF16 else self.torch.uint8

    def encode(self, kv, mu, out=None, stream=None):
        """Returns (container uint8 tensor, size in bytes)."""
        if out is None:
            out = self.torch.empty(self.max_bytes, dtype=self.torch.uint8, device=self.device)
        ws = self.workspace(SKV_OP_ENCODE)
        rc, nb = skv_encode(self.params, self.shape, kv.data_ptr(), _ptr(mu), out.data_ptr(),
                            out.numel(), ws.data_ptr(), ws.numel(), _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_encode")
        return out, nb

    def encode_with_bits(self, kv, mu, out=None, per_scalar=False, stream=None):
        """Encode and the ideal code length in one pass: (container, bytes, ideal
        bits[, per-scalar tensor])."""
        if out is None:
            out = self.torch.empty(self.max_bytes, dtype=self.torch.uint8, device=self.device)
        ps = None
        if per_scalar:
            ps = self.torch.empty(self.n, dtype=self.torch.float32, device=self.device)
        ws = self.workspace(SKV_OP_ENCODE)
        rc, nb, tot = skv_encode_with_bits(self.params, self.shape, kv.data_ptr(), _ptr(mu),
                                           out.data_ptr(), out.numel(),
                                           ps.data_ptr() if ps is not None else None,
                                           ws.data_ptr(), ws.numel(), _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_encode_with_bits")
        return (out, nb, tot, ps) if per_scalar else (out, nb, tot)

    def encode_with_bits_fused(self):
        """True where encode_with_bits computes the bits inside the encoder."""
        rc, f = skv_encode_with_bits_fused(self.params, self.shape)
        if rc:
            raise SkvError(rc, "skv_encode_with_bits_fused")
        return bool(f)

    def encode_range(self, kv, mu, chunk_begin, chunk_end, first=False, bits=False,
                     stream=None):
        """Enqueue the encode of chunks [chunk_begin, chunk_end) (no synchronisation);
        bits: their ideal bits too, added to the total encode_range_bits reads."""
        ws = self.workspace(SKV_OP_ENCODE)
        flags = (SKV_RANGE_FIRST if first else 0) | (SKV_RANGE_BITS if bits else 0)
        rc = skv_encode_range(self.params, self.shape, kv.data_ptr(), _ptr(mu), chunk_begin,
                              chunk_end, flags, ws.data_ptr(), ws.numel(), _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_encode_range")

    def encode_range_bits(self, stream=None):
        """Ideal bits of the ranges encoded with bits=True since the first one."""
        ws = self.workspace(SKV_OP_ENCODE)
        rc, tot = skv_encode_range_bits(self.params, self.shape, ws.data_ptr(), ws.numel(),
                                        _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_encode_range_bits")
        return tot

    def encode_finish(self, out=None, stream=None):
        """The container from the chunk ranges encoded so far: (tensor, bytes)."""
        if out is None:
            out = self.torch.empty(self.max_bytes, dtype=self.torch.uint8, device=self.device)
        ws = self.workspace(SKV_OP_ENCODE)
        rc, nb = skv_encode_finish(self.params, self.shape, out.data_ptr(), out.numel(),
                                   ws.data_ptr(), ws.numel(), _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_encode_finish")
        return out, nb

    def encode_commit(self, chunk_begin, chunk_end, out, end_bytes=None, stream=None):
        """Place the encoded chunks [chunk_begin, chunk_end) in `out` (no
        synchronisation); encode_finish(out=out) writes the header.  end_bytes:
        an int64 tensor element (device or pinned host) that receives the
        container's size so far."""
        ws = self.workspace(SKV_OP_ENCODE)
        rc = skv_encode_commit(self.params, self.shape, chunk_begin, chunk_end, out.data_ptr(),
                               out.numel(), _ptr(end_bytes), ws.data_ptr(), ws.numel(),
                               _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_encode_commit")

    def fingerprint(self, stream=None):
        ws = self.workspace(SKV_OP_IDEAL_BITS)
        rc, fp = skv_model_fingerprint(self.params, self.shape, ws.data_ptr(), ws.numel(),
                                       _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_model_fingerprint")
        return fp

    def num_chunks(self):
        s, tb = self.shape, self.params.token_block
        return s.layers * 2 * s.heads * ((s.tokens + tb - 1) // tb)

    def decode(self, buf, nbytes, mu, out=None, stream=None):
        if out is None:
            out = self.torch.empty(self.n, dtype=self.kv_dtype(), device=self.device)
        ws = self.workspace(SKV_OP_DECODE)
        rc = skv_decode(self.params, self.shape, buf.data_ptr(), nbytes, _ptr(mu),
                        out.data_ptr(), ws.data_ptr(), ws.numel(), _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_decode")
        return out

    def decode_range(self, buf, nbytes, chunk_begin, chunk_end, mu, out, pages=None,
                     num_pages=0, first=False, partial=False, stream=None):
        """Enqueue the decode of chunks [chunk_begin, chunk_end) into `out` (the
        [L,2,H,T,D] tensor, or a page pool when `pages` maps chunks to pages).
        partial: a container still being committed (nbytes = its capacity).
        No synchronisation; call decode_status() for the accumulated status."""
        ws = self.workspace(SKV_OP_DECODE)
        flags = (SKV_RANGE_FIRST if first else 0) | (SKV_RANGE_PARTIAL if partial else 0)
        rc = skv_decode_range(self.params, self.shape, buf.data_ptr(), nbytes, chunk_begin,
                              chunk_end, _ptr(mu), out.data_ptr(), _ptr(pages), num_pages,
                              flags, ws.data_ptr(), ws.numel(), _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_decode_range")

    def decode_status(self, stream=None):
        rc = skv_decode_status(self.workspace(SKV_OP_DECODE).data_ptr(), _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_decode_status")

    def ideal_bits(self, kv, mu, per_scalar=False, stream=None):
        ws = self.workspace(SKV_OP_IDEAL_BITS)
        ps = None
        if per_scalar:
            ps = self.torch.empty(self.n, dtype=self.torch.float32, device=self.device)
        rc, tot = skv_ideal_bits(self.params, self.shape, kv.data_ptr(), _ptr(mu),
                                 ps.data_ptr() if ps is not None else None, ws.data_ptr(),
                                 ws.numel(), _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_ideal_bits")
        return (tot, ps) if per_scalar else tot

    def model_bits(self, kv, mu, per_scalar=False, stream=None):
        """Code length under the coder's own frequencies: total (and per scalar)."""
        ws = self.workspace(SKV_OP_MODEL_BITS)
        ps = None
        if per_scalar:
            ps = self.torch.empty(self.n, dtype=self.torch.float32, device=self.device)
        rc, tot = skv_model_bits(self.params, self.shape, kv.data_ptr(), _ptr(mu),
                                 ps.data_ptr() if ps is not None else None, ws.data_ptr(),
                                 ws.numel(), _stream_handle(stream))
        if rc:
            raise SkvError(rc, "skv_model_bits")
        return (tot, ps) if per_scalar else tot
