"""Oracle for speculative KV coding -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the cpu-baseline / reference
leg of ``bench.py`` may import this package.  It wraps ``skv_oracle.c``, a
plain single-threaded C coder written from the pages of "推测式 KV 编码无损压缩
KV 缓存最高可达约 4 倍" (Speculative KV coding, lpnh.cn/news/878951); the
readings it takes where the pages are silent are listed in that file's header.
It shares no code with the CUDA library (``lossless_kv_cache_fixed_gb300``) and
never imports it.

The wrapper only marshals numpy arrays into the C calls; the arithmetic lives
in C.  ``ThreadPoolExecutor`` fans independent chunks out over host cores (the
C calls release the GIL); each chunk is still coded single-threaded.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libskv_oracle.so")
SRC = os.path.join(HERE, "skv_oracle.c")

BF16, E4M3 = 0, 1
NSYM = {BF16: 65282, E4M3: 254}
PRECISION = {BF16: 28, E4M3: 16}
OK, ERR_ARG, ERR_CAPACITY, ERR_SYMBOL, ERR_PARAM, ERR_CORRUPT = 0, -1, -2, -3, -4, -5


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE binary32/64, no contraction)."""
    os.makedirs(BUILD, exist_ok=True)
    hdr = os.path.join(HERE, "skv_oracle.h")
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC), os.path.getmtime(hdr))):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=gnu11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


class _Model(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("L", C.c_int32), ("H", C.c_int32), ("T", C.c_int32),
                ("D", C.c_int32), ("Tb", C.c_int32), ("G", C.c_int32), ("w1", C.c_int32),
                ("w3", C.c_int32), ("we", C.c_int32), ("block_scale", C.c_int32),
                ("adaptive", C.c_int32),
                ("sigma", C.c_void_p), ("E", C.c_void_p),
                ("counts", C.c_void_p)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(LIB)
        P = C.POINTER(_Model)
        u64, u32, i32, vp, dbl = C.c_uint64, C.c_uint32, C.c_int32, C.c_void_p, C.c_double
        sig = {
            "or_bf16_value": (dbl, [C.c_uint16]),
            "or_e4m3_value": (dbl, [C.c_uint8]),
            "or_phi_table": (None, [vp]),
            "or_nsym": (i32, [C.c_int]),
            "or_rank": (i32, [C.c_int, u32]),
            "or_bits": (u32, [C.c_int, i32]),
            "or_lo": (C.c_float, [C.c_int, i32]),
            "or_phi_q": (u32, [C.c_float]),
            "or_sigma_valid": (C.c_int, [C.c_float]),
            "or_cum": (u32, [P, i32, C.c_float, C.c_float]),
            "or_cum_all": (C.c_int, [P, C.c_float, C.c_float, vp]),
            "or_build_ecdf": (C.c_int, [vp, vp]),
            "or_model_hash": (u64, [P]),
            "or_num_chunks": (u64, [P]),
            "or_encode_chunk": (C.c_int, [P, vp, vp, u64, vp, u64, C.POINTER(u64)]),
            "or_decode_chunk": (C.c_int, [P, vp, u64, vp, u64, vp]),
            "or_max_encoded_bytes": (u64, [P]),
            "or_encode": (C.c_int, [P, vp, vp, vp, u64, C.POINTER(u64)]),
            "or_check_header": (C.c_int, [P, vp, u64]),
            "or_compare_chunks": (C.c_int, [P, vp, vp, vp, u64, u64, u64, C.POINTER(u64)]),
            "or_decode": (C.c_int, [P, vp, u64, vp, vp]),
            "or_scale_mult": (C.c_float, [i32]),
            "or_adaptive_table": (C.c_int, [P, vp, u64, vp, vp]),
            "or_chunk_scales": (C.c_int, [P, vp, vp, u64, vp]),
            "or_log_q": (dbl, [dbl]),
            "or_log_mass": (dbl, [dbl, dbl]),
            "or_ideal_bits_one": (dbl, [P, u32, C.c_uint16, C.c_float]),
            "or_ideal_bits": (C.c_int, [P, vp, vp, u64, u64, vp, C.POINTER(dbl)]),
            "or_model_bits_chunk": (C.c_int, [P, vp, vp, u64, C.POINTER(dbl)]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


class Model:
    """Coding model: shape, chunking and the (sigma, p-hat) tables."""

    def __init__(self, dtype, L, H, T, D, Tb, G, sigma, E=None, counts=None,
                 weights=(95, 3, 2), block_scale=False, adaptive=False):
        self.dtype = dtype
        # the order-0 baseline (weights (0, 0, 100)) reads no sigma: None is allowed
        self.sigma = None if sigma is None else np.ascontiguousarray(sigma, dtype=np.float32)
        assert self.sigma is None or self.sigma.size == L * 2 * H * D
        self.E = None if E is None else np.ascontiguousarray(E, dtype=np.uint32)
        self.counts = None if counts is None else np.ascontiguousarray(counts, dtype=np.uint64)
        if dtype == BF16:
            if self.E is None and self.counts is not None:
                self.E = build_ecdf(self.counts)
            assert self.E is not None and self.E.size == NSYM[BF16] + 1
        self.shape = (L, 2, H, T, D)
        self.s = _Model(dtype, L, H, T, D, Tb, G, weights[0], weights[1], weights[2],
                        1 if block_scale else 0, 1 if adaptive else 0, _ptr(self.sigma),
                        _ptr(self.E),
                        _ptr(self.counts))

    @property
    def ref(self):
        return C.byref(self.s)

    @property
    def n(self):
        L, _, H, T, D = self.shape
        return L * 2 * H * T * D

    def num_chunks(self):
        return int(lib().or_num_chunks(self.ref))


def phi_table():
    T = np.zeros(8193, dtype=np.uint32)
    lib().or_phi_table(_ptr(T))
    return T


def phi_q(z):
    return int(lib().or_phi_q(float(z)))


def rank(dtype, u):
    return int(lib().or_rank(dtype, int(u)))


def bits(dtype, r):
    return int(lib().or_bits(dtype, int(r)))


def lo(dtype, r):
    return float(lib().or_lo(dtype, int(r)))


def sigma_valid(s):
    return bool(lib().or_sigma_valid(float(s)))


def cum(model, r, mu, sigma):
    return int(lib().or_cum(model.ref, int(r), float(mu), float(sigma)))


def cum_all(model, mu, sigma):
    out = np.zeros(NSYM[model.dtype] + 1, dtype=np.uint32)
    lib().or_cum_all(model.ref, float(mu), float(sigma), _ptr(out))
    return out


def build_ecdf(counts):
    counts = np.ascontiguousarray(counts, dtype=np.uint64)
    assert counts.size == 65536
    E = np.zeros(NSYM[BF16] + 1, dtype=np.uint32)
    lib().or_build_ecdf(_ptr(counts), _ptr(E))
    return E


def model_hash(model):
    return int(lib().or_model_hash(model.ref))


def _as_sym(model, kv):
    dt = np.uint16 if model.dtype == BF16 else np.uint8
    kv = np.ascontiguousarray(kv).view(dt).reshape(-1)
    assert kv.size == model.n
    return kv


def _as_mu(model, mu):
    if mu is None:          # the order-0 baseline reads no mu
        return None
    mu = np.ascontiguousarray(mu).view(np.uint16).reshape(-1)
    assert mu.size == model.n
    return mu


def encode(model, kv, mu):
    """Whole container, single-threaded. Returns (rc, uint8 array)."""
    kv, mu = _as_sym(model, kv), _as_mu(model, mu)
    cap = int(lib().or_max_encoded_bytes(model.ref))
    out = np.zeros(cap, dtype=np.uint8)
    nb = C.c_uint64(0)
    rc = lib().or_encode(model.ref, _ptr(kv), _ptr(mu), _ptr(out), cap, C.byref(nb))
    return rc, out[: nb.value].copy()


def decode(model, buf, mu):
    mu = _as_mu(model, mu)
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    out = np.zeros(model.n, dtype=np.uint16 if model.dtype == BF16 else np.uint8)
    rc = lib().or_decode(model.ref, _ptr(buf), buf.size, _ptr(mu), _ptr(out))
    return rc, out


def check_header(model, buf):
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    return lib().or_check_header(model.ref, _ptr(buf), buf.size)


def compare_container(model, kv, mu, buf, threads=None, begin=0, end=None):
    """Chunks [begin, end) of container `buf` (default: all) against the oracle's
    encoding of each chunk, spread over the host cores (one slice of chunks per
    task; each chunk is still coded single-threaded).  The header is checked
    first.  Returns (status, first differing chunk or -1, threads used)."""
    kv, mu = _as_sym(model, kv), _as_mu(model, mu)
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    L = lib()
    rank(model.dtype, 0)          # the oracle's tables, built once before the threads
    rc = L.or_check_header(model.ref, _ptr(buf), buf.size)
    if rc:
        return rc, -1, 1
    nc = model.num_chunks()
    end = nc if end is None else end
    threads = threads or os.cpu_count() or 1
    nslice = max(1, min(end - begin, 16 * threads))
    cuts = [begin + (end - begin) * i // nslice for i in range(nslice + 1)]

    def one(i):
        bad = C.c_uint64(0)
        r = L.or_compare_chunks(model.ref, _ptr(kv), _ptr(mu), _ptr(buf), buf.size, cuts[i],
                                cuts[i + 1], C.byref(bad))
        return r, (int(bad.value) if r else -1)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(one, range(nslice)))
    for r, bad in res:
        if r:
            return r, bad, threads
    return OK, -1, threads


def encode_chunk(model, kv, mu, c):
    kv, mu = _as_sym(model, kv), _as_mu(model, mu)
    return _encode_chunk_raw(model, kv, mu, c)


def _encode_chunk_raw(model, kv, mu, c):
    L, _, H, T, D = model.shape
    cap = model.s.Tb * D + 2 * model.s.G + (D // 8 + 3) // 4
    out = np.zeros(cap, dtype=np.uint32)
    nw = C.c_uint64(0)
    rc = lib().or_encode_chunk(model.ref, _ptr(kv), _ptr(mu), int(c), _ptr(out), cap,
                               C.byref(nw))
    if rc:
        raise RuntimeError("oracle encode_chunk rc=%d" % rc)
    return out[: nw.value].copy()


def decode_chunk(model, words, mu, c, kv_out):
    mu = _as_mu(model, mu)
    words = np.ascontiguousarray(words, dtype=np.uint32)
    return lib().or_decode_chunk(model.ref, _ptr(words), words.size, _ptr(mu), int(c),
                                 _ptr(kv_out))


def encode_chunks(model, kv, mu, chunks, threads=None):
    """Encode the listed chunks on a thread pool; returns a list of word arrays."""
    kv, mu = _as_sym(model, kv), _as_mu(model, mu)
    threads = threads or os.cpu_count() or 1
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda c: _encode_chunk_raw(model, kv, mu, c), list(chunks)))


def ideal_bits(model, kv, mu, begin=0, end=None, per_scalar=False):
    kv, mu = _as_sym(model, kv), _as_mu(model, mu)
    end = model.n if end is None else end
    assert model.dtype == E4M3 or model.counts is not None
    ps = np.zeros(end - begin, dtype=np.float64) if per_scalar else None
    tot = C.c_double(0)
    rc = lib().or_ideal_bits(model.ref, _ptr(kv), _ptr(mu), begin, end, _ptr(ps),
                             C.byref(tot))
    if rc:
        raise RuntimeError("oracle ideal_bits rc=%d" % rc)
    return (tot.value, ps) if per_scalar else tot.value


def ideal_bits_one(model, sym, mu_bits, sigma):
    return float(lib().or_ideal_bits_one(model.ref, int(sym), int(mu_bits), float(sigma)))


def model_bits_chunk(model, kv, mu, c):
    kv, mu = _as_sym(model, kv), _as_mu(model, mu)
    b = C.c_double(0)
    rc = lib().or_model_bits_chunk(model.ref, _ptr(kv), _ptr(mu), int(c), C.byref(b))
    if rc:
        raise RuntimeError("oracle model_bits rc=%d" % rc)
    return b.value


def adaptive_table(model, kv, c):
    """(E table uint32[65283], P uint64[65282]) of chunk c of an adaptive model."""
    kv = _as_sym(model, kv)
    E = np.zeros(NSYM[BF16] + 1, dtype=np.uint32)
    P = np.zeros(NSYM[BF16], dtype=np.uint64)
    rc = lib().or_adaptive_table(model.ref, _ptr(kv), int(c), _ptr(E), _ptr(P))
    if rc:
        raise RuntimeError("oracle adaptive_table rc=%d" % rc)
    return E, P


def scale_mult(s):
    return float(lib().or_scale_mult(int(s)))


def chunk_scales(model, kv, mu, c):
    kv, mu = _as_sym(model, kv), _as_mu(model, mu)
    out = np.zeros(256, dtype=np.uint8)
    lib().or_chunk_scales(model.ref, _ptr(kv), _ptr(mu), int(c), _ptr(out))
    return out[: model.shape[4] // 8].copy()


def log_q(z):
    return float(lib().or_log_q(float(z)))


def log_mass(za, zb):
    return float(lib().or_log_mass(float(za), float(zb)))


def bf16_value(u):
    return float(lib().or_bf16_value(int(u)))


def e4m3_value(u):
    return float(lib().or_e4m3_value(int(u)))
