"""CPU oracle for the paged decode path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (``paged_kv_looped_gb300``)
never touches it, and it never touches the product: the two share no code.

The arithmetic lives in ``rlt_oracle.c`` (plain single-threaded C, fp64),
built here with gcc into ``librlt_oracle.so``; this module only marshals
numpy arrays.  Each function cites the page passage it restates:

* "Faster fuzzy minds" (dibbla.space), "When scheduler does the work": the KV
  is a flat pool of fixed-size slots addressed through a page table;
  "LOTUS": store_kv scatters each token's K/V to the slots it is handed;
  "Recurrent depth": iteration t of layer l uses bank t*L + l.
* vllm-rlt PR #152, Summary: per-plane layer map (prelude/coda on plane 0
  only); noise = f(request seed, position, channel) via a stage-wise
  SplitMix64-style hash, a 24-bit uniform and an inverse normal CDF onto
  N(0, initializer_range^2) truncated at +-3 sigma.

Every function is pinned by ``tests/test_oracle_*.py`` against something
other than itself (published SplitMix64 outputs, closed-form truncated-normal
moments, scipy's ndtri, dense numpy attention, brute-force invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rlt_oracle.c")
_LIB = os.path.join(_HERE, "librlt_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, portable flags) if it is missing or stale."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, u64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        sig = {
            "oracle_bank_map": (i32, [P, i32, i32, P]),
            "oracle_slot": (i64, [P, i32, i32, i64, i32]),
            "oracle_paged_gather": (None, [P, P, i64, i32, i32, i32, i32, P, i32, P, i32, i32, P, P]),
            "oracle_kv_append": (None, [P, P, i64, i32, i32, i32, i32, P, P, P, i32]),
            "oracle_decode_attn": (None, [P, P, P, i64, i32, i32, i32, i32, P, i32, P, i32, i32,
                                          f64, P, P, P]),
            "oracle_mix64": (u64, [u64]),
            "oracle_stage": (u64, [u64, u64]),
            "oracle_noise_key": (u64, [u64, i64, i32]),
            "oracle_noise_hash24": (None, [P, P, i64, i32, P]),
            "oracle_noise_value": (f64, [ctypes.c_uint32, f64]),
            "oracle_latent_noise_init": (None, [P, P, i64, i32, f64, P]),
            "oracle_bf16_round": (ctypes.c_uint16, [f64]),
            "oracle_rope": (None, [P, i32, i32, f64, i64, P]),
            "oracle_kv_append_rope": (None, [P, P, i64, i32, i32, i32, i32, P, P, P, P, i32, i32, f64]),
            "oracle_mark_written": (None, [P, i32, i32, P, P, P, i32]),
            "oracle_publishable_prefix": (None, [P, i32, i32, P, i32, i32, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ bank map

def bank_map(recurrent, num_planes: int):
    """(map int32[L][T], num_banks): plane 0 holds every layer, deeper planes the looped ones."""
    rec = _c(recurrent, np.uint8)
    m = np.empty((rec.size, num_planes), np.int32)
    n = _load().oracle_bank_map(_ptr(rec), rec.size, num_planes, _ptr(m))
    return m, int(n)


# ------------------------------------------------------- slots, gather, append

def slot(page_table, b: int, pos: int, page_size: int) -> int:
    pt = _c(page_table, np.int32)
    return int(_load().oracle_slot(_ptr(pt), pt.shape[1], b, pos, page_size))


def paged_gather(k_pool, v_pool, page_table, seq_lens, bank: int = 0, max_len: int | None = None):
    """Dense [B][max_len][Hkv][D] copies (bf16 bits) of each request's cached rows."""
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    nb, P, Hkv, ps, D = _pool_dims(k_pool)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    B = sl.size
    if max_len is None:
        max_len = int(sl.max()) if B else 0
    ko = np.zeros((B, max_len, Hkv, D), np.uint16)
    vo = np.zeros_like(ko)
    _load().oracle_paged_gather(_ptr(k_pool), _ptr(v_pool), P, Hkv, ps, D, bank, _ptr(pt),
                                pt.shape[1], _ptr(sl), B, max_len, _ptr(ko), _ptr(vo))
    return ko, vo


def kv_append(k_pool, v_pool, k_new, v_new, out_loc, bank: int = 0):
    """In-place store_kv on host pools (bf16 bits, [banks][pages][Hkv][ps][D] or one bank)."""
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    nb, P, Hkv, ps, D = _pool_dims(k_pool)
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    loc = _c(out_loc, np.int64)
    _load().oracle_kv_append(_ptr(k_pool), _ptr(v_pool), P, Hkv, ps, D, bank, _ptr(kn), _ptr(vn),
                             _ptr(loc), loc.size)


def _pool_dims(pool):
    if pool.ndim == 4:
        P, Hkv, ps, D = pool.shape
        return 1, P, Hkv, ps, D
    nb, P, Hkv, ps, D = pool.shape
    return nb, P, Hkv, ps, D


# ---------------------------------------------------------------- attention

def decode_attn(q, k_pool, v_pool, page_table, seq_lens, bank: int = 0, scale: float = 0.0):
    """fp64 (out [B][Hq][D], lse [B][Hq]) of softmax(q K^T * scale) V over each request's pages."""
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    nb, P, Hkv, ps, D = _pool_dims(k_pool)
    B, Hq, Dq = q.shape
    assert Dq == D and Hq % Hkv == 0
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    scratch = np.zeros(max(int(sl.max()) if B else 1, 1), np.float64)
    _load().oracle_decode_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), P, Hkv, ps, D, bank, _ptr(pt),
                               pt.shape[1], _ptr(sl), B, Hq, float(scale), _ptr(out), _ptr(lse),
                               _ptr(scratch))
    return out, lse


def decode_attn_rows(q, k_pool, v_pool, page_table, seq_lens, rows, bank: int = 0, scale: float = 0.0):
    """The oracle on a subset of requests ``rows`` only (for sampled checks of large cases)."""
    rows = np.asarray(rows, np.int64)
    pt = _c(page_table, np.int32)[rows]
    sl = _c(seq_lens, np.int32)[rows]
    return decode_attn(_c(q, np.uint16)[rows], k_pool, v_pool, pt, sl, bank, scale)


# -------------------------------------------------------------------- noise

def mix64(z: int) -> int:
    return int(_load().oracle_mix64(z & (2**64 - 1)))


def stage(h: int, x: int) -> int:
    return int(_load().oracle_stage(h & (2**64 - 1), x & (2**64 - 1)))


def noise_key(seed: int, position: int, channel: int) -> int:
    return int(_load().oracle_noise_key(seed & (2**64 - 1), position, channel))


def noise_hash24(seeds, positions, channels: int):
    s = _c(seeds, np.uint64)
    p = _c(positions, np.int64)
    out = np.empty((s.size, channels), np.uint32)
    _load().oracle_noise_hash24(_ptr(s), _ptr(p), s.size, channels, _ptr(out))
    return out


def noise_value(h24: int, initializer_range: float) -> float:
    return float(_load().oracle_noise_value(int(h24), float(initializer_range)))


def noise_values(h24, initializer_range: float):
    h = np.asarray(h24, np.uint32).ravel()
    f = _load().oracle_noise_value
    return np.array([f(int(x), float(initializer_range)) for x in h], np.float64).reshape(np.shape(h24))


def latent_noise_init(seeds, positions, channels: int, initializer_range: float):
    s = _c(seeds, np.uint64)
    p = _c(positions, np.int64)
    out = np.empty((s.size, channels), np.float64)
    _load().oracle_latent_noise_init(_ptr(s), _ptr(p), s.size, channels, float(initializer_range),
                                     _ptr(out))
    return out


# ------------------------------------------------------- RoPE, fused append

def bf16_round(x: float) -> int:
    """Correctly rounded (nearest, ties to even) bf16 bits of a double."""
    return int(_load().oracle_bf16_round(float(x)))


def rope(x, pos: int, rot_dim: int, base: float):
    """fp64 rotate-half RoPE of one row x[head_dim] at sequence position pos."""
    xx = _c(x, np.float64)
    out = np.empty_like(xx)
    _load().oracle_rope(_ptr(xx), xx.size, rot_dim, float(base), int(pos), _ptr(out))
    return out


def kv_append_rope(k_pool, v_pool, k_new, v_new, positions, out_loc, rot_dim: int, base: float, bank: int = 0):
    """In-place store_kv with the keys rotated at their positions (bf16 bits)."""
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    nb, P, Hkv, ps, D = _pool_dims(k_pool)
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    pos = _c(positions, np.int64)
    loc = _c(out_loc, np.int64)
    _load().oracle_kv_append_rope(_ptr(k_pool), _ptr(v_pool), P, Hkv, ps, D, bank, _ptr(kn), _ptr(vn),
                                  _ptr(pos), _ptr(loc), loc.size, rot_dim, float(base))


# ------------------------------------------------------ prefix publication

def mark_written(written, bank: int, request, positions, out_loc):
    """In place: written[bank][r] = max(written[bank][r], p + 1) for each appended token."""
    assert written.dtype == np.int32 and written.flags.c_contiguous
    req = _c(request, np.int32)
    _load().oracle_mark_written(_ptr(written), written.shape[1], bank, _ptr(req), _ptr(_c(positions, np.int64)),
                                _ptr(_c(out_loc, np.int64)), req.size)


def publishable_prefix(bank_map_, written, page_size: int):
    """Tokens per request written in every held (layer, plane) bank, in whole pages."""
    m = _c(bank_map_, np.int32)
    w = _c(written, np.int32)
    out = np.empty(w.shape[1], np.int32)
    _load().oracle_publishable_prefix(_ptr(m), m.shape[0], m.shape[1], _ptr(w), w.shape[1], page_size, _ptr(out))
    return out


# --------------------------------------------- extend (span) attention

def extend_rows(page_table, seq_lens, new_lens):
    """Per new query token: (request, its key count = causal limit).  Request b's n_b new
    tokens are its last n_b positions; the i-th sees keys 0 .. L_b - n_b + i."""
    req, lim = [], []
    for b, (L, n) in enumerate(zip(np.asarray(seq_lens), np.asarray(new_lens))):
        assert 0 <= n <= L
        for i in range(int(n)):
            req.append(b)
            lim.append(int(L) - int(n) + i + 1)
    return np.array(req, np.int64), np.array(lim, np.int32)


def extend_attn(q_ext, k_pool, v_pool, page_table, seq_lens, new_lens, bank: int = 0, scale: float = 0.0):
    """fp64 (out [N][Hq][D], lse [N][Hq]) of causal attention for every new token of every request
    ("Faster fuzzy minds", LOTUS: re-forwarding a span is an extend-prefill).  Each new token is a
    decode query over its own causal prefix, so this is decode_attn on per-token rows."""
    req, lim = extend_rows(page_table, seq_lens, new_lens)
    pt = np.ascontiguousarray(np.asarray(page_table, np.int32)[req])
    return decode_attn(q_ext, k_pool, v_pool, pt, lim, bank, scale)
