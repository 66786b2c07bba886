"""Python binding of librlt, the sm_103a paged-KV decode path for looped transformers.

Argument marshalling only: every step of the path runs in the CUDA kernels of
``librlt.so`` behind the C ABI declared in ``include/rlt.h``.  PyTorch
supplies device memory and streams.  There is no CPU fallback: if the library
has not been built, every call raises.

Functions keep the C names:

* ``rlt_bank_map``          (layer, plane) -> KV bank map (host).
* ``rlt_bank_index``        one (layer, plane) entry of that map (host).
* ``rlt_kv_append``         store_kv: scatter this step's K/V rows to their slots.
* ``rlt_paged_decode_attn`` split-K paged GQA decode attention (+ combine).
* ``rlt_latent_noise_init`` position-keyed truncated-normal latent noise.
* ``rlt_noise_hash24``      the 24-bit uniforms behind that noise.
* ``rlt_paged_gather``      page-table gather into dense rows (for checks).
* ``rlt_validate_batch``    host validation of page tables and append slots.
* ``rlt_get_device_error``  read and clear the kernels' error bits.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "RltError", "KVPool", "library_path", "load", "rlt_bank_map", "rlt_bank_index", "rlt_kv_append",
    "rlt_paged_decode_workspace_size", "rlt_paged_decode_attn", "rlt_paged_decode_attn_noalloc",
    "rlt_latent_noise_init",
    "rlt_noise_hash24", "rlt_paged_gather", "rlt_validate_batch", "rlt_get_device_error", "rlt_debug_fault_next_decode",
    "rlt_version", "PrefixPlan", "rlt_plan_prefix", "rlt_choose_chunk_tiles", "rlt_paged_decode_attn_prefix",
    "rlt_paged_decode_prefix_workspace_size", "rlt_kv_append_rope", "rlt_publishable_prefix",
    "ExtendPlan", "rlt_plan_extend", "rlt_paged_extend_attn", "ATTN_EARLY_START", "DEVERR_BAD_PAGE", "DEVERR_BAD_SLOT", "DEVERR_TIMEOUT", "DEVERR_BAD_LEN",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "librlt.so")

STATUS = {0: "RLT_OK", 1: "RLT_ERR_INVALID_ARG", 2: "RLT_ERR_OUT_OF_RANGE", 3: "RLT_ERR_UNSUPPORTED",
          4: "RLT_ERR_WORKSPACE_TOO_SMALL", 5: "RLT_ERR_CUDA"}
DEVERR_BAD_PAGE, DEVERR_BAD_SLOT, DEVERR_TIMEOUT, DEVERR_BAD_LEN = 1, 2, 4, 8
ATTN_EARLY_START = 1     # RLT_ATTN_EARLY_START: see include/rlt.h


class RltError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class rlt_kv_pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("num_banks", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


RLT_BF16 = 0


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load librlt.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with paged_kv_looped_gb300.build.build() "
                           "(nvcc, sm_103a); this package has no CPU fallback")
    lib = ctypes.CDLL(_LIB_PATH)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    u32 = ctypes.c_uint32
    pool_p = ctypes.POINTER(rlt_kv_pool)
    sigs = {
        "rlt_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "rlt_version": (i32, []),
        "rlt_bank_map": (i32, [P, i32, i32, P]),
        "rlt_bank_index": (i32, [P, i32, i32, i32, i32]),
        "rlt_kv_append": (ctypes.c_int, [pool_p, i32, P, P, P, i32, P]),
        "rlt_paged_decode_workspace_size": (sz, [i32, i32, i32, i32, i32, i32]),
        "rlt_paged_decode_attn": (ctypes.c_int, [pool_p, i32, P, P, P, i32, P, i32, P, i32, i32, f32, P, P, P,
                                                 sz, i32, u32, P]),
        "rlt_latent_noise_init": (ctypes.c_int, [P, P, P, i64, i32, f32, P]),
        "rlt_noise_hash24": (ctypes.c_int, [P, P, P, i64, i32, P]),
        "rlt_paged_gather": (ctypes.c_int, [pool_p, i32, P, i32, P, i32, i32, P, P, P]),
        "rlt_paged_decode_attn_noalloc": (ctypes.c_int, [pool_p, i32, P, i32, P, i32, P, i32, i32, f32, P, P,
                                                         i32, P]),
        "rlt_validate_batch": (ctypes.c_int, [P, i32, P, i32, P, i64, i32]),
        "rlt_plan_prefix": (ctypes.c_int, [P, i32, P, i32, i32, i32, i32, i32, P, i32, P, P, i32, P, P]),
        "rlt_paged_decode_prefix_workspace_size": (sz, [i32, i32, i32, i32, i32, i32, i32]),
        "rlt_choose_chunk_tiles": (i32, [P, i32, P, i32, i32, i32, i32, i32, i32]),
        "rlt_paged_decode_attn_prefix": (ctypes.c_int, [pool_p, i32, P, P, P, i32, P, i32, P, i32, i32, P, P, P, P, i32,
                                                        i32, i32, i32, i32, f32, P, P, P, sz, i32, i32, u32, P]),
        "rlt_get_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
        "rlt_debug_fault_next_decode": (ctypes.c_int, [ctypes.c_uint64]),
        "rlt_kv_append_rope": (ctypes.c_int, [pool_p, i32, P, P, P, P, i32, i32, ctypes.c_double, P, P, i32, P]),
        "rlt_publishable_prefix": (ctypes.c_int, [P, i32, i32, i32, P, P]),
        "rlt_plan_extend": (ctypes.c_int, [P, P, i32, i32, i32, i32, P, i32, P, P, i32, P, P, P]),
        "rlt_paged_extend_workspace_size": (sz, [i32, i32, i32, i32]),
        "rlt_paged_extend_attn": (ctypes.c_int, [pool_p, i32, P, i32, i32, P, i32, i32, P, P, P, P, P, i32, i32,
                                                 i32, i32, f32, P, P, P, sz, i32, u32, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != 0:
        raise RltError(status, where)


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _host(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


class KVPool:
    """A paged KV pool: bf16 CUDA tensors k, v of shape [banks][pages][Hkv][page_size][D]."""

    def __init__(self, k, v):
        import torch
        if k.shape != v.shape or k.dim() != 5:
            raise ValueError("k and v must both be [banks][pages][kv_heads][page_size][head_dim]")
        _dev(k, torch.bfloat16, "k")
        _dev(v, torch.bfloat16, "v")
        self.k, self.v = k, v
        nb, P, Hkv, ps, D = k.shape
        self.num_banks, self.num_pages, self.num_kv_heads, self.page_size, self.head_dim = nb, P, Hkv, ps, D
        self.struct = rlt_kv_pool(k.data_ptr(), v.data_ptr(), P, nb, Hkv, ps, D, RLT_BF16)

    @classmethod
    def empty(cls, num_banks, num_pages, num_kv_heads, page_size, head_dim, device="cuda"):
        import torch
        shape = (num_banks, num_pages, num_kv_heads, page_size, head_dim)
        return cls(torch.empty(shape, dtype=torch.bfloat16, device=device),
                   torch.empty(shape, dtype=torch.bfloat16, device=device))


# ---------------------------------------------------------------- host calls

def rlt_version() -> int:
    return int(load().rlt_version())


def rlt_bank_map(recurrent, num_planes: int):
    """(map int32 [num_layers][num_planes], num_banks); -1 where a plane does not hold a layer."""
    rec, rp = _host(recurrent, np.uint8)
    out = np.empty((rec.size, num_planes), np.int32)
    n = load().rlt_bank_map(rp, rec.size, num_planes, out.ctypes.data_as(ctypes.c_void_p))
    if n < 0:
        raise RltError(-n, "rlt_bank_map")
    return out, int(n)


def rlt_bank_index(bank_map, layer: int, plane: int) -> int:
    """The bank holding (layer, plane) in a map from rlt_bank_map, or -1 where the plane does not hold it."""
    m, mp = _host(bank_map, np.int32)
    if m.ndim != 2:
        raise ValueError("bank_map must be int32 [num_layers][num_planes]")
    return int(load().rlt_bank_index(mp, m.shape[0], m.shape[1], int(layer), int(plane)))


def rlt_validate_batch(page_table, seq_lens, new_slots, num_pages: int, page_size: int) -> int:
    """Host check of a decode batch; returns the status code (0 = valid)."""
    pt, ptp = _host(page_table, np.int32)
    sl, slp = _host(seq_lens, np.int32)
    ns, nsp = (None, None) if new_slots is None else _host(new_slots, np.int64)
    return int(load().rlt_validate_batch(ptp, pt.shape[1] if pt.ndim == 2 else 0, slp, sl.size, nsp,
                                         num_pages, page_size))


def rlt_get_device_error() -> int:
    """Read and clear the device error bits of the current device (synchronises it)."""
    v = ctypes.c_uint32(0)
    _check(load().rlt_get_device_error(ctypes.byref(v)), "rlt_get_device_error")
    return int(v.value)


def rlt_debug_fault_next_decode(wait_limit_ns: int):
    """Test hook: the next rlt_paged_decode_attn of this thread runs with this copy-wait limit and
    one tile copy left unissued, so that a wait runs out (see include/rlt.h)."""
    _check(load().rlt_debug_fault_next_decode(int(wait_limit_ns)), "rlt_debug_fault_next_decode")


# ------------------------------------------------------------- device calls

def rlt_kv_append(pool: KVPool, bank: int, k_new, v_new, out_loc, stream=None):
    """store_kv: k_new/v_new bf16 [N][Hkv][D], out_loc int64 [N] (negative = skip)."""
    import torch
    n = int(out_loc.numel())
    if k_new.shape != (n, pool.num_kv_heads, pool.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [N][num_kv_heads][head_dim] with N = out_loc.numel()")
    _check(load().rlt_kv_append(ctypes.byref(pool.struct), bank, _dev(k_new, torch.bfloat16, "k_new"),
                                _dev(v_new, torch.bfloat16, "v_new"), _dev(out_loc, torch.int64, "out_loc"),
                                n, _stream(stream)), "rlt_kv_append")


def rlt_kv_append_rope(pool: KVPool, bank: int, k_new, v_new, positions, out_loc, rot_dim: int,
                       rope_base: float, request=None, written=None, stream=None):
    """store_kv with RoPE on the keys at each token's sequence position (same for every plane)."""
    import torch
    n = int(out_loc.numel())
    batch = int(written.shape[1]) if written is not None else 0
    _check(load().rlt_kv_append_rope(
        ctypes.byref(pool.struct), bank, _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        _dev(positions, torch.int64, "positions"), _dev(out_loc, torch.int64, "out_loc"), n, int(rot_dim),
        float(rope_base), _dev(request, torch.int32, "request") if request is not None else ctypes.c_void_p(0),
        _dev(written, torch.int32, "written") if written is not None else ctypes.c_void_p(0), batch,
        _stream(stream)), "rlt_kv_append_rope")


def rlt_publishable_prefix(written, page_size: int, out=None, stream=None):
    """Tokens per request written in every bank (every held layer-plane), in whole pages."""
    import torch
    num_banks, batch = int(written.shape[0]), int(written.shape[1])
    if out is None:
        out = torch.empty(batch, dtype=torch.int32, device=written.device)
    _check(load().rlt_publishable_prefix(_dev(written, torch.int32, "written") if num_banks else ctypes.c_void_p(0),
                                         num_banks, batch, int(page_size), _dev(out, torch.int32, "out"),
                                         _stream(stream)), "rlt_publishable_prefix")
    return out


def rlt_paged_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                                    split_tokens=0) -> int:
    return int(load().rlt_paged_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                      max_seq_len, split_tokens))


def _check_q_out(pool, q, out, lse_out):
    """q [B][Hq][D] against the pool's head_dim; out (if given) shaped like q, lse_out [B][Hq].
    The C ABI takes no head_dim for q: a mismatch here would read and write past the arrays."""
    if q.dim() != 3:
        raise ValueError("q must be [B][Hq][head_dim]")
    B, Hq, D = q.shape
    if D != pool.head_dim:
        raise ValueError(f"q head_dim {D} does not match the pool's {pool.head_dim}")
    if out is not None and tuple(out.shape) != (B, Hq, D):
        raise ValueError(f"out must be [B][Hq][D] = {(B, Hq, D)}")
    if lse_out is not None and tuple(lse_out.shape) != (B, Hq):
        raise ValueError(f"lse_out must be [B][Hq] = {(B, Hq)}")


def _new_rows(k_new, v_new, B, Hkv, D):
    """Device pointers of the optional fused-append rows (bf16 [B][Hkv][D] each, or both None)."""
    import torch
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is None:
        return ctypes.c_void_p(0), ctypes.c_void_p(0)
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if tuple(t.shape) != (B, Hkv, D):
            raise ValueError(f"{name} must be [B][Hkv][D] = {(B, Hkv, D)}")
    return _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new")


def rlt_paged_decode_attn(pool: KVPool, bank: int, q, page_table, seq_lens, max_seq_len: int,
                          out=None, lse_out=None, workspace=None, scale: float = 0.0,
                          split_tokens: int = 0, stream=None, k_new=None, v_new=None, early_start: bool = False):
    """Paged decode attention of one bank. q bf16 [B][Hq][D]; page_table int32 [B][max_pages];
    seq_lens int32 [B].  With k_new / v_new (bf16 [B][Hkv][D]) each request's new token is
    stored at position seq_lens[b] - 1 by the same call (fused append).  early_start sets
    RLT_ATTN_EARLY_START (the call may start while the kernel ahead of it runs; see rlt.h for
    what that kernel must not write).  Returns out."""
    import torch
    _check_q_out(pool, q, out, lse_out)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    ws_need = rlt_paged_decode_workspace_size(B, Hq, pool.num_kv_heads, D, max_seq_len, split_tokens)
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    lse_ptr = _dev(lse_out, torch.float32, "lse_out") if lse_out is not None else ctypes.c_void_p(0)
    if page_table.dim() != 2 or page_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("page_table must be [B][max_pages] and seq_lens [B]")
    kn, vn = _new_rows(k_new, v_new, B, pool.num_kv_heads, D)
    _check(load().rlt_paged_decode_attn(
        ctypes.byref(pool.struct), bank, _dev(q, torch.bfloat16, "q"), kn, vn, Hq,
        _dev(page_table, torch.int32, "page_table"), page_table.shape[1],
        _dev(seq_lens, torch.int32, "seq_lens"), B, int(max_seq_len), float(scale),
        _dev(out, torch.bfloat16, "out"), lse_ptr, ws_ptr, ws_bytes, int(split_tokens),
        ATTN_EARLY_START if early_start else 0, _stream(stream)), "rlt_paged_decode_attn")
    return out


def rlt_paged_decode_attn_noalloc(pool: KVPool, bank: int, q, page_table, seq_lens, max_seq_len: int,
                                  out=None, lse_out=None, scale: float = 0.0, split_tokens: int = 0,
                                  stream=None):
    """rlt_paged_decode_attn with the split-K partials in the library's fixed scratch array.

    For callers that cannot allocate device memory at the point of the call (a host
    framework that owns all device allocations, or a decode loop that must not
    risk a synchronising cudaMalloc).  Allocates nothing when ``out`` is given.
    Calls on one device share the scratch array: calls that overlap on the GPU race.
    """
    import torch
    _check_q_out(pool, q, out, lse_out)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    lse_ptr = _dev(lse_out, torch.float32, "lse_out") if lse_out is not None else ctypes.c_void_p(0)
    if page_table.dim() != 2 or page_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("page_table must be [B][max_pages] and seq_lens [B]")
    _check(load().rlt_paged_decode_attn_noalloc(
        ctypes.byref(pool.struct), bank, _dev(q, torch.bfloat16, "q"), Hq,
        _dev(page_table, torch.int32, "page_table"), page_table.shape[1],
        _dev(seq_lens, torch.int32, "seq_lens"), B, int(max_seq_len), float(scale),
        _dev(out, torch.bfloat16, "out"), lse_ptr, int(split_tokens), _stream(stream)),
        "rlt_paged_decode_attn_noalloc")
    return out


NOALLOC_SCRATCH_BYTES = 64 << 20


def rlt_latent_noise_init(seeds, positions, channels: int, initializer_range: float, out=None,
                          stream=None):
    """fp32 [rows][channels] truncated-normal noise keyed by (seed, position, channel)."""
    import torch
    n = int(seeds.numel())
    if positions.numel() != n:
        raise ValueError("seeds and positions must have one entry per row")
    if out is None:
        out = torch.empty((n, channels), dtype=torch.float32, device=seeds.device)
    _check(load().rlt_latent_noise_init(_dev(out, torch.float32, "out"), _dev(seeds, torch.uint64, "seeds")
                                        if seeds.dtype == torch.uint64 else _dev(seeds, torch.int64, "seeds"),
                                        _dev(positions, torch.int64, "positions"), n, channels,
                                        float(initializer_range), _stream(stream)),
           "rlt_latent_noise_init")
    return out


def rlt_noise_hash24(seeds, positions, channels: int, out=None, stream=None):
    """uint32-valued (stored as int32) [rows][channels] 24-bit uniforms of the noise."""
    import torch
    n = int(seeds.numel())
    if out is None:
        out = torch.empty((n, channels), dtype=torch.int32, device=seeds.device)
    _check(load().rlt_noise_hash24(_dev(out, torch.int32, "out"), _dev(seeds, seeds.dtype, "seeds"),
                                   _dev(positions, torch.int64, "positions"), n, channels,
                                   _stream(stream)), "rlt_noise_hash24")
    return out


def rlt_paged_gather(pool: KVPool, bank: int, page_table, seq_lens, max_len: int, k_out=None,
                     v_out=None, stream=None):
    """Dense bf16 [B][max_len][Hkv][D] copies of each request's cached K and V rows."""
    import torch
    B = int(seq_lens.numel())
    shape = (B, max_len, pool.num_kv_heads, pool.head_dim)
    if k_out is None:
        k_out = torch.zeros(shape, dtype=torch.bfloat16, device=pool.k.device)
    if v_out is None:
        v_out = torch.zeros(shape, dtype=torch.bfloat16, device=pool.k.device)
    _check(load().rlt_paged_gather(ctypes.byref(pool.struct), bank, _dev(page_table, torch.int32, "page_table"),
                                   page_table.shape[1], _dev(seq_lens, torch.int32, "seq_lens"), B,
                                   int(max_len), _dev(k_out, torch.bfloat16, "k_out"),
                                   _dev(v_out, torch.bfloat16, "v_out"), _stream(stream)),
           "rlt_paged_gather")
    return k_out, v_out


# ------------------------------------------------------------ shared prefixes

SEG_FIELDS = 8


class PrefixPlan:
    """Host result of rlt_plan_prefix plus (after ``.to(device)``) its device copies."""

    def __init__(self, segments, members, member_limit, request_prefix, sizes, chunk_tiles, query_group):
        self.segments = segments            # int32 [n][8]
        self.members = members              # int32 [entries], ascending limits within a segment
        self.member_limit = member_limit    # int32 [entries]: tokens each member shares in its segment
        self.request_prefix = request_prefix  # int32 [B][2]
        self.num_segments, self.member_entries, self.max_chunks, self.max_prefix_slots, \
            self.max_members, self.max_rest_len, self.work_units = (int(x) for x in sizes)
        self.chunk_tiles = chunk_tiles
        self.query_group = query_group
        self.dev = None

    def to(self, device):
        import torch
        def t(a):
            a = np.ascontiguousarray(a, np.int32).reshape(-1)
            return torch.from_numpy(a if a.size else np.zeros(1, np.int32)).to(device)
        self.dev = (t(self.segments), t(self.members), t(self.member_limit), t(self.request_prefix))
        return self


def rlt_plan_prefix(page_table, seq_lens, page_size: int, chunk_tiles: int = 4,
                    private_tails: bool = False, query_group: int = 1) -> PrefixPlan:
    """Find the 128-token tiles several requests share (host arrays in, host plan out).
    With ``private_tails`` every request's remaining tokens get a one-member segment too.
    ``query_group`` = num_q_heads / num_kv_heads of the attention the plan is for."""
    pt, ptp = _host(page_table, np.int32)
    sl, slp = _host(seq_lens, np.int32)
    B = sl.size
    req = np.zeros((B, 2), np.int32)
    sizes = np.zeros(7, np.int32)
    lib = load()
    tails = 1 if private_tails else 0
    # one call with room for the usual plan (segments <= 2B: fewer than B shared member sets
    # plus B tails); a plan that needs more reports its sizes and is made again
    seg_cap, mem_cap = 2 * B + 1, 4 * B + 1
    for _ in range(2):
        seg = np.zeros((seg_cap, SEG_FIELDS), np.int32)
        mem = np.zeros(mem_cap, np.int32)
        lim = np.zeros(mem_cap, np.int32)
        st = lib.rlt_plan_prefix(ptp, pt.shape[1], slp, B, page_size, chunk_tiles, query_group, tails,
                                 seg.ctypes.data_as(ctypes.c_void_p), seg_cap,
                                 mem.ctypes.data_as(ctypes.c_void_p), lim.ctypes.data_as(ctypes.c_void_p),
                                 mem_cap, req.ctypes.data_as(ctypes.c_void_p),
                                 sizes.ctypes.data_as(ctypes.c_void_p))
        if st != 2:
            break
        seg_cap, mem_cap = max(int(sizes[0]), 1), max(int(sizes[1]), 1)
    _check(st, "rlt_plan_prefix")
    n = int(sizes[0])
    return PrefixPlan(seg[:n], mem[: int(sizes[1])], lim[: int(sizes[1])], req, sizes, chunk_tiles, query_group)


def rlt_choose_chunk_tiles(page_table, seq_lens, page_size: int, query_group: int, private_tails: bool,
                           num_kv_heads: int, num_ctas: int) -> int:
    """Tiles per work item for rlt_plan_prefix (host arrays in): see the C declaration."""
    pt, ptp = _host(page_table, np.int32)
    sl, slp = _host(seq_lens, np.int32)
    r = int(load().rlt_choose_chunk_tiles(ptp, pt.shape[1], slp, sl.size, int(page_size), int(query_group),
                                          1 if private_tails else 0, int(num_kv_heads), int(num_ctas)))
    if r < 1:
        raise RltError(-r, "rlt_choose_chunk_tiles")
    return r


def rlt_paged_decode_prefix_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_rest_len,
                                           max_prefix_slots, split_tokens=0) -> int:
    return int(load().rlt_paged_decode_prefix_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                             max_rest_len, max_prefix_slots, split_tokens))


def rlt_paged_decode_attn_prefix(pool: KVPool, bank: int, q, page_table, seq_lens, max_seq_len: int,
                                 plan: PrefixPlan, out=None, lse_out=None, workspace=None, scale: float = 0.0,
                                 split_tokens: int = 0, max_ctas: int = 0, stream=None, k_new=None, v_new=None,
                                 early_start: bool = False):
    """Paged decode attention reading shared-prefix tiles once (plan from rlt_plan_prefix, .to(device)).
    k_new / v_new: the fused append, and early_start, as in rlt_paged_decode_attn."""
    import torch
    _check_q_out(pool, q, out, lse_out)
    B, Hq, D = q.shape
    if page_table.dim() != 2 or page_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("page_table must be [B][max_pages] and seq_lens [B]")
    if plan.num_segments and plan.query_group != Hq // pool.num_kv_heads:
        raise ValueError("the plan was built for another query group")
    if plan.dev is None:
        plan.to(q.device)
    if out is None:
        out = torch.empty_like(q)
    rest = plan.max_rest_len if plan.num_segments else int(max_seq_len)
    need = rlt_paged_decode_prefix_workspace_size(B, Hq, pool.num_kv_heads, D, rest,
                                                  plan.max_prefix_slots, split_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    lse_ptr = _dev(lse_out, torch.float32, "lse_out") if lse_out is not None else ctypes.c_void_p(0)
    seg, mem, lim, req = plan.dev
    kn, vn = _new_rows(k_new, v_new, B, pool.num_kv_heads, D)
    _check(load().rlt_paged_decode_attn_prefix(
        ctypes.byref(pool.struct), bank, _dev(q, torch.bfloat16, "q"), kn, vn, Hq,
        _dev(page_table, torch.int32, "page_table"), page_table.shape[1],
        _dev(seq_lens, torch.int32, "seq_lens"), B, int(max_seq_len),
        _dev(seg, torch.int32, "segments"), _dev(mem, torch.int32, "members"),
        _dev(lim, torch.int32, "member_limit"), _dev(req, torch.int32, "request_prefix"), plan.num_segments, plan.work_units,
        plan.max_prefix_slots, plan.chunk_tiles, rest, float(scale),
        _dev(out, torch.bfloat16, "out"), lse_ptr, ctypes.c_void_p(workspace.data_ptr()),
        workspace.numel() * workspace.element_size(), int(split_tokens), int(max_ctas),
        ATTN_EARLY_START if early_start else 0, _stream(stream)), "rlt_paged_decode_attn_prefix")
    return out


# ------------------------------------------------------ extend attention

class ExtendPlan:
    """Host output of rlt_plan_extend; .to(device) uploads it for rlt_paged_extend_attn."""

    def __init__(self, segments, members, member_limit, row_prefix, row_len, sizes, chunk_tiles, query_group):
        self.segments, self.members, self.member_limit = segments, members, member_limit
        self.row_prefix, self.row_len = row_prefix, row_len
        (self.num_segments, self.num_rows, self.max_chunks, self.max_slots, self.max_members, _,
         self.work_units) = (int(x) for x in sizes)
        self.chunk_tiles, self.query_group = chunk_tiles, query_group
        self.dev = None

    def to(self, device):
        import torch
        self.dev = [torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)
                    for a in (self.segments, self.members, self.member_limit, self.row_prefix, self.row_len)]
        return self


def rlt_plan_extend(seq_lens, new_lens, page_size: int, chunk_tiles: int = 4, query_group: int = 1) -> ExtendPlan:
    """Lay out causal extend attention (new_lens[b] last tokens of request b) for the tensor-core kernel."""
    sl, _ = _host(seq_lens, np.int32)
    nl, _ = _host(new_lens, np.int32)
    B = sl.size
    sizes = np.zeros(7, np.int32)
    args = lambda seg, mem, lim, rp, rl, ms, mm: (
        sl.ctypes.data_as(ctypes.c_void_p), nl.ctypes.data_as(ctypes.c_void_p), B, page_size, chunk_tiles,
        query_group, seg, ms, mem, lim, mm, rp, rl, sizes.ctypes.data_as(ctypes.c_void_p))
    z = ctypes.c_void_p(0)
    st = load().rlt_plan_extend(*args(z, z, z, z, z, 0, 0))
    if st not in (0, 2):
        _check(st, "rlt_plan_extend")
    nseg, rows = int(sizes[0]), int(sizes[1])
    seg = np.zeros((max(nseg, 1), 8), np.int32)
    mem = np.zeros(max(rows, 1), np.int32)
    lim = np.zeros(max(rows, 1), np.int32)
    rp = np.zeros((max(rows, 1), 2), np.int32)
    rl = np.zeros(max(rows, 1), np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(load().rlt_plan_extend(*args(p(seg), p(mem), p(lim), p(rp), p(rl), seg.shape[0], mem.size)),
           "rlt_plan_extend")
    return ExtendPlan(seg[:nseg], mem[:rows], lim[:rows], rp[:rows], rl[:rows], sizes, chunk_tiles, query_group)


def rlt_paged_extend_attn(pool: KVPool, bank: int, q, page_table, plan: ExtendPlan, out=None, lse_out=None,
                          workspace=None, scale: float = 0.0, max_ctas: int = 0, stream=None,
                          early_start: bool = False):
    """Causal extend attention: q/out bf16 [new tokens][Hq][D] packed request by request.
    early_start as in rlt_paged_decode_attn."""
    import torch
    _check_q_out(pool, q, out, lse_out)
    N, Hq, D = q.shape
    if plan.num_rows != N:
        raise ValueError("the plan was built for another number of new tokens")
    if plan.num_segments and plan.query_group != Hq // pool.num_kv_heads:
        raise ValueError("the plan was built for another query group")
    if plan.dev is None:
        plan.to(q.device)
    if out is None:
        out = torch.empty_like(q)
    need = int(load().rlt_paged_extend_workspace_size(N, Hq, D, max(plan.max_slots, 1)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    lse_ptr = _dev(lse_out, torch.float32, "lse_out") if lse_out is not None else ctypes.c_void_p(0)
    seg, mem, lim, rp, rl = plan.dev
    _check(load().rlt_paged_extend_attn(
        ctypes.byref(pool.struct), bank, _dev(q, torch.bfloat16, "q"), Hq, N,
        _dev(page_table, torch.int32, "page_table"), page_table.shape[1], page_table.shape[0],
        _dev(seg, torch.int32, "segments"), _dev(mem, torch.int32, "members"), _dev(lim, torch.int32, "member_limit"),
        _dev(rp, torch.int32, "row_prefix"), _dev(rl, torch.int32, "row_len"), plan.num_segments, plan.work_units,
        max(plan.max_slots, 1), plan.chunk_tiles, float(scale), _dev(out, torch.bfloat16, "out"), lse_ptr,
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(), int(max_ctas),
        ATTN_EARLY_START if early_start else 0, _stream(stream)), "rlt_paged_extend_attn")
    return out
