"""The C-ABI library loads, exports every entry point include/rlt.h declares, and its host
logic (bank map, batch validation, argument checks that fail before any launch) behaves."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import paged_kv_looped_gb300 as rlt
import workloads as W
from paged_kv_looped_gb300 import build as rlt_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rlt.h")


@pytest.fixture(scope="module")
def lib():
    rlt_build.build()
    return rlt.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^RLT_API\s+[^;(]*?\b(rlt_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("rlt_kv_append", "rlt_paged_decode_attn", "rlt_latent_noise_init", "rlt_bank_map",
              "rlt_paged_gather", "rlt_noise_hash24"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", rlt.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for code, name in rlt.STATUS.items():
        assert lib.rlt_status_string(code).decode() == name
    assert rlt.rlt_version() >= 100


@pytest.mark.parametrize("rec,planes", [([1] * 24, 4), ([0, 0, 1, 1, 1, 1, 0, 0], 32), ([0] * 3, 1),
                                        ([1, 0, 1], 5)])
def test_bank_map_matches_oracle(lib, rec, planes):
    m, n = rlt.rlt_bank_map(np.array(rec, np.uint8), planes)
    mo, no = oracle.bank_map(np.array(rec, np.uint8), planes)
    assert n == no and np.array_equal(m, mo)


@pytest.mark.parametrize("rec,planes", [([1] * 24, 4), ([0, 0, 1, 1, 1, 1, 0, 0], 32), ([1, 0, 1], 5)])
def test_bank_index_matches_oracle_map(lib, rec, planes):
    """rlt_bank_index, one (layer, plane) lookup through the C ABI, against the oracle's whole map."""
    mo, _ = oracle.bank_map(np.array(rec, np.uint8), planes)
    m, _ = rlt.rlt_bank_map(np.array(rec, np.uint8), planes)
    for layer in range(len(rec)):
        for plane in range(planes):
            assert rlt.rlt_bank_index(m, layer, plane) == mo[layer, plane]
    # prelude / coda layers exist on plane 0 only; lookups outside the map give -1
    assert rlt.rlt_bank_index(m, -1, 0) == -1 and rlt.rlt_bank_index(m, len(rec), 0) == -1
    assert rlt.rlt_bank_index(m, 0, planes) == -1 and rlt.rlt_bank_index(m, 0, -1) == -1
    assert lib.rlt_bank_index(None, len(rec), planes, 0, 0) == -1


def test_bank_index_huginn_planes(lib):
    """Huginn: layers 0-1 and 6-7 (prelude, coda) only on plane 0; 2-5 on all 32 planes."""
    m, n = rlt.rlt_bank_map(np.array([0, 0, 1, 1, 1, 1, 0, 0], np.uint8), 32)
    assert n == 132
    for layer in (0, 1, 6, 7):
        assert rlt.rlt_bank_index(m, layer, 0) >= 0
        assert all(rlt.rlt_bank_index(m, layer, t) == -1 for t in range(1, 32))
    held = sorted(rlt.rlt_bank_index(m, l, t) for l in range(8) for t in range(32)
                  if rlt.rlt_bank_index(m, l, t) >= 0)
    assert held == list(range(132))


def test_bank_map_rejects_bad_sizes(lib):
    with pytest.raises(rlt.RltError):
        rlt.rlt_bank_map(np.zeros(0, np.uint8), 4)


def test_validate_batch_accepts_generated_workloads(lib):
    for name in W.WORKLOADS:
        c = W.config(name)
        assert rlt.rlt_validate_batch(c.page_table, c.seq_lens, c.new_slots, c.num_pages, c.page_size) == 0


def test_validate_batch_rejects_bad_batches(lib):
    c = W.config("huginn")
    args = lambda pt, sl, ns, P=c.num_pages: rlt.rlt_validate_batch(pt, sl, ns, P, c.page_size)  # noqa: E731
    pt = c.page_table.copy()
    pt[3, 2] = c.num_pages                                   # page id past the pool
    assert args(pt, c.seq_lens, c.new_slots) == 2
    pt = c.page_table.copy()
    pt[0, 0] = -1
    assert args(pt, c.seq_lens, c.new_slots) == 2
    sl = c.seq_lens.copy()
    sl[1] = c.max_pages * c.page_size + 1                     # longer than its table row
    assert args(c.page_table, sl, None) == 2
    ns = c.new_slots.copy()
    ns[2] = ns[2] + 1 if (c.seq_lens[2] % c.page_size) else ns[2] - 1   # not the last position
    assert args(c.page_table, c.seq_lens, ns) == 2
    ns = c.new_slots.copy()
    ns[5] = ns[4]                                            # two requests, one slot
    assert args(c.page_table, c.seq_lens, ns) != 0
    # an append into a page another request also reads (shared prefix) is refused
    pt = c.page_table.copy()
    b0_last = (c.seq_lens[0] - 1) // c.page_size
    pt[1, 0] = pt[0, b0_last]
    assert args(pt, c.seq_lens, c.new_slots) == 1
    assert args(c.page_table, c.seq_lens, None) == 0


def test_device_entry_points_reject_bad_arguments_before_launch(lib):
    # every one of these fails host-side checks, so no CUDA call is made
    null = ctypes.c_void_p(0)
    assert lib.rlt_kv_append(None, 0, null, null, null, 1, null) == 1
    pool = rlt.rlt_kv_pool(16, 16, 10, 1, 2, 16, 128)
    assert lib.rlt_kv_append(ctypes.byref(pool), 1, null, null, null, 1, null) == 2     # bank
    assert lib.rlt_kv_append(ctypes.byref(pool), 0, null, null, null, -1, null) == 1
    assert lib.rlt_kv_append(ctypes.byref(pool), 0, null, null, null, 0, null) == 0     # nothing to do
    bad = rlt.rlt_kv_pool(8, 16, 10, 1, 2, 16, 128)                                     # misaligned k
    assert lib.rlt_kv_append(ctypes.byref(bad), 0, null, null, null, 1, null) == 1
    attn = lambda p, hq, split=0, ws=0: lib.rlt_paged_decode_attn(                       # noqa: E731
        ctypes.byref(p), 0, null, null, null, hq, null, 1, null, 1, 64, 0.0, null, null, null, ws, split, 0, null)
    assert attn(pool, 3) == 1                                # Hq not a multiple of Hkv
    assert attn(pool, 6) == 3                                # group 3: no kernel
    assert attn(pool, 2, split=24) == 1                      # split not a multiple of 16
    odd_ps = rlt.rlt_kv_pool(16, 16, 10, 1, 2, 8, 128)
    assert attn(odd_ps, 2) == 3                              # page_size 8: no attention kernel
    d96 = rlt.rlt_kv_pool(16, 16, 10, 1, 2, 16, 96)
    assert attn(d96, 2) == 3
    assert attn(pool, 2) == 1                                # null q / tables / out
    # an unknown flag bit is refused before anything else
    assert lib.rlt_paged_decode_attn(ctypes.byref(pool), 0, null, null, null, 2, null, 1, null, 1, 64, 0.0, null,
                                     null, null, 0, 0, 2, null) == 1
    assert lib.rlt_paged_decode_attn_prefix(ctypes.byref(pool), 0, null, null, null, 2, null, 1, null, 1, 64, null,
                                            null, null, null, 0, 0, 0, 1, 0, 0.0, null, null, null, 0, 0, 0, 4,
                                            null) == 1
    assert lib.rlt_paged_extend_attn(ctypes.byref(pool), 0, null, 2, 1, null, 1, 1, null, null, null, null, null,
                                     1, 1, 1, 1, 0.0, null, null, null, 0, 0, 8, null) == 1
    assert lib.rlt_latent_noise_init(null, null, null, 5, 0, ctypes.c_float(0.02), null) == 1
    assert lib.rlt_latent_noise_init(null, null, null, 0, 8, ctypes.c_float(0.02), null) == 0
    assert lib.rlt_noise_hash24(null, null, null, -1, 8, null) == 1
    assert lib.rlt_paged_gather(ctypes.byref(pool), 0, null, 1, null, 2, 10, null, null, null) == 1
    assert lib.rlt_validate_batch(null, 1, null, 1, null, 10, 0) == 1
    assert lib.rlt_paged_decode_workspace_size(-1, 1, 1, 128, 10, 0) == 0


def test_fault_switch_rejects_limits_outside_its_range(lib):
    # only refusals here: a valid limit would arm the next decode call of this thread
    assert lib.rlt_debug_fault_next_decode(ctypes.c_uint64(0)) == 1
    assert lib.rlt_debug_fault_next_decode(ctypes.c_uint64(2_000_000_000)) == 1


def test_pool_dtype_other_than_bf16_is_refused(lib):
    null = ctypes.c_void_p(0)
    fp16 = rlt.rlt_kv_pool(16, 16, 10, 1, 2, 16, 128, 1)
    assert lib.rlt_kv_append(ctypes.byref(fp16), 0, null, null, null, 1, null) == 3
    assert lib.rlt_paged_decode_attn(ctypes.byref(fp16), 0, null, null, null, 2, null, 1, null, 1, 64, 0.0, null,
                                     null, null, 0, 0, 0, null) == 3
    assert lib.rlt_paged_gather(ctypes.byref(fp16), 0, null, 1, null, 2, 10, null, null, null) == 3


def test_noalloc_checks_arguments_before_the_scratch_size(lib):
    """The no-allocation entry point reports what rlt_paged_decode_attn would for a bad pool, bank,
    split or pointer, even for a shape whose partials would not fit its scratch array; only a
    well-formed call too large for the array gets RLT_ERR_WORKSPACE_TOO_SMALL.  Nothing launches:
    the pointers are aligned stand-ins that no kernel ever sees."""
    fake = ctypes.c_void_p(4096)
    pool = rlt.rlt_kv_pool(4096, 8192, 10, 1, 8, 16, 128)
    big = dict(Hq=64, batch=65535, max_len=1 << 20, split=16)
    call = lambda p, bank=0, split=16, q=fake, Hq=64: lib.rlt_paged_decode_attn_noalloc(  # noqa: E731
        ctypes.byref(p), bank, q, Hq, fake, 1 << 16, fake, big["batch"], big["max_len"], 0.0, fake, None, split, None)
    assert rlt.rlt_paged_decode_workspace_size(big["batch"], 64, 8, 128, big["max_len"], 16) > \
        rlt.NOALLOC_SCRATCH_BYTES
    assert call(pool) == 4                                   # well formed, too large: scratch size
    assert call(pool, bank=1) == 2                           # bank outside the pool
    assert call(pool, split=24) == 1                         # split not a multiple of 16
    assert call(pool, Hq=24) == 3                            # group 3: no kernel
    assert call(pool, Hq=12) == 1                            # Hq not a multiple of Hkv
    assert call(pool, q=ctypes.c_void_p(0)) == 1             # null q
    assert call(pool, q=ctypes.c_void_p(4100)) == 1          # misaligned q
    bad = rlt.rlt_kv_pool(4104, 8192, 10, 1, 8, 16, 128)     # misaligned k
    assert call(bad) == 1
    assert lib.rlt_paged_decode_attn_noalloc(None, 0, fake, 64, fake, 1, fake, 1, 16, 0.0, fake, None, 0,
                                             None) == 1


def test_wrappers_check_q_out_and_lse_shapes():
    """The binding checks what the C ABI cannot (it takes no head_dim for q): a q, out or lse_out
    of the wrong shape is refused before any pointer is passed on."""
    import types

    import torch
    pool = types.SimpleNamespace(head_dim=128)
    q = torch.zeros((4, 8, 128), dtype=torch.bfloat16)
    rlt._check_q_out(pool, q, None, None)
    rlt._check_q_out(pool, q, torch.zeros_like(q), torch.zeros((4, 8)))
    with pytest.raises(ValueError, match="head_dim"):
        rlt._check_q_out(pool, torch.zeros((4, 8, 64), dtype=torch.bfloat16), None, None)
    with pytest.raises(ValueError, match="out"):
        rlt._check_q_out(pool, q, torch.zeros((4, 8, 64), dtype=torch.bfloat16), None)
    with pytest.raises(ValueError, match="lse_out"):
        rlt._check_q_out(pool, q, None, torch.zeros((4, 9)))


def test_workspace_size_grows_with_splits(lib):
    one = lib.rlt_paged_decode_workspace_size(4, 8, 8, 128, 256, 256)
    assert one == 0                                          # a single split needs no partials
    many = lib.rlt_paged_decode_workspace_size(4, 8, 8, 128, 4096, 256)
    assert many >= 4 * 8 * 16 * (128 + 1) * 4


def test_package_refuses_to_run_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(rlt, "_lib", None)
    monkeypatch.setattr(rlt, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        rlt.load()
