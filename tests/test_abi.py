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
        ctypes.byref(p), 0, null, null, null, hq, null, 1, null, 1, 64, 0.0, null, null, null, ws, split, null)
    assert attn(pool, 3) == 1                                # Hq not a multiple of Hkv
    assert attn(pool, 6) == 3                                # group 3: no kernel
    assert attn(pool, 2, split=24) == 1                      # split not a multiple of 16
    odd_ps = rlt.rlt_kv_pool(16, 16, 10, 1, 2, 8, 128)
    assert attn(odd_ps, 2) == 3                              # page_size 8: no attention kernel
    d96 = rlt.rlt_kv_pool(16, 16, 10, 1, 2, 16, 96)
    assert attn(d96, 2) == 3
    assert attn(pool, 2) == 1                                # null q / tables / out
    assert lib.rlt_latent_noise_init(null, null, null, 5, 0, ctypes.c_float(0.02), null) == 1
    assert lib.rlt_latent_noise_init(null, null, null, 0, 8, ctypes.c_float(0.02), null) == 0
    assert lib.rlt_noise_hash24(null, null, null, -1, 8, null) == 1
    assert lib.rlt_paged_gather(ctypes.byref(pool), 0, null, 1, null, 2, 10, null, null, null) == 1
    assert lib.rlt_validate_batch(null, 1, null, 1, null, 10, 0) == 1
    assert lib.rlt_paged_decode_workspace_size(-1, 1, 1, 128, 10, 0) == 0


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
