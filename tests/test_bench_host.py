"""Host-side accounting of bench.py, checked without a GPU.

The algorithmic bytes of an attention call count every K/V row a request reads once, and
for shared prefixes ("Faster fuzzy minds", "When scheduler does the work": requests sharing a
prompt map the same physical pages) each physical row once -- what an ideal kernel must move
from HBM.  Here both counts are rebuilt by brute force from the page tables.  The committed
DRAM-traffic summaries are used only while the kernel sources they were taken on are unchanged.
"""
import os
import shutil

import numpy as np
import pytest

import bench
import workloads as W


def brute_force_tokens(case):
    """(logical, unique) K/V rows per kv head: positions read, and distinct pool slots."""
    slots = set()
    logical = 0
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        logical += L
        for p in range(L):
            slots.add(int(case.page_table[b, p // case.page_size]) * case.page_size + p % case.page_size)
    return logical, len(slots)


@pytest.mark.parametrize("name", ["tiny", "huginn"])
def test_attention_bytes_from_the_page_tables(name):
    case = W.config(name)
    logical, unique = brute_force_tokens(case)
    per_row = case.num_kv_heads * case.head_dim * 2 * 2            # K and V, bf16
    fixed = (case.batch * case.num_q_heads * case.head_dim * 2 * 2  # q in, o out
             + sum(-(-int(L) // case.page_size) for L in case.seq_lens) * 4 + case.batch * 4)
    assert bench.attn_bytes(case, unique=False) == logical * per_row + fixed
    assert bench.attn_bytes(case, unique=True) == unique * per_row + fixed
    if name == "huginn":
        assert unique < logical / 3                                 # the shared chain counted once
    else:
        assert unique == logical


def test_fused_append_bytes_drop_only_the_slot_list():
    case = W.config("tiny")
    n = int((case.new_slots >= 0).sum())
    rows = n * case.num_kv_heads * case.head_dim * 2                # bf16 rows of one of K / V
    assert bench.append_bytes(case) == 2 * 2 * rows + case.batch * 8
    assert bench.fused_append_bytes(case) == 2 * 2 * rows


def test_job_throughput_is_every_ranks_bytes_over_the_slowest_step():
    assert bench.job_gbs(10**9, 4, 2.0) == pytest.approx(2000.0)


def test_traffic_summary_is_dropped_when_a_kernel_source_changes(tmp_path, monkeypatch):
    src_profile = os.path.join(bench.ROOT, "profiles", "traffic_ouro.txt")
    text = open(src_profile).read()
    fields = dict(l.split(":", 1) for l in text.splitlines() if ":" in l)
    sources = fields["sources"].split()
    os.makedirs(tmp_path / "profiles")
    os.makedirs(tmp_path / "paged_kv_looped_gb300" / "csrc")
    shutil.copy(src_profile, tmp_path / "profiles" / "traffic_ouro.txt")
    for f in sources:
        shutil.copy(os.path.join(bench.ROOT, "paged_kv_looped_gb300", "csrc", f),
                    tmp_path / "paged_kv_looped_gb300" / "csrc" / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the copy's summary names the copied sources' hash (as a fresh capture would), whether or not
    # the committed summary is current
    import hashlib
    blob = b"".join(open(tmp_path / "paged_kv_looped_gb300" / "csrc" / f, "rb").read() for f in sources)
    digest = hashlib.sha256(blob).hexdigest()[:16]
    with open(tmp_path / "profiles" / "traffic_ouro.txt", "w") as fh:
        fh.write("\n".join(f"sources_sha256_16: {digest}" if l.startswith("sources_sha256_16:") else l
                           for l in text.splitlines()) + "\n")
    fused = fields.get("append", "plain").strip() == "fused"
    assert bench.profiled_traffic("ouro", fused) == float(fields["dram_bytes_per_call"])
    assert bench.profiled_traffic("ouro", not fused) is None        # taken with the other append form
    assert bench.profiled_traffic("gqa", fused) is None             # no such summary in the copy
    with open(tmp_path / "paged_kv_looped_gb300" / "csrc" / sources[0], "a") as fh:
        fh.write("\n// edited\n")
    assert bench.profiled_traffic("ouro", fused) is None


def test_noise_roofline_takes_the_issue_bound_from_the_current_profile(monkeypatch):
    # the committed ncu summary of the noise kernel was taken on the current noise.cu: the bench
    # reports the kernel against integer issue (SMs x 4 schedulers x 32 lanes x clock / the
    # profiled instructions per value) as well as against its HBM write
    ipv = bench.profiled_noise_instructions()
    assert ipv is not None and 20 < ipv < 100
    monkeypatch.setattr(bench, "sm_count_and_clock", lambda: (152, 2070.0))
    case = W.config("longctx")
    values = case.noise.rows * case.noise.channels
    peak = 152 * 4 * 32 * 2070e6 / ipv
    ms = values / (0.7 * peak) * 1e3                     # a launch at 70 % of the issue bound
    r = bench.noise_roofline(case, ms)
    assert r["values"] == values
    assert abs(r["alu"]["frac"] - 0.7) < 1e-3
    assert r["bound"] == "alu"                           # 4 bytes per value write far below the copy peak
    assert r["frac_of_hbm_peak"] < r["alu"]["frac"]
