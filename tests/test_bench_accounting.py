"""bench.py's byte accounting and its traffic lookup (CPU).

The bench line's `value` is unique key/value bytes per step over the step
time, and `roofline.achieved` is the algorithmic bytes of one attention call
over its duration; both rest on `_kv_bytes` / `_algo_bytes`.  These are
checked here against sums written out by hand for small batches (a shared
span counts once for its whole group, since every member's table names the
same physical blocks: zenaique "prefix sharing" answer; kgptalkie "Prefix
Sharing Is a Natural Extension").  `roofline.traffic` comes from the committed
ncu summaries in profiles/, and only while the kernel sources a summary names
are unchanged; every registered summary must parse, and the lookup must
answer exactly when its recorded hash matches the sources.
"""
import os
import re

import pytest

import bench
from paged_kv_cache_253_gb300 import workloads as wls

D128 = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)


@pytest.mark.parametrize("dtype,per_tok", [("bf16", 8 * 128 * 2 * 2), ("fp8", 8 * 128 * 2 * 1),
                                           ("f32", 8 * 128 * 2 * 4)])
def test_kv_bytes_count_every_cached_token(dtype, per_tok):
    wl = wls.make_workload("decode", lengths=[1, 17, 250], dtype=dtype, **D128)
    assert bench._kv_bytes(wl, [1, 17, 250]) == (1 + 17 + 250) * per_tok


def test_a_shared_span_counts_once_per_group():
    wl = wls.make_workload("decode", lengths=[40, 50, 60, 70, 80], **D128)
    per_tok = 8 * 128 * 2 * 2
    lens = [40, 50, 60, 70, 80]
    # two groups: members {0, 1, 2} share 2 blocks, members {3, 4} share 1 block
    groups = ([0, 3, 5], [0, 1, 2, 3, 4], [2, 1])
    unique = sum(lens) - (3 - 1) * 2 * 16 - (2 - 1) * 1 * 16
    assert bench._kv_bytes(wl, lens, groups) == unique * per_tok
    # no groups: every member's whole context
    assert bench._kv_bytes(wl, lens, ([0], [], [])) == sum(lens) * per_tok


def test_algorithmic_bytes_add_queries_outputs_tables_and_lengths():
    lens = [1, 17, 250]
    wl = wls.make_workload("decode", lengths=lens, **D128)
    S, Hq, D = 3, 32, 128
    kv = sum(lens) * 8 * 128 * 2 * 2
    q = S * Hq * D * 2                    # bf16 queries
    out = S * Hq * D * 4                  # fp32 output
    tables = (1 + 2 + 16) * 4             # ceil(L / 16) block ids per sequence
    assert bench._algo_bytes(wl, lens) == kv + q + out + tables + S * 4
    wl8 = wls.make_workload("decode", lengths=lens, dtype="fp8", **D128)
    assert bench._algo_bytes(wl8, lens) == kv // 2 + q + out + tables + S * 4


def _profile(name):
    text = open(os.path.join(bench.ROOT, "profiles", name)).read()
    srcs = re.search(r"sources:\s*`([^`]+)`", text)
    digest = re.search(r"source sha256\[:16\]:\s*`?([0-9a-f]{16})", text)
    traffic = re.search(r"dram bytes per launch:\s*\|?\s*`?([0-9]+)", text)
    return srcs, digest, traffic


@pytest.mark.parametrize("key", sorted(bench.TRAFFIC_PROFILES))
def test_registered_traffic_summaries_parse(key):
    srcs, digest, traffic = _profile(bench.TRAFFIC_PROFILES[key])
    assert srcs and digest and traffic, f"{key}: sources, hash or traffic line missing"
    for n in srcs.group(1).split():
        assert os.path.isfile(os.path.join(bench.ROOT, "paged_kv_cache_253_gb300", "csrc", n)), n
    assert int(traffic.group(1)) > 0


@pytest.mark.parametrize("key", sorted(bench.TRAFFIC_PROFILES))
def test_traffic_is_reported_only_for_unchanged_sources(key, monkeypatch):
    srcs, digest, traffic = _profile(bench.TRAFFIC_PROFILES[key])

    class W:
        name, dtype = key

    current = bench.source_digest(srcs.group(1).split())
    got = bench._traffic_from_profile(W())
    assert got == (int(traffic.group(1)) if digest.group(1) == current else None)
    # sources edited since the capture: no traffic figure
    monkeypatch.setattr(bench, "source_digest", lambda names: "0" * 16)
    assert bench._traffic_from_profile(W()) is None


def test_unregistered_workloads_have_no_traffic():
    class W:
        name, dtype = "tiny", "f32"

    assert bench._traffic_from_profile(W()) is None
