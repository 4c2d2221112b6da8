"""Host-side checks of bench.py's bookkeeping; no GPU work.

* every stored DRAM-traffic entry names a workload the bench can run, and is
  reported only while the kernel's sources still have the stored digest;
* the digest ignores comments and blank lines but not code;
* the FLOP and byte counts behind the reported rates match what they count:
  allowed (query, key) pairs, and the bytes of the merge's tensors.
"""

import os

import pytest

import bench
from sequence_exact_attention_gb300 import workloads as wl


def _all_names():
    return (set(wl.WORKLOADS) | set(wl.MERGE_WORKLOADS) | set(wl.VARLEN_WORKLOADS)
            | set(wl.ULYSSES_WORKLOADS) | set(wl.BWD_WORKLOADS))


def test_traffic_entries_name_real_workloads():
    names = _all_names()
    for kernel, entry in bench.TRAFFIC.items():
        assert kernel in bench.KERNEL_SOURCES
        for w, nbytes in entry["bytes_per_launch"].items():
            assert w in names, f"{kernel}: unknown workload {w}"
            assert nbytes > 0


def test_traffic_follows_the_source_digest(monkeypatch):
    w = wl.HEADLINE
    digest = bench._kernel_digest("attn_tc")
    entry = {"sha256_16": digest, "bytes_per_launch": {w: 1234567}}
    monkeypatch.setitem(bench.TRAFFIC, "attn_tc", entry)
    assert bench._traffic("attn_tc", w) == 1234567
    assert bench._traffic("attn_tc", "no_such_workload") is None
    monkeypatch.setitem(bench.TRAFFIC, "attn_tc", dict(entry, sha256_16="0" * 16))
    assert bench._traffic("attn_tc", w) is None


def test_digest_ignores_comments_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "sequence_exact_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.KERNEL_SOURCES, "probe", ("k.cu",))
    src = csrc / "k.cu"
    src.write_text("int f() {\n  return 1;\n}\n")
    d0 = bench._kernel_digest("probe")
    src.write_text("// a comment\nint f() {  // trailing\n\n  return 1;\n}\n")
    assert bench._kernel_digest("probe") == d0
    src.write_text("int f() {\n  return 2;\n}\n")
    assert bench._kernel_digest("probe") != d0


def test_recorded_digests_cover_existing_sources():
    for kernel, files in bench.KERNEL_SOURCES.items():
        for name in files:
            path = os.path.join(bench.ROOT, "sequence_exact_attention_gb300", "csrc", name)
            assert os.path.exists(path), path


def _allowed_pairs(S, causal):
    return sum((i + 1) if causal else S for i in range(S))


@pytest.mark.parametrize("causal", [False, True])
def test_forward_flop_counts_allowed_pairs(causal):
    """4*D FLOP per allowed (query, key) pair; the causal count is the usual
    S^2/2 convention, within S/2 pairs of the exact S(S+1)/2."""
    S, D, B, H = 96, 64, 2, 3
    w = wl.AttnWorkload("t", "bf16", B, H, H, S, D, 4, causal, "contiguous")
    exact = 4.0 * D * B * H * _allowed_pairs(S, causal)
    assert abs(w.flop - exact) <= 4.0 * D * B * H * S / 2
    if not causal:
        assert w.flop == exact
    assert wl.bwd_flop(w) == 2.5 * w.flop


def test_varlen_flop_is_the_sum_over_sequences():
    for w in wl.VARLEN_WORKLOADS.values():
        per_seq = sum(wl.AttnWorkload("s", w.dtype, 1, w.H_q, w.H_kv, n, w.D, w.P, w.causal,
                                      w.order).flop for n in w.lengths)
        assert w.flop == pytest.approx(per_seq)


def test_merge_bytes_equal_the_tensors_read_and_written():
    w = wl.MergeWorkload("t", "f32", 3, 1, 2, 8, 64, seed=1)
    os_, ls = wl.make_merge_parts(w)
    read = sum(t.numel() * t.element_size() for t in os_ + ls)
    written = os_[0].numel() * os_[0].element_size() + ls[0].numel() * ls[0].element_size()
    assert w.bytes == read + written


def test_headline_metric_names_only_the_headline():
    assert bench._fwd_metric(wl.WORKLOADS[wl.HEADLINE]) == bench.METRIC
    for name, w in wl.WORKLOADS.items():
        if name != wl.HEADLINE:
            assert name in bench._fwd_metric(w)


def test_stored_traffic_is_current():
    """Every stored DRAM capture belongs to the kernel sources as they are
    now; after a kernel change the traffic must be captured again (one ncu
    pass) or the bench reports null."""
    for kernel, entry in bench.TRAFFIC.items():
        assert entry["sha256_16"] == bench._kernel_digest(kernel), (
            f"{kernel}: sources changed since the stored DRAM traffic was captured")


def _ref_args(**kw):
    import argparse
    a = dict(gpus=1, steps=1, warmup=0, ref_rows=8)
    a.update(kw)
    return argparse.Namespace(**a)


def _last_json(capsys):
    import json
    return json.loads(capsys.readouterr().out.strip().splitlines()[-1])


@pytest.mark.parametrize("kind", ["varlen", "ulysses", "merge"])
def test_reference_arms_print_the_contract_line(kind, capsys):
    """Every workload family's --impl reference arm times the oracle on the
    host and prints the same metric and unit as the GPU arm."""
    if kind == "varlen":
        w = wl.VarlenWorkload("t", "bf16", (40, 0, 7, 100), 2, 1, 64, 2, True, "zigzag", seed=3)
        assert bench.run_varlen_reference(_ref_args(), w) == 0
        metric, unit = bench.VARLEN_METRIC, bench.UNIT
    elif kind == "ulysses":
        w = wl.AttnWorkload("t", "bf16", 2, 4, 2, 90, 64, 4, True, "contiguous", seed=4)
        assert bench.run_ulysses_reference(_ref_args(), w) == 0
        metric, unit = bench.ULYSSES_METRIC, bench.UNIT
    else:
        w = wl.MergeWorkload("t", "f32", 3, 1, 2, 512, 64, seed=5)
        assert bench.run_merge_reference(_ref_args(), w) == 0
        metric, unit = bench.MERGE_METRIC, "GB/s"
    line = _last_json(capsys)
    assert line["impl"] == "reference" and line["metric"] == metric and line["unit"] == unit
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["steps"] == 1


def test_parity_record_of_the_bench_line():
    """The bench line's parity record compares the timed output with the
    oracle rows of the CPU-baseline sample, against the tolerance."""
    import numpy as np
    import torch
    import oracle
    w = wl.AttnWorkload("t", "bf16", 1, 2, 2, 200, 64, 2, True, "zigzag", seed=9)
    q, k, v = wl.make_qkv(w)
    o, l = oracle.attention_naive(q, k, v, True, w.scale)
    out = torch.from_numpy(o).to(torch.bfloat16)
    lse = torch.from_numpy(l).float()
    want = []
    _, _, rows = bench._oracle_sample_rate(w, q, k, v, 16, seed=3, want=want)
    rec = bench._parity(w, out, lse, rows, want[0])
    assert rec["rows"] == 16 and rec["within_tolerance"], rec
    assert rec["out_max_abs_err"] < 1e-2 and rec["lse_max_abs_err"] < 1e-5
    bad = out.clone()
    bad[:, rows[0]] += 1.0
    assert not bench._parity(w, bad, lse, rows, want[0])["within_tolerance"]
    assert "error" in bench._parity(w, out, lse, rows, None)   # never raises


def test_device_info_never_raises():
    info = bench._device_info(0)
    assert ("name" in info and "sm_count" in info) or "error" in info


def test_l2_rule_follows_the_input_size():
    """Inputs larger than L2 are timed back to back; inputs that fit are
    flushed out of L2 before every timed launch, and the config says which."""
    big, small = wl.WORKLOADS[wl.HEADLINE], wl.WORKLOADS["bf16_s4k_causal"]
    assert bench._inputs_mib(big) > bench.L2_MIB
    assert "larger than L2" in bench._config(big)["l2"]
    assert bench._l2_flusher(big, None, None) is None
    assert bench._inputs_mib(small) <= bench.L2_MIB
    assert "flushed" in bench._config(small)["l2"]
    assert bench.FLUSH_MIB > bench.L2_MIB
