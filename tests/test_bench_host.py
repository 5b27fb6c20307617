"""Host-side logic of bench.py (no GPU): the byte accounting behind the roofline and
the rule that reports stored DRAM traffic only for the code it was measured on."""
import json

import numpy as np

import bench
import workloads as W


def test_kv_bytes_counts_the_used_blocks_tokens():
    w = W.config(4, small=True)
    per_tok = 2 * w.head_dim * w.elem_bytes
    full = bench.kv_bytes(w)
    # every listed block of every item: the item's tokens
    toks = sum(int(w.seq_lens[it // w.num_kv_heads]) for it in range(w.num_items))
    assert full == toks * per_tok
    # one block per item: a full 64-token block unless the sequence is shorter
    one = bench.kv_bytes(w, np.ones(w.num_items, dtype=np.int32))
    lists = bench.listed_blocks(w)
    expect = 0
    for it, lst in enumerate(lists):
        b = it // w.num_kv_heads
        expect += min(w.block_size, int(w.seq_lens[b]) - int(lst[0]) * w.block_size) * per_tok
    assert one == expect
    assert bench.kv_bytes(w, np.zeros(w.num_items, dtype=np.int32)) == 0
    assert bench.kv_bytes(w, -np.ones(w.num_items, dtype=np.int32)) == 0  # failed items read nothing counted


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    csrc = tmp_path / "kv_cache_early_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "art_kernel.cuh").write_text("// a comment\nint f() { return 1; }  // trailing\n/* block\n comment */\n")
    (csrc / "art_units.cuh").write_text("int g();\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h1 = bench.kernel_source_hash("one CTA per item")
    (csrc / "art_kernel.cuh").write_text("// another comment\n\nint f() { return 1; }\n")
    assert bench.kernel_source_hash("one CTA per item") == h1  # comments and blank lines only
    (csrc / "art_kernel.cuh").write_text("int f() { return 2; }\n")
    assert bench.kernel_source_hash("one CTA per item") != h1  # code
    hu, h_one = bench.kernel_source_hash("units"), bench.kernel_source_hash("one CTA per item")
    (csrc / "art_units.cuh").write_text("int g(int);\n")
    assert bench.kernel_source_hash("one CTA per item") == h_one  # not a source of the one-CTA path
    assert bench.kernel_source_hash("units") != hu  # a source of the unit path


def test_traffic_only_for_the_measured_code_and_path(tmp_path, monkeypatch):
    (tmp_path / "kv_cache_early_gb300" / "csrc").mkdir(parents=True)
    (tmp_path / "kv_cache_early_gb300" / "csrc" / "art_kernel.cuh").write_text("int f();\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash("one CTA per item")
    entry = {"kernel_hash": h, "captured_workload": "w-small", "dram_bytes": 1100, "algorithmic_bytes": 1000,
             "path": "one CTA per item"}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({"w": entry}))
    t, src = bench.load_traffic("w", 2000, "one CTA per item")
    assert t == 2200 and "scaled" in src  # a smaller capture, scaled by algorithmic bytes
    assert bench.load_traffic("w", 2000, "units") == (None, None)  # another kernel path
    assert bench.load_traffic("other", 2000, "one CTA per item") == (None, None)
    (tmp_path / "kv_cache_early_gb300" / "csrc" / "art_kernel.cuh").write_text("int f(int);\n")
    assert bench.load_traffic("w", 2000, "one CTA per item") == (None, None)  # the code changed since
