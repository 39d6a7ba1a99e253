"""The algorithmic work bench.py divides by the measured time (the roofline
numerators), checked against brute-force counts on small shapes: every
(query row, head, visible key) pair costs 4*D FLOPs (QK^T and PV), and the
byte counts are the tensors' sizes."""
import importlib.util
import os
import types

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _w(B, L, Hq, Hkv, D, V=1024, k=4):
    return types.SimpleNamespace(B=B, L=L, Hq=Hq, Hkv=Hkv, D=D, V=V, k=k, rows=B * L)


def test_attention_pairs():
    b = _bench()
    w = _w(3, 5, 4, 2, 8)
    ctx = np.array([7, 0, 11], np.int32)
    pairs = sum(w.Hq * w.L * (int(c) + w.L) for c in ctx)  # every query sees ctx + whole block
    assert b.attn_flops(w, ctx) == 4 * w.D * pairs


def test_causal_pairs():
    b = _bench()
    w = _w(2, 6, 4, 1, 16)
    ctx = np.array([9, 3], np.int32)
    pairs = 0
    for c in ctx:
        for l in range(w.L):
            pairs += w.Hq * (int(c) + l + 1)  # the cache and block keys 0..l
    assert b.causal_flops(w, ctx) == 4 * w.D * pairs


def test_training_pairs():
    b = _bench()
    w = _w(1, 1, 8, 2, 32)
    B, N, S = 2, 48, 8
    pairs = 0
    for n in range(N):
        j = n // S
        pairs += w.Hq * (j * S + S)  # clean prefix of the block, then the block itself
    assert b.train_flops(w, B, N, S) == 4 * w.D * B * pairs


def test_byte_counts():
    b = _bench()
    w = _w(2, 4, 8, 2, 16, V=512, k=3)
    ctx = np.array([5, 9], np.int32)
    kv_cache = 2 * 2 * w.Hkv * w.D * int(ctx.sum())          # K and V rows read once, bf16
    q_out = 2 * 2 * w.B * w.L * w.Hq * w.D                    # Q read, out written, bf16
    blk = 2 * 2 * w.B * w.L * w.Hkv * w.D                      # block K and V, bf16
    assert b.attn_bytes(w, ctx) == kv_cache + q_out + blk
    assert b.append_bytes(w) == 2 * blk                        # block read again, cache rows written
    masked = 6
    assert b.commit_bytes(w, masked) == masked * w.V * 4 + 2 * w.rows + 4 * min(w.k, w.L) * w.B


def test_profiled_traffic_entries_and_source_keys(tmp_path, monkeypatch):
    # Every traffic entry names an existing ncu summary and existing kernel
    # sources; the bench reports the DRAM bytes only while those sources hash
    # to the captured value (an edited kernel reports null).
    import json
    b = _bench()
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    assert t
    for kernel, entries in t.items():
        for workload, e in entries.items():
            assert os.path.exists(os.path.join(ROOT, e["capture"])), e["capture"]
            assert all(os.path.exists(os.path.join(ROOT, s)) for s in e["sources"])
            assert e["dram_bytes_per_launch"] > 0
            got = b.profiled_traffic(kernel, workload)
            assert got in (None, e["dram_bytes_per_launch"])
    # a changed source voids the entry
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    entry = {"dram_bytes_per_launch": 123, "sources": ["k.cu"], "capture": "x.md",
             "sources_sha256": b.sources_hash(["k.cu"])}
    (prof / "traffic.json").write_text(json.dumps({"attn": {"w": entry}}))
    assert b.profiled_traffic("attn", "w") == 123
    src.write_text("kernel v2")
    assert b.profiled_traffic("attn", "w") is None
    assert b.profiled_traffic("attn", "other") is None
