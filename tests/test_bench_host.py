"""Host logic of bench.py that needs no GPU: the roofline entry picks the bound
that the algorithmic work sets (HBM bytes or tensor flops) and reports the
achieved rate against that peak; stored ncu traffic is used only while the
kernel sources it was captured from are unchanged."""
import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import moe_synth  # noqa: E402

PK = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0, "source": "test"}


def test_roofline_picks_hbm_for_low_intensity():
    # 1 GB and 10 GFLOP: 125 us of HBM against 5 us of tensor work
    e = bench.roofline_entry("k", 0.25, 1e10, 1e9, PK, traffic=123)
    assert e["bound"] == "hbm" and e["unit"] == "GB/s"
    assert np.isclose(e["achieved"], 1e9 / 0.25e-3 / 1e9)          # 4000 GB/s
    assert np.isclose(e["frac"], 0.5)
    assert e["traffic"] == 123


def test_roofline_picks_tensor_for_high_intensity():
    # 1 PFLOP over 1 GB: 500 ms of tensor work against 125 us of HBM
    e = bench.roofline_entry("k", 1000.0, 1e15, 1e9, PK)
    assert e["bound"] == "tensor" and e["unit"] == "TFLOP/s"
    assert np.isclose(e["achieved"], 1000.0)
    assert np.isclose(e["frac"], 0.5)


def test_weight_gradient_bytes_cover_every_expert():
    spec = moe_synth.BF16_T2048
    cnt = np.zeros(spec.E, dtype=np.int64)
    cnt[0] = spec.T * spec.k                      # one active expert
    w = bench.work_per_group(spec, cnt, training=True)
    grads = (spec.E + spec.S) * 2 * spec.f * spec.d * 2
    # the gradients of experts that received no token are written too (as zeros)
    assert w["bwd_dw13"][1] >= grads
    assert w["bwd_dwd"][1] >= grads // 2
    # forward weight reads count only the experts that received tokens
    assert w["gateup"][1] < grads


def _entry(root, sources):
    h = hashlib.sha256()
    for s in sources:
        with open(os.path.join(root, s), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def test_stored_traffic_only_while_sources_unchanged(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "src").mkdir()
    (tmp_path / "src" / "a.cu").write_text("kernel a\n")
    (tmp_path / "src" / "b.h").write_text("constant b\n")
    srcs = ["src/a.cu", "src/b.h"]
    tab = {"gateup": {"dram_bytes_per_launch": 865548288, "sources": srcs,
                      "source_sha256_16": _entry(str(tmp_path), srcs)}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(tab))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.stored_traffic("gateup") == 865548288
    assert bench.stored_traffic("bwd_dw13") is None           # no capture for this kernel
    (tmp_path / "src" / "b.h").write_text("constant b changed\n")
    assert bench.stored_traffic("gateup") is None             # source changed since the capture
    (tmp_path / "src" / "b.h").unlink()
    assert bench.stored_traffic("gateup") is None             # source missing


def test_committed_traffic_entries_name_their_captures():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        tab = json.load(fh)
    for group, ent in tab.items():
        if group.startswith("_"):
            continue
        assert os.path.exists(os.path.join(ROOT, ent["capture"])), group
        for s in ent["sources"]:
            assert os.path.exists(os.path.join(ROOT, s)), (group, s)
        assert ent["dram_bytes_per_launch"] > 0
