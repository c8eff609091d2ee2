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


def test_layer_work_deepseek_v3_forward_matches_the_survey_figures():
    # every routed expert used, plus the shared one: 22.64 GB of bf16 expert weights, 3.7 MB of router
    # weight and 235 MB of x and y; 6.49 TFLOP of expert products plus 0.03 of router GEMM
    spec = moe_synth.DSV3_UNIFORM
    cnt = np.full(spec.E, spec.T * spec.k // spec.E)
    fl, by = bench.layer_work(spec, cnt)
    assert abs(by - (257 * 3 * 2048 * 7168 * 2 + 256 * 7168 * 2 + 2 * 8192 * 7168 * 2)) == 0
    assert np.isclose(by / 1e9, 22.88, atol=0.01)
    assert np.isclose(fl / 1e12, 6.49 + 0.03, atol=0.01)
    # an expert without tokens moves no weights
    cnt[:16] = 0
    _, by16 = bench.layer_work(spec, cnt)
    assert by - by16 == 16 * 3 * 2048 * 7168 * 2
    # the h and o round trips are not algorithmic work: the whole-call bytes stay well under the
    # per-kernel sum that counts them
    w = bench.work_per_group(spec, np.full(spec.E, 256), training=False)
    assert sum(w[g][1] for g in ("router_logits", "gateup", "down", "combine")) > by + 2.5e9


def test_layer_work_training_step_matches_the_survey_figures():
    # fwd: weights 1.107 GB + x, y 17 MB; bwd: weights read again 1.107 GB, weight gradients of every expert
    # 1.107 GB, x, dy, dx 25 MB, saved u, v 69 MB (written by the forward, read by the backward)
    spec = moe_synth.BF16_T2048
    cnt = np.full(spec.E, spec.T * spec.k // spec.E)
    fl_f, by_f = bench.layer_work(spec, cnt, "fwd")
    fl, by = bench.layer_work(spec, cnt, "fwd+bwd")
    W = 64 * 3 * 1408 * 2048 * 2
    assert np.isclose(W / 1e9, 1.107, atol=1e-3)
    assert by_f == W + 64 * 2048 * 2 + 2 * 2048 * 2048 * 2
    uv = 12288 * 2 * 1408 * 2
    assert by - by_f == W + W + 3 * 2048 * 2048 * 2 + 2 * uv
    assert np.isclose(fl_f / 1e9, 213, atol=1) and np.isclose((fl - fl_f) / 1e9, 426, atol=2)
    # fp32 storage doubles the bytes of the same shapes
    tiny = moe_synth.TINY_FP32
    _, by32 = bench.layer_work(tiny, np.full(tiny.E, 16))
    assert by32 == 8 * 3 * 128 * 256 * 4 + 8 * 256 * 4 + 2 * 64 * 256 * 4


def test_roof_line_bound_and_fraction():
    r = bench.roof_line(2.0, 2e12, 8e9, PK)                 # 1 ms of tensor work, 1 ms of HBM at 8 TB/s
    assert np.isclose(r["roofline_ms"], 1.0) and np.isclose(r["frac_of_roofline"], 0.5)
    r = bench.roof_line(2.0, 1e12, 8e9, PK)
    assert r["bound"] == "hbm" and np.isclose(r["roofline_ms"], 1.0)
    r = bench.roof_line(2.0, 8e12, 4e9, PK, tensor_peak=4000.0)   # a tensor peak other than bf16's
    assert r["bound"] == "tensor" and np.isclose(r["roofline_ms"], 2.0) and np.isclose(r["frac_of_roofline"], 1.0)


def test_mxfp8_step_work_ideal_once_and_per_chunk():
    spec = moe_synth.DSV3_MXFP8
    w_axis = 3 * 257 * 2048 * 7168 * (1 + 1 / 32)
    grads = 3 * 257 * 2048 * 7168 * 2
    acts = 4 * 8192 * 7168 * 2
    (fi, bi), (fc, bc) = bench.mx_step_work(spec, 4, 3, 6.5e12, 13e12)
    assert np.isclose(bi, 2 * w_axis + grads + acts)
    # 4 chunk forwards + 1 recomputed (3 ring slots), 4 chunk backwards: 9 weight streams
    assert np.isclose(bc, 9 * w_axis + grads + acts)
    assert np.isclose(bc / 1e9, 128.0, atol=1.5)
    assert np.isclose(fc, 6.5e12 * 1.25 + 13e12) and fi == 6.5e12 + 13e12
    # a ring that holds every chunk recomputes nothing
    _, (fc4, bc4) = bench.mx_step_work(spec, 4, 4, 6.5e12, 13e12)
    assert np.isclose(bc4, 8 * w_axis + grads + acts) and fc4 == fi


def test_both_arms_report_the_same_config():
    spec = moe_synth.BF16_T2048
    assert bench.bench_config(spec, 1) == bench.bench_config(spec, 1)
    assert bench.bench_config(spec, 2)["global_batch"] == 2 * spec.T


def test_host_cpu_reports_model_and_cores():
    h = bench.host_cpu()
    assert h["nproc"] == os.cpu_count() and isinstance(h["model"], str) and h["model"]
