"""The arithmetic behind bench.py's roofline fields, on the CPU: the method's
algorithmic work per (token, head), the roofline of a prefill launch, and
the reading of committed ncu summaries (used only while the kernel sources
they were taken on are unchanged)."""
import hashlib
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_helpers_mod",
                                                  os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_algorithmic_work_per_token_head(bench):
    """The hot-path scope's figures, written out: q, k, v and out in bf16,
    log alpha in fp32 and beta once per (token, head) at d = 128; the dense
    contractions K K^T, Q K^T, A^kk (beta V), A^kk (beta Gamma K), A^qk E
    (2 C d flop each) and W S, K_end^T E, Q_hat S (2 d^2 each) at C = 64."""
    d, C = 128, 64
    assert bench.path_bytes_per_tok_head(d) == (3 + 1) * d * 2 + d * 4 + 4 == 1540
    assert bench.prefill_flops_per_tok_head(d, C) == 5 * 2 * C * d + 3 * 2 * d * d == 180224
    assert bench.PATH_BYTES == 1540 and bench.PATH_FLOPS == 180224


def test_prefill_roofline_arithmetic(bench):
    """The dominant stage's time against the method's work for the launch's
    units; the whole call beside it; scratch traffic reported apart."""
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0, "source": "test"}
    units = 1_000_000
    r = bench.prefill_roofline({"prep": 2.0, "scan": 1.0, "out": 0.5}, units, 2.5, peaks,
                               traffic=123, traffic_note="n")
    assert r["kernel"] == "prep" and r["launch_ms"] == 2.0
    assert r["algorithmic_bytes_per_launch"] == 1540 * units
    assert r["achieved"] == pytest.approx(1540e6 / 2e-3 / 1e9)          # 770 GB/s
    assert r["frac"] == pytest.approx(0.77)
    assert r["tensor_tflops"] == pytest.approx(180224e6 / 2e-3 / 1e12)
    assert r["tensor_frac"] == pytest.approx(r["tensor_tflops"] / 100.0)
    assert r["whole_call"]["gbs"] == pytest.approx(1540e6 / 2.5e-3 / 1e9)
    assert r["whole_call"]["frac"] == pytest.approx(0.616)
    assert r["overhead_bytes"] == pytest.approx(bench.SCRATCH_BYTES["prep"] * units)
    assert r["traffic"] == 123 and r["traffic_note"] == "n"


def _summary(root, src_text, digest_of=None):
    """A kernel source and an ncu summary naming it, under `root`."""
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    src = os.path.join(root, "k.cu")
    with open(src, "w") as f:
        f.write(src_text)
    digest = hashlib.sha256((digest_of or src_text).encode()).hexdigest()
    with open(os.path.join(root, "profiles", "k.md"), "w") as f:
        f.write("# k\n\nsource_sha256: %s  (k.cu)\ndram_bytes_per_launch: 4096\n" % digest)


def test_profiled_traffic_follows_the_source_hash(bench, tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "PROFILE_FILES", {"k": ("k.md", 1000), "none": (None, None)})
    _summary(str(tmp_path), "kernel source\n")
    assert bench.profiled_traffic("k") == 4096
    # counters taken on other code: no traffic figure
    _summary(str(tmp_path), "changed kernel source\n", digest_of="kernel source\n")
    assert bench.profiled_traffic("k") is None
    assert bench.profiled_traffic("none") is None
    assert bench.profiled_traffic("unknown") is None


def test_profiled_traffic_scales_with_the_units(bench, tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "PROFILE_FILES", {"k": ("k.md", 1000)})
    _summary(str(tmp_path), "kernel source\n")
    t, note = bench.profiled_traffic_scaled("k", 1000)
    assert t == 4096 and note == "ncu capture of this workload"
    t, note = bench.profiled_traffic_scaled("k", 512_000)
    assert t == 4096 * 512 and "scaled by 512" in note
