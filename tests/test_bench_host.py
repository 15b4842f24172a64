"""Host logic of bench.py that decides what a bench line reports: the code
hash that keys the ncu traffic record (comments and blank lines do not count,
code does) and the record lookup itself."""
import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def test_source_hash_ignores_comments_not_code(tmp_path):
    b = _bench()
    (tmp_path / "common.cuh").write_text("// helpers\n__device__ int h() { return 1; }\n")
    k = tmp_path / "k.cu"
    k.write_text("// a kernel\n__global__ void k(int* p) { *p = 1; }  // store one\n\n")
    base = b.source_hash(str(k))
    k.write_text("// a kernel, described differently\n\n__global__ void k(int* p) { *p = 1; }\n")
    assert b.source_hash(str(k)) == base
    k.write_text("__global__ void k(int* p) { *p = 2; }\n")
    assert b.source_hash(str(k)) != base
    (tmp_path / "common.cuh").write_text("__device__ int h() { return 2; }\n")
    k.write_text("// a kernel\n__global__ void k(int* p) { *p = 1; }\n")
    assert b.source_hash(str(k)) != base


def test_traffic_record_entries_name_existing_sources():
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for key in ("k_fc2_gemm", "swiglu_producer"):
        src = os.path.join(ROOT, "diffusion_transformer_mlp_gb300", "csrc", rec[key]["source"])
        assert os.path.exists(src)
        assert rec[key]["bytes_per_launch"] > 0
        assert len(rec[key]["source_sha256_16"]) == 16


def test_quantize_only_bytes_and_percentiles():
    """The quantise-only workload's algorithmic bytes (two reads of the BF16
    input, QDATA and scales written once) and the percentile helper of the
    ragged-M report."""
    b = _bench()
    m, f = 37810, 5376
    assert b.quant_only_bytes(m, f) == 2 * m * f * 2 + 37888 * f // 2 + 37888 * (f // 16)
    # the SwiGLU producer writes the same NVFP4 bytes and reads twice the BF16
    # input (gate and up) in each of its two passes
    k = 14336
    assert b.producer_bytes(m, k) - 2 * (m * 2 * k * 2) == b.quant_only_bytes(m, k) - 2 * (m * k * 2)
    vals = list(range(1, 51))
    # nearest rank on the sorted runs: index round(q (n - 1))
    assert b._pct(vals, 0.5) == 25 and b._pct(vals, 0.9) == 45 and b._pct([3.0], 0.9) == 3.0
