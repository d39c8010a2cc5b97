"""Host-side accounting of bench.py: the algorithmic bytes behind the
roofline figure, the launch count it claims, and the gate that keeps an ncu
traffic figure from outliving the kernel source it was taken on."""

import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

HASHED = ("decode.cu", "gemm_common.cuh", "quant_math.cuh", "ptx.cuh", "internal.h")


def test_linear_bytes_closed_form():
    # packed codes N*K/2, one scale byte per 32 K, bf16 activations in, bf16 out
    assert bench.linear_bytes(1, 14336, 5120) == 14336 * 2560 + 14336 * 160 + 2 * 5120 + 2 * 14336
    # K not a multiple of 32: the last block still has a scale byte
    assert bench.linear_bytes(3, 1000, 5152) == 1000 * 2576 + 1000 * 161 + 2 * 3 * 5152 + 2 * 3 * 1000
    # the GEMM-only figure reads the quantized activations instead of bf16
    assert bench.gemm_kernel_bytes(16, 1024, 5120) == 1024 * 2560 + 1024 * 160 + 16 * 2560 + 16 * 160 + 2 * 16 * 1024


def test_decode_sweep_shape_and_step_bytes():
    cases = [(M, N, K) for M in bench.DECODE_MS for (N, K) in bench.DECODE_NK]
    assert len(cases) == 15
    step = sum(bench.linear_bytes(*c) for c in cases)
    weights = 5 * sum(N * K // 2 + N * K // 32 for (N, K) in bench.DECODE_NK)
    assert weights < step < weights * 1.03          # the weight stream is almost all the bytes


@pytest.mark.parametrize("M,want", [(1, 1), (8, 1), (9, 2), (16, 2), (64, 2)])
def test_launches_per_decode_call(M, want):
    assert bench.launches_per_call(M, 14336, 5120) == want


def _copy_sources(tmp_path):
    src = os.path.join(ROOT, "mxfp4_quantized_gemm_gb300", "csrc")
    dst = tmp_path / "mxfp4_quantized_gemm_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in HASHED:
        shutil.copy(os.path.join(src, f), dst / f)
    (tmp_path / "profiles").mkdir()
    return dst


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    with open(dst / "decode.cu", "a") as f:
        f.write("\n// a comment only\n\n")
    assert bench.kernel_source_hash() == h0
    with open(dst / "decode.cu", "a") as f:
        f.write("static int unused_probe_value = 1;   // code\n")
    assert bench.kernel_source_hash() != h0


def test_recorded_traffic_only_for_matching_source(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    ratios = "".join(f"ratio_{N}_{K} = 1.01\n" for (N, K) in bench.DECODE_NK)
    cases = [(1, 14336, 5120), (64, 34816, 5120)]
    traffic = tmp_path / "profiles" / "decode_gemm_traffic.txt"
    traffic.write_text(f"# test\nsource_hash = {bench.kernel_source_hash()}\n" + ratios)
    want = round(sum(1.01 * bench.linear_bytes(*c) for c in cases) / len(cases))
    assert bench.recorded_traffic(cases) == want
    traffic.write_text("source_hash = 0000000000000000\n" + ratios)
    assert bench.recorded_traffic(cases) is None    # taken on another kernel source
    traffic.unlink()
    assert bench.recorded_traffic(cases) is None
