"""The benchmark's roofline arithmetic, on CPU, against counts worked out by hand.

The bench line's `roofline.achieved` is algorithmic bytes (decode) or FLOPs (scan) over the
measured time, so a wrong count would misstate every fraction it prints.  Each expected value
below is written out from the shapes, not from the functions under test.
"""
from __future__ import annotations

import bench
from linear_attention_recurrence_gdn_gb300.workloads import (DECODE_B64, DECODE_B256_HM,
                                                             LONG_B2, PREFILL_B4)


def test_decode_bytes_of_the_two_decode_workloads():
    # state f32 read + write: 2 * 4 * B * Hv * Dv * Dk; q, k (bf16) per key head; v, z (bf16)
    # and y (f32) per value head row; two f32 gates per value head; the f32 norm weight
    def by_hand(B, Hk, Hv, D):
        state = 2 * 4 * B * Hv * D * D
        qk = 2 * B * Hk * D * 2
        vzy = B * Hv * (2 * D * 2 + 4 * D)
        gates = B * Hv * 8
        return state + qk + vzy + gates + 4 * D
    assert bench.decode_bytes(DECODE_B64) == by_hand(64, 16, 32, 128) == 271_073_792
    assert bench.decode_bytes(DECODE_B256_HM) == by_hand(256, 16, 32, 128) == 1_084_293_632


def test_scan_flops_is_six_dk_dv_per_token_head():
    assert bench.scan_flops(PREFILL_B4) == 6 * 128 * 128 * 4 * 4096 * 32 == 51_539_607_552
    assert bench.scan_flops(LONG_B2) == 6 * 128 * 128 * 2 * 16384 * 32


def test_chunked_kernel_issued_flops_per_chunk():
    # per head and 64-token chunk: 76 MMAs of N = 64 (tables 8, W 8, U 8, X 24, Y 16, O 12) and
    # 8 of N = 128 (the update), each M = 128, K = 16: 2 * 128 * N * 16 FLOP
    per_chunk = 76 * (2 * 128 * 64 * 16) + 8 * (2 * 128 * 128 * 16)
    one = PREFILL_B4.replace(B=1, S=64, Hk=1, Hv=1)
    assert bench.scan_wy_mma_flops(one) == per_chunk == 24_117_248
    # a ragged last chunk costs a whole chunk; heads multiply
    assert bench.scan_wy_mma_flops(PREFILL_B4.replace(B=2, S=65, Hk=1, Hv=3)) == 2 * 3 * 2 * per_chunk


def test_whole_job_rate_is_all_units_over_the_slowest_rank():
    assert bench.aggregate_rate(100.0, 4, 2.0) == 200.0


def test_peaks_fall_back_when_the_measured_file_is_absent(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback"
    assert p["hbm_gbs"] == bench.FALLBACK_HBM_GBS and p["bf16_tflops"] == bench.FALLBACK_BF16_TFLOPS
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 7000.5, "bf16_tflops": 1800.0}')
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["hbm_gbs"] == 7000.5 and p["bf16_tflops"] == 1800.0
