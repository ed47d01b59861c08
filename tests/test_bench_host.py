"""Host-side logic of bench.py (CPU only): the work model and the analytic
ring all-reduce time of "Tensor parallel serving" ("Communication cost")."""
import math

import bench


def test_ring_allreduce_time_model():
    B = bench.LINK_GBPS * 1e9
    assert bench.ring_allreduce_us(1, 1e9) == 0.0
    # p = 2: each rank sends and receives half the message twice -> bytes / B
    assert math.isclose(bench.ring_allreduce_us(2, 1e9), 1e9 / B * 1e6)
    # p = 8: 2 * 7/8 = 1.75 message lengths over the link
    assert math.isclose(bench.ring_allreduce_us(8, 4096 * 8192 * 2), 1.75 * 4096 * 8192 * 2 / B * 1e6)
    # grows towards 2 * bytes / B as p grows
    assert bench.ring_allreduce_us(1024, 1e9) < 2 * 1e9 / B * 1e6


def test_work_model_covers_every_workload():
    for name, w in bench.WORKLOADS.items():
        work = bench.kernel_work(w)
        assert work, name
        for flops, nbytes in work.values():
            assert flops > 0 and nbytes > 0, name
    # the prefill FFN: 2*M*d*(2 d_ff) for gate+up, 2*M*d_ff*d for down
    w = bench.WORKLOADS["swiglu_ffn_prefill_tp8"]
    work = bench.kernel_work(w)
    assert work["column"][0] == 2.0 * 4096 * 8192 * 2 * 28672
    assert work["row"][0] == 2.0 * 4096 * 28672 * 8192
    # decode: weight bytes dominate
    w = bench.WORKLOADS["swiglu_ffn_decode_tp4_b1"]
    col, row = bench.kernel_work(w)["column"], bench.kernel_work(w)["row"]
    assert abs(col[1] - 2 * 2 * 28672 * 8192) < 1e6 and abs(row[1] - 2 * 28672 * 8192) < 1e6
    # the uneven split's widths cover d_ff
    w = bench.WORKLOADS["column_uneven_decode_tp3_b8"]
    assert sum(w["widths"]) == w["dff"] and len(w["widths"]) == w["tp"]


def test_fp8_work_model_halves_weight_bytes():
    """FP8 workloads stream one byte per weight plus one fp32 scale per weight
    row (per shard on the row side); FLOPs are unchanged."""
    bf = bench.kernel_work(bench.WORKLOADS["swiglu_ffn_decode_tp4_b1"])
    f8 = bench.kernel_work(bench.WORKLOADS["swiglu_ffn_decode_tp4_b1_fp8"])
    d, dff, tp = 8192, 28672, 4
    assert f8["column"][0] == bf["column"][0] and f8["row"][0] == bf["row"][0]
    assert f8["column"][1] == bf["column"][1] - 2 * dff * d + 4 * 2 * dff
    assert f8["row"][1] == bf["row"][1] - dff * d + 4 * tp * d


def test_decode_extras_and_datasheet_denominators():
    """The default run also times the decode-shaped workloads; every fraction is
    reported against the measured peaks and against the datasheet figures."""
    assert set(bench.DECODE_EXTRAS) <= set(bench.WORKLOADS)
    for name in bench.DECODE_EXTRAS:
        w = bench.WORKLOADS[name]
        assert w["kind"] == "ffn" and w["M"] <= 64
        # decode is HBM-bound: its intensity is far below the ridge point
        flops = sum(f for f, _ in bench.kernel_work(w).values())
        nbytes = sum(b for _, b in bench.kernel_work(w).values())
        assert flops / nbytes < 100
    assert bench.DATASHEET["hbm_gbs"] == 8000.0 and bench.DATASHEET["bf16_tflops"] == 2250.0
