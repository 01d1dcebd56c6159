"""The measurement helpers in bench.py reproduce the analytic numbers the pages print."""

import os

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "wall_analytics.txt")
P, W_P = 70e9, 2.0
PER_TOKEN = bench.kv_bytes_per_token(80, 8, 128, 2)


def _rows():
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            kind, *kv = line.split()
            yield kind, {k: float(v) for k, v in (x.split("=") for x in kv)}


def test_per_token_bytes_of_the_70b_shape():
    assert PER_TOKEN == 327680


def test_wall_page_numbers():
    seen = set()
    for kind, a in _rows():
        seen.add(kind)
        if kind == "crossover":
            s = bench.traffic_crossover_tokens(P, W_P, int(a["batch"]), PER_TOKEN)
            assert round(s / 1e3, 1) == round(a["tokens"] / 1e3, 1)
        elif kind == "speedup":
            kvb = a["context"] * PER_TOKEN / 1e9
            assert round(bench.kv_speedup(P * W_P / 1e9, kvb, a["c"]), 2) == a["value"]
        elif kind == "stepbytes":
            assert round(P * W_P / 1e9 + a["context"] * PER_TOKEN / 1e9, 1) == a["gb"]
        elif kind == "intensity":
            assert bench.decode_intensity(int(a["g"]), a["w_kv"]) == a["flop_per_byte"]
    assert seen == {"crossover", "speedup", "stepbytes", "intensity"}


def test_workload_bytes_per_step_are_the_closed_form():
    from kvd_inputs import get

    assert get("llama8b").kv_bytes_per_step() == 32 * 8192 * bench.kv_bytes_per_token(32, 8, 128, 2)
    w = get("llama70b_fp8")
    assert w.kv_bytes_per_step() == 131072 * bench.kv_bytes_per_token(80, 8, 128, 1)
    assert w.kv_bytes_per_step() == 20 * 2 ** 30
