"""The cost-model module reproduces the numbers the pages print."""

import json
import os

import pytest

from megatron_tensor_layers_gb300 import costmodel as cm


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_decode_table_of_the_page(golden_dir):
    g = _golden(golden_dir, "aiinfra62_decode_cost_table.json")
    a = g["assumptions"]
    m = cm.DecodeModel(layers=a["layers"], hidden=a["hidden"], weight_bytes=a["weight_bytes"],
                       kv_bytes_per_token=a["kv_per_token"], ctx=a["ctx"], kv_rank_limit=a["kv_rank_limit"])
    for row in g["rows"]:
        r = cm.decode_step(m, row["tp"], row["batch"], a["hbm"], a["link"], a["alpha"])
        assert r["step_s"] * 1e3 == pytest.approx(row["step_ms"], abs=0.006)
        assert r["comm_s"] * 1e3 == pytest.approx(row["comm_ms"], abs=0.006)
        assert round(r["tokens_per_s"]) == row["tok_s"]
        assert round(r["tokens_per_s_per_gpu"]) == row["tok_s_per_gpu"]


def test_comm_versus_compute_of_the_page(golden_dir):
    g = _golden(golden_dir, "tpscratch_comm_cost.json")
    a, p = g["assumptions"], g["printed"]
    dec = cm.comm_per_forward(a["layers"], a["hidden"], 64, a["tp"], a["busbw"], a["alpha"])
    assert round(dec * 1e3, 1) == p["decode_batch64_comm_ms"]
    weight_floor = a["params"] * 2 / a["tp"] / a["hbm"]
    assert round(weight_floor * 1e3, 1) == p["decode_weight_floor_ms"]
    pre = cm.comm_per_forward(a["layers"], a["hidden"], 4096, a["tp"], a["busbw"], a["alpha"])
    assert round(pre * 1e3) == p["prefill_4096_comm_ms"]
    comp = cm.prefill_compute(a["params"], 4096, a["tp"], a["peak_flops"], a["mfu"])
    assert round(comp * 1e3) == p["prefill_4096_compute_ms"]


def test_simulated_allreduce_and_cli(capsys):
    assert cm.simulated_allreduce_time(1 << 20, 4, 5e12, 0.0) == pytest.approx(5 * (1 << 20) / 5e12)
    rows = cm.gb300_table({"hbm_bytes_per_s": 6.5e12, "launch_s": 3e-6})
    assert [r["tokens"] for r in rows] == [1, 64, 8192]
    assert rows[2]["nvlink_tp8_us"] == pytest.approx(522, rel=0.01)     # the page's "about 520 us"
    cm._main([])
    assert "42.55" in capsys.readouterr().out


def test_allreduces_per_forward_of_the_page(golden_dir):
    g = _golden(golden_dir, "tpscratch_allreduce_count.json")
    assert cm.allreduces_per_forward(g["layers"]) == g["prefill_forward_allreduces"]
    assert g["allreduce_per_layer"] * g["layers"] + g["embedding_allreduce"] == g["prefill_forward_allreduces"]
