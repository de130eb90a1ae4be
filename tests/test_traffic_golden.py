"""The roofline's byte and flop model against the numbers the hpc-ops FP8
decode benchmark prints ("[Feature Request] Support q_len > 1 for FP8
decode", hpc-ops issue #4): K+V at 1 B, Q at 1 B and O at 2 B per call times
the printed iterations per second must reproduce the printed GB/s, and
4 * bs * Hq * ctx * D flops the printed TFLOPS, for both implementations."""
import json
import os
import types

import pytest
import torch

from paged_split_kv_03_gb300.traffic import call_bytes, call_flops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hpcops_h200_fp8_decode.json")


def _shape(w):
    B, R = w["batch"], w["q_len"]
    return types.SimpleNamespace(
        page_size=w["block_size"], num_kv_heads=w["num_kv_heads"], head_dim=w["head_dim"],
        num_qo_heads=w["num_qo_heads"], kv_e4m3=True, q_e4m3=True, scale_mode=1,
        kv_len=torch.full((B,), w["kv_len"], dtype=torch.int32),
        qo_indptr=torch.arange(B + 1, dtype=torch.int32) * R, window=None)


@pytest.mark.parametrize("idx", [0, 1])
def test_byte_and_flop_model_reproduce_printed_numbers(idx):
    g = json.load(open(GOLDEN))
    wl = _shape(g["workload"])
    r = g["results"][idx]
    b = call_bytes(wl)
    moved = b["kv"] + b["q"] + b["out"]
    assert b["kv"] == 2 * 128 * 8 * 2048 * 128
    assert abs(moved * r["iter_per_s"] / 1e9 - r["GB_per_s"]) < 0.05
    assert abs(call_flops(wl) * r["iter_per_s"] / 1e12 - r["TFLOPS"]) < 0.005
    # the printed average time is the inverse of the printed rate
    assert abs(1e3 / r["iter_per_s"] - r["avg_ms"]) < 0.0006


def test_mla_latent_counts_once():
    """MLA: the latent is read as K and as V but moves from HBM once (the
    FlashMLA page's MBU); bf16 latent 576 x 2 B per token, records 640 B plus
    four fp32 block scales per token; out has the 512 value channels."""
    from paged_split_kv_03_gb300.synth import config_workload
    for name, per_tok in (("mla_bf16", 576 * 2), ("mla_fp8", 576), ("mla_fp8_mixed", 640 + 16)):
        wl = config_workload(name, bs=2, kv_lens=640)
        assert wl.v_pages is wl.k_pages
        b = call_bytes(wl)
        assert b["kv"] + (b["scales"] if name == "mla_fp8_mixed" else 0) == 2 * 640 * per_tok
        assert b["out"] == 2 * 16 * 512 * 2
        assert call_flops(wl) == 2 * (576 + 512) * 16 * 2 * 640
