"""The roofline arithmetic of bench.py (algorithmic bytes per kernel class and
FLOPs per step) against figures fixed independently of that code:

* KV bytes per token per step: 12 layers x 2 x 10 kv heads x 128 x 2 B = 61,440
  for the 3B-MoE shape and 36 x 2 x 8 x 128 x 2 = 147,456 for the dense 4B shape;
* the expert gate/up bytes of the committed ncu capture (13 active experts,
  4 rows): profiles/ncu_traffic.json;
* the LM-head bytes of a 128-row launch printed by a GPU run: 331,612,160;
* per-row FLOPs / 2 = the parameters a token meets, close to the ~570M active
  parameters the Jina-OCR-v1 abstract states for the 3B-MoE decoder."""
import json
import os

import pytest

import bench
import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _one(k, **extra):
    return {k: dict(launches=1, ms=1.0, **extra)}


@pytest.mark.parametrize("cfg,per_token", [(syn.MOE3B, 61_440), (syn.DENSE4B, 147_456)])
def test_kv_bytes_per_token(cfg, per_token):
    # attention reads L * ctx_sum * 2 * H_kv * d * 2 bytes: one token of context, one step
    cb = bench.class_bytes(cfg, {}, T=1, ctx_sum=1.0, n_steps=1)
    assert cb["attn_splitkv_merge"] == per_token


def test_gateup_bytes_match_the_profiled_capture():
    cap = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))["expert_gateup_swiglu"]["captured"]
    cb = bench.class_bytes(syn.MOE3B, _one("expert_gateup_swiglu", units=cap["active_experts"]), T=4, ctx_sum=0.0,
                           n_steps=1)
    assert cb["expert_gateup_swiglu"] == cap["algorithmic_bytes"]
    # 2 matrices x 896 x 1280 bf16 per expert, plus the step's activations
    assert cap["algorithmic_bytes"] == 13 * 2 * 896 * 1280 * 2 + 4 * 1280 * 4 + 4 * 8 * 896 * 4


def test_lmhead_bytes():
    cb = bench.class_bytes(syn.MOE3B, _one("lmhead_argmax_commit"), T=128, ctx_sum=0.0, n_steps=1)
    assert cb["lmhead_argmax_commit"] == 331_612_160 == 129_280 * 1280 * 2 + 128 * 1280 * 4


def test_fp8_weights_count_one_byte_and_the_row_scales():
    bf = bench.class_bytes(syn.MOE3B, _one("expert_down", units=1), T=1, ctx_sum=0.0, n_steps=1)["expert_down"]
    f8 = bench.class_bytes(syn.MOE3B_FP8, _one("expert_down", units=1), T=1, ctx_sum=0.0, n_steps=1)["expert_down"]
    act = 1 * 8 * 896 * 4 + 1 * 8 * 1280 * 4
    assert bf - act == 1280 * 896 * 2
    assert f8 - act == 1280 * (896 * 1 + 4)


def test_flops_per_row_are_the_active_parameters():
    cfg = syn.MOE3B
    per_row = bench.step_flops_of(cfg, T=1, R=1, ctx_sum=0.0, n_steps=1) / 2
    assert abs(per_row - 570e6) / 570e6 < 0.05          # "~570M active parameters per token"
    # attention FLOPs: 4 x keys x H_q x d per row and layer (QK^T and PV)
    extra = bench.step_flops_of(cfg, T=1, R=1, ctx_sum=100.0, n_steps=1) - 2 * per_row
    assert extra == 4 * cfg.n_layers * cfg.n_q_heads * cfg.head_dim * 100


def test_rejection_sampling_traffic_record_is_consistent():
    """The sampler's traffic record: its algorithmic bytes are the rows the
    rule must read (accepted drafts plus one row per sequence, V f32 each, as
    sampling_leg and --sampling-probe count them), and its ratio is the
    captured DRAM bytes over those."""
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))["rejection_sampling"]
    cap = rec["captured"]
    assert cap["algorithmic_bytes"] == (cap["accepted_total"] + 64) * 129_280 * 4
    ratio = (cap["dram_read_bytes"] + cap["dram_write_bytes"]) / cap["algorithmic_bytes"]
    assert abs(rec["traffic_over_algorithmic"] - ratio) < 1e-12
    # while the sources hash to the capture, the bench scales the ratio to a launch's bytes
    t = bench.traffic_for("rejection_sampling", 1e6)
    assert t is None or abs(t - 1e6 * ratio) < 1e-3
