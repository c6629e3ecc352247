"""Pins of the parameter-count oracle against the numbers the pages print."""
from oracle import llama_shapes as ls


def test_per_layer_and_totals(golden):
    g = golden("llama32_1b_params.json")
    s = ls.LLAMA_32_1B
    assert ls.layer_params(s) == g["per_layer"]
    assert s.num_layers * ls.layer_params(s) == g["layers_total"]
    assert ls.embedding_params(s) == g["embedding_vh"]
    assert ls.total_params(s) == g["total_approx"]
    # Without the final norm the total is short by exactly h (reading R1).
    no_norm = ls.LlamaShape(final_norm=False)
    assert g["total_approx"] - ls.total_params(no_norm) == s.hidden


def test_per_card_ledger(golden):
    g = golden("llama32_1b_params.json")
    s = ls.LLAMA_32_1B
    tot = ls.total_params(s)
    assert round(tot / 2 / 1e6, 1) == g["pp2_stage_millions_approx"]
    assert round(tot / 4 / 1e6, 1) == g["tp2_card_millions_approx"]
    stage = ls.tp_pp_stage0_tensors(s, tp=2, pp=2)
    n = sum(ls.numel(shp) for _, shp in stage)
    assert n == 374_636_544                      # exact stage-0 list (norms replicated over TP)
    assert round(n / 1e6, 1) == g["tp2_card_millions_approx"]
    b = g["bytes_per_param_zero1_dp2"] * n       # 2 + 4 + 12/dp with dp = 2
    assert 2 + 4 + 12 / 2 == g["bytes_per_param_zero1_dp2"]
    assert round(b / 1e9, 2) == g["per_card_gb_approx"]
    assert round(b / 2**30, 2) == g["per_card_gib_approx"]


def test_tp_split_shapes():
    s = ls.LLAMA_32_1B
    t = dict(ls.tp_layer_tensors(s, 2))
    assert t["qkv"] == (1536, 2048)      # (32 + 2*8) * 64 / 2
    assert t["proj"] == (2048, 1024)
    assert t["fc1"] == (8192, 2048)      # gate + up, 2f / TP
    assert t["fc2"] == (2048, 4096)
    # TP=1 layer tensors sum to the per-layer count of the page's formula.
    full = sum(ls.numel(shp) for _, shp in ls.tp_layer_tensors(s, 1))
    assert full == ls.layer_params(s)
