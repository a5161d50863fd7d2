"""Golden fixtures: the pages' printed workload facts, and a stored oracle
encoding of an explicit tiny input (regression pin of the oracle)."""
import os

import numpy as np

from nvfp4_linear_lora_gb300 import configs
from oracle import nvfp4

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _facts():
    out = {}
    for line in open(os.path.join(GOLDEN, "page_facts.txt")):
        if line.startswith("#") or not line.strip():
            continue
        key, val = line.split("|")[0].split()
        out[key] = int(val)
    return out


def test_page_facts_consistent():
    f = _facts()
    assert f["adapter_linear_targets"] == f["projections_per_block"] * (f["denoiser_blocks"] + f["token_refiner_blocks"])
    assert f["adapter_tensors_per_file"] == 3 * f["adapter_linear_targets"]   # A, B, alpha per target


def test_configs_follow_page_facts():
    f = _facts()
    ranks = {name: r for name, _, _, r, _ in configs.BLOCK_PROJECTIONS}
    assert len(configs.BLOCK_PROJECTIONS) == f["projections_per_block"] == f["nvfp4_matrices_per_block"]
    assert ranks["qkv"] == f["rank_alpha_fused_qkv"]
    assert ranks["attn_out"] == ranks["gate_up"] == ranks["down"] == f["rank_alpha_other"]
    assert configs.BLOCK_S == f["packed_S_16_token_prompt"]
    assert configs.SWITCH_S == f["packed_S_18_token_prompt"]


def test_oracle_tiny_golden():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    x, s = mg.tiny_input()
    packed, scales, ts = nvfp4.quantize(x, s)
    rows = {}
    for line in open(os.path.join(GOLDEN, "nvfp4_tiny.txt")):
        if line.startswith("#"):
            continue
        k, v = line.split()
        rows[k] = v
    assert int(rows["tensor_scale_f32_hex"], 16) == int(np.float32(ts).view(np.uint32))
    for r in range(packed.shape[0]):
        assert scales[r].tobytes().hex() == rows[f"scales_row{r}"]
        assert packed[r].tobytes().hex() == rows[f"codes_row{r}"]
