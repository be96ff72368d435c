"""The seeded input generators (CPU): the same seed gives the same bytes, a
row sample equals those rows of the full draw, the draws follow the stated
recipe (N(0,1) activations, N(0,0.02) weights, 1% of the activation channels
scaled by 50 in the prefill workload), and the module shares no code with the
oracle or the GPU library."""
import math
import os
import re

import pytest
import torch

import synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_same_seed_same_bytes_other_seed_other_bytes():
    a = synthetic.activation(8, 64, torch.bfloat16, seed=3)
    assert torch.equal(a, synthetic.activation(8, 64, torch.bfloat16, seed=3))
    assert not torch.equal(a, synthetic.activation(8, 64, torch.bfloat16, seed=4))
    w = synthetic.weight(16, 64, torch.bfloat16, seed=3)
    assert torch.equal(w, synthetic.weight(16, 64, torch.bfloat16, seed=3))
    # weights and activations of one seed are independent draws
    assert not torch.equal(w[:8].float() / 0.02, a.float())


@pytest.mark.parametrize("rows", [[0, 5, 1023, 1024, 1500, 2047], [2047, 3, 1024]])
def test_row_sample_equals_the_full_draw(rows):
    # rows on both sides of a 1024-row seed block, in any order
    full = synthetic.weight(2048, 48, torch.bfloat16, seed=11)
    part = synthetic.weight(2048, 48, torch.bfloat16, seed=11, row_subset=rows)
    assert torch.equal(part, full[rows])
    xf = synthetic.activation(2048, 64, torch.float16, seed=5, outlier_frac=0.01)
    xp = synthetic.activation(2048, 64, torch.float16, seed=5, outlier_frac=0.01,
                              row_subset=rows)
    assert torch.equal(xp, xf[rows])
    with pytest.raises(IndexError):
        synthetic.weight(16, 16, torch.float32, seed=1, row_subset=[16])


def test_distributions_follow_the_recipe():
    x = synthetic.activation(512, 1024, torch.float32, seed=21)
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1.0) < 0.01
    w = synthetic.weight(512, 1024, torch.float32, seed=21)
    assert abs(w.mean().item()) < 2e-4 and abs(w.std().item() - 0.02) < 2e-4
    # 16-bit storage is the float32 draw rounded once
    assert torch.equal(synthetic.weight(64, 64, torch.bfloat16, seed=2),
                       synthetic.weight(64, 64, torch.float32, seed=2).to(torch.bfloat16))


def test_outlier_channels():
    K = 4096
    ch = synthetic.outlier_channels(K, seed=7)
    assert ch.numel() == math.ceil(0.01 * K) == 41
    assert len(set(ch.tolist())) == ch.numel() and 0 <= ch.min() and ch.max() < K
    base = synthetic.activation(256, K, torch.float32, seed=7)
    x = synthetic.activation(256, K, torch.float32, seed=7, outlier_frac=0.01)
    mask = torch.zeros(K, dtype=torch.bool)
    mask[ch] = True
    # the outlier columns are the plain draw times 50, the rest untouched
    assert torch.equal(x[:, ~mask], base[:, ~mask])
    assert torch.allclose(x[:, mask], 50.0 * base[:, mask], rtol=0, atol=0)
    # the prefill workload uses them; the others have none
    assert synthetic.WORKLOADS["prefill_w8a8_outliers"].outlier_frac == 0.01
    for name in ("decode_w8a16", "llama3_8b_w8a8_sweep", "llama70b_static_fp8out"):
        assert synthetic.WORKLOADS[name].outlier_frac == 0.0


def test_workload_shapes_and_seeds():
    wl = synthetic.WORKLOADS
    dec = wl["decode_w8a16"]
    assert dec.kind == "w8a16" and dec.x_dtype == torch.float16 and len(dec.shapes) == 12
    assert {(n, k) for (_, n, k) in dec.shapes} == {(12288, 4096), (4096, 4096),
                                                    (22016, 4096), (4096, 11008)}
    assert {m for (m, _, _) in dec.shapes} == {1, 4, 16}
    assert wl["prefill_w8a8_outliers"].shapes == ((1024, 4096, 4096), (1024, 11008, 4096))
    assert len(wl["llama3_8b_w8a8_sweep"].shapes) == 20
    s70 = wl["llama70b_static_fp8out"]
    assert len(s70.shapes) == 16 and s70.act_scale == "static" and s70.out_dtype == "e4m3"
    # every shape of every workload has its own seed, distinct from the
    # calibration draws behind the static scales
    seeds = [w.seed(i) for w in wl.values() for i in range(len(w.shapes))]
    assert len(set(seeds)) == len(seeds)
    assert not set(seeds) & {synthetic.calibration_seed(s) for s in seeds}
    # every size obeys the divisible-by-16 rule of the FP8 products
    for w in wl.values():
        for (_, n, k) in w.shapes:
            assert n % 16 == 0 and k % 16 == 0


def test_generators_share_no_code_with_the_method():
    text = open(os.path.join(ROOT, "synthetic", "__init__.py")).read()
    assert not re.search(r"^\s*(import|from)\s+(oracle|fp8_quantized_linear_gb300)", text, re.M)
    assert "448" not in text  # no E4M3 range, scale or cast
    oracle_text = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert not re.search(r"^\s*(import|from)\s+fp8_quantized_linear_gb300", oracle_text, re.M)
