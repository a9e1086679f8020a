"""Checks of the seeded input generators and the MoE routing glue (CPU only)."""

import numpy as np
import torch

import synth


def test_same_seed_same_bytes_and_independent_streams():
    a = synth.normal_bf16((64, 256), 1.0, 0, synth.TAG_X)
    b = synth.normal_bf16((64, 256), 1.0, 0, synth.TAG_X)
    c = synth.normal_bf16((64, 256), 1.0, 0, synth.TAG_W)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a, c)


def test_outlier_recipes():
    z = synth.normal_f32((1000, 1000), 1.0, 0, 1, outlier_p=0.01, outlier_mult=50.0)
    frac = np.mean(np.abs(z) > 8)          # N(0,1) beyond 8 sigma is ~1e-15
    assert 0.007 < frac < 0.011
    t = synth.normal_f32((1000, 1000), 1.0, 0, 2, outlier_p=0.005, outlier_t_nu=2.0)
    assert np.max(np.abs(t)) > 10                      # heavy tail: N(0,1) never reaches this


def test_dense_case_shapes():
    c = synth.dense_case("tiny")
    assert c.x().shape == (256, 512) and c.w().shape == (256, 512)
    assert c.x().dtype == torch.bfloat16
    assert synth.dense_case("fprop").flops == 2 * 4096 * 18432 * 7168


def _route_bruteforce(x, R, bias, k):
    out = []
    for t in range(x.shape[0]):
        aff = [1.0 / (1.0 + np.exp(-float(np.float32(x[t] @ R[e])))) for e in range(R.shape[0])]
        sel = sorted(range(R.shape[0]), key=lambda e: (-(aff[e] + bias[e]), e))[:k]
        out.append(set(sel))
    return out


def test_routing_small_case():
    case = synth.MOE_SMALL
    x = synth.bf16_to_f32(case.tokens())
    R, bias = case.router(), case.bias()
    r = synth.moe_route(x, R, bias, case.topk)
    assert r["offsets"][0] == 0 and r["offsets"][-1] == case.rows
    assert np.all(np.diff(r["offsets"]) >= 0)
    assert r["counts"].sum() == case.rows
    for t in range(case.T):
        assert len(set(r["topk"][t].tolist())) == case.topk
    # rows ordered by expert, then token
    e, tok = r["expert_of_row"], r["token_of_row"]
    key = e * case.T + tok
    assert np.all(np.diff(key) > 0)
    for i in range(case.E):
        assert np.all(e[r["offsets"][i]:r["offsets"][i + 1]] == i)
    bf = _route_bruteforce(x, R, bias, case.topk)
    for t in range(case.T):
        assert set(r["topk"][t].tolist()) == bf[t]


def test_expert_weight_cpu_recipe():
    case = synth.MOE_SMALL
    w = synth.expert_weight(case, 3, "up")
    assert w.shape == (2 * case.I, case.H)
    assert torch.equal(w, synth.expert_weight(case, 3, "up"))
    assert not torch.equal(w, synth.expert_weight(case, 4, "up"))
    assert synth.expert_weight(case, 3, "down").shape == (case.H, case.I)


def test_ragged_offsets():
    assert synth.ragged_offsets([3, 0, 2]).tolist() == [0, 3, 3, 5]
