"""The LoRA+ learning-rate rule ("Chronicals", arXiv 2601.02609, abstract,
optimisation (3): adapter matrix B learns 16x faster than A) as parameter
groups: host logic, no GPU."""
import pytest
import torch

from fine_tuning_gb300.autograd import LORA_PLUS_RATIO, lora_plus_param_groups


class LoraLinear(torch.nn.Module):
    def __init__(self, d_in, d_out, r):
        super().__init__()
        self.base = torch.nn.Linear(d_in, d_out, bias=False)
        self.base.weight.requires_grad_(False)  # frozen base weight
        self.lora_A = torch.nn.Linear(d_in, r, bias=False)
        self.lora_B = torch.nn.Linear(r, d_out, bias=False)


class Model(torch.nn.Module):
    def __init__(self):
        super().__init__()
        self.q_proj = LoraLinear(8, 8, 2)
        self.v_proj = LoraLinear(8, 4, 2)
        self.norm = torch.nn.Parameter(torch.ones(8))


def test_groups_put_b_at_16x():
    m = Model()
    groups = lora_plus_param_groups(m.named_parameters(), lr=1e-4)
    assert LORA_PLUS_RATIO == 16.0
    assert [g["lr"] for g in groups] == [1e-4, 1.6e-3]
    ids = lambda ps: {id(p) for p in ps}
    assert ids(groups[1]["params"]) == ids([m.q_proj.lora_B.weight, m.v_proj.lora_B.weight])
    assert ids(groups[0]["params"]) == ids([m.q_proj.lora_A.weight, m.v_proj.lora_A.weight,
                                            m.norm])
    every = ids(groups[0]["params"]) | ids(groups[1]["params"])
    assert id(m.q_proj.base.weight) not in every  # frozen


@pytest.mark.parametrize("ratio", [16.0, 4.0])
def test_one_sgd_step_moves_b_ratio_times_as_far(ratio):
    torch.manual_seed(0)
    m = Model()
    before = {n: p.detach().clone() for n, p in m.named_parameters()}
    opt = torch.optim.SGD(lora_plus_param_groups(m.named_parameters(), lr=0.01, ratio=ratio))
    for p in m.parameters():
        if p.requires_grad:
            p.grad = torch.ones_like(p)
    opt.step()
    da = (before["q_proj.lora_A.weight"] - m.q_proj.lora_A.weight).abs().max().item()
    db = (before["q_proj.lora_B.weight"] - m.q_proj.lora_B.weight).abs().max().item()
    assert da == pytest.approx(0.01) and db == pytest.approx(0.01 * ratio)
    assert torch.equal(before["q_proj.base.weight"], m.q_proj.base.weight)


def test_weight_decay_and_empty_groups():
    lin = torch.nn.Linear(3, 3)
    groups = lora_plus_param_groups(lin.named_parameters(), lr=0.1, weight_decay=0.01)
    assert len(groups) == 1 and groups[0]["weight_decay"] == 0.01
