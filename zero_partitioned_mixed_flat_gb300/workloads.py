"""Workload definitions: tensor lists, units and step settings of the five
configurations the step is exercised on.

These are architectural sizes only (no weights).  The GPT-2 lists follow the
GPT-2 block (qkv, proj, fc, fc2 weights and biases, two LayerNorms) plus the
token/position embeddings and the final LayerNorm; the 7.5B ZeRO-3 case is a
32-layer d=4096 stack of the same blocks plus one "rest" unit that brings the
total to 7.5e9 parameters (the size of the Figure 1 example in the ZeRO paper
reading notes, "第13篇 · ZeRO" §3.3).  Hyper-parameters not stated for a
configuration take the tiny case's (AdamW, lr 1e-4, betas (0.9, 0.999),
eps 1e-8, wd 0.01, clip 1.0).
"""
from dataclasses import dataclass, field
from typing import List, Optional


def gpt2_block(d: int) -> List[int]:
    """Tensor sizes of one GPT-2 block of width d, in storage order."""
    return [
        d, d,                  # ln_1 gamma, beta
        d * 3 * d, 3 * d,      # attention qkv weight, bias
        d * d, d,              # attention projection weight, bias
        d, d,                  # ln_2 gamma, beta
        d * 4 * d, 4 * d,      # mlp fc weight, bias
        4 * d * d, d,          # mlp fc2 weight, bias
    ]


def gpt2_tensors(d: int, layers: int, vocab: int = 50257, ctx: int = 1024) -> List[int]:
    sizes = [vocab * d, ctx * d]
    for _ in range(layers):
        sizes += gpt2_block(d)
    sizes += [d, d]            # ln_f gamma, beta
    return sizes


def zero3_7p5b_tensors():
    """(sizes, unit_of_tensor) for the 7.5B ZeRO-3 case: unit 0 is the rest
    (embedding-like) unit, units 1..32 are the d=4096 blocks."""
    block = gpt2_block(4096)
    rest = 7_500_000_000 - 32 * sum(block)
    sizes = [rest]
    units = [0]
    for layer in range(32):
        sizes += block
        units += [layer + 1] * len(block)
    return sizes, units


@dataclass
class Workload:
    name: str
    sizes: List[int]
    n_ranks: int
    stage: int
    lp: int                      # 0 = fp16, 1 = bf16
    ranks: List[int]             # partitions updated per step
    steps: int
    loss_scale: float
    growth_interval: int         # <= 0: static loss scale
    grads_times_scale: bool      # grads are N(0, std) * S (fp16 cases)
    unit_of_tensor: Optional[List[int]] = None
    bucket_elems: int = 0
    inject_inf_step: int = 0     # 1-based step with a seeded +inf (0: none)
    gather: bool = False         # stage-3 per-unit forward + backward gathers
    grad_std: float = 1e-3
    master_std: float = 0.02
    align: int = 128
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    wd: float = 0.01
    adamw: bool = True
    clip: float = 1.0
    reduce_lp_accum: bool = False  # partial sums rounded to the lp type
    gather_quantized: bool = False  # stage 3: block-quantized gathers
    quant_format: int = 0           # their codes: 0 int8, 1 fp8 E4M3
    notes: str = field(default="")


def _make():
    w = {}
    w["tiny-zero1"] = Workload(
        name="tiny-zero1", sizes=[1 << 20], n_ranks=4, stage=1, lp=0,
        ranks=[0, 1, 2, 3], steps=3, loss_scale=1024.0, growth_interval=0,
        grads_times_scale=True,
        notes="psi=2^20 one tensor, N=4, all partitions, fp16 grads x 1024 (static)")
    w["gpt2-small-zero1"] = Workload(
        name="gpt2-small-zero1", sizes=gpt2_tensors(768, 12), n_ranks=8, stage=1, lp=1,
        ranks=list(range(8)), steps=3, loss_scale=1.0, growth_interval=0,
        grads_times_scale=False, bucket_elems=50_000_000,
        notes="GPT-2 small tensor list, N=8, all partitions, bf16, buckets of 5e7")
    w["gpt2-xl-zero2"] = Workload(
        name="gpt2-xl-zero2", sizes=gpt2_tensors(1600, 48), n_ranks=64, stage=2, lp=0,
        ranks=[0], steps=3, loss_scale=65536.0, growth_interval=1000,
        grads_times_scale=True, inject_inf_step=2,
        notes="GPT-2 1.5B tensor list, N=64 rank 0, fp16, dynamic scale 2^16, +inf on step 2")
    s, u = zero3_7p5b_tensors()
    w["7.5b-zero3"] = Workload(
        name="7.5b-zero3", sizes=s, unit_of_tensor=u, n_ranks=64, stage=3, lp=0,
        ranks=[0], steps=4, loss_scale=65536.0, growth_interval=1000,
        grads_times_scale=True, gather=True, bucket_elems=500_000_000,
        notes="7.5B, 33 units (rest + 32 d=4096 blocks), N=64 rank 0, fp16, gathers, "
              "reduce buckets of 5e8 elements")
    w["7.5b-zero3-q8"] = Workload(
        name="7.5b-zero3-q8", sizes=s, unit_of_tensor=u, n_ranks=64, stage=3, lp=0,
        ranks=[0], steps=4, loss_scale=65536.0, growth_interval=1000,
        grads_times_scale=True, gather=True, gather_quantized=True, bucket_elems=500_000_000,
        notes="7.5b-zero3 with ZeRO++-style int8 block-quantized gathers")
    w["7.5b-zero3-fp8"] = Workload(
        name="7.5b-zero3-fp8", sizes=s, unit_of_tensor=u, n_ranks=64, stage=3, lp=0,
        ranks=[0], steps=4, loss_scale=65536.0, growth_interval=1000,
        grads_times_scale=True, gather=True, gather_quantized=True, quant_format=1,
        bucket_elems=500_000_000,
        notes="7.5b-zero3 with fp8 (E4M3, power-of-two block scale) quantized gathers")
    w["13b-zero2"] = Workload(
        name="13b-zero2", sizes=[13_000_000_000], n_ranks=16, stage=2, lp=1,
        ranks=[0], steps=4, loss_scale=1.0, growth_interval=0,
        grads_times_scale=False,
        notes="13B one flat tensor, N=16 rank 0, bf16, HBM-capacity case")
    # small cases of the same kernels, for profiler captures (a few GB on the
    # device, inputs still larger than the 129 MB L2); not benchmark lines
    w["profile-zero2"] = Workload(
        name="profile-zero2", sizes=[16 << 25], n_ranks=16, stage=2, lp=1, ranks=[0],
        steps=4, loss_scale=1.0, growth_interval=0, grads_times_scale=False,
        notes="13b-zero2 kernels at 2^29 parameters (P = 2^25)")
    blocks = gpt2_block(1024)
    w["profile-zero3"] = Workload(
        name="profile-zero3", sizes=[64 << 20] + blocks + blocks,
        unit_of_tensor=[0] + [1] * len(blocks) + [2] * len(blocks), n_ranks=64, stage=3,
        lp=0, ranks=[0], steps=4, loss_scale=65536.0, growth_interval=1000,
        grads_times_scale=True, gather=True,
        notes="7.5b-zero3 kernels on 3 units (64M rest + two d=1024 blocks)")
    w["profile-zero3-q8"] = Workload(
        name="profile-zero3-q8", sizes=[1 << 28], unit_of_tensor=[0], n_ranks=4, stage=3,
        lp=0, ranks=[0], steps=4, loss_scale=65536.0, growth_interval=1000,
        grads_times_scale=True, gather=True, gather_quantized=True,
        notes="quantize and dequantizing-gather kernels on one 2^28 unit, N=4 (P = 2^26)")
    return w


WORKLOADS = _make()
