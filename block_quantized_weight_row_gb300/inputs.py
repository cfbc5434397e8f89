"""Seeded synthetic inputs for the block-quantized weight-row workloads.

This module only draws random numbers and names shapes; it holds none of the
method's arithmetic. The tests, the benchmark and the smoke check use it to
feed the SAME tensor to the CUDA path and to the CPU oracle. Values depend on
the device the generator runs on (torch's CPU and CUDA generators produce
different streams), so a caller draws once and copies to wherever it needs.

Workloads (shapes and distributions of the pages' models):
  tiny       W 1024 x 1024 ~ N(0, 0.02), x ~ N(0, 1), seed 0
  qwen3-0.6b 28 layers x {q 2048x1024, k 1024x1024, v 1024x1024, o 1024x2048,
             gate 3072x1024, up 3072x1024, down 1024x3072}  (M x K)
  7b         32 layers x {q,k,v,o 4096x4096, gate 11008x4096, up 11008x4096,
             down 4096x11008}
  prefill    X 512 x K ~ N(0, 1), W (M x K) ~ N(0, 0.02) for
             (4096, 4096), (11008, 4096), (4096, 11008)
  kv         per layer K, V [32768][8][128]; K = mu + N(0, 1) with
             mu[h][c] ~ U(-2, 2) per layer, V ~ N(0, 1); a separate 4096-token
             calibration draw of K gives the bias; 28 layers
  legacy     W 11008 x 4096 ~ N(0, 0.02) (8 draws), x ~ N(0, 1): the GEMV in
             Q4_1, Q5_0, Q5_1, Q4_K, Q6_K (and Q4_0 for comparison)
Seeds: workload index * 1000 + layer * 10 + matrix index.
"""
from dataclasses import dataclass

import torch

WEIGHT_STD = 0.02

# (name, M, K); q/k/v read the attention input, o the attention output,
# gate/up the FFN input, down the FFN hidden state.
QWEN3_0_6B_LAYER = (("q", 2048, 1024), ("k", 1024, 1024), ("v", 1024, 1024),
                    ("o", 1024, 2048), ("gate", 3072, 1024), ("up", 3072, 1024),
                    ("down", 1024, 3072))
LLAMA_7B_LAYER = (("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096),
                  ("o", 4096, 4096), ("gate", 11008, 4096), ("up", 11008, 4096),
                  ("down", 4096, 11008))
# which activation each matrix reads: matrices with the same input share one x
LAYER_INPUT = {"q": "attn_in", "k": "attn_in", "v": "attn_in", "o": "attn_out",
               "gate": "ffn_in", "up": "ffn_in", "down": "ffn_hidden"}

WORKLOADS = {
    "tiny": dict(index=0),
    "qwen3-0.6b-decode": dict(index=1, layers=28, layer=QWEN3_0_6B_LAYER),
    "7b-decode": dict(index=2, layers=32, layer=LLAMA_7B_LAYER),
    "prefill-q8_0": dict(index=3, tokens=512, shapes=((4096, 4096), (11008, 4096), (4096, 11008))),
    "kv-write": dict(index=4, layers=28, tokens=32768, kv_heads=8, head_dim=128, calib_tokens=4096),
    # the 7B gate/up shape in every legacy weight type
    "legacy-gemv": dict(index=5, shape=(11008, 4096)),
}


def seed_of(workload: str, layer: int = 0, matrix: int = 0) -> int:
    return WORKLOADS[workload]["index"] * 1000 + layer * 10 + matrix


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, device="cpu", mean: float = 0.0) -> torch.Tensor:
    """fp32 N(mean, std^2) draw of the given shape."""
    t = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def uniform(shape, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    t = torch.rand(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return t.mul_(hi - lo).add_(lo)


def weight(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    return normal((M, K), WEIGHT_STD, seed, device)


def chain_weight(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """W ~ N(0, 1/K): a product y = W x then has per-element variance equal to
    that of x, so that a chain of products (each reading the previous output)
    stays in range however long it is."""
    return normal((M, K), K ** -0.5, seed, device)


def activation(K: int, seed: int, device="cpu", rows: int | None = None) -> torch.Tensor:
    shape = (K,) if rows is None else (rows, K)
    return normal(shape, 1.0, seed, device)


def tiny(device="cpu"):
    """Tiny GEMV case: (W 1024x1024, x 1024), seed 0 for W and 1 for x."""
    return weight(1024, 1024, seed_of("tiny", 0, 0), device), activation(1024, seed_of("tiny", 0, 1), device)


@dataclass
class KVLayer:
    K: torch.Tensor        # [tokens][kv_heads][head_dim]
    V: torch.Tensor        # [tokens][kv_heads][head_dim]
    mu: torch.Tensor       # [kv_heads][head_dim] per-channel mean of K
    K_calib: torch.Tensor  # [calib_tokens][kv_heads][head_dim], a separate draw


def kv_layer(layer: int, tokens: int, kv_heads: int, head_dim: int, calib_tokens: int,
             device="cpu") -> KVLayer:
    mu = uniform((kv_heads, head_dim), -2.0, 2.0, seed_of("kv-write", layer, 0), device)
    K = normal((tokens, kv_heads, head_dim), 1.0, seed_of("kv-write", layer, 1), device)
    K.add_(mu)
    V = normal((tokens, kv_heads, head_dim), 1.0, seed_of("kv-write", layer, 2), device)
    Kc = normal((calib_tokens, kv_heads, head_dim), 1.0, seed_of("kv-write", layer, 3), device)
    Kc.add_(mu)
    return KVLayer(K, V, mu, Kc)


def adversarial_blocks(device="cpu") -> torch.Tensor:
    """Rows of 32-value blocks with the edge cases quantizers get wrong:
    all zero, a single spike, exact .5 ties, +-amax, constants, fp16-subnormal
    scales, huge dynamic range. Shape (n_blocks, 32)."""
    rows = []
    z = torch.zeros(32)
    rows.append(z.clone())                                   # all zero
    r = z.clone(); r[5] = 3.0; rows.append(r)                # single spike
    r = z.clone(); r[31] = -3.0; rows.append(r)              # single negative spike, last lane
    r = torch.arange(32, dtype=torch.float32) - 15.5; rows.append(r)  # .5 offsets
    r = torch.full((32,), 0.5); r[0] = 7.0; rows.append(r)   # Q4_0 ties at d = 1
    r = torch.full((32,), 2.5); r[0] = -7.0; rows.append(r)
    r = torch.full((32,), 63.5); r[1] = 127.0; rows.append(r)  # Q8_0 ties at d = 1
    r = torch.full((32,), 1.25); rows.append(r)              # constant block
    r = torch.full((32,), -1e-3); rows.append(r)             # constant negative
    r = torch.linspace(-1e-6, 1e-6, 32); rows.append(r)      # subnormal fp16 scale
    r = torch.linspace(-3e-8, 3e-8, 32); rows.append(r)      # scale underflows to 0
    r = torch.zeros(32); r[0] = 6e4; r[1] = 1e-3; rows.append(r)  # huge range
    r = torch.zeros(32); r[7] = -8.0; rows.append(r)         # negative amax
    r = torch.tensor([(-1.0) ** i * (i + 1) for i in range(32)]); rows.append(r)
    return torch.stack(rows).to(device)


INPUT_ORDER = ("attn_in", "attn_out", "ffn_in", "ffn_hidden")


@dataclass
class PlanEntry:
    layer: int
    name: str
    M: int
    K: int
    w_seed: int
    x_key: tuple   # (layer, input name); matrices with the same key share one x
    x_seed: int


def decode_plan(workload: str) -> list:
    """Matrices of one decode step in execution order, with their seeds.
    Weight seeds: workload*1000 + layer*10 + matrix index; activation seeds:
    workload*1000 + 500 + layer*10 + input index."""
    cfg = WORKLOADS[workload]
    plan = []
    for layer in range(cfg["layers"]):
        for mi, (name, M, K) in enumerate(cfg["layer"]):
            inp = LAYER_INPUT[name]
            plan.append(PlanEntry(layer, name, M, K, seed_of(workload, layer, mi), (layer, inp),
                                  cfg["index"] * 1000 + 500 + layer * 10 + INPUT_ORDER.index(inp)))
    return plan
