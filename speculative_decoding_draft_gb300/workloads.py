"""Seeded synthetic workloads for the DSpark per-step hot path.

This module only draws random inputs with the shapes and distributions of the
five benchmark configurations; it holds none of the method's arithmetic (no
bias, softmax, sampling, survival product or acceptance rule), so both the CUDA
path and the CPU oracle can consume what it produces.  The pages measure on
public benchmarks and live traffic that are not available here; these synthetic
inputs stand in for them, with the target rows generated as base logits plus
Gaussian noise so that per-position acceptance lands near the levels the pages
report.

Tensors are generated with ``torch`` on the requested device from a fixed
generator seed (data seed = 1234 + config index); large configurations should be
generated on the GPU.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Callable, Dict, Optional

import torch


@dataclass(frozen=True)
class Config:
    name: str
    index: int
    B: int                  # requests
    K_max: int              # block size (max draft length)
    V: int                  # vocabulary
    rank: int               # Markov-head rank r
    dtype: str              # "f32" | "bf16"
    u_std: float            # base draft logits ~ N(0, u_std)
    ew_std: float           # transition factors E, W ~ N(0, ew_std)
    ragged_k: bool = False  # per-request K uniform in 1..K_max
    greedy_frac: float = 0.0  # fraction of requests at temperature 0 (r mod 10 < 10 * frac)
    conf_kind: str = "sigmoid"   # "sigmoid" | "calibrated"
    noise: str = "const"         # target noise recipe
    noise_std: float = 1.0
    sps_kind: str = "tiny"
    sps_len: int = 65
    batch: int = 0               # which batch of requests (one per replica under torchrun)

    @property
    def philox_seed(self) -> int:
        return self.index + (self.batch << 32)

    @property
    def data_seed(self) -> int:
        return 1234 + self.index + 1000 * self.batch

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


CONFIGS: Dict[str, Config] = {
    "tiny": Config("tiny", 0, B=4, K_max=7, V=1000, rank=16, dtype="f32", u_std=2.0, ew_std=0.1,
                   noise="const", noise_std=0.5, sps_kind="tiny", sps_len=65),
    "qwen": Config("qwen", 1, B=64, K_max=7, V=151936, rank=256, dtype="bf16", u_std=3.0, ew_std=0.02,
                   noise="const", noise_std=1.0, sps_kind="qwen", sps_len=1025),
    "highc": Config("highc", 2, B=512, K_max=7, V=151936, rank=256, dtype="bf16", u_std=3.0, ew_std=0.02,
                    noise="halves", sps_kind="highc", sps_len=4097),
    "dsv4": Config("dsv4", 3, B=1024, K_max=5, V=129280, rank=256, dtype="bf16", u_std=3.0, ew_std=0.02,
                   conf_kind="calibrated", noise="const", noise_std=0.8, sps_kind="dsv4", sps_len=6145),
    "ragged": Config("ragged", 4, B=2048, K_max=7, V=151936, rank=256, dtype="bf16", u_std=3.0, ew_std=0.02,
                     ragged_k=True, greedy_frac=0.3, noise="uniform", sps_kind="ragged", sps_len=16385),
}

WORKLOAD_TEXT = {
    "tiny": "B=4 requests, K=7, V=1000, rank 16, fp32",
    "qwen": "Qwen3-4B-shaped step: B=64, K=7, V=151936, rank 256, bf16",
    "highc": "high concurrency: B=512, K=7, V=151936, rank 256, bf16",
    "dsv4": "DeepSeek-V4-shaped: B=1024, K=5, V=129280, rank 256, bf16",
    "ragged": "ragged mixed: B=2048, K in 1..7, V=151936, rank 256, bf16, 30% greedy",
}


def replica(cfg: Config, rank: int) -> Config:
    """The batch of requests that replica `rank` processes: the same recipe with its own data
    and random-stream seeds (rank 0 is the configuration itself)."""
    return replace(cfg, batch=rank)


def small_config(name: str = "qwen", **kw) -> Config:
    """A reduced copy of a configuration (same recipe, smaller sizes) for parity tests."""
    base = CONFIGS[name]
    sps_len = kw.pop("sps_len", None)
    c = replace(base, **kw)
    if sps_len is None:
        sps_len = c.B * (c.K_max + 1) + 1
    return replace(c, sps_len=sps_len)


def _gen(cfg: Config, device, salt: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(cfg.data_seed * 1000 + salt)
    return g


def _randn(shape, std, g, device):
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std


# ---------------------------------------------------------------------------
# draft inputs
# ---------------------------------------------------------------------------
def request_params(cfg: Config, device="cpu") -> dict:
    """anchor [B] int32, K_r [B] int32, temperature [B] float32."""
    g = _gen(cfg, device, 5)
    anchor = torch.randint(0, cfg.V, (cfg.B,), generator=g, device=device, dtype=torch.int32)
    if cfg.ragged_k:
        K_r = torch.randint(1, cfg.K_max + 1, (cfg.B,), generator=g, device=device, dtype=torch.int32)
    else:
        K_r = torch.full((cfg.B,), cfg.K_max, device=device, dtype=torch.int32)
    temperature = torch.ones(cfg.B, device=device, dtype=torch.float32)
    if cfg.greedy_frac > 0:
        r = torch.arange(cfg.B, device=device)
        temperature[(r % 10) < int(round(10 * cfg.greedy_frac))] = 0.0
    return dict(anchor=anchor, K_r=K_r, temperature=temperature)


def draft_inputs(cfg: Config, device="cpu") -> dict:
    """U [B,K_max,V], E [V,rank], W [rank,V] (storage dtype), anchor [B], K_r [B], temperature [B]."""
    g = _gen(cfg, device, 1)
    U = _randn((cfg.B, cfg.K_max, cfg.V), cfg.u_std, g, device).to(cfg.torch_dtype)
    E = _randn((cfg.V, cfg.rank), cfg.ew_std, g, device).to(cfg.torch_dtype)
    W = _randn((cfg.rank, cfg.V), cfg.ew_std, g, device).to(cfg.torch_dtype)
    return dict(U=U, E=E, W=W, **request_params(cfg, device))


def confidence_head(cfg: Config, device="cpu") -> dict:
    """Confidence-head inputs: conf_h [B, K_max] ~ N(1.5, 1), the backbone term (so that the
    head alone gives confidences like the scheduler inputs'), and conf_w [rank] ~ N(0, 1), the
    weights on the Markov embedding (with E ~ N(0, ew_std) the Markov term has standard
    deviation ew_std * sqrt(rank): 0.32 at rank 256, 0.4 for the fp32 case)."""
    g = _gen(cfg, device, 6)
    return dict(conf_h=_randn((cfg.B, cfg.K_max), 1.0, g, device) + 1.5, conf_w=_randn((cfg.rank,), 1.0, g, device))


def rnn_head(cfg: Config, device="cpu") -> dict:
    """RNN-head inputs: rnn_W [3 rank, 2 rank] ~ N(0, 1 / sqrt(2 rank)) in the storage dtype (unit-scale
    pre-activations from unit-scale inputs), rnn_x [B, K_max, 3 rank] ~ N(0, 1) float32 (the backbone term),
    and a feature scale: with the state in (-1, 1) the feature times W2 (~N(0, ew_std)) gives a bias of the
    Markov head's size when W2 is the configuration's."""
    g = _gen(cfg, device, 7)
    r = cfg.rank
    Wc = _randn((3 * r, 2 * r), 1.0 / math.sqrt(2 * r), g, device).to(cfg.torch_dtype)
    x = _randn((cfg.B, cfg.K_max, 3 * r), 1.0, g, device)
    return dict(rnn_W=Wc, rnn_x=x)


# ---------------------------------------------------------------------------
# scheduler inputs
# ---------------------------------------------------------------------------
def confidences(cfg: Config, device="cpu") -> torch.Tensor:
    """Per-position acceptance confidences c [B, K_max] in (0, 1]."""
    g = _gen(cfg, device, 2)
    if cfg.conf_kind == "sigmoid":
        return torch.sigmoid(torch.randn(cfg.B, cfg.K_max, generator=g, device=device) + 1.5)
    # calibrated: c_{r,j} = min(1, s_r^(1/K) * exp(N(0, 0.05))), s_r ~ U(0.05, 0.95)
    s = torch.rand(cfg.B, 1, generator=g, device=device) * 0.9 + 0.05
    jitter = torch.exp(torch.randn(cfg.B, cfg.K_max, generator=g, device=device) * 0.05)
    return torch.clamp(s ** (1.0 / cfg.K_max) * jitter, max=1.0)


def _sps_fn(kind: str) -> Callable[[float], float]:
    if kind == "tiny":
        return lambda b: b / (1.0 + b / 64.0)
    if kind == "qwen":
        return lambda b: min(b, 512) / 512.0
    if kind == "highc":
        return lambda b: 1.0 / (1.0 + math.ceil(b / 64.0) * 64.0 / 2048.0)
    if kind == "dsv4":
        return lambda b: (b / 3072.0) * (2.0 - b / 3072.0)
    if kind == "ragged":
        return lambda b: 1.0 if b <= 4096 else (0.8 if b <= 8192 else 0.6)
    raise ValueError(kind)


def sps_table(cfg: Config, variant: str = "literal") -> torch.Tensor:
    """SPS(B) cost table (fp64, CPU), index = verify batch tokens B, entry 0 unused.

    variant "literal" is the configuration's curve as written; "step" divides it
    by B (reading the curve as a token rate and converting it to steps/sec),
    which makes it fall with B so that the early stop is exercised.
    """
    f = _sps_fn(cfg.sps_kind)
    t = torch.zeros(cfg.sps_len, dtype=torch.float64)
    for b in range(1, cfg.sps_len):
        t[b] = f(float(b)) if variant == "literal" else f(float(b)) / float(b)
    return t


# ---------------------------------------------------------------------------
# target rows
# ---------------------------------------------------------------------------
def noise_std(cfg: Config, device="cpu") -> torch.Tensor:
    g = _gen(cfg, device, 3)
    r = torch.arange(cfg.B, device=device)
    if cfg.noise == "const":
        return torch.full((cfg.B,), cfg.noise_std, device=device)
    if cfg.noise == "halves":
        lo = torch.full((cfg.B,), 0.3, device=device)
        return torch.where(r < cfg.B // 2, lo, lo * 5.0)
    if cfg.noise == "uniform":
        return torch.rand(cfg.B, generator=g, device=device) * 1.8 + 0.2
    raise ValueError(cfg.noise)


def target_dense(cfg: Config, U: torch.Tensor, K_r: torch.Tensor, device=None) -> torch.Tensor:
    """Target logits for every position, [B, K_max+1, V] in the storage dtype.

    Row j < K_r is the base draft row U[:, j] plus N(0, sigma_r) noise (the
    target at draft position j+1); rows j >= K_r are fresh N(0, u_std) rows
    (the bonus row after the last draft position, and unused padding).
    """
    device = U.device if device is None else device
    g = _gen(cfg, device, 4)
    sig = noise_std(cfg, device).view(cfg.B, 1, 1)
    out = torch.empty(cfg.B, cfg.K_max + 1, cfg.V, dtype=cfg.torch_dtype, device=device)
    for j in range(cfg.K_max + 1):   # per position to bound temporary memory
        fresh = _randn((cfg.B, cfg.V), cfg.u_std, g, device)
        if j < cfg.K_max:
            noisy = U[:, j].float() + _randn((cfg.B, cfg.V), 1.0, g, device) * sig[:, 0]
            use = j < K_r.to(device)
            row = torch.where(use.view(-1, 1), noisy, fresh)
        else:
            row = fresh
        out[:, j] = row.to(cfg.torch_dtype)
    return out


def flatten_targets(tgt_dense: torch.Tensor, ell: torch.Tensor):
    """Gather rows 0..ell_r of each request into the flattened ragged layout.

    Returns (tgt_flat [sum(ell+1), V], tgt_off [B+1] int32).  Pure indexing.
    """
    B, Kp1, V = tgt_dense.shape
    ell = ell.to(tgt_dense.device).long()
    counts = ell + 1
    off = torch.zeros(B + 1, dtype=torch.int64, device=tgt_dense.device)
    off[1:] = torch.cumsum(counts, 0)
    req = torch.repeat_interleave(torch.arange(B, device=tgt_dense.device), counts)
    pos = torch.arange(int(off[-1]), device=tgt_dense.device) - off[req]
    flat = tgt_dense[req, pos]
    return flat.contiguous(), off.to(torch.int32)


def bf16_bits(t: torch.Tensor):
    """Host numpy view of a tensor for the oracle: float32 as is, bf16 as uint16 bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
