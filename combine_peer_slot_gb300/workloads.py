"""Seeded synthetic workloads for the AFD FFN-side step.

This module only draws inputs (shapes, lengths, activations, weights); it
holds none of the method's arithmetic, and both the CUDA path and the CPU
oracle consume the bytes it produces.

Recipe (per workload, numpy PCG64 ``default_rng(seed)``, in this order):
  1. seq_lens: fixed, or drawn (log-uniform rounded for the skewed workload,
     integer-uniform [1, 32] for the decode workload);
  2. x, one [n_p, hidden] block per peer, standard normal in fp32, then
     rounded once to the activation type (torch's round-to-nearest-even);
  3. router weight Wg [hidden, E] ~ N(0, 1/hidden), fp32;
  4. skewed workload only: per-expert bias b_e = 1.5 * ln(w_r), w_r the
     normalised Zipf(1.2) weight of rank r = e + 1.
Expert weights (per layer) are drawn with torch's normal generator seeded
with seed * 1000 + layer, on the device the caller names, in the order
W13 [E, 2I, hidden] ~ N(0, 1/hidden), Wd [E, hidden, I] ~ N(0, 1/I),
W13_s [2I_s, hidden] ~ N(0, 1/hidden), Wd_s [hidden, I_s] ~ N(0, 1/I_s),
then rounded to the activation type.  W13 rows 0..I-1 are the gate
projection, rows I..2I-1 the up projection.
"""
from dataclasses import dataclass, field
import math

import numpy as np


@dataclass
class Workload:
    name: str
    num_peers: int
    hidden: int
    act: str                 # "bf16" or "f32"
    num_experts: int
    topk: int
    renorm: bool
    inter: int
    shared_inter: int
    seed: int
    seq_lens: list = field(default_factory=list)
    skew_bias: bool = False
    layers: int = 1
    routed_scaling: float = 1.0
    token_cap: int = 0       # 0: the largest seq_len rounded up to 64
    description: str = ""

    @property
    def act_bytes(self):
        return 2 if self.act == "bf16" else 4

    @property
    def total_tokens(self):
        return int(sum(self.seq_lens))

    def flops_per_token(self):
        """Algorithmic FLOPs per token per layer: routed SwiGLU (gate, up,
        down) for k experts, the shared expert, and the router logits."""
        H, I, Is, k, E = self.hidden, self.inter, self.shared_inter, self.topk, self.num_experts
        return 6 * H * (k * I + Is) + 2 * H * E


def _draw_seq_lens(rng, name, num_peers):
    if name == "skewed":
        u = rng.uniform(math.log(64), math.log(16384), size=num_peers)
        return [int(round(math.exp(v))) for v in u]
    if name == "decode":
        return [int(v) for v in rng.integers(1, 33, size=num_peers)]
    raise KeyError(name)


def get(name):
    """The five workloads: a tiny fp32 smoke case, an odd-length two-peer
    fan-in, a DeepSeek-V2-Lite-shaped prefill layer, a skewed straggler
    prefill and a 26-layer decode-shaped pass."""
    if name == "tiny":
        w = Workload("tiny", 1, 128, "f32", 8, 2, True, 64, 0, 0, [16],
                     description="1 peer x 16 tokens, hidden 128 fp32, 8 experts top-2 renormalised, inter 64, no shared expert")
    elif name == "fanin":
        w = Workload("fanin", 2, 1024, "bf16", 16, 4, False, 512, 512, 1, [37, 91],
                     description="2 peers [37, 91], hidden 1024 bf16, 16 experts top-4, inter 512 + shared 512")
    elif name == "v2lite_prefill":
        w = Workload("v2lite_prefill", 4, 2048, "bf16", 64, 6, False, 1408, 2816, 2,
                     [512, 1536, 3072, 8192],
                     description="DeepSeek-V2-Lite MoE layer shape: 4 peers [512, 1536, 3072, 8192] = 13312 tokens, hidden 2048 bf16, 64 experts top-6, inter 1408, shared 2816")
    elif name == "skewed":
        w = Workload("skewed", 8, 2048, "bf16", 64, 6, False, 1408, 2816, 3, [],
                     skew_bias=True,
                     description="V2-Lite shapes, 8 peers log-uniform in [64, 16384], Zipf(1.2) router bias")
    elif name == "decode":
        w = Workload("decode", 16, 2048, "bf16", 64, 6, False, 1408, 2816, 4, [],
                     layers=26,
                     description="V2-Lite shapes, 16 peers x U{1..32} tokens, 26 layers with distinct weights")
    else:
        raise KeyError(name)
    rng = np.random.default_rng(w.seed)
    if not w.seq_lens:
        w.seq_lens = _draw_seq_lens(rng, name, w.num_peers)
    if not w.token_cap:
        w.token_cap = max(64, -(-max(w.seq_lens) // 64) * 64)
    w._rng_state = rng.bit_generator.state
    return w


NAMES = ("tiny", "fanin", "v2lite_prefill", "skewed", "decode")


def _to_act(a32, act):
    """fp32 numpy array -> activation storage (uint16 bf16 bits or float32)."""
    if act == "f32":
        return np.ascontiguousarray(a32, dtype=np.float32)
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def host_inputs(w):
    """seq_lens-shaped activations and the router parameters (numpy):
    {'x': [per-peer arrays], 'Wg': [H, E] fp32, 'bias': [E] fp32 or None}."""
    rng = np.random.default_rng(w.seed)
    rng.bit_generator.state = w._rng_state
    xs = [_to_act(rng.standard_normal((n, w.hidden), dtype=np.float32), w.act)
          for n in w.seq_lens]
    Wg = (rng.standard_normal((w.hidden, w.num_experts), dtype=np.float32)
          * np.float32(1.0 / math.sqrt(w.hidden))).astype(np.float32)
    bias = None
    if w.skew_bias:
        r = np.arange(1, w.num_experts + 1, dtype=np.float64)
        zw = r ** -1.2
        zw /= zw.sum()
        bias = (1.5 * np.log(zw)).astype(np.float32)
    return {"x": xs, "Wg": Wg, "bias": bias}


def expert_weights(w, layer, device="cpu"):
    """Per-layer expert weights as torch tensors on `device`, in the
    activation dtype: W13 [E, 2I, H], Wd [E, H, I], W13s [2Is, H] or None,
    Wds [H, Is] or None."""
    import torch
    dt = torch.bfloat16 if w.act == "bf16" else torch.float32
    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 1000 + layer)
    H, I, Is, E = w.hidden, w.inter, w.shared_inter, w.num_experts

    def draw(shape, fan_in):
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        return (t * (1.0 / math.sqrt(fan_in))).to(dt)

    W13 = draw((E, 2 * I, H), H)
    Wd = draw((E, H, I), I)
    W13s = draw((2 * Is, H), H) if Is > 0 else None
    Wds = draw((H, Is), Is) if Is > 0 else None
    return {"W13": W13, "Wd": Wd, "W13s": W13s, "Wds": Wds}


def weights_to_numpy(wt):
    """torch weight dict -> numpy arrays in storage form (uint16 bf16 bits or
    float32) for the oracle."""
    import torch
    out = {}
    for k, v in wt.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.bfloat16:
            out[k] = v.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        else:
            out[k] = v.detach().cpu().contiguous().numpy()
    return out


def custom(name, **overrides):
    """A named workload with some fields replaced (edge-case parity runs);
    new seq_lens also reset num_peers and token_cap."""
    w = get(name)
    for key, val in overrides.items():
        setattr(w, key, val)
    if "seq_lens" in overrides:
        w.num_peers = len(w.seq_lens)
        if "token_cap" not in overrides:
            w.token_cap = max(64, -(-max(max(w.seq_lens), 1) // 64) * 64)
    return w
