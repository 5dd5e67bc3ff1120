"""The synthetic workloads and their seeded input generator.

Each workload is a list of trainable linear layers, each with activations
A [B, T, d_in] and output errors E [B, T, d_out] (the upstream gradient of the
layer output), plus the step's clip bound C and noise multiplier sigma.

Readings of the workload descriptions (stated once here):
* "N(0, v)" names a variance, so N(0, 1e-4) has standard deviation 1e-2.
* "lognormal(0, s)" is exp(s * N(0, 1)), one draw per record, multiplying
  all of that record's E rows in every layer.
* "records 0 and 3 scaled x10": E of records 0 and 3 times 10.
* "10% of records x20": round(0.1 B) records, the first ones of a seeded
  permutation, E times 20.
* "A ~ N(0,1) after GELU": A = GELU_erf(Z), Z ~ N(0, 1).
* Student-t(3): Z / sqrt(V / 3) with V a sum of three squared N(0, 1) draws.
* LoRA adapters: each adapter is two registered layers, LoRA-A (d_in -> r)
  and LoRA-B (r -> d_out), each with its own independently drawn A and E.
* Data seed of a layer = 1000 * workload index + layer index; the per-record
  scale draws use seed 1000 * workload index + 999.  Noise seed 0, step 0.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class LayerSpec:
    name: str
    d_in: int
    d_out: int
    T: int
    has_bias: bool = False


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    dtype: str                 # "f32" or "bf16"
    B: int
    layers: tuple
    C: float
    sigma: float
    a_dist: str = "normal"     # "normal" | "gelu_normal"
    a_scale: float = 1.0
    e_dist: str = "normal"     # "normal" | "student_t3"
    e_std: float = 1.0
    record_scale: str = "none"  # "none" | "lognormal" | "first_records" | "perm_fraction"
    record_scale_param: float = 0.0
    record_scale_factor: float = 1.0
    record_list: tuple = ()
    noise_seed: int = 0
    step: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def ncoords(self) -> int:
        return sum(ly.d_out * ly.d_in + (ly.d_out if ly.has_bias else 0) for ly in self.layers)

    @property
    def input_bytes(self) -> int:
        esz = 4 if self.dtype == "f32" else 2
        return sum(self.B * ly.T * (ly.d_in + ly.d_out) * esz for ly in self.layers)

    def scaled(self, **kw) -> "Workload":
        d = {f: getattr(self, f) for f in self.__dataclass_fields__}
        d.update(kw)
        return Workload(**d)


def _lora_stack(n_blocks, targets, d_model, r, T):
    layers = []
    for blk in range(n_blocks):
        for t in targets:
            layers.append(LayerSpec(f"blk{blk}.{t}.lora_A", d_model, r, T))
            layers.append(LayerSpec(f"blk{blk}.{t}.lora_B", r, d_model, T))
    return tuple(layers)


def _llama_layer(T):
    r = 16
    layers = []
    for t in ("q", "k", "v", "o"):
        layers.append(LayerSpec(f"{t}_proj.lora_A", 4096, r, T))
        layers.append(LayerSpec(f"{t}_proj.lora_B", r, 4096, T))
    for t in ("gate", "up"):
        layers.append(LayerSpec(f"{t}_proj.lora_A", 4096, r, T))
        layers.append(LayerSpec(f"{t}_proj.lora_B", r, 14336, T))
    layers.append(LayerSpec("down_proj", 14336, 4096, T))
    return tuple(layers)


WORKLOADS = (
    Workload(1, "linear_f32_b8_t16_64to32_bias", "f32", 8,
             (LayerSpec("linear", 64, 32, 16, True),), C=1.0, sigma=1.0,
             record_scale="first_records", record_list=(0, 3), record_scale_factor=10.0,
             notes="single fp32 linear layer with bias; E of records 0 and 3 x10"),
    Workload(2, "opt125m_lora_r8_qv_b16_t128", "bf16", 16,
             _lora_stack(12, ("q", "v"), 768, 8, 128), C=1.0, sigma=1.0,
             e_std=1e-2, record_scale="lognormal", record_scale_param=1.0,
             notes="LoRA rank 8 on q and v of a 12-block d_model=768 stack (48 layers)"),
    Workload(3, "dense_4096x4096_b64_t512", "bf16", 64,
             (LayerSpec("linear", 4096, 4096, 512),), C=0.5, sigma=0.8,
             e_std=1e-2, record_scale="perm_fraction", record_scale_param=0.1,
             record_scale_factor=20.0,
             notes="full-weight 4096x4096 linear, ghost path"),
    Workload(4, "mlp_1024_4096_1024_t1_b4096", "bf16", 4096,
             (LayerSpec("fc1", 1024, 4096, 1), LayerSpec("fc2", 4096, 1024, 1)),
             C=1.0, sigma=1.1, a_dist="gelu_normal", e_dist="student_t3", e_std=1e-2,
             notes="non-sequence MLP, T = 1"),
    Workload(5, "llama3_8b_layer_lora_r16_down_full_b32_t2048", "bf16", 32,
             _llama_layer(2048), C=1.0, sigma=1.0,
             e_std=1e-3, record_scale="lognormal", record_scale_param=1.5,
             notes="LoRA r16 on q/k/v/o/gate/up + full-weight down_proj"),
)


def by_index(i: int) -> Workload:
    for w in WORKLOADS:
        if w.index == i:
            return w
    raise KeyError(i)


def by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def record_scales(w: Workload, device="cpu") -> torch.Tensor:
    """Per-record multiplier of E (float32 [B]); ones when the workload has none."""
    s = torch.ones(w.B, dtype=torch.float32)
    g = _gen("cpu", 1000 * w.index + 999)
    if w.record_scale == "lognormal":
        s = torch.exp(w.record_scale_param * torch.randn(w.B, generator=g, dtype=torch.float64)).float()
    elif w.record_scale == "first_records":
        for r in w.record_list:
            if r < w.B:
                s[r] = w.record_scale_factor
    elif w.record_scale == "perm_fraction":
        k = int(round(w.record_scale_param * w.B))
        perm = torch.randperm(w.B, generator=g)
        s[perm[:k]] = w.record_scale_factor
    return s.to(device)


def generate_layer(w: Workload, layer_index: int, device="cpu", T: int | None = None):
    """Draw (A, E) for one layer: tensors [B, T, d_in] and [B, T, d_out] in w's dtype.

    Values are drawn in float32 with a generator seeded by
    1000 * w.index + layer_index on ``device``, then rounded to the dtype.
    """
    ly = w.layers[layer_index]
    T = ly.T if T is None else T
    g = _gen(device, 1000 * w.index + layer_index)
    f32 = torch.float32
    A = torch.randn(w.B, T, ly.d_in, generator=g, device=device, dtype=f32)
    if w.a_dist == "gelu_normal":
        A = torch.nn.functional.gelu(A)
    if w.a_scale != 1.0:
        A.mul_(w.a_scale)
    if w.e_dist == "student_t3":
        Z = torch.randn(w.B, T, ly.d_out, generator=g, device=device, dtype=f32)
        V = torch.zeros_like(Z)
        for _ in range(3):
            V.add_(torch.randn(w.B, T, ly.d_out, generator=g, device=device, dtype=f32).square_())
        E = Z.div_(V.div_(3.0).sqrt_())
        del V
    else:
        E = torch.randn(w.B, T, ly.d_out, generator=g, device=device, dtype=f32)
    if w.e_std != 1.0:
        E.mul_(w.e_std)
    s = record_scales(w, device)
    if not bool((s == 1).all()):
        E.mul_(s.view(-1, 1, 1))
    return A.to(w.torch_dtype).contiguous(), E.to(w.torch_dtype).contiguous()
