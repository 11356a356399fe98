"""Seeded synthetic inputs for the MDN memory update (shared by tests/bench).

This module holds no arithmetic of the method: it only draws inputs with the
shapes and distributions of the benchmark workloads and offers the relative-L2
error metric.  Both the CUDA path's tests and the oracle consume what it
returns.

Distributions (per token and head):
  q, k   ~ N(0, 1), then L2-normalised over the head dimension in fp32
         (x / ||x||_2, no epsilon), then cast to the input dtype
  v      ~ N(0, 1), cast to the input dtype
  alpha  = exp(-U(0, 0.1))          retention
  mu     ~ U(0, 0.9)                momentum retention
  eta    = sigmoid(N(0, 1))         gradient scale
  beta   = 1 (passed as "absent"), or sigmoid(N(0, 1)) when requested
  S0, M0 = 0, or 0.01 * N(0, 1) (fp32)
Variable-length packing draws lengths from U{128..4096} while the running
total plus the draw stays below the target; the last sequence takes the
remainder (it may be shorter than 128).
"""
from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int = 1
    T: int = 0
    H: int = 1
    D: int = 128
    dtype: str = "bf16"          # dtype of q, k, v and o
    state: str = "zero"          # "zero" tensors, "none" (absent), "randn"
    varlen_total: int = 0        # > 0: packed variable-length sequences
    decode_steps: int = 0        # > 0: recurrent decode workload
    seed: int = 0
    chunk: int = 64
    notes: str = field(default="", compare=False)


# The five benchmark workloads (names describe the shape they stand for).
TINY_FP32 = Workload("tiny_fp32_B1_H2_T256_d64", B=1, T=256, H=2, D=64,
                     dtype="fp32", state="zero", seed=0)
PREFILL_400M = Workload("prefill_400m_B8_H8_T2048_d128", B=8, T=2048, H=8,
                        D=128, dtype="bf16", state="zero", seed=1)
PREFILL_1P3B_LONG = Workload("prefill_1p3b_B1_H16_T16384_d128", B=1, T=16384,
                             H=16, D=128, dtype="bf16", state="randn", seed=2)
VARLEN_PACKED = Workload("varlen_packed_T32768_H16_d128", B=1, T=32768, H=16,
                         D=128, dtype="bf16", state="none",
                         varlen_total=32768, seed=3)
DECODE = Workload("decode_N256_H16_d128_1000steps", B=256, T=1, H=16, D=128,
                  dtype="bf16", state="randn", decode_steps=1000, seed=4)

ALL = [TINY_FP32, PREFILL_400M, PREFILL_1P3B_LONG, VARLEN_PACKED, DECODE]
# fp32 inputs at the 400M-model shapes: a timing and parity case of the
# split-operand tensor-core path, not one of the five workloads above
PREFILL_400M_FP32 = Workload("prefill_400m_fp32_B8_H8_T2048_d128", B=8, T=2048, H=8, D=128,
                             dtype="fp32", state="zero", seed=1)
BY_NAME = {w.name: w for w in ALL + [PREFILL_400M_FP32]}

TORCH_DTYPE = {"fp32": torch.float32, "bf16": torch.bfloat16}


def varlen_lengths(total: int, seed: int, lo: int = 128, hi: int = 4096):
    """Sequence lengths summing exactly to ``total`` (see module docstring)."""
    g = torch.Generator().manual_seed(seed * 7919 + 17)
    lens = []
    acc = 0
    while True:
        x = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        if acc + x < total:
            lens.append(x)
            acc += x
        else:
            lens.append(total - acc)
            break
    return lens


def cu_from_lengths(lens):
    cu = [0]
    for x in lens:
        cu.append(cu[-1] + x)
    return torch.tensor(cu, dtype=torch.int32)


def _normalise(x):
    return x / x.norm(dim=-1, keepdim=True)


def draw_tokens(g, shape_tok, H, D, dtype, device):
    """q, k, v for ``shape_tok`` token positions: ``[*shape_tok, H, D]``."""
    shp = (*shape_tok, H, D)
    q = _normalise(torch.randn(shp, generator=g, device=device))
    k = _normalise(torch.randn(shp, generator=g, device=device))
    v = torch.randn(shp, generator=g, device=device)
    td = TORCH_DTYPE[dtype]
    return q.to(td), k.to(td), v.to(td)


def draw_gates(g, shape, device, with_beta=False):
    alpha = torch.exp(-torch.rand(shape, generator=g, device=device) * 0.1)
    mu = torch.rand(shape, generator=g, device=device) * 0.9
    eta = torch.sigmoid(torch.randn(shape, generator=g, device=device))
    beta = (torch.sigmoid(torch.randn(shape, generator=g, device=device))
            if with_beta else None)
    return alpha, mu, eta, beta


def make_prefill(w: Workload, device="cpu", with_beta=False,
                 T: Optional[int] = None, B: Optional[int] = None,
                 H: Optional[int] = None, D: Optional[int] = None,
                 seed: Optional[int] = None, state: Optional[str] = None,
                 lengths=None):
    """Inputs of a prefill workload (optionally resized for small tests).

    Returns a dict: q, k, v ``[B, T, H, D]`` (packed ``[1, sum T, H, D]`` for
    varlen), alpha, mu, eta, beta ``[B, T, H]`` fp32 (beta may be None),
    S0, M0 ``[n_seq, H, D, D]`` fp32 or None, cu_seqlens (int32 or None),
    n_seq.
    """
    B = w.B if B is None else B
    T = w.T if T is None else T
    H = w.H if H is None else H
    D = w.D if D is None else D
    seed = w.seed if seed is None else seed
    state = w.state if state is None else state
    g = torch.Generator(device=device).manual_seed(seed)
    cu = None
    if lengths is not None or w.varlen_total:
        if lengths is None:
            lengths = varlen_lengths(T, seed)
        cu = cu_from_lengths(lengths)
        B, T = 1, int(cu[-1])
        n_seq = len(lengths)
    else:
        n_seq = B
    q, k, v = draw_tokens(g, (B, T), H, D, w.dtype, device)
    alpha, mu, eta, beta = draw_gates(g, (B, T, H), device, with_beta)
    if state == "randn":
        S0 = torch.randn((n_seq, H, D, D), generator=g, device=device) * 0.01
        M0 = torch.randn((n_seq, H, D, D), generator=g, device=device) * 0.01
    elif state == "zero":
        S0 = torch.zeros((n_seq, H, D, D), device=device)
        M0 = torch.zeros((n_seq, H, D, D), device=device)
    else:
        S0 = M0 = None
    return dict(q=q, k=k, v=v, alpha=alpha, mu=mu, eta=eta, beta=beta,
                S0=S0, M0=M0, cu_seqlens=cu, n_seq=n_seq, B=B, T=T, H=H, D=D,
                dtype=w.dtype)


def make_decode_state(w: Workload, device="cpu", N=None, H=None, D=None):
    N = w.B if N is None else N
    H = w.H if H is None else H
    D = w.D if D is None else D
    g = torch.Generator(device=device).manual_seed(w.seed)
    S = torch.randn((N, H, D, D), generator=g, device=device) * 0.01
    M = torch.randn((N, H, D, D), generator=g, device=device) * 0.01
    return S, M


def make_decode_steps(w: Workload, steps, device="cpu", N=None, H=None,
                      D=None, with_beta=False):
    """Per-step inputs for ``steps`` decode steps, stacked on dim 0.

    Returns q, k, v ``[steps, N, H, D]`` and alpha, mu, eta (, beta)
    ``[steps, N, H]``.  The stream is seeded separately from the states.
    """
    N = w.B if N is None else N
    H = w.H if H is None else H
    D = w.D if D is None else D
    g = torch.Generator(device=device).manual_seed(w.seed * 1000003 + 1)
    q, k, v = draw_tokens(g, (steps, N), H, D, w.dtype, device)
    alpha, mu, eta, beta = draw_gates(g, (steps, N, H), device, with_beta)
    return dict(q=q, k=k, v=v, alpha=alpha, mu=mu, eta=eta, beta=beta)


def rel_l2(x, ref):
    """||x - ref||_2 / ||ref||_2 over the whole tensor, in fp64."""
    x = torch.as_tensor(x).detach().double().cpu()
    ref = torch.as_tensor(ref).detach().double().cpu()
    den = ref.norm().item()
    num = (x - ref).norm().item()
    if den == 0.0:
        return num
    return num / den
