"""Seeded synthetic rollout inputs, shared by the tests, the smoke check and the bench.

This module holds no estimator arithmetic: it only draws random arrays with the
shapes and distributions of the rl-triton workloads (README "Performance":
num_envs=4096, seq_len=128; usage example: [64, 512] float tensors) and the
five workload recipes listed below. Both the float64 oracle and the CUDA path
receive exactly these arrays.

Every tensor has its own independent stream, spawned in a fixed order from
``numpy.random.SeedSequence(seed)``, so adding a tensor never changes the
others. Arrays are numpy (fp32, int32 for ``x_int``), [N, T] row-major and
time-contiguous; ``bootstrap_value`` is [N].
"""
from dataclasses import dataclass, field
from typing import Dict, Tuple

import numpy as np

# Fixed draw order: one child stream per name.
_STREAMS = ("rewards", "values", "bootstrap_value", "dones", "next_values",
            "log_rhos", "q_values", "x", "x_int")


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: sizes, distributions and estimator settings."""
    name: str
    N: int
    T: int
    estimators: Tuple[str, ...]
    p_term: float
    p_trunc: float = 0.0
    gamma: float = 0.99
    lambda_: float = 0.95
    rho_bar: float = 1.0
    c_bar: float = 1.0
    log_rho_std: float = 0.5
    seed: int = 1000
    extra: Dict[str, float] = field(default_factory=dict)


ALL7 = ("gae", "lambda_returns", "discounted_returns", "vtrace", "retrace",
        "eligibility_traces", "episodic_prefix_sum")
TRUNC5 = ("gae", "vtrace", "retrace", "lambda_returns", "discounted_returns")

# The five workload recipes. Seeds are 1000 + the recipe's index.
WORKLOADS = {
    "gae_64x512": Workload("gae_64x512", 64, 512, ("gae",), p_term=0.01,
                           seed=1001),
    "all7_4096x128": Workload("all7_4096x128", 4096, 128, ALL7, p_term=0.01,
                              seed=1002),
    "trunc5_4096x128": Workload("trunc5_4096x128", 4096, 128, TRUNC5,
                                p_term=0.01, p_trunc=0.005, seed=1003),
    "longT_256x1024": Workload("longT_256x1024", 256, 1024, ALL7,
                               p_term=0.001, gamma=0.997, seed=1004),
    "longT_256x4096": Workload("longT_256x4096", 256, 4096, ALL7,
                               p_term=0.001, gamma=0.997, seed=1004),
    "longT_256x16384": Workload("longT_256x16384", 256, 16384, ALL7,
                                p_term=0.001, gamma=0.997, seed=1004),
    "vlong_8x131072": Workload("vlong_8x131072", 8, 131072,
                               ("vtrace", "retrace"), p_term=1e-4,
                               gamma=0.999, lambda_=1.0, seed=1005),
}


def rollout(N: int, T: int, seed: int, p_term: float, p_trunc: float = 0.0,
            log_rho_std: float = 0.5, int_range: int = 100) -> Dict[str, np.ndarray]:
    """Draw one rollout batch.

    rewards, values, q_values, x, next_values, bootstrap_value ~ N(0, 1);
    log_rhos ~ N(0, log_rho_std^2); x_int ~ U{-int_range..int_range} int32.
    Done masks come from one uniform u per step: u < p_term marks a terminated
    step, p_term <= u < p_term + p_trunc a truncated one, so the two masks are
    disjoint with the exact rates. Masks are 0/1 float32. ``truncateds`` and
    ``next_values`` are present only when p_trunc > 0.
    """
    children = np.random.SeedSequence(seed).spawn(len(_STREAMS))
    g = {name: np.random.Generator(np.random.PCG64(c))
         for name, c in zip(_STREAMS, children)}
    shape = (N, T)
    f32 = np.float32
    out = {
        "rewards": g["rewards"].standard_normal(shape, dtype=f32),
        "values": g["values"].standard_normal(shape, dtype=f32),
        "bootstrap_value": g["bootstrap_value"].standard_normal((N,), dtype=f32),
    }
    u = g["dones"].random(shape, dtype=np.float64)
    out["terminateds"] = (u < p_term).astype(f32)
    if p_trunc > 0.0:
        out["truncateds"] = ((u >= p_term) & (u < p_term + p_trunc)).astype(f32)
        out["next_values"] = g["next_values"].standard_normal(shape, dtype=f32)
    out["log_rhos"] = (g["log_rhos"].standard_normal(shape, dtype=f32)
                       * f32(log_rho_std))
    out["q_values"] = g["q_values"].standard_normal(shape, dtype=f32)
    out["x"] = g["x"].standard_normal(shape, dtype=f32)
    out["x_int"] = g["x_int"].integers(-int_range, int_range + 1, size=shape,
                                       dtype=np.int32)
    return out


def workload_inputs(w: Workload, N: int = None, T: int = None,
                    seed: int = None) -> Dict[str, np.ndarray]:
    """Inputs for a named workload; N, T or seed may be overridden (parity
    tests use a few rows of a full-size recipe)."""
    return rollout(w.N if N is None else N, w.T if T is None else T,
                   w.seed if seed is None else seed, w.p_term, w.p_trunc,
                   w.log_rho_std)


def affine_inputs(N: int, T: int, seed: int, p_reset: float = 0.01,
                  a_max: float = 0.99) -> Dict[str, np.ndarray]:
    """Raw coefficients for the generic affine scan: a ~ U(-a_max, a_max),
    b ~ N(0, 1), reset ~ Bernoulli(p_reset) as 0/1 float32, x_init ~ N(0, 1)
    per row. |a| < 1 keeps every partial sum bounded."""
    children = np.random.SeedSequence(seed).spawn(4)
    g = [np.random.Generator(np.random.PCG64(c)) for c in children]
    f32 = np.float32
    return {
        "a": g[0].uniform(-a_max, a_max, (N, T)).astype(f32),
        "b": g[1].standard_normal((N, T), dtype=f32),
        "reset": (g[2].random((N, T)) < p_reset).astype(f32),
        "x_init": g[3].standard_normal((N,), dtype=f32),
    }


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, exact."""
    return (np.ascontiguousarray(h).astype(np.uint32) << 16).view(np.float32)


def compact_rollout(N: int, T: int, seed: int, p_term: float, p_trunc: float = 0.0):
    """A rollout in compact formats: rewards, values, next_values as bf16 bit
    patterns (held as int16, which every torch version can move to a GPU),
    masks as uint8; bootstrap_value float32. Returns (compact, float32 view)
    where the float32 view holds exactly the values the compact arrays
    encode, for the oracle."""
    src = rollout(N, T, seed, p_term, p_trunc)
    comp = {"bootstrap_value": src["bootstrap_value"]}
    f32 = {"bootstrap_value": src["bootstrap_value"]}
    for k in ("rewards", "values", "next_values"):
        if k in src:
            bits = to_bf16_bits(src[k])
            comp[k] = bits.view(np.int16)
            f32[k] = bf16_bits_to_f32(bits)
    for k in ("terminateds", "truncateds"):
        if k in src:
            comp[k] = (src[k] != 0).astype(np.uint8)
            f32[k] = comp[k].astype(np.float32)
    return comp, f32


def device_rollout(torch, N: int, T: int, seed: int, p_term: float, fields: Tuple[str, ...],
                   device, time_major: bool = False, int_range: int = 100):
    """Draw the named fields of a rollout directly in device memory, for sizes
    too large to draw on the host (billions of elements). Same distributions
    as ``rollout`` for those fields (rewards, values ~ N(0, 1); terminateds
    Bernoulli(p_term) as 0/1 float32; x_int ~ U{-int_range..int_range} int32;
    bootstrap_value ~ N(0, 1) per environment), drawn by torch's seeded device
    generator, one generator per field seeded from ``seed`` and the field's
    position in the fixed draw order. Arrays are [N, T], or [T, N] with
    time_major. The values differ from ``rollout``'s for the same seed; any
    row can be copied to the host for the oracle."""
    shape = (T, N) if time_major else (N, T)
    out = {}
    for name in fields:
        g = torch.Generator(device=device)
        g.manual_seed(seed * 64 + _STREAMS.index("dones" if name == "terminateds" else name))
        if name in ("rewards", "values", "q_values", "x"):
            out[name] = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        elif name == "bootstrap_value":
            out[name] = torch.randn((N,), generator=g, device=device, dtype=torch.float32)
        elif name == "terminateds":
            u = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
            out[name] = (u < p_term).to(torch.float32)
            del u
        elif name == "x_int":
            out[name] = torch.randint(-int_range, int_range + 1, shape, generator=g,
                                      device=device, dtype=torch.int32)
        else:
            raise ValueError("device_rollout draws no %r" % (name,))
    return out
