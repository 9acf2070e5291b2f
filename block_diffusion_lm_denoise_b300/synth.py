"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds no arithmetic of the method: it only draws numbers. Every value is a
pure function of (seed, tensor name, element index), computed with exact integer
operations followed by one float32 multiply and one bf16 rounding, so the same call gives
bit-identical tensors on the CPU and on a GPU. Inputs can therefore be created directly in
device memory and still be reproduced on the host.

Generator (all arithmetic mod 2**32, carried in int64 so no operation overflows):
  H(x)      : "lowbias32" integer hash (xor-shift 16, multiply 0x7feb352d, xor-shift 15,
              multiply 0x846ca68b, xor-shift 16), published by C. Wellons (hash prospector).
  key       : k1 = H(crc32(name) ^ H(seed)), k2 = H(k1 ^ 0x9e3779b9)
  u(c)      : H(H(c ^ k1) + k2) for a 32-bit counter c
  element i : the four 16-bit halves of u(2i) and u(2i+1) are summed (Irwin-Hall of four
              discrete uniforms: mean 131070, std 37837.23), centred, converted exactly to
              float32 and multiplied by sigma / 37837.23 (float32) -> approximately
              N(0, sigma^2), bounded at about 3.46 sigma. bf16 tensors round that float32
              value to nearest-even.
Uniforms use the top 24 bits of u(2i) / 2**24.
"""

from __future__ import annotations

import math
import os
import zlib
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

M32 = 0xFFFFFFFF
_IH_STD = math.sqrt(4 * (65536.0 ** 2 - 1.0) / 12.0)   # std of a sum of four U{0..65535}
_IH_MEAN = 2 * 65535                                     # mean of that sum
_CHUNK = 1 << 25


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for int64 x in [0, 2**32) and a constant c < 2**32, exactly."""
    lo = x & 0xFFFF
    hi = x >> 16
    return (lo * c + (((hi * c) & 0xFFFF) << 16)) & M32


def _hash32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _hash32_int(x: int) -> int:
    x &= M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & M32
    x ^= x >> 16
    return x


def _keys(seed: int, name: str):
    k1 = _hash32_int(zlib.crc32(name.encode()) ^ _hash32_int(seed))
    k2 = _hash32_int(k1 ^ 0x9E3779B9)
    return k1, k2


def _u32(counter: torch.Tensor, k1: int, k2: int) -> torch.Tensor:
    return _hash32((_hash32(counter ^ k1) + k2) & M32)


def _hash32_np(x):
    """_hash32 on a numpy uint32 array (multiplication wraps mod 2**32 natively)."""
    import numpy as np
    x = x ^ (x >> np.uint32(16))
    x = x * np.uint32(0x7FEB352D)
    x = x ^ (x >> np.uint32(15))
    x = x * np.uint32(0x846CA68B)
    x = x ^ (x >> np.uint32(16))
    return x


def _normal_f32_flat_host(n: int, sigma: float, seed: int, name: str) -> torch.Tensor:
    """The same values as the device path, computed with numpy uint32 arithmetic on the host
    cores (chunks in parallel threads: numpy releases the interpreter lock in its loops)."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor
    k1, k2 = _keys(seed, name)
    k1n, k2n = np.uint32(k1), np.uint32(k2)
    scale = np.float32(float(torch.tensor(sigma / _IH_STD, dtype=torch.float32)))
    out = np.empty(n, dtype=np.float32)
    step = 1 << 22

    def work(s0):
        s1 = min(n, s0 + step)
        i = np.arange(s0, s1, dtype=np.uint64)
        c = ((2 * i) & np.uint64(M32)).astype(np.uint32)
        a = _hash32_np(_hash32_np(c ^ k1n) + k2n)
        b = _hash32_np(_hash32_np((c + np.uint32(1)) ^ k1n) + k2n)
        sm = ((a & np.uint32(0xFFFF)).astype(np.int32) + (a >> np.uint32(16)).astype(np.int32)
              + (b & np.uint32(0xFFFF)).astype(np.int32) + (b >> np.uint32(16)).astype(np.int32)
              - _IH_MEAN)
        out[s0:s1] = sm.astype(np.float32) * scale

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(work, range(0, n, step)))
    return torch.from_numpy(out)


def _normal_f32_flat(n: int, sigma: float, seed: int, name: str, device) -> torch.Tensor:
    if torch.device(device).type == "cpu":
        return _normal_f32_flat_host(n, sigma, seed, name)
    k1, k2 = _keys(seed, name)
    out = torch.empty(n, dtype=torch.float32, device=device)
    scale = torch.tensor(float(torch.tensor(sigma / _IH_STD, dtype=torch.float32)),
                         dtype=torch.float32, device=device)
    for s0 in range(0, n, _CHUNK):
        s1 = min(n, s0 + _CHUNK)
        i = torch.arange(s0, s1, dtype=torch.int64, device=device)
        a = _u32((2 * i) & M32, k1, k2)
        b = _u32((2 * i + 1) & M32, k1, k2)
        s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16) - _IH_MEAN
        out[s0:s1] = s.to(torch.float32) * scale
    return out


def normal(shape, sigma: float, seed: int, name: str, device="cpu",
           dtype=torch.bfloat16) -> torch.Tensor:
    """Approximately N(0, sigma^2) values (see module doc), as `dtype` (bf16 or fp32)."""
    n = int(math.prod(shape))
    x = _normal_f32_flat(n, sigma, seed, name, device)
    return x.to(dtype).reshape(shape)


def uniform(shape, lo: float, hi: float, seed: int, name: str, device="cpu") -> torch.Tensor:
    """float32 values lo + (hi - lo) * k / 2**24, k uniform on 0..2**24-1."""
    n = int(math.prod(shape))
    k1, k2 = _keys(seed, name)
    i = torch.arange(n, dtype=torch.int64, device=device)
    u = (_u32((2 * i) & M32, k1, k2) >> 8).to(torch.float32) * (1.0 / 16777216.0)
    lo_t = torch.tensor(lo, dtype=torch.float32, device=device)
    span = torch.tensor(hi - lo, dtype=torch.float32, device=device)
    return (lo_t + u * span).reshape(shape)


def integers(shape, high: int, seed: int, name: str, device="cpu") -> torch.Tensor:
    """int32 values in [0, high) (u mod high)."""
    n = int(math.prod(shape))
    k1, k2 = _keys(seed, name)
    i = torch.arange(n, dtype=torch.int64, device=device)
    return (_u32((2 * i) & M32, k1, k2) % high).to(torch.int32).reshape(shape)


def bernoulli(shape, p: float, seed: int, name: str, device="cpu") -> torch.Tensor:
    """bool values, True with probability p (top 24 bits below p * 2**24)."""
    n = int(math.prod(shape))
    k1, k2 = _keys(seed, name)
    i = torch.arange(n, dtype=torch.int64, device=device)
    return ((_u32((2 * i) & M32, k1, k2) >> 8) < int(p * 16777216)).reshape(shape)


# ----------------------------------------------------------------------------------------
# Workload presets
# ----------------------------------------------------------------------------------------

@dataclass
class Dims:
    B: int
    S: int
    d: int
    Hq: int
    Hkv: int
    D: int
    V: int
    Lmax: int
    n_layers: int

    def as_dict(self):
        return dict(B=self.B, S=self.S, d=self.d, Hq=self.Hq, Hkv=self.Hkv, D=self.D,
                    V=self.V, Lmax=self.Lmax, n_layers=self.n_layers)


@dataclass
class Workload:
    """All tensors of one synthetic problem (weights stored [out, in])."""
    name: str
    dims: Dims
    gamma: float
    T: int
    t: int
    layers: List[Dict[str, torch.Tensor]] = field(default_factory=list)
    w_lm: Optional[torch.Tensor] = None
    emb: Optional[torch.Tensor] = None
    pos: Optional[torch.Tensor] = None
    h: Optional[torch.Tensor] = None
    phi_table: Optional[torch.Tensor] = None
    tokens: Optional[torch.Tensor] = None
    masked: Optional[torch.Tensor] = None
    ctx_len: Optional[torch.Tensor] = None


def _layer(seed: int, l: int, dm: Dims, sig_w_in: float, sig_w_o: float, sig_kv: float,
           device, B_kv: Optional[int] = None) -> Dict[str, torch.Tensor]:
    Bk = dm.B if B_kv is None else B_kv
    N = (dm.Hq + 2 * dm.Hkv) * dm.D
    return dict(
        wqkv=normal((N, dm.d), sig_w_in, seed, f"L{l}.wqkv", device),
        wo=normal((dm.d, dm.Hq * dm.D), sig_w_o, seed, f"L{l}.wo", device),
        ada_E=normal((6, dm.d), 0.02, seed, f"L{l}.ada_E", device, torch.float32),
        k_ctx=normal((Bk, dm.Hkv, dm.Lmax, dm.D), sig_kv, seed, f"L{l}.k_ctx", device),
        v_ctx=normal((Bk, dm.Hkv, dm.Lmax, dm.D), sig_kv, seed, f"L{l}.v_ctx", device),
    )


def phi_table(T: int, d: int, seed: int, device="cpu", sigma: float = 0.25) -> torch.Tensor:
    """Shared adaLN-single timestep vectors phi(t) for t = 1..T, fp32 [T, 6, d].

    The pages do not define the timestep MLP; these are seeded stand-ins, one independent
    draw per step (row t-1 belongs to tau = t / T)."""
    return normal((T, 6, d), sigma, seed, "phi_table", device, torch.float32)


# Global hidden-state scale for the mid-size single step; produced by
# tests/golden/calibrate_mid_scale.py from the oracle (fraction of masked rows with
# conf >= 0.8 near 30%).
MID_STEP_H_SCALE = 6.5


def tiny_step(device="cpu", seed: int = 0) -> Workload:
    """B=1, L=64, S=16 all [MASK], 1 layer, d=256, Hq=4, Hkv=1, D=64, V=1024, t=1 of 16,
    every weight / activation / KV ~ N(0, 1/sqrt(fan_in)), adaLN table ~ N(0, 0.02)."""
    dm = Dims(B=1, S=16, d=256, Hq=4, Hkv=1, D=64, V=1024, Lmax=64, n_layers=1)
    wl = Workload("tiny_step", dm, gamma=0.8, T=16, t=1)
    wl.layers = [_layer(seed, 0, dm, 1 / math.sqrt(dm.d), 1 / math.sqrt(dm.Hq * dm.D),
                        1 / math.sqrt(dm.D), device)]
    wl.w_lm = normal((dm.V, dm.d), 1 / math.sqrt(dm.d), seed, "w_lm", device)
    wl.h = normal((dm.B * dm.S, dm.d), 1 / math.sqrt(dm.d), seed, "h", device)
    wl.phi_table = phi_table(wl.T, dm.d, seed, device)
    wl.tokens = torch.full((dm.B, dm.S), dm.V, dtype=torch.int32, device=device)
    wl.masked = torch.ones((dm.B, dm.S), dtype=torch.uint8, device=device)
    return wl


def mid_step(device="cpu", seed: int = 1, B: int = 8, L: int = 2048) -> Workload:
    """B=8, L=2048, S=16 with a seeded 50% already committed, 1 layer, d=4096, Hq=32,
    Hkv=2, D=128, V=131072; LM head ~ N(0, 0.02); hidden rows scaled by MID_STEP_H_SCALE."""
    dm = Dims(B=B, S=16, d=4096, Hq=32, Hkv=2, D=128, V=131072, Lmax=L, n_layers=1)
    wl = Workload("mid_step", dm, gamma=0.8, T=16, t=8)
    wl.layers = [_layer(seed, 0, dm, 1 / math.sqrt(dm.d), 1 / math.sqrt(dm.Hq * dm.D), 1.0,
                        device)]
    wl.w_lm = normal((dm.V, dm.d), 0.02, seed, "w_lm", device)
    wl.h = normal((dm.B * dm.S, dm.d), MID_STEP_H_SCALE, seed, "h", device)
    wl.phi_table = phi_table(wl.T, dm.d, seed, device)
    committed = bernoulli((dm.B, dm.S), 0.5, seed, "committed", device)
    toks = integers((dm.B, dm.S), dm.V, seed, "tokens", device)
    wl.tokens = torch.where(committed, toks, torch.full_like(toks, dm.V))
    wl.masked = (~committed).to(torch.uint8)
    return wl


def attention_sweep(L: int, device="cpu", seed: int = 2, B: int = 32) -> Workload:
    """Fused-attention workload: B=32, S=16, Hq=32, Hkv=2, D=128, q/K/V ~ N(0, 1) bf16."""
    dm = Dims(B=B, S=16, d=4096, Hq=32, Hkv=2, D=128, V=131072, Lmax=L, n_layers=1)
    wl = Workload(f"attention_L{L}", dm, gamma=0.8, T=16, t=1)
    wl.layers = [dict(
        q=normal((B, dm.S, dm.Hq, dm.D), 1.0, seed, "q", device),
        k_blk=normal((B, dm.S, dm.Hkv, dm.D), 1.0, seed, "k_blk", device),
        v_blk=normal((B, dm.S, dm.Hkv, dm.D), 1.0, seed, "v_blk", device),
        k_ctx=normal((B, dm.Hkv, L, dm.D), 1.0, seed, "k_ctx", device),
        v_ctx=normal((B, dm.Hkv, L, dm.D), 1.0, seed, "v_ctx", device),
    )]
    return wl


def lmhead_sweep(M: int, S: int, gamma: float, device="cpu", seed: int = 3,
                 d: int = 4096, V: int = 131072) -> Workload:
    """LM-head + commit workload: rows M = B*S, h ~ N(0, 1) / temp_row with a per-row
    temperature ~ U(0.2, 2.0), W_lm ~ N(0, 0.02), all positions masked."""
    assert M % S == 0
    B = M // S
    dm = Dims(B=B, S=S, d=d, Hq=32, Hkv=2, D=128, V=V, Lmax=0, n_layers=0)
    wl = Workload(f"lmhead_M{M}_S{S}_g{gamma}", dm, gamma=gamma, T=16, t=1)
    wl.w_lm = normal((V, d), 0.02, seed, "w_lm", device)
    temp = uniform((M, 1), 0.2, 2.0, seed, "temp", device)
    h32 = normal((M, d), 1.0, seed, "h", device, torch.float32)
    wl.h = (h32 / temp).to(torch.bfloat16)
    wl.tokens = torch.full((B, S), V, dtype=torch.int32, device=device)
    wl.masked = torch.ones((B, S), dtype=torch.uint8, device=device)
    return wl


DECODE_V = 131072

# LM-head weight scale of the decode workload whose logits are as sharp as the mid-size
# step's: about 30 % of the positions clear gamma = 0.8 in the first step (0.312 in the
# oracle on four of its sequences); produced by tests/golden/calibrate_decode_scale.py.
DECODE_W_LM_SIGMA = 0.09


def decode_loop(device="cpu", seed: int = 4, B: int = 64, L: int = 8192, n_layers: int = 6,
                kv_rows: Optional[List[int]] = None, w_lm_sigma: float = 0.02,
                emb_rows: Optional[List[int]] = None) -> Workload:
    """Full block decode: B=64, L=8192, S=16, T=16, 6 layers each with its own context KV
    (~N(0,1)), d=4096, Hq=32, Hkv=2, D=128, V=131072, gamma=0.8; emb [V+1, d] and the
    position stand-in [S, d] ~ N(0, 1); weights ~ N(0, 1/sqrt(fan_in)), W_lm ~ N(0, sigma^2)
    (w_lm_sigma: 0.02, or DECODE_W_LM_SIGMA for logits as sharp as the mid-size step's).

    kv_rows: generate the context KV only for these sequences (host-side oracle subsets);
    emb_rows: only these rows of the embedding table, stacked in the given order (a host-side
    subset for steps whose tokens are known). Values are those of the full tensors' rows (the
    generator is per element)."""
    dm = Dims(B=B, S=16, d=4096, Hq=32, Hkv=2, D=128, V=131072, Lmax=L, n_layers=n_layers)
    wl = Workload("decode_loop", dm, gamma=0.8, T=16, t=1)
    for l in range(n_layers):
        if kv_rows is None:
            wl.layers.append(_layer(seed, l, dm, 1 / math.sqrt(dm.d),
                                    1 / math.sqrt(dm.Hq * dm.D), 1.0, device))
        else:
            lay = _layer(seed, l, Dims(**{**dm.as_dict(), "Lmax": 0}), 1 / math.sqrt(dm.d),
                         1 / math.sqrt(dm.Hq * dm.D), 1.0, device)
            lay["k_ctx"] = kv_subset((B, dm.Hkv, L, dm.D), kv_rows, 1.0, seed,
                                     f"L{l}.k_ctx", device)
            lay["v_ctx"] = kv_subset((B, dm.Hkv, L, dm.D), kv_rows, 1.0, seed,
                                     f"L{l}.v_ctx", device)
            wl.layers.append(lay)
    wl.w_lm = normal((dm.V, dm.d), w_lm_sigma, seed, "w_lm", device)
    wl.emb = (normal((dm.V + 1, dm.d), 1.0, seed, "emb", device) if emb_rows is None else
              kv_subset((dm.V + 1, dm.d), emb_rows, 1.0, seed, "emb", device))
    wl.pos = normal((dm.S, dm.d), 1.0, seed, "pos", device)
    wl.phi_table = phi_table(wl.T, dm.d, seed, device)
    wl.tokens = torch.full((B, dm.S), dm.V, dtype=torch.int32, device=device)
    wl.masked = torch.ones((B, dm.S), dtype=torch.uint8, device=device)
    return wl


def kv_subset(full_shape, rows: List[int], sigma: float, seed: int, name: str,
              device="cpu") -> torch.Tensor:
    """Rows `rows` (first axis) of normal(full_shape, ...) without building the rest."""
    per = int(math.prod(full_shape[1:]))
    k1, k2 = _keys(seed, name)
    scale = torch.tensor(float(torch.tensor(sigma / _IH_STD, dtype=torch.float32)),
                         dtype=torch.float32, device=device)
    outs = []
    for r in rows:
        i = torch.arange(r * per, (r + 1) * per, dtype=torch.int64, device=device)
        a = _u32((2 * i) & M32, k1, k2)
        b = _u32((2 * i + 1) & M32, k1, k2)
        s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16) - _IH_MEAN
        outs.append((s.to(torch.float32) * scale).to(torch.bfloat16))
    return torch.stack(outs).reshape((len(rows),) + tuple(full_shape[1:]))
