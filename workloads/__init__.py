"""Seeded synthetic inputs for the PISA prefill and decode workloads.

This module is shared by the CPU oracle's tests and by the GPU library's tests and
benchmark. It holds none of the method's arithmetic: only random numbers and the
structure of the inputs (block-mean key offsets, planted "needle" keys).

Random numbers are counter based, so any slice of any tensor can be produced on any
device without producing the rest, and CPU and GPU produce identical bits:

* SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014): output n of a stream with key ``k`` is ``mix64(k + (n+1)*GOLDEN)``.
* A standard-normal-like variate from 12 uniform 16-bit integers (Irwin-Hall sum,
  three SplitMix64 outputs per element): ``x = (sum - 393210) / 65536`` has mean 0
  and variance ``1 - 2**-32``.  Every step is integer arithmetic or an exact float
  operation, so the value is bit-identical on every device; it is rounded once to
  bf16 (round to nearest even) by torch's conversion.

Layouts (all row-major, last dimension contiguous):
  Q  [B, N, H_q, d]     K, V [B, H_kv, N, d]
  decode step: q [B, H_q, d], k, v [B, H_kv, d]
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

# stream identifiers
S_Q, S_K, S_V, S_OFF, S_NEEDLE, S_DQ, S_DK, S_DV = 1, 2, 3, 4, 5, 6, 7, 8

IH_MEAN = 12 * 65535 // 2          # 393210 = 12 * 32767.5
IH_SCALE = 1.0 / 65536.0


def _s64(x: int) -> int:
    x &= MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


_S_GOLDEN, _S_MIX1, _S_MIX2 = _s64(GOLDEN), _s64(MIX1), _s64(MIX2)


def mix64(z: int) -> int:
    """SplitMix64 finaliser on Python integers (reference for small draws)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    return mix64((mix64(seed) + stream) & MASK64)


class Stream:
    """Sequential SplitMix64 stream on Python integers."""

    def __init__(self, seed: int, stream: int):
        self.key = stream_key(seed, stream)
        self.n = 0

    def next(self) -> int:
        self.n += 1
        return mix64((self.key + self.n * GOLDEN) & MASK64)

    def below(self, m: int) -> int:
        return self.next() % m


def _lsr(x: torch.Tensor, s: int) -> torch.Tensor:
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix_t(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _S_MIX1
    z = (z ^ _lsr(z, 27)) * _S_MIX2
    return z ^ _lsr(z, 31)


def splitmix_outputs(key: int, n: torch.Tensor) -> torch.Tensor:
    """Output number ``n`` (int64 tensor, 0-based) of the stream with this key."""
    return _mix_t(_s64(key) + (n + 1) * _S_GOLDEN)


def normal_f32(key: int, idx: torch.Tensor) -> torch.Tensor:
    """Irwin-Hall(12) variate for each element index in ``idx`` (int64), as float32."""
    base = idx * 3
    s = torch.zeros_like(idx)
    for j in range(3):
        h = splitmix_outputs(key, base + j)
        s += h & 0xFFFF
        s += _lsr(h, 16) & 0xFFFF
        s += _lsr(h, 32) & 0xFFFF
        s += _lsr(h, 48)
    return (s - IH_MEAN).to(torch.float32) * IH_SCALE


def normal_bf16(key: int, start: int, count: int, device, chunk: int = 1 << 24) -> torch.Tensor:
    """bf16 variates for the contiguous element range [start, start+count)."""
    out = torch.empty(count, dtype=torch.bfloat16, device=device)
    for c0 in range(0, count, chunk):
        c1 = min(count, c0 + chunk)
        idx = torch.arange(start + c0, start + c1, dtype=torch.int64, device=device)
        out[c0:c1] = normal_f32(key, idx).to(torch.bfloat16)
    return out


# ----------------------------------------------------------------------------------------
# workload configurations
# ----------------------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    index: int           # 1-based position in the workload list; part of the seed
    B: int
    N: int
    H_q: int
    H_kv: int
    d: int
    K: int
    C: int = 64
    g: int = 2
    offsets: bool = False          # per-(b, h_kv, leaf) key offset ~ N(0, 0.5^2 I)
    needles: int = 0               # planted needle keys per (b, h_kv)
    decode_steps: int = 0          # >0: batched decode workload, N = initial cache length
    description: str = ""

    @property
    def seed(self) -> int:
        return 0x5049534100 + self.index

    @property
    def G_Q(self) -> int:
        return self.H_q // self.H_kv

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, B=1, N=1024, H_q=4, H_kv=1, d=64, K=4, needles=2,
                     description="tiny causal prefill, N=1024, G_Q=4, d=64, K=4, 2 needles per KV head"),
    "prefill_4k": Workload("prefill_4k", 2, B=4, N=4096, H_q=16, H_kv=1, d=128, K=16, offsets=True, needles=8,
                           description="causal prefill at 4K, B=4, G_Q=16, d=128, K=16, offsets, 8 needles"),
    "prefill_32k": Workload("prefill_32k", 3, B=1, N=32768, H_q=32, H_kv=2, d=128, K=16, offsets=True, needles=32,
                            description="long causal prefill, N=32768, H_q=32, H_kv=2, d=128, K=16, offsets, 32 needles"),
    "prefill_256k": Workload("prefill_256k", 4, B=1, N=262144, H_q=16, H_kv=1, d=128, K=16, offsets=True,
                             description="selection-scale prefill, N=262144, G_Q=16, d=128, K=16, offsets"),
    "decode_128k": Workload("decode_128k", 5, B=64, N=131072, H_q=32, H_kv=8, d=128, K=16, offsets=True,
                            decode_steps=256,
                            description="batched decode, 64 sequences x 131072 cached tokens, G_Q=4, 256 steps"),
}


# ----------------------------------------------------------------------------------------
# element-indexed generators
# ----------------------------------------------------------------------------------------
def q_rows(w: Workload, b: int, ts, device="cpu") -> torch.Tensor:
    """Q[b, ts, :, :] as bf16 [len(ts), H_q, d] (computed for these rows only)."""
    ts = torch.as_tensor(ts, dtype=torch.int64, device=device)
    e = torch.arange(w.H_q * w.d, dtype=torch.int64, device=device)
    idx = ((b * w.N + ts)[:, None] * (w.H_q * w.d) + e[None, :]).reshape(-1)
    x = normal_f32(stream_key(w.seed, S_Q), idx).to(torch.bfloat16)
    return x.reshape(len(ts), w.H_q, w.d)


def make_q(w: Workload, device="cpu") -> torch.Tensor:
    n = w.B * w.N * w.H_q * w.d
    return normal_bf16(stream_key(w.seed, S_Q), 0, n, device).reshape(w.B, w.N, w.H_q, w.d)


def _offsets(w: Workload, b: int, g: int, device) -> torch.Tensor:
    M1 = (w.N + w.C - 1) // w.C
    start = ((b * w.H_kv + g) * M1) * w.d
    idx = torch.arange(start, start + M1 * w.d, dtype=torch.int64, device=device)
    return (normal_f32(stream_key(w.seed, S_OFF), idx) * 0.5).reshape(M1, w.d)


@dataclass
class Needle:
    b: int
    g: int
    pos: int
    rows: list            # 8 (t', h) query rows the needle is aimed at
    key: np.ndarray       # bf16 bit patterns [d], uint16


def needles(w: Workload) -> list:
    """Needle placements, deterministic in the workload's seed.

    Per (b, h_kv): ``w.needles`` distinct positions drawn uniformly from [C, N-1)
    (so the needle lies in a selectable past block of some later query).  Each needle
    aims at 8 query rows (t', h) with t' > pos and h in the KV head's group; its key is
    ``4 * sqrt(d) * m / |m|`` with m the mean of those 8 query vectors, rounded to
    float32 and then to bf16.  The needle replaces the key at ``pos`` (no offset).
    """
    out = []
    if w.needles <= 0 or w.N <= w.C + 1:
        return out
    st = Stream(w.seed, S_NEEDLE)
    for b in range(w.B):
        for g in range(w.H_kv):
            used = set()
            while len(used) < min(w.needles, w.N - 1 - w.C):
                p = w.C + st.below(w.N - 1 - w.C)
                if p in used:
                    continue
                used.add(p)
                rows = []
                for _ in range(8):
                    tq = p + 1 + st.below(w.N - 1 - p)
                    h = g * w.G_Q + st.below(w.G_Q)
                    rows.append((tq, h))
                qv = torch.stack([q_rows(w, b, [tq])[0, h].to(torch.float64) for tq, h in rows])
                m = qv.mean(dim=0).numpy()
                nrm = float(np.sqrt(np.sum(m * m)))
                kv = (4.0 * math.sqrt(w.d) / nrm) * m if nrm > 0 else m
                key = torch.from_numpy(kv.astype(np.float32)).to(torch.bfloat16)
                out.append(Needle(b, g, p, rows, key.view(torch.int16).numpy().view(np.uint16).copy()))
    return out


def kv_slice(w: Workload, which: str, b: int, g: int, n: int | None = None, device="cpu",
             needle_list=None) -> torch.Tensor:
    """K[b, g, :n, :] or V[b, g, :n, :] as bf16 [n, d]."""
    n = w.N if n is None else n
    stream = S_K if which == "K" else S_V
    start = ((b * w.H_kv + g) * w.N) * w.d
    x = torch.empty(n * w.d, dtype=torch.float32, device=device)
    chunk = 1 << 24
    key = stream_key(w.seed, stream)
    for c0 in range(0, n * w.d, chunk):
        c1 = min(n * w.d, c0 + chunk)
        idx = torch.arange(start + c0, start + c1, dtype=torch.int64, device=device)
        x[c0:c1] = normal_f32(key, idx)
    x = x.reshape(n, w.d)
    if which == "K" and w.offsets:
        off = _offsets(w, b, g, device)
        leaf = torch.arange(n, device=device) // w.C
        x = x + off[leaf]
    out = x.to(torch.bfloat16)
    if which == "K":
        nl = needles(w) if needle_list is None else needle_list
        for nd in nl:
            if nd.b == b and nd.g == g and nd.pos < n:
                out[nd.pos] = torch.from_numpy(nd.key.view(np.int16)).view(torch.bfloat16).to(device)
    return out


def make_kv(w: Workload, which: str, device="cpu", n_cap: int | None = None) -> torch.Tensor:
    """Full K or V as bf16 [B, H_kv, n_cap, d]; rows >= N are zero."""
    n_cap = w.N if n_cap is None else n_cap
    out = torch.zeros(w.B, w.H_kv, n_cap, w.d, dtype=torch.bfloat16, device=device)
    nl = needles(w) if which == "K" else []
    for b in range(w.B):
        for g in range(w.H_kv):
            out[b, g, :w.N] = kv_slice(w, which, b, g, device=device, needle_list=nl)
    return out


def prefill_inputs(w: Workload, device="cpu"):
    return make_q(w, device), make_kv(w, "K", device), make_kv(w, "V", device)


def decode_step_inputs(w: Workload, step: int, device="cpu"):
    """Per-step q [B,H_q,d], k, v [B,H_kv,d]: plain variates, seed advanced by the step."""
    seed = w.seed + 1 + step
    q = normal_bf16(stream_key(seed, S_DQ), 0, w.B * w.H_q * w.d, device).reshape(w.B, w.H_q, w.d)
    k = normal_bf16(stream_key(seed, S_DK), 0, w.B * w.H_kv * w.d, device).reshape(w.B, w.H_kv, w.d)
    v = normal_bf16(stream_key(seed, S_DV), 0, w.B * w.H_kv * w.d, device).reshape(w.B, w.H_kv, w.d)
    return q, k, v


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy, contiguous)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
