"""Seeded synthetic inputs for ragged batched log-probabilities.

Shared by the tests and ``bench.py`` as the ONLY common code between the CUDA path
and the oracle.  It draws random numbers and builds the input layout (lengths,
input row offsets, echo flags, tokens); it holds none of the method's arithmetic
(no output offsets, no softmax, no top-k).

Workloads (stand-ins for serving traffic; the pages measure nothing on a public
dataset, so nothing real is replaced):

* ``tiny``    B=4, lengths {3,5,1,7}, V=1000, levels=3, echo {T,F,T,F};
              N(0, 2) logits; row 0 gets its maximum copied to a second id.
* ``decode``  B=256 next-token rows, V=128256 (the Llama-3 vocabulary), levels=3,
              no echo; N(0, 3) plus one token per row spiked by +12.
* ``prefill`` B=8, lengths U[64, 2048], V=32000, levels=3, all echo; N(0, 2.5).
* ``mixed``   B=64, lengths U[1, 512], V=152064, levels=3, echo ~ Bernoulli(0.5);
              Student-t (df=3) x 2, 1 % of entries -inf, 0.1 % of rows with a
              duplicated maximum.
* ``wide``    B=32, lengths U[128, 1024], V=256000, levels=6, all echo; N(0, 1)
              rounded to multiples of 1/16 (many exact ties).

Two input variants apply to any workload: per-batch temperatures
(``with_temperatures``: uniform in [0.25, 2.0], some exactly 1.0) and VARIABLE
logits (``make_batch(..., variable_extra=n)``: the logits tensor holds only each
sequence's last positions — all of them for echo batches, 1 + U{0..n} (capped by the
length) otherwise — and ``input_row_offsets`` describes the positions).

Host-side structure comes from ``numpy.random.default_rng(seed)``; logits come from
a ``torch.Generator`` on the target device, drawn in fixed row chunks so the values
depend only on (seed, shape, device type).
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

CONFIGS = {
    "tiny": dict(B=4, lengths=[3, 5, 1, 7], V=1000, levels=3, echo=[1, 0, 1, 0],
                 dist="normal", scale=2.0, tie_rows=[0], seed=0),
    "decode": dict(B=256, next_token=True, V=128256, levels=3, echo=0,
                   dist="normal", scale=3.0, spike=12.0, seed=1),
    "prefill": dict(B=8, len_range=(64, 2048), V=32000, levels=3, echo=1,
                    dist="normal", scale=2.5, seed=2),
    "mixed": dict(B=64, len_range=(1, 512), V=152064, levels=3, echo_p=0.5,
                  dist="student_t3", scale=2.0, neg_inf_frac=0.01, dup_max_row_frac=0.001, seed=3),
    "wide": dict(B=32, len_range=(128, 1024), V=256000, levels=6, echo=1,
                 dist="normal", scale=1.0, quant=1.0 / 16.0, seed=4),
}

_CHUNK_ROWS = 512


@dataclasses.dataclass
class Batch:
    """One ragged batch. Integer tensors are int32 storage of uint32 values."""
    name: str
    logits: torch.Tensor            # f32 [T, V] (VARIABLE: [T_logits, V])
    logit_row_offsets: torch.Tensor  # int32 [B+1], rows of ``logits`` per batch
    tokens: torch.Tensor            # int32 [T_in]
    sampled_tokens: torch.Tensor    # int32 [B]
    echo: torch.Tensor              # uint8 [B]
    levels: int
    B: int
    T: int                          # rows of ``logits``
    V: int
    input_row_offsets: Optional[torch.Tensor] = None  # int32 [B+1], positions (VARIABLE only)
    temperatures: Optional[torch.Tensor] = None       # f32 [B]

    def host(self):
        """numpy copies of the integer inputs (logits stay where they are)."""
        return (self.logit_row_offsets.cpu().numpy().view(np.uint32),
                self.tokens.cpu().numpy().view(np.uint32),
                self.sampled_tokens.cpu().numpy().view(np.uint32),
                self.echo.cpu().numpy().astype(bool))

    def host_variant(self):
        """numpy copies of the optional inputs: (input offsets or None, temperatures or None)."""
        ioff = None if self.input_row_offsets is None else self.input_row_offsets.cpu().numpy().view(np.uint32)
        tau = None if self.temperatures is None else self.temperatures.cpu().numpy().astype(np.float32)
        return ioff, tau

    @property
    def positions_offsets(self) -> torch.Tensor:
        return self.logit_row_offsets if self.input_row_offsets is None else self.input_row_offsets


def _fill_logits(out: torch.Tensor, dist: str, scale: float, gen: torch.Generator,
                 neg_inf_frac: float = 0.0, quant: Optional[float] = None) -> None:
    T, V = out.shape
    dev = out.device
    for a in range(0, T, _CHUNK_ROWS):
        b = min(T, a + _CHUNK_ROWS)
        blk = out[a:b]
        if dist == "normal":
            torch.randn(blk.shape, generator=gen, device=dev, out=blk)
        elif dist == "gumbel":
            u = torch.rand(blk.shape, generator=gen, device=dev)
            u.clamp_(min=1e-20)
            blk.copy_(-torch.log(-torch.log(u)))
        elif dist == "student_t3":
            z = torch.randn(blk.shape, generator=gen, device=dev)
            chi = torch.zeros_like(z)
            for _ in range(3):
                w = torch.randn(blk.shape, generator=gen, device=dev)
                chi.addcmul_(w, w)
            blk.copy_(z / torch.sqrt(chi / 3.0))
        else:
            raise ValueError(dist)
        blk.mul_(scale)
        if quant:
            blk.div_(quant).round_().mul_(quant)
        if neg_inf_frac:
            mask = torch.rand(blk.shape, generator=gen, device=dev) < neg_inf_frac
            blk.masked_fill_(mask, float("-inf"))


def _duplicate_max(logits: torch.Tensor, rows, rng: np.random.Generator) -> None:
    """Copy each chosen row's maximum value onto a second, random id."""
    V = logits.shape[1]
    for r in rows:
        r = int(r)
        amax = int(torch.argmax(logits[r]).item())
        j = int(rng.integers(0, V - 1))
        if j >= amax:
            j += 1
        logits[r, j] = logits[r, amax]


def make_batch(name: str, device="cpu", *, B: Optional[int] = None, V: Optional[int] = None,
               max_len: Optional[int] = None, levels: Optional[int] = None,
               seed: Optional[int] = None, variable_extra: Optional[int] = None) -> Batch:
    """Build a named workload, optionally shrunk (fewer batches, smaller vocab,
    shorter sequences) while keeping its distribution and structure.

    ``variable_extra`` switches to VARIABLE logits (see the module docstring)."""
    cfg = dict(CONFIGS[name])
    seed = cfg["seed"] if seed is None else seed
    rng = np.random.default_rng(seed)
    Bn = cfg["B"] if B is None else B
    Vn = cfg["V"] if V is None else V
    lv = cfg["levels"] if levels is None else levels

    if cfg.get("next_token"):
        lengths = np.ones(Bn, dtype=np.int64)
    elif "lengths" in cfg and B is None:
        lengths = np.asarray(cfg["lengths"], dtype=np.int64)
    elif "lengths" in cfg:
        lengths = rng.integers(1, max(cfg["lengths"]) + 1, size=Bn)
    else:
        lo, hi = cfg["len_range"]
        if max_len is not None:
            hi = max(lo, min(hi, max_len))
            lo = min(lo, hi)
        lengths = rng.integers(lo, hi + 1, size=Bn)
    if max_len is not None:
        lengths = np.minimum(lengths, max_len)

    if "echo_p" in cfg:
        echo = (rng.random(Bn) < cfg["echo_p"]).astype(np.uint8)
    elif isinstance(cfg["echo"], list) and B is None:
        echo = np.asarray(cfg["echo"], dtype=np.uint8)
    elif isinstance(cfg["echo"], list):
        echo = (np.arange(Bn) % 2 == 0).astype(np.uint8)
    else:
        echo = np.full(Bn, cfg["echo"], dtype=np.uint8)

    offsets = np.zeros(Bn + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(lengths)
    T = int(offsets[-1])
    tokens = rng.integers(0, Vn, size=T, dtype=np.int64)
    sampled = rng.integers(0, Vn, size=Bn, dtype=np.int64)
    input_offsets = None
    if variable_extra is not None:
        # present logits rows: all positions of an echo batch, else the last 1 + extra
        extra = rng.integers(0, variable_extra + 1, size=Bn)
        present = np.where(echo != 0, lengths, np.minimum(lengths, 1 + extra))
        input_offsets = offsets
        offsets = np.zeros(Bn + 1, dtype=np.int64)
        offsets[1:] = np.cumsum(present)
        T = int(offsets[-1])

    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    logits = torch.empty((T, Vn), dtype=torch.float32, device=dev)
    _fill_logits(logits, cfg["dist"], cfg["scale"], gen,
                 neg_inf_frac=cfg.get("neg_inf_frac", 0.0), quant=cfg.get("quant"))
    if cfg.get("spike"):
        ids = torch.from_numpy(rng.integers(0, Vn, size=T)).to(dev)
        logits[torch.arange(T, device=dev), ids] += cfg["spike"]
    tie_rows = list(cfg.get("tie_rows", []))
    if cfg.get("dup_max_row_frac"):
        n = max(1, int(round(T * cfg["dup_max_row_frac"])))
        tie_rows += list(rng.choice(T, size=min(n, T), replace=False))
    _duplicate_max(logits, [r for r in tie_rows if r < T], rng)

    as_i32 = lambda a: torch.from_numpy(np.asarray(a, dtype=np.int64).astype(np.uint32).view(np.int32)).to(dev)
    return Batch(name=name if variable_extra is None else name + "_variable", logits=logits,
                 logit_row_offsets=as_i32(offsets), tokens=as_i32(tokens),
                 sampled_tokens=as_i32(sampled), echo=torch.from_numpy(echo).to(dev),
                 levels=lv, B=Bn, T=T, V=Vn,
                 input_row_offsets=None if input_offsets is None else as_i32(input_offsets))


def with_temperatures(batch: Batch, seed: int = 0, lo: float = 0.25, hi: float = 2.0,
                      values=None) -> Batch:
    """The same batch with per-batch temperatures: uniform in [lo, hi] with every
    fourth batch exactly 1.0, or the given ``values``."""
    if values is None:
        rng = np.random.default_rng(seed + 7919)
        values = rng.uniform(lo, hi, size=batch.B)
        values[::4] = 1.0
    tau = torch.tensor(np.asarray(values, dtype=np.float32), device=batch.logits.device)
    return dataclasses.replace(batch, name=batch.name + "_tau", temperatures=tau)


def make_next_token_batch(B: int, V: int, levels: int, dist: str = "normal", scale: float = 1.0,
                          device="cpu", seed: int = 0) -> Batch:
    """Next-token logits ``[B, V]``, offsets ``0..B``, no echo (batch/vocab grid
    and normal/Gumbel logits as in the FlashInfer sampling tests)."""
    rng = np.random.default_rng(seed)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    logits = torch.empty((B, V), dtype=torch.float32, device=dev)
    _fill_logits(logits, dist, scale, gen)
    as_i32 = lambda a: torch.from_numpy(np.asarray(a, dtype=np.int64).astype(np.uint32).view(np.int32)).to(dev)
    return Batch(name=f"next_token_{dist}_{B}x{V}", logits=logits,
                 logit_row_offsets=as_i32(np.arange(B + 1)), tokens=as_i32(rng.integers(0, V, size=B)),
                 sampled_tokens=as_i32(rng.integers(0, V, size=B)),
                 echo=torch.zeros(B, dtype=torch.uint8, device=dev), levels=levels, B=B, T=B, V=V)


def make_custom_batch(logits: torch.Tensor, lengths, echo, levels: int, seed: int = 0,
                      tokens=None, sampled=None) -> Batch:
    """Wrap caller-built logits with a ragged layout (edge-case tests)."""
    rng = np.random.default_rng(seed)
    dev = logits.device
    T, V = logits.shape
    lengths = np.asarray(lengths, dtype=np.int64)
    offsets = np.zeros(len(lengths) + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(lengths)
    if tokens is None:
        tokens = rng.integers(0, V, size=T)
    if sampled is None:
        sampled = rng.integers(0, V, size=len(lengths))
    as_i32 = lambda a: torch.from_numpy(np.asarray(a, dtype=np.int64).astype(np.uint32).view(np.int32)).to(dev)
    return Batch(name="custom", logits=logits, logit_row_offsets=as_i32(offsets), tokens=as_i32(tokens),
                 sampled_tokens=as_i32(sampled),
                 echo=torch.from_numpy(np.asarray(echo, dtype=np.uint8)).to(dev),
                 levels=levels, B=len(lengths), T=T, V=V)
