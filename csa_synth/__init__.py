"""Seeded synthetic inputs for one layer of Compressed Sparse Attention.

This module is shared by the CPU oracle tests, the GPU parity tests and the
bench.  It only draws random numbers and lays them out in the buffer formats
the library takes; it holds none of the method's arithmetic (no projection,
pooling, normalisation, rotation, scoring or softmax).  Every tensor is drawn
from its own PCG64 stream keyed by ``[seed, config id, tensor id, extra...]``,
in float32, and converted to the storage dtype by torch's own cast, so both
sides of a comparison see identical bytes.

Shapes follow the DeepSeek-V4-Flash layer described in "feat: add DeepSeek-V4
(Pro/Flash) model support" (mlx-lm #1189, Thump604's fixes: ratio-4
compressor ``ape (4, 1024)``, ``wkv/wgate (1024, 4096)``; stepnoy's notes on
``index_topk`` 512 and the 128-token sliding window) and in "DeepSeek-V4-Flash:
native deepseek_v4 AR backend" (MTPLX #216, "What V4 adds": 64 query heads over
one 512-dim latent, per-head sink logits).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np
import torch

SEED = 0

# tensor ids of the per-tensor random streams
_T_X, _T_Q, _T_KV, _T_IQ, _T_IW = 1, 2, 3, 4, 5
_T_WKV, _T_WGATE, _T_APE = 10, 11, 12
_T_SINK = 20
_T_POOL, _T_IKEY, _T_WIN, _T_FRONT_A, _T_FRONT_I = 30, 31, 32, 33, 34
_T_HIDDEN = 40
_POOL_ATTN, _POOL_INDEX = 0, 1


@dataclass(frozen=True)
class Config:
    """One workload: layer dimensions plus the run shape."""

    cid: int
    name: str
    dtype: str  # "f32" or "bf16": storage dtype of activations, weights, caches
    B: int
    H: int
    D: int
    R: int
    W: int
    ratio: int
    Hi: int
    Di: int
    topk: int
    X: int
    rope_base: float
    ctx: int = 0  # tokens already in the cache when the run starts
    steps: int = 0  # decode steps
    T: int = 0  # prefill chunk length (0: decode workload)
    prefill_tokens: int = 0  # tokens compressed from seeded hidden states before decoding
    rms_eps: float = 1e-6
    rollback: int = 0  # extra ring slots for exact trims (window W + rollback, frontier + rollback)
    extra: dict = field(default_factory=dict)

    @property
    def lanes(self) -> int:
        return 2 if self.ratio == 4 else 1

    @property
    def frontier_slots(self) -> int:
        """Frontier ring slots, the rollback journal included."""
        return (2 * self.ratio if self.ratio == 4 else self.ratio) + self.rollback

    @property
    def ring_slots(self) -> int:
        """Window ring slots: W plus the rollback margin."""
        return self.W + self.rollback

    @property
    def has_indexer(self) -> bool:
        return self.ratio == 4

    @property
    def storage(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / np.sqrt(self.D)))

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


_FLASH = dict(dtype="bf16", H=64, D=512, R=64, W=128, ratio=4, Hi=64, Di=128, topk=512, X=4096,
              rope_base=160000.0)

CONFIGS = {
    1: Config(cid=1, name="tiny-f32-decode-256", dtype="f32", B=1, H=8, D=64, R=16, W=32, ratio=4,
              Hi=4, Di=32, topk=16, X=128, rope_base=10000.0, ctx=0, steps=256),
    2: Config(cid=2, name="flash-decode-b1-ctx8k", B=1, ctx=0, steps=1, prefill_tokens=8192, **_FLASH),
    3: Config(cid=3, name="flash-decode-b32-ctx32k", B=32, ctx=32768, steps=256, **_FLASH),
    4: Config(cid=4, name="flash-r128-decode-b16-ctx256k", B=16, ctx=262144, steps=64,
              **{**_FLASH, "ratio": 128}),
    5: Config(cid=5, name="flash-prefill-t4096-ctx64k", B=1, ctx=65536, T=4096, **_FLASH),
}


def _rng(cfg: Config, tensor_id: int, *extra: int) -> np.random.Generator:
    return np.random.default_rng([SEED, cfg.cid, tensor_id, *[int(e) for e in extra]])


def _normal(cfg: Config, shape, tensor_id: int, *extra: int, scale: float = 1.0) -> np.ndarray:
    a = _rng(cfg, tensor_id, *extra).standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        a = a * np.float32(scale)
    return a


def _as(cfg: Config, a: np.ndarray) -> torch.Tensor:
    """fp32 draws -> storage dtype (torch's round-to-nearest-even cast)."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(cfg.storage)


def inv_freq(cfg: Config) -> torch.Tensor:
    """RoPE frequency table passed to the library: base^(-2i/R), i < R/2, as fp32.

    The layer takes this table as an input (a caller could pass a YaRN-scaled
    table instead); compress layers use base 160000, the tiny case 10000.
    """
    i = np.arange(cfg.R // 2, dtype=np.float64)
    return torch.from_numpy((cfg.rope_base ** (-2.0 * i / cfg.R)).astype(np.float32))


@dataclass
class Compressor:
    wkv: torch.Tensor  # [L*d, X] storage dtype
    wgate: torch.Tensor  # [L*d, X]
    ape: torch.Tensor  # [r, L*d] fp32
    norm_w: torch.Tensor  # [d] fp32
    d: int


def compressor(cfg: Config, which: str) -> Compressor:
    """Weights of the attention pool ("attn", d = D) or the index pool ("index", d = Di)."""
    pid = _POOL_ATTN if which == "attn" else _POOL_INDEX
    d = cfg.D if which == "attn" else cfg.Di
    L = cfg.lanes
    s = 1.0 / np.sqrt(cfg.X)
    wkv = _as(cfg, _normal(cfg, (L * d, cfg.X), _T_WKV, pid, scale=s))
    wgate = _as(cfg, _normal(cfg, (L * d, cfg.X), _T_WGATE, pid, scale=s))
    ape = torch.from_numpy(_normal(cfg, (cfg.ratio, L * d), _T_APE, pid))
    norm_w = torch.ones(d, dtype=torch.float32)
    return Compressor(wkv=wkv, wgate=wgate, ape=ape, norm_w=norm_w, d=d)


def sinks(cfg: Config) -> torch.Tensor:
    return torch.from_numpy(_normal(cfg, (cfg.H,), _T_SINK))


@dataclass
class StepInputs:
    x: torch.Tensor  # [B, 1, X]
    q: torch.Tensor  # [B, H, D]
    kv: torch.Tensor  # [B, D]
    iq: torch.Tensor  # [B, Hi, Di]
    iw: torch.Tensor  # [B, Hi]


def step_inputs(cfg: Config, step: int, B: int | None = None) -> StepInputs:
    """Per-token activations of decode step ``step`` (N(0,1), rounded to storage)."""
    B = cfg.B if B is None else B
    return StepInputs(
        x=_as(cfg, _normal(cfg, (B, 1, cfg.X), _T_X, 1, step)),
        q=_as(cfg, _normal(cfg, (B, cfg.H, cfg.D), _T_Q, 1, step)),
        kv=_as(cfg, _normal(cfg, (B, cfg.D), _T_KV, 1, step)),
        iq=_as(cfg, _normal(cfg, (B, cfg.Hi, cfg.Di), _T_IQ, 1, step)),
        iw=_as(cfg, _normal(cfg, (B, cfg.Hi), _T_IW, 1, step)),
    )


def hidden(cfg: Config, T: int, B: int | None = None, tag: int = 0) -> torch.Tensor:
    """Hidden states [B, T, X] fed to the compressors before decoding (cache build)."""
    B = cfg.B if B is None else B
    return _as(cfg, _normal(cfg, (B, T, cfg.X), _T_HIDDEN, tag))


def chunk_inputs(cfg: Config, T: int | None = None) -> StepInputs:
    """Activations of one prefill chunk of T tokens (batch 1): x [1,T,X], q [T,H,D] ..."""
    T = cfg.T if T is None else T
    return StepInputs(
        x=_as(cfg, _normal(cfg, (1, T, cfg.X), _T_X, 2)),
        q=_as(cfg, _normal(cfg, (T, cfg.H, cfg.D), _T_Q, 2)),
        kv=_as(cfg, _normal(cfg, (T, cfg.D), _T_KV, 2)),
        iq=_as(cfg, _normal(cfg, (T, cfg.Hi, cfg.Di), _T_IQ, 2)),
        iw=_as(cfg, _normal(cfg, (T, cfg.Hi), _T_IW, 2)),
    )


@dataclass
class Cache:
    """Per-layer state in the library's buffer formats (all torch CPU tensors)."""

    pool: torch.Tensor  # [B, cap, D] storage
    ikeys: torch.Tensor | None  # [B, cap, Di] storage (ratio-4 layers only)
    window: torch.Tensor  # [B, W, D] ring, slot t mod W
    front_attn: torch.Tensor  # [B, F, 2*L*D] ring of projected (kv | gate) rows, slot t mod F
    front_index: torch.Tensor | None  # [B, F, 2*L*Di]
    n_rows: torch.Tensor  # [B] int32
    pos: torch.Tensor  # [B] int32: position of the next token

    def clone(self) -> "Cache":
        return Cache(**{k: (None if v is None else v.clone()) for k, v in vars(self).items()})


def empty_cache(cfg: Config, cap: int, B: int | None = None) -> Cache:
    B = cfg.B if B is None else B
    L, F = cfg.lanes, cfg.frontier_slots
    z = lambda *s: torch.zeros(*s, dtype=cfg.storage)  # noqa: E731
    return Cache(
        pool=z(B, cap, cfg.D),
        ikeys=z(B, cap, cfg.Di) if cfg.has_indexer else None,
        window=z(B, cfg.ring_slots, cfg.D),
        front_attn=z(B, F, 2 * L * cfg.D),
        front_index=z(B, F, 2 * L * cfg.Di) if cfg.has_indexer else None,
        n_rows=torch.zeros(B, dtype=torch.int32),
        pos=torch.zeros(B, dtype=torch.int32),
    )


def synth_cache(cfg: Config, cap: int, B: int | None = None, ctx: int | None = None) -> Cache:
    """A cache holding ``ctx`` tokens, filled directly with seeded N(0,1) values.

    Running the compressor over 32 x 32768 tokens in a single-threaded oracle is
    out of reach, so the long-context workloads start from caches drawn at random
    in the same formats: ``ctx // ratio`` pool and index-key rows, a full window
    ring, and a frontier ring whose slots hold the projected (kv | gate) rows of
    the last tokens.  Each sequence has its own stream, so a subset of sequences
    can be regenerated alone.
    """
    B = cfg.B if B is None else B
    ctx = cfg.ctx if ctx is None else ctx
    if cfg.rollback:
        return with_rollback_slots(synth_cache(cfg.replace(rollback=0), cap, B, ctx), cfg, ctx)
    n = ctx // cfg.ratio
    assert n <= cap
    c = empty_cache(cfg, cap, B)
    L, F = cfg.lanes, cfg.frontier_slots
    for b in range(B):
        c.pool[b, :n] = _as(cfg, _normal(cfg, (n, cfg.D), _T_POOL, b))
        if cfg.has_indexer:
            c.ikeys[b, :n] = _as(cfg, _normal(cfg, (n, cfg.Di), _T_IKEY, b))
            c.front_index[b] = _as(cfg, _normal(cfg, (F, 2 * L * cfg.Di), _T_FRONT_I, b))
        c.window[b] = _as(cfg, _normal(cfg, (cfg.W, cfg.D), _T_WIN, b))
        c.front_attn[b] = _as(cfg, _normal(cfg, (F, 2 * L * cfg.D), _T_FRONT_A, b))
    c.n_rows[:] = n
    c.pos[:] = ctx
    return c


def with_rollback_slots(cache: Cache, cfg: Config, ctx: int) -> Cache:
    """The same cache (built without rollback slots, position ctx) in rings with cfg.rollback extra slots: token t's
    window row moves from slot t mod W to slot t mod (W + rollback), and its frontier entry from slot t mod F0 to
    t mod (F0 + rollback); the new slots hold zeros (no earlier tokens exist in them)."""
    out = empty_cache(cfg, cache.pool.shape[1], cache.pool.shape[0])
    out.pool.copy_(cache.pool)
    if out.ikeys is not None:
        out.ikeys.copy_(cache.ikeys)
    out.n_rows.copy_(cache.n_rows)
    out.pos.copy_(cache.pos)
    W, Wr = cfg.W, cfg.ring_slots
    F0, F = cache.front_attn.shape[1], cfg.frontier_slots
    for t in range(max(0, ctx - W), ctx):
        out.window[:, t % Wr] = cache.window[:, t % W]
    for t in range(max(0, ctx - F0), ctx):
        out.front_attn[:, t % F] = cache.front_attn[:, t % F0]
        if out.front_index is not None:
            out.front_index[:, t % F] = cache.front_index[:, t % F0]
    return out
